// Tensor-core path of the bf16 forward (tcgen05 MMA, TMA loads, TMEM accumulators).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>

#include "tc.h"

namespace mlora {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

}  // namespace

TcWorkspaceNeeds tc_workspace_needs(bool bf16, const PoolDims& d) {
    TcWorkspaceNeeds n{};
    n.need_v32 = true;
    n.partial_bytes = 0;
    n.counter_bytes = 0;
    (void)bf16;
    (void)d;
    return n;
}

bool tc_encode_up_map(CUtensorMap* map, void* up_block, int rpad, int dout) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)rpad, (cuuint64_t)dout};
    cuuint64_t strides[1] = {(cuuint64_t)rpad * 2};
    cuuint32_t box[2] = {16, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, up_block, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tc_supported(const PoolDims& d, int T) {
    (void)d;
    (void)T;
    return false;
}

cudaError_t tc_forward(const TcForwardArgs& a, cudaStream_t st) {
    (void)a;
    (void)st;
    return cudaErrorNotSupported;
}

}  // namespace mlora
