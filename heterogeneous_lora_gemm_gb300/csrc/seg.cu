// Standalone segment-builder kernel (one CTA of 1024 threads), used by
// mlora_debug_segments and by the fp32 forward.  The bf16 forward runs the same
// builder (seg.cuh) in the prologue of its tensor-core shrink instead.
#include "internal.h"
#include "seg.cuh"

namespace mlora {

namespace {

constexpr int SEG_THREADS = 1024;

__global__ void __launch_bounds__(SEG_THREADS, 1)
seg_build_kernel(const int32_t* __restrict__ row_adapter, int T, const SlotRec* __restrict__ slots, Workspace ws,
                 int S, int P, int max_chunks) {
    extern __shared__ int smem[];
    const seg::Scratch sc = seg::carve(smem, S, P, max_chunks);
    seg::build<false>(row_adapter, T, slots, S, P, max_chunks, sc, true, ws);
}

}  // namespace

int seg_warps_for(int S, int warps, int scratch_ints_avail, int max_chunks, int T) {
    // as many row ranges as fit the scratch (per-(warp, slot) counters), at most one per warp
    int P = warps;
    while (P > 1 && seg::scratch_ints(S, P, max_chunks, T) > scratch_ints_avail) --P;
    return seg::scratch_ints(S, P, max_chunks, T) <= scratch_ints_avail ? P : 0;
}

cudaError_t seg_init() {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, seg_build_kernel);
    // static shared memory counts against the same per-block limit
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(seg_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - (int)fa.sharedSizeBytes);
    return e;
}

cudaError_t launch_seg_build(const int32_t* row_adapter, int T, const SlotRec* slots, const Workspace& ws,
                             const PoolDims& d, cudaStream_t st) {
    const int P = seg_warps_for(d.S, SEG_THREADS / 32, (200 * 1024) / 4, d.max_chunks, T);
    if (P < 1) return cudaErrorInvalidConfiguration;
    const size_t smem = sizeof(int) * (size_t)seg::scratch_ints(d.S, P, d.max_chunks, T);
    seg_build_kernel<<<1, SEG_THREADS, smem, st>>>(row_adapter, T, slots, ws, d.S, P, d.max_chunks);
    return cudaGetLastError();
}

}  // namespace mlora
