// Tensor-core (tcgen05 / TMA / TMEM) path of the bf16 forward: declarations.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace mlora {

struct TcWorkspaceNeeds {
    bool need_v32;          // the SIMT shrink/expand path is still reachable for this pool
    size_t partial_bytes;   // split-K partial tiles
    size_t counter_bytes;   // split-K arrival counters
};
TcWorkspaceNeeds tc_workspace_needs(bool bf16, const PoolDims& d);

// Encodes the TMA descriptor of one adapter's Up block [dout x rpad] (bf16,
// row-major): boxes of 16 rank columns x 128 output rows, 32-byte swizzle,
// columns past rpad read as zero.
bool tc_encode_up_map(CUtensorMap* map, void* up_block, int rpad, int dout);

// Encodes the TMA descriptor of one adapter's Down block [rank x din] (bf16,
// row-major): boxes of 64 din columns x 16 rank rows, 128-byte swizzle, rows past
// the rank read as zero.
bool tc_encode_down_map(CUtensorMap* map, void* down_block, int rank, int din);

// Raises the dynamic shared memory cap of the tensor-core kernels (call outside capture).
cudaError_t tc_init();

// Whether the tensor-core forward takes this pool shape and batch size.
bool tc_supported(const PoolDims& d, int T);

struct TcForwardArgs {
    const void* X;
    const void* W;
    void* Y;
    int T;
    bool lora;
    const int32_t* row_adapter;
    const SlotRec* slots;
    const CUtensorMap* up_maps;
    const CUtensorMap* down_maps;
    const void* arena_down;
    Workspace ws;
    PoolDims dims;
    int ext_chunk_cap;      // upper bound of K-extension chunks (sum over loaded slots)
    cudaEvent_t ev_start;   // optional profiling events around the projection kernel
    cudaEvent_t ev_stop;
};

// Records a profiling event; inside stream capture it becomes an event-record node.
cudaError_t record_profile(cudaEvent_t ev, cudaStream_t st);

// Prefill-shaped projection (T > 256), tc_prefill.cu.
cudaError_t prefill_init();
cudaError_t launch_prefill(const TcForwardArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                           const CUtensorMap& tmV, int num_sms, bool after_shrink, cudaStream_t st);
cudaError_t tc_forward(const TcForwardArgs& a, cudaStream_t st);

}  // namespace mlora
