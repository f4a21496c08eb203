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
    size_t tmask_bytes;     // per token tile of 256, one byte per chunk: the shrink computed it
};
TcWorkspaceNeeds tc_workspace_needs(bool bf16, const PoolDims& d);

// TMA descriptors of the whole adapter arena (bf16), encoded once per pool:
//   down   : 2D {din, units}, boxes of 64 din columns x 16 rank rows, 128-byte swizzle
//   up128  : 3D {8, dout, units/8}, boxes of 8 rank columns x 128 rows x 2 blocks, no swizzle
//   up256  : the same with 256 rows per box (prefill tiles)
//   upw128, upw256: the same boxes seen as rows of 128 bytes (8 output rows x 8 rank
//           columns: 3D {64, dout/8, units/8}): the same bytes in shared memory, in an
//           eighth of the TMA rows; only when dout % 8 == 0 (up_rows == 8), else copies
//           of up128 / up256 (up_rows == 1)
struct TcArenaMaps {
    CUtensorMap down, up128, up256, upw128, upw256;
    int up_rows;   // output rows per row of the upw maps (8, or 1 for the plain maps)
};
bool tc_encode_arena_maps(TcArenaMaps* maps, void* arena_down, void* arena_up, int units, int din, int dout);

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
    TcArenaMaps maps;
    const void* arena_down;
    const void* arena_up;   // the Up arena [units / 8][dout][8]
    Workspace ws;
    PoolDims dims;
    int n_chunks;           // chunks of the loaded slots (entries of ws.chunks: by module, then arena order)
    int tile_span;          // largest arena span of 8 consecutive chunks (first unit to last unit + 16)
    int run_stride;         // most common arena stride (rank units) of 4-chunk units, 0 = none
    int units;              // rank units of the arena
    int n_loaded;           // loaded slots
    unsigned long long* stamps;   // profiling records of the kernels' CTAs (NULL = off)
    int stamp_cap;
    // decode projection over a quantized W (W unused): 1 int8 codes [dout x din] with an
    // fp32 scale per row (qscale [dout]); 2 4-bit codes [dout x din/2] (even column in the
    // low nibble) with an fp32 scale per row and 64 columns (qscale [din/64][dout]) and
    // the 16-entry codebook qcb.  Needs T <= 256 and din % 64 == 0, and for 4-bit codes
    // dout % 4 == 0 and qscale 16-byte aligned (tc_quantized_fits).
    int qmode;
    const void* Wq;
    const float* qscale;
    float qcb[16];
};
bool tc_quantized_fits(const PoolDims& d, int T, bool nf4);

// Shrink on the CUDA cores for decode batches over many adapters with a few rows each
// (shrink_gemv.cu): one CTA per chunk of the pool plus the segment builder's CTA.
cudaError_t gemv_init();
bool gemv_shrink_fits(const PoolDims& d, int T);
cudaError_t launch_shrink_gemv(const TcForwardArgs& a, bool prefetch, cudaStream_t st);

// Prefill-shaped projection (T > 256), tc_prefill.cu.
cudaError_t prefill_init();
cudaError_t launch_prefill(const TcForwardArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                           const CUtensorMap& tmV, int num_sms, bool after_shrink, cudaStream_t st);

// Base projection Y = X W^T (T <= 256, bf16) on the decode kernel with caller-given
// scratch: `partials` (partial_bytes of fp32 partial tiles) and `counters`
// (max_tiles zeroed ints, one per 128 output features), `status` one word.
cudaError_t tc_project_with_scratch(const void* X, const void* W, int T, int din, int dout, void* Y,
                                   float* partials, size_t partial_bytes, int32_t* counters, int max_tiles,
                                   uint32_t* status, cudaStream_t st);

// Static merge of one adapter into a bf16 W on the tensor cores (merge_tc.cu).
cudaError_t merge_tc_init();
cudaError_t launch_merge_tc(void* W, const SlotRec* slots, int slot, const TcArenaMaps& maps, uint32_t* status,
                            const PoolDims& d, float sign, cudaStream_t st);
// The merge into an int8 base (codes [dout x din], din % 16 == 0, 16-byte aligned; one
// fp32 scale per row) on the tensor cores: the merged rows' max, their new codes, then
// their new scales.  `row_max`: dout words of scratch, zero on entry and on return.
cudaError_t launch_merge_quant_tc(int8_t* Wq, float* row_scale, uint32_t* row_max, const SlotRec* slots, int slot,
                                  const TcArenaMaps& maps, uint32_t* status, const PoolDims& d, cudaStream_t st);

// Encodes a bf16 tensor map (used by both tensor-core translation units).
bool tc_encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
               const cuuint32_t* box, CUtensorMapSwizzle sw);
bool tc_encode_typed(CUtensorMap* map, CUtensorMapDataType type, const void* base, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw);
cudaError_t tc_forward(const TcForwardArgs& a, cudaStream_t st);

}  // namespace mlora
