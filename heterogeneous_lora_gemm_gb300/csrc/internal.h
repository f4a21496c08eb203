// Declarations shared by the translation units of libmlora.so (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

namespace mlora {

// Device slot table entry (one per adapter slot).
struct SlotRec {
    int32_t rank;    // 0 = empty slot
    int32_t rpad;    // roundup(rank, 8): rank units the adapter holds
    float scale;
    int32_t unit;    // first rank unit in the arena (a multiple of 8)
    int32_t chunk0;  // index of the slot's first chunk in the chunk table
};

// Arena layout, per rank unit u (one rank row of one adapter):
//   Down half: row u = [din] elements at u*din   (Down_a row k is unit u_a + k)
//   Up half:   units come in blocks of 8; block b = [dout x 8] row-major at b*8*dout,
//              so Up_a[o][k] sits at ((u_a + k) / 8 * dout + o) * 8 + (u_a + k) % 8.
__host__ __device__ inline size_t up_index(int unit, int k, int o, int dout) {
    const int u = unit + k;
    return ((size_t)(u >> 3) * dout + o) * 8 + (u & 7);
}

// One K-extension chunk of a loaded adapter: 16 rank columns (fewer in the last
// chunk of a rank that is not a multiple of 16).  The pool keeps the chunks of all
// loaded slots, in ascending slot order, in a device table that changes only on
// load, unload and compaction.
struct ChunkRec {
    int32_t slot;
    int32_t unit;    // arena rank unit of the chunk's first column (a multiple of 8)
    int32_t kval;    // valid rank columns, 1..16
    float scale;
    int32_t row0, row1;   // output rows [row0, row1) its Up columns reach (a module of a fused
                          // projection); every row for an adapter of the whole layer
};

// Bits of the device status word.
enum : uint32_t { STATUS_BAD_ROW = 1u, STATUS_TIMEOUT = 2u };

// Width of one K-extension chunk of the low-rank intermediate (one bf16 MMA K step).
constexpr int CHUNK = 16;

// Per-forward device workspace (all carved from one allocation at pool creation).
struct Workspace {
    uint32_t* status;      // [1]
    int32_t* counts;       // [S]     rows per slot
    int32_t* offsets;      // [S+1]   exclusive scan of counts
    int32_t* perm;         // [max_tokens] rows in segment order, -1 past n_valid
    int32_t* meta;         // [8]     0: n_valid, 1: n_chunks, 2: n_touched
    int32_t* chunk_slot;   // [max_chunks] slot of each K-extension chunk (touched slots ascending)
    int32_t* chunk_unit;   // [max_chunks] arena rank unit of the chunk's first rank column
    int32_t* chunk_kval;   // [max_chunks] valid rank columns of the chunk (<= CHUNK)
    float* v32;            // [max_tokens x max_rank] scale * Down x per row (SIMT path)
    uint16_t* vt;          // [max_chunks x 2 x tcap x 8] bf16 scale * Down x per loaded chunk (tensor path),
                           // each chunk's 16 rank columns as two blocks of 8 (a block's 8 tokens
                           // are one 128-byte row); written for the (chunk, token tile) pairs
                           // tmask marks, read only there
    float* partials;       // split-K partial tiles
    int32_t* tile_ctr;     // split-K arrival counters (zero between forwards)
    const ChunkRec* chunks;   // [max_chunks] chunks of the loaded slots (pool state, not per forward)
    uint8_t* tmask;        // [token tiles of 256][max_chunks] 1 = a row of the token tile uses the chunk's slot
};

struct PoolDims {
    int S, din, dout, max_rank, max_tokens, max_chunks, tcap;
};

// Sets the text returned by mlora_last_error() in the calling thread.
void set_last_error(const std::string& msg);

// ---- launchers (each returns the launch's cudaError_t) ----
cudaError_t seg_init();   // raises the segment builder's shared memory cap (outside capture)
// Row ranges (warps, at most `warps`) the segment builder can use with
// `scratch_ints_avail` ints of shared memory, and whether the row map is staged
// there too; P = 0 if even one range does not fit.
struct SegPlan {
    int P;
    bool stage_rows;
    int ints;
};
SegPlan seg_plan(int S, int warps, int scratch_ints_avail, int T);
cudaError_t launch_seg_build(const int32_t* row_adapter, int T, const SlotRec* slots,
                             const Workspace& ws, const PoolDims& d, cudaStream_t st);

// SIMT path (fp32 and bf16): shrink into v32, then base + expand into Y.
cudaError_t launch_shrink_simt(bool bf16, const void* X, const int32_t* row_adapter, int T,
                               const SlotRec* slots, const void* arena_down, const Workspace& ws,
                               const PoolDims& d, cudaStream_t st);
cudaError_t launch_base_expand_simt(bool bf16, const void* X, const void* W,
                                    const int32_t* row_adapter, int T, void* Y,
                                    const SlotRec* slots, const void* arena_up, const Workspace& ws,
                                    const PoolDims& d, bool with_lora, cudaStream_t st);
// Quantized base (quant.cu): int8 codes x per-row scale.
cudaError_t launch_dequant(bool bf16, const int8_t* q, const float* s, int dout, int din, void* W, cudaStream_t st);
cudaError_t launch_merge_quant(bool bf16, int8_t* q, float* s, const SlotRec* slots, int slot, const void* arena_down,
                               const void* arena_up, const PoolDims& d, cudaStream_t st);
// NF4 base (quant.cu): 4-bit codes [dout x din/2], absmax [din/64][dout], codebook [16] (host).
cudaError_t launch_dequant_nf4(bool bf16, const uint8_t* q, const float* absmax, const float* codebook, int dout,
                               int din, void* W, cudaStream_t st);
cudaError_t launch_merge_nf4(bool bf16, uint8_t* q, float* absmax, const float* codebook, const SlotRec* slots,
                             int slot, const void* arena_down, const void* arena_up, const PoolDims& d,
                             cudaStream_t st);
cudaError_t launch_merge_simt(bool bf16, void* W, const SlotRec* slots, int slot,
                              const void* arena_down, const void* arena_up, const PoolDims& d, float sign,
                              cudaStream_t st);

}  // namespace mlora
