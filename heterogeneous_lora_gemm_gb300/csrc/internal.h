// Declarations shared by the translation units of libmlora.so (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace mlora {

// Device slot table entry (one per adapter slot).
struct SlotRec {
    int32_t rank;    // 0 = empty slot
    int32_t rpad;    // roundup(rank, 8): row length of the stored Up block [dout x rpad]
    float scale;
    int32_t unit;    // unit offset in the arena: Down at unit*din, Up at unit*dout elements
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
    int32_t* chunk_col;    // [max_chunks] first rank column of the chunk inside its adapter
    float* v32;            // [max_tokens x max_rank] scale * Down x per row (SIMT path)
    uint16_t* vt;          // [max_chunks x tcap x CHUNK] bf16 scale * Down x, chunked (tensor path)
    float* partials;       // split-K partial tiles
    int32_t* tile_ctr;     // split-K arrival counters (zero between forwards)
};

struct PoolDims {
    int S, din, dout, max_rank, max_tokens, max_chunks, tcap;
};

// ---- launchers (each returns the launch's cudaError_t) ----
cudaError_t seg_init();   // raises the segment builder's shared memory cap (outside capture)
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
cudaError_t launch_merge_simt(bool bf16, void* W, const SlotRec* slots, int slot,
                              const void* arena_down, const void* arena_up, const PoolDims& d,
                              cudaStream_t st);

}  // namespace mlora
