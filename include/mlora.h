/*
 * mlora.h -- C ABI of the GB300 (sm_103a) multi-LoRA linear layer.
 *
 * What the layer computes (ai-infra-kb "M031" multi-LoRA tutorial, §02; airsota
 * card "multi-LoRA serving vs merging", part 三.1; wiblog "vLLM LoRA adapter
 * batch scheduling", section on Punica's grouped matmul):
 *
 *   for a mixed batch of T rows X[T x din] in which row t names adapter a_t or none,
 *       Y[t,:] = W X[t,:]  +  scale_a * Up_a (Down_a X[t,:])      (a = a_t)
 *       Y[t,:] = W X[t,:]                                          (no adapter)
 *   with W [dout x din], Down_a [r_a x din], Up_a [dout x r_a]; the shared base
 *   product covers every row in one call, ranks may differ per adapter, and each
 *   result is written to the row it came from (original row order).
 *
 * and, as a separate call (M031 §04), the static merge W <- W + scale_a Up_a Down_a.
 *
 * Conventions for every call below
 *   - Matrices are dense and row-major: X [T x din], W [dout x din] (the layout of
 *     a torch Linear weight), Y [T x dout], Down [r x din], Up [dout x r].
 *   - Element type is the pool's dtype (MLORA_BF16: bf16 in, fp32 accumulate, bf16
 *     out with one final rounding; MLORA_F32: fp32 throughout, CUDA-core FMA only).
 *   - X, W, Y, row_adapter, perm and offsets are DEVICE pointers on the pool's
 *     device; for MLORA_BF16 X, W and Y must be 16-byte aligned.  The caller owns
 *     them.  Adapter sources given to mlora_load_adapter may be host or device
 *     memory and may be freed as soon as that call returns.
 *   - Calls taking a stream only enqueue work on it and return; errors of
 *     arguments are returned before anything is enqueued.  A pool serves one
 *     stream at a time: its forward and merge calls share the pool's workspace,
 *     so calls on one pool that overlap on the GPU race.  Calls on one pool must
 *     not be made from several host threads at once.
 *   - No call traps or asserts on the device.  A row that names a slot outside
 *     [0, max_slots) or an empty slot is treated as a row without adapter and
 *     raises a device status bit, read by mlora_pool_status.
 */
#ifndef MLORA_H
#define MLORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mlora_pool* mlora_pool_t;
/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* mlora_stream_t;

typedef enum mlora_status {
    MLORA_OK = 0,
    MLORA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, T > max_tokens */
    MLORA_ERR_BAD_SLOT = 2,      /* slot outside [0, max_slots) */
    MLORA_ERR_RANK = 3,          /* rank < 1 or rank > max_rank */
    MLORA_ERR_NOT_LOADED = 4,    /* the slot holds no adapter */
    MLORA_ERR_OOM = 5,           /* rank budget exhausted, or a device allocation failed */
    MLORA_ERR_CUDA = 6,          /* a CUDA runtime call failed (no device, launch failure, ...) */
    MLORA_ERR_DEVICE_ROW = 7,    /* (mlora_pool_status) a row named an invalid or empty slot */
    MLORA_ERR_UNSUPPORTED = 8,   /* shape outside what the kernels handle (see mlora_pool_create) */
    MLORA_ERR_DEVICE_TIMEOUT = 9 /* (mlora_pool_status) a kernel pipeline wait gave up after its limit */
} mlora_status;

typedef enum mlora_dtype { MLORA_F32 = 0, MLORA_BF16 = 1 } mlora_dtype;

typedef struct mlora_pool_info_s {
    int32_t din, dout, dtype, max_slots, max_rank, max_tokens;
    int32_t rank_units;          /* capacity of the adapter arena, in rank units */
    int32_t rank_units_used;     /* units held by loaded adapters (rank rounded up to 8 each) */
    int32_t loaded;              /* number of loaded slots */
    int32_t device;              /* CUDA device the pool lives on */
    uint64_t arena_bytes;        /* device bytes of the adapter arena (Down and Up) */
    uint64_t table_bytes;        /* device bytes of the slot table and per-slot descriptors */
    uint64_t workspace_bytes;    /* device bytes of the per-forward workspace */
    int32_t ext_run_stride;      /* bf16 pools: arena stride (rank units) at which the loaded
                                    adapters' chunks most often lie in runs of 4 of one module;
                                    the decode projection loads such a run's Up tiles in one
                                    TMA box (0 = no run) */
    int32_t reserved;
} mlora_pool_info_t;

/* Text for a status code (static storage). */
const char* mlora_status_string(mlora_status s);

/* Detail of the most recent failure in the calling thread ("" if none). */
const char* mlora_last_error(void);

/*
 * Creates an adapter pool on the current CUDA device: the device-resident slot
 * pool that M031 §06 and the wiblog section on max_loras describe (slots fixed
 * up front), sized by a total rank budget instead of max_slots x max_rank so that
 * one high-rank adapter does not inflate every slot (wiblog failure mode
 * "max_lora_rank set too large").
 *
 *   max_slots   number of adapter slots (ids 0..max_slots-1), 0..4096; 0 makes a
 *               pool whose forward is the plain base projection
 *   rank_budget total rank resident at once; an adapter of rank r holds
 *               roundup(r, 8) units of it; rounded up to a multiple of 8
 *   max_rank    largest rank one adapter may have, 1..256
 *   din, dout   layer shape, >= 1; MLORA_BF16 needs din % 8 == 0
 *   dtype       element type of X, W, Y, Down and Up
 *   max_tokens  largest T a forward may pass, >= 1
 *   out         receives the pool handle (NULL on failure)
 *
 * All device memory the pool uses is allocated here (arena, slot table,
 * workspace); forward, merge, load and unload allocate nothing.
 * Errors: INVALID_ARG, UNSUPPORTED, OOM, CUDA.  Argument checks run before any
 * CUDA call.
 */
mlora_status mlora_pool_create(int max_slots, int rank_budget, int max_rank, int din, int dout,
                               mlora_dtype dtype, int max_tokens, mlora_pool_t* out);

/* Waits for the pool's outstanding work and frees all its device memory. NULL is a no-op. */
mlora_status mlora_pool_destroy(mlora_pool_t pool);

/*
 * Copies an adapter into a slot (M031 §06: weights must be in place before a
 * forward uses them; the slot is overwritten only after its last reader).
 *
 *   slot   0..max_slots-1; an adapter already in the slot is replaced
 *   down   Down [rank x din], row-major, pool dtype, host or device memory
 *   up     Up [dout x rank], row-major, pool dtype, host or device memory
 *   rank   1..max_rank
 *   scale  the adapter's scale (alpha / r in the airsota card's notation)
 *
 * Blocks the calling thread until the pool's last enqueued forward or merge has
 * finished, then copies, updates the device slot table and bumps the slot's
 * version; returns when the copy is complete.  If the rank budget has no room
 * left, live adapters are compacted first; OOM if it still does not fit.
 * Errors: INVALID_ARG, BAD_SLOT, RANK, OOM, CUDA.  On error the slot is unchanged.
 */
mlora_status mlora_load_adapter(mlora_pool_t pool, int slot, const void* down, const void* up,
                                int rank, float scale);

/* Empties a slot after its last reader (same waiting rule as load); bumps its version.
 * Errors: BAD_SLOT, NOT_LOADED, CUDA. */
mlora_status mlora_unload_adapter(mlora_pool_t pool, int slot);

/*
 * Loads one tenant's adapters of several modules of a fused projection into one slot
 * (airsota card "multi-LoRA serving vs merging", section 四 item ④: engines serve
 * adapters of mixed ranks and of different target modules).  The pool's W is the
 * modules' weights stacked by rows (e.g. q, k, v as one [3 x 4096] x 4096 qkv
 * projection); module m owns output rows [row_offset[m], row_offset[m] + rows[m]) and
 * has Down [rank[m] x din], Up [rows[m] x rank[m]] and scale[m], or rank[m] == 0 when
 * the tenant does not adapt it.  A forward then adds, to every row of this slot,
 * scale[m] Up[m] (Down[m] x) on module m's rows, for every adapted module, in the one
 * launch of the fused projection.  The slot holds one combined adapter whose rank
 * is the sum of the modules' ranks, each rounded up to 16 (at most max_rank);
 * module m's rank chunks only reach its own rows, and a projection tile skips the
 * chunks of modules whose rows it does not hold.  When the modules' scales differ,
 * each module's Up is scaled before it is stored (one rounding to the pool dtype).
 * Ownership and lifecycle as mlora_load_adapter.
 * Errors: INVALID_ARG (NULL arrays, a module outside [0, dout)), BAD_SLOT, RANK, OOM, CUDA.
 */
mlora_status mlora_load_adapter_modules(mlora_pool_t pool, int slot, int n_modules, const int* row_offset,
                                        const int* rows, const void* const* down, const void* const* up,
                                        const int* rank, const float* scale);

/* Version counter of a slot: 0 before the first load, +1 at every load and unload
 * (the immutable compute identity of M031 §07). Errors: BAD_SLOT, INVALID_ARG. */
mlora_status mlora_adapter_version(mlora_pool_t pool, int slot, uint64_t* version);

/*
 * Host (cold) tier of adapters (M031 §06: cold adapters on the host, hot ones on the
 * device, fetched for the batch that needs them; the weights must be in place before
 * the forward runs, and a slot is overwritten only after its last reader).
 *
 * mlora_host_adapter_add copies an adapter into pinned host memory owned by the
 * pool, under the caller's `id` (any int; an existing id is replaced once no
 * prefetch still copies out of it).  Down [rank x din], Up [dout x rank] as for
 * mlora_load_adapter, host or device memory, pool dtype; the caller may free them
 * when the call returns.  Errors: INVALID_ARG, RANK, OOM, CUDA.
 */
mlora_status mlora_host_adapter_add(mlora_pool_t pool, int id, const void* down, const void* up, int rank,
                                   float scale);
/* Frees the host-tier copy of `id` (waits for a prefetch still copying out of it).
 * Errors: INVALID_ARG, NOT_LOADED (no such id), CUDA. */
mlora_status mlora_host_adapter_remove(mlora_pool_t pool, int id);
/*
 * Loads host-tier adapter `id` into `slot` without waiting on the host.  On the
 * pool's copy stream, the weights go into free arena units at once (overlapping
 * forwards already enqueued); the slot and chunk tables change only once the
 * forwards enqueued so far have finished (a GPU-side wait on their last event); the
 * slot's previous adapter keeps its units until then.  `stream` is made to wait for
 * the update: forwards enqueued on it afterwards see the new adapter, forwards
 * enqueued before see the old one.  Forwards on other streams must be ordered after
 * `stream` by the caller.  The slot's version advances.  When only the slot's own
 * units or a compaction make room, or forwards of the pool were captured into a
 * graph, the call waits for the pool's readers on the host first.
 * Errors: INVALID_ARG, BAD_SLOT, NOT_LOADED (no such id), OOM (rank budget), CUDA.
 */
mlora_status mlora_prefetch(mlora_pool_t pool, int slot, int id, mlora_stream_t stream);

/*
 * The multi-LoRA forward (M031 §02): Y = X W^T for all T rows, plus
 * scale_a Up_a (Down_a x) on every row x whose adapter is a, in original row
 * order.  Segment build, shrink, base projection and expand all run in this
 * library's kernels on `stream`.
 *
 *   X            device [T x din], pool dtype
 *   W            device [dout x din], pool dtype
 *   row_adapter  device int32 [T]: slot id per row, -1 = no adapter; NULL = all -1
 *   T            0..max_tokens; T == 0 enqueues nothing and returns OK
 *   Y            device [T x dout], pool dtype, overwritten; must not overlap X or W
 *   stream       CUDA stream
 *
 * Rows naming an invalid or empty slot get no delta and set the status bit
 * reported by mlora_pool_status.  Errors: INVALID_ARG, CUDA.
 */
mlora_status mlora_forward(mlora_pool_t pool, const void* X, const void* W,
                           const int32_t* row_adapter, int T, void* Y, mlora_stream_t stream);

/*
 * Static merge of one adapter into a base weight, in place (M031 §04):
 *   W[o,i] <- W[o,i] + scale * sum_k Up[o,k] Down[k,i]      (fp32 sum, one rounding)
 * The merged weight is valid for rows of this adapter only.  Keep the original
 * W if the merge may need to be undone: it is not reversible exactly.
 *   W      device [dout x din], pool dtype
 *   slot   a loaded slot
 * Errors: INVALID_ARG, BAD_SLOT, NOT_LOADED, CUDA.
 */
mlora_status mlora_merge(mlora_pool_t pool, void* W, int slot, mlora_stream_t stream);

/*
 * Un-merge: subtracts the same update again, in place (airsota card "multi-LoRA
 * serving vs merging", section 四 item ③ -- a merge overwrites the base, so
 * switching back means re-subtracting the adapter's update or restoring a kept
 * original):
 *   W[o,i] <- W[o,i] - scale * sum_k Up[o,k] Down[k,i]      (fp32 sum, one rounding)
 * Applied to the output of mlora_merge with the same slot, it returns the original W
 * up to the two roundings: per element |W'' - W| <= u (|W'| + |W''|) with W' the
 * merged weight and u the unit roundoff of the pool dtype (2^-8 for bf16, 2^-24
 * for fp32), plus the fp32 error of the update sum.  Keep the original W when an
 * exact return is needed.  Arguments, ownership and errors as mlora_merge.
 */
mlora_status mlora_unmerge(mlora_pool_t pool, void* W, int slot, mlora_stream_t stream);

/*
 * Quantized base weight (M031 §05): int8 codes with one scale per output row,
 *   W[o,i] = Wq[o,i] * row_scale[o]          (symmetric; Wq device int8 [dout x din],
 *                                            row_scale device fp32 [dout])
 * The logical matrix is the restored W; a LoRA update is added to it, never to the
 * codes (that would mix two numeric spaces).
 *
 * mlora_dequantize: W = Wq * row_scale, rounded once to `dtype`, into the caller's
 *   buffer W [dout x din] (device).  Wq and W 16-byte aligned.  Errors: INVALID_ARG, CUDA.
 * mlora_forward_quantized: the dynamic LoRA branch over the restored base.  A bf16 pool
 *   with T <= 256 and din a multiple of 64 reads the codes in its projection kernel
 *   (each W tile restored in shared memory: the same values as mlora_dequantize, half
 *   the bytes of a bf16 W; W_scratch unused, may be NULL); otherwise it dequantizes into
 *   W_scratch (device [dout x din], pool dtype, caller-owned) and runs mlora_forward on
 *   it.  Arguments otherwise as mlora_forward.
 * mlora_merge_quantized: the merge on a quantized base, in place: restore each row,
 *   add scale * Up Down (fp32), then quantize the merged row again: new
 *   row_scale[o] = max_i |w[o,i]| / 127 (fp32; 0 for an all-zero row), codes
 *   rint(w / row_scale[o]) (to nearest, ties to even) clamped to [-127, 127].  The
 *   re-quantization adds at most half a step (row_scale[o] / 2) per element on top
 *   of the merged float weight.  Wq 16-byte aligned.  A bf16 pool with din a
 *   multiple of 16 runs it on the tensor cores in three launches (the merged rows'
 *   max, their codes, their scales; the fp32 sum over the rank may then round
 *   differently from a sequential one, which moves a code by one only at a tie);
 *   otherwise one CUDA-core launch holds each merged row in shared memory.
 *   Errors: INVALID_ARG (also, on the CUDA-core path, din too large for a row in
 *   shared memory, about 51 000), BAD_SLOT, NOT_LOADED, CUDA.
 */
mlora_status mlora_dequantize(const void* Wq, const float* row_scale, int dout, int din, mlora_dtype dtype, void* W,
                              mlora_stream_t stream);
mlora_status mlora_forward_quantized(mlora_pool_t pool, const void* X, const void* Wq, const float* row_scale,
                                     void* W_scratch, const int32_t* row_adapter, int T, void* Y,
                                     mlora_stream_t stream);
mlora_status mlora_merge_quantized(mlora_pool_t pool, void* Wq, float* row_scale, int slot, mlora_stream_t stream);

/*
 * NF4 base weight (M031 §05: the logical matrix is W restored by scale and codebook;
 * the page names the NF4 codebook): 4-bit codes with an fp32 absmax per output row and
 * block of 64 input columns and a 16-entry codebook,
 *   W[o,i] = codebook[code[o,i]] * absmax[i / 64][o]
 *   codes    device uint8 [dout x din/2]: column 2m of a row in the low nibble of byte
 *            m, column 2m+1 in the high nibble; 16-byte aligned
 *   absmax   device fp32 [din/64][dout] (block-major: one block's rows adjacent)
 *   codebook HOST fp32 [16], copied at the call (e.g. the NormalFloat values)
 * din must be a multiple of 64.
 *
 * mlora_dequantize_nf4: W = codebook[code] * absmax, rounded once to `dtype`, into the
 *   caller's W [dout x din] (device, 16-byte aligned).  Errors: INVALID_ARG, CUDA.
 * mlora_forward_nf4: the dynamic LoRA branch over the restored base.  A bf16 pool with
 *   T <= 256, dout a multiple of 4 and absmax 16-byte aligned reads the codes (and the
 *   block scales) in its projection kernel (each W tile restored in shared memory, the
 *   same values as mlora_dequantize_nf4; W_scratch unused, may be NULL);
 *   otherwise W_scratch (device [dout x din], pool dtype) receives the restored W and
 *   mlora_forward runs on it.  Arguments otherwise as mlora_forward.
 * mlora_merge_nf4: the merge on an NF4 base, in place: per row and block, restore
 *   (fp32 codebook value * absmax), add scale * sum_k Up[o,k] Down[k,i] (fp32), take the
 *   block's new absmax = max |w|, and give each w / absmax (fp32) the code of the
 *   nearest codebook value (the lower code on a tie).  The codebook must be ascending
 *   and hold 0 (an all-zero block keeps absmax 0).  Errors: INVALID_ARG, BAD_SLOT,
 *   NOT_LOADED, CUDA.
 */
mlora_status mlora_dequantize_nf4(const void* codes, const float* absmax, const float* codebook, int dout, int din,
                                  mlora_dtype dtype, void* W, mlora_stream_t stream);
mlora_status mlora_forward_nf4(mlora_pool_t pool, const void* X, const void* codes, const float* absmax,
                               const float* codebook, void* W_scratch, const int32_t* row_adapter, int T, void* Y,
                               mlora_stream_t stream);
mlora_status mlora_merge_nf4(mlora_pool_t pool, void* codes, float* absmax, const float* codebook, int slot,
                             mlora_stream_t stream);

/*
 * Synchronizes `stream`, then reads and clears the pool's device status word.
 * Returns MLORA_OK, MLORA_ERR_DEVICE_ROW (a forward since the last call saw a row
 * naming an invalid or empty slot), MLORA_ERR_DEVICE_TIMEOUT (a pipeline wait in a
 * kernel gave up after its bounded limit; that call's output is not valid) or
 * MLORA_ERR_CUDA (the stream reported an error).
 */
mlora_status mlora_pool_status(mlora_pool_t pool, mlora_stream_t stream);

/* Fills `info` with the pool's configuration and memory split. Errors: INVALID_ARG. */
mlora_status mlora_pool_info(mlora_pool_t pool, mlora_pool_info_t* info);

/*
 * Runs only the segment builder of mlora_forward (M031 §03: rows grouped by
 * adapter, original order kept inside a group, groups in ascending slot id) and
 * copies its result to the caller's device buffers:
 *   perm     device int32 [T]: original row indices in segment order; entries past
 *            the number of rows with a valid adapter are set to -1
 *   offsets  device int32 [max_slots + 1]: offsets[s]..offsets[s+1] is slot s's range
 * Errors: INVALID_ARG, CUDA.
 */
mlora_status mlora_debug_segments(mlora_pool_t pool, const int32_t* row_adapter, int T,
                                  int32_t* perm, int32_t* offsets, mlora_stream_t stream);

/*
 * Reads back the segments (M031 §03: rows grouped by adapter, original order kept
 * inside a group, groups in ascending slot id) that the most recent mlora_forward
 * of this pool built with its row map -- on the bf16 path, the builder that runs
 * inside the shrink kernel; otherwise the standalone segment kernel -- into the
 * caller's device buffers, on `stream` (order it after that forward):
 *   T        the rows of that forward (INVALID_ARG if it had another T, if no forward
 *            with a row map ran since the pool was made, or if mlora_debug_segments
 *            ran after it)
 *   perm     device int32 [T], layout as in mlora_debug_segments
 *   offsets  device int32 [max_slots + 1]
 * Errors: INVALID_ARG, CUDA.
 */
mlora_status mlora_debug_last_segments(mlora_pool_t pool, int T, int32_t* perm, int32_t* offsets,
                                       mlora_stream_t stream);

/*
 * Profiling records of the tensor-core kernels' thread blocks, for measuring kernel
 * durations inside a timed run (no work is skipped or changed; each block adds one
 * atomic add and one 32-byte store as it ends).  With cap > 0, every CTA of the
 * shrink and projection kernels launched by later forwards of this pool (captured
 * forwards included: the buffer is baked into the launch) appends one record to
 * `records`, a caller-owned device buffer of 8-byte words, 8-byte aligned, of
 * 4 + 4 cap words:
 *   records[0]            number of records appended so far (the caller zeroes it)
 *   records[4+4i .. 7+4i] record i: start and end of the block in the device's
 *                         %globaltimer nanoseconds, the kernel kind (0 shrink,
 *                         1 decode projection, 2 prefill projection) and the block's
 *                         linear index
 * Records past `cap` are counted but not stored.  cap == 0 turns recording off.
 * Errors: INVALID_ARG.
 */
mlora_status mlora_profile_stamps(mlora_pool_t pool, void* records, int cap);

/*
 * Base projection Y = X W^T for a decode-sized batch that allocates nothing.
 * The pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory when they need the projection -- plugins whose host
 * runtime owns the device-memory budget and forbids allocations after start-up,
 * and latency-critical loops that cannot take the device-wide synchronisation an
 * allocation may cause.  Such callers cannot create a pool, whose workspace comes
 * from cudaMalloc.
 *
 *   X   device [T x din] bf16, W device [dout x din] bf16, Y device [T x dout] bf16,
 *       all 16-byte aligned, owned by the caller; Y is overwritten
 *   T   0..256 (T == 0 enqueues nothing); din a positive multiple of 8;
 *       dout 1..262144
 *
 * It runs the split-K tensor-core projection of mlora_forward (no adapters) on
 * `stream`, with that kernel's scratch (fp32 partial tiles, arrival counters and
 * a status word) in one fixed device array of about 8 MiB that every GPU loading
 * this library holds until the process exits; larger shapes are rejected with
 * MLORA_ERR_UNSUPPORTED, never served from anywhere else.  No cudaMalloc, cudaFree
 * or allocating library routine is called.  The first call on a device looks up
 * the array's device address and raises the kernel's shared-memory cap (host
 * calls that run once per device).  All calls share the one array
 * (it keeps what the last call left; the counters are cleared on every call), so
 * calls whose work overlaps on the GPU -- on different streams, or from several
 * host threads -- race and must be ordered by the caller.  A pipeline wait of
 * the kernel that gives up after its bounded limit leaves that call's Y invalid
 * and sets a bit in the array's status word, which stays set until
 * mlora_project_noalloc_status reads it.
 * Errors: INVALID_ARG (NULL or misaligned pointer), UNSUPPORTED, CUDA.
 */
mlora_status mlora_project_noalloc(const void* X, const void* W, int T, int din, int dout, void* Y,
                                   mlora_stream_t stream);

/*
 * Status of the allocation-free calls made on the current device since the last
 * read: synchronizes `stream`, then reads and clears the status word of the fixed
 * scratch array (no allocation).  Returns MLORA_OK, MLORA_ERR_DEVICE_TIMEOUT (a
 * pipeline wait in one of those calls gave up after its bounded limit; that call's
 * Y is not valid) or MLORA_ERR_CUDA.  Like the calls it reports on, its first use
 * on a device looks up the array's address.
 */
mlora_status mlora_project_noalloc_status(mlora_stream_t stream);

/*
 * Test hook for the status above: enqueues on `stream` one kernel whose single
 * pipeline wait has nothing to wait for and gives up after `cycles` SM clock
 * cycles (1 .. 2^31), with the same bounded wait the projection kernels use, so
 * that mlora_project_noalloc_status then reports MLORA_ERR_DEVICE_TIMEOUT.
 * Nothing faults or hangs.  Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
mlora_status mlora_debug_noalloc_expire_wait(long long cycles, mlora_stream_t stream);

/*
 * Host-only view of the arena allocator the pool uses (no CUDA calls), for tests
 * of the placement logic.  An arena has `units` rank units; an allocation of
 * `n` units is placed first-fit at a multiple of 8.  mlora_arena_compact slides
 * every live block toward offset 0, keeping their order, and reports the moves.
 */
typedef struct mlora_arena* mlora_arena_t;
mlora_arena_t mlora_arena_new(int units);
void mlora_arena_delete(mlora_arena_t arena);
/* Returns the unit offset of the new block of `id`, or -1 if no hole fits. */
int mlora_arena_alloc(mlora_arena_t arena, int id, int n);
/* Frees the block of `id`; returns 0, or -1 if `id` holds no block. */
int mlora_arena_free(mlora_arena_t arena, int id);
/* Gives the block of `from` to `to` in place (the pool quarantines an evicted
 * adapter's block this way until its last reader has finished); returns 0, or -1
 * if `from` holds no block or `to` already holds one. */
int mlora_arena_rename(mlora_arena_t arena, int from, int to);
/* Compacts; writes up to `cap` moves as (id, old_offset, new_offset) triples; returns the count. */
int mlora_arena_compact(mlora_arena_t arena, int32_t* moves, int cap);
/* Units in use and largest free hole. */
int mlora_arena_used(mlora_arena_t arena);
int mlora_arena_largest_hole(mlora_arena_t arena);

#ifdef __cplusplus
}
#endif

#endif /* MLORA_H */
