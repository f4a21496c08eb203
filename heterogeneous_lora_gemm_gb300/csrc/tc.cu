// Tensor-core path of the bf16 forward: tcgen05 MMA with TMEM accumulators, TMA
// loads into swizzled shared memory, warp-specialised pipeline.
//
// "swap-AB" GEMM kernel, in two modes.  The weight-like operand is the MMA's M
// side (128 rows per tile) and the tokens are the N side (N = up to 256 tokens,
// a multiple of 16), so the weight streams through the tensor cores once however
// few rows the batch has.
//
// Shrink (any T; token tiles of 256 along grid z): rows = 8 chunks of 16 rank rows
// of the loaded adapters' Down (the pool's chunk table), K = din, giving
// Down_c X^T for every token of the tile.  A CTA loads only the chunks whose slot
// some token of its token tile uses, and marks them in tmask; Vt entries of the
// other (chunk, token tile) pairs are never read.  The epilogue keeps the entry
// of a token only if the token belongs to the chunk's adapter, scales it, rounds
// it to bf16 and writes Vt[c][t][:], zero for every other token.  CTA (0,0,0)
// also runs the segment builder (seg.cuh), in its epilogue warps while its MMAs
// run, and publishes the segments.
//
// Projection (T <= 256): rows = output features.  The K loop of a tile is the din
// columns of W followed by a K-extension over the loaded adapters' chunks
// (ai-infra-kb "M031" §02: each row adds scale_a Up_a (Down_a x)):
//
//     Y^T[o, t] = sum_i W[o, i] X[t, i]  +  sum_c Up_{a(c)}[o, col(c) + j] Vt[c][t][j]
//
// over the chunks c whose slot some row of the batch uses.  The delta lands in
// the same fp32 accumulator as the base product, on the row's own column, and the
// output is rounded once.  The projection is launched while the shrink still runs
// (programmatic dependent launch): it streams W and the Up tiles of its chunks
// before it waits for Vt.
//
// Work split: a grid of (row tile, K split, token tile).  Split s takes a
// contiguous share of the K steps and holds an fp32 partial tile in TMEM.  The
// splits of a tile form a thread-block cluster: each stages its partial tile in
// its own shared memory and, after a cluster barrier, sums one slice of tokens
// over the shared memory of all splits, in split order (so the result does not
// depend on timing), in as many passes as the staging space needs.  A caller
// without clusters (the allocation-free entry point) meets through global memory
// instead: the last split to arrive sums the partials in split order.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>

#include "seg.cuh"
#include "tc.h"
#include "tc_ptx.cuh"

namespace mlora {

using namespace ptx;

namespace {

// ---------------------------------------------------------------- host helpers
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

bool tc_encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
               const cuuint32_t* box, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    }
    return n;
}

// ---------------------------------------------------------------- constants
constexpr int BM = 128;            // rows per tile (MMA M)
constexpr int BK = 64;             // K per pipeline step (128 bytes of bf16)
constexpr int EXT_SUB = 4;         // K-extension chunks per pipeline step
constexpr int A_BYTES = BM * BK * 2;            // 16 KiB: W tile, 4 Up chunk tiles or 8 Down chunk tiles
constexpr int NUM_THREADS = 192;   // warp 0 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr int MAX_N = 256;
constexpr int CHUNKS_PER_TILE = BM / CHUNK;     // shrink: 8 chunks of 16 rank rows
constexpr int CHUNK_BYTES = CHUNK * BK * 2;     // 2 KiB: 16 rank rows x 64 din columns of Down
constexpr int MAX_SPLITS = 16;     // K splits per tile at most
constexpr int MAX_CLUSTER = 8;     // K splits of a tile reduced inside one (portable) cluster
constexpr int MAX_STAGES = 8;
constexpr int EXT_CAP = 256;       // projection: K-extension chunks of a CTA kept in shared memory
constexpr int MAX_SLOT_WORDS = 4096 / 32;

// where the publishing shrink CTA builds the segments
enum { SEG_NONE = 0, SEG_BEFORE = 1, SEG_BESIDE = 2 };

__host__ __device__ constexpr int b_bytes(int n) { return n * BK * 2; }
__host__ __device__ constexpr int stage_bytes(int n) { return A_BYTES + b_bytes(n); }

// Shared-memory tail after the stage ring and the segment scratch.
struct Tail {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t acc_full;
    int stage_kind[MAX_STAGES];       // -1 = din step, else bit mask of the K-extension chunks loaded
    uint32_t tmem_slot;
    int abort_flag;
    int flags[2];                     // [0] an MMA was issued, [1] last arrival (global reduction)
    int tile_chunks;                  // shrink: chunks of this row tile some token uses
    int my_c[CHUNKS_PER_TILE];        // shrink, per compacted chunk: index in the chunk table,
    int my_slot[CHUNKS_PER_TILE];     //   slot, arena unit, valid rank columns, scale
    int my_unit[CHUNKS_PER_TILE];
    int my_kval[CHUNKS_PER_TILE];
    float my_scale[CHUNKS_PER_TILE];
    int tile_ra[MAX_N];               // shrink: slot id of each token of the token tile
    uint32_t slot_bits[MAX_SLOT_WORDS];   // projection: slots some row of the batch uses
    int ext_unit[EXT_CAP];            // projection: arena unit of each K-extension chunk, -1 = skip
    int ext_slot[EXT_CAP];
};

struct GemmParams {
    const ChunkRec* chunks;         // chunk table of the loaded slots
    const int32_t* row_adapter;     // slot id per token
    const SlotRec* slots;           // shrink: slot table (segment builder)
    __nv_bfloat16* Y;               // projection output [T x dout]
    __nv_bfloat16* vt;              // shrink output [max_chunks][tcap][16]
    uint8_t* tmask;                 // shrink output [token tile][max_chunks]
    float* partials;                // global reduction: [tile][split][N][BM]
    int32_t* tile_ctr;              // global reduction: [tile] arrival counters
    uint32_t* status;
    int T, dout, N, kb_total, splits, stages, tcap;
    int n_chunks;                   // chunks in the table
    int ext_units;                  // projection: K-extension steps (EXT_SUB chunks each)
    int a_bytes;                    // bytes of the A operand in a stage
    int ring_bytes;                 // the stage ring; also the cluster reduction's staging space
    int tail_off;                   // offset of the Tail
    int pdl;                        // launched while the shrink may still run: wait before reading Vt
    int cluster;                    // the K splits of a tile form a cluster (else: global reduction)
    int S, max_chunks;
    int seg_mode, seg_P, seg_stage_rows, scratch_off;   // shrink: segment builder of CTA (0,0,0)
    Workspace ws;
};

// ---------------------------------------------------------------- the GEMM kernel
template <bool SHRINK>
__global__ void __launch_bounds__(NUM_THREADS, 1)
swapab_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmArena,
                   GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Tail& tl = *reinterpret_cast<Tail*>(smem + p.tail_off);
    volatile int* abort_flag = &tl.abort_flag;
    const int NS = p.stages;
    const int SB = p.a_bytes + b_bytes(p.N);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, split = blockIdx.y, ztile = blockIdx.z;
    const int tok0 = ztile * MAX_N;                  // first token of this token tile
    const int T = min(p.T - tok0, p.N);              // tokens in this tile
    const bool publisher = SHRINK && (blockIdx.x | blockIdx.y | blockIdx.z) == 0;

    if (SHRINK) {
        pdl_trigger();   // the projection may launch and stream W meanwhile
        if (publisher && p.seg_mode == SEG_BEFORE) {
            // too many slots or rows for scratch beside the ring: the whole CTA builds
            // the segments in the ring memory before any load
            const seg::Scratch sc = seg::carve(reinterpret_cast<int*>(smem), p.S, p.seg_P, p.seg_stage_rows != 0);
            seg::build<seg::GROUP_BLOCK>(p.row_adapter, p.T, p.slots, p.S, p.seg_P, p.max_chunks, sc, p.ws);
        }
    }

    const int kb0 = (int)((long long)split * p.kb_total / p.splits);
    const int kb1 = (int)((long long)(split + 1) * p.kb_total / p.splits);
    const int eu0 = SHRINK ? 0 : (int)((long long)split * p.ext_units / p.splits);
    const int eu1 = SHRINK ? 0 : (int)((long long)(split + 1) * p.ext_units / p.splits);
    const int n_steps = (kb1 - kb0) + (eu1 - eu0);
    const uint32_t ncols = p.N <= 32 ? 32 : (p.N <= 64 ? 64 : (p.N <= 128 ? 128 : 256));

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&tl.full[s], 1);
            mbar_init(&tl.empty[s], 1);
        }
        mbar_init(&tl.acc_full, 1);
        tl.abort_flag = 0;
        tl.flags[0] = 0;
        tl.flags[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!SHRINK) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
        if (SHRINK || p.ext_units > 0) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmArena) : "memory");
    }
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tl.tmem_slot)),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 2 && SHRINK) {
        // Which of this row tile's chunks does some token of the token tile use?  The
        // row ids and the chunk entries are read together; a chunk is needed if a
        // token names its slot (ids of empty or invalid slots match no chunk).
        const int cb = tile * CHUNKS_PER_TILE;
        int av[MAX_N / 32];
#pragma unroll
        for (int i = 0; i < MAX_N / 32; ++i) {
            const int t = lane + 32 * i;
            av[i] = t < T ? p.row_adapter[tok0 + t] : -1;
        }
        ChunkRec cr{-2, 0, 0, 0.f};
        if (lane < CHUNKS_PER_TILE && cb + lane < p.n_chunks) cr = p.chunks[cb + lane];
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < CHUNKS_PER_TILE; ++j) {
            const int sl = __shfl_sync(0xffffffffu, cr.slot, j);
            bool hit = false;
#pragma unroll
            for (int i = 0; i < MAX_N / 32; ++i) hit |= av[i] == sl;
            if (__any_sync(0xffffffffu, hit)) m |= 1u << j;
        }
#pragma unroll
        for (int i = 0; i < MAX_N / 32; ++i) {
            const int t = lane + 32 * i;
            if (t < T) tl.tile_ra[t] = av[i];
        }
        if (lane < CHUNKS_PER_TILE && ((m >> lane) & 1u)) {
            const int k = __popc(m & ((1u << lane) - 1u));   // compacted position
            tl.my_c[k] = cb + lane;
            tl.my_slot[k] = cr.slot;
            tl.my_unit[k] = cr.unit;
            tl.my_kval[k] = cr.kval;
            tl.my_scale[k] = cr.scale;
        }
        if (lane == 0) tl.tile_chunks = __popc(m);
        if (split == 0 && lane < CHUNKS_PER_TILE && cb + lane < p.n_chunks)
            p.tmask[(size_t)ztile * p.max_chunks + cb + lane] = (uint8_t)((m >> lane) & 1u);
    }
    if (warp == 2 && !SHRINK && eu1 > eu0) {
        // The slots the batch uses, then this CTA's K-extension chunks: the arena unit
        // of each chunk whose slot is used, -1 for the others (never loaded).
        int av[MAX_N / 32];
#pragma unroll
        for (int i = 0; i < MAX_N / 32; ++i) {
            const int t = lane + 32 * i;
            av[i] = t < T ? p.row_adapter[t] : -1;
        }
        const int c0 = eu0 * EXT_SUB;
        const int nx = min((eu1 - eu0) * EXT_SUB, EXT_CAP);
        for (int k = lane; k < nx; k += 32) {
            const int c = c0 + k;
            int sl = -1, un = -1;
            if (c < p.n_chunks) {
                const ChunkRec cr = p.chunks[c];
                sl = cr.slot;
                un = cr.unit;
            }
            tl.ext_slot[k] = sl;
            tl.ext_unit[k] = un;
        }
        for (int w = lane; w < (p.S + 31) / 32; w += 32) tl.slot_bits[w] = 0;
        __syncwarp();
#pragma unroll
        for (int i = 0; i < MAX_N / 32; ++i)
            if (av[i] >= 0 && av[i] < p.S) atomicOr(&tl.slot_bits[av[i] >> 5], 1u << (av[i] & 31));
        __syncwarp();
        for (int k = lane; k < nx; k += 32) {
            const int sl = tl.ext_slot[k];
            if (sl < 0 || !((tl.slot_bits[sl >> 5] >> (sl & 31)) & 1u)) tl.ext_unit[k] = -1;
        }
    }
    // A block barrier needs converged warps: lanes that skipped a one-thread branch
    // above (barrier set-up, the TMA and MMA roles) wait here for it first.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tl.tmem_slot;
    const int tile_chunks = SHRINK ? tl.tile_chunks : 0;
    const bool seg_here = publisher && p.seg_mode == SEG_BESIDE;
    auto run_seg = [&]() {   // warps 2..5 of the publishing CTA, beside the TMA and MMA warps
        const seg::Scratch sc =
            seg::carve(reinterpret_cast<int*>(smem + p.scratch_off), p.S, p.seg_P, p.seg_stage_rows != 0);
        seg::build<seg::GROUP_EPI>(p.row_adapter, p.T, p.slots, p.S, p.seg_P, p.max_chunks, sc, p.ws);
    };
    if (SHRINK && tile_chunks <= 0) {   // no token of the token tile uses a chunk of this row tile
        if (seg_here && warp >= 2) run_seg();
        if (warp == 1) {
            __syncwarp();
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
        }
        return;
    }

    if (warp == 0 && lane == 0) {
        // ---------------- producer: TMA loads into the stage ring
        int s = 0;
        uint32_t ph = 0;
        bool waited = false;
        int armed[MAX_STAGES] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int i = 0; i < n_steps; ++i) {
            if (!mbar_wait(&tl.empty[s], ph ^ 1, abort_flag, p.status)) break;
            ++armed[s];
            uint8_t* a = smem + (size_t)s * SB;
            uint8_t* b = a + p.a_bytes;
            const int kb = kb0 + i;
            if (SHRINK) {
                tl.stage_kind[s] = -1;
                mbar_expect_tx(&tl.full[s], (uint32_t)(tile_chunks * CHUNK_BYTES + b_bytes(p.N)));
                for (int j = 0; j < tile_chunks; ++j)
                    tma_2d(a + j * CHUNK_BYTES, &tmArena, &tl.full[s], kb * BK, tl.my_unit[j]);
                tma_2d(b, &tmX, &tl.full[s], kb * BK, tok0);
            } else if (kb < kb1) {
                tl.stage_kind[s] = -1;
                mbar_expect_tx(&tl.full[s], (uint32_t)SB);
                tma_2d(a, &tmW, &tl.full[s], kb * BK, tile * BM);
                tma_2d(b, &tmX, &tl.full[s], kb * BK, 0);
            } else {
                const int u = eu0 + (kb - kb1);
                const int kx = (u - eu0) * EXT_SUB;
                int un[EXT_SUB];
                uint32_t mask = 0;
#pragma unroll
                for (int j = 0; j < EXT_SUB; ++j) {
                    const int c = u * EXT_SUB + j;
                    int v = -1;
                    if (c < p.n_chunks) {
                        if (kx + j < EXT_CAP) {
                            v = tl.ext_unit[kx + j];
                        } else {
                            const ChunkRec cr = p.chunks[c];
                            if ((tl.slot_bits[cr.slot >> 5] >> (cr.slot & 31)) & 1u) v = cr.unit;
                        }
                    }
                    un[j] = v;
                    if (v >= 0) mask |= 1u << j;
                }
                tl.stage_kind[s] = (int)mask;
                if (mask == 0) {
                    mbar_expect_tx(&tl.full[s], 0);
                } else {
                    // Up tiles (two blocks of 8 rank columns x 128 rows) are the pool's own
                    // data: issue them before waiting for the shrink, then its Vt
                    mbar_expect_tx_only(&tl.full[s], (uint32_t)(__popc(mask) * (BM * 32)));
#pragma unroll
                    for (int j = 0; j < EXT_SUB; ++j)
                        if ((mask >> j) & 1u)
                            tma_3d(a + j * (BM * 32), &tmArena, &tl.full[s], 0, tile * BM, un[j] >> 3);
                    if (!waited) {
                        if (p.pdl) pdl_wait();
                        waited = true;
                    }
                    mbar_expect_tx(&tl.full[s], (uint32_t)b_bytes(p.N));
                    tma_3d(b, &tmV, &tl.full[s], 0, 0, u * EXT_SUB);
                }
            }
            if (++s == NS) {
                s = 0;
                ph ^= 1;
            }
        }
        if (*abort_flag) {
            // let loads already issued land before the CTA's shared memory goes away
            for (int j = 0; j < NS; ++j) {
                if (armed[j] == 0) continue;
                const long long t0 = clock64();
                while (!mbar_try_wait(&tl.full[j], (uint32_t)((armed[j] - 1) & 1)) && clock64() - t0 < 200000000ll) {
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        const uint32_t idesc = idesc_bf16(BM, p.N);
        int s = 0;
        uint32_t ph = 0;
        uint32_t acc = 0;
        for (int i = 0; i < n_steps; ++i) {
            if (!mbar_wait(&tl.full[s], ph, abort_flag, p.status)) break;
            tc_fence_after();
            const uint32_t a = smem_u32(smem + (size_t)s * SB);
            const uint32_t b = a + p.a_bytes;
            const int kind = tl.stage_kind[s];
            if (kind < 0) {
                // A spans 128 rows (16 KiB) from a; in the shrink, rows past the loaded
                // chunks hold whatever lies there and give accumulator rows nobody reads
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    mma_bf16(tmem, sdesc(a + k * 32, 1024, SW128), sdesc(b + k * 32, 1024, SW128), idesc, acc);
                    acc = 1;
                }
            } else {
                // Up chunk: [2 blocks of 8 columns][128 rows][16 B], no swizzle (K-direction core
                // matrices BM*16 bytes apart, M-direction 128 bytes); Vt chunk: 32-byte swizzle
#pragma unroll
                for (int j = 0; j < EXT_SUB; ++j)
                    if ((kind >> j) & 1) {
                        mma_bf16(tmem, sdesc_lbo(a + j * (BM * 32), BM * 16, 128, SW_NONE),
                                 sdesc(b + j * (p.N * 32), 256, SW32), idesc, acc);
                        acc = 1;
                    }
            }
            mma_commit(&tl.empty[s]);
            if (++s == NS) {
                s = 0;
                ph ^= 1;
            }
        }
        tl.flags[0] = (int)acc;
        mma_commit(&tl.acc_full);
        if (*abort_flag) {   // MMAs already issued must finish before TMEM is released
            const long long t0 = clock64();
            while (!mbar_try_wait(&tl.acc_full, 0) && clock64() - t0 < 200000000ll) {
            }
        }
    } else if (warp >= 2) {
        if (seg_here) run_seg();   // the segment build overlaps this CTA's loads and MMAs
        // ---------------- epilogue: TMEM -> partial tile, or the final values
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;          // row of the tile
        const bool ok = mbar_wait(&tl.acc_full, 0, abort_flag, p.status);
        __syncwarp();   // reconverge: lanes may leave the wait loop apart; tcgen05.ld is warp-collective
        tc_fence_after();
        const bool have = __all_sync(0xffffffffu, ok) && tl.flags[0] != 0;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);

        // final write of 16 consecutive tokens t0..t0+15 of this row
        int c_slot = -1, c_idx = 0;
        float c_scale = 0.f;
        if (SHRINK && (row / CHUNK) < tile_chunks) {
            const int k = row / CHUNK;
            c_idx = tl.my_c[k];
            c_slot = tl.my_slot[k];
            // rank columns past the adapter's rank belong to the next adapter in the arena
            c_scale = (row % CHUNK) < tl.my_kval[k] ? tl.my_scale[k] : 0.f;
        }
        const int o = tile * BM + row;
        auto emit = [&](int t0, const float* v) {
            if (SHRINK) {
                if (c_slot < 0) return;
                __nv_bfloat16* dst = p.vt + ((size_t)c_idx * p.tcap + tok0) * CHUNK + (row % CHUNK);
                for (int j = 0; j < 16 && t0 + j < T; ++j) {
                    const bool mine = tl.tile_ra[t0 + j] == c_slot;
                    dst[(size_t)(t0 + j) * CHUNK] = __float2bfloat16_rn(mine ? c_scale * v[j] : 0.f);
                }
            } else if (o < p.dout) {
                for (int j = 0; j < 16 && t0 + j < T; ++j)
                    p.Y[(size_t)(t0 + j) * p.dout + o] = __float2bfloat16_rn(v[j]);
            }
        };

        // final write of rows r0..r0+3 (a multiple of 4) of token t
        auto emit4 = [&](int t, int r0, const float4& v) {
            if (SHRINK) {
                const int k = r0 / CHUNK;
                if (k >= tile_chunks) return;
                const int kval = tl.my_kval[k];
                const int k0 = r0 % CHUNK;
                const float sc = tl.tile_ra[t] == tl.my_slot[k] ? tl.my_scale[k] : 0.f;
                __nv_bfloat162 lo = __floats2bfloat162_rn(k0 < kval ? sc * v.x : 0.f, k0 + 1 < kval ? sc * v.y : 0.f);
                __nv_bfloat162 hi = __floats2bfloat162_rn(k0 + 2 < kval ? sc * v.z : 0.f, k0 + 3 < kval ? sc * v.w : 0.f);
                uint2 w;
                w.x = *reinterpret_cast<uint32_t*>(&lo);
                w.y = *reinterpret_cast<uint32_t*>(&hi);
                *reinterpret_cast<uint2*>(p.vt + ((size_t)tl.my_c[k] * p.tcap + tok0 + t) * CHUNK + k0) = w;
            } else {
                const int o0 = tile * BM + r0;
                __nv_bfloat16* y = p.Y + (size_t)t * p.dout + o0;
                if (p.dout % 4 == 0 && o0 + 4 <= p.dout) {
                    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
                    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
                    uint2 w;
                    w.x = *reinterpret_cast<uint32_t*>(&lo);
                    w.y = *reinterpret_cast<uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(y) = w;
                } else {
                    const float vv[4] = {v.x, v.y, v.z, v.w};
                    for (int j = 0; j < 4; ++j)
                        if (o0 + j < p.dout) y[j] = __float2bfloat16_rn(vv[j]);
                }
            }
        };

        if (p.splits == 1) {
            for (int t0 = 0; t0 < T; t0 += 16) {
                float v[16];
                if (have) tmem_ld16(tbase + t0, v);
                else
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                emit(t0, v);
            }
        } else if (p.cluster) {
            // Stage this split's partial tile [token][row] in its own shared memory (the
            // ring is idle: every load has been consumed by the finished MMAs), then,
            // after a cluster barrier, reduce one slice of tokens over the shared
            // memory of all splits, summed in split order, and write it.  Passes of
            // tp tokens when the whole tile does not fit the ring.
            float* part_s = reinterpret_cast<float*>(smem);
            const uint32_t part_a = smem_u32(part_s);
            const int tp = min(p.N, (p.ring_bytes / (BM * 4)) & ~15);
            for (int p0 = 0; p0 < T; p0 += tp) {
                const int pt = min(tp, T - p0);
                for (int t0 = 0; t0 < pt; t0 += 16) {
                    float v[16];
                    if (have) tmem_ld16(tbase + p0 + t0, v);
                    else
                        for (int j = 0; j < 16; ++j) v[j] = 0.f;
#pragma unroll
                    for (int j = 0; j < 16; ++j) part_s[(t0 + j) * BM + row] = v[j];
                }
                __syncwarp();
                cluster_sync();
                const int ts = (pt + p.splits - 1) / p.splits;
                const int t_lo = (int)cluster_rank() * ts;
                const int t_hi = min(pt, t_lo + ts);
                for (int g = threadIdx.x - 64; g < (t_hi - t_lo) * (BM / 4); g += 128) {
                    const int t = t_lo + g / (BM / 4), r0 = (g % (BM / 4)) * 4;
                    const uint32_t off = part_a + (uint32_t)((t * BM + r0) * 4);
                    float4 q4[MAX_CLUSTER];
#pragma unroll
                    for (int sp = 0; sp < MAX_CLUSTER; ++sp)
                        if (sp < p.splits) q4[sp] = ld_cluster_f4(map_cluster(off, (uint32_t)sp));
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int sp = 0; sp < MAX_CLUSTER; ++sp)
                        if (sp < p.splits) {
                            acc.x += q4[sp].x;
                            acc.y += q4[sp].y;
                            acc.z += q4[sp].z;
                            acc.w += q4[sp].w;
                        }
                    emit4(p0 + t, r0, acc);
                }
                __syncwarp();
                cluster_sync();   // no CTA refills or leaves while the others still read its shared memory
            }
        } else {
            // partial tile layout [split][token][row] fp32: for a fixed token the 128 rows
            // of a tile are contiguous, so both the stores below and the reduction's
            // loads are coalesced
            const int ctr = tile * gridDim.z + ztile;
            const size_t tile_base = (size_t)ctr * p.splits * p.N * BM;
            float* mine = p.partials + tile_base + (size_t)split * p.N * BM + row;
            for (int t0 = 0; t0 < T; t0 += 16) {
                float v[16];
                if (have) tmem_ld16(tbase + t0, v);
                else
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) mine[(size_t)(t0 + j) * BM] = v[j];
            }
            __threadfence();
            epi_bar();
            if (threadIdx.x == 64) {
                const int prev = atomicAdd(&p.tile_ctr[ctr], 1);
                const int last = prev == p.splits - 1;
                if (last) {
                    p.tile_ctr[ctr] = 0;
                    __threadfence();
                }
                tl.flags[1] = last;
            }
            epi_bar();
            if (tl.flags[1]) {
                // last split of the tile: sum the partials in split order (independent of
                // arrival order).  The 128 epilogue threads sweep the tile as float4
                // groups of 4 rows of one token; the loads of all splits are independent.
                const float4* base = reinterpret_cast<const float4*>(p.partials + tile_base);
                const int groups = T * (BM / 4);
                const size_t sstride4 = (size_t)p.N * (BM / 4);
                const int et = threadIdx.x - 64;
                for (int g = et; g < groups; g += 128) {
                    float4 q4[MAX_SPLITS];
#pragma unroll
                    for (int sp = 0; sp < MAX_SPLITS; ++sp)
                        if (sp < p.splits) q4[sp] = __ldcg(base + sp * sstride4 + g);
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int sp = 0; sp < MAX_SPLITS; ++sp)
                        if (sp < p.splits) {
                            acc.x += q4[sp].x;
                            acc.y += q4[sp].y;
                            acc.z += q4[sp].z;
                            acc.w += q4[sp].w;
                        }
                    emit4(g / (BM / 4), (g % (BM / 4)) * 4, acc);
                }
            }
        }
    }
    if (warp < 2 && p.cluster && p.splits > 1) {   // the epilogue warps' cluster barriers, two per pass
        __syncwarp();
        const int tp = min(p.N, (p.ring_bytes / (BM * 4)) & ~15);
        for (int p0 = 0; p0 < T; p0 += tp) {
            cluster_sync();
            cluster_sync();
        }
    }
    // A block barrier needs converged warps: lanes that skipped a one-thread branch
    // above (barrier set-up, the TMA and MMA roles) wait here for it first.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();   // reconverge: lane 0 ran the MMA loop alone, dealloc is warp-collective
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
    }
}

}  // namespace

// ---------------------------------------------------------------- host side
cudaError_t record_profile(cudaEvent_t ev, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return e;
    return cs != cudaStreamCaptureStatusNone ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, st);
}

namespace {

// Shared-memory budgets: the projection and the shrink that precedes it may share
// an SM while both run, so their rings together stay inside one SM's 228 KiB.
constexpr int PROJ_SMEM_BUDGET = 136 * 1024;
constexpr int SHRINK_SMEM_BUDGET = 84 * 1024;

int clamp_stages(int ns) { return ns < 2 ? 2 : (ns > MAX_STAGES ? MAX_STAGES : ns); }

// the K splits of a tile as a cluster: a power of two, at most MAX_CLUSTER
int cluster_splits(int s) {
    int c = 1;
    while (c * 2 <= s && c * 2 <= MAX_CLUSTER) c *= 2;
    return c;
}

// K splits so that row tiles x token tiles x splits fill the SMs once, with the
// partial tiles of a tile (splits x N x 128 floats) bounded.
int k_splits(int tiles, int kb_total, int N) {
    int s = sm_count() / (tiles > 0 ? tiles : 1);
    const int cap = 1024 / (N > 0 ? N : 1);
    if (s > cap) s = cap;
    if (s > MAX_SPLITS) s = MAX_SPLITS;
    if (s > kb_total) s = kb_total;
    if (s < 1) s = 1;
    return s;
}

int max_dyn_smem() {
    static int v = 0;
    if (!v) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || v <= 0)
            v = 227 * 1024;
    }
    return v;
}

size_t align16(size_t v) { return (v + 15) / 16 * 16; }

// dynamic shared memory of one CTA: alignment slack, ring (+ segment scratch), tail
size_t smem_bytes(const GemmParams& p) { return 1024 + (size_t)p.tail_off + sizeof(Tail); }

int proj_tiles(const PoolDims& d) { return (d.dout + BM - 1) / BM; }
int token_tiles(int T) { return (T + MAX_N - 1) / MAX_N; }

}  // namespace

cudaError_t tc_init() {
    // the cap on dynamic shared memory is raised once, outside any stream capture
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    // static shared memory counts against the same per-block limit
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, swapab_gemm_kernel<false>);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(swapab_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - (int)fa.sharedSizeBytes);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, swapab_gemm_kernel<true>);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(swapab_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - (int)fa.sharedSizeBytes);
    // the same (largest) shared-memory carve-out for every kernel of a forward, so that
    // consecutive kernels can share an SM without reconfiguring it
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(swapab_gemm_kernel<false>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(swapab_gemm_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess) e = prefill_init();
    return e;
}

TcWorkspaceNeeds tc_workspace_needs(bool bf16, const PoolDims& d) {
    TcWorkspaceNeeds n{};
    n.need_v32 = !bf16;   // fp32 pools use the FMA path
    if (bf16) {
        // the global reduction (allocation-free entry point aside, only used when a
        // tile's splits cannot form a cluster): tiles x splits <= SMs partial tiles
        const int ncap = d.max_tokens < MAX_N ? (d.max_tokens + 15) / 16 * 16 : MAX_N;
        n.partial_bytes = (size_t)sm_count() * BM * ncap * sizeof(float);
        n.counter_bytes = sizeof(int32_t) * (size_t)proj_tiles(d);
        n.tmask_bytes = (size_t)token_tiles(d.max_tokens) * d.max_chunks;
    }
    return n;
}

bool tc_encode_arena_maps(TcArenaMaps* m, void* arena_down, void* arena_up, int units, int din, int dout) {
    {
        cuuint64_t dims[2] = {(cuuint64_t)din, (cuuint64_t)units};
        cuuint64_t strides[1] = {(cuuint64_t)din * 2};
        cuuint32_t box[2] = {BK, (cuuint32_t)CHUNK};
        if (!tc_encode(&m->down, arena_down, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return false;
    }
    cuuint64_t dims[3] = {8, (cuuint64_t)dout, (cuuint64_t)(units / 8)};
    cuuint64_t strides[2] = {16, (cuuint64_t)dout * 16};
    cuuint32_t box128[3] = {8, 128, 2};
    cuuint32_t box256[3] = {8, 256, 2};
    return tc_encode(&m->up128, arena_up, 3, dims, strides, box128, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           tc_encode(&m->up256, arena_up, 3, dims, strides, box256, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool tc_supported(const PoolDims& d, int T) {
    (void)d;
    return T >= 1;
}

cudaError_t tc_forward(const TcForwardArgs& a, cudaStream_t st) {
    const PoolDims& d = a.dims;
    const int T = a.T;
    const bool decode = T <= MAX_N;
    const int kb_total = (d.din + BK - 1) / BK;
    const int n_chunks = a.lora ? a.n_chunks : 0;
    const bool shrink = n_chunks > 0;
    cudaError_t e;

    // ---- shrink: Vt = masked scale * Down_chunks X^T, per token tile, the used chunks
    if (shrink) {
        const int Ns = decode ? (T + 15) / 16 * 16 : MAX_N;
        CUtensorMap tmXs, tmNone;
        std::memset(&tmNone, 0, sizeof tmNone);
        cuuint64_t dims[2] = {(cuuint64_t)d.din, (cuuint64_t)T};
        cuuint64_t strides[1] = {(cuuint64_t)d.din * 2};
        cuuint32_t box[2] = {BK, (cuuint32_t)Ns};
        if (!tc_encode(&tmXs, a.X, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        const int tiles = (n_chunks + CHUNKS_PER_TILE - 1) / CHUNKS_PER_TILE;
        const int ztiles = token_tiles(T);
        GemmParams g{};
        g.chunks = a.ws.chunks;
        g.row_adapter = a.row_adapter;
        g.slots = a.slots;
        g.vt = (__nv_bfloat16*)a.ws.vt;
        g.tmask = a.ws.tmask;
        g.partials = a.ws.partials;
        g.tile_ctr = a.ws.tile_ctr;
        g.status = a.ws.status;
        g.T = T;
        g.N = Ns;
        g.kb_total = kb_total;
        g.tcap = d.tcap;
        g.n_chunks = n_chunks;
        g.S = d.S;
        g.max_chunks = d.max_chunks;
        g.ws = a.ws;
        // A holds the chunks of one row tile: fewer than 8 when fewer are loaded
        g.a_bytes = (n_chunks < CHUNKS_PER_TILE ? n_chunks : CHUNKS_PER_TILE) * CHUNK_BYTES;
        const int sb = g.a_bytes + b_bytes(Ns);
        g.splits = cluster_splits(k_splits(tiles * ztiles, kb_total, Ns));
        g.stages = clamp_stages(SHRINK_SMEM_BUDGET / sb);
        // the MMA reads 128 rows of A from every stage: slack after the last one
        g.ring_bytes = g.stages * sb + (A_BYTES - g.a_bytes);
        // segment builder of CTA (0,0,0): scratch beside the ring, built by the epilogue
        // warps while the loads run, if it fits; else by the whole CTA before its loads
        const int room = max_dyn_smem() - 1024 - (int)sizeof(Tail) - 16 - g.ring_bytes;
        SegPlan sp = seg_plan(d.S, 4, room > 0 ? room / 4 : 0, T);
        size_t scratch = 0;
        if (sp.P >= 1) {
            g.seg_mode = SEG_BESIDE;
            scratch = align16((size_t)sp.ints * 4);
        } else {
            sp = seg_plan(d.S, NUM_THREADS / 32, (max_dyn_smem() - 1024 - (int)sizeof(Tail) - 16) / 4, T);
            if (sp.P < 1) return cudaErrorInvalidConfiguration;
            g.seg_mode = SEG_BEFORE;
            if ((size_t)g.ring_bytes < (size_t)sp.ints * 4) g.ring_bytes = (int)align16((size_t)sp.ints * 4);
        }
        g.seg_P = sp.P;
        g.seg_stage_rows = sp.stage_rows ? 1 : 0;
        g.scratch_off = g.ring_bytes;
        g.tail_off = (int)align16((size_t)g.ring_bytes + scratch);
        g.cluster = g.splits > 1 ? 1 : 0;
        // first kernel of the forward: an ordinary launch (it overwrites the Vt the
        // previous forward's projection read)
        e = launch_k(swapab_gemm_kernel<true>, dim3(tiles, g.splits, ztiles), dim3(NUM_THREADS), smem_bytes(g), st,
                     false, g.cluster ? g.splits : 1, tmNone, tmXs, tmNone, a.maps.down, g);
        if (e != cudaSuccess) return e;
    }

    const int N = decode ? (T + 15) / 16 * 16 : 128;     // token rows per tile
    CUtensorMap tmW, tmX, tmV;
    {
        cuuint64_t dims[2] = {(cuuint64_t)d.din, (cuuint64_t)d.dout};
        cuuint64_t strides[1] = {(cuuint64_t)d.din * 2};
        cuuint32_t box[2] = {BK, decode ? (cuuint32_t)BM : 256u};
        if (!tc_encode(&tmW, a.W, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)d.din, (cuuint64_t)T};
        cuuint64_t strides[1] = {(cuuint64_t)d.din * 2};
        cuuint32_t box[2] = {BK, (cuuint32_t)N};
        if (!tc_encode(&tmX, a.X, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[3] = {(cuuint64_t)CHUNK, (cuuint64_t)d.tcap, (cuuint64_t)d.max_chunks};
        cuuint64_t strides[2] = {(cuuint64_t)CHUNK * 2, (cuuint64_t)d.tcap * CHUNK * 2};
        cuuint32_t box[3] = {CHUNK, (cuuint32_t)N, EXT_SUB};
        if (!tc_encode(&tmV, a.ws.vt, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_32B)) return cudaErrorInvalidValue;
    }

    if (!decode) {
        if (a.ev_start && (e = record_profile(a.ev_start, st)) != cudaSuccess) return e;
        if ((e = launch_prefill(a, tmX, tmW, tmV, sm_count(), shrink, st)) != cudaSuccess) return e;
        if (a.ev_stop && (e = record_profile(a.ev_stop, st)) != cudaSuccess) return e;
        return cudaSuccess;
    }

    const int tiles = proj_tiles(d);
    GemmParams p{};
    p.chunks = a.ws.chunks;
    p.row_adapter = a.row_adapter;
    p.Y = (__nv_bfloat16*)a.Y;
    p.partials = a.ws.partials;
    p.tile_ctr = a.ws.tile_ctr;
    p.status = a.ws.status;
    p.T = T;
    p.dout = d.dout;
    p.N = N;
    p.kb_total = kb_total;
    p.n_chunks = n_chunks;
    p.ext_units = shrink ? (n_chunks + EXT_SUB - 1) / EXT_SUB : 0;
    p.splits = cluster_splits(k_splits(tiles, kb_total, N));
    p.stages = clamp_stages(PROJ_SMEM_BUDGET / stage_bytes(N));
    p.a_bytes = A_BYTES;
    p.ring_bytes = p.stages * stage_bytes(N);
    p.tail_off = p.ring_bytes;
    p.tcap = d.tcap;
    p.pdl = shrink ? 1 : 0;
    p.cluster = p.splits > 1 ? 1 : 0;
    p.S = d.S;
    p.max_chunks = d.max_chunks;
    if (a.ev_start && (e = record_profile(a.ev_start, st)) != cudaSuccess) return e;
    e = launch_k(swapab_gemm_kernel<false>, dim3(tiles, p.splits, 1), dim3(NUM_THREADS), smem_bytes(p), st,
                 shrink && !a.ev_start, p.cluster ? p.splits : 1, tmW, tmX, tmV, a.maps.up128, p);
    if (e != cudaSuccess) return e;
    if (a.ev_stop && (e = record_profile(a.ev_stop, st)) != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t tc_project_with_scratch(const void* X, const void* W, int T, int din, int dout, void* Y,
                                   float* partials, size_t partial_bytes, int32_t* counters, int max_tiles,
                                   uint32_t* status, cudaStream_t st) {
    if (T < 1 || T > MAX_N) return cudaErrorInvalidValue;
    const int N = (T + 15) / 16 * 16;
    const int tiles = (dout + BM - 1) / BM;
    const int kb_total = (din + BK - 1) / BK;
    if (tiles > max_tiles) return cudaErrorInvalidValue;
    CUtensorMap tmW, tmX, tmNone;
    std::memset(&tmNone, 0, sizeof tmNone);
    {
        cuuint64_t dims[2] = {(cuuint64_t)din, (cuuint64_t)dout};
        cuuint64_t strides[1] = {(cuuint64_t)din * 2};
        cuuint32_t box[2] = {BK, (cuuint32_t)BM};
        if (!tc_encode(&tmW, W, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)din, (cuuint64_t)T};
        cuuint64_t strides[1] = {(cuuint64_t)din * 2};
        cuuint32_t box[2] = {BK, (cuuint32_t)N};
        if (!tc_encode(&tmX, X, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    GemmParams p{};
    p.Y = (__nv_bfloat16*)Y;
    p.partials = partials;
    p.tile_ctr = counters;
    p.status = status;
    p.T = T;
    p.dout = dout;
    p.N = N;
    p.kb_total = kb_total;
    p.ext_units = 0;
    // as many K splits as fill the SMs and whose partial tiles fit the scratch
    int splits = k_splits(tiles, kb_total, N);
    const size_t per_split = (size_t)tiles * BM * N * sizeof(float);
    while (splits > 1 && (size_t)splits * per_split > partial_bytes) --splits;
    p.splits = splits;
    p.stages = clamp_stages(PROJ_SMEM_BUDGET / stage_bytes(N));
    p.a_bytes = A_BYTES;
    p.ring_bytes = p.stages * stage_bytes(N);
    p.tail_off = p.ring_bytes;
    p.tcap = 0;
    p.pdl = 0;
    p.cluster = 0;   // the K splits meet through the given scratch
    return launch_k(swapab_gemm_kernel<false>, dim3(tiles, p.splits, 1), dim3(NUM_THREADS), smem_bytes(p), st, false,
                    1, tmW, tmX, tmNone, tmNone, p);
}

}  // namespace mlora
