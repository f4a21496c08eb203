// Tensor-core path of the bf16 forward: tcgen05 MMA with TMEM accumulators, TMA
// loads into 128B/32B-swizzled shared memory, warp-specialised pipeline.
//
// "swap-AB" GEMM kernel, in two modes.  The weight-like operand is the MMA's M
// side (128 rows per tile) and the tokens are the N side (N = up to 256 tokens,
// a multiple of 16), so the weight streams through the tensor cores once however
// few rows the batch has.
//
// Projection (T <= 256): rows = output features.  The K loop of a tile is the din
// columns of W followed by a K-extension over the touched adapters (ai-infra-kb
// "M031" §02: each row adds scale_a Up_a (Down_a x)):
//
//     Y^T[o, t] = sum_i W[o, i] X[t, i]  +  sum_c Up_{a(c)}[o, col(c) + j] Vt[c][t][j]
//
// where chunk c holds 16 rank columns of one touched adapter and Vt[c][t][:] is
// scale_a Down_a x_t for rows t of that adapter and zero for every other row.  The
// delta therefore lands in the same fp32 accumulator as the base product, on the
// row's own column, and the output is rounded once.  Up is read once per output
// tile through per-slot TMA descriptors whose out-of-range columns read as zero.
//
// Shrink (any T; token tiles of 256 along grid z): rows = 8 chunks of 16 rank rows
// of the touched adapters' Down (per-slot descriptors; rows past the rank read as
// zero), K = din, giving Down_c X^T for every token.  The epilogue keeps the
// entry of a token only if the token belongs to the chunk's adapter, scales it,
// rounds it to bf16 and writes Vt; every other entry is written as zero, so Vt
// needs no clearing.
//
// Work split: a grid of (row tile, K split, token tile).  Split s takes a
// contiguous share of the K steps.  Each split writes an fp32 partial tile; the
// last split to arrive (atomic counter, no waiting) adds all partials in split
// order and writes the result, so it does not depend on arrival order.
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
constexpr int MAX_SPLITS = 16;     // K splits per tile at most
constexpr int MAX_CLUSTER = 8;     // K splits of a tile reduced inside one (portable) cluster

__host__ __device__ constexpr int b_bytes(int n) { return n * BK * 2; }
__host__ __device__ constexpr int stage_bytes(int n) { return A_BYTES + b_bytes(n); }

struct GemmParams {
    const int32_t* chunk_slot;      // projection: chunk table of the touched slots (from the shrink)
    const int32_t* chunk_unit;
    const int32_t* meta;            // meta[1] = number of chunks of the touched slots
    const int32_t* row_adapter;     // shrink: slot id per token
    const SlotRec* slots;
    __nv_bfloat16* Y;               // projection output [T x dout]
    __nv_bfloat16* vt;              // shrink output [max_chunks][tcap][16]
    float* partials;                // [tile][z][split][BM][N]
    int32_t* tile_ctr;              // [tile][z] arrival counters
    uint32_t* status;
    int T, dout, N, kb_total, ext_units, splits, stages, tcap;
    int pdl;    // launched while an earlier kernel may still run: wait before reading its outputs
    // shrink prologue: segment builder over S slots with segP row ranges, in
    // scratch_bytes at the start of shared memory (the ring region is at least that
    // large); seg_warp: one warp builds it (segP = 1)
    int S, segP, max_chunks, scratch_bytes, seg_warp;
    // the K splits of a tile form a cluster and reduce through distributed shared memory
    int cluster;
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
    const int NS = p.stages;
    const int SB = stage_bytes(p.N);
    const int ring = max(NS * SB, SHRINK ? p.scratch_bytes : 0);
    uint64_t* full = (uint64_t*)(smem + ring);
    uint64_t* empty = full + NS;
    uint64_t* acc_full = empty + NS;
    int* stage_kind = (int*)(acc_full + 1);          // -1 = din step, else number of valid chunks
    uint32_t* tmem_slot = (uint32_t*)(stage_kind + NS);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    int* flags = (int*)(tmem_slot + 2);              // [0] issued-any, [1] last-arrival
    int* my_chunk = flags + 2;                       // shrink: [4][8] slot, unit, valid columns, scale
    int* tile_ra = my_chunk + 4 * CHUNKS_PER_TILE;   // shrink: slot of each token of this token tile
    int* tile_chunks_s = tile_ra + MAX_N;            // shrink: chunks of this row tile

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, split = blockIdx.y, ztile = blockIdx.z;
    const int tok0 = ztile * MAX_N;                  // first token of this token tile
    const int T = min(p.T - tok0, p.N);              // tokens in this tile

    if (SHRINK) {
        pdl_trigger();   // the projection may launch and stream W meanwhile
        // Segment build (M031 §02/§03) in the stage memory, before any load uses it.
        // Every CTA builds the same table; CTA (0,0,0) publishes it (perm, offsets,
        // chunk table, meta) for the projection and for the caller.  Small batches
        // are built by warp 2 alone while warps 0 and 1 set up barriers and TMEM.
        if (!p.seg_warp || warp == 2) {
            const seg::Scratch sc = seg::carve(reinterpret_cast<int*>(smem), p.S, p.segP, p.max_chunks);
            const bool publish = (blockIdx.x | blockIdx.y | blockIdx.z) == 0;
            const int n_chunks =
                p.seg_warp ? seg::build<true>(p.row_adapter, p.T, p.slots, p.S, 1, p.max_chunks, sc, publish, p.ws)
                           : seg::build<false>(p.row_adapter, p.T, p.slots, p.S, p.segP, p.max_chunks, sc, publish,
                                               p.ws);
            const int gt = p.seg_warp ? lane : (int)threadIdx.x, gn = p.seg_warp ? 32 : (int)blockDim.x;
            const int tc = min(CHUNKS_PER_TILE, n_chunks - tile * CHUNKS_PER_TILE);
            if (gt == 0) *tile_chunks_s = tc;
            if (gt < CHUNKS_PER_TILE && gt < tc) {
                const int c = tile * CHUNKS_PER_TILE + gt;
                my_chunk[gt] = sc.c_slot[c];
                my_chunk[CHUNKS_PER_TILE + gt] = sc.c_unit[c];
                my_chunk[2 * CHUNKS_PER_TILE + gt] = sc.c_kval[c];
                my_chunk[3 * CHUNKS_PER_TILE + gt] = __float_as_int(p.slots[sc.c_slot[c]].scale);
            }
            // the epilogue masks tokens by their slot: keep this token tile's row map at hand
            for (int t = gt; t < T; t += gn) tile_ra[t] = sc.ra_s[tok0 + t];
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
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        flags[0] = 0;
        flags[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!SHRINK) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
    }
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // A block barrier needs converged warps: lanes that skipped a one-thread branch
    // above (barrier set-up, the TMA and MMA roles) wait here for it first.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int tile_chunks = SHRINK ? *tile_chunks_s : 0;
    if (SHRINK && tile_chunks <= 0) {   // no chunk of the touched slots falls in this row tile
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
        int n_chunks = -1;
        int armed[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int i = 0; i < n_steps; ++i) {
            if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.status)) break;
            ++armed[s];
            uint8_t* a = smem + (size_t)s * SB;
            uint8_t* b = a + A_BYTES;
            const int kb = kb0 + i;
            if (SHRINK) {
                stage_kind[s] = -1;
                mbar_expect_tx(&full[s], (uint32_t)(tile_chunks * CHUNK * BK * 2 + b_bytes(p.N)));
                for (int j = 0; j < tile_chunks; ++j)
                    tma_2d(a + j * (CHUNK * BK * 2), &tmArena, &full[s], kb * BK, my_chunk[CHUNKS_PER_TILE + j]);
                tma_2d(b, &tmX, &full[s], kb * BK, tok0);
            } else if (kb < kb1) {
                stage_kind[s] = -1;
                mbar_expect_tx(&full[s], (uint32_t)SB);
                tma_2d(a, &tmW, &full[s], kb * BK, tile * BM);
                tma_2d(b, &tmX, &full[s], kb * BK, 0);
            } else {
                if (n_chunks < 0) {
                    if (p.pdl) pdl_wait();   // chunk table and Vt come from the kernels before
                    n_chunks = p.meta[1];
                }
                const int u = eu0 + (kb - kb1);
                const int c0 = u * EXT_SUB;
                int nv = n_chunks - c0;
                nv = nv < 0 ? 0 : (nv > EXT_SUB ? EXT_SUB : nv);
                stage_kind[s] = nv;
                if (nv == 0) {
                    mbar_expect_tx(&full[s], 0);
                } else {
                    mbar_expect_tx(&full[s], (uint32_t)(nv * (BM * 32) + b_bytes(p.N)));
                    tma_3d(b, &tmV, &full[s], 0, 0, c0);
                    for (int j = 0; j < nv; ++j)   // two blocks of 8 rank columns x 128 rows
                        tma_3d(a + j * (BM * 32), &tmArena, &full[s], 0, tile * BM, p.chunk_unit[c0 + j] >> 3);
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
                while (!mbar_try_wait(&full[j], (uint32_t)((armed[j] - 1) & 1)) && clock64() - t0 < 200000000ll) {
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
            if (!mbar_wait(&full[s], ph, abort_flag, p.status)) break;
            tc_fence_after();
            const uint32_t a = smem_u32(smem + (size_t)s * SB);
            const uint32_t b = a + A_BYTES;
            const int kind = stage_kind[s];
            if (kind < 0) {
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    mma_bf16(tmem, sdesc(a + k * 32, 1024, SW128), sdesc(b + k * 32, 1024, SW128), idesc, acc);
                    acc = 1;
                }
            } else {
                // Up chunk: [2 blocks of 8 columns][128 rows][16 B], no swizzle (K-direction core
                // matrices BM*16 bytes apart, M-direction 128 bytes); Vt chunk: 32-byte swizzle
                for (int j = 0; j < kind; ++j) {
                    mma_bf16(tmem, sdesc_lbo(a + j * (BM * 32), BM * 16, 128, SW_NONE),
                             sdesc(b + j * (p.N * 32), 256, SW32), idesc, acc);
                    acc = 1;
                }
            }
            mma_commit(&empty[s]);
            if (++s == NS) {
                s = 0;
                ph ^= 1;
            }
        }
        flags[0] = (int)acc;
        mma_commit(acc_full);
        if (*abort_flag) {   // MMAs already issued must finish before TMEM is released
            const long long t0 = clock64();
            while (!mbar_try_wait(acc_full, 0) && clock64() - t0 < 200000000ll) {
            }
        }
    } else if (warp >= 2) {
        // ---------------- epilogue: TMEM -> partial tile, or the final values
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;          // row of the tile
        const bool ok = mbar_wait(acc_full, 0, abort_flag, p.status);
        __syncwarp();   // reconverge: lanes may leave the wait loop apart; tcgen05.ld is warp-collective
        tc_fence_after();
        const bool have = __all_sync(0xffffffffu, ok) && flags[0] != 0;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);

        // final write of 16 consecutive tokens t0..t0+15 of this row
        int c_slot = -1, c_idx = 0;
        float c_scale = 0.f;
        if (SHRINK && (row / CHUNK) < tile_chunks) {
            c_idx = tile * CHUNKS_PER_TILE + row / CHUNK;
            c_slot = my_chunk[row / CHUNK];
            // rank columns past the adapter's rank belong to the next adapter in the arena
            c_scale = (row % CHUNK) < my_chunk[2 * CHUNKS_PER_TILE + row / CHUNK]
                          ? __int_as_float(my_chunk[3 * CHUNKS_PER_TILE + row / CHUNK])
                          : 0.f;
        }
        const int o = tile * BM + row;
        auto emit = [&](int t0, const float* v) {
            if (SHRINK) {
                if (c_slot < 0) return;
                __nv_bfloat16* dst = p.vt + ((size_t)c_idx * p.tcap + tok0) * CHUNK + (row % CHUNK);
                for (int j = 0; j < 16 && t0 + j < T; ++j) {
                    const bool mine = tile_ra[t0 + j] == c_slot;
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
                const int ci = r0 / CHUNK;
                if (ci >= tile_chunks) return;
                const int slot = my_chunk[ci];
                const int kval = my_chunk[2 * CHUNKS_PER_TILE + ci];
                const int k0 = r0 % CHUNK;
                const bool mine = tile_ra[t] == slot;
                const float sc = mine ? __int_as_float(my_chunk[3 * CHUNKS_PER_TILE + ci]) : 0.f;
                __nv_bfloat162 lo = __floats2bfloat162_rn(k0 < kval ? sc * v.x : 0.f, k0 + 1 < kval ? sc * v.y : 0.f);
                __nv_bfloat162 hi = __floats2bfloat162_rn(k0 + 2 < kval ? sc * v.z : 0.f, k0 + 3 < kval ? sc * v.w : 0.f);
                uint2 w;
                w.x = *reinterpret_cast<uint32_t*>(&lo);
                w.y = *reinterpret_cast<uint32_t*>(&hi);
                *reinterpret_cast<uint2*>(p.vt + ((size_t)(tile * CHUNKS_PER_TILE + ci) * p.tcap + tok0 + t) * CHUNK + k0) = w;
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

        const int ctr = tile * gridDim.z + ztile;
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
            // memory of all splits, summed in split order, and write it.
            float* part_s = reinterpret_cast<float*>(smem);
            for (int t0 = 0; t0 < T; t0 += 16) {
                float v[16];
                if (have) tmem_ld16(tbase + t0, v);
                else
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) part_s[(t0 + j) * BM + row] = v[j];
            }
            __syncwarp();
            cluster_sync();
            const int ts = (T + p.splits - 1) / p.splits;
            const int t_lo = (int)cluster_rank() * ts;
            const int t_hi = min(T, t_lo + ts);
            const uint32_t part_a = smem_u32(part_s);
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
                emit4(t, r0, acc);
            }
            __syncwarp();
            cluster_sync();   // no CTA leaves while the others still read its shared memory
        } else {
            // partial tile layout [split][token][row] fp32: for a fixed token the 128 rows
            // of a tile are contiguous, so both the stores below and the reduction's
            // loads are coalesced
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
                flags[1] = last;
            }
            epi_bar();
            if (flags[1]) {
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
    if (warp < 2 && p.cluster && p.splits > 1) {   // the epilogue warps' two cluster barriers
        __syncwarp();
        cluster_sync();
        cluster_sync();
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

int ring_stages(int N, int budget) {
    int ns = budget / stage_bytes(N);
    if (ns < 2) ns = 2;
    if (ns > 8) ns = 8;
    return ns;
}

// K splits so that row tiles x token tiles x splits fill the SMs once, with the
// partial tiles the last split reads back (splits x N x 128 floats) bounded.
int k_splits(int tiles, int kb_total, int N) {
    int s = sm_count() / (tiles > 0 ? tiles : 1);
    const int cap = 1024 / (N > 0 ? N : 1);
    if (s > cap) s = cap;
    if (s > MAX_SPLITS) s = MAX_SPLITS;
    if (s > kb_total) s = kb_total;
    if (s < 1) s = 1;
    return s;
}

// dynamic shared memory of one CTA: alignment slack, the ring (or the segment
// scratch, if larger), barriers, stage kinds, TMEM slot / flags, chunk info
size_t smem_bytes(int stages, int N, int scratch_bytes = 0) {
    size_t ring = (size_t)stages * stage_bytes(N);
    if ((size_t)scratch_bytes > ring) ring = (size_t)scratch_bytes;
    return 1024 + ring + (size_t)(2 * stages + 1) * 8 + (size_t)stages * 4 + 16 + 4 * CHUNKS_PER_TILE * 4 +
           MAX_N * 4 + 16;
}

int proj_tiles(const PoolDims& d) { return (d.dout + BM - 1) / BM; }
int shrink_tiles(const PoolDims& d) { return (d.max_chunks + CHUNKS_PER_TILE - 1) / CHUNKS_PER_TILE; }
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
        // partial tiles exist only when a split count > 1, i.e. tiles x token tiles x
        // splits <= SMs; each of the two kernels gets its own region
        const int ncap = d.max_tokens < MAX_N ? (d.max_tokens + 15) / 16 * 16 : MAX_N;
        const size_t region = (size_t)sm_count() * BM * ncap * sizeof(float);
        n.partial_bytes = 2 * region;
        n.counter_bytes =
            sizeof(int32_t) * ((size_t)proj_tiles(d) + (size_t)shrink_tiles(d) * token_tiles(d.max_tokens));
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
    const int ext_chunks = a.lora ? a.ext_chunk_cap : 0;
    const bool shrink = a.lora && ext_chunks > 0;
    const size_t region_floats =
        (size_t)sm_count() * BM * (d.max_tokens < MAX_N ? (d.max_tokens + 15) / 16 * 16 : MAX_N);
    cudaError_t e;

    // ---- shrink: Vt = masked scale * Down_chunks X^T, all tokens, every chunk of the touched slots
    if (shrink) {
        const int Ns = decode ? (T + 15) / 16 * 16 : MAX_N;
        CUtensorMap tmXs, tmNone;
        std::memset(&tmNone, 0, sizeof tmNone);
        cuuint64_t dims[2] = {(cuuint64_t)d.din, (cuuint64_t)T};
        cuuint64_t strides[1] = {(cuuint64_t)d.din * 2};
        cuuint32_t box[2] = {BK, (cuuint32_t)Ns};
        if (!tc_encode(&tmXs, a.X, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        const int tiles = (ext_chunks + CHUNKS_PER_TILE - 1) / CHUNKS_PER_TILE;
        const int ztiles = token_tiles(T);
        GemmParams g{};
        g.meta = a.ws.meta;
        g.row_adapter = a.row_adapter;
        g.slots = a.slots;
        g.vt = (__nv_bfloat16*)a.ws.vt;
        g.partials = a.ws.partials + region_floats;
        g.tile_ctr = a.ws.tile_ctr + proj_tiles(d);
        g.status = a.ws.status;
        g.T = T;
        g.N = Ns;
        g.kb_total = kb_total;
        g.splits = k_splits(tiles * ztiles, kb_total, Ns);
        if (g.splits > 8) g.splits = 8;   // the shrink's K loop is short: fewer, longer splits
        g.stages = ring_stages(Ns, SHRINK_SMEM_BUDGET);
        g.tcap = d.tcap;
        g.pdl = 0;
        g.S = d.S;
        g.max_chunks = d.max_chunks;
        g.ws = a.ws;
        // segment scratch in the ring memory: as many row ranges as fit (at most one per warp)
        const int ring_ints = g.stages * stage_bytes(Ns) / 4;
        g.seg_warp = T <= MAX_N && d.S <= 1024;   // decode-sized: one warp builds the segments
        g.segP = g.seg_warp ? 1 : seg_warps_for(d.S, NUM_THREADS / 32, ring_ints, d.max_chunks, T);
        if (g.segP < 1) g.segP = 1;   // the ring grows to the scratch (many slots, long batches)
        g.scratch_bytes = 4 * seg::scratch_ints(d.S, g.segP, d.max_chunks, T);
        // first kernel of the forward: an ordinary launch (it may overwrite the workspace
        // the previous forward's kernels read)
        g.cluster = g.splits > 1 && g.splits <= MAX_CLUSTER && Ns * BM * 4 <= g.stages * stage_bytes(Ns);
        e = launch_k(swapab_gemm_kernel<true>, dim3(tiles, g.splits, ztiles), dim3(NUM_THREADS),
                     smem_bytes(g.stages, Ns, g.scratch_bytes), st, false, g.cluster ? g.splits : 1, tmNone, tmXs, tmNone, a.maps.down, g);
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
    p.chunk_slot = a.ws.chunk_slot;
    p.chunk_unit = a.ws.chunk_unit;
    p.meta = a.ws.meta;
    p.Y = (__nv_bfloat16*)a.Y;
    p.partials = a.ws.partials;
    p.tile_ctr = a.ws.tile_ctr;
    p.status = a.ws.status;
    p.T = T;
    p.dout = d.dout;
    p.N = N;
    p.kb_total = kb_total;
    p.ext_units = (ext_chunks + EXT_SUB - 1) / EXT_SUB;
    p.splits = k_splits(tiles, kb_total, N);
    p.stages = ring_stages(N, PROJ_SMEM_BUDGET);
    p.tcap = d.tcap;
    p.pdl = shrink ? 1 : 0;
    if (a.ev_start && (e = record_profile(a.ev_start, st)) != cudaSuccess) return e;
    if (p.splits > MAX_CLUSTER && N * BM * 4 <= p.stages * stage_bytes(N)) p.splits = MAX_CLUSTER;
    p.cluster = p.splits > 1 && N * BM * 4 <= p.stages * stage_bytes(N);
    e = launch_k(swapab_gemm_kernel<false>, dim3(tiles, p.splits, 1), dim3(NUM_THREADS), smem_bytes(p.stages, N), st,
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
    p.stages = ring_stages(N, PROJ_SMEM_BUDGET);
    p.tcap = 0;
    p.pdl = 0;
    p.cluster = 0;   // the K splits meet through the given scratch
    return launch_k(swapab_gemm_kernel<false>, dim3(tiles, p.splits, 1), dim3(NUM_THREADS), smem_bytes(p.stages, N),
                    st, false, 1, tmW, tmX, tmNone, tmNone, p);
}

}  // namespace mlora
