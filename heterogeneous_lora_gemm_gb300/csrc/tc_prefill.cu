// Prefill-shaped batches (T > 256): persistent tcgen05 GEMM with the fused expand.
//
// Tiles are 128 tokens x 256 output features (one tcgen05.mma.cta_group::1 of
// M = 128, N = 256, K = 16 per 32 bytes of K).  One CTA per SM walks its share of
// the tiles in a grouped raster order (8 token tiles share each weight tile, so
// the weight tiles in flight stay in L2).  Warp 0 issues TMA loads into a 4-stage
// ring, warp 1 issues the MMAs into one of two TMEM accumulators (2 x 256
// columns), and warps 2-5 drain the other accumulator to bf16 Y while the next
// tile is being multiplied.  The raster walks all weight tiles for a group of token
// tiles whose X tiles together take about 40 MB, so that they stay in L2 while the
// weight streams past: W is read once per group (groups of 8 token tiles re-read it
// from DRAM once per 1024 tokens, three times the algorithmic bytes in all).  As in the decode kernel, the K loop of every tile is
// din columns of X W^T followed by the K-extension over the loaded adapters'
// chunks (ai-infra-kb "M031" §02), so each row's delta is added to its own output
// row before the single rounding.  A tile multiplies only the chunks the shrink
// marked as used by its token tile (tmask); the others' Up tiles are not loaded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tc.h"
#include "tc_ptx.cuh"

namespace mlora {

using namespace ptx;

namespace {

constexpr int PM = 128;                         // tokens per tile
constexpr int PN = 256;                         // output features per tile
constexpr int PK = 64;                          // K per pipeline step
constexpr int PA_BYTES = PM * PK * 2;           // 16 KiB
constexpr int PB_BYTES = PN * PK * 2;           // 32 KiB
constexpr int PSTAGE = PA_BYTES + PB_BYTES;     // 48 KiB
constexpr int PSTAGES = 4;
constexpr int P_THREADS = 192;
constexpr int GROUP_MIN = 8;                    // token tiles per raster group, at least
constexpr size_t GROUP_X_BYTES = 40u << 20;     // X bytes of one raster group, about
constexpr int EXT_SUB = 4;

struct PrefillParams {
    const ChunkRec* chunks;     // chunk table of the loaded slots
    const uint8_t* tmask;       // [token tile of 256][max_chunks], from the shrink
    __nv_bfloat16* Y;
    uint32_t* status;
    int T, dout, kb_total, m_tiles, n_tiles, vec_store;
    int n_chunks, max_chunks;
    int ext_steps;              // K-extension steps per tile (EXT_SUB chunks each), 0 without adapters
    int pdl;    // launched while the shrink may still run: wait before reading its outputs
    int group_m;   // token tiles per raster group
    unsigned long long* stamps;   // profiling records (NULL = off), see ptx::stamp_record
    int up_rows;                  // output rows per row of the Up map (8 or 1)
    int stamp_cap;
};

__device__ __forceinline__ void tile_coords(int i, int m_tiles, int n_tiles, int group_m, int& m, int& n) {
    const int per_group = group_m * n_tiles;
    const int first_m = (i / per_group) * group_m;
    const int gm = min(m_tiles - first_m, group_m);
    const int r = i % per_group;
    m = first_m + r % gm;
    n = r / gm;
}

__global__ void __launch_bounds__(P_THREADS, 1)
prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmUp,
                    PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(smem + (size_t)PSTAGES * PSTAGE);
    uint64_t* empty = full + PSTAGES;
    uint64_t* tfull = empty + PSTAGES;     // [2] accumulator ready
    uint64_t* tempty = tfull + 2;          // [2] accumulator drained
    uint64_t* drain = tempty + 2;          // MMA completion on the give-up path
    int* stage_kind = (int*)(drain + 1);   // -1 = din step, else bit mask of the chunks loaded
    uint32_t* tmem_slot = (uint32_t*)(stage_kind + PSTAGES);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = p.m_tiles * p.n_tiles;
    const unsigned long long t_start = (p.stamps && threadIdx.x == 0) ? gtimer() : 0ull;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
    }
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(512)
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
    const int steps = p.kb_total + p.ext_steps;
    pdl_trigger();   // the next forward's shrink may get resident and set up meanwhile

    if (warp == 0 && lane == 0) {
        // ---------------- producer
        int s = 0;
        uint32_t ph = 0;
        bool waited = false;
        int armed[PSTAGES] = {0, 0, 0, 0};
        for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
            int m, n;
            tile_coords(tile, p.m_tiles, p.n_tiles, p.group_m, m, n);
            for (int i = 0; i < steps; ++i) {
                if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.status)) break;
                ++armed[s];
                uint8_t* a = smem + (size_t)s * PSTAGE;
                uint8_t* b = a + PA_BYTES;
                if (i < p.kb_total) {
                    stage_kind[s] = -1;
                    mbar_expect_tx(&full[s], PSTAGE);
                    tma_2d(a, &tmX, &full[s], i * PK, m * PM);
                    tma_2d(b, &tmW, &full[s], i * PK, n * PN);
                } else {
                    if (!waited) {   // tmask and Vt come from the shrink
                        if (p.pdl) pdl_wait();
                        waited = true;
                    }
                    const int c0 = (i - p.kb_total) * EXT_SUB;
                    const uint8_t* tm = p.tmask + (size_t)(m * PM / 256) * p.max_chunks;
                    int used[EXT_SUB], un[EXT_SUB];
#pragma unroll
                    for (int j = 0; j < EXT_SUB; ++j) {   // independent loads, then the mask
                        const bool in = c0 + j < p.n_chunks;
                        used[j] = in ? tm[c0 + j] : 0;
                        un[j] = in ? p.chunks[c0 + j].unit : 0;
                    }
                    uint32_t mask = 0;
#pragma unroll
                    for (int j = 0; j < EXT_SUB; ++j)
                        if (used[j]) mask |= 1u << j;
                    stage_kind[s] = (int)mask;
                    if (mask == 0) {
                        mbar_expect_tx(&full[s], 0);
                    } else {
                        mbar_expect_tx(&full[s], (uint32_t)(PA_BYTES + __popc(mask) * (PN * 32)));
                        tma_3d(a, &tmV, &full[s], 0, m * PM / 8, c0 * 2);
#pragma unroll
                        for (int j = 0; j < EXT_SUB; ++j)   // two blocks of 8 rank columns x 256 rows
                            if ((mask >> j) & 1u) tma_3d(b + j * (PN * 32), &tmUp, &full[s], 0, n * PN / p.up_rows, un[j] >> 3);
                    }
                }
                if (++s == PSTAGES) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
        if (*abort_flag) {
            for (int j = 0; j < PSTAGES; ++j) {
                if (armed[j] == 0) continue;
                const long long t0 = clock64();
                while (!mbar_try_wait(&full[j], (uint32_t)((armed[j] - 1) & 1)) && clock64() - t0 < 200000000ll) {
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        const uint32_t idesc = idesc_bf16(PM, PN);
        int s = 0;
        uint32_t ph = 0;
        int local = 0;
        for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x, ++local) {
            const int buf = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            if (!mbar_wait(&tempty[buf], (use & 1) ^ 1, abort_flag, p.status)) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(buf * PN);
            uint32_t acc = 0;
            for (int i = 0; i < steps; ++i) {
                if (!mbar_wait(&full[s], ph, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t a = smem_u32(smem + (size_t)s * PSTAGE);
                const uint32_t b = a + PA_BYTES;
                const int kind = stage_kind[s];
                if (kind < 0) {
#pragma unroll
                    for (int k = 0; k < PK / 16; ++k) {
                        mma_bf16(d, sdesc(a + k * 32, 1024, SW128), sdesc(b + k * 32, 1024, SW128), idesc, acc);
                        acc = 1;
                    }
                } else {
                    // Vt chunk: [2 blocks of 8 columns][128 tokens][16 B]; Up chunk: [2 blocks of 8
                    // columns][256 rows][16 B]; no swizzle (K-direction core matrices PM*16 or
                    // PN*16 bytes apart, M/N-direction 128)
#pragma unroll
                    for (int j = 0; j < EXT_SUB; ++j)
                        if ((kind >> j) & 1) {
                            mma_bf16(d, sdesc_lbo(a + j * (PM * 32), PM * 16, 128, SW_NONE),
                                     sdesc_lbo(b + j * (PN * 32), PN * 16, 128, SW_NONE), idesc, acc);
                            acc = 1;
                        }
                }
                mma_commit(&empty[s]);
                if (++s == PSTAGES) {
                    s = 0;
                    ph ^= 1;
                }
            }
            mma_commit(&tfull[buf]);
        }
        if (*abort_flag) {   // MMAs already issued must finish before TMEM is released
            mma_commit(drain);
            const long long t0 = clock64();
            while (!mbar_try_wait(drain, 0) && clock64() - t0 < 200000000ll) {
            }
        }
    } else if (warp >= 2) {
        // ---------------- epilogue
        const int q = warp & 3;
        int local = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
            int m, n;
            tile_coords(tile, p.m_tiles, p.n_tiles, p.group_m, m, n);
            const int buf = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            const bool got = mbar_wait(&tfull[buf], use & 1, abort_flag, p.status);
            __syncwarp();   // reconverge: lanes may leave the wait loop apart; tcgen05.ld is warp-collective
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            const int t = m * PM + q * 32 + lane;
            const uint32_t taddr = tmem + (uint32_t)(buf * PN) + ((uint32_t)(q * 32) << 16);
            __nv_bfloat16* yrow = p.Y + (size_t)t * p.dout;
            for (int c0 = 0; c0 < PN; c0 += 16) {
                float v[16];
                tmem_ld16(taddr + c0, v);
                const int o = n * PN + c0;
                if (t < p.T) {
                    if (p.vec_store && o + 16 <= p.dout) {
                        uint4 w[2];
                        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(w);
#pragma unroll
                        for (int j = 0; j < 8; ++j) h[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
                        *reinterpret_cast<uint4*>(yrow + o) = w[0];
                        *reinterpret_cast<uint4*>(yrow + o + 8) = w[1];
                    } else {
                        for (int j = 0; j < 16; ++j)
                            if (o + j < p.dout) yrow[o + j] = __float2bfloat16_rn(v[j]);
                    }
                }
            }
            tc_fence_before();
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&tempty[buf])) : "memory");
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
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
    if (threadIdx.x == 0) stamp_record(p.stamps, p.stamp_cap, t_start, STAMP_PREFILL);
}

}  // namespace

cudaError_t prefill_init() {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, prefill_gemm_kernel);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - (int)fa.sharedSizeBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_gemm_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    return e;
}

cudaError_t launch_prefill(const TcForwardArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                           const CUtensorMap& tmV, int num_sms, bool after_shrink, cudaStream_t st) {
    const PoolDims& d = a.dims;
    PrefillParams p{};
    p.chunks = a.ws.chunks;
    p.tmask = a.ws.tmask;
    p.Y = (__nv_bfloat16*)a.Y;
    p.status = a.ws.status;
    p.T = a.T;
    p.dout = d.dout;
    p.kb_total = (d.din + PK - 1) / PK;
    p.m_tiles = (a.T + PM - 1) / PM;
    p.n_tiles = (d.dout + PN - 1) / PN;
    p.n_chunks = a.lora ? a.n_chunks : 0;
    p.max_chunks = d.max_chunks;
    p.ext_steps = after_shrink ? (p.n_chunks + EXT_SUB - 1) / EXT_SUB : 0;
    p.vec_store = (d.dout % 8 == 0) ? 1 : 0;
    p.pdl = after_shrink ? 1 : 0;
    {
        const size_t per_tile = (size_t)PM * d.din * 2;
        size_t g = GROUP_X_BYTES / (per_tile > 0 ? per_tile : 1);
        g = g < (size_t)GROUP_MIN ? (size_t)GROUP_MIN : g;
        p.group_m = (int)(g < (size_t)p.m_tiles ? g : (size_t)p.m_tiles);
        if (p.group_m < 1) p.group_m = 1;
    }
    p.stamps = a.stamps;
    p.up_rows = a.maps.up_rows;
    p.stamp_cap = a.stamp_cap;
    const int total = p.m_tiles * p.n_tiles;
    const int grid = total < num_sms ? total : num_sms;
    const size_t smem = 1024 + (size_t)PSTAGES * PSTAGE + (2 * PSTAGES + 5) * 8 + PSTAGES * 4 + 16;
    return launch_k(prefill_gemm_kernel, dim3(grid), dim3(P_THREADS), smem, st, after_shrink, 1, tmX,
                    tmW, tmV, a.maps.upw256, p);
}

}  // namespace mlora
