// Tensor-core path of the bf16 forward: tcgen05 MMA with TMEM accumulators, TMA
// loads into 128B/32B-swizzled shared memory, warp-specialised pipeline.
//
// Decode-shaped batches (T <= 256) use one kernel, "swap-AB": the weight is the M
// operand (128 output features per tile) and the tokens are the N operand
// (N = T rounded up to 16), so W streams through the tensor cores exactly once
// however few rows the batch has.  The K loop of every tile is the din columns of
// W followed by a K-extension over the touched adapters (ai-infra-kb "M031" §02:
// each row adds scale_a Up_a (Down_a x)):
//
//     Y^T[o, t] = sum_i W[o, i] X[t, i]  +  sum_c Up_{a(c)}[o, col(c) + j] Vt[c][t][j]
//
// where chunk c holds 16 rank columns of one touched adapter and Vt[c][t][:] is
// scale_a Down_a x_t for rows t of that adapter and zero for every other row.
// The delta therefore lands in the same fp32 accumulator as the base product,
// on the row's own column, and the output is rounded once.  Up is read from the
// adapter arena once per output tile, through per-slot TMA descriptors whose
// out-of-range columns read as zero (ranks that are not a multiple of 16).
//
// Work split: a grid of (output tile, K split).  Split s takes a contiguous
// share of the din steps and of the K-extension steps of its tile.  Each split
// writes an fp32 partial tile; the last split to arrive (atomic counter, no
// waiting) adds all partials in split order and writes bf16 Y, so the result
// does not depend on arrival order.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

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

bool encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

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
constexpr int BM = 128;            // output features per tile (MMA M)
constexpr int BK = 64;             // din columns per pipeline step (128 bytes of bf16)
constexpr int EXT_SUB = 4;         // K-extension chunks per pipeline step
constexpr int A_BYTES = BM * BK * 2;            // 16 KiB: W tile, or 4 Up chunk tiles
constexpr int NUM_THREADS = 192;   // warp 0 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr int MAX_N = 256;

__host__ __device__ constexpr int b_bytes(int n) { return n * BK * 2; }
__host__ __device__ constexpr int stage_bytes(int n) { return A_BYTES + b_bytes(n); }

struct DecodeParams {
    const CUtensorMap* up_maps;   // per-slot Up descriptors (global memory)
    const int32_t* chunk_slot;
    const int32_t* chunk_col;
    const int32_t* meta;          // meta[1] = number of K-extension chunks
    __nv_bfloat16* Y;
    float* partials;
    int32_t* tile_ctr;
    uint32_t* status;
    int T, dout, N, kb_total, ext_units, splits, stages;
};

// ---------------------------------------------------------------- decode kernel
__global__ void __launch_bounds__(NUM_THREADS, 1)
decode_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmV, DecodeParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int NS = p.stages;
    const int SB = stage_bytes(p.N);
    uint64_t* full = (uint64_t*)(smem + (size_t)NS * SB);
    uint64_t* empty = full + NS;
    uint64_t* acc_full = empty + NS;
    int* stage_kind = (int*)(acc_full + 1);          // -1 = din step, else number of valid chunks
    uint32_t* tmem_slot = (uint32_t*)(stage_kind + NS);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    int* flags = (int*)(tmem_slot + 2);              // [0] issued-any, [1] last-arrival

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, split = blockIdx.y;
    const int kb0 = (int)((long long)split * p.kb_total / p.splits);
    const int kb1 = (int)((long long)(split + 1) * p.kb_total / p.splits);
    const int eu0 = (int)((long long)split * p.ext_units / p.splits);
    const int eu1 = (int)((long long)(split + 1) * p.ext_units / p.splits);
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
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

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
            if (kb < kb1) {
                stage_kind[s] = -1;
                mbar_expect_tx(&full[s], (uint32_t)SB);
                tma_2d(a, &tmW, &full[s], kb * BK, tile * BM);
                tma_2d(b, &tmX, &full[s], kb * BK, 0);
            } else {
                if (n_chunks < 0) n_chunks = p.meta[1];
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
                    for (int j = 0; j < nv; ++j) {
                        const CUtensorMap* um = p.up_maps + p.chunk_slot[c0 + j];
                        tensormap_acquire(um);
                        tma_2d(a + j * (BM * 32), um, &full[s], p.chunk_col[c0 + j], tile * BM);
                    }
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
                for (int j = 0; j < kind; ++j) {
                    mma_bf16(tmem, sdesc(a + j * (BM * 32), 256, SW32), sdesc(b + j * (p.N * 32), 256, SW32), idesc,
                             acc);
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
        // ---------------- epilogue: TMEM -> partial tile or bf16 Y
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;          // row of the tile = output feature
        const int o = tile * BM + row;
        const bool ok = mbar_wait(acc_full, 0, abort_flag, p.status);
        tc_fence_after();
        const bool have = ok && flags[0] != 0;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
        const int T = p.T;
        if (p.splits == 1) {
            for (int t0 = 0; t0 < T; t0 += 16) {
                float v[16];
                if (have) tmem_ld16(tbase + t0, v);
                else
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                if (o < p.dout)
                    for (int j = 0; j < 16 && t0 + j < T; ++j)
                        p.Y[(size_t)(t0 + j) * p.dout + o] = __float2bfloat16_rn(v[j]);
            }
        } else {
            float* mine = p.partials + ((size_t)(tile * p.splits + split) * p.N) * BM;
            for (int t0 = 0; t0 < T; t0 += 16) {
                float v[16];
                if (have) tmem_ld16(tbase + t0, v);
                else
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                for (int j = 0; j < 16 && t0 + j < T; ++j) mine[(size_t)(t0 + j) * BM + row] = v[j];
            }
            __threadfence();
            epi_bar();
            if (threadIdx.x == 64) {
                const int prev = atomicAdd(&p.tile_ctr[tile], 1);
                const int last = prev == p.splits - 1;
                if (last) {
                    p.tile_ctr[tile] = 0;
                    __threadfence();
                }
                flags[1] = last;
            }
            epi_bar();
            if (flags[1]) {
                const float* base = p.partials + (size_t)tile * p.splits * p.N * BM;
                for (int t0 = 0; t0 < T; t0 += 16) {
                    float v[16];
                    if (have) tmem_ld16(tbase + t0, v);
                    else
                        for (int j = 0; j < 16; ++j) v[j] = 0.f;
                    for (int j = 0; j < 16 && t0 + j < T; ++j) {
                        float sum = 0.f;
                        for (int sp = 0; sp < p.splits; ++sp)
                            sum += (sp == split) ? v[j] : __ldcg(base + ((size_t)sp * p.N + t0 + j) * BM + row);
                        if (o < p.dout) p.Y[(size_t)(t0 + j) * p.dout + o] = __float2bfloat16_rn(sum);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
    }
}

// ---------------------------------------------------------------- shrink into chunks
// Vt[c][t][j] = bf16(scale_a * sum_i Down_a[col(c) + j, i] x_t[i]) if row t belongs to
// the chunk's adapter a and col(c) + j < rank_a, else 0.  One warp per (chunk, row).
constexpr int SHRINK_ROWS = 32;   // rows per block (8 warps x 4 rows)

__global__ void __launch_bounds__(256)
shrink_chunks_kernel(const __nv_bfloat16* __restrict__ X, const int32_t* __restrict__ row_adapter,
                     const SlotRec* __restrict__ slots, const __nv_bfloat16* __restrict__ arena_down,
                     const int32_t* __restrict__ chunk_slot, const int32_t* __restrict__ chunk_col,
                     const int32_t* __restrict__ meta, __nv_bfloat16* __restrict__ vt, int T, int din, int S,
                     int tcap) {
    const int c = blockIdx.x;
    if (c >= meta[1]) return;
    const int slot = chunk_slot[c], col0 = chunk_col[c];
    const SlotRec rec = slots[slot];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kmax = min(CHUNK, rec.rank - col0);
    const __nv_bfloat16* down = arena_down + ((size_t)rec.unit + col0) * din;
    for (int r = warp; r < SHRINK_ROWS; r += 8) {
        const int t = blockIdx.y * SHRINK_ROWS + r;
        if (t >= T) break;
        const int a = row_adapter[t];
        float acc[CHUNK];
#pragma unroll
        for (int j = 0; j < CHUNK; ++j) acc[j] = 0.f;
        if (a == slot) {
            const __nv_bfloat16* x = X + (size_t)t * din;
            for (int i = lane * 8; i < din; i += 32 * 8) {
                const uint4 xv = *reinterpret_cast<const uint4*>(x + i);
                const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xv);
                float xf[8];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float2 f = __bfloat1622float2(x2[h]);
                    xf[2 * h] = f.x;
                    xf[2 * h + 1] = f.y;
                }
#pragma unroll
                for (int j = 0; j < CHUNK; ++j) {
                    if (j < kmax) {
                        const uint4 dv = *reinterpret_cast<const uint4*>(down + (size_t)j * din + i);
                        const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const float2 f = __bfloat1622float2(d2[h]);
                            acc[j] = fmaf(f.x, xf[2 * h], acc[j]);
                            acc[j] = fmaf(f.y, xf[2 * h + 1], acc[j]);
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < CHUNK; ++j)
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], d);
        }
        // lane j < 16 writes element j of the row's 32-byte chunk entry
        if (lane < CHUNK) {
            float v = 0.f;
#pragma unroll
            for (int j = 0; j < CHUNK; ++j)
                if (j == lane) v = acc[j];
            vt[((size_t)c * tcap + t) * CHUNK + lane] = __float2bfloat16_rn(a == slot ? rec.scale * v : 0.f);
        }
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

static int decode_splits(int tiles, int kb_total, int ext_units) {
    const int slots = 2 * sm_count();
    int s = slots / (tiles > 0 ? tiles : 1);
    if (s < 1) s = 1;
    if (s > 16) s = 16;
    if (s > kb_total) s = kb_total;
    (void)ext_units;
    return s;
}

static int decode_stages(int N) {
    int ns = (100 * 1024) / stage_bytes(N);
    if (ns < 2) ns = 2;
    if (ns > 8) ns = 8;
    return ns;
}

cudaError_t tc_init() {
    // the cap on dynamic shared memory is raised once, outside any stream capture
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, decode_gemm_kernel);
    // static shared memory counts against the same per-block limit
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - (int)fa.sharedSizeBytes);
    if (e == cudaSuccess) e = prefill_init();
    return e;
}

TcWorkspaceNeeds tc_workspace_needs(bool bf16, const PoolDims& d) {
    TcWorkspaceNeeds n{};
    n.need_v32 = !bf16;   // fp32 pools use the FMA path
    if (bf16) {
        const int tiles = (d.dout + BM - 1) / BM;
        const int ncap = d.max_tokens < MAX_N ? (d.max_tokens + 15) / 16 * 16 : MAX_N;
        const int kb_total = (d.din + BK - 1) / BK;
        const int splits = decode_splits(tiles, kb_total, 0);
        n.partial_bytes = (size_t)tiles * splits * ncap * BM * sizeof(float);
        n.counter_bytes = (size_t)tiles * sizeof(int32_t);
    }
    return n;
}

bool tc_encode_up_map(CUtensorMap* map, void* up_block, int rpad, int dout) {
    cuuint64_t dims[2] = {(cuuint64_t)rpad, (cuuint64_t)dout};
    cuuint64_t strides[1] = {(cuuint64_t)rpad * 2};
    cuuint32_t box[2] = {16, (cuuint32_t)BM};
    return encode(map, up_block, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_32B);
}

bool tc_supported(const PoolDims& d, int T) {
    (void)d;
    return T >= 1;
}

cudaError_t tc_forward(const TcForwardArgs& a, cudaStream_t st) {
    const PoolDims& d = a.dims;
    const int T = a.T;
    const bool decode = T <= MAX_N;
    const int N = decode ? (T + 15) / 16 * 16 : 128;     // token rows per tile
    const int tiles = (d.dout + BM - 1) / BM;
    const int kb_total = (d.din + BK - 1) / BK;
    const int ext_chunks = a.lora ? a.ext_chunk_cap : 0;
    const int ext_units = (ext_chunks + EXT_SUB - 1) / EXT_SUB;

    CUtensorMap tmW, tmX, tmV;
    {
        cuuint64_t dims[2] = {(cuuint64_t)d.din, (cuuint64_t)d.dout};
        cuuint64_t strides[1] = {(cuuint64_t)d.din * 2};
        cuuint32_t box[2] = {BK, decode ? (cuuint32_t)BM : 256u};
        if (!encode(&tmW, a.W, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)d.din, (cuuint64_t)T};
        cuuint64_t strides[1] = {(cuuint64_t)d.din * 2};
        cuuint32_t box[2] = {BK, (cuuint32_t)N};
        if (!encode(&tmX, a.X, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[3] = {(cuuint64_t)CHUNK, (cuuint64_t)d.tcap, (cuuint64_t)d.max_chunks};
        cuuint64_t strides[2] = {(cuuint64_t)CHUNK * 2, (cuuint64_t)d.tcap * CHUNK * 2};
        cuuint32_t box[3] = {CHUNK, (cuuint32_t)N, EXT_SUB};
        if (!encode(&tmV, a.ws.vt, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_32B)) return cudaErrorInvalidValue;
    }

    cudaError_t e;
    if (a.lora && ext_chunks > 0) {
        dim3 grid(ext_chunks, (T + SHRINK_ROWS - 1) / SHRINK_ROWS);
        shrink_chunks_kernel<<<grid, 256, 0, st>>>(
            (const __nv_bfloat16*)a.X, a.row_adapter, a.slots, (const __nv_bfloat16*)a.arena_down,
            a.ws.chunk_slot, a.ws.chunk_col, a.ws.meta, (__nv_bfloat16*)a.ws.vt, T, d.din, d.S, d.tcap);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }

    if (!decode) {
        if (a.ev_start && (e = record_profile(a.ev_start, st)) != cudaSuccess) return e;
        if ((e = launch_prefill(a, tmX, tmW, tmV, sm_count(), st)) != cudaSuccess) return e;
        if (a.ev_stop && (e = record_profile(a.ev_stop, st)) != cudaSuccess) return e;
        return cudaSuccess;
    }

    DecodeParams p{};
    p.up_maps = a.up_maps;
    p.chunk_slot = a.ws.chunk_slot;
    p.chunk_col = a.ws.chunk_col;
    p.meta = a.ws.meta;
    p.Y = (__nv_bfloat16*)a.Y;
    p.partials = a.ws.partials;
    p.tile_ctr = a.ws.tile_ctr;
    p.status = a.ws.status;
    p.T = T;
    p.dout = d.dout;
    p.N = N;
    p.kb_total = kb_total;
    p.ext_units = ext_units;
    p.splits = decode_splits(tiles, kb_total, ext_units);
    p.stages = decode_stages(N);
    const size_t smem = 1024 + (size_t)p.stages * stage_bytes(N) + (size_t)(2 * p.stages + 1) * 8 +
                        (size_t)p.stages * 4 + 16;
    dim3 grid(tiles, p.splits);
    if (a.ev_start && (e = record_profile(a.ev_start, st)) != cudaSuccess) return e;
    decode_gemm_kernel<<<grid, NUM_THREADS, smem, st>>>(tmW, tmX, tmV, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.ev_stop && (e = record_profile(a.ev_stop, st)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace mlora
