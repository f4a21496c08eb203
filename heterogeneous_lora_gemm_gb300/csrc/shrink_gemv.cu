// Shrink for decode batches spread over many adapters with a few rows each
// (ai-infra-kb "M031" §02: V = scale_a Down_a x for the rows of adapter a; wiblog
// "vLLM LoRA adapter batch scheduling", section on batch fragmentation, whose
// extreme case is one row per adapter).
//
// One CTA per K-extension chunk of the pool (16 rank rows of one loaded adapter):
// it finds the rows of the batch whose slot is the chunk's, computes
// scale * Down_chunk x for each of them over the whole din on the CUDA cores -- no
// K split, so no partial sums meet between CTAs -- and writes the chunk's Vt for
// every row of the batch: bf16(scale * Down_chunk x_t) for its own rows, zero for
// the others (the projection's K-extension multiplies Up by Vt over all rows).  A
// chunk that no row uses writes nothing; the projection skips its slot.  One more
// CTA runs the segment builder (seg.cuh).
//
// With few rows per adapter, the tensor-core shrink spends most of its work and
// its split-K reductions on rows that the mask then drops; here each Down row is
// read once from HBM and multiplied only by the rows that use it.
//
// Launched first in the forward with programmatic dependent launch: the chunk
// record and (optionally) an L2 prefetch of the chunk's Down rows -- pool data --
// go out before the wait for the kernel before, which may produce X and the row
// map and may still read Vt.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "seg.cuh"
#include "tc.h"
#include "tc_ptx.cuh"

namespace mlora {

using namespace ptx;

namespace {

constexpr int G_THREADS = 256;
constexpr int G_WARPS = G_THREADS / 32;
constexpr int G_NT = 8;                    // rows of the chunk's adapter per pass over its Down rows
constexpr int G_XS_BYTES = 64 * 1024;      // shared memory for the X rows of one pass
constexpr int G_MAX_T = 256;               // decode batches only

struct GemvParams {
    const __nv_bfloat16* X;        // [T x din]
    const int32_t* row_adapter;    // [T]
    const ChunkRec* chunks;        // chunk table of the loaded slots
    const __nv_bfloat16* down;     // arena Down half [units x din]
    __nv_bfloat16* vt;             // [max_chunks][tcap][16]
    const SlotRec* slots;          // segment builder
    Workspace ws;
    int T, din, n_chunks, tcap, S, max_chunks;
    int seg_P, seg_stage_rows;
    int nt;                        // rows per pass (X rows staged in shared memory)
    int prefetch;                  // L2 prefetch of the chunk's Down rows before the wait
    unsigned long long* stamps;    // profiling records (NULL = off)
    int stamp_cap;
};

// 8 bf16 of a 16-byte word, as floats (exact)
__device__ __forceinline__ void bf16x8(const uint4 w, float* f) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}

__global__ void __launch_bounds__(G_THREADS) shrink_gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int rows_s[G_MAX_T];          // the chunk's rows, in row order
    __shared__ int pos_s[G_MAX_T];           // row -> its index in rows_s, or -1
    __shared__ float vals_s[G_MAX_T][CHUNK];  // scale * Down_chunk x per row of rows_s
    __shared__ int n_rows_s;
    const unsigned long long t_start = (p.stamps && threadIdx.x == 0) ? gtimer() : 0ull;
    const int c = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (c == p.n_chunks) {
        // the segment builder: slot table and arguments staged before the wait, only
        // the row map read after it
        const seg::Scratch sc = seg::carve(reinterpret_cast<int*>(smem), p.S, p.seg_P, p.seg_stage_rows != 0);
        seg::stage(p.slots, p.S, p.ws, p.row_adapter, p.T, p.max_chunks, sc);
        pdl_wait();
        pdl_trigger();
        seg::build(p.S, p.seg_P, sc);
        if (threadIdx.x == 0) stamp_record(p.stamps, p.stamp_cap, t_start, STAMP_SHRINK);
        return;
    }

    const ChunkRec cr = p.chunks[c];
    const int din = p.din;
    if (p.prefetch && threadIdx.x < cr.kval) {
        const __nv_bfloat16* row = p.down + (size_t)(cr.unit + threadIdx.x) * din;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row), "r"((uint32_t)din * 2u) : "memory");
    }
    pdl_wait();
    pdl_trigger();

    // rows of the chunk's slot, in row order (warp 0), and the inverse map
    for (int t = threadIdx.x; t < p.T; t += G_THREADS) pos_s[t] = -1;
    __syncthreads();
    if (warp == 0) {
        int n = 0;
        for (int base = 0; base < p.T; base += 32) {
            const int t = base + lane;
            const bool mine = t < p.T && p.row_adapter[t] == cr.slot;
            const unsigned b = __ballot_sync(0xffffffffu, mine);
            if (mine) {
                const int k = n + __popc(b & seg::lanemask_lt());
                rows_s[k] = t;
                pos_s[t] = k;
            }
            n += __popc(b);
        }
        if (lane == 0) n_rows_s = n;
    }
    __syncthreads();
    const int n = n_rows_s;
    if (n == 0) {
        if (threadIdx.x == 0) stamp_record(p.stamps, p.stamp_cap, t_start, STAMP_SHRINK);
        return;
    }

    // warp w owns rank rows w and w + 8 of the chunk; lane l covers din columns
    // l*8 .. l*8+7 of every 256
    __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem);
    const int r0 = warp, r1 = warp + G_WARPS;
    const bool has0 = r0 < cr.kval, has1 = r1 < cr.kval;
    const uint4* d0p = reinterpret_cast<const uint4*>(p.down + (size_t)(cr.unit + (has0 ? r0 : 0)) * din);
    const uint4* d1p = reinterpret_cast<const uint4*>(p.down + (size_t)(cr.unit + (has1 ? r1 : 0)) * din);
    const int words = din / 8;   // 16-byte words per row
    for (int g0 = 0; g0 < n; g0 += p.nt) {
        const int ng = min(p.nt, n - g0);
        for (int i = threadIdx.x; i < ng * words; i += G_THREADS) {
            const int j = i / words, k = i - j * words;
            reinterpret_cast<uint4*>(xs)[i] = reinterpret_cast<const uint4*>(p.X + (size_t)rows_s[g0 + j] * din)[k];
        }
        __syncthreads();
        float acc0[G_NT], acc1[G_NT];
#pragma unroll
        for (int j = 0; j < G_NT; ++j) acc0[j] = acc1[j] = 0.f;
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 4
        for (int k = lane; k < words; k += 32) {
            float w0[8], w1[8];
            bf16x8(has0 ? __ldg(d0p + k) : zero, w0);
            bf16x8(has1 ? __ldg(d1p + k) : zero, w1);
#pragma unroll
            for (int j = 0; j < G_NT; ++j) {
                if (j < ng) {
                    float x[8];
                    bf16x8(reinterpret_cast<const uint4*>(xs)[j * words + k], x);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        acc0[j] = fmaf(w0[e], x[e], acc0[j]);
                        acc1[j] = fmaf(w1[e], x[e], acc1[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < G_NT; ++j) {
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                acc0[j] += __shfl_xor_sync(0xffffffffu, acc0[j], d);
                acc1[j] += __shfl_xor_sync(0xffffffffu, acc1[j], d);
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < G_NT; ++j)
                if (j < ng) {
                    vals_s[g0 + j][r0] = acc0[j];
                    vals_s[g0 + j][r1] = acc1[j];
                }
        }
        __syncthreads();   // the X rows of the next pass overwrite xs
    }

    // Vt[c][t][0..15] for every row of the batch, 32 bytes each: the scaled values
    // for the chunk's own rows (zero past the chunk's valid columns), zero elsewhere
    for (int t = threadIdx.x; t < p.T; t += G_THREADS) {
        const int k = pos_s[t];
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float a = 0.f, b = 0.f;
            if (k >= 0) {
                a = 2 * e < cr.kval ? cr.scale * vals_s[k][2 * e] : 0.f;
                b = 2 * e + 1 < cr.kval ? cr.scale * vals_s[k][2 * e + 1] : 0.f;
            }
            __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
            w[e] = *reinterpret_cast<uint32_t*>(&h);
        }
        uint4* dst = reinterpret_cast<uint4*>(p.vt + ((size_t)c * p.tcap + t) * CHUNK);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    if (threadIdx.x == 0) stamp_record(p.stamps, p.stamp_cap, t_start, STAMP_SHRINK);
}

int max_dyn_smem_gemv() {
    static int v = 0;
    if (!v) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || v <= 0)
            v = 227 * 1024;
    }
    return v;
}

}  // namespace

cudaError_t gemv_init() {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, shrink_gemv_kernel);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(shrink_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 max_dyn_smem_gemv() - (int)fa.sharedSizeBytes);
    return e;
}

bool gemv_shrink_fits(const PoolDims& d, int T) {
    return T >= 1 && T <= G_MAX_T && d.din % 8 == 0;
}

cudaError_t launch_shrink_gemv(const TcForwardArgs& a, bool prefetch, cudaStream_t st) {
    const PoolDims& d = a.dims;
    GemvParams p{};
    p.X = (const __nv_bfloat16*)a.X;
    p.row_adapter = a.row_adapter;
    p.chunks = a.ws.chunks;
    p.down = (const __nv_bfloat16*)a.arena_down;
    p.vt = (__nv_bfloat16*)a.ws.vt;
    p.slots = a.slots;
    p.ws = a.ws;
    p.T = a.T;
    p.din = d.din;
    p.n_chunks = a.n_chunks;
    p.tcap = d.tcap;
    p.S = d.S;
    p.max_chunks = d.max_chunks;
    p.nt = G_XS_BYTES / (d.din * 2);
    p.nt = p.nt < 1 ? 1 : (p.nt > G_NT ? G_NT : p.nt);
    p.prefetch = prefetch ? 1 : 0;
    p.stamps = a.stamps;
    p.stamp_cap = a.stamp_cap;
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, shrink_gemv_kernel);
    if (e != cudaSuccess) return e;
    const int avail_ints = (max_dyn_smem_gemv() - (int)fa.sharedSizeBytes) / 4;
    const size_t xs_bytes = (size_t)p.nt * d.din * 2;
    // the builder CTA uses the same dynamic shared memory: as many row ranges as fit
    SegPlan sp = seg_plan(d.S, G_WARPS, (int)(xs_bytes / 4), a.T);
    if (sp.P < 1) sp = seg_plan(d.S, G_WARPS, avail_ints, a.T);
    if (sp.P < 1) return cudaErrorInvalidConfiguration;
    p.seg_P = sp.P;
    p.seg_stage_rows = sp.stage_rows ? 1 : 0;
    const size_t smem = xs_bytes > (size_t)sp.ints * 4 ? xs_bytes : (size_t)sp.ints * 4;
    return launch_k(shrink_gemv_kernel, dim3(a.n_chunks + 1), dim3(G_THREADS), smem, st, true, 1, p);
}

}  // namespace mlora
