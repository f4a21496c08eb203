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
constexpr int G_TOK = 2;                   // rows of the chunk's adapter per pass over its Down rows
constexpr int G_U = 4;                     // 16-byte words of a row per lane in flight at once
constexpr int G_MAX_T = G_THREADS;         // decode batches only: one row id per thread

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
    int prefetch;                  // L2 prefetch of the chunk's Down rows before the wait
    unsigned long long* stamps;    // profiling records (NULL = off)
    int stamp_cap;
};

// sum over the 8 bf16 pairs of two 16-byte words, added to acc (fp32 FMAs)
__device__ __forceinline__ float dot8(const uint4 a, const uint4 b, float acc) {
    const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc = fmaf(__uint_as_float(ua[i] << 16), __uint_as_float(ub[i] << 16), acc);
        acc = fmaf(__uint_as_float(ua[i] & 0xFFFF0000u), __uint_as_float(ub[i] & 0xFFFF0000u), acc);
    }
    return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    return v;
}

__global__ void __launch_bounds__(G_THREADS, 1) shrink_gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(16) uint8_t smem[];   // the segment builder's scratch
    __shared__ int rows_s[G_MAX_T];          // the chunk's rows, in row order
    __shared__ int pos_s[G_MAX_T];           // row -> its index in rows_s, or -1
    __shared__ float vals_s[G_MAX_T][CHUNK];  // Down_chunk x per row of rows_s
    __shared__ int warp_n[G_WARPS];
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

    // rows of the chunk's slot, in row order: one row id per thread, one round trip
    const int t = threadIdx.x;
    const bool mine = t < p.T && p.row_adapter[t] == cr.slot;
    const unsigned b = __ballot_sync(0xffffffffu, mine);
    if (lane == 0) warp_n[warp] = __popc(b);
    __syncthreads();
    int off = 0, n = 0;
#pragma unroll
    for (int w = 0; w < G_WARPS; ++w) {
        off += w < warp ? warp_n[w] : 0;
        n += warp_n[w];
    }
    if (t < p.T) {
        const int k = mine ? off + __popc(b & seg::lanemask_lt()) : -1;
        pos_s[t] = k;
        if (mine) rows_s[k] = t;
    }
    __syncthreads();
    if (n == 0) {
        if (threadIdx.x == 0) stamp_record(p.stamps, p.stamp_cap, t_start, STAMP_SHRINK);
        return;
    }

    // warp w owns rank rows w and w + 8 of the chunk; lane l the 16-byte words
    // l, l + 32, ... of a row; X rows come from L2 (written by the kernel before)
    const int r0 = warp, r1 = warp + G_WARPS;
    const bool has0 = r0 < cr.kval, has1 = r1 < cr.kval;
    const uint4* d0p = reinterpret_cast<const uint4*>(p.down + (size_t)(cr.unit + (has0 ? r0 : 0)) * din);
    const uint4* d1p = reinterpret_cast<const uint4*>(p.down + (size_t)(cr.unit + (has1 ? r1 : 0)) * din);
    const int words = din / 8;
    for (int g0 = 0; g0 < n; g0 += G_TOK) {
        const bool two = g0 + 1 < n;
        // (rows past the chunk's valid ones read row 0 and a missing second row reads the
        // first: the loads need no predicate, and the Vt write drops those values)
        const uint4* xa = reinterpret_cast<const uint4*>(p.X + (size_t)rows_s[g0] * din);
        const uint4* xb = reinterpret_cast<const uint4*>(p.X + (size_t)rows_s[two ? g0 + 1 : g0] * din);
        float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
        // G_U words per lane in flight at once: every load of a block is issued before
        // any of them is used
        int k0 = lane;
        for (; k0 + 32 * (G_U - 1) < words; k0 += 32 * G_U) {
            uint4 w0[G_U], w1[G_U], x0[G_U], x1[G_U];
#pragma unroll
            for (int u = 0; u < G_U; ++u) {
                w0[u] = __ldg(d0p + k0 + 32 * u);
                w1[u] = __ldg(d1p + k0 + 32 * u);
                x0[u] = __ldcg(xa + k0 + 32 * u);
                x1[u] = __ldcg(xb + k0 + 32 * u);
            }
#pragma unroll
            for (int u = 0; u < G_U; ++u) {
                a00 = dot8(w0[u], x0[u], a00);
                a10 = dot8(w1[u], x0[u], a10);
                a01 = dot8(w0[u], x1[u], a01);
                a11 = dot8(w1[u], x1[u], a11);
            }
        }
        for (; k0 < words; k0 += 32) {
            const uint4 w0 = __ldg(d0p + k0), w1 = __ldg(d1p + k0);
            const uint4 x0 = __ldcg(xa + k0), x1 = __ldcg(xb + k0);
            a00 = dot8(w0, x0, a00);
            a10 = dot8(w1, x0, a10);
            a01 = dot8(w0, x1, a01);
            a11 = dot8(w1, x1, a11);
        }
        a00 = warp_sum(a00);
        a10 = warp_sum(a10);
        a01 = warp_sum(a01);
        a11 = warp_sum(a11);
        if (lane == 0) {
            vals_s[g0][r0] = a00;
            vals_s[g0][r1] = a10;
            if (two) {
                vals_s[g0 + 1][r0] = a01;
                vals_s[g0 + 1][r1] = a11;
            }
        }
    }
    __syncthreads();

    // Vt[c][t][0..15] for every row of the batch, 32 bytes each: the scaled values
    // for the chunk's own rows (zero past the chunk's valid columns), zero elsewhere
    if (t < p.T) {
        const int k = pos_s[t];
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float lo = 0.f, hi = 0.f;
            if (k >= 0) {
                lo = 2 * e < cr.kval ? cr.scale * vals_s[k][2 * e] : 0.f;
                hi = 2 * e + 1 < cr.kval ? cr.scale * vals_s[k][2 * e + 1] : 0.f;
            }
            __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
            w[e] = *reinterpret_cast<uint32_t*>(&h);
        }
        // Vt [chunk][block of 8 rank columns][tcap][8]
        __nv_bfloat16* dst = p.vt + ((size_t)c * 2 * p.tcap + t) * 8;
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(dst + (size_t)p.tcap * 8) = make_uint4(w[4], w[5], w[6], w[7]);
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
    p.prefetch = prefetch ? 1 : 0;
    p.stamps = a.stamps;
    p.stamp_cap = a.stamp_cap;
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, shrink_gemv_kernel);
    if (e != cudaSuccess) return e;
    // the builder CTA's scratch is the only dynamic shared memory: as many row ranges
    // as fit a small budget, more memory only if not even one does
    SegPlan sp = seg_plan(d.S, G_WARPS, 16 * 1024 / 4, a.T);
    if (sp.P < 1) sp = seg_plan(d.S, G_WARPS, (max_dyn_smem_gemv() - (int)fa.sharedSizeBytes) / 4, a.T);
    if (sp.P < 1) return cudaErrorInvalidConfiguration;
    p.seg_P = sp.P;
    p.seg_stage_rows = sp.stage_rows ? 1 : 0;
    return launch_k(shrink_gemv_kernel, dim3(a.n_chunks + 1), dim3(G_THREADS), (size_t)sp.ints * 4, st, true, 1, p);
}

}  // namespace mlora
