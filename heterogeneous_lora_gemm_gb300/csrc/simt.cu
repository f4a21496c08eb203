// CUDA-core (FMA) kernels of the multi-LoRA layer.
//
// These serve the fp32 pools (no TF32 anywhere: the fp32 path keeps full fp32
// products and sums) and the bf16 shapes the tensor-core kernels do not take.
//   shrink      v32[t, k] = scale_a * sum_i Down_a[k, i] x_t[i]       (rows of the segments)
//   base_expand Y[t, o]  = sum_i W[o, i] x_t[i] + sum_k Up_a[o, k] v32[t, k]
//   merge       W[o, i] += sign * scale * sum_k Up[o, k] Down[k, i]   (sign -1: un-merge)
// (ai-infra-kb "M031" tutorial §02 and §04.)  The expand reads the row's own
// adapter and writes Y at the row's own index, so the result is in original row
// order by construction.
#include <cuda_bf16.h>

#include "internal.h"

namespace mlora {

namespace {

template <typename E>
__device__ __forceinline__ float to_f32(E v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename E>
__device__ __forceinline__ E from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ bool valid_slot(int a, int S, const SlotRec* slots) {
    return a >= 0 && a < S && slots[a].rank > 0;
}

// One block per segment entry i (grid covers T; entries past n_valid exit).
// Each warp takes rank rows k = warp, warp + nwarps, ... of the row's adapter.
template <typename E>
__global__ void shrink_simt_kernel(const E* __restrict__ X, const SlotRec* __restrict__ slots,
                                   const E* __restrict__ arena_down, Workspace ws, const int32_t* __restrict__ row_adapter,
                                   int din, int max_rank) {
    const int i = blockIdx.x;
    if (i >= ws.meta[0]) return;
    const int t = ws.perm[i];
    const int a = row_adapter[t];
    const SlotRec rec = slots[a];
    const E* x = X + (size_t)t * din;
    const E* down = arena_down + (size_t)rec.unit * din;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int k = warp; k < rec.rank; k += nw) {
        const E* d = down + (size_t)k * din;
        float acc = 0.f;
        for (int c = lane; c < din; c += 32) acc = fmaf(to_f32(d[c]), to_f32(x[c]), acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) ws.v32[(size_t)t * max_rank + k] = rec.scale * acc;
    }
}

// Tiled FMA GEMM: a 64 (rows t) x 64 (outputs o) tile per block, 256 threads,
// 4 x 4 outputs per thread, K in steps of 16 through shared memory.  The
// expand of each output is added to the same fp32 accumulator before the single
// final rounding.
constexpr int BT = 64, BO = 64, BK = 16;

template <typename E>
__global__ void __launch_bounds__(256)
base_expand_simt_kernel(const E* __restrict__ X, const E* __restrict__ W, const int32_t* __restrict__ row_adapter,
                        int T, int din, int dout, E* __restrict__ Y, const SlotRec* __restrict__ slots,
                        const E* __restrict__ arena_up, const float* __restrict__ v32, int S, int max_rank,
                        int with_lora) {
    __shared__ float xs[BK][BT + 1];
    __shared__ float wsm[BK][BO + 1];
    const int t0 = blockIdx.y * BT, o0 = blockIdx.x * BO;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;   // 16 x 16 threads
    float acc[4][4] = {};
    for (int k0 = 0; k0 < din; k0 += BK) {
        for (int idx = threadIdx.x; idx < BK * BT; idx += 256) {
            const int r = idx / BK, c = idx % BK;
            const int t = t0 + r, k = k0 + c;
            xs[c][r] = (t < T && k < din) ? to_f32(X[(size_t)t * din + k]) : 0.f;
            const int o = o0 + r;
            wsm[c][r] = (o < dout && k < din) ? to_f32(W[(size_t)o * din + k]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < BK; ++c) {
            float xv[4], wv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) xv[i] = xs[c][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) wv[j] = wsm[c][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= T) continue;
        int a = with_lora ? row_adapter[t] : -1;
        const bool lora = with_lora && valid_slot(a, S, slots);
        SlotRec rec{};
        if (lora) rec = slots[a];
        const float* v = v32 + (size_t)t * max_rank;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int o = o0 + tx * 4 + j;
            if (o >= dout) continue;
            float y = acc[i][j];
            if (lora)
                for (int k = 0; k < rec.rank; ++k) y = fmaf(to_f32(arena_up[up_index(rec.unit, k, o, dout)]), v[k], y);
            Y[(size_t)t * dout + o] = from_f32<E>(y);
        }
    }
}

// W[o, i] += scale * sum_k Up[o, k] Down[k, i] (M031 §04), fp32 sum, one rounding.
// Merge.  A block owns a tile of MERGE_ROWS rows x MERGE_COLS columns of W; each
// thread owns 8 rows x 8 consecutive columns (one 16-byte vector of a bf16 row).  The
// thread's old W values are loaded first, so that the HBM round trip overlaps the
// adapter loads and the FMAs.  Per chunk of MERGE_KC rank columns, the Down slab
// [k][MERGE_COLS] (fp32) and the Up slab [MERGE_ROWS][k] sit in shared memory: a
// thread reads its 8 Down values of column k once and multiplies them by the 8 Up
// values of its rows (broadcast across the warp).  Sums in fp32, one rounding.
constexpr int MERGE_ROWS = 64, MERGE_COLS = 256, MERGE_KC = 32, MERGE_THREADS = 256;

__device__ __forceinline__ void load8(const __nv_bfloat16* p, bool vec, int n, float* v) {
    if (vec) {
        const uint4 q = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(h[j]);
            v[2 * j] = f.x;
            v[2 * j + 1] = f.y;
        }
    } else {
        for (int j = 0; j < 8; ++j) v[j] = j < n ? __bfloat162float(p[j]) : 0.f;
    }
}
__device__ __forceinline__ void load8(const float* p, bool vec, int n, float* v) {
    if (vec) {
        const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
        v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
    } else {
        for (int j = 0; j < 8; ++j) v[j] = j < n ? p[j] : 0.f;
    }
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, bool vec, int n, const float* v) {
    if (vec) {
        uint4 q;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
        for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
        *reinterpret_cast<uint4*>(p) = q;
    } else {
        for (int j = 0; j < n; ++j) p[j] = __float2bfloat16_rn(v[j]);
    }
}
__device__ __forceinline__ void store8(float* p, bool vec, int n, const float* v) {
    if (vec) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
    } else {
        for (int j = 0; j < n; ++j) p[j] = v[j];
    }
}

template <typename E>
__global__ void __launch_bounds__(MERGE_THREADS, 2)
merge_simt_kernel(E* __restrict__ W, const SlotRec* __restrict__ slots, int slot,
                  const E* __restrict__ arena_down, const E* __restrict__ arena_up, int din, int dout,
                  float sign) {
    __shared__ __align__(16) float down_s[MERGE_KC][MERGE_COLS];
    __shared__ float up_s[MERGE_ROWS][MERGE_KC + 1];
    const SlotRec rec = slots[slot];
    if (rec.rank <= 0) return;
    const int cg = threadIdx.x & 31, rg = threadIdx.x >> 5;   // column group (8 columns), row group (8 rows)
    const int c0 = blockIdx.x * MERGE_COLS, i0 = c0 + cg * 8;
    const int o0 = blockIdx.y * MERGE_ROWS + rg * 8;
    const int ncol = min(8, din - i0);                         // columns of this thread inside W
    // 16-byte vectors need whole, aligned groups of 8 columns
    const bool vec = ncol == 8 && (din % 8) == 0;

    // bf16 rows as whole vectors: the raw 16 bytes of each of the 8 rows, loaded now
    constexpr bool BF16 = sizeof(E) == 2;
    const bool pre = BF16 && vec;
    uint4 w_raw[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
        w_raw[r] = (pre && o0 + r < dout) ? *reinterpret_cast<const uint4*>(W + (size_t)(o0 + r) * din + i0)
                                          : make_uint4(0u, 0u, 0u, 0u);
    float acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[r][j] = 0.f;

    const E* down = arena_down + (size_t)rec.unit * din;
    const bool dvec = (din % 8) == 0;
    for (int k0 = 0; k0 < rec.rank; k0 += MERGE_KC) {
        const int kn = min(MERGE_KC, rec.rank - k0);
        __syncthreads();
        for (int idx = threadIdx.x; idx < kn * (MERGE_COLS / 8); idx += MERGE_THREADS) {
            const int k = idx / (MERGE_COLS / 8), c8 = (idx % (MERGE_COLS / 8)) * 8;
            const int n = min(8, din - (c0 + c8));
            float v[8];
            if (n > 0) load8(down + (size_t)(k0 + k) * din + c0 + c8, dvec && n == 8, n, v);
            else
                for (int j = 0; j < 8; ++j) v[j] = 0.f;
            *reinterpret_cast<float4*>(&down_s[k][c8]) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(&down_s[k][c8 + 4]) = make_float4(v[4], v[5], v[6], v[7]);
        }
        for (int idx = threadIdx.x; idx < MERGE_ROWS * kn; idx += MERGE_THREADS) {
            const int r = idx / kn, k = idx % kn;
            const int o = blockIdx.y * MERGE_ROWS + r;
            up_s[r][k] = o < dout ? to_f32(arena_up[up_index(rec.unit, k0 + k, o, dout)]) : 0.f;
        }
        __syncthreads();
        for (int k = 0; k < kn; ++k) {
            const float4 da = *reinterpret_cast<const float4*>(&down_s[k][cg * 8]);
            const float4 db = *reinterpret_cast<const float4*>(&down_s[k][cg * 8 + 4]);
            const float dv[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float u = up_s[rg * 8 + r][k];
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[r][j] = fmaf(u, dv[j], acc[r][j]);
            }
        }
    }
    if (ncol <= 0) return;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        if (o0 + r >= dout) break;
        E* w = W + (size_t)(o0 + r) * din + i0;
        float old[8];
        if (pre) {
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w_raw[r]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __bfloat1622float2(h[j]);
                old[2 * j] = f.x;
                old[2 * j + 1] = f.y;
            }
        } else {
            load8(w, vec, ncol, old);
        }
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = fmaf(sign * rec.scale, acc[r][j], old[j]);
        store8(w, vec, ncol, v);
    }
}

}  // namespace

cudaError_t launch_shrink_simt(bool bf16, const void* X, const int32_t* row_adapter, int T,
                               const SlotRec* slots, const void* arena_down, const Workspace& ws,
                               const PoolDims& d, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    if (bf16)
        shrink_simt_kernel<__nv_bfloat16><<<T, 128, 0, st>>>(
            (const __nv_bfloat16*)X, slots, (const __nv_bfloat16*)arena_down, ws, row_adapter, d.din, d.max_rank);
    else
        shrink_simt_kernel<float><<<T, 128, 0, st>>>((const float*)X, slots, (const float*)arena_down, ws,
                                                     row_adapter, d.din, d.max_rank);
    return cudaGetLastError();
}

cudaError_t launch_base_expand_simt(bool bf16, const void* X, const void* W,
                                    const int32_t* row_adapter, int T, void* Y,
                                    const SlotRec* slots, const void* arena_up, const Workspace& ws,
                                    const PoolDims& d, bool with_lora, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    dim3 grid((d.dout + BO - 1) / BO, (T + BT - 1) / BT);
    if (bf16)
        base_expand_simt_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            (const __nv_bfloat16*)X, (const __nv_bfloat16*)W, row_adapter, T, d.din, d.dout, (__nv_bfloat16*)Y,
            slots, (const __nv_bfloat16*)arena_up, ws.v32, d.S, d.max_rank, with_lora ? 1 : 0);
    else
        base_expand_simt_kernel<float><<<grid, 256, 0, st>>>((const float*)X, (const float*)W, row_adapter, T,
                                                            d.din, d.dout, (float*)Y, slots, (const float*)arena_up,
                                                            ws.v32, d.S, d.max_rank, with_lora ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_merge_simt(bool bf16, void* W, const SlotRec* slots, int slot,
                              const void* arena_down, const void* arena_up, const PoolDims& d, float sign,
                              cudaStream_t st) {
    const dim3 grid((d.din + MERGE_COLS - 1) / MERGE_COLS, (d.dout + MERGE_ROWS - 1) / MERGE_ROWS);
    if (bf16)
        merge_simt_kernel<__nv_bfloat16><<<grid, MERGE_THREADS, 0, st>>>(
            (__nv_bfloat16*)W, slots, slot, (const __nv_bfloat16*)arena_down, (const __nv_bfloat16*)arena_up, d.din,
            d.dout, sign);
    else
        merge_simt_kernel<float><<<grid, MERGE_THREADS, 0, st>>>((float*)W, slots, slot, (const float*)arena_down,
                                                          (const float*)arena_up, d.din, d.dout, sign);
    return cudaGetLastError();
}

}  // namespace mlora
