// A quantized base weight (ai-infra-kb "M031" tutorial §05): int8 codes with one
// scale per output row, W[o, i] = code[o, i] * row_scale[o] (symmetric).
//
//   dequant_kernel      W = code * row_scale, rounded once to the pool dtype: the
//                       logical matrix that the dynamic LoRA branch runs over
//   merge_quant_kernel  the merge on a quantized base: dequantize, add
//                       scale * Up Down (fp32), and quantize the merged rows again
//                       (new row scale max|w| / 127, codes rounded to nearest even and
//                       clamped to [-127, 127]), in place.  Adding the update to the
//                       codes themselves would mix two numeric spaces (§05).
//
// Both are bandwidth-bound sweeps over W.  The merge here serves fp32 pools and code
// rows that are not whole 16-byte units (bf16 pools otherwise merge on the tensor
// cores, merge_tc.cu).  It runs one CTA per group of rows (each Down value loaded
// serves all of them): the rows are read, updated and held in shared memory (fp32),
// reduced to their max, then written back as codes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace mlora {

namespace {

constexpr int DQ_THREADS = 256;
constexpr int MQ_THREADS = 256;
constexpr int MQ_SMEM_MAX = 200 * 1024;      // merged rows held in shared memory (fp32)

template <typename E>
__device__ __forceinline__ E from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <typename E>
__device__ __forceinline__ float as_f32(E v);
template <>
__device__ __forceinline__ float as_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float as_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// 8 consecutive values as fp32: one 16-byte (bf16) or two 16-byte (fp32) loads when
// `vec` (8 whole, aligned values), else one by one up to n.
__device__ __forceinline__ void load8f(const __nv_bfloat16* p, bool vec, int n, float* v) {
    if (vec) {
        const uint4 raw = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(h[j]);
            v[2 * j] = f.x;
            v[2 * j + 1] = f.y;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = j < n ? __bfloat162float(p[j]) : 0.f;
    }
}
__device__ __forceinline__ void load8f(const float* p, bool vec, int n, float* v) {
    if (vec) {
        const float4 a = *reinterpret_cast<const float4*>(p);
        const float4 b = *reinterpret_cast<const float4*>(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = j < n ? p[j] : 0.f;
    }
}

// A code as a float without a conversion instruction: 2^23 + 128 + c holds c + 128 in
// its low mantissa bits.
__device__ __forceinline__ float code_f32(int8_t c) { return __int_as_float(0x4B000000 + 128 + (int)c) - 8388736.f; }

// Groups of 16 codes of a row (din % 16 == 0: one 16-byte load each), four groups
// per thread and step with their loads issued first; else one code per thread.
template <typename E>
__device__ __forceinline__ void dequant16(const int4 raw, float so, E* dst) {
    const int8_t* c = reinterpret_cast<const int8_t*>(&raw);
    __align__(16) E out[16];
    if constexpr (sizeof(E) == 2) {   // bf16: two values per rounding instruction
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(out);
#pragma unroll
        for (int j = 0; j < 8; ++j) o2[j] = __floats2bfloat162_rn(code_f32(c[2 * j]) * so, code_f32(c[2 * j + 1]) * so);
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) out[j] = from_f32<E>(code_f32(c[j]) * so);
    }
    const int4* src = reinterpret_cast<const int4*>(out);
    int4* d = reinterpret_cast<int4*>(dst);
#pragma unroll
    for (int j = 0; j < (int)(16 * sizeof(E) / 16); ++j) d[j] = src[j];
}

template <typename E>
__global__ void __launch_bounds__(DQ_THREADS)
dequant_kernel(const int8_t* __restrict__ q, const float* __restrict__ s, int dout, int din, E* __restrict__ W) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t first = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if ((din % 16) == 0) {
        const size_t groups = (size_t)dout * (din / 16);
        const uint32_t gpr = (uint32_t)(din / 16);          // groups per row
        const bool narrow = groups <= 0xFFFFFFFFull;        // row of a group by a 32-bit division
        for (size_t g0 = first; g0 < groups; g0 += 4 * stride) {
            int4 raw[4];
            float so[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const size_t g = g0 + u * stride;
                if (g < groups) {
                    raw[u] = *reinterpret_cast<const int4*>(q + g * 16);
                    so[u] = s[narrow ? (size_t)((uint32_t)g / gpr) : g / gpr];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const size_t g = g0 + u * stride;
                if (g < groups) dequant16<E>(raw[u], so[u], W + g * 16);
            }
        }
    } else {
        const size_t n = (size_t)dout * din;
        for (size_t g = first; g < n; g += stride) W[g] = from_f32<E>((float)q[g] * s[g / din]);
    }
}

// CTA per R consecutive output rows.  Each thread owns 8 consecutive columns of a
// 2048-column block and all R rows of them (an R x 8 register tile): the update
// scale * Up[rows, k] Down[k, cols] (fp32, k ascending), plus the restored codes,
// goes to shared memory [R][din]; then each row's max, its new scale, and its codes.
template <typename E, int R>
__global__ void __launch_bounds__(MQ_THREADS)
merge_quant_kernel(int8_t* __restrict__ q, float* __restrict__ s, const SlotRec* __restrict__ slots, int slot,
                   const E* __restrict__ arena_down, const E* __restrict__ arena_up, int din, int dout) {
    extern __shared__ float wsh[];   // [R][din] merged rows, then [R][rank] Up of the rows
    __shared__ float red[MQ_THREADS / 32][R];
    __shared__ float sn_s[R];
    const SlotRec rec = slots[slot];
    const int o0 = blockIdx.x * R;
    const int nr = min(R, dout - o0);
    float* up_s = wsh + (size_t)R * din;
    for (int idx = threadIdx.x; idx < R * rec.rank; idx += MQ_THREADS) {
        const int r = idx / rec.rank, k = idx % rec.rank;
        up_s[idx] = r < nr ? as_f32(arena_up[up_index(rec.unit, k, o0 + r, dout)]) : 0.f;
    }
    __syncthreads();
    const E* down = arena_down + (size_t)rec.unit * din;
    float m[R];
#pragma unroll
    for (int r = 0; r < R; ++r) m[r] = 0.f;
    for (int c0 = 0; c0 < din; c0 += MQ_THREADS * 8) {
        const int i0 = c0 + threadIdx.x * 8;
        if (i0 >= din) continue;
        const int nc = min(8, din - i0);
        const bool vec = nc == 8 && (din % 8) == 0;   // whole, 16-byte aligned groups of 8
        float acc[R][8];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[r][j] = 0.f;
        // four rank steps' Down loads in flight, then their FMAs (k ascending)
        for (int k0 = 0; k0 < rec.rank; k0 += 4) {
            float d[4][8];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                if (k0 + kk < rec.rank) load8f(down + (size_t)(k0 + kk) * din + i0, vec, nc, d[kk]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                if (k0 + kk >= rec.rank) break;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float u = up_s[r * rec.rank + k0 + kk];
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[r][j] = fmaf(u, d[kk][j], acc[r][j]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r >= nr) break;
            const int o = o0 + r;
            const float so = s[o];
            __align__(8) int8_t c8[8];
            if (vec) {
                *reinterpret_cast<uint2*>(c8) = *reinterpret_cast<const uint2*>(q + (size_t)o * din + i0);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) c8[j] = j < nc ? q[(size_t)o * din + i0 + j] : (int8_t)0;
            }
            float w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                w[j] = fmaf(rec.scale, acc[r][j], (float)c8[j] * so);
                if (j < nc) m[r] = fmaxf(m[r], fabsf(w[j]));
            }
            float* dst = wsh + (size_t)r * din + i0;
            if (vec) {
                *reinterpret_cast<float4*>(dst) = make_float4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(w[4], w[5], w[6], w[7]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < nc) dst[j] = w[j];
            }
        }
    }
    // the rows' max: warp shuffle, then across warps
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float v = m[r];
#pragma unroll
        for (int dd = 16; dd > 0; dd >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, dd));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5][r] = v;
    }
    __syncthreads();
    if (threadIdx.x < R) {
        float v = 0.f;
        for (int w = 0; w < MQ_THREADS / 32; ++w) v = fmaxf(v, red[w][threadIdx.x]);
        sn_s[threadIdx.x] = v / 127.f;   // new row scale (0 for an all-zero row: codes 0)
        if (threadIdx.x < nr) s[o0 + threadIdx.x] = sn_s[threadIdx.x];
    }
    __syncthreads();
    // codes: each thread its own 8 columns of each row (as in the first pass)
    for (int r = 0; r < nr; ++r) {
        const float sn = sn_s[r];
        const int o = o0 + r;
        for (int c0 = 0; c0 < din; c0 += MQ_THREADS * 8) {
            const int i0 = c0 + threadIdx.x * 8;
            if (i0 >= din) continue;
            const int nc = min(8, din - i0);
            const bool vec = nc == 8 && (din % 8) == 0;
            const float* src = wsh + (size_t)r * din + i0;
            float w[8];
            if (vec) {
                const float4 a = *reinterpret_cast<const float4*>(src);
                const float4 b = *reinterpret_cast<const float4*>(src + 4);
                w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
                w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) w[j] = j < nc ? src[j] : 0.f;
            }
            __align__(8) int8_t c8[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int c = 0;
                if (j < nc && sn > 0.f) {
                    c = __float2int_rn(w[j] / sn);
                    c = c > 127 ? 127 : (c < -127 ? -127 : c);
                }
                c8[j] = (int8_t)c;
            }
            int8_t* dst = q + (size_t)o * din + i0;
            if (vec) {
                *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(c8);
            } else {
                for (int j = 0; j < nc; ++j) dst[j] = c8[j];
            }
        }
    }
}

int quant_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    }
    return n;
}

}  // namespace

cudaError_t launch_dequant(bool bf16, const int8_t* q, const float* s, int dout, int din, void* W, cudaStream_t st) {
    const size_t groups = (din % 16) == 0 ? (size_t)dout * (din / 16) : (size_t)dout * din;
    size_t blocks = (groups + DQ_THREADS - 1) / DQ_THREADS;
    const size_t cap = (size_t)quant_sms() * 8;   // grid-stride beyond 8 CTAs per SM
    blocks = blocks < cap ? blocks : cap;
    if (blocks == 0) return cudaSuccess;
    if (bf16)
        dequant_kernel<__nv_bfloat16><<<(unsigned)blocks, DQ_THREADS, 0, st>>>(q, s, dout, din, (__nv_bfloat16*)W);
    else
        dequant_kernel<float><<<(unsigned)blocks, DQ_THREADS, 0, st>>>(q, s, dout, din, (float*)W);
    return cudaGetLastError();
}

template <typename E, int R>
cudaError_t launch_merge_quant_r(int8_t* q, float* s, const SlotRec* slots, int slot, const void* arena_down,
                                 const void* arena_up, const PoolDims& d, cudaStream_t st) {
    const size_t smem = sizeof(float) * ((size_t)R * d.din + (size_t)R * d.max_rank);
    cudaError_t e = cudaFuncSetAttribute(merge_quant_kernel<E, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    merge_quant_kernel<E, R><<<(unsigned)((d.dout + R - 1) / R), MQ_THREADS, smem, st>>>(
        q, s, slots, slot, (const E*)arena_down, (const E*)arena_up, d.din, d.dout);
    return cudaGetLastError();
}

template <typename E>
cudaError_t launch_merge_quant_e(int8_t* q, float* s, const SlotRec* slots, int slot, const void* arena_down,
                                 const void* arena_up, const PoolDims& d, cudaStream_t st) {
    // as many rows per CTA (4, 2, 1) as leave the held rows in shared memory
    const size_t per_row = sizeof(float) * ((size_t)d.din + (size_t)d.max_rank);
    if (4 * per_row <= (size_t)MQ_SMEM_MAX) return launch_merge_quant_r<E, 4>(q, s, slots, slot, arena_down, arena_up, d, st);
    if (2 * per_row <= (size_t)MQ_SMEM_MAX) return launch_merge_quant_r<E, 2>(q, s, slots, slot, arena_down, arena_up, d, st);
    if (per_row <= (size_t)MQ_SMEM_MAX) return launch_merge_quant_r<E, 1>(q, s, slots, slot, arena_down, arena_up, d, st);
    return cudaErrorInvalidValue;   // a row of din fp32 does not fit
}

cudaError_t launch_merge_quant(bool bf16, int8_t* q, float* s, const SlotRec* slots, int slot, const void* arena_down,
                               const void* arena_up, const PoolDims& d, cudaStream_t st) {
    return bf16 ? launch_merge_quant_e<__nv_bfloat16>(q, s, slots, slot, arena_down, arena_up, d, st)
                : launch_merge_quant_e<float>(q, s, slots, slot, arena_down, arena_up, d, st);
}

// ---------------------------------------------------------------- NF4 base
// 4-bit codes, two per byte (column 2m in the low nibble of byte m of a row), an fp32
// absmax per output row and block of 64 input columns stored block-major
// ([din/64][dout]: consecutive rows of one block are adjacent), and a 16-entry
// codebook (ai-infra-kb "M031" §05: W restored by scale and codebook).
namespace {

constexpr int NF4_BLOCK = 64;

struct Codebook {
    float v[16];
};

// 16 codes (8 bytes) of row o from column i0 (a multiple of 16): W = codebook[code] *
// absmax, rounded once to the pool dtype.
template <typename E>
__global__ void __launch_bounds__(DQ_THREADS)
dequant_nf4_kernel(const uint8_t* __restrict__ q, const float* __restrict__ absmax, Codebook cb, int dout, int din,
                   E* __restrict__ W) {
    __shared__ float cb_s[16];
    if (threadIdx.x < 16) cb_s[threadIdx.x] = cb.v[threadIdx.x];
    __syncthreads();
    const size_t groups = (size_t)dout * (din / 16);
    const uint32_t gpr = (uint32_t)(din / 16);
    for (size_t g = blockIdx.x * (size_t)blockDim.x + threadIdx.x; g < groups; g += (size_t)gridDim.x * blockDim.x) {
        const size_t o = g / gpr;
        const int i0 = (int)(g - o * gpr) * 16;
        const uint2 raw = *reinterpret_cast<const uint2*>(q + o * (din / 2) + i0 / 2);
        const float sc = absmax[(size_t)(i0 / NF4_BLOCK) * dout + o];
        const uint32_t b[2] = {raw.x, raw.y};
        __align__(16) E out[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t byte = (b[j >> 2] >> (8 * (j & 3))) & 0xFFu;
            out[2 * j] = from_f32<E>(cb_s[byte & 15u] * sc);
            out[2 * j + 1] = from_f32<E>(cb_s[byte >> 4] * sc);
        }
        const int4* src = reinterpret_cast<const int4*>(out);
        int4* d = reinterpret_cast<int4*>(W + o * din + i0);
#pragma unroll
        for (int j = 0; j < (int)(16 * sizeof(E) / 16); ++j) d[j] = src[j];
    }
}

// The merge on an NF4 base, in place.  One CTA per (block of 64 columns, 64 rows): the
// block's Down columns and the rows' Up values go to shared memory once (fp32); each
// warp then takes 8 rows, lane l columns 2l and 2l+1 (one byte of codes).  Restore
// (fp32 codebook value times the block's absmax), add scale * sum_k Up[o,k] Down[k,i]
// (fp32, k ascending), take the block's new absmax, and give each w / absmax (fp32
// division) the code of the nearest codebook value (fp32 distances, the first of equal
// ones).
constexpr int MN4_ROWS = 256;   // output rows per CTA of the NF4 merge: one per thread

// The nearest codebook entry to v (fp32 distances, the lower code on a tie), for an
// ascending codebook: bisection to the two entries that bracket v, then their
// distances.  (An entry further out is strictly further in fp32 as well: the gaps of
// the codebook are far above the rounding of a difference of values in [-1, 1].)
__device__ __forceinline__ uint32_t nf4_code_of(float v, const float* cb) {
    int j = 0;   // entries below v, at most 15
#pragma unroll
    for (int step = 8; step > 0; step >>= 1)
        if (cb[j + step - 1] < v) j += step;
    if (j == 0) return 0u;
    return fabsf(v - cb[j]) < fabsf(v - cb[j - 1]) ? (uint32_t)j : (uint32_t)(j - 1);
}

template <typename E>
__global__ void __launch_bounds__(MN4_ROWS)
merge_nf4_kernel(uint8_t* __restrict__ q, float* __restrict__ absmax, Codebook cb, const SlotRec* __restrict__ slots,
                 int slot, const E* __restrict__ arena_down, const E* __restrict__ arena_up, int din, int dout,
                 int aligned) {
    extern __shared__ float4 mn4_s[];   // [rank][64] Down columns of the block, fp32
    __shared__ float cb_s[16];
    const SlotRec rec = slots[slot];
    const int rank = rec.rank;
    const int blk = blockIdx.x;
    const int o = blockIdx.y * MN4_ROWS + threadIdx.x;   // this thread's output row
    float* down_s = reinterpret_cast<float*>(mn4_s);
    if (threadIdx.x < 16) cb_s[threadIdx.x] = cb.v[threadIdx.x];
    const E* down = arena_down + (size_t)rec.unit * din + blk * NF4_BLOCK;
    for (int idx = threadIdx.x; idx < rank * NF4_BLOCK; idx += blockDim.x) {
        const int k = idx / NF4_BLOCK, c = idx % NF4_BLOCK;
        down_s[idx] = as_f32(down[(size_t)k * din + c]);
    }
    __syncthreads();
    if (o >= dout) return;
    // the row's 64 codes of the block (32 bytes) and its scale
    uint8_t* qb = q + (size_t)o * (din / 2) + blk * (NF4_BLOCK / 2);
    uint32_t cw[8];
    if (aligned) {
        const uint4 a = *reinterpret_cast<const uint4*>(qb), b = *reinterpret_cast<const uint4*>(qb + 16);
        cw[0] = a.x; cw[1] = a.y; cw[2] = a.z; cw[3] = a.w; cw[4] = b.x; cw[5] = b.y; cw[6] = b.z; cw[7] = b.w;
    } else {
        for (int i = 0; i < 8; ++i)
            cw[i] = qb[4 * i] | (qb[4 * i + 1] << 8) | (qb[4 * i + 2] << 16) | ((uint32_t)qb[4 * i + 3] << 24);
    }
    float* am = absmax + (size_t)blk * dout + o;
    const float old = *am;
    // u = Up[o, :] Down[:, block] in fp32, k ascending
    float u[NF4_BLOCK];
#pragma unroll
    for (int c = 0; c < NF4_BLOCK; ++c) u[c] = 0.f;
    for (int k0 = 0; k0 < rank; k0 += 8) {
        float upk[8];   // eight Up values requested at once
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            upk[kk] = k0 + kk < rank ? as_f32(arena_up[up_index(rec.unit, k0 + kk, o, dout)]) : 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            if (k0 + kk >= rank) break;
            const float4* dk = mn4_s + (k0 + kk) * (NF4_BLOCK / 4);
#pragma unroll
            for (int c4 = 0; c4 < NF4_BLOCK / 4; ++c4) {
                const float4 d = dk[c4];   // (the same address in every thread: a broadcast)
                u[4 * c4] = fmaf(upk[kk], d.x, u[4 * c4]);
                u[4 * c4 + 1] = fmaf(upk[kk], d.y, u[4 * c4 + 1]);
                u[4 * c4 + 2] = fmaf(upk[kk], d.z, u[4 * c4 + 2]);
                u[4 * c4 + 3] = fmaf(upk[kk], d.w, u[4 * c4 + 3]);
            }
        }
    }
    // merged values (restored + scale * u) and the block's new absmax
    float m = 0.f;
#pragma unroll
    for (int c = 0; c < NF4_BLOCK; ++c) {
        const uint32_t code = (cw[c >> 3] >> (4 * (c & 7))) & 15u;
        u[c] = cb_s[code] * old + rec.scale * u[c];
        m = fmaxf(m, fabsf(u[c]));
    }
    // the codes of w / absmax, two per byte (even column in the low nibble)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float v = m > 0.f ? u[8 * i + e] / m : 0.f;
            word |= nf4_code_of(v, cb_s) << (4 * e);
        }
        cw[i] = word;
    }
    if (aligned) {
        *reinterpret_cast<uint4*>(qb) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        *reinterpret_cast<uint4*>(qb + 16) = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    } else {
        for (int i = 0; i < 32; ++i) qb[i] = (uint8_t)(cw[i >> 2] >> (8 * (i & 3)));
    }
    *am = m;
}

}  // namespace

cudaError_t launch_dequant_nf4(bool bf16, const uint8_t* q, const float* absmax, const float* codebook, int dout,
                               int din, void* W, cudaStream_t st) {
    Codebook cb;
    for (int j = 0; j < 16; ++j) cb.v[j] = codebook[j];
    const size_t groups = (size_t)dout * (din / 16);
    size_t blocks = (groups + DQ_THREADS - 1) / DQ_THREADS;
    const size_t cap = (size_t)quant_sms() * 8;
    blocks = blocks < cap ? blocks : cap;
    if (blocks == 0) return cudaSuccess;
    if (bf16)
        dequant_nf4_kernel<__nv_bfloat16><<<(unsigned)blocks, DQ_THREADS, 0, st>>>(q, absmax, cb, dout, din,
                                                                                  (__nv_bfloat16*)W);
    else
        dequant_nf4_kernel<float><<<(unsigned)blocks, DQ_THREADS, 0, st>>>(q, absmax, cb, dout, din, (float*)W);
    return cudaGetLastError();
}

cudaError_t launch_merge_nf4(bool bf16, uint8_t* q, float* absmax, const float* codebook, const SlotRec* slots,
                             int slot, const void* arena_down, const void* arena_up, const PoolDims& d,
                             cudaStream_t st) {
    Codebook cb;
    for (int j = 0; j < 16; ++j) cb.v[j] = codebook[j];
    if (d.dout == 0 || d.din == 0) return cudaSuccess;
    // shared memory for the largest rank the pool takes: Down [rank][64], fp32
    const size_t smem = sizeof(float) * (size_t)d.max_rank * NF4_BLOCK;
    const dim3 grid((unsigned)(d.din / NF4_BLOCK), (unsigned)((d.dout + MN4_ROWS - 1) / MN4_ROWS));
    const int aligned = ((uintptr_t)q & 15u) == 0 ? 1 : 0;   // rows of din / 2 bytes, din % 64 == 0
    cudaError_t e;
    if (bf16) {
        e = cudaFuncSetAttribute(merge_nf4_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        merge_nf4_kernel<__nv_bfloat16><<<grid, MN4_ROWS, smem, st>>>(
            q, absmax, cb, slots, slot, (const __nv_bfloat16*)arena_down, (const __nv_bfloat16*)arena_up, d.din, d.dout,
            aligned);
    } else {
        e = cudaFuncSetAttribute(merge_nf4_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        merge_nf4_kernel<float><<<grid, MN4_ROWS, smem, st>>>(q, absmax, cb, slots, slot, (const float*)arena_down,
                                                            (const float*)arena_up, d.din, d.dout, aligned);
    }
    return cudaGetLastError();
}

}  // namespace mlora
