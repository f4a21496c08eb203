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
// Both are bandwidth-bound sweeps over W.  The merge runs one CTA per group of rows,
// one row at a time: the row is read, updated and held in shared memory (fp32),
// reduced to its max, then written back as codes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace mlora {

namespace {

constexpr int DQ_THREADS = 256;
constexpr int MQ_THREADS = 256;
constexpr int MQ_ROWS = 4;                   // rows per CTA of the merge
constexpr int MQ_SMEM_MAX = 200 * 1024;      // one merged row held in shared memory (fp32)

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

// One thread per 16 codes of a row (din % 16 == 0: one 16-byte load), else per code.
template <typename E>
__global__ void __launch_bounds__(DQ_THREADS)
dequant_kernel(const int8_t* __restrict__ q, const float* __restrict__ s, int dout, int din, E* __restrict__ W) {
    const bool vec = (din % 16) == 0;
    const size_t groups = vec ? (size_t)dout * (din / 16) : (size_t)dout * din;
    for (size_t g = blockIdx.x * (size_t)blockDim.x + threadIdx.x; g < groups; g += (size_t)gridDim.x * blockDim.x) {
        if (vec) {
            const size_t e0 = g * 16;
            const int o = (int)(e0 / din);
            const float so = s[o];
            const int4 raw = *reinterpret_cast<const int4*>(q + e0);
            const int8_t* c = reinterpret_cast<const int8_t*>(&raw);
            __align__(16) E out[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) out[j] = from_f32<E>((float)c[j] * so);
            const int4* src = reinterpret_cast<const int4*>(out);
            int4* dst = reinterpret_cast<int4*>(W + e0);
#pragma unroll
            for (int j = 0; j < (int)(16 * sizeof(E) / 16); ++j) dst[j] = src[j];
        } else {
            const int o = (int)(g / din);
            W[g] = from_f32<E>((float)q[g] * s[o]);
        }
    }
}

// CTA per `rows` consecutive output rows, one after the other (shared memory: din fp32).
template <typename E>
__global__ void __launch_bounds__(MQ_THREADS)
merge_quant_kernel(int8_t* __restrict__ q, float* __restrict__ s, const SlotRec* __restrict__ slots, int slot,
                   const E* __restrict__ arena_down, const E* __restrict__ arena_up, int din, int dout, int rows) {
    extern __shared__ float wsh[];   // [din]: the row being merged
    __shared__ float red[MQ_THREADS / 32];
    const SlotRec rec = slots[slot];
    const int o0 = blockIdx.x * rows;
    const int nr = min(rows, dout - o0);
    const E* down = arena_down + (size_t)rec.unit * din;
    for (int r = 0; r < nr; ++r) {
        const int o = o0 + r;
        const float so = s[o];
        float m = 0.f;
        for (int i = threadIdx.x; i < din; i += MQ_THREADS) {
            float acc = 0.f;
            for (int k = 0; k < rec.rank; ++k)
                acc = fmaf(as_f32(arena_up[up_index(rec.unit, k, o, dout)]), as_f32(down[(size_t)k * din + i]), acc);
            const float w = fmaf(rec.scale, acc, (float)q[(size_t)o * din + i] * so);
            wsh[i] = w;
            m = fmaxf(m, fabsf(w));
        }
        // max over the row: warp shuffle, then across warps
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x < 32) {
            float v = threadIdx.x < MQ_THREADS / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
            if (threadIdx.x == 0) red[0] = v;
        }
        __syncthreads();
        const float mx = red[0];
        __syncthreads();   // red is reused by the next row
        const float sn = mx / 127.f;   // new row scale (0 for an all-zero row: codes 0)
        for (int i = threadIdx.x; i < din; i += MQ_THREADS) {
            int c = 0;
            if (sn > 0.f) {
                c = __float2int_rn(wsh[i] / sn);
                c = c > 127 ? 127 : (c < -127 ? -127 : c);
            }
            q[(size_t)o * din + i] = (int8_t)c;
        }
        if (threadIdx.x == 0) s[o] = sn;
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

cudaError_t launch_merge_quant(bool bf16, int8_t* q, float* s, const SlotRec* slots, int slot, const void* arena_down,
                               const void* arena_up, const PoolDims& d, cudaStream_t st) {
    const int rows = MQ_ROWS;
    const size_t smem = sizeof(float) * (size_t)d.din;
    if (smem > (size_t)MQ_SMEM_MAX) return cudaErrorInvalidValue;   // din above 51 200
    const unsigned grid = (unsigned)((d.dout + rows - 1) / rows);
    cudaError_t e;
    if (bf16) {
        e = cudaFuncSetAttribute(merge_quant_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        merge_quant_kernel<__nv_bfloat16><<<grid, MQ_THREADS, smem, st>>>(
            q, s, slots, slot, (const __nv_bfloat16*)arena_down, (const __nv_bfloat16*)arena_up, d.din, d.dout, rows);
    } else {
        e = cudaFuncSetAttribute(merge_quant_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        merge_quant_kernel<float><<<grid, MQ_THREADS, smem, st>>>(q, s, slots, slot, (const float*)arena_down,
                                                                  (const float*)arena_up, d.din, d.dout, rows);
    }
    return cudaGetLastError();
}

}  // namespace mlora
