// Static merge of one adapter into a bf16 base weight on the tensor cores
// (ai-infra-kb "M031" tutorial §04):
//
//     W[o, i] <- bf16( W[o, i] + scale * sum_k Up[o, k] Down[k, i] )      (fp32 sum)
//
// and, with the sign flipped, the un-merge that re-subtracts the same update
// (airsota card "multi-LoRA serving vs merging", section 四 item ③: a merge
// overwrites the base; switching back means subtracting it again, or restoring a
// kept original).
//
// The update is an outer product with K = rank: one CTA per tile of 128 rows (o) x
// 128 columns (i) computes it as tcgen05 MMAs of M = 128, N = 128, K = 16, one per 16
// rank columns, into a TMEM accumulator.  A = the adapter's Up columns, read from the
// arena's 8-column blocks without swizzle (K-major, as in the forward's
// K-extension); B = the adapter's Down rows [16 x 128], which are N-contiguous, so
// they are read as an MN-major operand (128-byte swizzle).  The W tile comes in by
// TMA first (it is needed last); the epilogue adds scale * acc to it in shared
// memory, rounds once, and TMA stores the tile back, so W is read and written in
// whole lines.  Warp 0 issues the loads, warp 1 allocates TMEM and issues the MMAs,
// warps 2..5 run the epilogue; every wait is bounded.
//
// The same kernel merges into a quantized base (M031 §05: restore, merge in floating
// point, quantize again; int8 codes with one fp32 scale per output row) in two
// launches over tiles of 128 x 128 codes, one TMA box each:
//   MODE_QMAX   w = scale * acc + code * row_scale for the tile, and each row's max |w|
//               folded into a per-row word (atomicMax on the bits: w >= 0 orders
//               like its bits);
//   MODE_QCODES the same w again (same MMAs, same order: the same bits), codes
//               round(w / (max / 127)) to nearest even, clamped to +-127, stored in place.
// A third launch then writes the new row scales max / 127 and clears the words.
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

constexpr int MG_BM = 128;                         // rows (o) per tile
constexpr int MG_THREADS = 192;
constexpr int MG_STAGES = 2;                       // rank chunks in flight (4 CTAs fit an SM)
constexpr int MG_UP_BYTES = MG_BM * CHUNK * 2;     // 4 KiB: 2 blocks of 8 rank columns x 128 rows

constexpr int MODE_BF16 = 0;    // W tile bf16, W += sign * scale * Up Down
constexpr int MODE_QMAX = 1;    // codes tile: the merged rows' max |w|
constexpr int MODE_QCODES = 2;  // codes tile: the merged rows' new codes

// Tile of MG_BM rows x BN columns: the W tile is BN/64 blocks of 128 rows x 64 columns
// (bf16; codes: BN/128 blocks of 128 rows x 128 columns), a rank chunk's Down is BN/64
// blocks of 16 rows x 64 columns.
template <int BN, int MODE = MODE_BF16>
struct MergeShape {
    static constexpr int W_BYTES = MG_BM * BN * (MODE == MODE_BF16 ? 2 : 1);
    static constexpr int DOWN_BYTES = CHUNK * BN * 2;
    static constexpr int STAGE = DOWN_BYTES + MG_UP_BYTES;
};

struct MergeTail {
    uint64_t full[MG_STAGES];
    uint64_t empty[MG_STAGES];
    uint64_t wfull;
    uint64_t acc_full;
    uint32_t tmem_slot;
    int abort_flag;
};

struct MergeParams {
    const SlotRec* slots;
    int slot;
    float sign;             // +1 merge, -1 un-merge
    uint32_t* status;
    const float* row_scale; // quantized base: the codes' scale per output row
    uint32_t* row_max;      // quantized base: max |w| per output row (fp32 bits)
    int dout;
    int up_rows;            // output rows per row of the Up map (8: 128-byte rows, or 1)
};


template <int BN, int MODE>
__global__ void __launch_bounds__(MG_THREADS, 1)
merge_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmDown,
                const __grid_constant__ CUtensorMap tmUp, MergeParams p) {
    using Sh = MergeShape<BN, MODE>;
    static_assert(MODE == MODE_BF16 || BN % 128 == 0, "a codes tile is whole 128-byte rows");
    constexpr int MG_BN = BN, MG_W_BYTES = Sh::W_BYTES, MG_DOWN_BYTES = Sh::DOWN_BYTES, MG_STAGE = Sh::STAGE;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* wt = smem;                                 // W tile
    uint8_t* ring = smem + MG_W_BYTES;                  // rank-chunk stages: Down then Up
    MergeTail& tl = *reinterpret_cast<MergeTail*>(ring + MG_STAGES * MG_STAGE);
    volatile int* abort_flag = &tl.abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = blockIdx.x * MG_BN, o0 = blockIdx.y * MG_BM;
    const SlotRec rec = p.slots[p.slot];
    const int nk = (rec.rank + CHUNK - 1) / CHUNK;     // rank chunks (MMA K steps)
    const float sc = p.sign * rec.scale;

    if (threadIdx.x == 0) {
        for (int s = 0; s < MG_STAGES; ++s) {
            mbar_init(&tl.full[s], 1);
            mbar_init(&tl.empty[s], 1);
        }
        mbar_init(&tl.wfull, 1);
        mbar_init(&tl.acc_full, 1);
        tl.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tl.tmem_slot)),
                     "r"(MG_BN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tl.tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---- loads: the W tile, then the rank chunks through the ring
        mbar_expect_tx(&tl.wfull, (uint32_t)MG_W_BYTES);
        if (MODE == MODE_BF16)
            for (int j = 0; j < MG_BN / 64; ++j) tma_2d(wt + j * (MG_BM * 128), &tmW, &tl.wfull, i0 + 64 * j, o0);
        else
            for (int j = 0; j < MG_BN / 128; ++j) tma_2d(wt + j * (MG_BM * 128), &tmW, &tl.wfull, i0 + 128 * j, o0);
        int s = 0;
        uint32_t ph = 0;
        int issued = 0;
        for (; issued < nk; ++issued) {
            if (!mbar_wait(&tl.empty[s], ph ^ 1, abort_flag, p.status)) break;
            uint8_t* dn = ring + s * MG_STAGE;
            uint8_t* up = dn + MG_DOWN_BYTES;
            const int u = rec.unit + issued * CHUNK;   // first arena unit of the chunk (a multiple of 8)
            mbar_expect_tx(&tl.full[s], (uint32_t)MG_STAGE);
            for (int j = 0; j < MG_BN / 64; ++j) tma_2d(dn + j * (CHUNK * 128), &tmDown, &tl.full[s], i0 + 64 * j, u);
            tma_3d(up, &tmUp, &tl.full[s], 0, o0 / p.up_rows, u >> 3);
            if (++s == MG_STAGES) {
                s = 0;
                ph ^= 1;
            }
        }
        if (*abort_flag) {   // let issued loads land before the shared memory goes away
            const long long t0 = clock64();
            while (!mbar_try_wait(&tl.wfull, 0) && clock64() - t0 < 200000000ll) {
            }
            for (int j = 0; j < MG_STAGES && j < issued; ++j) {
                const int fills = (issued - 1 - j) / MG_STAGES + 1;
                const long long t1 = clock64();
                while (!mbar_try_wait(&tl.full[j], (uint32_t)((fills - 1) & 1)) && clock64() - t1 < 200000000ll) {
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMAs: D[o, i] += Up[o, 16 ranks] Down[16 ranks, i]
        const uint32_t idesc = idesc_bf16(MG_BM, MG_BN) | (1u << 16);   // B is MN-major
        int s = 0;
        uint32_t ph = 0;
        uint32_t acc = 0;
        for (int c = 0; c < nk; ++c) {
            if (!mbar_wait(&tl.full[s], ph, abort_flag, p.status)) break;
            tc_fence_after();
            uint8_t* dn = ring + s * MG_STAGE;
            uint8_t* up = dn + MG_DOWN_BYTES;
            // Arena units past round8(rank) in the last chunk belong to the next adapter:
            // zero that half of the Up columns (the padding up to round8 is zero already)
            if (rec.rank - c * CHUNK <= 8) {
                for (int q = 0; q < MG_BM; ++q)
                    *reinterpret_cast<uint4*>(up + MG_BM * 16 + q * 16) = make_uint4(0u, 0u, 0u, 0u);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            // Up: [2 blocks of 8 columns][128 rows][16 B] without swizzle (K-direction core
            // matrices 128*16 bytes apart, M-direction 128 bytes);  Down: [BN/64 blocks of 64
            // columns][16 rows][128 B], 128-byte swizzle, MN-major (MN blocks 2 KiB apart,
            // 8-row K groups 1 KiB apart)
            mma_bf16(tmem, sdesc_lbo(smem_u32(up), MG_BM * 16, 128, SW_NONE),
                     sdesc_lbo(smem_u32(dn), CHUNK * 128, 1024, SW128), idesc, acc);
            acc = 1;
            mma_commit(&tl.empty[s]);
            if (++s == MG_STAGES) {
                s = 0;
                ph ^= 1;
            }
        }
        mma_commit(&tl.acc_full);
        if (*abort_flag) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&tl.acc_full, 0) && clock64() - t0 < 200000000ll) {
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue: W tile (swizzled rows of 128 B) += scale * acc, in place, then store
        //      (codes: the merged rows' max, or their new codes stored in place)
        const int q = warp & 3;
        const int row = q * 32 + lane;   // row of the tile = TMEM lane
        const bool ok_acc = mbar_wait(&tl.acc_full, 0, abort_flag, p.status);
        const bool ok_w = mbar_wait(&tl.wfull, 0, abort_flag, p.status);
        __syncwarp();
        tc_fence_after();
        const bool have = __all_sync(0xffffffffu, ok_acc && ok_w) && nk > 0;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
        if constexpr (MODE != MODE_BF16) {
            // codes: 16 columns = one 16-byte chunk of the row's 128 bytes, swizzled by
            // the row's position in its 8-row group
            const int o = o0 + row;
            const float so = o < p.dout ? p.row_scale[o] : 0.f;
            const float sn = MODE == MODE_QCODES && o < p.dout ? __uint_as_float(p.row_max[o]) / 127.f : 0.f;
            // 1 / sn for the quotients (0 for an all-zero row: codes 0); an sn so small
            // that it has no finite reciprocal takes every quotient exactly
            const float inv = sn > 0.f ? 1.f / sn : 0.f;
            const bool fast = inv <= 3.0e38f;
            float m = 0.f;
            for (int c16 = 0; c16 < MG_BN / 16; ++c16) {
                float v[16];
                if (have) tmem_ld16(tbase + c16 * 16, v);
                else
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                uint4* cell = reinterpret_cast<uint4*>(wt + (c16 >> 3) * (MG_BM * 128) + row * 128 +
                                                      (((c16 & 7) ^ (row & 7)) * 16));
                uint4 raw = *cell;
                int8_t* c8 = reinterpret_cast<int8_t*>(&raw);
                float w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    // the code as a float without a conversion instruction: 2^23 + 128 + c
                    // has c + 128 in its low mantissa bits
                    const float cf = __int_as_float(0x4B000000 + 128 + (int)c8[j]) - 8388736.f;
                    w[j] = fmaf(sc, v[j], cf * so);
                }
                if constexpr (MODE == MODE_QMAX) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(w[j]));
                } else {
                    // The code is the nearest integer (ties to even) to the fp32 quotient
                    // w / sn, |w / sn| < 128.  w * inv (two roundings) lies within
                    // 128 * 3 * 2^-24 < 2^-15 of it: farther than 2^-14 from every
                    // half-integer, both round to the same integer, found by adding
                    // 1.5 * 2^23 (the sum's low mantissa bits are the rounded value);
                    // nearer, the quotient is taken exactly.
                    constexpr float RND = 12582912.f;   // 1.5 * 2^23
                    uint32_t near = fast ? 0u : 0xFFFFu;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float qf = w[j] * inv;
                        const float t = qf + RND;
                        if (fabsf(qf - (t - RND)) > 0.5f - 0x1p-14f) near |= 1u << j;
                        int c = __float_as_int(t) - __float_as_int(RND);
                        c = c > 127 ? 127 : (c < -127 ? -127 : c);
                        c8[j] = (int8_t)c;
                    }
                    if (near && sn > 0.f) {
                        for (int j = 0; j < 16; ++j)
                            if ((near >> j) & 1u) {
                                int c = __float2int_rn(w[j] / sn);
                                c8[j] = (int8_t)(c > 127 ? 127 : (c < -127 ? -127 : c));
                            }
                    } else if (near) {
                        for (int j = 0; j < 16; ++j) c8[j] = 0;
                    }
                }
                if (MODE == MODE_QCODES) *cell = raw;
            }
            // columns past din hold zero codes and zero Down (TMA fill): w = 0 there
            if (MODE == MODE_QMAX && have && o < p.dout) atomicMax(p.row_max + o, __float_as_uint(m));
        } else {
            for (int c16 = 0; c16 < MG_BN / 16; ++c16) {
                float v[16];
                if (have) tmem_ld16(tbase + c16 * 16, v);
                else
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                // columns c16*16 .. +15: block c16/4, 16-byte chunks 2(c16%4) and +1, swizzled
                // by the row's position in its 8-row group
                uint8_t* blk = wt + (c16 >> 2) * (MG_BM * 128) + row * 128;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int ch = ((c16 & 3) * 2 + h) ^ (row & 7);
                    uint4* cell = reinterpret_cast<uint4*>(blk + ch * 16);
                    uint4 w = *cell;
                    __nv_bfloat162* hw = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 f = __bfloat1622float2(hw[j]);
                        hw[j] = __floats2bfloat162_rn(fmaf(sc, v[h * 8 + 2 * j], f.x),
                                                      fmaf(sc, v[h * 8 + 2 * j + 1], f.y));
                    }
                    *cell = w;
                }
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> TMA store
        __syncwarp();
        epi_bar();
        if (threadIdx.x == 64 && have && MODE != MODE_QMAX) {
            const int bw = MODE == MODE_BF16 ? 64 : 128;   // columns per stored block
            for (int j = 0; j < MG_BN / bw; ++j)
                asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(&tmW),
                             "r"(i0 + bw * j), "r"(o0), "r"(smem_u32(wt + j * (MG_BM * 128)))
                             : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");   // the tile is read before exit
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(MG_BN) : "memory");
    }
}

template <int BN, int MODE>
size_t merge_smem() {
    return 1024 + MergeShape<BN, MODE>::W_BYTES + MG_STAGES * MergeShape<BN, MODE>::STAGE + sizeof(MergeTail);
}

// columns per tile (128: 4 CTAs per SM, their loads, MMAs and stores interleave)
constexpr int MG_BN_USED = 128;

template <int MODE>
cudaError_t merge_attrs() {
    cudaError_t e = cudaFuncSetAttribute(merge_tc_kernel<MG_BN_USED, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)merge_smem<MG_BN_USED, MODE>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(merge_tc_kernel<MG_BN_USED, MODE>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    return e;
}

// New row scales after a quantized merge, and the per-row words cleared for the next.
__global__ void row_scale_kernel(float* __restrict__ s, uint32_t* __restrict__ row_max, int dout) {
    const int o = blockIdx.x * blockDim.x + threadIdx.x;
    if (o < dout) {
        s[o] = __uint_as_float(row_max[o]) / 127.f;   // 0 for an all-zero row: its codes are 0
        row_max[o] = 0u;
    }
}

// A 2D int8 tensor map (the codes), 128-byte swizzle.
bool encode_u8(CUtensorMap* map, const void* base, const cuuint64_t* dims, const cuuint64_t* strides,
               const cuuint32_t* box) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
        fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    }
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t merge_tc_init() {
    cudaError_t e = merge_attrs<MODE_BF16>();
    if (e == cudaSuccess) e = merge_attrs<MODE_QMAX>();
    if (e == cudaSuccess) e = merge_attrs<MODE_QCODES>();
    return e;
}

cudaError_t launch_merge_quant_tc(int8_t* Wq, float* row_scale, uint32_t* row_max, const SlotRec* slots, int slot,
                                  const TcArenaMaps& maps, uint32_t* status, const PoolDims& d, cudaStream_t st) {
    if (d.din % 16 != 0 || ((uintptr_t)Wq & 15u) != 0) return cudaErrorInvalidValue;   // TMA row stride and base
    CUtensorMap tmQ;
    cuuint64_t dims[2] = {(cuuint64_t)d.din, (cuuint64_t)d.dout};
    cuuint64_t strides[1] = {(cuuint64_t)d.din};
    cuuint32_t box[2] = {128, (cuuint32_t)MG_BM};
    if (!encode_u8(&tmQ, Wq, dims, strides, box)) return cudaErrorInvalidValue;
    MergeParams p{slots, slot, 1.f, status, row_scale, row_max, d.dout, maps.up_rows};
    const dim3 grid((d.din + MG_BN_USED - 1) / MG_BN_USED, (d.dout + MG_BM - 1) / MG_BM);
    cudaError_t e = launch_k(merge_tc_kernel<MG_BN_USED, MODE_QMAX>, grid, dim3(MG_THREADS),
                             merge_smem<MG_BN_USED, MODE_QMAX>(), st, false, 1, tmQ, maps.down, maps.upw128, p);
    if (e != cudaSuccess) return e;
    e = launch_k(merge_tc_kernel<MG_BN_USED, MODE_QCODES>, grid, dim3(MG_THREADS), merge_smem<MG_BN_USED, MODE_QCODES>(),
                 st, false, 1, tmQ, maps.down, maps.upw128, p);
    if (e != cudaSuccess) {   // the words hold this call's maxima: clear them for the next call
        cudaMemsetAsync(row_max, 0, sizeof(uint32_t) * (size_t)d.dout, st);
        return e;
    }
    row_scale_kernel<<<(d.dout + 255) / 256, 256, 0, st>>>(row_scale, row_max, d.dout);
    return cudaGetLastError();
}

cudaError_t launch_merge_tc(void* W, const SlotRec* slots, int slot, const TcArenaMaps& maps, uint32_t* status,
                            const PoolDims& d, float sign, cudaStream_t st) {
    CUtensorMap tmW;
    cuuint64_t dims[2] = {(cuuint64_t)d.din, (cuuint64_t)d.dout};
    cuuint64_t strides[1] = {(cuuint64_t)d.din * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)MG_BM};
    if (!tc_encode(&tmW, W, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    MergeParams p{slots, slot, sign, status, nullptr, nullptr, d.dout, maps.up_rows};
    const dim3 grid((d.din + MG_BN_USED - 1) / MG_BN_USED, (d.dout + MG_BM - 1) / MG_BM);
    return launch_k(merge_tc_kernel<MG_BN_USED, MODE_BF16>, grid, dim3(MG_THREADS), merge_smem<MG_BN_USED, MODE_BF16>(),
                    st, false, 1, tmW, maps.down, maps.upw128, p);
}

}  // namespace mlora
