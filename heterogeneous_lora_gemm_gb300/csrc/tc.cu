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
// it to bf16 and writes Vt[c][t][:], zero for every other token.  One more grid
// column holds the segment builder (seg.cuh): its first CTA builds and publishes
// the segments while the others multiply.
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
    return tc_encode_typed(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides, box, sw);
}

bool tc_encode_typed(CUtensorMap* map, CUtensorMapDataType type, const void* base, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};   // (element strides, up to rank 5)
    CUresult r = fn(map, type, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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
constexpr int EXT_SUB = 4;         // K-extension chunks per pipeline step (one int4 of the step plan)
constexpr int A_BYTES = BM * BK * 2;            // 16 KiB: W tile, 4 Up chunk tiles or 8 Down chunk tiles
constexpr int NUM_THREADS = 192;   // warp 0 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr int MAX_N = 256;
constexpr int CHUNKS_PER_TILE = BM / CHUNK;     // shrink: 8 chunks of 16 rank rows
constexpr int CHUNK_BYTES = CHUNK * BK * 2;     // 2 KiB: 16 rank rows x 64 din columns of Down
constexpr int MAX_SPLITS = 16;     // K splits per tile at most
constexpr int MAX_CLUSTER = 8;     // K splits of a tile reduced inside one (portable) cluster
constexpr int MAX_STAGES = 12;
constexpr int EXT_CAP = 256;       // projection: K-extension chunks of a CTA kept in shared memory
constexpr int UNUSED = 1 << 30;    // projection: flag of a listed chunk's arena unit the batch does not use
constexpr int RUN_UNITS_MAX = (1 << 23) - 1;   // arenas read as runs: a step plan entry packs unit + 1 << 8
// the arena unit of a listed chunk the batch uses, else -1
__host__ __device__ constexpr int used_unit(int v) { return v >= 0 && !(v & UNUSED) ? v : -1; }
constexpr int MAX_SLOT_WORDS = 4096 / 32;
constexpr int EXT_LEAD = 0;        // projection: K-extension steps go this many K chunks of 64 before the end
constexpr int PUSH_MAX_N = 64;     // projection: tokens up to which the splits push their partials
constexpr int PROJ_KC = 2;         // projection: K chunks of 64 per pipeline step (one 3D box each for W and X)
constexpr int PROJ_ZT_N = 128;     // projection: tokens per token tile of a wide decode batch
constexpr int PROJ_ZT_MIN = 224;   // a decode batch of more tokens than this runs as token tiles
constexpr int QUANT_KC = 2;        // projection over codes: K chunks of 64 per pipeline step
constexpr int QMODE_INT8 = 1, QMODE_NF4 = 2;

__host__ __device__ constexpr int b_bytes(int n) { return n * BK * 2; }
__host__ __device__ constexpr int stage_bytes(int n) { return A_BYTES + b_bytes(n); }

// Shared-memory tail after the stage ring and the segment scratch.
struct Tail {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t conv[MAX_STAGES];        // projection over codes: the stage's W tile is restored
    uint64_t acc_full;
    uint64_t info_ready;              // projection: the K-extension chunk info is in place
    uint64_t rx_bar;                  // projection, push reduction: all splits' slices have landed
    int stage_kind[MAX_STAGES];       // -1 = din step, else bit mask of the K-extension chunks loaded
    uint32_t tmem_slot;
    int abort_flag;
    int flags[2];                     // [0] an MMA was issued, [1] last arrival (global reduction)
    int tile_chunks;                  // shrink: chunks of this row tile some token uses
    int win_u0;                       // shrink: arena unit of the window's first row
    int my_c[CHUNKS_PER_TILE];        // shrink, per compacted chunk: index in the chunk table,
    int my_slot[CHUNKS_PER_TILE];     //   slot, arena unit,
    int my_unit[CHUNKS_PER_TILE];
    int my_off[CHUNKS_PER_TILE];      //   first accumulator row, valid rank columns, scale
    int my_kval[CHUNKS_PER_TILE];
    float my_scale[CHUNKS_PER_TILE];
    int tile_ra[MAX_N];               // shrink: slot id of each token of the token tile
    uint32_t slot_bits[MAX_SLOT_WORDS];   // projection: slots some row of the batch uses
    int ext_unit[EXT_CAP];            // projection: arena unit of each K-extension chunk of this tile's
                                      // module (| UNUSED when the batch does not use it), -1 = none
    int ext_slot[EXT_CAP];            // (then: the K-extension units with a chunk to multiply)
    int n_ext, ext_first;             // projection: this split's share of that list
    int4 ext_plan[EXT_CAP / EXT_SUB]; // projection: per listed step of this split, its chunks' arena
                                      // units (-1 = not loaded), and
    int ext_plan_u[EXT_CAP / EXT_SUB];   // its unit (bits 0-7) | (arena unit of its first chunk + 1)
                                         // << 8 when its 4 chunks form a run (else 0 there)
    unsigned long long t_start;       // profiling: globaltimer at the CTA's start
};

struct GemmParams {
    const ChunkRec* chunks;         // chunk table of the loaded slots (ascending arena unit)
    const int32_t* row_adapter;     // slot id per token
    const SlotRec* slots;           // shrink: slot table (segment builder)
    __nv_bfloat16* Y;               // projection output [T x dout]
    __nv_bfloat16* vt;              // shrink output [max_chunks][tcap][16]
    uint8_t* tmask;                 // shrink output [token tile][max_chunks]
    float* partials;                // global reduction: [tile][split][N][BM]
    int32_t* tile_ctr;              // global reduction: [tile] arrival counters
    uint32_t* status;
    int T, dout, N, splits, stages, tcap;
    int kc;                         // K chunks of 64 columns per pipeline step
    int ksteps;                     // pipeline steps over din (ceil(din / (64 kc)))
    int a_sub;                      // bytes of the A operand per K chunk
    int window;                     // shrink: A is one window of win_rows arena rows per K chunk
    int win_rows;
    int n_chunks;                   // chunks in the table
    int ext_units;                  // projection: K-extension steps (EXT_SUB chunks each)
    int ring_bytes;                 // the stage ring; also the staging space of the reduction
    int tail_off;                   // offset of the Tail
    int pdl;                        // projection: launched while the shrink may still run
    int cluster;                    // the K splits of a tile form a cluster (else: global reduction)
    int push;                       // projection: the splits push their partial slices (bulk copies)
    int ext_lead;                   // projection: pipeline steps after the K-extension steps
    int xwait;                      // projection without shrink: launched early, griddepcontrol.wait
                                    // before reading X (W of the first stages goes out before)
    int rx_off;                     // push: offset of the receive buffer [split][BM][N / splits] fp32
    int S, max_chunks;
    int seg_tile, seg_P, seg_stage_rows;   // shrink: grid column of the segment builder, its plan
    Workspace ws;
    unsigned long long* stamps;     // profiling records (NULL = off), see ptx::stamp_record
    int stamp_cap;
    // projection over a quantized W (tmW maps the codes): 0 bf16 W; QMODE_INT8 int8 codes
    // with an fp32 scale per output row; QMODE_NF4 4-bit codes (two per byte, the even
    // column in the low nibble) with an fp32 scale per output row and 64 columns
    int qmode;
    int q_x;                        // code bytes per row and K chunk of 64 columns
    const float* qscale;            // QMODE_INT8: [dout]; QMODE_NF4: [din / 64][dout]
    float qcb[16];                  // QMODE_NF4: the codebook
    int qtab_off;                   // QMODE_NF4: shared-memory offset of the codebook (16 floats)
    int up_rows;                    // projection: output rows per row of the Up map (8 or 1)
    // projection: a K-extension step whose 4 chunks lie at a stride of run_b blocks of
    // 8 rank columns loads their Up tiles in one box of the runs map ({64, dout / 8,
    // run_b, run_groups}); run_b = 0: never (always over codes)
    int run_b, run_groups;
};

// Sum of one slice of the staged partial tiles: groups g in [et, ng) step nthr of 4
// rows x 1 token (rb staged rows per token), gpt groups per token, group i of a token
// at staged row row_of(i),
// loaded from the shared memory of all NSP CTAs of the cluster (or, NSP = 1, of this
// CTA), 8 float4 loads in flight per thread, summed in split order.  A group that
// need(token, i) rejects is not loaded: it is emitted as zeros.
template <int NSP, typename RowOf, typename Need, typename Emit>
__device__ __forceinline__ void staged_reduce(uint32_t part_a, int rb, int t_lo, int ng, int gpt, int et, int nthr,
                                              RowOf&& row_of, Need&& need, Emit&& emit) {
    constexpr int U = NSP >= 8 ? 1 : 8 / NSP;
    for (int g0 = et; g0 < ng; g0 += nthr * U) {
        float4 q[U][NSP];
        bool ok[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int g = g0 + nthr * u;
            ok[u] = g < ng && need(t_lo + g / gpt, g % gpt);
            if (ok[u]) {
                const int t = t_lo + g / gpt;
                const uint32_t off = part_a + (uint32_t)((t * rb + row_of(g % gpt)) * 4);
                if (NSP == 1) {
                    q[u][0] = ld_shared_f4(off);
                } else {
#pragma unroll
                    for (int sp = 0; sp < NSP; ++sp) q[u][sp] = ld_cluster_f4(map_cluster(off, (uint32_t)sp));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int g = g0 + nthr * u;
            if (g < ng) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ok[u]) {
                    acc = q[u][0];
#pragma unroll
                    for (int sp = 1; sp < NSP; ++sp) {
                        acc.x += q[u][sp].x;
                        acc.y += q[u][sp].y;
                        acc.z += q[u][sp].z;
                        acc.w += q[u][sp].w;
                    }
                }
                emit(t_lo + g / gpt, g % gpt, acc);
            }
        }
    }
}

// Two values bf16(v0 * sc), bf16(v1 * sc) (v0 in the low half): the products in fp32,
// one rounding each, two lanes per instruction; with bias, v = f + bias first (exact
// for the code floats below).
__device__ __forceinline__ uint32_t scaled_pair_bf16(uint32_t f0, uint32_t f1, float bias, float sc) {
    uint32_t r;
    asm("{\n\t.reg .b64 t, b, s;\n\t.reg .f32 lo, hi;\n\t"
        "mov.b64 t, {%1, %2};\n\t"
        "mov.b64 b, {%3, %3};\n\t"
        "mov.b64 s, {%4, %4};\n\t"
        "add.rn.f32x2 t, t, b;\n\t"
        "mul.rn.f32x2 t, t, s;\n\t"
        "mov.b64 {lo, hi}, t;\n\t"
        "cvt.rn.bf16x2.f32 %0, hi, lo;\n\t}"
        : "=r"(r)
        : "r"(f0), "r"(f1), "f"(bias), "f"(sc));
    return r;
}
__device__ __forceinline__ uint32_t scaled_pair_bf16(float2 v, float sc) {
    uint32_t r;
    asm("{\n\t.reg .b64 t, s;\n\t.reg .f32 lo, hi;\n\t"
        "mov.b64 t, {%1, %2};\n\t"
        "mov.b64 s, {%3, %3};\n\t"
        "mul.rn.f32x2 t, t, s;\n\t"
        "mov.b64 {lo, hi}, t;\n\t"
        "cvt.rn.bf16x2.f32 %0, hi, lo;\n\t}"
        : "=r"(r)
        : "f"(v.x), "f"(v.y), "f"(sc));
    return r;
}

// One row of a stage's W tile restored from its codes: 64 columns of bf16(code value *
// scale) -- the value and the single rounding of the restore kernels -- written as the
// 128-byte row `row` of a K-major tile with the 128-byte swizzle (16-byte chunk j of the
// row at position j ^ (row % 8)), the layout a TMA load of a bf16 W tile leaves.  The
// 16-byte reads start at a row-dependent chunk to spread shared-memory banks.
// int8: the code byte c becomes the float 2^23 + 128 + c by a byte permutation (its
// low mantissa bits), and c exactly by subtracting 2^23 + 128.  NF4: the row's 16
// restored values bf16(codebook[i] * scale) are formed once per K block and kept as
// byte tables in registers (low bytes, high bytes); byte permutations then look up
// four codes at a time, no per-code arithmetic and no memory access.
// 16 int8 codes -> 16 restored bf16 values (8 pairs, column order)
__device__ __forceinline__ void int8_group_bf16(const uint4& raw, float sc, uint32_t (&w)[8]) {
    const uint32_t wd[4] = {raw.x ^ 0x80808080u, raw.y ^ 0x80808080u, raw.z ^ 0x80808080u,
                            raw.w ^ 0x80808080u};   // bytes c + 128
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t f0 = __byte_perm(wd[e], 0x4B000000u, 0x7540), f1 = __byte_perm(wd[e], 0x4B000000u, 0x7541);
        const uint32_t f2 = __byte_perm(wd[e], 0x4B000000u, 0x7542), f3 = __byte_perm(wd[e], 0x4B000000u, 0x7543);
        w[2 * e] = scaled_pair_bf16(f0, f1, -8388736.f, sc);
        w[2 * e + 1] = scaled_pair_bf16(f2, f3, -8388736.f, sc);
    }
}

__device__ __forceinline__ void restore_row(const uint8_t* codes, uint8_t* arow, int row, float sc, int qmode,
                                            const float* qcb) {
    const int sw = row & 7;
    if (qmode == QMODE_INT8) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int j = (jj + row) & 3;   // codes of columns 16j .. 16j+15
            const uint4 raw = *reinterpret_cast<const uint4*>(codes + 16 * j);
            uint32_t w[8];
            int8_group_bf16(raw, sc, w);
            *reinterpret_cast<uint4*>(arow + (((2 * j) ^ sw) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(arow + (((2 * j + 1) ^ sw) * 16)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
    } else {
        uint32_t lo_t[4], hi_t[4];   // lo_t[j] byte e: low byte of value 4j + e; hi_t: high bytes
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 c4 = reinterpret_cast<const float4*>(qcb)[j];
            const uint32_t p0 = scaled_pair_bf16(make_float2(c4.x, c4.y), sc);
            const uint32_t p1 = scaled_pair_bf16(make_float2(c4.z, c4.w), sc);
            lo_t[j] = __byte_perm(p0, p1, 0x6420);
            hi_t[j] = __byte_perm(p0, p1, 0x7531);
        }
        // the values of four codes given one per byte (0..15): their low and high bytes
        auto lookup4 = [&](uint32_t nb, uint32_t& lob, uint32_t& hib) {
            const uint32_t v = nb & 0x07070707u;
            const uint32_t sel = __byte_perm(v | (v >> 4), 0u, 0x0020);   // nibble k: code k mod 8
            const uint32_t m = ((nb >> 3) & 0x01010101u) * 0xFFu;         // byte k all ones: code k >= 8
            lob = (__byte_perm(lo_t[0], lo_t[1], sel) & ~m) | (__byte_perm(lo_t[2], lo_t[3], sel) & m);
            hib = (__byte_perm(hi_t[0], hi_t[1], sel) & ~m) | (__byte_perm(hi_t[2], hi_t[3], sel) & m);
        };
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int j = (jj + row) & 1;   // codes of columns 32j .. 32j+31, two per byte
            const uint4 raw = *reinterpret_cast<const uint4*>(codes + 16 * j);
            const uint32_t b4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // 16-byte chunk 4j + q: columns 32j + 8q .. +7
                uint32_t le, he, lo, ho;   // even columns (low nibbles), odd columns (high nibbles)
                lookup4(b4[q] & 0x0F0F0F0Fu, le, he);
                lookup4((b4[q] >> 4) & 0x0F0F0F0Fu, lo, ho);
                const uint32_t t1 = __byte_perm(le, he, 0x5140), t2 = __byte_perm(lo, ho, 0x5140);   // columns 0,2 / 1,3
                const uint32_t t3 = __byte_perm(le, he, 0x7362), t4 = __byte_perm(lo, ho, 0x7362);   // columns 4,6 / 5,7
                *reinterpret_cast<uint4*>(arow + (((4 * j + q) ^ sw) * 16)) =
                    make_uint4(__byte_perm(t1, t2, 0x5410), __byte_perm(t1, t2, 0x7632), __byte_perm(t3, t4, 0x5410),
                               __byte_perm(t3, t4, 0x7632));
            }
        }
    }
}

// The int8 codes of one row over a stage's two K chunks (128 bytes: chunk 0's 64 codes,
// then chunk 1's) restored into both chunks' W rows as restore_row does, all eight
// 16-byte reads issued first (starting at a row-dependent group: conflict-free across
// 8 rows), so that one thread carries eight independent conversions.
__device__ __forceinline__ void restore_row_int8x2(const uint8_t* codes, uint8_t* arow0, uint8_t* arow1, int row,
                                                   float sc) {
    const int sw = row & 7;
    uint4 raw[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) raw[g] = *reinterpret_cast<const uint4*>(codes + 16 * ((g + row) & 7));
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const int gg = (g + row) & 7;   // chunk gg / 4, columns 16 (gg % 4) ..
        uint8_t* arow = gg < 4 ? arow0 : arow1;
        const int j = gg & 3;
        uint32_t w[8];
        int8_group_bf16(raw[g], sc, w);
        *reinterpret_cast<uint4*>(arow + (((2 * j) ^ sw) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(arow + (((2 * j + 1) ^ sw) * 16)) = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

// ---------------------------------------------------------------- the GEMM kernel
// Two CTAs per SM: a shrink CTA and a projection CTA launched behind it share an SM.
// MT: 128-row W tiles per projection CTA (1 or 2), sharing each X stage; with 2 the CTA
// owns 256 output rows, two MMAs per K slice into two accumulators (no K-extension, no
// codes, split-K through the staged cluster reduction, N <= 128).
template <bool SHRINK, int MT = 1>
__global__ void __launch_bounds__(NUM_THREADS, 2)
swapab_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmArena,
                   const __grid_constant__ CUtensorMap tmAux, GemmParams p) {
    // tmAux: over 4-bit codes, the block scales; else, with adapters, the Up arena as runs
    const CUtensorMap& tmQs = tmAux;
    const CUtensorMap& tmRun = tmAux;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Tail& tl = *reinterpret_cast<Tail*>(smem + p.tail_off);
    volatile int* abort_flag = &tl.abort_flag;
    const int NS = p.stages;
    const int B_SUB = b_bytes(p.N);                  // bytes of the B operand per K chunk
    const int A_STAGE = p.kc * p.a_sub;
    const int Q_OFF = A_STAGE + p.kc * B_SUB;        // projection over codes: the code tile [row][kc * q_x]
    // over 4-bit codes the stage also holds the K block's 128 fp32 scales
    const int QS_OFF = Q_OFF + BM * p.q_x * p.kc;    // 4-bit codes: the scales [kc][row]
    const int Q_BYTES = (BM * p.q_x + (p.qmode == QMODE_NF4 ? BM * 4 : 0)) * p.kc;   // codes (+ scales)
    // (stages start on 1024-byte swizzle atoms)
    const int SB = (!SHRINK && p.qmode) ? (Q_OFF + Q_BYTES + 1023) & ~1023 : Q_OFF;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, split = blockIdx.y, ztile = blockIdx.z;
    static_assert(MT == 1 || (!SHRINK && MT == 2), "two row tiles only in the projection");
    constexpr int RB = MT * BM;                         // output rows of this CTA
    constexpr int kStampKind = SHRINK ? STAMP_SHRINK : STAMP_PROJECTION;
    const int tok0 = ztile * p.N;                    // first token of this token tile
    const int T = min(p.T - tok0, p.N);              // tokens in this tile

    if (SHRINK) {
        if (tile == p.seg_tile) {
            // (the builder's scratch may cover the Tail: this start time stays in a register)
            const unsigned long long t_seg = (p.stamps && threadIdx.x == 0) ? gtimer() : 0ull;
            // the segment builder's column: its first CTA builds and publishes the
            // segments (and the bad-row status), the others have nothing to do.  The
            // slot table and the arguments are staged before the wait for the kernel
            // before: only the row map is read after it.
            const bool builder = split == 0 && ztile == 0;
            const seg::Scratch sc = seg::carve(reinterpret_cast<int*>(smem), p.S, p.seg_P, p.seg_stage_rows != 0);
            if (builder) seg::stage(p.slots, p.S, p.ws, p.row_adapter, p.T, p.max_chunks, sc);
            pdl_wait();
            pdl_trigger();
            if (builder) seg::build(p.S, p.seg_P, sc);
            if (threadIdx.x == 0) stamp_record(p.stamps, p.stamp_cap, t_seg, kStampKind);
            return;
        }
    }
    if (p.stamps && threadIdx.x == 0) tl.t_start = gtimer();

    const int kb0 = (int)((long long)split * p.ksteps / p.splits);
    const int kb1 = (int)((long long)(split + 1) * p.ksteps / p.splits);
    // K-extension units (EXT_SUB consecutive chunks of the table): the first LU are
    // listed per row tile (those with a chunk this tile and token tile use, divided
    // evenly over the K splits); the units past them are split by index, all kept
    constexpr int LU_CAP = EXT_CAP / EXT_SUB;
    const int LU = SHRINK ? 0 : min(p.ext_units, LU_CAP);
    const int xu = SHRINK ? 0 : p.ext_units - LU;
    const int eu0 = LU + (int)((long long)split * xu / p.splits);
    const int eu1 = LU + (int)((long long)(split + 1) * xu / p.splits);
    // pipeline steps: the din steps, with the K-extension steps inserted at `ins`; how
    // many of those run is known once the CTA's chunk list is built (info_ready)
    const int nw = kb1 - kb0;
    const int ins = max(0, nw - p.ext_lead);
    const int ne0 = LU + (eu1 - eu0);   // K-extension steps at most (exactly once listed)
    auto ext_steps = [&]() { return tl.n_ext + (eu1 - eu0); };
    auto ext_unit_at = [&](int e) { return e < tl.n_ext ? tl.ext_slot[tl.ext_first + e] : eu0 + (e - tl.n_ext); };
    const int acc_cols = MT * p.N;   // TMEM columns of the accumulators (MT of N columns)
    const uint32_t ncols = acc_cols <= 32 ? 32 : (acc_cols <= 64 ? 64 : (acc_cols <= 128 ? 128 : (acc_cols <= 256 ? 256 : 512)));

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&tl.full[s], 1);
            mbar_init(&tl.empty[s], 1);
            mbar_init(&tl.conv[s], 4);   // one arrival per converting (epilogue) warp
        }
        mbar_init(&tl.acc_full, 1);
        mbar_init(&tl.info_ready, 1);
        mbar_init(&tl.rx_bar, 1);
        tl.abort_flag = 0;
        tl.flags[0] = 0;
        tl.flags[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!SHRINK && p.push) mbar_expect_tx(&tl.rx_bar, (uint32_t)(BM * p.N * 4));   // every split's slice
        if (!SHRINK) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
        if (!SHRINK && p.qmode == QMODE_NF4) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmQs) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
        if (SHRINK || p.ext_units > 0) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmArena) : "memory");
        if (!SHRINK && p.run_b > 0) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmRun) : "memory");
    }
    if (!SHRINK && p.qmode == QMODE_NF4 && threadIdx.x < 16)   // the codebook of the 4-bit restore
        reinterpret_cast<float*>(smem + p.qtab_off)[threadIdx.x] = p.qcb[threadIdx.x];
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tl.tmem_slot)),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (SHRINK) {
        // Launched while the stream's previous kernel may still run (it may produce X
        // or the row map, or read the Vt this kernel overwrites): wait for it here,
        // after the set-up, then let the projection launch and stream W meanwhile.
        pdl_wait();
        pdl_trigger();
    }
    // (the projection lets the next kernel launch once its last MMA is issued: CTAs of
    // the next forward that got resident earlier would only wait, holding the shared
    // memory and registers that this kernel's later CTAs need)
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
        ChunkRec cr{-2, 0, 0, 0.f, 0, 0};
        if (lane < CHUNKS_PER_TILE && cb + lane < p.n_chunks) cr = p.chunks[cb + lane];
        // the table is in arena order within the tile (window mode): the window of the
        // tile starts at its first chunk
        const int u0 = __shfl_sync(0xffffffffu, cr.unit, 0);
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
            tl.my_off[k] = p.window ? cr.unit - u0 : k * CHUNK;   // first accumulator row of the chunk
            tl.my_kval[k] = cr.kval;
            tl.my_scale[k] = cr.scale;
        }
        if (lane == 0) {
            tl.tile_chunks = __popc(m);
            tl.win_u0 = u0;
        }
        if (p.tmask && split == 0 && lane < CHUNKS_PER_TILE && cb + lane < p.n_chunks)
            p.tmask[(size_t)ztile * p.max_chunks + cb + lane] = (uint8_t)((m >> lane) & 1u);
    }
    // A block barrier needs converged warps: lanes that skipped a one-thread branch
    // above (barrier set-up, the TMA and MMA roles) wait here for it first.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tl.tmem_slot;
    const int tile_chunks = SHRINK ? tl.tile_chunks : 0;
    // push reduction: this CTA's receive barrier is set up (the epilogues wait for all;
    // the mbarrier-init fence above orders it)
    if (!SHRINK && p.push) cluster_arrive_relaxed();
    if (SHRINK && tile_chunks <= 0) {   // no token of the token tile uses a chunk of this row tile
        if (warp == 1) {
            __syncwarp();
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
        }
        if (threadIdx.x == 0) stamp_record(p.stamps, p.stamp_cap, tl.t_start, kStampKind);
        return;
    }

    if (warp == 2 && !SHRINK && LU > 0) {
        // While the producer streams W: the slots the batch uses, then the listed
        // K-extension chunks, the arena unit of each chunk whose slot is used and whose
        // rows meet this tile, -1 for the others (never loaded).  The producer waits for
        // it at its first K-extension step.
        int av[MAX_N / 32];
#pragma unroll
        for (int i = 0; i < MAX_N / 32; ++i) {
            const int t = lane + 32 * i;
            av[i] = t < T ? p.row_adapter[tok0 + t] : -1;
        }
        const int nx = LU * EXT_SUB;
#pragma unroll
        for (int it = 0; it < EXT_CAP / 32; ++it) {   // (all records requested at once)
            const int k = lane + 32 * it, c = k;
            if (k >= nx) continue;
            int sl = -1, un = -1;
            if (c < p.n_chunks) {
                const ChunkRec cr = p.chunks[c];
                sl = cr.slot;
                // a chunk of a module whose rows miss this tile adds nothing here
                un = (cr.row0 < (tile + 1) * BM && cr.row1 > tile * BM) ? cr.unit : -1;
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
            if (tl.ext_unit[k] >= 0 && (sl < 0 || !((tl.slot_bits[sl >> 5] >> (sl & 31)) & 1u)))
                tl.ext_unit[k] |= UNUSED;
        }
        __syncwarp();
        // The tile's K-extension steps: only the listed units with a chunk to multiply
        // (a step with nothing to load would still cost a pipeline round trip), in
        // table order, this split taking its share of them.
        int n_all = 0;
        for (int u0 = 0; u0 < LU; u0 += 32) {
            const int uu = u0 + lane;
            bool any = false;
            if (uu < LU)
#pragma unroll
                for (int j = 0; j < EXT_SUB; ++j) any |= used_unit(tl.ext_unit[uu * EXT_SUB + j]) >= 0;
            const unsigned m = __ballot_sync(0xffffffffu, any);
            __syncwarp();   // (the list overwrites the slot ids read above)
            if (any) tl.ext_slot[n_all + __popc(m & ((1u << lane) - 1u))] = uu;
            n_all += __popc(m);
        }
        {
            // this split's steps, each with its unit and its chunks' arena units in one
            // 16-byte entry: the producer reads one entry per step instead of a chain
            const int f0 = (int)((long long)split * n_all / p.splits);
            const int n_my = (int)((long long)(split + 1) * n_all / p.splits) - f0;
            for (int e = lane; e < n_my; e += 32) {
                const int uu = tl.ext_slot[f0 + e];
                tl.ext_plan[e] = make_int4(used_unit(tl.ext_unit[uu * EXT_SUB]), used_unit(tl.ext_unit[uu * EXT_SUB + 1]),
                                           used_unit(tl.ext_unit[uu * EXT_SUB + 2]),
                                           used_unit(tl.ext_unit[uu * EXT_SUB + 3]));
                // a run: all 4 chunks in the table and in this tile's module, at the stride
                // of the run map, inside it (chunks the batch does not use are loaded too,
                // and not multiplied)
                int r0 = -1;
                if (p.run_b > 0) {
                    int cu[EXT_SUB];
                    bool ok = true;
#pragma unroll
                    for (int j = 0; j < EXT_SUB; ++j) {
                        const int v = tl.ext_unit[uu * EXT_SUB + j];
                        cu[j] = v & ~UNUSED;
                        ok = ok && v >= 0;
                    }
                    const int b0 = cu[0] >> 3;
#pragma unroll
                    for (int j = 1; j < EXT_SUB; ++j) ok = ok && cu[j] - cu[0] == j * 8 * p.run_b;
                    ok = ok && (cu[0] & 7) == 0 && b0 % p.run_b + 2 <= p.run_b && b0 / p.run_b + EXT_SUB <= p.run_groups;
                    if (ok) r0 = cu[0];
                }
                tl.ext_plan_u[e] = uu | ((r0 + 1) << 8);
            }
            if (lane == 0) {
                tl.ext_first = f0;
                tl.n_ext = n_my;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_expect_tx(&tl.info_ready, 0);
    }

    // epilogue warps: the TMEM lane quarter a warp may access, its row of the tile, and
    // whether the accumulator holds this CTA's products (else it counts as zero)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
    bool have = false;
    // projection: final write of rows r0..r0+3 (a multiple of 4) of token t
    auto emit4 = [&](int t, int r0, const float4& v) {
        const int o0 = tile * RB + r0;
        __nv_bfloat16* y = p.Y + (size_t)(tok0 + t) * p.dout + o0;
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
    };
    // the K splits sum their partial tiles by staging them in shared memory
    const bool staged = SHRINK || (p.splits > 1 && !p.push && p.cluster);

    if (warp == 0 && lane == 0) {
        // ---------------- producer: TMA loads into the stage ring
        int s = 0;
        uint32_t ph = 0;
        bool waited = false;
        int issued = 0;   // steps whose loads went out
        if (!SHRINK && p.xwait) {
            // Launched while the kernel before may still run (it may produce X): the W
            // tiles of the first stages go out now, their X tiles once it has completed.
            const int pre = min(NS, max(0, (kb1 - kb0) - p.ext_lead));
            for (int i = 0; i < pre; ++i) {
                uint8_t* a = smem + (size_t)i * SB;
                tl.stage_kind[i] = -1;
                if (p.qmode) {
                    mbar_expect_tx_only(&tl.full[i], (uint32_t)Q_BYTES);
                    tma_2d(a + Q_OFF, &tmW, &tl.full[i], (kb0 + i) * p.kc * p.q_x, tile * BM);
                    if (p.qmode == QMODE_NF4) tma_2d(a + QS_OFF, &tmQs, &tl.full[i], tile * BM, (kb0 + i) * p.kc);
                } else {
                    mbar_expect_tx_only(&tl.full[i], (uint32_t)A_STAGE);
                    if (p.kc > 1) tma_3d(a, &tmW, &tl.full[i], 0, tile * RB, (kb0 + i) * p.kc);
                    else tma_2d(a, &tmW, &tl.full[i], (kb0 + i) * BK, tile * RB);
                }
            }
            pdl_wait();
            for (int i = 0; i < pre; ++i) {
                uint8_t* b = smem + (size_t)i * SB + A_STAGE;
                mbar_expect_tx(&tl.full[i], (uint32_t)(p.kc * B_SUB));
                if (p.kc > 1) tma_3d(b, &tmX, &tl.full[i], 0, tok0, (kb0 + i) * p.kc);
                else tma_2d(b, &tmX, &tl.full[i], (kb0 + i) * BK, tok0);
            }
            issued = pre;
            s = pre % NS;
            ph = pre == NS ? 1u : 0u;
        }
        int ne = ne0;   // K-extension steps (an upper bound until listed)
        for (; issued < nw + ne; ++issued) {
            const int i = issued;
            if (!mbar_wait(&tl.empty[s], ph ^ 1, abort_flag, p.status)) break;
            uint8_t* a = smem + (size_t)s * SB;
            uint8_t* b = a + A_STAGE;
            // din steps, with the K-extension steps placed EXT_LEAD steps before the end
            // so that their Vt loads overlap the last W tiles
            if (i == ins && LU > 0) {
                if (!mbar_wait(&tl.info_ready, 0, abort_flag, p.status)) break;
                ne = ext_steps();
                if (i == nw + ne) break;   // nothing left: no K-extension step, no din step after
            }
            const bool ext = i >= ins && i < ins + ne;
            const int kb = kb0 + (i < ins ? i : i - ne);
            if (SHRINK) {
                tl.stage_kind[s] = -1;
                if (p.window) {
                    // one box each: win_rows arena rows x kc K chunks of Down, N tokens x kc K chunks of X
                    mbar_expect_tx(&tl.full[s], (uint32_t)SB);
                    tma_3d(a, &tmArena, &tl.full[s], 0, tl.win_u0, kb * p.kc);
                    tma_3d(b, &tmX, &tl.full[s], 0, tok0, kb * p.kc);
                } else {
                    mbar_expect_tx(&tl.full[s], (uint32_t)(tile_chunks * CHUNK_BYTES + B_SUB));
                    for (int j = 0; j < tile_chunks; ++j)
                        tma_2d(a + j * CHUNK_BYTES, &tmArena, &tl.full[s], kb * BK, tl.my_unit[j]);
                    tma_2d(b, &tmX, &tl.full[s], kb * BK, tok0);
                }
            } else if (!ext && p.qmode) {
                // the code tile and X; the epilogue warps restore the bf16 W tile from the codes
                tl.stage_kind[s] = -1;
                mbar_expect_tx(&tl.full[s], (uint32_t)(Q_BYTES + p.kc * B_SUB));
                tma_2d(a + Q_OFF, &tmW, &tl.full[s], kb * p.kc * p.q_x, tile * BM);
                if (p.qmode == QMODE_NF4) tma_2d(a + QS_OFF, &tmQs, &tl.full[s], tile * BM, kb * p.kc);
                if (p.kc > 1) tma_3d(b, &tmX, &tl.full[s], 0, tok0, kb * p.kc);
                else tma_2d(b, &tmX, &tl.full[s], kb * BK, tok0);
            } else if (!ext) {
                tl.stage_kind[s] = -1;
                mbar_expect_tx(&tl.full[s], (uint32_t)SB);
                if (p.kc > 1) {   // kc K chunks of W (128 rows) and of X (N tokens), one box each
                    tma_3d(a, &tmW, &tl.full[s], 0, tile * RB, kb * p.kc);
                    tma_3d(b, &tmX, &tl.full[s], 0, tok0, kb * p.kc);
                } else {
                    tma_2d(a, &tmW, &tl.full[s], kb * BK, tile * RB);
                    tma_2d(b, &tmX, &tl.full[s], kb * BK, tok0);
                }
            } else {
                const int e = i - ins;
                int u, un[EXT_SUB], run0 = -1;
                uint32_t mask = 0;
                if (e < tl.n_ext) {   // a listed step: its entry of the plan
                    const int4 pl = tl.ext_plan[e];
                    const int pu = tl.ext_plan_u[e];
                    u = pu & 0xFF;
                    run0 = (pu >> 8) - 1;
                    un[0] = pl.x;
                    un[1] = pl.y;
                    un[2] = pl.z;
                    un[3] = pl.w;
                } else {              // a unit past the listed ones (split by index)
                    u = ext_unit_at(e);
#pragma unroll
                    for (int j = 0; j < EXT_SUB; ++j) {
                        const int c = u * EXT_SUB + j;
                        int v = -1;
                        if (c < p.n_chunks) {
                            const ChunkRec cr = p.chunks[c];
                            if (((tl.slot_bits[cr.slot >> 5] >> (cr.slot & 31)) & 1u) && cr.row0 < (tile + 1) * BM &&
                                cr.row1 > tile * BM)
                                v = cr.unit;
                        }
                        un[j] = v;
                    }
                }
#pragma unroll
                for (int j = 0; j < EXT_SUB; ++j)
                    if (un[j] >= 0) mask |= 1u << j;
                tl.stage_kind[s] = (int)mask;
                if (mask == 0) {
                    mbar_expect_tx(&tl.full[s], 0);
                } else {
                    // Up tiles (two blocks of 8 rank columns x 128 rows) are the pool's own
                    // data: issue them before waiting for the shrink, then its Vt.  A run's
                    // 4 chunks are one box (the same layout: chunk j at j x 4 KiB)
                    if (run0 >= 0) {
                        mbar_expect_tx_only(&tl.full[s], (uint32_t)(EXT_SUB * (BM * 32)));
                        tma_4d(a, &tmRun, &tl.full[s], 0, tile * BM / 8, (run0 >> 3) % p.run_b, (run0 >> 3) / p.run_b);
                    } else {
                        mbar_expect_tx_only(&tl.full[s], (uint32_t)(__popc(mask) * (BM * 32)));
#pragma unroll
                        for (int j = 0; j < EXT_SUB; ++j)
                            if ((mask >> j) & 1u)
                                tma_3d(a + j * (BM * 32), &tmArena, &tl.full[s], 0, tile * BM / p.up_rows, un[j] >> 3);
                    }
                    if (!waited) {
                        if (p.pdl) pdl_wait();   // Vt comes from the shrink
                        waited = true;
                    }
                    mbar_expect_tx(&tl.full[s], (uint32_t)B_SUB);
                    tma_3d(b, &tmV, &tl.full[s], 0, tok0 / 8, u * EXT_SUB * 2);
                }
            }
            if (++s == NS) {
                s = 0;
                ph ^= 1;
            }
        }
        if (*abort_flag) {
            // let loads already issued land before the CTA's shared memory goes away:
            // step i filled stage i % NS in its phase (i / NS) & 1
            for (int j = 0; j < NS && j < issued; ++j) {
                const int fills = (issued - 1 - j) / NS + 1;
                const long long t0 = clock64();
                while (!mbar_try_wait(&tl.full[j], (uint32_t)((fills - 1) & 1)) && clock64() - t0 < 200000000ll) {
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        const uint32_t idesc = idesc_bf16(BM, p.N);
        int s = 0;
        uint32_t ph = 0;
        uint32_t acc = 0;
        uint32_t cph = 0;   // over codes: parity of each stage's next conversion
        int ne_m = ne0;
        for (int i = 0; i < nw + ne_m; ++i) {
            if (i == ins && LU > 0) {   // as many K-extension steps as the producer issues
                if (!mbar_wait(&tl.info_ready, 0, abort_flag, p.status)) break;
                ne_m = ext_steps();
                if (i == nw + ne_m) break;
            }
            const bool din_step = !(i >= ins && i < ins + ne_m);
            if (!SHRINK && p.qmode && din_step) {
                // the epilogue warps saw the stage land and restored its W tile from the codes
                if (!mbar_wait(&tl.conv[s], (cph >> s) & 1u, abort_flag, p.status)) break;
                cph ^= 1u << s;
            } else if (!mbar_wait(&tl.full[s], ph, abort_flag, p.status)) {
                break;
            }
            tc_fence_after();
            const uint32_t a = smem_u32(smem + (size_t)s * SB);
            const uint32_t b = a + A_STAGE;
            const int kind = (!SHRINK && p.qmode && din_step) ? -1 : tl.stage_kind[s];
            if (kind < 0) {
                // each K chunk: A spans 128 rows (16 KiB) from its sub-block; in the shrink,
                // rows past the loaded ones hold whatever lies there and give accumulator
                // rows nobody reads
                for (int kc = 0; kc < p.kc; ++kc) {
                    const uint32_t ak = a + kc * p.a_sub, bk = b + kc * B_SUB;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        // tile u's rows follow tile u-1's in the W box (128-row blocks of
                        // the 128-byte swizzle); each accumulator starts fresh on its first MMA
#pragma unroll
                        for (int u = 0; u < MT; ++u)
                            mma_bf16(tmem + (uint32_t)(u * p.N), sdesc(ak + u * A_BYTES + k * 32, 1024, SW128),
                                     sdesc(bk + k * 32, 1024, SW128), idesc, acc);
                        acc = 1;
                    }
                }
            } else {
                // Up chunk: [2 blocks of 8 columns][128 rows][16 B], Vt chunk: [2 blocks of 8
                // columns][N tokens][16 B]; no swizzle (K-direction core matrices 128 or N rows
                // x 16 bytes apart, M/N-direction 128 bytes)
#pragma unroll
                for (int j = 0; j < EXT_SUB; ++j)
                    if ((kind >> j) & 1) {
                        mma_bf16(tmem, sdesc_lbo(a + j * (BM * 32), BM * 16, 128, SW_NONE),
                                 sdesc_lbo(b + j * (p.N * 32), p.N * 16, 128, SW_NONE), idesc, acc);
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
        if (!SHRINK) pdl_trigger();
        if (*abort_flag) {   // MMAs already issued must finish before TMEM is released
            const long long t0 = clock64();
            while (!mbar_try_wait(&tl.acc_full, 0) && clock64() - t0 < 200000000ll) {
            }
        }
    } else if (warp >= 2) {
        if (!SHRINK && p.qmode) {
            // ---------------- over codes: restore each din step's W tile (row `row` per
            // thread) once its codes land, then release the stage to the MMA warp
            const int o = tile * BM + row;
            const float row_sc = (p.qmode == QMODE_INT8 && o < p.dout) ? __ldg(p.qscale + o) : 0.f;
            int ne_c = ne0;
            int s = 0;
            uint32_t ph = 0;
            for (int i = 0; i < nw + ne_c; ++i) {
                if (i == ins && LU > 0) {   // the stages the K-extension steps take
                    if (!mbar_wait(&tl.info_ready, 0, abort_flag, p.status)) break;
                    ne_c = ext_steps();
                    if (i == nw + ne_c) break;
                }
                if (!(i >= ins && i < ins + ne_c)) {
                    // every din step is waited for in order (the MMA waits for this warp's
                    // release), so the parity never runs a phase ahead
                    const bool got = mbar_wait(&tl.full[s], ph, abort_flag, p.status);
                    __syncwarp();
                    if (!__all_sync(0xffffffffu, got)) break;
                    uint8_t* stg = smem + (size_t)s * SB;
                    if (p.qmode == QMODE_INT8 && p.kc == 2) {   // both K chunks of the stage at once
                        restore_row_int8x2(stg + Q_OFF + row * 2 * p.q_x, stg + row * 128, stg + p.a_sub + row * 128, row,
                                           row_sc);
                    } else {
                        for (int j = 0; j < p.kc; ++j) {   // the stage's K chunks
                            // (4-bit codes: the row's scale of this K block came with the codes)
                            const float sc =
                                p.qmode == QMODE_NF4 ? reinterpret_cast<const float*>(stg + QS_OFF)[j * BM + row] : row_sc;
                            restore_row(stg + Q_OFF + (row * p.kc + j) * p.q_x, stg + j * p.a_sub + row * 128, row, sc,
                                        p.qmode, reinterpret_cast<const float*>(smem + p.qtab_off));
                        }
                    }
                    fence_proxy_async_smem();   // the MMA (async proxy) reads what these threads wrote
                    __syncwarp();
                    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&tl.conv[s]))
                                                : "memory");
                }
                if (++s == NS) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
        // ---------------- epilogue: TMEM -> partial tile, or the final values
        const bool ok = mbar_wait(&tl.acc_full, 0, abort_flag, p.status);
        __syncwarp();   // reconverge: lanes may leave the wait loop apart; tcgen05.ld is warp-collective
        tc_fence_after();
        have = __all_sync(0xffffffffu, ok) && tl.flags[0] != 0;

        if (!SHRINK && p.splits == 1) {
            const int o = tile * BM + row;
            for (int t0 = 0; t0 < T; t0 += 16) {
                float v[16];
                if (have) tmem_ld16(tbase + t0, v);
                else
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                if (o < p.dout)
                    for (int j = 0; j < 16 && t0 + j < T; ++j)
                        p.Y[(size_t)(tok0 + t0 + j) * p.dout + o] = __float2bfloat16_rn(v[j]);
            }
        } else if (!SHRINK && p.push) {
            // Push reduction.  Stage this split's partial tile [token][row] in its idle
            // ring: the tokens of split j's slice are then one contiguous block, which
            // one bulk copy sends into CTA j's receive buffer [src][token][row],
            // signalling j's receive barrier.  Each CTA then sums its own slice over the
            // sources in split order and writes it.  A second cluster barrier keeps
            // every CTA alive until all the copies out of its shared memory have landed.
            const int ts = p.N / p.splits;
            const uint32_t me = cluster_rank();
            float* part_s = reinterpret_cast<float*>(smem);
            for (int t0 = 0; t0 < p.N; t0 += 16) {
                float v[16];
                if (have) tmem_ld16(tbase + t0, v);
                else
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) part_s[(t0 + j) * BM + row] = v[j];
            }
            fence_proxy_async_smem();
            __syncwarp();
            epi_bar();
            cluster_wait();   // every CTA of the cluster has set up its receive barrier
            const uint32_t rx_a = smem_u32(smem + p.rx_off);
            const uint32_t slice = (uint32_t)(ts * BM * 4);
            if (threadIdx.x == 64)
                for (int j = 0; j < p.splits; ++j)
                    bulk_s2s(map_cluster(rx_a + me * slice, (uint32_t)j), smem_u32(part_s) + (uint32_t)j * slice, slice,
                             map_cluster(smem_u32(&tl.rx_bar), (uint32_t)j));
            mbar_wait(&tl.rx_bar, 0, abort_flag, p.status);
            __syncwarp();
            cluster_arrive();   // every copy into this CTA has landed
            const int et = threadIdx.x - 64;
            for (int g = et; g < ts * (BM / 4); g += 128) {
                const int t = g / (BM / 4), r0 = (g % (BM / 4)) * 4;
                float4 acc = ld_shared_f4(rx_a + (uint32_t)((t * BM + r0) * 4));
                for (int src = 1; src < p.splits; ++src) {
                    const float4 q4 = ld_shared_f4(rx_a + src * slice + (uint32_t)((t * BM + r0) * 4));
                    acc.x += q4.x;
                    acc.y += q4.y;
                    acc.z += q4.z;
                    acc.w += q4.w;
                }
                if ((int)me * ts + t < T) emit4((int)me * ts + t, r0, acc);
            }
            __syncwarp();
            cluster_wait();   // ... and into every other CTA: the copies out of this one are done
        } else if (!SHRINK && !p.cluster) {
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
    if (warp < 2 && !SHRINK && p.push) {   // the epilogue warps' two split cluster barriers
        __syncwarp();
        cluster_wait();
        cluster_arrive();
        cluster_wait();
    }
    if (staged && (warp >= 2 || p.splits > 1)) {
        // Staged reduction: each split stages its partial tile [token][row] in its
        // own shared memory (the ring is idle: every load has been consumed by the
        // finished MMAs), then, after a barrier (over the cluster when the splits
        // form one), sums one slice of tokens over the shared memory of all splits,
        // in split order, and writes it.  Passes of tp tokens when the whole tile
        // does not fit the ring.  The shrink stages only the rows of its window
        // (or of its chunks) and writes each used chunk's 16 columns of Vt, in
        // groups of 4: the row's value for this chunk's own rank columns (scaled,
        // for the tokens of the chunk's adapter), zero elsewhere.  Across a cluster,
        // warps 0 and 1 (done with the loads and the MMAs) share the sums.
        __syncwarp();   // lane 0 of warps 0 and 1 ran its role alone
        float* part_s = reinterpret_cast<float*>(smem);
        const uint32_t part_a = smem_u32(part_s);
        const bool multi = p.splits > 1;
        const int tp = min(p.N, (p.ring_bytes / (RB * 4)) & ~15);
        const int rows = SHRINK ? (p.window ? p.win_rows : tile_chunks * CHUNK) : BM;
        const int gpt = SHRINK ? tile_chunks * 4 : RB / 4;   // groups of 4 rows per token
        const int et = multi ? (int)threadIdx.x : (int)threadIdx.x - 64;
        const int nthr = multi ? NUM_THREADS : 128;
        auto row_of = [&](int gi) { return SHRINK ? tl.my_off[gi >> 2] + (gi & 3) * 4 : gi * 4; };
        for (int p0 = 0; p0 < T; p0 += tp) {
            const int pt = min(tp, T - p0);
            if (warp >= 2 && q * 32 < rows)
#pragma unroll
                for (int u = 0; u < MT; ++u)   // accumulator u holds rows u * 128 + row
                    for (int t0 = 0; t0 < pt; t0 += 16) {
                        float v[16];
                        if (have) tmem_ld16(tbase + (uint32_t)(u * p.N) + p0 + t0, v);
                        else
                            for (int j = 0; j < 16; ++j) v[j] = 0.f;
#pragma unroll
                        for (int j = 0; j < 16; ++j) part_s[(t0 + j) * RB + u * BM + row] = v[j];
                    }
            __syncwarp();
            if (multi) cluster_sync();
            else epi_bar();
            const int ts = (pt + p.splits - 1) / p.splits;
            const int t_lo = multi ? (int)cluster_rank() * ts : 0;
            const int t_hi = min(pt, t_lo + ts);
            const int ng = t_hi > t_lo ? (t_hi - t_lo) * gpt : 0;
            // the shrink keeps a chunk's values only for the tokens of the chunk's adapter
            // (the others are written as zeros): their sums need no loads
            auto need = [&](int t, int gi) { return !SHRINK || tl.tile_ra[p0 + t] == tl.my_slot[gi >> 2]; };
            auto emit_g = [&](int t, int gi, const float4& v) {
                if (SHRINK) {
                    const int k = gi >> 2, j0 = (gi & 3) * 4;
                    const int kval = tl.my_kval[k];
                    const float sc = tl.tile_ra[p0 + t] == tl.my_slot[k] ? tl.my_scale[k] : 0.f;
                    __nv_bfloat162 lo = __floats2bfloat162_rn(j0 < kval ? sc * v.x : 0.f,
                                                              j0 + 1 < kval ? sc * v.y : 0.f);
                    __nv_bfloat162 hi = __floats2bfloat162_rn(j0 + 2 < kval ? sc * v.z : 0.f,
                                                              j0 + 3 < kval ? sc * v.w : 0.f);
                    uint2 w;
                    w.x = *reinterpret_cast<uint32_t*>(&lo);
                    w.y = *reinterpret_cast<uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(p.vt + (((size_t)tl.my_c[k] * 2 + (j0 >> 3)) * p.tcap + tok0 + p0 + t) * 8 +
                                              (j0 & 7)) = w;
                } else {
                    emit4(p0 + t, gi * 4, v);
                }
            };
            if (p.splits == 1) staged_reduce<1>(part_a, RB, t_lo, ng, gpt, et, nthr, row_of, need, emit_g);
            else if (p.splits == 2) staged_reduce<2>(part_a, RB, t_lo, ng, gpt, et, nthr, row_of, need, emit_g);
            else if (p.splits == 3) staged_reduce<3>(part_a, RB, t_lo, ng, gpt, et, nthr, row_of, need, emit_g);
            else if (p.splits == 4) staged_reduce<4>(part_a, RB, t_lo, ng, gpt, et, nthr, row_of, need, emit_g);
            else if (p.splits == 6) staged_reduce<6>(part_a, RB, t_lo, ng, gpt, et, nthr, row_of, need, emit_g);
            else staged_reduce<8>(part_a, RB, t_lo, ng, gpt, et, nthr, row_of, need, emit_g);
            __syncwarp();
            // no CTA refills or leaves while the others still read its shared memory
            if (multi) cluster_sync();
            else epi_bar();
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
    if (threadIdx.x == 0) stamp_record(p.stamps, p.stamp_cap, tl.t_start, kStampKind);
}

}  // namespace

// ---------------------------------------------------------------- host side
namespace {

// Shared-memory budgets of the rings.  A decode projection takes PROJ_SMEM_BUDGET
// (one CTA per SM) or PROJ_SMEM_BUDGET_2 (two per SM).  The decode shrink launched
// before it either runs on the SMs that the projection leaves idle (a few row tiles:
// SHRINK_SMEM_BUDGET_APART) or shares SMs with it, both rings then sized to fit one
// SM's 228 KiB together with their tails (PROJ_ and SHRINK_SMEM_BUDGET_SHARED).
// Otherwise (prefill, two projection CTAs per SM) the shrink takes SHRINK_SMEM_BUDGET.
// A projection with no shrink in its forward takes PROJ_SMEM_BUDGET_ALONE when one CTA
// per SM runs: a deeper ring keeps more W (and, for wide batches, X) in flight.
constexpr int PROJ_SMEM_BUDGET = 136 * 1024;
constexpr int PROJ_SMEM_BUDGET_ALONE = 208 * 1024;
constexpr int PROJ_SMEM_BUDGET_2 = 100 * 1024;   // two projection CTAs per SM
constexpr int PROJ_SMEM_BUDGET_SHARED = 112 * 1024;
constexpr int SHRINK_SMEM_BUDGET = 84 * 1024;
constexpr int SHRINK_SMEM_BUDGET_APART = 108 * 1024;
constexpr int SHRINK_SMEM_BUDGET_SHARED = 104 * 1024;

int clamp_stages(int ns) { return ns < 2 ? 2 : (ns > MAX_STAGES ? MAX_STAGES : ns); }

// the K splits of a tile as a cluster: a power of two, at most MAX_CLUSTER
int cluster_splits(int s) {
    int c = 1;
    while (c * 2 <= s && c * 2 <= MAX_CLUSTER) c *= 2;
    return c;
}

// K splits so that row tiles x token tiles x splits fill the SMs once; through
// global memory, with the partial tiles of a tile (splits x N x 128 floats) bounded.
int k_splits(int tiles, int kb_total, int N, bool global_reduction) {
    int s = sm_count() / (tiles > 0 ? tiles : 1);
    const int cap = 1024 / (N > 0 ? N : 1);
    if (global_reduction && s > cap) s = cap;
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
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, swapab_gemm_kernel<false, 2>);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(swapab_gemm_kernel<false, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
        e = cudaFuncSetAttribute(swapab_gemm_kernel<false, 2>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(swapab_gemm_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess) e = prefill_init();
    if (e == cudaSuccess) e = gemv_init();
    if (e == cudaSuccess) e = merge_tc_init();
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
    if (!tc_encode(&m->up128, arena_up, 3, dims, strides, box128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tc_encode(&m->up256, arena_up, 3, dims, strides, box256, CU_TENSOR_MAP_SWIZZLE_NONE))
        return false;
    m->upw128 = m->up128;
    m->upw256 = m->up256;
    m->up_rows = 1;
    if (dout % 8 == 0) {
        cuuint64_t wdims[3] = {64, (cuuint64_t)dout / 8, (cuuint64_t)(units / 8)};
        cuuint64_t wstrides[2] = {128, (cuuint64_t)dout * 16};
        cuuint32_t wbox128[3] = {64, 16, 2};
        cuuint32_t wbox256[3] = {64, 32, 2};
        if (!tc_encode(&m->upw128, arena_up, 3, wdims, wstrides, wbox128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !tc_encode(&m->upw256, arena_up, 3, wdims, wstrides, wbox256, CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
        m->up_rows = 8;
    }
    return true;
}

bool tc_quantized_fits(const PoolDims& d, int T, bool nf4) {
    // 4-bit codes: the block scales come by TMA (rows of 16-byte multiples)
    return T >= 1 && T <= MAX_N && d.din % BK == 0 && (!nf4 || d.dout % 4 == 0);
}

bool tc_supported(const PoolDims& d, int T) {
    (void)d;
    return T >= 1;
}

namespace {

// Launch shape of the decode projection for N token rows per tile; `budget1` is the
// ring budget when one CTA per SM runs.
struct DecodeShape {
    int splits;   // K splits of a tile (the cluster)
    int budget;   // shared-memory budget of the ring
    int pkc;      // K chunks of 64 per pipeline step
    int ksteps;   // pipeline steps over din
};

DecodeShape decode_shape(const PoolDims& d, int N, int budget1, int zt, int mt) {
    const int tiles = (d.dout + mt * BM - 1) / (mt * BM) * zt;   // (row tile, token tile) pairs
    auto stage_bytes = [&](int n) { return mt * A_BYTES + b_bytes(n); };
    const int kb_total = (d.din + BK - 1) / BK;
    // K splits of a tile: as many as fill the SMs with one CTA each (a power of two);
    // when that leaves a quarter of the SMs idle (few row tiles, long K), two CTAs per
    // SM with a smaller ring
    int splits = cluster_splits(k_splits(tiles, kb_total, N, false));
    int budget = budget1;
    if (tiles >= sm_count()) {
        // more row tiles than SMs (e.g. a fused gate|up of 22016 features): two CTAs
        // per SM and three K splits, so that the waves of small work units balance
        splits = kb_total < 3 ? kb_total : 3;
        budget = PROJ_SMEM_BUDGET_2;
    } else if (tiles * splits < 3 * sm_count() / 4) {
        int s2 = 2 * sm_count() / tiles;
        // clusters of s2 CTAs stay inside a GPC: filling more than nine tenths of the
        // SMs' two CTA slots leaves a cluster or two without room until the first CTAs
        // end (a second wave of a whole CTA lifetime), so take a split fewer there
        while (s2 > 1 && 10 * tiles * s2 > 9 * 2 * sm_count()) --s2;
        s2 = s2 > kb_total ? kb_total : s2;
        s2 = s2 >= 8 ? 8 : (s2 >= 6 ? 6 : (s2 >= 4 ? 4 : s2));   // cluster sizes with a reducer
        if (s2 > splits) {
            splits = s2;
            budget = PROJ_SMEM_BUDGET_2;
        }
    }
    // W and X as 3D views {64, rows, K chunks}, so that one box carries up to PROJ_KC
    // K chunks (needs din % 64 == 0): at least two stages, and three or more narrower
    // ones rather than two wide ones
    int pkc = d.din % BK == 0 ? PROJ_KC : 1;
    const int avail = budget - (N <= PUSH_MAX_N ? BM * N * 4 : 0);
    while (pkc > 1 && (2 * pkc * stage_bytes(N) > avail ||
                       (avail / (pkc * stage_bytes(N)) < 3 && avail / stage_bytes(N) >= 3)))
        --pkc;
    DecodeShape s;
    s.budget = budget;
    s.pkc = pkc;
    s.ksteps = (kb_total + pkc - 1) / pkc;
    s.splits = splits < s.ksteps ? splits : s.ksteps;
    return s;
}

}  // namespace

cudaError_t tc_forward(const TcForwardArgs& a, cudaStream_t st) {
    const PoolDims& d = a.dims;
    const int T = a.T;
    const bool decode = T <= MAX_N;
    const int kb_total = (d.din + BK - 1) / BK;
    const int n_chunks = a.lora ? a.n_chunks : 0;
    const bool shrink = n_chunks > 0;
    cudaError_t e;
    const int N = decode ? (T + 15) / 16 * 16 : 128;     // token rows per tile
    if (a.qmode && !(decode && d.din % BK == 0)) return cudaErrorInvalidValue;
    // A decode batch of more than 224 tokens runs its shrink and its projection as token
    // tiles of 128 (grid z): half the K splits per row tile, and a split's partial tile
    // half as large, for the same number of CTAs.  The token tiles of a row tile read
    // the same W slice at about the same time, so W is fetched from DRAM about once.
    // Up to 224 tokens one tile is faster: the second tile would hold few tokens and
    // take W into its SMs all the same.
    // Over codes every token tile would restore the W tile again: one tile there.  Both
    // kernels tile alike: a token tile's projection reads the Vt of exactly the chunks
    // whose slots its own tokens use, which its shrink tile wrote.
    const int q_x = a.qmode == QMODE_INT8 ? BK : (a.qmode == QMODE_NF4 ? BK / 2 : 0);   // code bytes per row and K chunk
    // over codes: a stage of QUANT_KC K chunks (codes, restored W tiles, X), and whether
    // a ring of two such stages fits shared memory at n tokens
    auto qstage = [&](int n) {
        return (QUANT_KC * (stage_bytes(n) + BM * q_x + (a.qmode == QMODE_NF4 ? BM * 4 : 0)) + 1023) & ~1023;
    };
    auto qfits = [&](int n) {
        const int rest = (n <= PUSH_MAX_N ? BM * n * 4 : 0) + 64 + (int)sizeof(Tail) + 1024;   // receive buffer, codebook
        return 2 * qstage(n) + rest <= max_dyn_smem();
    };
    const int zt = (decode && !a.qmode && N > PROJ_ZT_MIN) ? (T + PROJ_ZT_N - 1) / PROJ_ZT_N : 1;
    const int Np = zt > 1 ? PROJ_ZT_N : N;               // token rows per projection tile
    // More 128-row tiles than SMs and no adapters (the 7B layer's gate|up, 172 tiles):
    // each CTA takes two row tiles that share its X stages, so that the K splits of half
    // as many tiles fit the SMs' two CTA slots in one wave (instead of 1.7 waves), and
    // each X tile is delivered to the SMs half as often.
    int mt = (decode && !a.qmode && !shrink && Np > PUSH_MAX_N && Np <= 128 && proj_tiles(d) >= sm_count()) ? 2 : 1;
    DecodeShape ds = decode_shape(d, decode ? Np : 16, shrink ? PROJ_SMEM_BUDGET : PROJ_SMEM_BUDGET_ALONE, zt, mt);
    if (mt > 1 && ds.splits < 2) {   // (two tiles per CTA only through the staged split-K reduction)
        mt = 1;
        ds = decode_shape(d, Np, PROJ_SMEM_BUDGET_ALONE, zt, mt);
    }
    if (a.qmode) {
        // over codes: QUANT_KC K chunks per stage (one 2D box of codes, one of scales);
        // a stage also holds the restored 16 KiB W tile of each chunk, which comes from
        // no load.  Each stage costs a round trip through the converting warps, so the
        // steps carry two chunks, and the ring budget is the deep one.  Where two such
        // stages do not fit (int8 above 224 tokens: 112 KiB a stage at 256), one chunk (two
        // token tiles of two chunks were slower at 256 tokens: 28.9 against 26.0 us).
        if (ds.budget == PROJ_SMEM_BUDGET || ds.budget == PROJ_SMEM_BUDGET_SHARED) ds.budget = PROJ_SMEM_BUDGET_ALONE;
        ds.pkc = (kb_total >= QUANT_KC && qfits(Np)) ? QUANT_KC : 1;
        ds.ksteps = (kb_total + ds.pkc - 1) / ds.pkc;
        ds.splits = ds.splits < ds.ksteps ? ds.splits : ds.ksteps;
    }
    // A decode batch with at most two rows per loaded adapter (on average) takes the
    // CUDA-core shrink: its adapters are read once each, with no split-K reduction.
    const bool gemv = decode && shrink && gemv_shrink_fits(d, T) && a.n_loaded > 0 && T <= 2 * a.n_loaded;
    int shrink_budget = SHRINK_SMEM_BUDGET;
    if (gemv) {
        // its Down rows are prefetched into L2 before the wait for the kernel before
        // when most loaded adapters are likely to be used
        if ((e = launch_shrink_gemv(a, T >= a.n_loaded, st)) != cudaSuccess) return e;
    } else if (decode && shrink && ds.budget == PROJ_SMEM_BUDGET) {
        // a shrink whose CTAs fit the SMs that the projection leaves idle gets a larger
        // ring there; a larger one shares SMs with the projection, both rings smaller
        const int stiles = (n_chunks + CHUNKS_PER_TILE - 1) / CHUNKS_PER_TILE;
        const int shrink_ctas = (stiles + 1) * zt * cluster_splits(k_splits(stiles * zt, kb_total, Np, false));
        if (shrink_ctas <= sm_count() - proj_tiles(d) * zt * ds.splits) {
            shrink_budget = SHRINK_SMEM_BUDGET_APART;
        } else {
            shrink_budget = SHRINK_SMEM_BUDGET_SHARED;
            ds = decode_shape(d, Np, PROJ_SMEM_BUDGET_SHARED, zt, mt);
        }
    }

    // ---- shrink: Vt = masked scale * Down_chunks X^T, per token tile, the used chunks
    if (shrink && !gemv) {
        const int Ns = decode ? Np : MAX_N;
        CUtensorMap tmXs, tmNone, tmDown;
        std::memset(&tmNone, 0, sizeof tmNone);
        const int tiles = (n_chunks + CHUNKS_PER_TILE - 1) / CHUNKS_PER_TILE;
        const int ztiles = decode ? zt : token_tiles(T);
        GemmParams g{};
        g.chunks = a.ws.chunks;
        g.row_adapter = a.row_adapter;
        g.slots = a.slots;
        g.vt = (__nv_bfloat16*)a.ws.vt;
        g.tmask = decode ? nullptr : a.ws.tmask;   // (the prefill projection reads it)
        g.partials = a.ws.partials;
        g.tile_ctr = a.ws.tile_ctr;
        g.status = a.ws.status;
        g.T = T;
        g.N = Ns;
        g.tcap = d.tcap;
        g.n_chunks = n_chunks;
        g.S = d.S;
        g.max_chunks = d.max_chunks;
        g.ws = a.ws;
        // Window mode: the chunks of a row tile (8 consecutive entries of the table, in
        // arena order) lie within win_rows <= 128 arena rows, so one box of win_rows
        // rows x kc K chunks loads them all; X comes as one box of Ns tokens x kc K
        // chunks.  Both views need din % 64 == 0.  Otherwise every chunk is a box of
        // its own, one K chunk per step.
        g.window = (d.din % BK == 0 && a.tile_span <= BM) ? 1 : 0;
        if (g.window) {
            int R = 16;
            while (R < a.tile_span) R *= 2;
            g.win_rows = R;
            g.a_sub = R * BK * 2;
            const int per = g.a_sub + b_bytes(Ns);
            g.kc = shrink_budget / (2 * per);
            g.kc = g.kc < 1 ? 1 : (g.kc > 4 ? 4 : g.kc);
            cuuint64_t dims[3] = {(cuuint64_t)BK, (cuuint64_t)T, (cuuint64_t)kb_total};
            cuuint64_t strides[2] = {(cuuint64_t)d.din * 2, (cuuint64_t)BK * 2};
            cuuint32_t box[3] = {BK, (cuuint32_t)Ns, (cuuint32_t)g.kc};
            if (!tc_encode(&tmXs, a.X, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
                return cudaErrorInvalidValue;
            cuuint64_t ddims[3] = {(cuuint64_t)BK, (cuuint64_t)a.units, (cuuint64_t)kb_total};
            cuuint32_t dbox[3] = {BK, (cuuint32_t)R, (cuuint32_t)g.kc};
            if (!tc_encode(&tmDown, a.arena_down, 3, ddims, strides, dbox, CU_TENSOR_MAP_SWIZZLE_128B))
                return cudaErrorInvalidValue;
        } else {
            g.kc = 1;
            // A holds the chunks of one row tile: fewer than 8 when fewer are loaded
            g.a_sub = (n_chunks < CHUNKS_PER_TILE ? n_chunks : CHUNKS_PER_TILE) * CHUNK_BYTES;
            cuuint64_t dims[2] = {(cuuint64_t)d.din, (cuuint64_t)T};
            cuuint64_t strides[1] = {(cuuint64_t)d.din * 2};
            cuuint32_t box[2] = {BK, (cuuint32_t)Ns};
            if (!tc_encode(&tmXs, a.X, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
                return cudaErrorInvalidValue;
            tmDown = a.maps.down;
        }
        g.ksteps = (kb_total + g.kc - 1) / g.kc;
        const int sb = g.kc * (g.a_sub + b_bytes(Ns));
        g.splits = cluster_splits(k_splits(tiles * ztiles, g.ksteps, Ns, false));
        g.stages = clamp_stages(shrink_budget / sb);
        // the MMA reads 128 rows of A from each K chunk's sub-block: slack after the ring
        const int slack = A_BYTES - g.a_sub - b_bytes(Ns) * g.kc;
        g.ring_bytes = g.stages * sb + (slack > 0 ? slack : 0);
        g.tail_off = g.ring_bytes;
        // the segment builder's CTA (grid column `tiles`) uses the same shared memory:
        // as many row ranges as fit it, or more memory for every CTA if none does
        const int have_ints = (int)((size_t)g.ring_bytes + sizeof(Tail)) / 4;
        SegPlan sp = seg_plan(d.S, NUM_THREADS / 32, have_ints, T);
        if (sp.P < 1) {
            sp = seg_plan(d.S, NUM_THREADS / 32, (max_dyn_smem() - 1024) / 4, T);
            if (sp.P < 1) return cudaErrorInvalidConfiguration;
            g.ring_bytes = (int)align16((size_t)sp.ints * 4);
            g.tail_off = g.ring_bytes;
        }
        g.seg_tile = tiles;
        g.seg_P = sp.P;
        g.seg_stage_rows = sp.stage_rows ? 1 : 0;
        g.cluster = g.splits > 1 ? 1 : 0;
        g.stamps = a.stamps;
        g.stamp_cap = a.stamp_cap;
        // first kernel of the forward: it may launch while the stream's previous kernel
        // runs, and waits for it before reading X or the row map
        e = launch_k(swapab_gemm_kernel<true>, dim3(tiles + 1, g.splits, ztiles), dim3(NUM_THREADS), smem_bytes(g),
                     st, true, g.cluster ? g.splits : 1, tmNone, tmXs, tmNone, tmDown, tmNone, g);
        if (e != cudaSuccess) return e;
    }

    CUtensorMap tmW, tmX, tmV, tmQs;
    std::memset(&tmQs, 0, sizeof tmQs);
    if (a.qmode == QMODE_NF4) {
        // the block scales [din / 64][dout] fp32: boxes of 128 rows of one K block
        cuuint64_t dims[2] = {(cuuint64_t)d.dout, (cuuint64_t)(d.din / BK)};
        cuuint64_t strides[1] = {(cuuint64_t)d.dout * 4};
        cuuint32_t box[2] = {(cuuint32_t)BM, (cuuint32_t)ds.pkc};
        if (!tc_encode_typed(&tmQs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.qscale, 2, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    if (a.qmode) {
        // the codes as bytes {din / (8 / bits), dout}; boxes of a step's K chunks x 128 rows
        cuuint64_t dims[2] = {(cuuint64_t)d.din / (BK / q_x), (cuuint64_t)d.dout};
        cuuint64_t strides[1] = {(cuuint64_t)(d.din / (BK / q_x))};
        cuuint32_t box[2] = {(cuuint32_t)(q_x * ds.pkc), (cuuint32_t)BM};
        if (!tc_encode_typed(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Wq, 2, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        cuuint64_t dims[2] = {(cuuint64_t)d.din, (cuuint64_t)d.dout};
        cuuint64_t strides[1] = {(cuuint64_t)d.din * 2};
        cuuint32_t box[2] = {BK, decode ? (cuuint32_t)(mt * BM) : 256u};
        if (!tc_encode(&tmW, a.W, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)d.din, (cuuint64_t)T};
        cuuint64_t strides[1] = {(cuuint64_t)d.din * 2};
        cuuint32_t box[2] = {BK, (cuuint32_t)Np};
        if (!tc_encode(&tmX, a.X, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    {
        // Vt [chunk][block of 8 rank columns][tcap][8] seen as rows of 128 bytes (8 tokens
        // of one block): one box is a K-extension step's EXT_SUB chunks x 2 blocks x Np
        // tokens, in the layout the MMA reads without swizzle, in Np / 8 rows per block
        cuuint64_t dims[3] = {64, (cuuint64_t)d.tcap / 8, (cuuint64_t)d.max_chunks * 2};
        cuuint64_t strides[2] = {128, (cuuint64_t)d.tcap * 16};
        cuuint32_t box[3] = {64, (cuuint32_t)Np / 8, 2 * EXT_SUB};
        if (!tc_encode(&tmV, a.ws.vt, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE)) return cudaErrorInvalidValue;
    }

    if (!decode) {
        return launch_prefill(a, tmX, tmW, tmV, sm_count(), shrink, st);
    }
    // the Up arena seen as runs: {64 (8 rows x 8 columns), dout / 8, run_b blocks of 8
    // rank columns, groups of run_b blocks}; a box is a K-extension step's 4 chunks of a
    // run (2 blocks each) over 128 output rows
    CUtensorMap tmRun;
    std::memset(&tmRun, 0, sizeof tmRun);
    int run_b = 0, run_groups = 0;
    if (shrink && !a.qmode && a.run_stride >= CHUNK && a.run_stride % 8 == 0 && a.maps.up_rows == 8 && a.arena_up &&
        a.units <= RUN_UNITS_MAX) {
        run_b = a.run_stride / 8;
        run_groups = a.units / a.run_stride;
        cuuint64_t dims[4] = {64, (cuuint64_t)d.dout / 8, (cuuint64_t)run_b, (cuuint64_t)run_groups};
        cuuint64_t strides[3] = {128, (cuuint64_t)d.dout * 16, (cuuint64_t)d.dout * 16 * run_b};
        cuuint32_t box[4] = {64, BM / 8, 2, EXT_SUB};
        if (run_groups < EXT_SUB || !tc_encode(&tmRun, a.arena_up, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            run_b = run_groups = 0;
    }

    const int tiles = (d.dout + mt * BM - 1) / (mt * BM);   // CTAs' row blocks
    const int budget = ds.budget, pkc = ds.pkc;
    if (pkc > 1) {
        cuuint64_t wdims[3] = {(cuuint64_t)BK, (cuuint64_t)d.dout, (cuuint64_t)kb_total};
        cuuint64_t strides[2] = {(cuuint64_t)d.din * 2, (cuuint64_t)BK * 2};
        cuuint32_t wbox[3] = {BK, (cuuint32_t)(mt * BM), (cuuint32_t)pkc};
        if (!a.qmode && !tc_encode(&tmW, a.W, 3, wdims, strides, wbox, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        cuuint64_t xdims[3] = {(cuuint64_t)BK, (cuuint64_t)T, (cuuint64_t)kb_total};
        cuuint32_t xbox[3] = {BK, (cuuint32_t)Np, (cuuint32_t)pkc};
        if (!tc_encode(&tmX, a.X, 3, xdims, strides, xbox, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    GemmParams p{};
    p.chunks = a.ws.chunks;
    p.row_adapter = a.row_adapter;
    p.Y = (__nv_bfloat16*)a.Y;
    p.partials = a.ws.partials;
    p.tile_ctr = a.ws.tile_ctr;
    p.status = a.ws.status;
    p.T = T;
    p.dout = d.dout;
    p.N = Np;
    p.kc = pkc;
    p.ksteps = ds.ksteps;
    p.n_chunks = n_chunks;
    p.ext_units = shrink ? (n_chunks + EXT_SUB - 1) / EXT_SUB : 0;
    p.splits = ds.splits;
    // small batches: the splits push their partial slices into a receive buffer
    p.push = (p.splits > 1 && Np <= PUSH_MAX_N && Np % p.splits == 0) ? 1 : 0;
    // K-extension steps: after the W steps, or, behind the CUDA-core shrink (done early
    // in the W stream), a quarter of the way into them, where their Up tiles' DRAM
    // latency overlaps the W stream
    p.ext_lead = gemv ? 3 * (ds.ksteps / ds.splits) / 4 : (EXT_LEAD + pkc - 1) / pkc;
    const int rx_bytes = p.push ? BM * Np * 4 : 0;
    // (over codes, the code tile too, and over 4-bit codes the K block's scales)
    const int sbytes = (pkc * (stage_bytes(Np) + (mt - 1) * A_BYTES + BM * q_x + (a.qmode == QMODE_NF4 ? BM * 4 : 0)) +
                        1023) & ~1023;
    const int qtab_bytes = a.qmode == QMODE_NF4 ? 64 : 0;
    p.stages = clamp_stages((budget - rx_bytes - qtab_bytes) / sbytes);
    p.a_sub = mt * A_BYTES;
    p.ring_bytes = p.stages * sbytes;
    p.rx_off = p.ring_bytes;
    p.qtab_off = p.ring_bytes + rx_bytes;
    p.tail_off = p.qtab_off + qtab_bytes;
    p.tcap = d.tcap;
    p.pdl = shrink ? 1 : 0;
    // Without a shrink the projection is the forward's first kernel: launched while the
    // kernel before it may run, its W goes out at once and its X after that kernel
    // has completed.  After a shrink it launches once the shrink has seen the kernel
    // before the forward complete, so X may be read at once.
    p.xwait = shrink ? 0 : 1;
    p.cluster = p.splits > 1 ? 1 : 0;
    p.S = d.S;
    p.max_chunks = d.max_chunks;
    p.stamps = a.stamps;
    p.stamp_cap = a.stamp_cap;
    p.qmode = a.qmode;
    p.q_x = q_x;
    p.qscale = a.qscale;
    p.up_rows = a.maps.up_rows;
    p.run_b = run_b;
    p.run_groups = run_groups;
    for (int i = 0; i < 16; ++i) p.qcb[i] = a.qcb[i];
    return launch_k(mt > 1 ? swapab_gemm_kernel<false, 2> : swapab_gemm_kernel<false, 1>, dim3(tiles, p.splits, zt),
                    dim3(NUM_THREADS), smem_bytes(p), st, true,
                    p.cluster ? p.splits : 1, tmW, tmX, tmV, a.maps.upw128, a.qmode ? tmQs : tmRun, p);
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
    p.kc = 1;
    p.ksteps = kb_total;
    p.ext_units = 0;
    // as many K splits as fill the SMs and whose partial tiles fit the scratch
    int splits = k_splits(tiles, kb_total, N, true);
    const size_t per_split = (size_t)tiles * BM * N * sizeof(float);
    while (splits > 1 && (size_t)splits * per_split > partial_bytes) --splits;
    p.splits = splits;
    p.stages = clamp_stages(PROJ_SMEM_BUDGET / stage_bytes(N));
    p.a_sub = A_BYTES;
    p.ring_bytes = p.stages * stage_bytes(N);
    p.tail_off = p.ring_bytes;
    p.tcap = 0;
    p.pdl = 0;
    p.cluster = 0;   // the K splits meet through the given scratch
    return launch_k(swapab_gemm_kernel<false>, dim3(tiles, p.splits, 1), dim3(NUM_THREADS), smem_bytes(p), st, false,
                    1, tmW, tmX, tmNone, tmNone, tmNone, p);
}

}  // namespace mlora
