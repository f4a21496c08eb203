// Row -> adapter segment builder as a device function over a group of threads
// (ai-infra-kb "M031" tutorial §02/§03; wiblog section on Punica's grouped
// matmul): group the rows of a mixed batch by adapter slot, keep the original
// order inside each group (P, R before Q in the page's example) and order groups
// by ascending slot id.
//
// Published to the workspace, bit-exactly:
//   counts[S]      rows per slot
//   offsets[S+1]   exclusive prefix sum of counts
//   perm[T]        original row indices in segment order, -1 past the valid rows
//   chunk table    the touched slots (count > 0) in ascending order, each split into
//                  ceil(rank/16) chunks of 16 rank columns.  Per chunk: slot,
//                  absolute rank-unit index in the arena (unit of the slot + first
//                  column) and the number of valid rank columns (<= 16).
//   meta           [0] valid rows, [1] chunks of the touched slots, [2] touched slots
//   status         STATUS_BAD_ROW if a row names an invalid or empty slot
//
// Stable scatter without a sort: the rows are split into P contiguous ranges, one
// per warp.  Pass 1 counts rows per (warp, slot) with __match_any_sync (one
// leader per group of equal ids in each 32-row step).  The counts become
// per-(warp, slot) cursors: offsets[s] + rows of slot s in earlier warps.  Pass 2
// walks the same ranges again; a row's position is its warp's cursor for its
// slot plus the number of lower lanes with the same id in that step.  Ranges and
// steps are in row order, so the result is the stable order.
//
// The whole block of one CTA runs it (no CTA ever waits on another): the
// standalone segment kernel, or a CTA of its own in the tensor-core shrink's grid.
// It runs in two steps: stage() copies the slot table and the builder's arguments
// into shared memory, build() then reads only the row map from global memory.  In
// the shrink's grid, stage() runs before the wait for the kernel before (the slot
// table is pool state that no kernel writes), so that only the row map's round
// trip follows the wait.
#pragma once
#include "internal.h"

namespace mlora {
namespace seg {

// The builder's arguments, staged in shared memory.
struct Staged {
    Workspace ws;
    const int32_t* row_adapter;
    int T;
    int max_chunks;
};
constexpr int STAGED_INTS = (int)((sizeof(Staged) + 15) / 16 * 4);   // 16-byte multiple

struct Scratch {
    Staged* in;      // the arguments
    int* rank_s;     // [S]
    int* unit_s;     // [S]
    int* scan;       // [S]
    int* cur;        // [P*S]
    int* misc;       // [40]: warp_tmp[0..32], [33] bad row
    int* ra_s;       // [T] the row map staged once, or nullptr (read from global memory)
};

__host__ __device__ inline int scratch_ints(int S, int P, int T_staged) {
    return STAGED_INTS + 3 * S + P * S + 40 + T_staged;
}

// `base` 16-byte aligned
__device__ inline Scratch carve(int* base, int S, int P, bool stage_rows) {
    Scratch s;
    s.in = reinterpret_cast<Staged*>(base);
    s.rank_s = base + STAGED_INTS;
    s.unit_s = s.rank_s + S;
    s.scan = s.unit_s + S;
    s.cur = s.scan + S;
    s.misc = s.cur + P * S;
    s.ra_s = stage_rows ? s.misc + 40 : nullptr;
    return s;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive scan of n ints in shared memory, in place, by the block.  Returns the total.
__device__ inline int block_exclusive_scan(int* a, int n, int* warp_tmp) {
    const int nt = blockDim.x, lane = threadIdx.x & 31;
    const int tid = threadIdx.x, warp = threadIdx.x >> 5, nwarps = nt >> 5;
    const int per = (n + nt - 1) / nt;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += a[i];
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) warp_tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < nwarps ? warp_tmp[lane] : 0;
        int wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, d);
            if (lane >= d) wi += v;
        }
        if (lane < nwarps) warp_tmp[lane] = wi - w;
        if (lane == 31) warp_tmp[32] = wi;
    }
    __syncthreads();
    int run = warp_tmp[warp] + incl - local;
    for (int i = lo; i < hi; ++i) {
        const int v = a[i];
        a[i] = run;
        run += v;
    }
    const int total = warp_tmp[32];
    __syncthreads();
    return total;
}

// Copies the slot table and the builder's arguments into shared memory.  Every
// thread of the block must call it (the block barrier is in build()).
__device__ inline void stage(const SlotRec* __restrict__ slots, int S, const Workspace& ws,
                             const int32_t* row_adapter, int T, int max_chunks, const Scratch& sc) {
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const SlotRec r = slots[s];
        sc.rank_s[s] = r.rank;
        sc.unit_s[s] = r.unit;
    }
    if (threadIdx.x == 0) {
        sc.in->ws = ws;
        sc.in->row_adapter = row_adapter;
        sc.in->T = T;
        sc.in->max_chunks = max_chunks;
    }
}

// Builds the segments of the staged row map over S slots in shared memory, with P
// row ranges (at most the block's warps; warps past P only help with the scans),
// and publishes them to the workspace.  Every thread of the block must call it,
// after stage().
__device__ inline void build(int S, int P, const Scratch& sc) {
    const int nt = blockDim.x, lane = threadIdx.x & 31;
    const int tid = threadIdx.x, warp = threadIdx.x >> 5;
    int* warp_tmp = sc.misc;
    __syncthreads();   // the staged arguments
    const Workspace& ws = sc.in->ws;
    const int32_t* row_adapter = sc.in->row_adapter;
    const int T = sc.in->T, max_chunks = sc.in->max_chunks;
    // the builder's only global reads: the row map
    if (sc.ra_s)
        for (int t = tid; t < T; t += nt) sc.ra_s[t] = row_adapter[t];
    for (int i = tid; i < P * S; i += nt) sc.cur[i] = 0;
    if (tid == 0) sc.misc[33] = 0;
    __syncthreads();
    const int32_t* ra = sc.ra_s ? sc.ra_s : row_adapter;

    // ---- pass 1: per (warp, slot) counts
    const int t_lo = warp < P ? (int)((long long)warp * T / P) : 0;
    const int t_hi = warp < P ? (int)((long long)(warp + 1) * T / P) : 0;
    for (int base = t_lo; base < t_hi; base += 32) {
        const int t = base + lane;
        int a = -1;
        if (t < t_hi) {
            a = ra[t];
            if (!(a >= 0 && a < S && sc.rank_s[a] > 0)) {
                if (a != -1) sc.misc[33] = 1;
                a = -1;
            }
        }
        const unsigned grp = __match_any_sync(0xffffffffu, a);
        if (a >= 0 && (grp & lanemask_lt()) == 0) sc.cur[warp * S + a] += __popc(grp);
        __syncwarp();
    }
    __syncthreads();

    // ---- totals, offsets and per-warp cursors
    for (int s = tid; s < S; s += nt) {
        int tot = 0;
        for (int w = 0; w < P; ++w) tot += sc.cur[w * S + s];
        sc.scan[s] = tot;
        ws.counts[s] = tot;
    }
    __syncthreads();
    const int n_valid = block_exclusive_scan(sc.scan, S, warp_tmp);
    for (int s = tid; s < S; s += nt) {
        const int off = sc.scan[s];
        ws.offsets[s] = off;
        int run = off;
        for (int w = 0; w < P; ++w) {
            const int c = sc.cur[w * S + s];
            sc.cur[w * S + s] = run;
            run += c;
        }
    }
    if (tid == 0) ws.offsets[S] = n_valid;
    __syncthreads();

    // ---- pass 2: stable scatter
    for (int base = t_lo; base < t_hi; base += 32) {
        const int t = base + lane;
        int a = -1;
        if (t < t_hi) {
            a = ra[t];
            if (!(a >= 0 && a < S && sc.rank_s[a] > 0)) a = -1;
        }
        const unsigned grp = __match_any_sync(0xffffffffu, a);
        int pos = 0;
        if (a >= 0) pos = sc.cur[warp * S + a] + __popc(grp & lanemask_lt());
        __syncwarp();
        if (a >= 0) {
            ws.perm[pos] = t;
            if ((grp & lanemask_lt()) == 0) sc.cur[warp * S + a] += __popc(grp);
        }
        __syncwarp();
    }
    for (int i = n_valid + tid; i < T; i += nt) ws.perm[i] = -1;
    __syncthreads();

    // ---- chunks of the touched slots (non-empty segments), ascending slot id;
    // cur[0..S) is reused for the per-slot chunk counts
    for (int s = tid; s < S; s += nt) {
        const int off = sc.scan[s];
        const int nxt = (s + 1 < S) ? sc.scan[s + 1] : n_valid;
        sc.cur[s] = (nxt > off) ? (sc.rank_s[s] + CHUNK - 1) / CHUNK : 0;
    }
    __syncthreads();
    const int n_chunks_raw = block_exclusive_scan(sc.cur, S, warp_tmp);
    const int n_chunks = min(n_chunks_raw, max_chunks);
    int touched = 0;
    for (int s = tid; s < S; s += nt) {
        const int off = sc.scan[s];
        const int nxt = (s + 1 < S) ? sc.scan[s + 1] : n_valid;
        if (nxt > off) {
            ++touched;
            const int nc = (sc.rank_s[s] + CHUNK - 1) / CHUNK;
            for (int j = 0; j < nc; ++j) {
                const int c = sc.cur[s] + j;
                if (c < max_chunks) {
                    ws.chunk_slot[c] = s;
                    ws.chunk_unit[c] = sc.unit_s[s] + j * CHUNK;
                    ws.chunk_kval[c] = min(CHUNK, sc.rank_s[s] - j * CHUNK);
                }
            }
        }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) touched += __shfl_xor_sync(0xffffffffu, touched, d);
    __syncthreads();   // warp_tmp reuse below
    if (lane == 0) warp_tmp[warp] = touched;
    __syncthreads();
    if (tid == 0) {
        int tt = 0;
        for (int w = 0; w < (nt >> 5); ++w) tt += warp_tmp[w];
        ws.meta[0] = n_valid;
        ws.meta[1] = n_chunks;
        ws.meta[2] = tt;
        if (sc.misc[33]) atomicOr(ws.status, STATUS_BAD_ROW);
    }
    __syncthreads();
}

}  // namespace seg
}  // namespace mlora
