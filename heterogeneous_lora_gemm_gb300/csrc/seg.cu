// Row -> adapter segment builder (ai-infra-kb "M031" tutorial §02/§03; wiblog section
// on Punica's grouped matmul): group the rows of a mixed batch by adapter slot, keep
// the original order inside each group (P, R before Q in the page's example), and
// order groups by ascending slot id.  Produces, bit-exactly:
//   counts[S]      rows per slot
//   offsets[S+1]   exclusive prefix sum of counts
//   perm[T]        original row indices in segment order, -1 past the valid rows
//   chunk table    the touched slots (count > 0) in ascending order, each split into
//                  ceil(rank/16) chunks of 16 rank columns: the K-extension layout
//                  of the tensor-core expand
// One CTA does all of it: T is at most a few ten thousand rows and S at most
// 4096, and a single CTA needs no inter-CTA wait of any kind.
//
// Stable scatter without a sort: the rows are split into P contiguous ranges, one
// per warp.  Pass 1 counts rows per (warp, slot) with __match_any_sync (one leader
// per group of equal ids in each 32-row step).  The counts are turned into
// per-(warp, slot) cursors: offsets[s] + rows of slot s in earlier warps.  Pass 2
// walks the same ranges again; a row's position is its warp's cursor for its slot
// plus the number of lower lanes with the same id in that step.  Ranges are in
// row order and steps are in row order, so the result is the stable order.
#include "internal.h"

namespace mlora {

namespace {

constexpr int SEG_THREADS = 1024;
constexpr int SEG_WARPS = SEG_THREADS / 32;

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive scan of n ints in shared memory, in place, by the whole block.
// Returns the total (valid in every thread after the call).
__device__ int block_exclusive_scan(int* a, int n, int* warp_tmp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + SEG_THREADS - 1) / SEG_THREADS;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += a[i];
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) warp_tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tmp[lane];
        int wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int v = __shfl_up_sync(0xffffffffu, wi, d);
            if (lane >= d) wi += v;
        }
        warp_tmp[lane] = wi - w;           // exclusive prefix of warp totals
        if (lane == 31) warp_tmp[32] = wi;  // grand total
    }
    __syncthreads();
    int run = warp_tmp[warp] + incl - local;
    for (int i = lo; i < hi; ++i) {
        int v = a[i];
        a[i] = run;
        run += v;
    }
    int total = warp_tmp[32];
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(SEG_THREADS, 1)
seg_build_kernel(const int32_t* __restrict__ row_adapter, int T, const SlotRec* __restrict__ slots,
                 Workspace ws, int S, int P, int max_chunks) {
    extern __shared__ int smem[];
    int* rank_s = smem;                 // [S]
    int* scan = rank_s + S;             // [S]   counts, then offsets
    int* cur = scan + S;                // [P*S] per-(warp, slot) counts, then cursors
    __shared__ int warp_tmp[33];
    __shared__ int bad_row;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the shrink that follows may launch now; it reads this kernel's output only after its wait
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int s = tid; s < S; s += SEG_THREADS) {
        rank_s[s] = slots[s].rank;
        scan[s] = 0;
    }
    for (int i = tid; i < P * S; i += SEG_THREADS) cur[i] = 0;
    if (tid == 0) bad_row = 0;
    __syncthreads();

    // ---- pass 1: per (warp, slot) counts
    const int t_lo = (int)((long long)warp * T / P);
    const int t_hi = (int)((long long)(warp + 1) * T / P);
    if (warp < P) {
        for (int base = t_lo; base < t_hi; base += 32) {
            const int t = base + lane;
            int a = -1;
            if (t < t_hi) {
                a = row_adapter[t];
                const bool ok = a >= 0 && a < S && rank_s[a] > 0;
                if (!ok) {
                    if (a != -1) bad_row = 1;
                    a = -1;
                }
            }
            const unsigned grp = __match_any_sync(0xffffffffu, a);
            if (a >= 0 && (grp & lanemask_lt()) == 0) cur[warp * S + a] += __popc(grp);
            __syncwarp();
        }
    }
    __syncthreads();

    // ---- totals, offsets and per-warp cursors
    for (int s = tid; s < S; s += SEG_THREADS) {
        int tot = 0;
        for (int w = 0; w < P; ++w) tot += cur[w * S + s];
        scan[s] = tot;
        ws.counts[s] = tot;
    }
    __syncthreads();
    const int n_valid = block_exclusive_scan(scan, S, warp_tmp);
    for (int s = tid; s < S; s += SEG_THREADS) {
        ws.offsets[s] = scan[s];
        int run = scan[s];
        for (int w = 0; w < P; ++w) {
            const int c = cur[w * S + s];
            cur[w * S + s] = run;
            run += c;
        }
    }
    if (tid == 0) ws.offsets[S] = n_valid;
    __syncthreads();

    // ---- pass 2: stable scatter
    if (warp < P) {
        for (int base = t_lo; base < t_hi; base += 32) {
            const int t = base + lane;
            int a = -1;
            if (t < t_hi) {
                a = row_adapter[t];
                if (!(a >= 0 && a < S && rank_s[a] > 0)) a = -1;
            }
            const unsigned grp = __match_any_sync(0xffffffffu, a);
            int pos = 0;
            if (a >= 0) pos = cur[warp * S + a] + __popc(grp & lanemask_lt());
            __syncwarp();
            if (a >= 0) {
                ws.perm[pos] = t;
                if ((grp & lanemask_lt()) == 0) cur[warp * S + a] += __popc(grp);
            }
            __syncwarp();
        }
    }
    for (int i = n_valid + tid; i < T; i += SEG_THREADS) ws.perm[i] = -1;
    __syncthreads();

    // ---- K-extension chunks of the touched slots, ascending slot id
    for (int s = tid; s < S; s += SEG_THREADS)
        scan[s] = (ws.counts[s] > 0) ? (rank_s[s] + CHUNK - 1) / CHUNK : 0;
    __syncthreads();
    const int n_chunks = block_exclusive_scan(scan, S, warp_tmp);
    for (int s = tid; s < S; s += SEG_THREADS) {
        if (ws.counts[s] > 0) {
            const int nc = (rank_s[s] + CHUNK - 1) / CHUNK;
            for (int j = 0; j < nc; ++j) {
                const int c = scan[s] + j;
                if (c < max_chunks) {
                    ws.chunk_slot[c] = s;
                    ws.chunk_col[c] = j * CHUNK;
                }
            }
        }
    }
    if (tid == 0) {
        ws.meta[0] = n_valid;
        ws.meta[1] = min(n_chunks, max_chunks);
        if (bad_row) atomicOr(ws.status, STATUS_BAD_ROW);
    }
    // number of touched slots
    int touched = 0;
    for (int s = tid; s < S; s += SEG_THREADS) touched += (ws.counts[s] > 0);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) touched += __shfl_xor_sync(0xffffffffu, touched, d);
    if (lane == 0) warp_tmp[warp] = touched;
    __syncthreads();
    if (tid == 0) {
        int tt = 0;
        for (int w = 0; w < SEG_WARPS; ++w) tt += warp_tmp[w];
        ws.meta[2] = tt;
    }
}

}  // namespace

cudaError_t seg_init() {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, seg_build_kernel);
    // static shared memory counts against the same per-block limit
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(seg_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - (int)fa.sharedSizeBytes);
    return e;
}

cudaError_t launch_seg_build(const int32_t* row_adapter, int T, const SlotRec* slots,
                             const Workspace& ws, const PoolDims& d, cudaStream_t st) {
    const int S = d.S;
    int P = S > 0 ? 10240 / S : SEG_WARPS;
    P = P < 1 ? 1 : (P > SEG_WARPS ? SEG_WARPS : P);
    const size_t smem = sizeof(int) * ((size_t)2 * S + (size_t)P * S);
    seg_build_kernel<<<1, SEG_THREADS, smem, st>>>(row_adapter, T, slots, ws, S, P, d.max_chunks);
    return cudaGetLastError();
}

}  // namespace mlora
