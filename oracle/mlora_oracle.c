/*
 * mlora_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, obviously correct fp64 CPU statement of the multi-LoRA linear
 * layer for a mixed batch.  Only tests/, the smoke check of __graft_entry__ and
 * the cpu_baseline / reference leg of bench.py may load this library.  It shares
 * no code, header, table or helper with the CUDA path under
 * heterogeneous_lora_gemm_gb300/csrc, and it includes nothing from there.
 *
 * Sources (the pages that define the method):
 *   [M031]    ai-infra-kb "M031" multi-LoRA tutorial page, sections 02-06.
 *   [AIRSOTA] airsota interview card "multi-LoRA serving vs merging", part 三
 *             (mathematical derivation).
 *   [WIBLOG]  wiblog "vLLM LoRA adapter batch scheduling", section on the Punica
 *             grouped matmul ("分组矩阵乘的直觉").
 *
 * Every routine below is pinned by tests/test_oracle_pins.py against facts the
 * pages print or against independent mathematics (see the test file).
 *
 * Conventions shared with the callers (plain C arrays, all row-major):
 *   X    [T x din]        input rows
 *   W    [dout x din]     base weight (the torch Linear layout)
 *   Down_s [r_s x din]    adapter s, first LoRA matrix (stored at down_all + down_off[s])
 *   Up_s   [dout x r_s]   adapter s, second LoRA matrix (stored at up_all + up_off[s])
 *   row_adapter[T]        slot id per row, -1 = no adapter
 *   ranks[S]              rank of slot s; 0 means "slot not loaded"
 * A row whose id is outside [0, S) or names an unloaded slot is treated exactly
 * like a row with -1 (it keeps the base output) and is counted as invalid.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int valid_slot(int32_t a, int32_t S, const int32_t* ranks)
{
    return a >= 0 && a < S && ranks[a] > 0;
}

/* ------------------------------------------------------------------------- */
/* Segments: [M031] §02/§03.  The rows that carry an adapter are grouped by
 * adapter id; inside a group the rows keep their original order (the page's
 * group order for rows P(A),Q(B),R(A),S(-) is P,R then Q).  Across groups the
 * order is ascending slot id.  Definition used here: sort the pairs
 * (slot, row) of all valid rows lexicographically.  Since every pair is unique
 * any correct sort gives the same sequence.                                  */

typedef struct { int32_t slot; int64_t row; } seg_pair;

static int cmp_seg_pair(const void* pa, const void* pb)
{
    const seg_pair* a = (const seg_pair*)pa;
    const seg_pair* b = (const seg_pair*)pb;
    if (a->slot != b->slot) return a->slot < b->slot ? -1 : 1;
    if (a->row != b->row) return a->row < b->row ? -1 : 1;
    return 0;
}

/* counts[S]: rows per slot.  offsets[S+1]: exclusive prefix sum of counts.
 * perm[n_valid]: original row indices in segment order.  Returns n_valid and
 * stores the number of rows whose id was not a loaded slot (and not -1) in
 * *n_invalid. */
int64_t oracle_segments(int64_t T, const int32_t* row_adapter, int32_t S,
                        const int32_t* ranks, int32_t* counts, int32_t* offsets,
                        int32_t* perm, int64_t* n_invalid)
{
    seg_pair* pairs = (seg_pair*)malloc(sizeof(seg_pair) * (size_t)(T > 0 ? T : 1));
    int64_t n = 0, bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        int32_t a = row_adapter[t];
        if (valid_slot(a, S, ranks)) {
            pairs[n].slot = a;
            pairs[n].row = t;
            ++n;
        } else if (a != -1) {
            ++bad;
        }
    }
    qsort(pairs, (size_t)n, sizeof(seg_pair), cmp_seg_pair);
    for (int32_t s = 0; s < S; ++s) counts[s] = 0;
    for (int64_t i = 0; i < n; ++i) {
        counts[pairs[i].slot] += 1;
        perm[i] = (int32_t)pairs[i].row;
    }
    offsets[0] = 0;
    for (int32_t s = 0; s < S; ++s) offsets[s + 1] = offsets[s] + counts[s];
    free(pairs);
    if (n_invalid) *n_invalid = bad;
    return n;
}

/* ------------------------------------------------------------------------- */
/* Forward: [M031] §02 and [AIRSOTA] 三.1.  For every requested row t:
 *   y_t[o] = sum_i W[o,i] x_t[i]                         (shared base, all rows)
 *   if row t carries adapter a:
 *       v_k     = sum_i Down_a[k,i] x_t[i]               (k < r_a)
 *       y_t[o] += scale_a * sum_k Up_a[o,k] v_k
 * written to Y[j,:] for the j-th requested row (rows == NULL: all rows, j = t),
 * i.e. in the original row order.  fp64 throughout, one row at a time. */
void oracle_forward(int64_t T, int64_t din, int64_t dout,
                    const double* X, const double* W, const int32_t* row_adapter,
                    int32_t S, const int32_t* ranks, const double* scales,
                    const int64_t* down_off, const int64_t* up_off,
                    const double* down_all, const double* up_all,
                    const int64_t* rows, int64_t n_rows, double* Y)
{
    int32_t max_rank = 1;
    for (int32_t s = 0; s < S; ++s)
        if (ranks[s] > max_rank) max_rank = ranks[s];
    if (rows == NULL) n_rows = T;

#pragma omp parallel
    {
        double* v = (double*)malloc(sizeof(double) * (size_t)max_rank);
#pragma omp for schedule(dynamic, 1)
        for (int64_t j = 0; j < n_rows; ++j) {
            int64_t t = rows ? rows[j] : j;
            const double* x = X + t * din;
            double* y = Y + j * dout;
            for (int64_t o = 0; o < dout; ++o) {
                const double* w = W + o * din;
                double acc = 0.0;
                for (int64_t i = 0; i < din; ++i) acc += w[i] * x[i];
                y[o] = acc;
            }
            int32_t a = (row_adapter != NULL) ? row_adapter[t] : -1;
            if (!valid_slot(a, S, ranks)) continue;
            int32_t r = ranks[a];
            const double* down = down_all + down_off[a];
            const double* up = up_all + up_off[a];
            for (int32_t k = 0; k < r; ++k) {
                const double* d = down + (int64_t)k * din;
                double acc = 0.0;
                for (int64_t i = 0; i < din; ++i) acc += d[i] * x[i];
                v[k] = acc;
            }
            for (int64_t o = 0; o < dout; ++o) {
                const double* u = up + o * r;
                double acc = 0.0;
                for (int32_t k = 0; k < r; ++k) acc += u[k] * v[k];
                y[o] += scales[a] * acc;
            }
        }
        free(v);
    }
}

/* ------------------------------------------------------------------------- */
/* Merge: [M031] §04 and [AIRSOTA] 三.2.
 *   W_out[o,i] = W[o,i] + scale * sum_k Up[o,k] Down[k,i]
 * The merged matrix serves rows of this one adapter only. */
void oracle_merge(int64_t din, int64_t dout, const double* W, int32_t rank,
                  double scale, const double* down, const double* up, double* W_out)
{
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < dout; ++o) {
        for (int64_t i = 0; i < din; ++i) {
            double acc = 0.0;
            for (int32_t k = 0; k < rank; ++k) acc += up[o * rank + k] * down[(int64_t)k * din + i];
            W_out[o * din + i] = W[o * din + i] + scale * acc;
        }
    }
}

/* Un-merge ([AIRSOTA] section 四 item ③: a merge overwrites the base; switching back
 * re-subtracts the adapter's update): W_out = W - scale * Up Down, in fp64. */
void oracle_unmerge(int64_t din, int64_t dout, const double* W, int32_t rank,
                    double scale, const double* down, const double* up, double* W_out)
{
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < dout; ++o) {
        const double* u = up + o * rank;   /* row o of Up */
        for (int64_t i = 0; i < din; ++i) {
            double acc = 0.0;
            for (int32_t k = 0; k < rank; ++k) acc += u[k] * down[(int64_t)k * din + i];
            W_out[o * din + i] = W[o * din + i] - scale * acc;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Low-rank work count: [M031] §03.  Each adapter group costs
 * 2 * rows * rank * (din + dout) FLOP (Down then Up, multiply and add); the
 * coarse alternative that gives every row of the batch a dense branch at the
 * largest rank present costs 2 * T * r_max * (din + dout). */
void oracle_lora_flops(int64_t T, int64_t din, int64_t dout, const int32_t* row_adapter,
                       int32_t S, const int32_t* ranks, int64_t* exact, int64_t* padded)
{
    int64_t e = 0;
    int32_t r_max = 0;
    for (int64_t t = 0; t < T; ++t) {
        int32_t a = row_adapter ? row_adapter[t] : -1;
        if (!valid_slot(a, S, ranks)) continue;
        e += 2 * (int64_t)ranks[a] * (din + dout);
        if (ranks[a] > r_max) r_max = ranks[a];
    }
    *exact = e;
    *padded = 2 * T * (int64_t)r_max * (din + dout);
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
