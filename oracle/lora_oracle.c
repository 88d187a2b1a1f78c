/*
 * lora_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU reference of the multi-tenant LoRA adapted linear layer.
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg load it;
 * the GPU library never links or calls it, and it shares no code with the GPU path.
 *
 * What it computes (pages: "m07 -- Multi-Adapter (LoRA) Serving", section 6 "Deep Dive
 * A: Batching Heterogeneous Adapters", the forward y = Wx + (B.A)x.(alpha/r), with the
 * scale passed in directly; "12. Adapter Serving and Multi-Tenant Customization",
 * section "What an adapter adds to a forward pass", W*x + B*A*x with A [r, d] and
 * B [d, r]; section 2 "Scale Numbers" for the factor shapes A: (r, d_in), B: (d_out, r)):
 *
 *   for every row i with adapter a = ids[i]:
 *     y_i[o] = sum_k W[o,k] x_i[k]  +  s * sum_j B_a[o,j] * ( sum_k A_a[j,k] x_i[k] )
 *
 * and for a row whose id is -1 (a base-only request, "12. Adapter Serving ...",
 * section "Scheduling with adapter awareness", the base-only group) only the first sum.
 * Inputs are bf16 bit patterns, widened exactly; every product and sum is fp64, in the
 * order written above. Rows are independent, so any subset of rows can be computed.
 *
 * It also gives the row grouping the batched kernels rely on ("m07", section 6: an index
 * vector maps each sequence to its adapter slot; "LoRA, quotas and noisy neighbours",
 * section "One weight read, many adapters": rows tagged with their adapter, grouped into
 * segments): a stable ordering of rows by adapter id, written with the textbook
 * definition of a stable rank.
 */
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * y[s * d_out + o] for the selected rows rows[0..n_sel-1] (indices into x / ids).
 *   x      : bf16 [n_rows_total, d_in]
 *   W      : bf16 [d_out, d_in]
 *   ids    : int32 [n_rows_total], -1 = base only, else 0 <= id < n_adapters
 *   ranks  : int32 [n_adapters] (0 = adapter has no factors for this module)
 *   A[a]   : bf16 [ranks[a], d_in]
 *   B[a]   : bf16 [d_out, ranks[a]]
 *   t_out  : optional fp64 [n_sel, max_rank] shrink result (unscaled), may be NULL
 * Returns 0, or -1 on an id outside [-1, n_adapters) / an id whose adapter has rank 0.
 */
int oracle_adapted_linear(int n_sel, const int64_t *rows, int d_in, int d_out,
                          const uint16_t *x, const uint16_t *W, const int32_t *ids,
                          int n_adapters, const int32_t *ranks,
                          const uint16_t *const *A, const uint16_t *const *B,
                          double scale, double *y, double *t_out, int max_rank, int n_threads)
{
    for (int s = 0; s < n_sel; ++s) {
        int a = ids[rows[s]];
        if (a < -1 || a >= n_adapters) return -1;
        if (a >= 0 && (ranks[a] <= 0 || ranks[a] > max_rank)) return -1;
    }
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    /* the shrink: t_i[j] = sum_k A_a[j,k] x_i[k] */
    double *t = t_out;
    if (t == NULL) return -1;
    long long n_t = (long long)n_sel * max_rank;
#pragma omp parallel for schedule(static)
    for (long long e = 0; e < n_t; ++e) {
        int s = (int)(e / max_rank), j = (int)(e % max_rank);
        int a = ids[rows[s]];
        double acc = 0.0;
        if (a >= 0 && j < ranks[a]) {
            const uint16_t *xi = x + rows[s] * (int64_t)d_in;
            const uint16_t *Aj = A[a] + (int64_t)j * d_in;
            for (int k = 0; k < d_in; ++k) acc += bf16_to_f64(Aj[k]) * bf16_to_f64(xi[k]);
        }
        t[e] = acc;
    }
    /* the base term plus the scaled expand: y_i[o] = sum_k W[o,k] x_i[k] + s * sum_j B_a[o,j] t_i[j] */
    long long n_y = (long long)n_sel * d_out;
#pragma omp parallel for schedule(static)
    for (long long e = 0; e < n_y; ++e) {
        int s = (int)(e / d_out), o = (int)(e % d_out);
        int a = ids[rows[s]];
        const uint16_t *xi = x + rows[s] * (int64_t)d_in;
        const uint16_t *Wo = W + (int64_t)o * d_in;
        double base = 0.0;
        for (int k = 0; k < d_in; ++k) base += bf16_to_f64(Wo[k]) * bf16_to_f64(xi[k]);
        double delta = 0.0;
        if (a >= 0) {
            int r = ranks[a];
            const uint16_t *Bo = B[a] + (int64_t)o * r;
            for (int j = 0; j < r; ++j) delta += bf16_to_f64(Bo[j]) * t[(int64_t)s * max_rank + j];
        }
        y[e] = base + scale * delta;
    }
    return 0;
}

/*
 * Stable grouping of rows by adapter id (ascending; -1, the base-only rows, first; rows
 * keep their original order inside a group).  The position of row i is
 *     #{ j : id_j < id_i }  +  #{ j < i : id_j == id_i },
 * so perm[pos(i)] = i.  seg_start[0..n_seg] bounds the groups, seg_adapter[s] is the id
 * of group s.  perm, seg_start, seg_adapter must hold n, n+1 and n entries.
 */
int oracle_segments(int n, const int32_t *ids, int32_t *perm, int32_t *seg_start,
                    int32_t *seg_adapter, int32_t *n_seg)
{
    for (int i = 0; i < n; ++i) {
        int pos = 0;
        for (int j = 0; j < n; ++j) {
            if (ids[j] < ids[i]) ++pos;
            else if (ids[j] == ids[i] && j < i) ++pos;
        }
        perm[pos] = i;
    }
    int ns = 0;
    for (int p = 0; p < n; ++p) {
        int id = ids[perm[p]];
        if (p == 0 || id != ids[perm[p - 1]]) {
            seg_start[ns] = p;
            seg_adapter[ns] = id;
            ++ns;
        }
    }
    seg_start[ns] = n;
    *n_seg = ns;
    return 0;
}
