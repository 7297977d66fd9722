/*
 * CPU oracle for the multi-LoRA mixed-batch adapter update.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header, table or helper with the CUDA library; the product path never
 * calls it.
 *
 * What it computes ("Multi-LoRA Serving - S-LoRA/Punica Batching, Adapter
 * Hot-Swap & Memory", section "The kernel trick: gather, do not merge"): for
 * request i using adapter a(i),
 *
 *     y_i = x_i W^T + scale_a * (x_i A_a^T) B_a^T
 *
 * which in this library's orientation (A_T_a is r x h_in, its row j is the
 * j-th low-rank direction; B_a is r x h_out) reads
 *
 *     v[t][j] = sum_k x[t][k] * A_T_a[j][k]                   ("shrink")
 *     y[t][n] = y0[t][n] + sum_k x[t][k] * W[n][k]             (base, optional)
 *                        + scale_a * sum_j v[t][j] * B_a[j][n]  ("expand")
 *
 * Segments (SGMV: runs of consecutive tokens that share an adapter) are
 * expanded to one adapter id per token by a plain loop.  Mixed ranks (S-LoRA
 * slide 10: adapters of different ranks are gathered without padding them to
 * one rank) are handled by giving each adapter its own rank: the sums over j
 * run to that rank only.
 *
 * Conventions the pages leave open, taken here:
 *   - adapter id < 0 means "no adapter": the token gets no low-rank term;
 *   - an id >= n_adapters or an adapter whose rank is < 0 (not loaded) is an
 *     error: the token gets no low-rank term and ORC_ERR_ADAPTER is set;
 *   - a rank 0 adapter adds nothing.
 *
 * Every floating-point input is an exact value (fp32 or bf16 widened) and all
 * arithmetic is in double.  The loops are the definition, in the order above;
 * an OpenMP loop over output rows only splits independent rows across threads.
 */
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_SEGMENTS 1
#define ORC_ERR_ADAPTER 2
#define ORC_ERR_RANK 4

/* Largest rank orc_layer accepts (its per-row v lives on the stack). */
#define ORC_MAX_RANK 4096

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Segments -> one adapter id per token.  seg_starts has S+1 entries: segment s
 * covers tokens seg_starts[s] .. seg_starts[s+1]-1 and uses seg_adapter[s].
 * Requires seg_starts[0] == 0, non-decreasing starts and seg_starts[S] == T;
 * otherwise returns ORC_ERR_SEGMENTS and leaves token_adapter unspecified.
 */
int orc_token_adapters(int S, const int32_t *seg_starts, const int32_t *seg_adapter,
                       int T, int32_t *token_adapter)
{
    if (S < 0 || T < 0 || seg_starts[0] != 0 || seg_starts[S] != T)
        return ORC_ERR_SEGMENTS;
    for (int s = 0; s < S; ++s)
        if (seg_starts[s + 1] < seg_starts[s])
            return ORC_ERR_SEGMENTS;
    for (int s = 0; s < S; ++s)
        for (int t = seg_starts[s]; t < seg_starts[s + 1]; ++t)
            token_adapter[t] = seg_adapter[s];
    return ORC_OK;
}

/* Classify token t's adapter: returns the adapter (>= 0), -1 for "none",
 * or -2 for an invalid id (sets *status). */
static int adapter_of(const int32_t *token_adapter, int t, int n_adapters,
                      const int32_t *rank, int ld_v, int *status)
{
    int a = token_adapter[t];
    if (a < 0)
        return -1;
    if (a >= n_adapters || rank[a] < 0) {
        *status |= ORC_ERR_ADAPTER;
        return -2;
    }
    if (ld_v >= 0 && rank[a] > ld_v) {
        *status |= ORC_ERR_RANK;
        return -2;
    }
    return a;
}

/*
 * Shrink for the listed rows: v[i][j] = sum_k x[rows[i]][k] * A_T_a[j][k] for
 * j < rank[a], a = token_adapter[rows[i]].  v is n_rows x ld_v; entries at
 * j >= rank[a], and rows without a valid adapter, are not written.
 */
int orc_shrink(int T, int h_in, const double *x, const int32_t *token_adapter,
               int n_adapters, const int32_t *rank, const double *AT, const int64_t *at_off,
               int n_rows, const int32_t *rows, int ld_v, double *v)
{
    int status = ORC_OK;
    (void)T;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int i = 0; i < n_rows; ++i) {
        int t = rows[i];
        int st = 0;
        int a = adapter_of(token_adapter, t, n_adapters, rank, ld_v, &st);
        status |= st;
        if (a < 0)
            continue;
        const double *xt = x + (size_t)t * h_in;
        const double *at = AT + at_off[a];
        for (int j = 0; j < rank[a]; ++j) {
            double acc = 0.0;
            for (int k = 0; k < h_in; ++k)
                acc += xt[k] * at[(size_t)j * h_in + k];
            v[(size_t)i * ld_v + j] = acc;
        }
    }
    return status;
}

/*
 * Expand for the listed rows: y[i][n] += scale[a] * sum_j v[i][j] * B_a[j][n].
 * y is n_rows x h_out and holds the starting output (y0) on entry; v is
 * n_rows x ld_v (row i belongs to token rows[i]).
 */
int orc_expand(int T, int h_out, const double *v, int ld_v, const int32_t *token_adapter,
               int n_adapters, const int32_t *rank, const double *scale,
               const double *B, const int64_t *b_off,
               int n_rows, const int32_t *rows, double *y)
{
    int status = ORC_OK;
    (void)T;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int i = 0; i < n_rows; ++i) {
        int t = rows[i];
        int st = 0;
        int a = adapter_of(token_adapter, t, n_adapters, rank, ld_v, &st);
        status |= st;
        if (a < 0)
            continue;
        const double *vi = v + (size_t)i * ld_v;
        const double *b = B + b_off[a];
        for (int n = 0; n < h_out; ++n) {
            double acc = 0.0;
            for (int j = 0; j < rank[a]; ++j)
                acc += vi[j] * b[(size_t)j * h_out + n];
            y[(size_t)i * h_out + n] += scale[a] * acc;
        }
    }
    return status;
}

/*
 * Whole adapted layer for the listed rows:
 *   y[i][n] += sum_k x[t][k] * W[n][k]                        (if W != NULL)
 *            + scale[a] * sum_j (sum_k x[t][k] * A_T_a[j][k]) * B_a[j][n]
 * with t = rows[i] and a = token_adapter[t].  W is h_out x h_in (row n is
 * output feature n).  y (n_rows x h_out) holds y0 on entry.  A row whose
 * adapter id is invalid gets the base term only and is flagged.
 */
int orc_layer(int T, int h_in, int h_out, const double *x, const double *W,
              const int32_t *token_adapter, int n_adapters, const int32_t *rank,
              const double *scale, const double *AT, const int64_t *at_off,
              const double *B, const int64_t *b_off,
              int n_rows, const int32_t *rows, double *y)
{
    int status = ORC_OK;
    (void)T;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int i = 0; i < n_rows; ++i) {
        int t = rows[i];
        int st = 0;
        int a = adapter_of(token_adapter, t, n_adapters, rank, -1, &st);
        status |= st;
        const double *xt = x + (size_t)t * h_in;
        double *yi = y + (size_t)i * h_out;
        if (W) {
            for (int n = 0; n < h_out; ++n) {
                double acc = 0.0;
                for (int k = 0; k < h_in; ++k)
                    acc += xt[k] * W[(size_t)n * h_in + k];
                yi[n] += acc;
            }
        }
        if (a < 0 || rank[a] == 0)
            continue;
        double vt[ORC_MAX_RANK];
        const double *at = AT + at_off[a];
        const double *b = B + b_off[a];
        int r = rank[a];
        if (r > ORC_MAX_RANK) {
            status |= ORC_ERR_RANK;
            continue;
        }
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int k = 0; k < h_in; ++k)
                acc += xt[k] * at[(size_t)j * h_in + k];
            vt[j] = acc;
        }
        for (int n = 0; n < h_out; ++n) {
            double acc = 0.0;
            for (int j = 0; j < r; ++j)
                acc += vt[j] * b[(size_t)j * h_out + n];
            yi[n] += scale[a] * acc;
        }
    }
    return status;
}
