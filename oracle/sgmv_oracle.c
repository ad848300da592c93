/*
 * sgmv_oracle.c -- plain fp64 CPU oracle for Segmented Gather Matrix-Vector
 * multiplication (SGMV), the multi-LoRA kernel of Punica.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg are the only code that may load this file's library.  The
 * product (the CUDA library and its Python binding) never calls it, includes
 * it or shares anything with it.
 *
 * Pages this follows (cited by title and section):
 *   [Article]  "Punica: when LoRA fine-tuned models need multi-tenant serving"
 *              (omica.com.cn practitioner article, in Chinese)
 *                §2.1 LoRA computation: y = xW + xAB, A is [H1, r], B is [r, H2].
 *                §2.2 SGMV: step 1 gathers each request's A_i out of one
 *                     contiguous stack of all adapters and forms v_i = x_i A_i
 *                     (a vector of length r); step 2 multiplies v_i by B_i,
 *                     all B_i stacked the same way.
 *                §5.1 the batch builder groups requests by LoRA id.
 *   [Review]   "Punica: Multi-Tenant LoRA Serving" (nubint.ai paper review),
 *                "Proposed method": SGMV batches the different LoRA models'
 *                GPU work by operating on segmented inputs and outputs.
 *   [Q&A]      "How to deploy several LoRA adapters without reloading the base
 *              model (Punica, S-LoRA)?" (aivaro.ru)
 *                §3.1 each request computes x = x + (x @ A) @ B with its own
 *                     A and B;
 *                §3.2 adapter weights live in one contiguous buffer and the
 *                     kernel selects them by index (segmented gather/scatter).
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes):
 *   - the LoRA delta is multiplied by one scalar `scale` per call;
 *   - stacked layouts are A[L][H1][r] and B[L][r][H2], row-major;
 *   - a segment whose adapter id is -1 has no adapter: its v rows are zero
 *     and its Y rows are left as they are;
 *   - `perm` (optional) maps a sorted position p to the physical row of X
 *     and Y that sits there; NULL means position p is row p;
 *   - grouping is a stable sort by adapter id: ascending id, original row
 *     order within an id, one segment per id that occurs.
 *
 * Everything is computed in double precision, sums taken in index order.
 * There is no blocking, fusion or reordering beyond the definition.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

/* Physical row of sorted position p. */
static int32_t row_of(const int32_t *perm, int32_t p)
{
    return perm ? perm[p] : p;
}

/*
 * Group rows by adapter id ([Article] §5.1; [Q&A] §3.2).
 *
 * row_adapter[T]: adapter id of each row, in [-1, L).
 * Outputs: perm[T] (sorted position -> row), seg_ptr[S+1], idx[S], *S_out.
 * Returns 0, or 1 if an id is outside [-1, L) (outputs are then undefined).
 */
int oracle_build_segments(const int32_t *row_adapter, int32_t T, int32_t L,
                          int32_t *perm, int32_t *seg_ptr, int32_t *idx,
                          int32_t *S_out)
{
    for (int32_t t = 0; t < T; ++t)
        if (row_adapter[t] < -1 || row_adapter[t] >= L)
            return 1;

    int32_t s = 0, p = 0;
    seg_ptr[0] = 0;
    for (int32_t id = -1; id < L; ++id) {
        int32_t first = p;
        for (int32_t t = 0; t < T; ++t)
            if (row_adapter[t] == id)
                perm[p++] = t;
        if (p > first) {
            idx[s] = id;
            seg_ptr[s + 1] = p;
            ++s;
        }
    }
    *S_out = s;
    return 0;
}

/*
 * Shrink, the first SGMV step ([Article] §2.2):
 *   v[p][k] = sum_h X[row(p)][h] * A[idx[s]][h][k]   for p in segment s.
 * v is [T][r], indexed by sorted position.  Rows of segments with idx -1
 * get v = 0.  Positions outside every segment are not written.
 */
void oracle_sgmv_shrink(double *v, const double *X, const double *A,
                        const int32_t *perm, const int32_t *seg_ptr,
                        const int32_t *idx, int32_t S, int32_t H1, int32_t r)
{
    for (int32_t s = 0; s < S; ++s) {
        int32_t a = idx[s];
        for (int32_t p = seg_ptr[s]; p < seg_ptr[s + 1]; ++p) {
            const double *x = X + (size_t)row_of(perm, p) * H1;
            for (int32_t k = 0; k < r; ++k) {
                double acc = 0.0;
                if (a >= 0)
                    for (int32_t h = 0; h < H1; ++h)
                        acc += x[h] * A[((size_t)a * H1 + h) * r + k];
                v[(size_t)p * r + k] = acc;
            }
        }
    }
}

/*
 * Expand, the second SGMV step ([Article] §2.2), added to the output
 * ([Q&A] §3.1):
 *   Y[row(p)][j] += scale * sum_k v[p][k] * B[idx[s]][k][j]   for p in segment s.
 * Segments with idx -1 leave their rows unchanged.
 */
void oracle_sgmv_expand(double *Y, const double *v, const double *B,
                        double scale, const int32_t *perm,
                        const int32_t *seg_ptr, const int32_t *idx, int32_t S,
                        int32_t H2, int32_t r)
{
    for (int32_t s = 0; s < S; ++s) {
        int32_t a = idx[s];
        if (a < 0)
            continue;
        for (int32_t p = seg_ptr[s]; p < seg_ptr[s + 1]; ++p) {
            double *y = Y + (size_t)row_of(perm, p) * H2;
            for (int32_t j = 0; j < H2; ++j) {
                double acc = 0.0;
                for (int32_t k = 0; k < r; ++k)
                    acc += v[(size_t)p * r + k] * B[((size_t)a * r + k) * H2 + j];
                y[j] += scale * acc;
            }
        }
    }
}

/*
 * Whole SGMV LoRA update: shrink, then expand.  T is the number of sorted
 * positions (size of the temporary v).  Returns 0, or 1 if the temporary
 * cannot be allocated.
 */
int oracle_sgmv_apply(double *Y, const double *X, const double *A,
                      const double *B, double scale, const int32_t *perm,
                      const int32_t *seg_ptr, const int32_t *idx, int32_t S,
                      int32_t T, int32_t H1, int32_t H2, int32_t r)
{
    double *v = (double *)calloc((size_t)(T > 0 ? T : 1) * (size_t)(r > 0 ? r : 1),
                                 sizeof(double));
    if (!v)
        return 1;
    oracle_sgmv_shrink(v, X, A, perm, seg_ptr, idx, S, H1, r);
    oracle_sgmv_expand(Y, v, B, scale, perm, seg_ptr, idx, S, H2, r);
    free(v);
    return 0;
}

/*
 * Fused base linear + LoRA: the LoRA layer of [Article] §2.1, y = xW + xAB,
 * in one call, as [Q&A] §3.2 ("Fused Kernel": the LoRA transform merged into
 * the base model's linear layer) describes it:
 *   Y[t][j] = sum_h X[t][h] * W[h][j]                          every row t,
 *   then the SGMV update above for every segment with an adapter.
 * W is [H1][H2] (x W, like x A and v B).  Y [T][H2] is overwritten: rows of
 * no adapter hold the base output alone.  Returns 0, or 1 if the temporary
 * of the update cannot be allocated.
 */
int oracle_fused_linear_lora(double *Y, const double *X, const double *W,
                             const double *A, const double *B, double scale,
                             const int32_t *perm, const int32_t *seg_ptr,
                             const int32_t *idx, int32_t S, int32_t T,
                             int32_t H1, int32_t H2, int32_t r)
{
    for (int32_t t = 0; t < T; ++t) {
        const double *x = X + (size_t)t * H1;
        double *y = Y + (size_t)t * H2;
        for (int32_t j = 0; j < H2; ++j) {
            double acc = 0.0;
            for (int32_t h = 0; h < H1; ++h)
                acc += x[h] * W[(size_t)h * H2 + j];
            y[j] = acc;
        }
    }
    return oracle_sgmv_apply(Y, X, A, B, scale, perm, seg_ptr, idx, S, T, H1, H2, r);
}
