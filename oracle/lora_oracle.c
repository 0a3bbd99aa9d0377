/*
 * lora_oracle.c -- plain fp64 reference of the LoRA adapter product.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; both sides only see the same seeded input arrays.
 *
 * Every function works in double precision on dense row-major arrays that hold
 * the exact (widened) values of the inputs.  Every output element is one sum
 * over its contraction index in ascending order, started from 0.0 and scaled
 * once at the end; the loops are nested so that inner loops walk contiguous
 * memory, and the only parallelism is OpenMP over independent output rows or
 * blocks of output elements, so the order of each sum is fixed.  The build
 * turns off floating-point contraction (no fused multiply-add), so results
 * are the same on every host.
 *
 * Sources (cited by page title and API entry):
 *   [NeMo lora_kernel] "nemo_automodel.components._peft.lora_kernel" API page:
 *       lora_forward_kernel / inner_kernel / block_vector_mul (forward),
 *       lora_da_dx_kernel / lora_da_dx_update_wrapper (dX, dlora_A),
 *       lora_db_kernel / lora_db_update_wrapper (dlora_B).
 *   [mstar lora.ops] "mstar.engine.resources.lora.ops" page:
 *       shrink, expand_fused, apply_linear_, gather_shrink, and the note on
 *       unspecified rows of h (zero adapter, columns past a slot's rank).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   R1  The forward adds into the output (block_vector_mul "adds the result").
 *   R2  The scale multiplies the final product once.
 *   R3  All single-adapter ops use the forward roles A (K x r), B (r x L).
 *   R7  Stacks: a [S][n*R][in], h [T][n*R], b [S][O][R]; one rank per slot.
 *   R8  A token whose slot is outside [0,S) or whose rank is outside [1,R]
 *       contributes nothing (same rule as an out-of-range id).
 *   R9  gather_shrink: an id outside [0,V) gives a zero row (written).
 *   R10 Unspecified h entries are written as zeros here.
 *
 * Parity pins (tests/test_oracle_pins.py): brute force through a different
 * association, rank-1 closed form, exact finite differences, invariants,
 * hand-worked fixtures.  Every function below is pinned by at least one of
 * them; none is "parity unpinned".
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Rows of dA / columns of dB whose running sums one thread keeps together
 * (cache blocking only: every element is still one ascending sum). */
#define ORACLE_KB 64
#define ORACLE_LB 256

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* A token takes part when its slot is in range and that slot's rank is in
 * [1, R] (reading R8 of the mstar lora.ops page). */
static int slot_active(int32_t slot, int32_t S, int32_t R, const int32_t *ranks)
{
    if (slot < 0 || slot >= S) return 0;
    return ranks[slot] >= 1 && ranks[slot] <= R;
}

/* ---------------------------------------------------------------------------
 * Single adapter, forward.  [NeMo lora_kernel] lora_forward_kernel computes
 * D = A x B x C with A (M,K) the input, B (K,N) lora_A, C (N,L) lora_B;
 * inner_kernel forms the (M,N) product with the scale and block_vector_mul
 * adds its product with C into D.  Here: Y = Y0 + s * (X*A)*B.
 * X [M][K], A [K][r], B [r][L], Y0/Y [M][L].
 * ------------------------------------------------------------------------- */
void oracle_lora_forward(int64_t M, int64_t K, int64_t L, int64_t r,
                         const double *X, const double *A, const double *B,
                         const double *Y0, double s, double *Y)
{
    /* Every sum runs over its contraction index in ascending order, starting
     * from 0.0; the loops are nested so that the inner loop walks contiguous
     * memory (h[j] and acc[l] are the running sums of their elements). */
    #pragma omp parallel
    {
        double *h = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
        double *acc = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        #pragma omp for schedule(static)
        for (int64_t m = 0; m < M; ++m) {
            for (int64_t j = 0; j < r; ++j) h[j] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double xk = X[m * K + k];
                for (int64_t j = 0; j < r; ++j) h[j] += xk * A[k * r + j];
            }
            for (int64_t l = 0; l < L; ++l) acc[l] = 0.0;
            for (int64_t j = 0; j < r; ++j) {
                const double hj = h[j];
                for (int64_t l = 0; l < L; ++l) acc[l] += hj * B[j * L + l];
            }
            for (int64_t l = 0; l < L; ++l) Y[m * L + l] = Y0[m * L + l] + s * acc[l];
        }
        free(acc);
        free(h);
    }
}

/* ---------------------------------------------------------------------------
 * Single adapter, backward for dX and dA.  [NeMo lora_kernel]
 * lora_da_dx_kernel forms DYB = DY x B and DX = DY x B x A (the backward
 * passes lora_B and lora_A transposed), and lora_da_dx_update_wrapper reduces
 * dlora_A from the input and DYB.  In forward roles:
 *   dyb = dY * B^T             [M][r]
 *   dX  = s * dyb * A^T        [M][K]
 *   dA  = s * X^T * dyb        [K][r]
 * ------------------------------------------------------------------------- */
void oracle_lora_backward_dx_da(int64_t M, int64_t K, int64_t L, int64_t r,
                                const double *X, const double *dY,
                                const double *A, const double *B, double s,
                                double *dX, double *dA)
{
    double *dyb = (double *)malloc(sizeof(double) * (size_t)(M * r > 0 ? M * r : 1));
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t l = 0; l < L; ++l) acc += dY[m * L + l] * B[j * L + l];
            dyb[m * r + j] = acc;
        }
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t j = 0; j < r; ++j) acc += dyb[m * r + j] * A[k * r + j];
            dX[m * K + k] = s * acc;
        }
    }
    /* dA[k][j] = s * (sum over m ascending of X[m][k] * dyb[m][j]); the rows k
     * are taken in blocks of ORACLE_KB so that a block's running sums stay in
     * cache while m advances. */
    #pragma omp parallel for schedule(static)
    for (int64_t k0 = 0; k0 < K; k0 += ORACLE_KB) {
        const int64_t k1 = k0 + ORACLE_KB < K ? k0 + ORACLE_KB : K;
        for (int64_t k = k0; k < k1; ++k)
            for (int64_t j = 0; j < r; ++j) dA[k * r + j] = 0.0;
        for (int64_t m = 0; m < M; ++m)
            for (int64_t k = k0; k < k1; ++k) {
                const double xk = X[m * K + k];
                for (int64_t j = 0; j < r; ++j) dA[k * r + j] += xk * dyb[m * r + j];
            }
        for (int64_t k = k0; k < k1; ++k)
            for (int64_t j = 0; j < r; ++j) dA[k * r + j] = s * dA[k * r + j];
    }
    free(dyb);
}

/* ---------------------------------------------------------------------------
 * Single adapter, backward for dB.  [NeMo lora_kernel] lora_db_kernel forms
 * AXT = lora_A^T x X^T, i.e. (X*A)^T, and lora_db_update_wrapper multiplies it
 * by the output gradient:  h = X*A [M][r],  dB = s * h^T * dY  [r][L].
 * ------------------------------------------------------------------------- */
void oracle_lora_backward_db(int64_t M, int64_t K, int64_t L, int64_t r,
                             const double *X, const double *A, const double *dY,
                             double s, double *dB)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)(M * r > 0 ? M * r : 1));
    /* h[m][j] = sum over k ascending of X[m][k] * A[k][j] */
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        double *hm = h + m * r;
        for (int64_t j = 0; j < r; ++j) hm[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double xk = X[m * K + k];
            for (int64_t j = 0; j < r; ++j) hm[j] += xk * A[k * r + j];
        }
    }
    /* dB[j][l] = s * (sum over m ascending of h[m][j] * dY[m][l]), the columns l
     * in blocks of ORACLE_LB whose running sums stay in cache while m advances */
    #pragma omp parallel for schedule(static)
    for (int64_t l0 = 0; l0 < L; l0 += ORACLE_LB) {
        const int64_t l1 = l0 + ORACLE_LB < L ? l0 + ORACLE_LB : L;
        for (int64_t j = 0; j < r; ++j)
            for (int64_t l = l0; l < l1; ++l) dB[j * L + l] = 0.0;
        for (int64_t m = 0; m < M; ++m)
            for (int64_t j = 0; j < r; ++j) {
                const double hj = h[m * r + j];
                for (int64_t l = l0; l < l1; ++l) dB[j * L + l] += hj * dY[m * L + l];
            }
        for (int64_t j = 0; j < r; ++j)
            for (int64_t l = l0; l < l1; ++l) dB[j * L + l] = s * dB[j * L + l];
    }
    free(h);
}

/* ---------------------------------------------------------------------------
 * Multi-adapter grouping of tokens by slot (the integer step in front of the
 * segmented kernels; the mstar lora.ops page requires it to run without a host
 * sync).  Definition: counts[s] = number of active tokens on slot s; perm lists
 * the active tokens ordered by (slot, token index).  Returns their number.
 * ------------------------------------------------------------------------- */
int64_t oracle_lora_group_by_slot(int64_t T, int32_t S, int32_t R,
                                  const int32_t *slots, const int32_t *ranks,
                                  int32_t *counts, int32_t *perm)
{
    int64_t n = 0;
    for (int32_t s = 0; s < S; ++s) counts[s] = 0;
    for (int64_t t = 0; t < T; ++t)
        if (slot_active(slots[t], S, R, ranks)) counts[slots[t]] += 1;
    for (int32_t s = 0; s < S; ++s) {
        if (counts[s] == 0) continue;
        for (int64_t t = 0; t < T; ++t)
            if (slots[t] == s && slot_active(s, S, R, ranks)) perm[n++] = (int32_t)t;
    }
    return n;
}

/* ---------------------------------------------------------------------------
 * shrink.  [mstar lora.ops] shrink: h[t] = x[t] @ a[slot(t)]^T, with
 * num_slices stacked rank blocks in a.  a [S][n*R][in], x [T][in],
 * h [T][n*R]:  h[t][i*R + j] = sum_k x[t][k] * a[slot][i*R + j][k], j < rank.
 * Rows of inactive tokens and columns j >= rank are unspecified (written 0).
 * ------------------------------------------------------------------------- */
void oracle_lora_shrink(int64_t T, int64_t in, int32_t S, int32_t R, int32_t n,
                        const int32_t *slots, const int32_t *ranks,
                        const double *x, const double *a, double *h)
{
    const int64_t NR = (int64_t)n * R;
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < NR; ++c) h[t * NR + c] = 0.0;
        int32_t slot = slots[t];
        if (!slot_active(slot, S, R, ranks)) continue;
        int32_t rank = ranks[slot];
        const double *as = a + (int64_t)slot * NR * in;
        for (int32_t i = 0; i < n; ++i) {
            for (int32_t j = 0; j < rank; ++j) {
                const double *arow = as + ((int64_t)i * R + j) * in;
                double acc = 0.0;
                for (int64_t k = 0; k < in; ++k) acc += x[t * in + k] * arow[k];
                h[t * NR + (int64_t)i * R + j] = acc;
            }
        }
    }
}

/* ---------------------------------------------------------------------------
 * expand.  [mstar lora.ops] expand_fused:
 *   y[t, slice i] += scalings[slot(t)] * h[t, slice i] @ b[slot(t), slice i]^T
 * Slice i covers output columns off_i .. off_i + out_slices[i] - 1 (off_i the
 * running sum); b [S][O][R]; only j < rank is read (the page: the expand does
 * not read columns past the rank nor rows of the zero adapter).
 * Y0 is the incoming y, Y the result.
 * ------------------------------------------------------------------------- */
void oracle_lora_expand(int64_t T, int32_t S, int32_t R, int32_t n,
                        const int32_t *out_slices, const int32_t *slots,
                        const int32_t *ranks, const double *scalings,
                        const double *h, const double *b,
                        const double *Y0, double *Y)
{
    int64_t O = 0;
    for (int32_t i = 0; i < n; ++i) O += out_slices[i];
    const int64_t NR = (int64_t)n * R;
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < O; ++c) Y[t * O + c] = Y0[t * O + c];
        int32_t slot = slots[t];
        if (!slot_active(slot, S, R, ranks)) continue;
        int32_t rank = ranks[slot];
        double sc = scalings[slot];
        const double *bs = b + (int64_t)slot * O * R;
        int64_t off = 0;
        for (int32_t i = 0; i < n; ++i) {
            for (int64_t c = 0; c < out_slices[i]; ++c) {
                double acc = 0.0;
                for (int32_t j = 0; j < rank; ++j)
                    acc += h[t * NR + (int64_t)i * R + j] * bs[(off + c) * R + j];
                Y[t * O + off + c] = Y0[t * O + off + c] + sc * acc;
            }
            off += out_slices[i];
        }
    }
}

/* ---------------------------------------------------------------------------
 * apply_linear.  [mstar lora.ops] apply_linear_: shrink, then expand into y
 * (the page allows a backend to fuse them; the oracle composes them).
 * ------------------------------------------------------------------------- */
void oracle_lora_apply_linear(int64_t T, int64_t in, int32_t S, int32_t R, int32_t n,
                              const int32_t *out_slices, const int32_t *slots,
                              const int32_t *ranks, const double *scalings,
                              const double *x, const double *a, const double *b,
                              const double *Y0, double *Y)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)(T * n * R > 0 ? T * n * R : 1));
    oracle_lora_shrink(T, in, S, R, n, slots, ranks, x, a, h);
    oracle_lora_expand(T, S, R, n, out_slices, slots, ranks, scalings, h, b, Y0, Y);
    free(h);
}

/* ---------------------------------------------------------------------------
 * gather_shrink.  [mstar lora.ops] gather_shrink: h[t] = a[slot(t)][:, ids[t]],
 * the shrink of the token's one-hot row; an id outside [0, V) contributes
 * nothing (reading R9: a zero row).  a [S][R][V], h [T][R].
 * ------------------------------------------------------------------------- */
void oracle_lora_gather_shrink(int64_t T, int64_t V, int32_t S, int32_t R,
                               const int32_t *slots, const int32_t *ranks,
                               const int64_t *ids, const double *a, double *h)
{
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < R; ++j) h[t * R + j] = 0.0;
        int32_t slot = slots[t];
        if (!slot_active(slot, S, R, ranks)) continue;
        int64_t id = ids[t];
        if (id < 0 || id >= V) continue;
        int32_t rank = ranks[slot];
        for (int32_t j = 0; j < rank; ++j)
            h[t * R + j] = a[((int64_t)slot * R + j) * V + id];
    }
}
