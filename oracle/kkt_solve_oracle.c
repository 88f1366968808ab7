/*
 * Plain CPU oracle for the chunk-forward kkt_solve step of Gated DeltaNet.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code with the CUDA path.
 *
 * What it computes (all arithmetic in IEEE double, dense explicit loops):
 *   For every sequence, every chunk [s, s+L) of at most C tokens counted from
 *   the sequence start, and every head h:
 *     A[i][j] = beta_i * (sum_d k_i[d] * k_j[d]) * exp(g_i - g_j)   for j < i < L
 *     A[i][j] = 0                                                   otherwise
 *     X = (I + A)^{-1}, found row by row by forward substitution:
 *         X[i][:] = e_i - sum_{j<i} A[i][j] * X[j][:]
 *     out[s+i][h][j] = X[i][j] for j < L, and 0 for L <= j < C.
 * Sources:
 *   - MindSpeed-Ops PR #135 page ("feat(triton): add
 *     chunk_gated_delta_rule_fwd_kkt_solve"), section "What this PR does":
 *     one call equals solve_tril(chunk_scaled_dot_kkt_fwd(...)), i.e. a scaled
 *     K*K^T inside each chunk followed by a lower-triangular solve; the API
 *     block says the result is (I + A)^{-1} with shape [B, T, H, chunk].
 *   - same page, bot summary ("主要改动"): the gate factor is the natural
 *     exponential of a difference of the cumulative log-gates; chunks restart
 *     at each cu_seqlens boundary (the T_local fix); g = None and beta = None
 *     are allowed.
 *   - PyPTO page "GatedDeltaRule算子性能优化案例", section 3.3.1: the inverse is
 *     a fixed-count row-by-row update, which is the forward substitution above.
 * The two halves of that chain are also given on their own, as the page's
 * unfused chain has them (same page, "What this PR does": the fused call
 * replaces chunk_scaled_dot_kkt_fwd followed by solve_tril, which write and
 * read A as [B, T, H, chunk]):
 *   oracle_chunk_A*      A itself, rows of real tokens, zero on and above the
 *                        diagonal and past the chunk;
 *   oracle_solve_tril*   (I + A)^{-1} of a given A by the same substitution,
 *                        reading only its strictly lower part.
 * Readings where the pages are silent: beta scales row i; the exponent is not
 *   clamped here (the Ascend kernel clamps it to [-50, 50], which never binds
 *   for chunk-local decays); g = NULL means g = 0, beta = NULL means beta = 1.
 * The pages print no output values, so the oracle is pinned by mathematics:
 * closed forms, brute-force inversion and invariants (tests/test_oracle_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* One chunk of one head.
 *   L      rows in the chunk (1 <= L <= C)
 *   C      chunk size = output row width
 *   K      head dimension
 *   kc     row r of the chunk's keys is kc[r*ldk + d], d < K
 *   g, beta  element r is g[r*ldg] (NULL allowed)
 *   out    row r is out[r*ldo + j], j < C
 * Returns 0, or -1 when a scratch allocation fails. */
int oracle_kkt_solve_chunk(int64_t L, int64_t C, int64_t K,
                           const double *kc, int64_t ldk,
                           const double *g, int64_t ldg,
                           const double *beta, int64_t ldb,
                           double *out, int64_t ldo)
{
    double *A = (double *)calloc((size_t)(L * L), sizeof(double));
    double *X = (double *)calloc((size_t)(L * L), sizeof(double));
    if (!A || !X) {
        free(A);
        free(X);
        return -1;
    }
    /* Step 1: the strictly lower matrix A. */
    for (int64_t i = 0; i < L; ++i) {
        for (int64_t j = 0; j < i; ++j) {
            double dot = 0.0;
            for (int64_t d = 0; d < K; ++d)
                dot += kc[i * ldk + d] * kc[j * ldk + d];
            double bi = beta ? beta[i * ldb] : 1.0;
            double gate = g ? exp(g[i * ldg] - g[j * ldg]) : 1.0;
            A[i * L + j] = bi * dot * gate;
        }
    }
    /* Step 2: (I + A) X = I, one row at a time. */
    for (int64_t i = 0; i < L; ++i) {
        for (int64_t c = 0; c < L; ++c) {
            double v = (i == c) ? 1.0 : 0.0;
            for (int64_t j = 0; j < i; ++j)
                v -= A[i * L + j] * X[j * L + c];
            X[i * L + c] = v;
        }
    }
    /* Step 3: rows of real tokens only; columns past the chunk are zero. */
    for (int64_t i = 0; i < L; ++i)
        for (int64_t c = 0; c < C; ++c)
            out[i * ldo + c] = (c < L) ? X[i * L + c] : 0.0;
    free(A);
    free(X);
    return 0;
}

/* The whole tensor for heads [h_begin, h_end).
 *   k     [Ntok, H, K]   (Ntok = nseq*T fixed-length, or T packed)
 *   g     [Ntok, H] or NULL;  beta [Ntok, H] or NULL
 *   cu    NULL: sequence n covers rows [n*T, (n+1)*T) for n < nseq;
 *         else sequence n covers rows [cu[n], cu[n+1]) for n < nseq.
 *   out   [Ntok, H, C]; rows of real tokens are written, others untouched.
 * Returns 0, -1 on an allocation failure, -2 on a bad argument. */
int oracle_kkt_solve(const double *k, const double *g, const double *beta,
                     const int32_t *cu, int64_t nseq, int64_t T, int64_t H,
                     int64_t K, int64_t C, double *out,
                     int64_t h_begin, int64_t h_end)
{
    if (!k || !out || nseq < 0 || T < 0 || H <= 0 || K <= 0 || C <= 0)
        return -2;
    for (int64_t n = 0; n < nseq; ++n) {
        int64_t s = cu ? (int64_t)cu[n] : n * T;
        int64_t e = cu ? (int64_t)cu[n + 1] : (n + 1) * T;
        if (e < s)
            return -2;
        for (int64_t c0 = s; c0 < e; c0 += C) {
            int64_t L = (e - c0 < C) ? (e - c0) : C;
            for (int64_t h = h_begin; h < h_end; ++h) {
                int rc = oracle_kkt_solve_chunk(
                    L, C, K, k + (c0 * H + h) * K, H * K,
                    g ? g + c0 * H + h : NULL, H,
                    beta ? beta + c0 * H + h : NULL, H,
                    out + (c0 * H + h) * C, H * C);
                if (rc)
                    return rc;
            }
        }
    }
    return 0;
}

/* A of one chunk: out row r is A[r][0..C), A[i][j] as above for j < i < L and
 * 0 elsewhere.  Same arguments as oracle_kkt_solve_chunk. */
int oracle_chunk_A_chunk(int64_t L, int64_t C, int64_t K,
                         const double *kc, int64_t ldk,
                         const double *g, int64_t ldg,
                         const double *beta, int64_t ldb,
                         double *out, int64_t ldo)
{
    for (int64_t i = 0; i < L; ++i) {
        for (int64_t j = 0; j < C; ++j) {
            double a = 0.0;
            if (j < i) {
                double dot = 0.0;
                for (int64_t d = 0; d < K; ++d)
                    dot += kc[i * ldk + d] * kc[j * ldk + d];
                double bi = beta ? beta[i * ldb] : 1.0;
                double gate = g ? exp(g[i * ldg] - g[j * ldg]) : 1.0;
                a = bi * dot * gate;
            }
            out[i * ldo + j] = a;
        }
    }
    return 0;
}

/* (I + A)^{-1} of one chunk from a given A (row r is Ain[r*lda + j]; only
 * j < r < L is read), by forward substitution; out rows as in
 * oracle_kkt_solve_chunk.  Returns 0, or -1 when a scratch allocation fails. */
int oracle_solve_tril_chunk(int64_t L, int64_t C, const double *Ain, int64_t lda,
                            double *out, int64_t ldo)
{
    double *X = (double *)calloc((size_t)(L * L), sizeof(double));
    if (!X)
        return -1;
    for (int64_t i = 0; i < L; ++i) {
        for (int64_t c = 0; c < L; ++c) {
            double v = (i == c) ? 1.0 : 0.0;
            for (int64_t j = 0; j < i; ++j)
                v -= Ain[i * lda + j] * X[j * L + c];
            X[i * L + c] = v;
        }
    }
    for (int64_t i = 0; i < L; ++i)
        for (int64_t c = 0; c < C; ++c)
            out[i * ldo + c] = (c < L) ? X[i * L + c] : 0.0;
    free(X);
    return 0;
}

/* Whole-tensor forms for heads [h_begin, h_end), with the sequence layout of
 * oracle_kkt_solve.  oracle_chunk_A writes A [Ntok, H, C] from k, g, beta;
 * oracle_solve_tril reads A [Ntok, H, C] and writes out [Ntok, H, C]. */
int oracle_chunk_A(const double *k, const double *g, const double *beta,
                   const int32_t *cu, int64_t nseq, int64_t T, int64_t H,
                   int64_t K, int64_t C, double *A,
                   int64_t h_begin, int64_t h_end)
{
    if (!k || !A || nseq < 0 || T < 0 || H <= 0 || K <= 0 || C <= 0)
        return -2;
    for (int64_t n = 0; n < nseq; ++n) {
        int64_t s = cu ? (int64_t)cu[n] : n * T;
        int64_t e = cu ? (int64_t)cu[n + 1] : (n + 1) * T;
        if (e < s)
            return -2;
        for (int64_t c0 = s; c0 < e; c0 += C) {
            int64_t L = (e - c0 < C) ? (e - c0) : C;
            for (int64_t h = h_begin; h < h_end; ++h)
                oracle_chunk_A_chunk(L, C, K, k + (c0 * H + h) * K, H * K,
                                     g ? g + c0 * H + h : NULL, H,
                                     beta ? beta + c0 * H + h : NULL, H,
                                     A + (c0 * H + h) * C, H * C);
        }
    }
    return 0;
}

int oracle_solve_tril(const double *A, const int32_t *cu, int64_t nseq, int64_t T,
                      int64_t H, int64_t C, double *out, int64_t h_begin, int64_t h_end)
{
    if (!A || !out || nseq < 0 || T < 0 || H <= 0 || C <= 0)
        return -2;
    for (int64_t n = 0; n < nseq; ++n) {
        int64_t s = cu ? (int64_t)cu[n] : n * T;
        int64_t e = cu ? (int64_t)cu[n + 1] : (n + 1) * T;
        if (e < s)
            return -2;
        for (int64_t c0 = s; c0 < e; c0 += C) {
            int64_t L = (e - c0 < C) ? (e - c0) : C;
            for (int64_t h = h_begin; h < h_end; ++h) {
                int rc = oracle_solve_tril_chunk(L, C, A + (c0 * H + h) * C, H * C,
                                                 out + (c0 * H + h) * C, H * C);
                if (rc)
                    return rc;
            }
        }
    }
    return 0;
}
