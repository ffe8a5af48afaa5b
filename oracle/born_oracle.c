/*
 * CPU oracle for causal Born attention — TEST INFRASTRUCTURE ONLY (tests, the
 * package smoke check and the benchmark's CPU baseline call it; the CUDA
 * library never links or calls it).
 *
 * Source: "Complex Phase-State Dynamics Reduce the Optimization Steps of
 * Sequence Models" (arXiv 2608.14691), section 5.5, equation (5), and
 * Appendix A, Algorithm 3.  Per head, with complex queries q_i, keys k_j and
 * values v_j in C^D and a positive temperature tau_i per query position:
 *     s_ij = |<q_i | k_j>|^2 / (D tau_i)          for j <= i
 *     psi_i = (sum_{j<=i} s_ij v_j) / (sum_{j<=i} s_ij)
 * where <q|k> = sum_a conj(q_a) k_a (the bra conjugates).  The steps are taken
 * in that order, in double precision, one query at a time.
 *
 * Reading: the pages do not say what psi_i is when every s_ij of a row is zero
 * (q_i orthogonal to every earlier key); the ratio is then 0/0 and psi_i is
 * returned as 0.
 *
 * A second function evaluates the same quantity through an independent route,
 * the feature-map (recurrent) form: |<q|k>|^2 = q^H (k k^H) q, so
 *     D tau_i sum_j s_ij v_j[m] = q_i^H W_i[m] q_i,  W_i[m] = sum_{j<=i} v_j[m] k_j k_j^H
 *     D tau_i sum_j s_ij        = q_i^H Z_i q_i,     Z_i    = sum_{j<=i} k_j k_j^H
 * carried as D x D matrices from position to position.  It shares no
 * arithmetic with the direct form and is used only to pin it.
 *
 * Layouts (row-major; complex = interleaved [re, im] doubles):
 *   q, k, v, psi [Bz,T,H,D]     tau [Bz,T,H]
 */
#include <complex.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

typedef double complex cplx;

static cplx cld(const double* p, int64_t i) { return p[2 * i] + I * p[2 * i + 1]; }
static void cst(double* p, int64_t i, cplx v) {
    p[2 * i] = creal(v);
    p[2 * i + 1] = cimag(v);
}

/* Algorithm 3, step by step. */
void oracle_born_attention(int64_t Bz, int64_t T, int64_t H, int64_t D, const double* q, const double* k,
                           const double* v, const double* tau, double* psi) {
#pragma omp parallel for collapse(2)
    for (int64_t b = 0; b < Bz; ++b)
        for (int64_t h = 0; h < H; ++h) {
            cplx* num = (cplx*)malloc((size_t)D * sizeof(cplx));
            for (int64_t i = 0; i < T; ++i) {
                const int64_t qi = ((b * T + i) * H + h) * D;
                for (int64_t m = 0; m < D; ++m) num[m] = 0;
                double den = 0.0;
                for (int64_t j = 0; j <= i; ++j) {
                    const int64_t kj = ((b * T + j) * H + h) * D;
                    cplx g = 0;
                    for (int64_t a = 0; a < D; ++a) g += conj(cld(q, qi + a)) * cld(k, kj + a);  /* <q_i|k_j> */
                    const double s = (creal(g) * creal(g) + cimag(g) * cimag(g)) / ((double)D * tau[(b * T + i) * H + h]);
                    for (int64_t m = 0; m < D; ++m) num[m] += s * cld(v, kj + m);
                    den += s;
                }
                for (int64_t m = 0; m < D; ++m) cst(psi, qi + m, den != 0.0 ? num[m] / den : 0.0);
            }
            free(num);
        }
}

/* The feature-map form (see the header); independent of the function above. */
void oracle_born_attention_feature_map(int64_t Bz, int64_t T, int64_t H, int64_t D, const double* q,
                                       const double* k, const double* v, double* psi) {
#pragma omp parallel for collapse(2)
    for (int64_t b = 0; b < Bz; ++b)
        for (int64_t h = 0; h < H; ++h) {
            cplx* W = (cplx*)calloc((size_t)(D * D * D), sizeof(cplx)); /* W[m][a][c] */
            cplx* Z = (cplx*)calloc((size_t)(D * D), sizeof(cplx));     /* Z[a][c]    */
            for (int64_t t = 0; t < T; ++t) {
                const int64_t o = ((b * T + t) * H + h) * D;
                for (int64_t a = 0; a < D; ++a)
                    for (int64_t c = 0; c < D; ++c) {
                        const cplx kk = cld(k, o + a) * conj(cld(k, o + c));  /* (k k^H)[a][c] */
                        Z[a * D + c] += kk;
                        for (int64_t m = 0; m < D; ++m) W[(m * D + a) * D + c] += cld(v, o + m) * kk;
                    }
                /* q^H M q = sum_{a,c} conj(q_a) M[a][c] q_c */
                double den = 0.0;
                for (int64_t a = 0; a < D; ++a)
                    for (int64_t c = 0; c < D; ++c) den += creal(conj(cld(q, o + a)) * Z[a * D + c] * cld(q, o + c));
                for (int64_t m = 0; m < D; ++m) {
                    cplx nm = 0;
                    for (int64_t a = 0; a < D; ++a)
                        for (int64_t c = 0; c < D; ++c) nm += conj(cld(q, o + a)) * W[(m * D + a) * D + c] * cld(q, o + c);
                    cst(psi, o + m, den != 0.0 ? nm / den : 0.0);
                }
            }
            free(W);
            free(Z);
        }
}
