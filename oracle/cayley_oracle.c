/*
 * CPU oracle for the per-coordinate Cayley-phase recurrence — TEST
 * INFRASTRUCTURE ONLY (tests, the package smoke check and the benchmark's CPU
 * baseline call it; the CUDA library never links or calls it).
 *
 * Source: "Complex Phase-State Dynamics Reduce the Optimization Steps of
 * Sequence Models" (arXiv 2608.14691).
 *   - Section 5.2, equations (2)-(3): per head, a complex state psi in C^N
 *     evolves coordinatewise, psi <- a_t (.) psi + b_t, with
 *     a_t = alpha_t lambda_t, alpha = sigmoid(u) (the gate, |a| = alpha) and
 *     lambda = (1 + i phi) / (1 - i phi) (the diagonal Cayley phase, |lambda| = 1).
 *     Appendix A, Algorithm 1 computes a from (phi, u) in exactly this order.
 *   - Section 5.5: the state-space readout y_t = conj(C_t) (.) psi_t, taken
 *     after the update (the readout of the state that includes b_t).
 *   - Section 5.3, equation (4), and Appendix A, Algorithm 2: the chunked polar
 *     scan.  Per chunk of length C: l = clamp(cumsum(log|a|), lo, 0),
 *     theta = cumsum(arg a), P = e^l e^{i theta}, P^-1 = e^-l e^{-i theta},
 *     states = P (.) (x0 + cumsum(b (.) P^-1)), and the chunk's last state
 *     seeds the next chunk.  The pages clamp at lo = -30.
 *
 * Reading: the recurrence (2) is the definition.  Algorithm 2 reaches it
 * exactly (up to rounding) only while no within-chunk cumulative log-gate
 * falls below the clamp; below it the clamp changes the result, so the
 * algorithm is restated here step by step as a second function, with the
 * clamp as a parameter (lo = -infinity turns it off).
 *
 * Index convention: token t updates the state with (a_t, b_t) and is then
 * read out; psi before token 0 is psi0 (zero when absent).
 *
 * Layouts (row-major; complex = interleaved [re, im] doubles):
 *   phi, u [Bz,T,H,N]   b, C, y [Bz,T,H,N]   psi0, psi_final [Bz,H,N]
 */
#include <complex.h>
#include <math.h>
#include <stdint.h>

typedef double complex cplx;

static cplx cld(const double* p, int64_t i) { return p[2 * i] + I * p[2 * i + 1]; }
static void cst(double* p, int64_t i, cplx v) {
    p[2 * i] = creal(v);
    p[2 * i + 1] = cimag(v);
}

/* Algorithm 1: the transition coefficient of one coordinate. */
static cplx cayley_coefficient(double phi, double u) {
    const cplx lambda = (1.0 + I * phi) / (1.0 - I * phi);
    const double alpha = 1.0 / (1.0 + exp(-u));
    return alpha * lambda;
}

void oracle_cayley_coefficients(int64_t n, const double* phi, const double* u, double* a) {
    for (int64_t i = 0; i < n; ++i) cst(a, i, cayley_coefficient(phi[i], u[i]));
}

/* Equation (2) step by step, with the section 5.5 readout. */
void oracle_cayley_recurrence(int64_t Bz, int64_t T, int64_t H, int64_t N, const double* phi, const double* u,
                              const double* b, const double* C, const double* psi0, double* y,
                              double* psi_final) {
#pragma omp parallel for collapse(3)
    for (int64_t bb = 0; bb < Bz; ++bb)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t k = 0; k < N; ++k) {
                const int64_t s = (bb * H + h) * N + k;
                cplx psi = psi0 ? cld(psi0, s) : 0.0;
                for (int64_t t = 0; t < T; ++t) {
                    const int64_t i = ((bb * T + t) * H + h) * N + k;
                    psi = cayley_coefficient(phi[i], u[i]) * psi + cld(b, i);
                    cst(y, i, conj(cld(C, i)) * psi);
                }
                if (psi_final) cst(psi_final, s, psi);
            }
}

/* Algorithm 2 with the clamp bound `lo` (the pages use -30; -INFINITY = off). */
void oracle_cayley_chunked(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t chunk, double lo,
                           const double* phi, const double* u, const double* b, const double* C,
                           const double* psi0, double* y, double* psi_final) {
#pragma omp parallel for collapse(3)
    for (int64_t bb = 0; bb < Bz; ++bb)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t k = 0; k < N; ++k) {
                const int64_t s = (bb * H + h) * N + k;
                cplx x0 = psi0 ? cld(psi0, s) : 0.0;
                for (int64_t c0 = 0; c0 < T; c0 += chunk) {
                    const int64_t m = (T - c0 < chunk) ? T - c0 : chunk;
                    double cum_log = 0.0, cum_arg = 0.0; /* the two cumsums of line 1 */
                    cplx acc = 0.0;                      /* cumsum(b (.) P^-1) */
                    cplx state = x0;
                    for (int64_t r = 0; r < m; ++r) {
                        const int64_t i = ((bb * T + c0 + r) * H + h) * N + k;
                        const cplx a = cayley_coefficient(phi[i], u[i]);
                        cum_log += log(cabs(a));
                        cum_arg += carg(a);
                        const double l = fmin(fmax(cum_log, lo), 0.0);
                        const cplx P = exp(l) * cexp(I * cum_arg);
                        const cplx Pinv = exp(-l) * cexp(-I * cum_arg);
                        acc += cld(b, i) * Pinv;
                        state = P * (x0 + acc);
                        cst(y, i, conj(cld(C, i)) * state);
                    }
                    x0 = state; /* the final state carried to the next chunk */
                }
                if (psi_final) cst(psi_final, s, x0);
            }
}
