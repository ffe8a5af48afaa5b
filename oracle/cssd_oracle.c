/*
 * CPU oracle for the complex SSD (complex-valued diagonal state space) —
 * TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, double-precision restatement of what the method computes.  Only
 * the tests, the package's smoke check and the benchmark's CPU-baseline leg
 * call it; the CUDA library never links or calls it, and the two share no code.
 *
 * Sources (the pages' notation: x_t token content, B_t input coupling, C_t
 * readout, dt_t raw step, A per-head complex rate, state h_t of N x P per head):
 *   - Discretisation a_t = exp(softplus(dt_t) * A), softplus on the real dt
 *     first, then the complex exponential: "Complex-Valued State Spaces"
 *     (Mamba-3-Lite docs), sections "Discretization" and "The discretization".
 *   - Sequential recurrence h_t = a_t h_{t-1} + B_t x_t^T (outer product, no
 *     conjugate), readout after the update y_t = C_t^T h_t (sum over the N
 *     state rows, no conjugate): same page, "The discretization" code
 *     walkthrough, and "SSD Theory" section 2.  The skip term + D x_t and a
 *     complex y are the readout of the recurrence as the workload states it.
 *   - Chunkwise decomposition (pad, inclusive within-chunk cumsum, segment
 *     matrix L, Y_diag, per-chunk states S_c, inter-chunk state, Y_off):
 *     "The Chunkwise Complex SSD Algorithm" sections 4.1-4.5 and "SSD Theory"
 *     sections 4.2-4.5.  The carry-in state follows the theorem
 *     H_c = sum_{c'<c} exp(CD[c-1] - CD[c']) S_c' ("SSD Theory" 4.5), not the
 *     page's own propagation code, which that page's Pitfalls section shows
 *     to be misaligned when chunk totals differ.
 *   - Constant-input closed form: burn-mamba "Module step_constant", the
 *     geometric series in the per-step factor, specialised to this recurrence
 *     (no input rotation, trapezoid weights beta = 0, gamma = 1).
 *
 * Readings where the pages leave a step open:
 *   - padded positions (t >= T inside the last chunk) contribute x = B = C = 0
 *     and decay exactly 1, so the final state is the state after token T-1;
 *   - y is complex (its real part is the pages' real output when D = 0);
 *   - D is a real per-head scalar broadcast over P.
 *
 * Complex numbers are interleaved [re, im] doubles.  Row-major layouts:
 *   x [Bz,T,H,P]  dt [Bz,T,H]  A [H]  B, C [Bz,T,H,N]  D [H]
 *   y [Bz,T,H,P]  h0, h_final [Bz,H,N,P]
 */
#include <complex.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef double complex cplx;

static double softplus(double v) {
    /* log(1 + e^v), written so that neither branch overflows. */
    return fmax(v, 0.0) + log1p(exp(-fabs(v)));
}

static cplx ld(const double* p, int64_t i) { return p[2 * i] + I * p[2 * i + 1]; }
static void st(double* p, int64_t i, cplx v) {
    p[2 * i] = creal(v);
    p[2 * i + 1] = cimag(v);
}

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sequential recurrence over T tokens for every (batch, head).
 * h0 may be NULL (zero initial state); h_final may be NULL. */
void oracle_cssd_naive(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P,
                       const double* x, const double* dt, const double* A,
                       const double* B, const double* C, const double* D,
                       const double* h0, double* y, double* h_final) {
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int64_t b = 0; b < Bz; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            cplx* s = (cplx*)calloc((size_t)(N * P), sizeof(cplx));
            if (h0)
                for (int64_t i = 0; i < N * P; ++i) s[i] = ld(h0, (b * H + h) * N * P + i);
            const cplx Ah = ld(A, h);
            for (int64_t t = 0; t < T; ++t) {
                const int64_t bth = (b * T + t) * H + h;
                const cplx a = cexp(softplus(dt[bth]) * Ah);
                for (int64_t n = 0; n < N; ++n) {
                    const cplx bn = ld(B, bth * N + n);
                    for (int64_t p = 0; p < P; ++p)
                        s[n * P + p] = a * s[n * P + p] + bn * ld(x, bth * P + p);
                }
                for (int64_t p = 0; p < P; ++p) {
                    cplx acc = 0;
                    for (int64_t n = 0; n < N; ++n) acc += ld(C, bth * N + n) * s[n * P + p];
                    st(y, bth * P + p, acc + D[h] * ld(x, bth * P + p));
                }
            }
            if (h_final)
                for (int64_t i = 0; i < N * P; ++i) st(h_final, (b * H + h) * N * P + i, s[i]);
            free(s);
        }
    }
}

/* One token of the same recurrence on a given state: h <- a h + B x^T, then
 * y = C^T h + D x.  h [Bz,H,N,P] in/out; x [Bz,H,P]; dt [Bz,H]; B, C [Bz,H,N]. */
void oracle_cssd_step(int64_t Bz, int64_t H, int64_t N, int64_t P, double* hstate,
                      const double* x, const double* dt, const double* A,
                      const double* B, const double* C, const double* D, double* y) {
#pragma omp parallel for collapse(2)
    for (int64_t b = 0; b < Bz; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            const int64_t bh = b * H + h;
            const cplx a = cexp(softplus(dt[bh]) * ld(A, h));
            for (int64_t n = 0; n < N; ++n)
                for (int64_t p = 0; p < P; ++p) {
                    const int64_t i = bh * N * P + n * P + p;
                    st(hstate, i, a * ld(hstate, i) + ld(B, bh * N + n) * ld(x, bh * P + p));
                }
            for (int64_t p = 0; p < P; ++p) {
                cplx acc = 0;
                for (int64_t n = 0; n < N; ++n)
                    acc += ld(C, bh * N + n) * ld(hstate, bh * N * P + n * P + p);
                st(y, bh * P + p, acc + D[h] * ld(x, bh * P + p));
            }
        }
    }
}

/* The chunkwise decomposition with chunk length Cz, zero initial state.
 * Used to pin the decomposition and its bookkeeping against the sequential
 * recurrence; it is not the definition the CUDA path is checked against. */
void oracle_cssd_chunked(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int64_t Cz,
                         const double* x, const double* dt, const double* A,
                         const double* B, const double* C, const double* D,
                         double* y, double* h_final) {
    /* Step 1: pad to a whole number of chunks. */
    const int64_t pad = (Cz - (T % Cz)) % Cz;
    const int64_t nch = (T + pad) / Cz;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int64_t b = 0; b < Bz; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            const cplx Ah = ld(A, h);
            cplx* Xc = (cplx*)calloc((size_t)(Cz * P), sizeof(cplx));
            cplx* Bc = (cplx*)calloc((size_t)(Cz * N), sizeof(cplx));
            cplx* Cc = (cplx*)calloc((size_t)(Cz * N), sizeof(cplx));
            cplx* Acs = (cplx*)calloc((size_t)Cz, sizeof(cplx));
            cplx* G = (cplx*)calloc((size_t)(Cz * Cz), sizeof(cplx));
            cplx* S = (cplx*)calloc((size_t)(nch * N * P), sizeof(cplx)); /* S_c per chunk */
            cplx* ct = (cplx*)calloc((size_t)nch, sizeof(cplx));           /* chunk totals */
            cplx* Hin = (cplx*)calloc((size_t)(N * P), sizeof(cplx));
            for (int64_t c = 0; c < nch; ++c) {
                /* Gather chunk c; padded positions are zero with zero log-decay. */
                cplx run = 0;
                for (int64_t l = 0; l < Cz; ++l) {
                    const int64_t t = c * Cz + l;
                    const int real_tok = t < T;
                    const int64_t bth = (b * T + (real_tok ? t : 0)) * H + h;
                    for (int64_t p = 0; p < P; ++p) Xc[l * P + p] = real_tok ? ld(x, bth * P + p) : 0;
                    for (int64_t n = 0; n < N; ++n) {
                        Bc[l * N + n] = real_tok ? ld(B, bth * N + n) : 0;
                        Cc[l * N + n] = real_tok ? ld(C, bth * N + n) : 0;
                    }
                    /* Step 2: A_log = softplus(dt) A and its inclusive cumsum. */
                    run += real_tok ? softplus(dt[bth]) * Ah : 0;
                    Acs[l] = run;
                }
                ct[c] = Acs[Cz - 1];
                /* Step 5a: S_c[n,p] = sum_l exp(Acs[C-1] - Acs[l]) B[l,n] X[l,p]. */
                for (int64_t l = 0; l < Cz; ++l) {
                    const cplx ds = cexp(Acs[Cz - 1] - Acs[l]);
                    for (int64_t n = 0; n < N; ++n)
                        for (int64_t p = 0; p < P; ++p)
                            S[(c * N + n) * P + p] += ds * Bc[l * N + n] * Xc[l * P + p];
                }
                /* Step 5b: carry-in state of chunk c from the theorem,
                 * H_c = sum_{c'<c} exp(CD[c-1] - CD[c']) S_c', CD the inclusive
                 * cumsum of chunk totals. */
                memset(Hin, 0, (size_t)(N * P) * sizeof(cplx));
                for (int64_t cp = 0; cp < c; ++cp) {
                    cplx seg = 0; /* CD[c-1] - CD[c'] = sum_{c'' = c'+1}^{c-1} ct[c''] */
                    for (int64_t k = cp + 1; k <= c - 1; ++k) seg += ct[k];
                    const cplx dec = cexp(seg);
                    for (int64_t i = 0; i < N * P; ++i) Hin[i] += dec * S[cp * N * P + i];
                }
                /* Steps 3-4: G = C B^T, L[l,s] = exp(Acs[l] - Acs[s]) 1[l >= s]. */
                for (int64_t l = 0; l < Cz; ++l)
                    for (int64_t s = 0; s < Cz; ++s) {
                        cplx g = 0;
                        for (int64_t n = 0; n < N; ++n) g += Cc[l * N + n] * Bc[s * N + n];
                        G[l * Cz + s] = (l >= s) ? g * cexp(Acs[l] - Acs[s]) : 0;
                    }
                for (int64_t l = 0; l < Cz; ++l) {
                    const int64_t t = c * Cz + l;
                    if (t >= T) continue; /* slice the padding away */
                    const int64_t bth = (b * T + t) * H + h;
                    const cplx ein = cexp(Acs[l]);
                    for (int64_t p = 0; p < P; ++p) {
                        cplx yd = 0, yo = 0;
                        for (int64_t s = 0; s <= l; ++s) yd += G[l * Cz + s] * Xc[s * P + p];
                        for (int64_t n = 0; n < N; ++n) yo += Cc[l * N + n] * Hin[n * P + p];
                        st(y, bth * P + p, yd + ein * yo + D[h] * Xc[l * P + p]);
                    }
                }
            }
            if (h_final) {
                /* State after the last chunk: the theorem's sum one chunk on. */
                memset(Hin, 0, (size_t)(N * P) * sizeof(cplx));
                for (int64_t cp = 0; cp < nch; ++cp) {
                    cplx seg = 0;
                    for (int64_t k = cp + 1; k <= nch - 1; ++k) seg += ct[k];
                    const cplx dec = cexp(seg);
                    for (int64_t i = 0; i < N * P; ++i) Hin[i] += dec * S[cp * N * P + i];
                }
                for (int64_t i = 0; i < N * P; ++i) st(h_final, (b * H + h) * N * P + i, Hin[i]);
            }
            free(Xc); free(Bc); free(Cc); free(Acs); free(G); free(S); free(ct); free(Hin);
        }
    }
}

/* Constant input held for n steps from h0, in closed form:
 *   a = exp(softplus(dt) A),  a^n = exp(n softplus(dt) A),
 *   h_n = a^n h0 + (1 - a^n) / (1 - a) B x^T,
 *   y_n = C^T h_n + D x,      y_inf = (C^T B) / (1 - a) x + D x.
 * Shapes as oracle_cssd_step; h_n, y_n, y_inf are outputs (y_inf may be NULL).
 * Requires a != 1 (Re A != 0 or Im A not a multiple of 2 pi / softplus(dt)). */
void oracle_geom_closed_form(int64_t Bz, int64_t H, int64_t N, int64_t P, int64_t nsteps,
                             const double* h0, const double* x, const double* dt,
                             const double* A, const double* B, const double* C,
                             const double* D, double* h_n, double* y_n, double* y_inf) {
#pragma omp parallel for collapse(2)
    for (int64_t b = 0; b < Bz; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            const int64_t bh = b * H + h;
            const cplx alog = softplus(dt[bh]) * ld(A, h);
            const cplx a = cexp(alog);
            const cplx an = cexp((double)nsteps * alog);
            const cplx geo = (1.0 - an) / (1.0 - a);
            for (int64_t n = 0; n < N; ++n)
                for (int64_t p = 0; p < P; ++p) {
                    const int64_t i = bh * N * P + n * P + p;
                    st(h_n, i, an * ld(h0, i) + geo * ld(B, bh * N + n) * ld(x, bh * P + p));
                }
            cplx cb = 0;
            for (int64_t n = 0; n < N; ++n) cb += ld(C, bh * N + n) * ld(B, bh * N + n);
            for (int64_t p = 0; p < P; ++p) {
                cplx acc = 0;
                for (int64_t n = 0; n < N; ++n) acc += ld(C, bh * N + n) * ld(h_n, bh * N * P + n * P + p);
                const cplx xp = ld(x, bh * P + p);
                st(y_n, bh * P + p, acc + D[h] * xp);
                if (y_inf) st(y_inf, bh * P + p, cb / (1.0 - a) * xp + D[h] * xp);
            }
        }
    }
}
