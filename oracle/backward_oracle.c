/*
 * CPU oracle for the gradients of the complex SSD forward — TEST
 * INFRASTRUCTURE ONLY (tests and the benchmark's CPU baseline call it; the
 * CUDA library never links or calls it).
 *
 * Forward (the oracle's sequential recurrence, "Complex-Valued State Spaces",
 * sections "Discretization" / "The discretization"; "SSD Theory" section 2):
 *     a_t = exp(z_t),  z_t = softplus(dt_t) A,  h_t = a_t h_{t-1} + B_t x_t^T,
 *     y_t = C_t^T h_t + D x_t,  h_{-1} = 0.
 * "The Chunkwise Complex SSD Algorithm" (its backward section) differentiates
 * this forward through the chunk quantities; here the gradients are taken of
 * the sequential recurrence directly, which is the definition.
 *
 * Convention: given the upstream gradient dy, the loss changes by
 *     dL = Re sum conj(g_w) dw
 * for every input w, i.e. a complex input's gradient is dL/dRe w + i dL/dIm w
 * and a real input's is dL/dw (the convention of complex automatic
 * differentiation in PyTorch).  With G_t the gradient with respect to h_t
 * (reverse-mode adjoint):
 *     G_t   = conj(a_{t+1}) G_{t+1} + conj(C_t) dy_t^T           (G_T = 0)
 *     gx_t  = sum_n conj(B_t[n]) G_t[n,:] + D dy_t
 *     gB_t  = sum_p G_t[:,p] conj(x_t[p])
 *     gC_t  = sum_p conj(h_t[:,p]) dy_t[p]
 *     ga_t  = sum_{n,p} G_t[n,p] conj(h_{t-1}[n,p]),   gz_t = conj(a_t) ga_t
 *     gdt_t = Re(conj(gz_t) A) sigmoid(dt_t),   gA = sum_{b,t} softplus(dt_t) gz_t
 *     gD    = sum_{b,t,p} Re(conj(dy_t[p]) x_t[p])
 * taken one token at a time, newest first, with every forward state stored
 * (memory (T + 1) N P complex per (batch, head): small cases only).
 *
 * Layouts as the forward oracle: x, dy, gx [Bz,T,H,P]; dt, gdt [Bz,T,H];
 * A, gA [H] (complex); B, C, gB, gC [Bz,T,H,N]; D, gD [H] (real).
 */
#include <complex.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef double complex cplx;

static cplx bld(const double* p, int64_t i) { return p[2 * i] + I * p[2 * i + 1]; }
static void bst(double* p, int64_t i, cplx v) {
    p[2 * i] = creal(v);
    p[2 * i + 1] = cimag(v);
}
static double bsoftplus(double v) { return fmax(v, 0.0) + log1p(exp(-fabs(v))); }
static double bsigmoid(double v) { return v >= 0 ? 1.0 / (1.0 + exp(-v)) : exp(v) / (1.0 + exp(v)); }

void oracle_cssd_backward(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, const double* x,
                          const double* dt, const double* A, const double* B, const double* C, const double* D,
                          const double* dy, double* gx, double* gdt, double* gA, double* gB, double* gC,
                          double* gD) {
    /* per-(batch, head) partial sums of gA and gD, reduced over the batch in order afterwards */
    cplx* gA_part = (cplx*)calloc((size_t)(Bz * H), sizeof(cplx));
    double* gD_part = (double*)calloc((size_t)(Bz * H), sizeof(double));
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < Bz; ++b)
        for (int64_t h = 0; h < H; ++h) {
            const cplx Ah = bld(A, h);
            const double Dh = D[h];
            const int64_t NP = N * P;
            cplx* hs = (cplx*)calloc((size_t)((T + 1) * NP), sizeof(cplx)); /* hs[t + 1] = h_t, hs[0] = h_{-1} = 0 */
            cplx* G = (cplx*)calloc((size_t)NP, sizeof(cplx));
            /* forward, every state kept */
            for (int64_t t = 0; t < T; ++t) {
                const int64_t bt = (b * T + t) * H + h;
                const cplx a = cexp(bsoftplus(dt[bt]) * Ah);
                const cplx* prev = hs + t * NP;
                cplx* cur = hs + (t + 1) * NP;
                for (int64_t n = 0; n < N; ++n)
                    for (int64_t p = 0; p < P; ++p)
                        cur[n * P + p] = a * prev[n * P + p] + bld(B, bt * N + n) * bld(x, bt * P + p);
            }
            /* reverse sweep */
            cplx gAh = 0;
            double gDh = 0;
            for (int64_t t = T - 1; t >= 0; --t) {
                const int64_t bt = (b * T + t) * H + h;
                const double sp = bsoftplus(dt[bt]);
                const cplx a = cexp(sp * Ah);
                const cplx* hcur = hs + (t + 1) * NP;
                const cplx* hprev = hs + t * NP;
                /* G <- G_t: add the readout of token t */
                for (int64_t n = 0; n < N; ++n)
                    for (int64_t p = 0; p < P; ++p) G[n * P + p] += conj(bld(C, bt * N + n)) * bld(dy, bt * P + p);
                for (int64_t p = 0; p < P; ++p) {
                    cplx s = Dh * bld(dy, bt * P + p);
                    for (int64_t n = 0; n < N; ++n) s += conj(bld(B, bt * N + n)) * G[n * P + p];
                    bst(gx, bt * P + p, s);
                    gDh += creal(conj(bld(dy, bt * P + p)) * bld(x, bt * P + p));
                }
                for (int64_t n = 0; n < N; ++n) {
                    cplx sb = 0, sc = 0;
                    for (int64_t p = 0; p < P; ++p) {
                        sb += G[n * P + p] * conj(bld(x, bt * P + p));
                        sc += conj(hcur[n * P + p]) * bld(dy, bt * P + p);
                    }
                    bst(gB, bt * N + n, sb);
                    bst(gC, bt * N + n, sc);
                }
                cplx ga = 0;
                for (int64_t i = 0; i < NP; ++i) ga += G[i] * conj(hprev[i]);
                const cplx gz = conj(a) * ga;
                gdt[bt] = creal(conj(gz) * Ah) * bsigmoid(dt[bt]);
                gAh += sp * gz;
                /* G_{t-1} = conj(a_t) G_t + (readout of t - 1, added next iteration) */
                for (int64_t i = 0; i < NP; ++i) G[i] *= conj(a);
            }
            gA_part[b * H + h] = gAh;
            gD_part[b * H + h] = gDh;
            free(hs);
            free(G);
        }
    for (int64_t h = 0; h < H; ++h) {
        cplx sa = 0;
        double sd = 0;
        for (int64_t b = 0; b < Bz; ++b) {
            sa += gA_part[b * H + h];
            sd += gD_part[b * H + h];
        }
        bst(gA, h, sa);
        gD[h] = sd;
    }
    free(gA_part);
    free(gD_part);
}
