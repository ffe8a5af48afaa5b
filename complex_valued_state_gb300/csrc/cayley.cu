// Per-coordinate Cayley-phase recurrence ("Complex Phase-State Dynamics Reduce
// the Optimization Steps of Sequence Models", section 5.2 equations (2)-(3),
// section 5.5 readout, Appendix A Algorithms 1-2).
//
// Every (batch, head, coordinate) is an independent scalar complex
// recurrence,
//     a_t = sigmoid(u_t) (1 + i phi_t) / (1 - i phi_t),
//     psi_t = a_t psi_{t-1} + b_t,      y_t = conj(C_t) psi_t,
// so the kernel runs one thread per coordinate along the sequence: there is
// nothing to contract, and the work is streaming 32 bytes per coordinate and
// token (phi, u, b, C in; y out).  Consecutive threads are consecutive
// coordinates of one token, so each warp's accesses are contiguous; the loads
// run a group of PF tokens ahead of the arithmetic (registers) to keep enough
// bytes in flight for HBM.
//
// Two evaluations:
//   - log_clamp = -inf: the recurrence itself, step by step (exact up to fp32
//     rounding; no reciprocal of a cumulative decay is ever formed).
//   - finite log_clamp (the paper uses -30): Algorithm 2, the chunked polar
//     scan, reproduced including its clamp.  Within a chunk,
//         l_m = clamp(sum_{r<=m} log|a_r|, log_clamp, 0),  Lambda_m = prod_{r<=m} lambda_r,
//         psi_m = e^{l_m} Lambda_m (x0 + sum_{r<=m} e^{-l_r} conj(Lambda_r) b_r),
//     and the chunk's last state is x0 of the next.  The cumulative phase is
//     kept as the running product of the unit Cayley factors rather than as
//     the sum of their angles 2 arctan(phi) followed by polar(): the two are
//     equal up to rounding, and the product needs no arctan or sincos.
//     log|a| = log sigmoid(u) = -softplus(-u) = -(max(-u, 0) + log(1 + e^{-|u|})).

#include "cssd_common.cuh"
#include "cssd_internal.h"

namespace cssd {
namespace {

constexpr int kThreads = 64;  // small blocks spread the coordinates evenly over the SMs
constexpr int PF = 8;  // tokens per load group

template <bool CLAMPED>
__global__ void __launch_bounds__(kThreads)
    cayley_scan_kernel(const float* __restrict__ phi, const float* __restrict__ u, const float2* __restrict__ b,
                       const float2* __restrict__ C, const float2* __restrict__ psi0, float2* __restrict__ y,
                       float2* __restrict__ psi_final, int T, int HN, long long BHN, int chunk, float lo) {
    const long long g = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (g >= BHN) return;
    const long long bb = g / HN;
    const int hk = (int)(g - bb * HN);
    const size_t base = (size_t)bb * T * HN + hk;  // element of token 0; tokens are HN apart

    float2 psi = psi0 ? psi0[g] : make_float2(0.f, 0.f);
    // Algorithm 2 state: chunk seed, running sum, cumulative phase and log-gate
    float2 x0 = psi, acc = make_float2(0.f, 0.f), lam_cum = make_float2(1.f, 0.f);
    float lsum = 0.f;
    int r = 0;

    float pn[PF], un[PF];
    float2 bn[PF], cn[PF];
    auto load = [&](int t0) {
#pragma unroll
        for (int j = 0; j < PF; ++j) {
            const int t = t0 + j;
            if (t < T) {
                const size_t i = base + (size_t)t * HN;
                pn[j] = __ldcs(phi + i);
                un[j] = __ldcs(u + i);
                bn[j] = __ldcs(b + i);
                cn[j] = __ldcs(C + i);
            }
        }
    };
    load(0);
    for (int t0 = 0; t0 < T; t0 += PF) {
        float pc[PF], uc[PF];
        float2 bc[PF], cc[PF];
#pragma unroll
        for (int j = 0; j < PF; ++j) {
            pc[j] = pn[j];
            uc[j] = un[j];
            bc[j] = bn[j];
            cc[j] = cn[j];
        }
        load(t0 + PF);  // the next group is in flight while this one is computed
#pragma unroll
        for (int j = 0; j < PF; ++j) {
            if (t0 + j >= T) break;
            // Algorithm 1: lambda = (1 + i phi) / (1 - i phi) = ((1 - phi^2) + 2 i phi) / (1 + phi^2)
            const float p = pc[j], p2 = p * p;
            const float inv = 1.f / (1.f + p2);
            const float2 lam = make_float2((1.f - p2) * inv, 2.f * p * inv);
            const float e = __expf(-fabsf(uc[j]));  // e^{-|u|}
            if constexpr (CLAMPED) {
                // + log sigmoid(u); log(1 + e) by the hardware logarithm: its absolute
                // error (~4e-7) is far below what a chunk's sum tolerates, and the
                // accurate log1pf cost 6 % of this kernel's time
                lsum -= fmaxf(-uc[j], 0.f) + __logf(1.f + e);
                lam_cum = cmul(lam_cum, lam);
                const float l = fminf(fmaxf(lsum, lo), 0.f);
                const float ep = __expf(l), en = __expf(-l);
                const float2 w = make_float2(en * lam_cum.x, -en * lam_cum.y);  // e^{-l} conj(Lambda)
                acc = cfma(w, bc[j], acc);
                psi = cscale(ep, cmul(lam_cum, cadd(x0, acc)));
                if (++r == chunk) {
                    r = 0;
                    x0 = psi;
                    acc = make_float2(0.f, 0.f);
                    lam_cum = make_float2(1.f, 0.f);
                    lsum = 0.f;
                }
            } else {
                const float alpha = uc[j] >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);  // sigmoid(u)
                psi = cfma(cscale(alpha, lam), psi, bc[j]);
            }
            // y = conj(C) psi
            const float2 cj = cc[j];
            __stcs(y + base + (size_t)(t0 + j) * HN,
                   make_float2(fmaf(cj.x, psi.x, cj.y * psi.y), fmaf(cj.x, psi.y, -cj.y * psi.x)));
        }
    }
    if (psi_final) psi_final[g] = psi;
}

}  // namespace

cudaError_t launch_cayley_scan(const CayleyArgs& a, cudaStream_t st) {
    const long long BHN = a.Bz * a.H * a.N;
    const unsigned grid = (unsigned)((BHN + kThreads - 1) / kThreads);
    const bool clamped = a.log_clamp > -INFINITY;
    if (clamped)
        cayley_scan_kernel<true><<<grid, kThreads, 0, st>>>(a.phi, a.u, a.b, a.C, a.psi0, a.y, a.psi_final, (int)a.T,
                                                            (int)(a.H * a.N), BHN, a.chunk, a.log_clamp);
    else
        cayley_scan_kernel<false><<<grid, kThreads, 0, st>>>(a.phi, a.u, a.b, a.C, a.psi0, a.y, a.psi_final,
                                                             (int)a.T, (int)(a.H * a.N), BHN, a.chunk, a.log_clamp);
    return cudaGetLastError();
}

}  // namespace cssd
