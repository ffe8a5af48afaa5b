// Decode step: one token of h <- a h + B x^T, y = C^T h + D x for every
// (batch, head).  Memory-bound: the whole N x P state of each head is read
// and written once per call, with 16-byte (two complex) coalesced accesses and
// streaming cache hints; the readout reduces over the N rows in registers and
// then across thread groups in shared memory.
//
// The recurrence is the sequential loop of "Complex-Valued State Spaces"
// (Mamba-3-Lite docs), "The discretization", one iteration of it.
//
// Constant-input shortcuts ("Constant-input stepping shortcuts —
// step_n_approx / step_infinite", burn-mamba docs, module step_constant): when
// the same (x, dt, B, C) is fed n times, the n steps collapse to one geometric
// series in the per-step factor a = exp(z), z = softplus(dt) A,
//     h_n = a^n h_0 + g_n B x^T,   g_n = sum_{k<n} a^k = expm1(n z) / expm1(z),
// and as n -> infinity (|a| < 1) the readout tends to
//     y_inf = (C^T B) x / (1 - a) + D x,
// with no state at all.  The pages state the series for a block whose input
// also rotates from step to step; in this recurrence the rotation is part of
// the complex a, so the series is the plain scalar one above.  The same kernel
// runs it with per-head coefficients (a^n, g_n) in place of (a, 1), so n steps
// cost one step's memory traffic.

#include "cssd_common.cuh"
#include "cssd_internal.h"

namespace cssd {
namespace {

template <int N, int P>
struct StepShape {
    static constexpr int QP = P / 2;                                  // float4 per state row
    static constexpr int NT = (N * P / 2 < 256) ? (N * P / 2) : 256;  // threads per head
    static constexpr int G = NT / QP;                                 // row groups
    static constexpr int RPT = N / G;                                 // rows per thread
    static_assert(G * RPT == N && G * QP == NT, "step tiling");
};

// One CTA per (batch, head).  Thread tid owns the column pair q = tid % QP
// and the rows n = g + G * i (g = tid / QP), so that for each i a warp touches
// one contiguous 512-byte run of the state.
// Coefficients of n steps of a constant input: a^n = exp(n z) and
// g_n = sum_{k<n} exp(k z) = expm1(n z) / expm1(z), z = softplus(dt) A.
// softplus and the angle n Im z are taken in double, since n multiplies their
// rounding errors; the angle is reduced mod 2 pi (two-part 2 pi, one fma each)
// before any trigonometry.  The rest is fp32, with the complex expm1 in the
// cancellation-free form
//     expm1(u + iv) = (expm1(u) cos v - 2 sin^2(v / 2)) + i e^u sin v,
// so that g_n stays accurate when z is small (g_n -> n as z -> 0; exactly n
// when z = 0).  Only a few double operations: one thread per CTA runs this
// while the state loads are in flight.
__device__ void const_input_coeffs(float dtv, float2 Ah, long long n, float2& an, float2& gn) {
    const double v = (double)dtv;
    const double sp = fmax(v, 0.0) + log1p(exp(-fabs(v)));
    const double nzi = (double)n * (sp * (double)Ah.y);
    constexpr double kTwoPiHi = 6.283185307179586232, kTwoPiLo = 2.4492935982947064e-16;
    const double k = rint(nzi * 0.15915494309189533577);
    const float phi = (float)fma(-k, kTwoPiLo, fma(-k, kTwoPiHi, nzi));
    const float nr = (float)((double)n * (sp * (double)Ah.x));
    const float zr = (float)(sp * (double)Ah.x), zi = (float)(sp * (double)Ah.y);
    float sn, cn, sz, cz;
    sincosf(phi, &sn, &cn);
    sincosf(zi, &sz, &cz);
    const float en = expf(nr);
    an = make_float2(en * cn, en * sn);
    const float hn = sinf(0.5f * phi), hz = sinf(0.5f * zi);
    const float ur = expm1f(nr) * cn - 2.f * hn * hn, ui = en * sn;           // expm1(n z)
    const float dr = expm1f(zr) * cz - 2.f * hz * hz, di = expf(zr) * sz;     // expm1(z)
    const float den = dr * dr + di * di;
    if (den == 0.f) {
        gn = make_float2((float)n, 0.f);
        return;
    }
    gn = make_float2((ur * dr + ui * di) / den, (ui * dr - ur * di) / den);
}

// MULTI = false: one ordinary step.  MULTI = true: `nsteps` steps of the same
// input, as h <- a^n h + B (g_n x)^T.
template <int N, int P, bool MULTI>
__global__ void __launch_bounds__(StepShape<N, P>::NT)
    step_kernel(float4* __restrict__ h, const float2* __restrict__ x, const float* __restrict__ dt,
                const float2* __restrict__ A, const float2* __restrict__ Bm, const float2* __restrict__ Cm,
                const float* __restrict__ D, float2* __restrict__ y, int H, long long nsteps) {
    using S = StepShape<N, P>;
    __shared__ float2 sB[N], sC[N];
    __shared__ float2 part[S::G][P];
    __shared__ float2 s_coef[2];  // (a^n, g_n) when MULTI
    const int bh = blockIdx.x;
    const int hd = bh % H;
    const int tid = threadIdx.x;
    const int q = tid % S::QP, g = tid / S::QP;

    float4* hs = h + (size_t)bh * (N * P / 2);
    // Issue the state loads first: they are independent of everything below.
    float4 hv[S::RPT];
#pragma unroll
    for (int i = 0; i < S::RPT; ++i) hv[i] = __ldcs(hs + (g + S::G * i) * S::QP + q);

    for (int n = tid; n < N; n += S::NT) {
        sB[n] = Bm[(size_t)bh * N + n];
        sC[n] = Cm[(size_t)bh * N + n];
    }
    const float4 xv = reinterpret_cast<const float4*>(x + (size_t)bh * P)[q];
    float2 x0 = make_float2(xv.x, xv.y), x1 = make_float2(xv.z, xv.w);
    float2 a;
    if constexpr (MULTI) {
        if (tid == 0) const_input_coeffs(dt[bh], A[hd], nsteps, s_coef[0], s_coef[1]);
    } else {
        a = cexpf2(alog_of(dt[bh], A[hd]));
    }
    __syncthreads();
    if constexpr (MULTI) {
        a = s_coef[0];
        x0 = cmul(s_coef[1], x0);
        x1 = cmul(s_coef[1], x1);
    }

    float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
#pragma unroll
    for (int i = 0; i < S::RPT; ++i) {
        const int n = g + S::G * i;
        const float2 bn = sB[n], cn = sC[n];
        const float2 h0 = cfma(bn, x0, cmul(a, make_float2(hv[i].x, hv[i].y)));
        const float2 h1 = cfma(bn, x1, cmul(a, make_float2(hv[i].z, hv[i].w)));
        __stcs(hs + n * S::QP + q, make_float4(h0.x, h0.y, h1.x, h1.y));
        acc0 = cfma(cn, h0, acc0);
        acc1 = cfma(cn, h1, acc1);
    }
    part[g][2 * q] = acc0;
    part[g][2 * q + 1] = acc1;
    __syncthreads();
    for (int p = tid; p < P; p += S::NT) {
        float2 s = make_float2(0.f, 0.f);
#pragma unroll
        for (int gg = 0; gg < S::G; ++gg) s = cadd(s, part[gg][p]);
        const float2 xp = x[(size_t)bh * P + p];
        y[(size_t)bh * P + p] = cadd(s, cscale(D[hd], xp));
    }
}

// Output of a constant input held forever: one warp per (batch, head)
// reduces C^T B over the state rows, then y = (C^T B) / (1 - a) x + D x with
// 1 / (1 - a) = -1 / expm1(z) (fp32, cancellation-free form as above).
template <int N>
__global__ void __launch_bounds__(256)
    step_infinite_kernel(const float2* __restrict__ x, const float* __restrict__ dt, const float2* __restrict__ A,
                         const float2* __restrict__ Bm, const float2* __restrict__ Cm, const float* __restrict__ D,
                         float2* __restrict__ y, int H, int BH, int P) {
    const int bh = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (bh >= BH) return;
    const int hd = bh % H;
    float2 xs[2];  // P <= 64: at most two columns per lane, fetched first
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int pp = lane + 32 * k;
        xs[k] = pp < P ? x[(size_t)bh * P + pp] : make_float2(0.f, 0.f);
    }
    float2 cb = make_float2(0.f, 0.f);
#pragma unroll
    for (int n = lane; n < N; n += 32) cb = cfma(Cm[(size_t)bh * N + n], Bm[(size_t)bh * N + n], cb);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        cb.x += __shfl_xor_sync(0xffffffffu, cb.x, o);
        cb.y += __shfl_xor_sync(0xffffffffu, cb.y, o);
    }
    const float2 z = alog_of(dt[bh], A[hd]);
    float sz, cz;
    sincosf(z.y, &sz, &cz);
    const float sh = sinf(0.5f * z.y);
    const float er = expm1f(z.x) * cz - 2.f * sh * sh, ei = expf(z.x) * sz;  // expm1(z) = a - 1
    const float den = er * er + ei * ei;
    // r = C^T B / (1 - a) = -C^T B / expm1(z)
    const float2 r = make_float2(-(cb.x * er + cb.y * ei) / den, -(cb.y * er - cb.x * ei) / den);
    const float Dh = D[hd];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int pp = lane + 32 * k;
        if (pp < P) y[(size_t)bh * P + pp] = cfma(r, xs[k], cscale(Dh, xs[k]));
    }
}

template <int N, int P>
cudaError_t launch_step_np(const StepArgs& a, cudaStream_t st) {
    const unsigned grid = (unsigned)(a.Bz * a.H);
    if (a.nsteps < 0)
        step_kernel<N, P, false><<<grid, StepShape<N, P>::NT, 0, st>>>(
            reinterpret_cast<float4*>(a.h), a.x, a.dt, a.A, a.B, a.C, a.D, a.y, (int)a.H, 1);
    else
        step_kernel<N, P, true><<<grid, StepShape<N, P>::NT, 0, st>>>(
            reinterpret_cast<float4*>(a.h), a.x, a.dt, a.A, a.B, a.C, a.D, a.y, (int)a.H, (long long)a.nsteps);
    return cudaGetLastError();
}

template <int N>
cudaError_t launch_step_n(const StepArgs& a, cudaStream_t st) {
    switch (a.P) {
        case 16: return launch_step_np<N, 16>(a, st);
        case 32: return launch_step_np<N, 32>(a, st);
        case 64: return launch_step_np<N, 64>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_step_infinite(const StepArgs& a, cudaStream_t st) {
    const int BH = (int)(a.Bz * a.H);
    const unsigned grid = (unsigned)((BH + 7) / 8);
    switch (a.N) {
        case 16: step_infinite_kernel<16><<<grid, 256, 0, st>>>(a.x, a.dt, a.A, a.B, a.C, a.D, a.y, (int)a.H, BH, (int)a.P); break;
        case 32: step_infinite_kernel<32><<<grid, 256, 0, st>>>(a.x, a.dt, a.A, a.B, a.C, a.D, a.y, (int)a.H, BH, (int)a.P); break;
        case 64: step_infinite_kernel<64><<<grid, 256, 0, st>>>(a.x, a.dt, a.A, a.B, a.C, a.D, a.y, (int)a.H, BH, (int)a.P); break;
        case 128: step_infinite_kernel<128><<<grid, 256, 0, st>>>(a.x, a.dt, a.A, a.B, a.C, a.D, a.y, (int)a.H, BH, (int)a.P); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_step(const StepArgs& a, cudaStream_t st) {
    switch (a.N) {
        case 16: return launch_step_n<16>(a, st);
        case 32: return launch_step_n<32>(a, st);
        case 64: return launch_step_n<64>(a, st);
        case 128: return launch_step_n<128>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace cssd
