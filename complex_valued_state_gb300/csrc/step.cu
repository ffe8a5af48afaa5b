// Decode step: one token of h <- a h + B x^T, y = C^T h + D x for every
// (batch, head).  Memory-bound: the whole N x P state of each head is read
// and written once per call, with 16-byte (two complex) coalesced accesses and
// streaming cache hints; the readout reduces over the N rows in registers and
// then across thread groups in shared memory.
//
// The recurrence is the sequential loop of "Complex-Valued State Spaces"
// (Mamba-3-Lite docs), "The discretization", one iteration of it.

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
template <int N, int P>
__global__ void __launch_bounds__(StepShape<N, P>::NT)
    step_kernel(float4* __restrict__ h, const float2* __restrict__ x, const float* __restrict__ dt,
                const float2* __restrict__ A, const float2* __restrict__ Bm, const float2* __restrict__ Cm,
                const float* __restrict__ D, float2* __restrict__ y, int H) {
    using S = StepShape<N, P>;
    __shared__ float2 sB[N], sC[N];
    __shared__ float2 part[S::G][P];
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
    const float2 x0 = make_float2(xv.x, xv.y), x1 = make_float2(xv.z, xv.w);
    const float2 a = cexpf2(alog_of(dt[bh], A[hd]));
    __syncthreads();

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

template <int N, int P>
cudaError_t launch_step_np(const StepArgs& a, cudaStream_t st) {
    const unsigned grid = (unsigned)(a.Bz * a.H);
    step_kernel<N, P><<<grid, StepShape<N, P>::NT, 0, st>>>(reinterpret_cast<float4*>(a.h), a.x, a.dt, a.A, a.B,
                                                           a.C, a.D, a.y, (int)a.H);
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
