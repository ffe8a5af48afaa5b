// Gradients of the chunked forward with respect to every input.
//
// Forward (per batch row and head): a_t = exp(z_t), z_t = softplus(dt_t) A,
// h_t = a_t h_{t-1} + B_t x_t^T, y_t = C_t^T h_t + D x_t.  Given the upstream
// gradient dy, with the convention dL = Re sum conj(g_w) dw, the adjoint state
// G_t = dL/dh_t obeys G_t = conj(a_{t+1}) G_{t+1} + conj(C_t) dy_t^T, and
//     gx_t = sum_n conj(B_t[n]) G_t[n,:] + D dy_t
//     gB_t = sum_p G_t[:,p] conj(x_t[p])
//     gC_t = sum_p conj(h_t[:,p]) dy_t[p]
// Each of these is itself a run of the forward recurrence, so the library's
// own forward kernels compute it:
//   gx: time reversed, input dy, input coupling conj(C), readout conj(B),
//       rate conj(A) (conj(a) = exp(softplus(dt) conj(A))), the step of token
//       t + 1 at reversed position T - 1 - t, skip D;
//   gB: the same reversed run with the state transposed (input conj(C) of
//       width N, coupling dy of width P, readout conj(x)), no skip;
//   gC: the forward run with the state transposed (input B, coupling x,
//       readout conj(dy)), no skip; gC = conj(output).
// The step and rate gradients need G_t and h_{t-1} together; since y is linear
// in x, with r_t = sum_p (conj(dy_t[p]) y_t[p] - x_t[p] conj(gx_t[p])) and
// R_t = sum_{u >= t} r_u one has dL/dz_t = conj(R_t), so
//     gdt_t = Re(R_t A) sigmoid(dt_t),   gA = sum_{b,t} softplus(dt_t) conj(R_t),
// and gD = sum_{b,t,p} Re(conj(dy) x).  The total of r vanishes (R_0 = 0: the
// first step multiplies the zero initial state), so R_t = -sum_{u < t} r_u too.
// r_t is a small difference of two sums of P products, so y and gx, which it
// is formed from, are computed to about fp32 accuracy (with operands rounded
// to 11 significant bits the error reached 1e-2 of the largest gdt): by the
// split-precision tensor-core kernel where its shape applies, else by the
// fp32 CUDA-core chunk kernels.  gB and gC, read directly, take the plain
// tensor-core kernel where it applies.
// The derivation differentiates the sequential recurrence ("Complex-Valued
// State Spaces", "The discretization"; "SSD Theory" section 2), which the
// chunked form computes exactly up to rounding.

#include "cssd_common.cuh"
#include "cssd_internal.h"

namespace cssd {
namespace {

constexpr int EB = 256;  // threads per block of the element kernels

// dst[b, tau, :] = (conj?) src[b, T - 1 - tau, :], rows of `row` complex
// numbers; one block per output row (grid-stride over rows), so each block
// copies one contiguous row to another.
__global__ void reverse_rows_kernel(const float2* __restrict__ src, float2* __restrict__ dst, int64_t Bz, int64_t T,
                                    int64_t row, bool conj_) {
    for (int64_t o = blockIdx.x; o < Bz * T; o += gridDim.x) {
        const int64_t b = o / T, tau = o - b * T;
        const float2* s = src + (b * T + (T - 1 - tau)) * row;
        float2* d = dst + o * row;
        for (int64_t e = threadIdx.x; e < row; e += EB) {
            float2 v = s[e];
            if (conj_) v.y = -v.y;
            d[e] = v;
        }
    }
}

// dst = conj(src), n complex numbers.
__global__ void conj_kernel(const float2* __restrict__ src, float2* __restrict__ dst, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * EB + threadIdx.x; i < n; i += (int64_t)gridDim.x * EB) {
        const float2 v = src[i];
        dst[i] = make_float2(v.x, -v.y);
    }
}

// Step of the reversed runs: position tau takes the step of token T - tau
// (the decay between tokens T - 1 - tau and T - tau); position 0 has no
// predecessor and takes 0.  Also conj(A) and a zero skip per head.
__global__ void reverse_steps_kernel(const float* __restrict__ dt, float* __restrict__ dts, int64_t Bz, int64_t T,
                                     int64_t H, const float2* __restrict__ A, float2* __restrict__ Ac,
                                     float* __restrict__ zero) {
    const int64_t total = Bz * T * H;
    for (int64_t i = (int64_t)blockIdx.x * EB + threadIdx.x; i < total; i += (int64_t)gridDim.x * EB) {
        const int64_t b = i / (T * H), r = i - b * T * H;
        const int64_t tau = r / H, h = r - tau * H;
        dts[i] = tau == 0 ? 0.f : dt[(b * T + (T - tau)) * H + h];
        if (i < H) {
            Ac[i] = make_float2(A[i].x, -A[i].y);
            zero[i] = 0.f;
        }
    }
}

// One warp per token-head: r = sum_p (conj(dy) y - x conj(gx)) and
// d = sum_p Re(conj(dy) x).
__global__ void token_terms_kernel(const float2* __restrict__ x, const float2* __restrict__ y,
                                   const float2* __restrict__ dy, const float2* __restrict__ gx, float2* __restrict__ r,
                                   float* __restrict__ d, int64_t units, int P) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (EB / 32);
    for (int64_t u = ((int64_t)blockIdx.x * EB + threadIdx.x) >> 5; u < units; u += warps) {
        float rr = 0.f, ri = 0.f, dd = 0.f;
        for (int p = lane; p < P; p += 32) {
            const int64_t i = u * P + p;
            const float2 a = dy[i], yy = y[i], xx = x[i], g = gx[i];
            // conj(dy) y - x conj(g)
            rr += a.x * yy.x + a.y * yy.y - (xx.x * g.x + xx.y * g.y);
            ri += a.x * yy.y - a.y * yy.x - (xx.y * g.x - xx.x * g.y);
            dd += a.x * xx.x + a.y * xx.y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            rr += __shfl_xor_sync(0xffffffffu, rr, o);
            ri += __shfl_xor_sync(0xffffffffu, ri, o);
            dd += __shfl_xor_sync(0xffffffffu, dd, o);
        }
        if (lane == 0) {
            r[u] = make_float2(rr, ri);
            d[u] = dd;
        }
    }
}

// Inclusive scan of one double2 per thread across the block (EB threads),
// in thread order; scratch holds EB / 32 double2.
__device__ __forceinline__ double2 block_scan(double2 v, double2* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double ux = __shfl_up_sync(0xffffffffu, v.x, o), uy = __shfl_up_sync(0xffffffffu, v.y, o);
        if (lane >= o) {
            v.x += ux;
            v.y += uy;
        }
    }
    if (lane == 31) scratch[warp] = v;
    __syncthreads();
    double2 off = make_double2(0.0, 0.0);
    for (int w = 0; w < warp; ++w) {
        off.x += scratch[w].x;
        off.y += scratch[w].y;
    }
    __syncthreads();
    return make_double2(v.x + off.x, v.y + off.y);
}

// One CTA per (batch, head): R_t, gdt_t = Re(R_t A) sigmoid(dt_t), and the
// (batch, head) sums of softplus(dt_t) conj(R_t) and of d_t.  Since the total
// of r vanishes, R_t = sum_{u >= t} r_u = -sum_{u < t} r_u; the shorter side is
// summed (in double), so R_0 = 0 exactly and rounding grows with
// min(t, T - t) rather than with T.  Thread k holds the tokens
// [k L, (k + 1) L) of the sequence.
constexpr int SCAN_L = 16;  // tokens per thread and pass
__global__ void __launch_bounds__(EB) reverse_scan_kernel(const float2* __restrict__ r, const float* __restrict__ d,
                                                          const float* __restrict__ dt, const float2* __restrict__ A,
                                                          float* __restrict__ gdt, double2* __restrict__ gA_part,
                                                          double* __restrict__ gD_part, int64_t T, int64_t H) {
    __shared__ double2 scratch[EB / 32];
    __shared__ double2 red[EB / 32];
    __shared__ double redd[EB / 32];
    const int64_t bh = blockIdx.x;
    const int64_t b = bh / H, h = bh - b * H;
    const float2 Ah = A[h];
    const int64_t half = (T + 1) / 2;  // token 0 is always on the prefix side: R_0 = 0
    const int tid = threadIdx.x;
    double ga_r = 0.0, ga_i = 0.0, gd = 0.0;
    auto emit = [&](int64_t t, double Rr, double Ri) {
        const int64_t i = (b * T + t) * H + h;
        const float v = dt[i];
        const float sig = v >= 0.f ? 1.f / (1.f + __expf(-v)) : __expf(v) / (1.f + __expf(v));
        gdt[i] = (float)(Rr * Ah.x - Ri * Ah.y) * sig;
        const double sp = softplusf(v);
        ga_r += sp * Rr;
        ga_i -= sp * Ri;
        gd += d[i];
    };
    // Prefix side, tokens [0, half) in passes of EB * SCAN_L: R_t = -(r_0 + ... + r_{t-1}).
    double2 carry = make_double2(0.0, 0.0);
    for (int64_t base = 0; base < half; base += (int64_t)EB * SCAN_L) {
        const int64_t t0 = base + (int64_t)tid * SCAN_L;
        double2 loc[SCAN_L];
        double2 sum = make_double2(0.0, 0.0);
#pragma unroll
        for (int k = 0; k < SCAN_L; ++k) {
            const int64_t t = t0 + k;
            const float2 v = t < half ? r[(b * T + t) * H + h] : make_float2(0.f, 0.f);
            loc[k] = sum;  // exclusive within the thread
            sum.x += v.x;
            sum.y += v.y;
        }
        const double2 incl = block_scan(sum, scratch);
        const double2 excl = make_double2(carry.x + incl.x - sum.x, carry.y + incl.y - sum.y);
#pragma unroll
        for (int k = 0; k < SCAN_L; ++k) {
            const int64_t t = t0 + k;
            if (t < half) emit(t, -(excl.x + loc[k].x), -(excl.y + loc[k].y));
        }
        if (tid == EB - 1) scratch[0] = incl;  // the pass total
        __syncthreads();
        carry.x += scratch[0].x;
        carry.y += scratch[0].y;
        __syncthreads();
    }
    // Suffix side, tokens [half, T) newest first: R_t = r_t + ... + r_{T-1}.
    carry = make_double2(0.0, 0.0);
    for (int64_t base = T - 1; base >= half; base -= (int64_t)EB * SCAN_L) {
        const int64_t t0 = base - (int64_t)tid * SCAN_L;  // this thread's newest token
        double2 loc[SCAN_L];
        double2 sum = make_double2(0.0, 0.0);
#pragma unroll
        for (int k = 0; k < SCAN_L; ++k) {
            const int64_t t = t0 - k;
            const float2 v = t >= half ? r[(b * T + t) * H + h] : make_float2(0.f, 0.f);
            sum.x += v.x;
            sum.y += v.y;
            loc[k] = sum;  // inclusive within the thread
        }
        const double2 incl = block_scan(sum, scratch);
        const double2 excl = make_double2(carry.x + incl.x - sum.x, carry.y + incl.y - sum.y);
#pragma unroll
        for (int k = 0; k < SCAN_L; ++k) {
            const int64_t t = t0 - k;
            if (t >= half) emit(t, excl.x + loc[k].x, excl.y + loc[k].y);
        }
        if (tid == EB - 1) scratch[0] = incl;
        __syncthreads();
        carry.x += scratch[0].x;
        carry.y += scratch[0].y;
        __syncthreads();
    }
    // Block sums of the rate and skip gradients.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ga_r += __shfl_xor_sync(0xffffffffu, ga_r, o);
        ga_i += __shfl_xor_sync(0xffffffffu, ga_i, o);
        gd += __shfl_xor_sync(0xffffffffu, gd, o);
    }
    if ((tid & 31) == 0) {
        red[tid >> 5] = make_double2(ga_r, ga_i);
        redd[tid >> 5] = gd;
    }
    __syncthreads();
    if (tid == 0) {
        double2 s2 = make_double2(0.0, 0.0);
        double sd = 0.0;
        for (int w = 0; w < EB / 32; ++w) {
            s2.x += red[w].x;
            s2.y += red[w].y;
            sd += redd[w];
        }
        gA_part[bh] = s2;
        gD_part[bh] = sd;
    }
}

// R at the chunk boundaries, from the states the two split-precision runs
// published (T a multiple of 64): at t = 64 c, 0 < c < nc,
//     R_t = a_t sum_{n,p} conj(G_t[n,p]) h_{t-1}[n,p]
// (the product of the adjoint state after token t and the forward state before
// it), an inner product of the forward run's state handed to chunk c (slot c)
// and the reversed run's state handed on after original token t (slot nc - c),
// each rotated back from its run's frame.  One block per (boundary, batch,
// head); written to Rb[bh * (nc + 1) + c].
__global__ void __launch_bounds__(EB) boundary_kernel(const float* __restrict__ Hd, const float2* __restrict__ Hrot,
                                                      const float* __restrict__ Gd, const float2* __restrict__ Grot,
                                                      const float* __restrict__ dt, const float2* __restrict__ A,
                                                      double2* __restrict__ Rb, int64_t T, int64_t H, int nc) {
    __shared__ double2 red[EB / 32];
    constexpr int S = 64 * 64;  // state elements (dstate = headdim = 64)
    const int64_t q = blockIdx.x;
    const int c = (int)(q % (nc - 1)) + 1;
    const int64_t bh = q / (nc - 1), b = bh / H, h = bh - b * H;
    const float* hs = Hd + ((size_t)bh * (nc + 1) + c) * (2 * S);
    const float* gs = Gd + ((size_t)bh * (nc + 1) + (nc - c)) * (2 * S);
    // element i of both dumps is the same (n, p): the sum does not depend on
    // their layout.
    // per-thread partial sums of 16 products in fp32 (the states themselves
    // carry ~22 significant bits; FP64 arithmetic is slow on this part), the
    // block reduction in double
    float fr = 0.f, fi = 0.f;
    for (int i = threadIdx.x; i < S; i += EB) {
        const float hr = hs[i], hi = hs[S + i], gr = gs[i], gi = gs[S + i];
        fr = fmaf(gr, hr, fmaf(gi, hi, fr));  // conj(g) h
        fi = fmaf(gr, hi, fmaf(-gi, hr, fi));
    }
    double kr = fr, ki = fi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        kr += __shfl_xor_sync(0xffffffffu, kr, o);
        ki += __shfl_xor_sync(0xffffffffu, ki, o);
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_double2(kr, ki);
    __syncthreads();
    if (threadIdx.x == 0) {
        kr = ki = 0.0;
        for (int w = 0; w < EB / 32; ++w) {
            kr += red[w].x;
            ki += red[w].y;
        }
        // frames: h = e^{i thH} h~, G = e^{i thG} G~, so conj(G) h = e^{i (thH - thG)} conj(G~) h~
        const float2 rh = Hrot[(size_t)bh * (nc + 1) + c], rg = Grot[(size_t)bh * (nc + 1) + (nc - c)];
        const double er = (double)rh.x * rg.x + (double)rh.y * rg.y, ei = (double)rh.y * rg.x - (double)rh.x * rg.y;
        const double pr = er * kr - ei * ki, pi = er * ki + ei * kr;
        // a_t = exp(softplus(dt_t) A)
        const double sp = softplusf(dt[((size_t)b * T + 64 * (size_t)c) * H + h]);
        const double m = exp(sp * (double)A[h].x), ang = sp * (double)A[h].y;
        const double ar = m * cos(ang), ai = m * sin(ang);
        Rb[(size_t)bh * (nc + 1) + c] = make_double2(ar * pr - ai * pi, ar * pi + ai * pr);
    }
}

// The step and rate gradients from chunk-local sums (T a multiple of 64): for
// t in chunk c, R_t = r_t + ... + r_{64 c + 63} + R_{64 (c + 1)} with the
// boundary value from boundary_kernel (0 after the last chunk), so no sum runs
// across a chunk.  One CTA per (batch, head), four chunks per pass of 256
// threads (one token each); outputs as reverse_scan_kernel.
__global__ void __launch_bounds__(EB) chunk_scan_kernel(const float2* __restrict__ r, const float* __restrict__ d,
                                                        const float* __restrict__ dt, const float2* __restrict__ A,
                                                        const double2* __restrict__ Rb, float* __restrict__ gdt,
                                                        double2* __restrict__ gA_part, double* __restrict__ gD_part,
                                                        int64_t T, int64_t H, int nc) {
    __shared__ double2 tot[EB / 32];
    __shared__ double2 red[EB / 32];
    __shared__ double redd[EB / 32];
    const int64_t bh = blockIdx.x;
    const int64_t b = bh / H, h = bh - b * H;
    const float2 Ah = A[h];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    double ga_r = 0.0, ga_i = 0.0, gd = 0.0;
    for (int c0 = 0; c0 < nc; c0 += EB / 64) {
        const int c = c0 + (tid >> 6);
        const int64_t t = 64 * (int64_t)c + (tid & 63);
        const bool valid = c < nc && t < T;
        const int64_t i = (b * T + t) * H + h;
        double2 v = make_double2(0.0, 0.0);
        if (valid) {
            const float2 rv = r[i];
            v = make_double2(rv.x, rv.y);
        }
        // suffix sums within the warp (32 tokens), then the upper warp's total
        // added to the lower warp of the same chunk
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double ux = __shfl_down_sync(0xffffffffu, v.x, o), uy = __shfl_down_sync(0xffffffffu, v.y, o);
            if (lane + o < 32) {
                v.x += ux;
                v.y += uy;
            }
        }
        if (lane == 0) tot[warp] = v;
        __syncthreads();
        if ((warp & 1) == 0) {
            v.x += tot[warp + 1].x;
            v.y += tot[warp + 1].y;
        }
        __syncthreads();
        if (valid) {
            const double2 Rn = (c + 1 < nc) ? Rb[(size_t)bh * (nc + 1) + c + 1] : make_double2(0.0, 0.0);
            const double Rr = v.x + Rn.x, Ri = v.y + Rn.y;
            const float dv = dt[i];
            const float sig = dv >= 0.f ? 1.f / (1.f + __expf(-dv)) : __expf(dv) / (1.f + __expf(dv));
            gdt[i] = (float)(Rr * Ah.x - Ri * Ah.y) * sig;
            const double sp = softplusf(dv);
            ga_r += sp * Rr;
            ga_i -= sp * Ri;
            gd += d[i];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ga_r += __shfl_xor_sync(0xffffffffu, ga_r, o);
        ga_i += __shfl_xor_sync(0xffffffffu, ga_i, o);
        gd += __shfl_xor_sync(0xffffffffu, gd, o);
    }
    if (lane == 0) {
        red[warp] = make_double2(ga_r, ga_i);
        redd[warp] = gd;
    }
    __syncthreads();
    if (tid == 0) {
        double2 s2 = make_double2(0.0, 0.0);
        double sd = 0.0;
        for (int w = 0; w < EB / 32; ++w) {
            s2.x += red[w].x;
            s2.y += red[w].y;
            sd += redd[w];
        }
        gA_part[bh] = s2;
        gD_part[bh] = sd;
    }
}

// gA[h], gD[h]: the batch rows' partial sums, added in order (deterministic).
__global__ void head_sums_kernel(const double2* __restrict__ gA_part, const double* __restrict__ gD_part,
                                 float2* __restrict__ gA, float* __restrict__ gD, int64_t Bz, int64_t H) {
    const int64_t h = (int64_t)blockIdx.x * EB + threadIdx.x;
    if (h >= H) return;
    double ar = 0.0, ai = 0.0, dd = 0.0;
    for (int64_t b = 0; b < Bz; ++b) {
        ar += gA_part[b * H + h].x;
        ai += gA_part[b * H + h].y;
        dd += gD_part[b * H + h];
    }
    gA[h] = make_float2((float)ar, (float)ai);
    gD[h] = (float)dd;
}

unsigned grid_for(int64_t n) {
    const int64_t blocks = (n + EB - 1) / EB;
    return (unsigned)(blocks < 65535 * 8 ? (blocks < 1 ? 1 : blocks) : 65535 * 8);
}

unsigned grid_rows(int64_t rows) { return (unsigned)(rows < 65535 * 8 ? rows : 65535 * 8); }

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// The forward to about fp32 accuracy: the split-precision tensor-core kernel
// (each operand as two half parts, three products per product) where it is
// built (headdim 64, dstate 64), else the fp32 CUDA-core chunk kernels
// (dstate 128 among them).
bool precise_on_tc(int64_t N, int64_t P, int chunk) {
    return tc_forward_supported(N, P, chunk) && tc_full_shape(N, P) && N == 64;
}
size_t precise_forward_workspace_bytes(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk) {
    if (precise_on_tc(N, P, chunk)) return tc_forward_workspace_bytes(Bz, T, H, N);
    return seq_forward_workspace_bytes(Bz, T, H, N, P, chunk);
}
cudaError_t launch_precise_forward(FwdArgs f, void* ws, cudaStream_t st) {
    if (!precise_on_tc(f.N, f.P, f.chunk)) return launch_seq_forward(f, ws, st);
    f.split_operands = true;
    return launch_tc_forward(f, ws, st);
}

// The adjoint runs take the tensor-core kernel's index and sign modes (time
// reversal, conjugated operands and output, no skip) when both the state and
// its transpose are tensor-core shapes; otherwise they run on reversed and
// conjugated copies of the inputs.
bool folded_runs(int64_t N, int64_t P, int chunk) {
    return tc_forward_supported(N, P, chunk) && tc_full_shape(N, P) && tc_full_shape(P, N);
}

// With the folded runs and T a multiple of 64, R_t comes from chunk-local sums
// and the boundary inner products of the two runs' published states.
bool boundary_sums(int64_t T, int64_t N, int64_t P, int chunk) {
    return folded_runs(N, P, chunk) && N == 64 && P == 64 && T % 64 == 0;
}

// Workspace regions of the backward, in order (the copies only without the
// folded runs, the state dumps only with the boundary sums).
struct BwdLayout {
    size_t y, dyR, dts, ccR, bcR, xcR, dyc, tmp, Ac, zero, r, d, gAp, gDp, Hd, Gd, Hrot, Grot, Rb, fwd, total;
};

BwdLayout bwd_layout(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk) {
    const size_t TP = (size_t)(Bz * T * H * P) * sizeof(float2), TN = (size_t)(Bz * T * H * N) * sizeof(float2);
    const size_t TH = (size_t)(Bz * T * H);
    const bool folded = folded_runs(N, P, chunk);
    BwdLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += align256(bytes);
        return o;
    };
    L.y = take(TP);
    if (!folded) {
        L.dyR = take(TP);
        L.dts = take(TH * sizeof(float));
        L.ccR = take(TN);
        L.bcR = take(TN);
        L.xcR = take(TP);
        L.dyc = take(TP);
        L.tmp = take(TP > TN ? TP : TN);
        L.Ac = take((size_t)H * sizeof(float2));
        L.zero = take((size_t)H * sizeof(float));
    }
    L.r = take(TH * sizeof(float2));
    L.d = take(TH * sizeof(float));
    L.gAp = take((size_t)(Bz * H) * sizeof(double2));
    L.gDp = take((size_t)(Bz * H) * sizeof(double));
    if (boundary_sums(T, N, P, chunk)) {
        const size_t slots = (size_t)(Bz * H) * (size_t)(T / 64 + 1);
        L.Hd = take(slots * 2 * 64 * 64 * sizeof(float));
        L.Gd = take(slots * 2 * 64 * 64 * sizeof(float));
        L.Hrot = take(slots * sizeof(float2));
        L.Grot = take(slots * sizeof(float2));
        L.Rb = take(slots * sizeof(double2));
    }
    const size_t f1 = precise_forward_workspace_bytes(Bz, T, H, N, P, chunk);  // y and gx runs
    const size_t f2 = forward_workspace_bytes(Bz, T, H, P, N, chunk);          // transposed-state runs
    L.fwd = take(f1 > f2 ? f1 : f2);
    L.total = off;
    return L;
}

}  // namespace

bool backward_supported(int64_t N, int64_t P) {
    auto ok = [](int64_t v) { return v == 16 || v == 32 || v == 64; };
    return (ok(N) || N == 128) && ok(P);
}

size_t backward_workspace_bytes(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk) {
    return bwd_layout(Bz, T, H, N, P, chunk).total;
}

cudaError_t launch_backward(const BwdArgs& a, void* workspace, cudaStream_t st) {
    const int64_t Bz = a.Bz, T = a.T, H = a.H, N = a.N, P = a.P;
    const BwdLayout L = bwd_layout(Bz, T, H, N, P, a.chunk);
    unsigned char* w = static_cast<unsigned char*>(workspace);
    auto f2p = [&](size_t o) { return reinterpret_cast<float2*>(w + o); };
    auto fp = [&](size_t o) { return reinterpret_cast<float*>(w + o); };
    void* fws = w + L.fwd;
    cudaError_t e = cudaSuccess;
    auto check = [&]() { return (e = cudaGetLastError()) == cudaSuccess; };

    const bool bsum = boundary_sums(T, N, P, a.chunk);
    float* Hd = bsum ? fp(L.Hd) : nullptr;
    float* Gd = bsum ? fp(L.Gd) : nullptr;
    float2* Hrot = bsum ? f2p(L.Hrot) : nullptr;
    float2* Grot = bsum ? f2p(L.Grot) : nullptr;

    // Forward output, to about fp32 accuracy (and its chunk states).
    const float2* y = f2p(L.y);
    {
        FwdArgs f{Bz, T, H, N, P, a.chunk, a.x, a.dt, a.A, a.B, a.C, a.D, f2p(L.y), nullptr};
        if (bsum) {
            f.mode = kFwdDump;
            f.dump = Hd;
            f.rot_dump = Hrot;
        }
        if ((e = launch_precise_forward(f, fws, st)) != cudaSuccess) return e;
    }

    if (folded_runs(N, P, a.chunk)) {
        // gx: the adjoint run, time reversed (the step of token t + 1 at
        // reversed position T - 1 - t), input dy, coupling conj(C), readout
        // conj(B), rate conj(A), skip D; written in token order.
        {
            FwdArgs f{Bz, T, H, N, P, a.chunk, a.dy, a.dt, a.A, a.C, a.B, a.D, a.gx, nullptr};
            f.mode = kFwdReverse | kFwdShiftDt | kFwdConjA | kFwdConjB | kFwdConjC;
            if (bsum) {
                f.mode |= kFwdDump;
                f.dump = Gd;
                f.rot_dump = Grot;
            }
            if ((e = launch_precise_forward(f, fws, st)) != cudaSuccess) return e;
        }
        // gB: the same reversed run with the state transposed: input conj(C),
        // coupling dy, readout conj(x), no skip.
        {
            FwdArgs f{Bz, T, H, P, N, a.chunk, a.C, a.dt, a.A, a.dy, a.x, nullptr, a.gB, nullptr};
            f.mode = kFwdReverse | kFwdShiftDt | kFwdConjA | kFwdConjX | kFwdConjC;
            if ((e = launch_forward(f, fws, st)) != cudaSuccess) return e;
        }
        // gC: the forward run with the state transposed (input B, coupling x,
        // readout conj(dy)), output conjugated, no skip.
        {
            FwdArgs f{Bz, T, H, P, N, a.chunk, a.B, a.dt, a.A, a.x, a.dy, nullptr, a.gC, nullptr};
            f.mode = kFwdConjC | kFwdConjY;
            if ((e = launch_forward(f, fws, st)) != cudaSuccess) return e;
        }
    } else {
        // Reversed and conjugated inputs.
        float2 *dyR = f2p(L.dyR), *ccR = f2p(L.ccR), *bcR = f2p(L.bcR), *xcR = f2p(L.xcR), *dyc = f2p(L.dyc);
        float2* Ac = f2p(L.Ac);
        float *dts = fp(L.dts), *zero = fp(L.zero);
        reverse_rows_kernel<<<grid_rows(Bz * T), EB, 0, st>>>(a.dy, dyR, Bz, T, H * P, false);
        reverse_rows_kernel<<<grid_rows(Bz * T), EB, 0, st>>>(a.C, ccR, Bz, T, H * N, true);
        reverse_rows_kernel<<<grid_rows(Bz * T), EB, 0, st>>>(a.B, bcR, Bz, T, H * N, true);
        reverse_rows_kernel<<<grid_rows(Bz * T), EB, 0, st>>>(a.x, xcR, Bz, T, H * P, true);
        conj_kernel<<<grid_for(Bz * T * H * P), EB, 0, st>>>(a.dy, dyc, Bz * T * H * P);
        reverse_steps_kernel<<<grid_for(Bz * T * H), EB, 0, st>>>(a.dt, dts, Bz, T, H, a.A, Ac, zero);
        if (!check()) return e;

        float2* tmp = f2p(L.tmp);
        // gx: reversed run (about fp32 accuracy), then back to token order.
        {
            FwdArgs f{Bz, T, H, N, P, a.chunk, dyR, dts, Ac, ccR, bcR, a.D, tmp, nullptr};
            if ((e = launch_precise_forward(f, fws, st)) != cudaSuccess) return e;
            reverse_rows_kernel<<<grid_rows(Bz * T), EB, 0, st>>>(tmp, a.gx, Bz, T, H * P, false);
            if (!check()) return e;
        }
        // gB: reversed run with the state transposed (dstate P, headdim N).
        {
            FwdArgs f{Bz, T, H, P, N, a.chunk, ccR, dts, Ac, dyR, xcR, zero, tmp, nullptr};
            if ((e = launch_forward(f, fws, st)) != cudaSuccess) return e;
            reverse_rows_kernel<<<grid_rows(Bz * T), EB, 0, st>>>(tmp, a.gB, Bz, T, H * N, false);
            if (!check()) return e;
        }
        // gC: forward run with the state transposed; gC = conj(output).
        {
            FwdArgs f{Bz, T, H, P, N, a.chunk, a.B, a.dt, a.A, a.x, dyc, zero, tmp, nullptr};
            if ((e = launch_forward(f, fws, st)) != cudaSuccess) return e;
            conj_kernel<<<grid_for(Bz * T * H * N), EB, 0, st>>>(tmp, a.gC, Bz * T * H * N);
            if (!check()) return e;
        }
    }
    // Step, rate and skip gradients.
    float2* r = f2p(L.r);
    float* d = fp(L.d);
    double2* gAp = reinterpret_cast<double2*>(w + L.gAp);
    double* gDp = reinterpret_cast<double*>(w + L.gDp);
    token_terms_kernel<<<grid_for(Bz * T * H * 32), EB, 0, st>>>(a.x, y, a.dy, a.gx, r, d, Bz * T * H, (int)P);
    if (bsum) {
        const int nc = (int)(T / 64);
        double2* Rb = reinterpret_cast<double2*>(w + L.Rb);
        if (nc > 1)
            boundary_kernel<<<(unsigned)((int64_t)(nc - 1) * Bz * H), EB, 0, st>>>(Hd, Hrot, Gd, Grot, a.dt, a.A, Rb,
                                                                                   T, H, nc);
        chunk_scan_kernel<<<(unsigned)(Bz * H), EB, 0, st>>>(r, d, a.dt, a.A, Rb, a.gdt, gAp, gDp, T, H, nc);
    } else {
        reverse_scan_kernel<<<(unsigned)(Bz * H), EB, 0, st>>>(r, d, a.dt, a.A, a.gdt, gAp, gDp, T, H);
    }
    head_sums_kernel<<<grid_for(H), EB, 0, st>>>(gAp, gDp, a.gA, a.gD, Bz, H);
    check();
    return e;
}

}  // namespace cssd
