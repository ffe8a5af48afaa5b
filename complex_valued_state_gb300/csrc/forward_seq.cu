// Chunk-parallel forward, CUDA-core version.
//
// Three launches on the caller's stream:
//   1. chunk_state   (grid chunks x heads x batch): runs the recurrence over
//      the chunk's tokens from a zero state and stores the chunk's end state
//      S_c (N x P) and its total decay E_c = exp(sum of the chunk's log-steps);
//   2. state_scan    (grid state-slices x heads*batch): the inter-chunk scan
//      H_{c+1} = E_c H_c + S_c, H_0 = the initial state (zero unless given),
//      written over S_c in place, plus the final state;
//   3. chunk_output  (grid chunks x heads x batch): the recurrence over the
//      chunk again, started from H_c, with the readout y = C^T h + D x.
// The split into per-chunk end states, a short scan over chunks and a
// per-chunk readout from the carried-in state is the chunkwise decomposition
// of "The Chunkwise Complex SSD Algorithm" (Mamba-3-Lite docs), sections 4.1
// and 4.5; padded positions of the last chunk are masked (zero input, decay 1)
// so the final state is the state after the last real token.

#include "cssd_common.cuh"
#include "cssd_internal.h"

namespace cssd {
namespace {

constexpr int kTB = 16;  // tokens staged in shared memory per step

template <int N, int P>
struct SeqShape {
    static constexpr int NPT = (N >= 16) ? 16 : N;  // state rows per thread
    static constexpr int R = N / NPT;                // threads sharing a column
    static constexpr int NT = P * R;                 // threads per CTA
};

// Thread t owns column p = t / R and rows n = r + R * i (r = t % R); the R
// threads of a column are adjacent lanes, so the readout reduces by shuffles.
template <int N, int P, bool READOUT>
__global__ void __launch_bounds__(SeqShape<N, P>::NT)
    chunk_seq_kernel(const float2* __restrict__ x, const float* __restrict__ dt, const float2* __restrict__ A,
                     const float2* __restrict__ Bm, const float2* __restrict__ Cm, const float* __restrict__ D,
                     float2* __restrict__ y, float2* __restrict__ Sbuf, float2* __restrict__ Ebuf, int T, int H,
                     int chunk, int nc) {
    using S = SeqShape<N, P>;
    __shared__ float2 sB[kTB][N];
    __shared__ float2 sC[READOUT ? kTB : 1][N];
    __shared__ float2 sX[kTB][P];
    __shared__ float2 sA[kTB];
    __shared__ float2 sLog[kTB];

    const int c = blockIdx.x, hd = blockIdx.y, b = blockIdx.z;
    const int t = threadIdx.x;
    const int r = t % S::R, p = t / S::R;
    const size_t bhc = ((size_t)b * H + hd) * nc + c;
    float2* state = Sbuf + bhc * (N * P);

    float2 s[S::NPT];
#pragma unroll
    for (int i = 0; i < S::NPT; ++i)
        s[i] = READOUT ? state[(r + S::R * i) * P + p] : make_float2(0.f, 0.f);
    const float2 Ah = A[hd];
    const float Dh = D[hd];
    float2 logsum = make_float2(0.f, 0.f);

    const int t0 = c * chunk;
    const int tend = min(t0 + chunk, T);
    for (int tb = t0; tb < tend; tb += kTB) {
        const int nt = min(kTB, tend - tb);
        __syncthreads();
        for (int i = t; i < kTB * N; i += S::NT) {
            const int j = i / N, n = i % N;
            const size_t row = ((size_t)b * T + tb + j) * H + hd;
            const bool ok = j < nt;
            sB[j][n] = ok ? Bm[row * N + n] : make_float2(0.f, 0.f);
            if (READOUT) sC[j][n] = ok ? Cm[row * N + n] : make_float2(0.f, 0.f);
        }
        for (int i = t; i < kTB * P; i += S::NT) {
            const int j = i / P, pp = i % P;
            const size_t row = ((size_t)b * T + tb + j) * H + hd;
            sX[j][pp] = (j < nt) ? x[row * P + pp] : make_float2(0.f, 0.f);
        }
        if (t < kTB) {
            float2 lg = make_float2(0.f, 0.f);
            if (t < nt) lg = alog_of(dt[((size_t)b * T + tb + t) * H + hd], Ah);
            sLog[t] = lg;
            sA[t] = cexpf2(lg);
        }
        __syncthreads();
        if (!READOUT && t == 0)
            for (int j = 0; j < nt; ++j) logsum = cadd(logsum, sLog[j]);
        for (int j = 0; j < nt; ++j) {
            const float2 a = sA[j];
            const float2 xv = sX[j][p];
#pragma unroll
            for (int i = 0; i < S::NPT; ++i) s[i] = cfma(sB[j][r + S::R * i], xv, cmul(a, s[i]));
            if (READOUT) {
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < S::NPT; ++i) acc = cfma(sC[j][r + S::R * i], s[i], acc);
#pragma unroll
                for (int off = S::R / 2; off > 0; off >>= 1) {
                    acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
                    acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
                }
                if (r == 0) {
                    const size_t row = ((size_t)b * T + tb + j) * H + hd;
                    y[row * P + p] = cadd(acc, cscale(Dh, xv));
                }
            }
        }
    }
    if (!READOUT) {
#pragma unroll
        for (int i = 0; i < S::NPT; ++i) state[(r + S::R * i) * P + p] = s[i];
        if (t == 0) Ebuf[bhc] = cexpf2(logsum);
    }
}

// Inter-chunk scan: each thread carries two complex entries of one head's
// state through all chunks.  S_c is replaced by H_c (the state entering c).
// Grid: x = batch * head, y = 256-wide slices of the state.
__global__ void __launch_bounds__(256)
    state_scan_kernel(float4* __restrict__ Sbuf, const float2* __restrict__ Ebuf, const float4* __restrict__ h0,
                      float4* __restrict__ h_final, int np2, int nc) {
    const int idx = blockIdx.y * blockDim.x + threadIdx.x;
    if (idx >= np2) return;
    const size_t bh = blockIdx.x;
    float4* Sp = Sbuf + bh * (size_t)nc * np2 + idx;
    const float2* E = Ebuf + bh * nc;
    float2 c0 = make_float2(0.f, 0.f), c1 = c0;
    if (h0) {  // the caller's state before the first token
        const float4 v = h0[bh * np2 + idx];
        c0 = make_float2(v.x, v.y);
        c1 = make_float2(v.z, v.w);
    }
    constexpr int U = 8;
    for (int cb = 0; cb < nc; cb += U) {
        float4 v[U];
        float2 e[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (cb + k < nc) {
                v[k] = __ldcs(Sp + (size_t)(cb + k) * np2);
                e[k] = E[cb + k];
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (cb + k < nc) {
                Sp[(size_t)(cb + k) * np2] = make_float4(c0.x, c0.y, c1.x, c1.y);
                c0 = cfma(e[k], c0, make_float2(v[k].x, v[k].y));
                c1 = cfma(e[k], c1, make_float2(v[k].z, v[k].w));
            }
        }
    }
    if (h_final) h_final[bh * np2 + idx] = make_float4(c0.x, c0.y, c1.x, c1.y);
}

template <int N, int P>
cudaError_t launch_np(const FwdArgs& a, float2* Sbuf, float2* Ebuf, cudaStream_t st) {
    const int nc = (int)((a.T + a.chunk - 1) / a.chunk);
    const dim3 grid(nc, (unsigned)a.H, (unsigned)a.Bz);
    constexpr int NT = SeqShape<N, P>::NT;
    chunk_seq_kernel<N, P, false><<<grid, NT, 0, st>>>(a.x, a.dt, a.A, a.B, a.C, a.D, a.y, Sbuf, Ebuf, (int)a.T,
                                                        (int)a.H, a.chunk, nc);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int np2 = (int)(a.N * a.P / 2);
    state_scan_kernel<<<dim3((unsigned)(a.Bz * a.H), (np2 + 255) / 256), 256, 0, st>>>(
        reinterpret_cast<float4*>(Sbuf), Ebuf, reinterpret_cast<const float4*>(a.h0),
        reinterpret_cast<float4*>(a.h_final), np2, nc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (g_prof_begin) cudaEventRecord(g_prof_begin, st);
    chunk_seq_kernel<N, P, true><<<grid, NT, 0, st>>>(a.x, a.dt, a.A, a.B, a.C, a.D, a.y, Sbuf, Ebuf, (int)a.T,
                                                       (int)a.H, a.chunk, nc);
    e = cudaGetLastError();
    if (g_prof_end) cudaEventRecord(g_prof_end, st);
    return e;
}

template <int N>
cudaError_t launch_n(const FwdArgs& a, float2* S, float2* E, cudaStream_t st) {
    switch (a.P) {
        case 16: return launch_np<N, 16>(a, S, E, st);
        case 32: return launch_np<N, 32>(a, S, E, st);
        case 64: return launch_np<N, 64>(a, S, E, st);
        case 128:
            // headdim 128 with dstate up to 64: the gradient runs of dstate 128
            // (their state is the transpose, headdim and dstate swapped)
            if constexpr (N <= 64) return launch_np<N, 128>(a, S, E, st);
            break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace

size_t seq_forward_workspace_bytes(int64_t Bz, int64_t T, int64_t H, int64_t N, int64_t P, int chunk) {
    const int64_t nc = (T + chunk - 1) / chunk;
    const size_t states = (size_t)(Bz * H * nc) * (size_t)(N * P) * sizeof(float2);
    const size_t totals = (size_t)(Bz * H * nc) * sizeof(float2);
    return states + ((totals + 255) / 256) * 256;
}

cudaError_t launch_seq_forward(const FwdArgs& a, void* ws, cudaStream_t st) {
    const int64_t nc = (a.T + a.chunk - 1) / a.chunk;
    float2* S = static_cast<float2*>(ws);
    float2* E = S + (size_t)(a.Bz * a.H * nc) * (size_t)(a.N * a.P);
    switch (a.N) {
        case 16: return launch_n<16>(a, S, E, st);
        case 32: return launch_n<32>(a, S, E, st);
        case 64: return launch_n<64>(a, S, E, st);
        case 128: return launch_n<128>(a, S, E, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace cssd
