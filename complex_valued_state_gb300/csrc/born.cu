// Causal Born attention on the tcgen05 tensor cores ("Complex Phase-State
// Dynamics Reduce the Optimization Steps of Sequence Models", section 5.5,
// equation (5), Appendix A Algorithm 3).  Per (batch, head):
//     s_ij  = |<q_i|k_j>|^2 / (D tau_i),  <q|k> = sum_a conj(q_a) k_a,  j <= i
//     psi_i = sum_{j<=i} s_ij v_j / sum_{j<=i} s_ij
// The factor 1/(D tau_i) is common to a row's numerator and denominator and is
// left out (psi does not depend on it).
//
// One CTA of 256 threads owns 128 queries of one head, one per tensor-memory
// lane, and walks the key blocks of 64 up to the diagonal (a head's CTAs are
// launched together, its longest first, so its keys and values are read from
// DRAM about once).  Per key block the real and imaginary scores are real
// GEMMs into two accumulators, the threads square them in place, and the
// value GEMM reads the squared scores from tensor memory; a row of ones in
// the value operand makes one accumulator column the running sum of scores.
// Scores need no rescaling between key blocks: they are non-negative and the
// normalisation is a plain sum, so numerator and denominator accumulate in
// fp32 in tensor memory across all blocks.

#include <atomic>

#include "cssd_common.cuh"
#include "cssd_internal.h"
#include "tcgen05.cuh"

namespace cssd {
namespace {

constexpr long long kBornWait = 4000000000LL;  // ~2 s at 2 GHz

__device__ __forceinline__ uint32_t kofs(int row, int k, int rows) {
    return (uint32_t)((((k >> 2) * (rows >> 3) + (row >> 3)) << 7) + ((row & 7) << 4) + ((k & 3) << 2));
}
__device__ __forceinline__ float rna_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}
__device__ __forceinline__ void sts(unsigned char* base, uint32_t off, float v) {
    *reinterpret_cast<float*>(base + off) = v;
}
__device__ __forceinline__ void sts2(unsigned char* base, uint32_t off, float a, float b) {
    *reinterpret_cast<float2*>(base + off) = make_float2(a, b);
}

// ------------------------------------------------------------------ 128 queries per CTA
// born_kernel_q128<D>: 128 queries per CTA, one per tensor-memory lane, the
// real and imaginary scores in two accumulators:
//   Re G = [Qr | Qi] [Kr | Ki]^T            (K = 2D)
//   Im G = Qr Ki^T - Qi Kr^T                (the two K = D halves of the same
//                                            operands, the second negated)
//   S = (Re G)^2 + (Im G)^2                  over Re G in tensor memory
//   ACC += S [Vr; Vi; 1]^T                   (A = S from tensor memory)
// so each lane ends with its query's numerator and score sum.  256 threads
// (two per lane, one column half each) and 256 tensor-memory columns; 56 KB
// of shared memory at width 16, 104 KB at 32: two CTAs per SM.
template <int D>
struct BornQ {
static constexpr int BQ = 128;                    // queries per CTA
static constexpr int NT = 256;                    // threads
static constexpr int BK = 64;                     // keys per block
static constexpr int K2 = 2 * D;                  // K of the score GEMM
static constexpr int NB = 2 * D + 16;             // value operand rows: Vr, Vi, ones, zeros
static constexpr int Q_BYTES = BQ * K2 * 4;       // rows q, K = [qr | qi]
static constexpr int K_BYTES = BK * K2 * 4;       // rows j, K = [kr | ki]
static constexpr int V_BYTES = NB * BK * 4;       // rows m, K = j
static constexpr int KV_BYTES = K_BYTES + V_BYTES;
static constexpr int SMEM = Q_BYTES + 2 * KV_BYTES;  // two key blocks in flight
static constexpr int ITEMS = BK * D / 2 / NT;     // float4 of keys (and of values) per thread per key block
static constexpr uint32_t COL_RE = 0, COL_IM = BK, COL_ACC = 2 * BK, TMEM_COLS = 256;  // S over Re G
static constexpr uint32_t Q_LBO = (BQ / 8) * 128, K_LBO = (BK / 8) * 128, V_LBO = (NB / 8) * 128, SBO = 128;
static constexpr int KSTEPS = K2 / 8;             // MMAs of K = 8 over [Re | Im]
static constexpr int NACC = (NB + 15) / 16 * 16;  // accumulator columns read back
static_assert(COL_ACC + NB <= TMEM_COLS && ITEMS * NT * 2 == BK * D, "budget and item mapping");
static_assert(2 * (SMEM + 2048) <= 227 * 1024, "two CTAs per SM");
};

template <int D>
__global__ void __launch_bounds__(256, 2) born_kernel_q128(const float4* __restrict__ q, const float4* __restrict__ k,
                                                          const float4* __restrict__ v, float2* __restrict__ psi,
                                                          int T, int H, int nqb, unsigned* status) {
    using bw = BornQ<D>;
    constexpr int BQ2 = bw::BQ, BK = bw::BK, NB = bw::NB, IT = bw::ITEMS;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t mbar[3];  // G done, drain, ACC update done
    __shared__ int s_gave_up;
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char* sq = smem;
    auto skb = [&](int buf) { return smem + bw::Q_BYTES + buf * bw::KV_BYTES; };
    auto svb = [&](int buf) { return skb(buf) + bw::K_BYTES; };
    // The query blocks of one head are consecutive CTAs, its latest (longest) block first.
    const int bh = (int)(blockIdx.x / nqb);
    const int qb = nqb - 1 - (int)(blockIdx.x % nqb);
    const int b = bh / H, h = bh - b * H;
    const int i0 = qb * BQ2;
    auto tok = [&](const float4* base, int t) { return base + ((size_t)((size_t)b * T + t) * H + h) * (D / 2); };

    if (warp == 0) {
        tc::tmem_alloc(&s_tmem, bw::TMEM_COLS);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        s_gave_up = 0;
        for (int i = 0; i < 3; ++i) tc::mbar_init(&mbar[i], 1);
        tc::mbar_fence_init();
    }
    // Rows 2D.. of both value operands: ones (the score sum), then zeros.
    for (int e = tid; e < 2 * (NB - 2 * D) * BK; e += bw::NT) {
        const int buf = e / ((NB - 2 * D) * BK), f = e % ((NB - 2 * D) * BK);
        const int r = 2 * D + f / BK, j = f % BK;
        sts(svb(buf), kofs(r, j, NB), r == 2 * D ? 1.f : 0.f);
    }
    // [Qr | Qi] (rows q, K = 32): item e is float4 c (two complex) of query e / (D / 2).
    for (int e = tid; e < BQ2 * D / 2; e += bw::NT) {
        const int i = e / (D / 2), c = 2 * (e % (D / 2));
        const float4 x = (i0 + i < T) ? __ldg(tok(q, i0 + i) + c / 2) : make_float4(0.f, 0.f, 0.f, 0.f);
        sts2(sq, kofs(i, c, BQ2), rna_tf32(x.x), rna_tf32(x.z));
        sts2(sq, kofs(i, D + c, BQ2), rna_tf32(x.y), rna_tf32(x.w));
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;

    // Tensor-memory lane L = 32 (warp mod 4) + lane = query i0 + L; column half ch.
    const int L = (warp & 3) * 32 + lane, ch = warp >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    // Keys and values of a block in registers: item e = tid + NT i is float4
    // c (two complex) of key e / (D / 2), so 8 consecutive lanes read one key row.
    const int j0 = tid / (D / 2), c0 = 2 * (tid % (D / 2));
    constexpr int JS = bw::NT / (D / 2);  // keys between a thread's items
    const size_t tok_stride = (size_t)H * (D / 2);
    const float4* kbase = tok(k, 0) + (size_t)j0 * tok_stride + c0 / 2;
    const float4* vbase = tok(v, 0) + (size_t)j0 * tok_stride + c0 / 2;
    float4 kr[IT], vr[IT];
    auto load_kv = [&](int kb) {
#pragma unroll
        for (int i = 0; i < IT; ++i) {
            const int t = kb * BK + j0 + JS * i;
            const size_t o = (size_t)(kb * BK + JS * i) * tok_stride;
            kr[i] = t < T ? __ldg(kbase + o) : make_float4(0.f, 0.f, 0.f, 0.f);
            vr[i] = t < T ? __ldg(vbase + o) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    auto write_kv = [&](int buf) {
        unsigned char* sk = skb(buf);
        unsigned char* sv = svb(buf);
#pragma unroll
        for (int i = 0; i < IT; ++i) {
            const int j = j0 + JS * i;
            sts2(sk, kofs(j, c0, BK), rna_tf32(kr[i].x), rna_tf32(kr[i].z));
            sts2(sk, kofs(j, D + c0, BK), rna_tf32(kr[i].y), rna_tf32(kr[i].w));
            sts(sv, kofs(c0, j, NB), rna_tf32(vr[i].x));
            sts(sv, kofs(c0 + 1, j, NB), rna_tf32(vr[i].z));
            sts(sv, kofs(D + c0, j, NB), rna_tf32(vr[i].y));
            sts(sv, kofs(D + c0 + 1, j, NB), rna_tf32(vr[i].w));
        }
        tc::fence_proxy_async();
    };
    const uint32_t ID_G = tc::idesc_tf32(128, BK), ID_GN = tc::idesc_tf32(128, BK, false, true);
    const uint32_t ID_V = tc::idesc_tf32(128, NB);
    constexpr uint64_t Q_STEP = (2 * bw::Q_LBO) >> 4, K_STEP = (2 * bw::K_LBO) >> 4, V_STEP = (2 * bw::V_LBO) >> 4;
    const uint64_t a_q = tc::make_desc(tc::smem_u32(sq), bw::Q_LBO, bw::SBO);
    // Re G and Im G of block kb (operands in buffer kb & 1).  One MMA takes
    // K = 8: the first half of the steps covers the real parts, the second
    // the imaginary ones.
    auto issue_g = [&](int kb) {
        const uint64_t b_k = tc::make_desc(tc::smem_u32(skb(kb & 1)), bw::K_LBO, bw::SBO);
        constexpr int HS = bw::KSTEPS / 2;  // steps over one half (the real or the imaginary parts)
#pragma unroll
        for (int ks = 0; ks < bw::KSTEPS; ++ks)
            tc::mma_tf32(tmem + bw::COL_RE, a_q + ks * Q_STEP, b_k + ks * K_STEP, ID_G, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < HS; ++ks)  // Qr Ki^T
            tc::mma_tf32(tmem + bw::COL_IM, a_q + ks * Q_STEP, b_k + (HS + ks) * K_STEP, ID_G, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < HS; ++ks)  // - Qi Kr^T
            tc::mma_tf32(tmem + bw::COL_IM, a_q + (HS + ks) * Q_STEP, b_k + ks * K_STEP, ID_GN, 1u);
        tc::commit(&mbar[0]);
    };

    const int nkb = (T + BK - 1) / BK;
    const int last = min((i0 + BQ2) / BK, nkb) - 1;  // the key blocks up to the query block's last position
    bool ok = true;
    load_kv(0);
    write_kv(0);
    if (last > 0) load_kv(1);
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        tc::fence_after_sync();
        issue_g(0);
    }
#pragma unroll 1
    for (int kb = 0; kb <= last; ++kb) {
        const int buf = kb & 1;
        ok = tc::mbar_wait_bounded(&mbar[0], (uint32_t)(kb & 1), kBornWait) && ok;
        tc::fence_after_sync();
        // S = (Re G)^2 + (Im G)^2 over Re G, this thread's lane and column half
        {
            uint32_t re[32], im[32];
            const uint32_t col = tmem + lane_base + 32 * ch;
            tc::tmem_ld16(col + bw::COL_RE, *reinterpret_cast<uint32_t(*)[16]>(re));
            tc::tmem_ld16(col + bw::COL_RE + 16, *reinterpret_cast<uint32_t(*)[16]>(re + 16));
            tc::tmem_ld16(col + bw::COL_IM, *reinterpret_cast<uint32_t(*)[16]>(im));
            tc::tmem_ld16(col + bw::COL_IM + 16, *reinterpret_cast<uint32_t(*)[16]>(im + 16));
            tc::tmem_wait_ld();
            const int kq = i0 + L - kb * BK - 32 * ch;  // the last key of this column half the query may see
            if (kq < 31) {  // a block on the diagonal: keys after the query are masked
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float gr = __uint_as_float(re[j]), gi = __uint_as_float(im[j]);
                    re[j] = __float_as_uint(j <= kq ? fmaf(gr, gr, gi * gi) : 0.f);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float gr = __uint_as_float(re[j]), gi = __uint_as_float(im[j]);
                    re[j] = __float_as_uint(fmaf(gr, gr, gi * gi));
                }
            }
            tc::tmem_st16(col + bw::COL_RE, *reinterpret_cast<uint32_t(*)[16]>(re));
            tc::tmem_st16(col + bw::COL_RE + 16, *reinterpret_cast<uint32_t(*)[16]>(re + 16));
            tc::tmem_wait_st();
        }
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            const uint64_t b_v = tc::make_desc(tc::smem_u32(svb(buf)), bw::V_LBO, bw::SBO);
#pragma unroll
            for (int ks = 0; ks < BK / 8; ++ks)
                tc::mma_tf32_ts(tmem + bw::COL_ACC, tmem + bw::COL_RE + 8 * ks, b_v + ks * V_STEP, ID_V,
                                (kb > 0 || ks > 0) ? 1u : 0u);
            tc::commit(&mbar[2]);
        }
        if (kb < last) {
            // The other buffer was last read by G and the ACC update of block
            // kb - 1, both complete.
            write_kv(buf ^ 1);
            if (kb + 1 < last) load_kv(kb + 2);
            // Re G and Im G are free once this block's ACC update is done.
            ok = tc::mbar_wait_bounded(&mbar[2], (uint32_t)(kb & 1), kBornWait) && ok;
            tc::fence_before_sync();
            __syncthreads();
            if (tid == 0) {
                tc::fence_after_sync();
                issue_g(kb + 1);
            }
        }
    }
    ok = tc::mbar_wait_bounded(&mbar[2], (uint32_t)(last & 1), kBornWait) && ok;
    tc::fence_after_sync();

    // Epilogue: lane L holds its query's numerator (columns 0 to D-1 real,
    // D to 2D-1 imaginary parts) and score sum (column 2D).
    uint32_t acc[bw::NACC];
    if (ch == 0) {  // warp-uniform: the tensor-memory loads are collective over the warp
#pragma unroll
        for (int cb = 0; cb < bw::NACC / 16; ++cb)
            tc::tmem_ld16(tmem + lane_base + bw::COL_ACC + 16 * cb, *reinterpret_cast<uint32_t(*)[16]>(acc + 16 * cb));
        tc::tmem_wait_ld();
    }
    if (ch == 0 && i0 + L < T) {
        const float den = __uint_as_float(acc[2 * D]);
        const float inv = den != 0.f ? 1.f / den : 0.f;
        float2* out = psi + ((size_t)((size_t)b * T + i0 + L) * H + h) * D;
#pragma unroll
        for (int m = 0; m < D; m += 2)
            *reinterpret_cast<float4*>(out + m) =
                make_float4(__uint_as_float(acc[m]) * inv, __uint_as_float(acc[D + m]) * inv,
                            __uint_as_float(acc[m + 1]) * inv, __uint_as_float(acc[D + m + 1]) * inv);
    }
    if (!ok) s_gave_up = 1;  // a completion wait gave up
    __syncthreads();
    if (s_gave_up && tid == 0) {
        if (status) atomicOr(status, kStatusBornMma);
        tc::drain_mmas(&mbar[1], kBornWait);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, bw::TMEM_COLS);
}

template <int D>
static cudaError_t launch_born_q128(const BornArgs& a, cudaStream_t st) {
    using bw = BornQ<D>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<bool> attr_set[128];
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(born_kernel_q128<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bw::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    const int64_t BH = a.Bz * a.H, nqb = (a.T + bw::BQ - 1) / bw::BQ;
    born_kernel_q128<D><<<(unsigned)(BH * nqb), bw::NT, bw::SMEM, st>>>(
        reinterpret_cast<const float4*>(a.q), reinterpret_cast<const float4*>(a.k), reinterpret_cast<const float4*>(a.v),
        a.psi, (int)a.T, (int)a.H, (int)nqb, status_word());
    return cudaGetLastError();
}

}  // namespace

bool born_supported(int64_t D) { return D == 16 || D == 32; }

cudaError_t launch_born(const BornArgs& a, cudaStream_t st) {
    return a.D == 16 ? launch_born_q128<16>(a, st) : launch_born_q128<32>(a, st);
}

}  // namespace cssd
