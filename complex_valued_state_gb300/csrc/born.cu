// Causal Born attention on the tcgen05 tensor cores ("Complex Phase-State
// Dynamics Reduce the Optimization Steps of Sequence Models", section 5.5,
// equation (5), Appendix A Algorithm 3).  Per (batch, head):
//     s_ij  = |<q_i|k_j>|^2 / (D tau_i),  <q|k> = sum_a conj(q_a) k_a,  j <= i
//     psi_i = sum_{j<=i} s_ij v_j / sum_{j<=i} s_ij
// The factor 1/(D tau_i) is common to a row's numerator and denominator and is
// left out (psi does not depend on it).
//
// One CTA owns 128 queries of one head, one per tensor-memory lane, and walks
// the key blocks of 32 up to the diagonal (a head's CTAs are launched
// together, its longest first, so its keys and values are read from DRAM
// about once).  Per key block the real and imaginary scores are real GEMMs,
// math warps square them in tensor memory, and the value GEMM reads the
// squared scores from there.  Scores need no rescaling between key blocks:
// they are non-negative and the normalisation is a plain sum, so numerator
// and denominator accumulate in fp32 in tensor memory across all blocks.

#include <atomic>

#include "cssd_common.cuh"
#include "cssd_internal.h"
#include "tcgen05.cuh"

namespace cssd {
namespace {

constexpr long long kBornWait = 4000000000LL;  // ~2 s at 2 GHz

__device__ __forceinline__ float rna_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}
__device__ __forceinline__ void sts(unsigned char* base, uint32_t off, float v) {
    *reinterpret_cast<float*>(base + off) = v;
}

// ------------------------------------------------------------------ the kernel
// born_kernel_ws<D>: 128 queries per CTA, blocks of 32 keys.  Eight math
// warps (two per lane quarter, one half of the key block each), one warp
// that runs the MMA loop (one elected lane issuing) and, at width 16, four
// loader warps:
//   G  = Q [K; K']^T          A = Q from tensor memory (the query rows as
//                             stored: re, im interleaved), B = the key block
//                             as stored and as (im, -re), so that columns
//                             0..31 hold Re <q|k> and 32..63 Im <q|k>
//   S  = (Re G)^2 + (Im G)^2  by the math warps, over Re G
//   ACC += S V^T              A = S from tensor memory, V rows interleaved
//                             (re, im) so that ACC is psi's row as stored
// The score sum: at width 16 a row of ones in V gives it an accumulator
// column; at width 32 (no tensor-memory columns left) each math thread
// rounds its S to TF32 and adds them up.  Queries, keys and values are
// rounded to TF32 on the way in.
// The score accumulator is double-buffered: the MMA warp queues G of block
// kb + 2 as soon as the value GEMM of block kb has read its scores, so the
// tensor core works on one block while the math warps square the next.  Key
// and value blocks go through shared-memory operand slots.  At width 16 the
// loader warps fill them: raw rows by cp.async six blocks ahead, rounded and
// stored by the thread that copied them.  At width 32 the math warps fill
// them two blocks ahead, from registers loaded two blocks before that.
template <int D>
struct BornW {
    static constexpr int BQ = 128;         // queries per CTA
    static constexpr int NMATH = 256;      // math threads: two per tensor-memory lane
    // Width 16: four loader warps stage the key/value blocks.  Width 32: the
    // math warps do (its raw blocks are twice the size, and a ring deep
    // enough for the loaders does not fit beside the operand slots).
    static constexpr bool LOADERS = D == 16;
    static constexpr int NLOAD = LOADERS ? 128 : 0;
    static constexpr int NT = NMATH + 32 + NLOAD;  // math warps 0-7, the MMA warp 8, loader warps 9-12
    static constexpr int BK = 32;          // keys per block
    static constexpr int K2 = 2 * D;       // K of the score GEMM
    static constexpr int NR = D == 16 ? 4 : 3;     // operand slots
    static constexpr int NRAW = LOADERS ? 6 : 0;   // raw key/value slots: blocks in flight from global memory
    static constexpr int IT = D / 16;      // float4 of keys (and of values) per math thread per block (math staging)
    static constexpr int LIT = LOADERS ? BK * D / 2 / NLOAD : 0;  // the same per loader thread
    // [K; K'] operand: 2 BK rows, K2 columns.  The k-group stride is one row
    // group set plus 16 bytes, so the eight lanes that store one key row's
    // eight 16-byte groups hit eight different bank groups.
    static constexpr uint32_t K_SBO = 128, K_LBO = (2 * BK / 8) * 128 + 16;
    static constexpr uint32_t K_BYTES = (K2 / 4) * K_LBO;
    // V operand: NB rows (component a's re in row 2a, im in row 2a + 1; at
    // width 16 a row of ones, whose accumulator column is the score sum, and
    // zeros), BK columns.  Row groups 144 bytes apart make the four-byte
    // column stores of a warp (four keys x eight float4) fall on 32 distinct
    // banks.
    static constexpr bool ONES = D == 16;
    static constexpr int NB = ONES ? 2 * D + 16 : 2 * D;
    static constexpr uint32_t V_SBO = 144, V_LBO = (NB / 8) * V_SBO;
    static constexpr uint32_t V_BYTES = (BK / 4) * V_LBO;
    static constexpr uint32_t SLOT = K_BYTES + V_BYTES;
    // Raw slot (loader staging): the block's key rows then its value rows as stored.
    static constexpr uint32_t RAW_HALF = BK * (D / 2) * 16, RAW = 2 * RAW_HALF;
    static constexpr uint32_t RAW0 = NR * SLOT;
    // At least 80 KB, so that no third CTA shares an SM (its tensor-memory
    // allocation would have to wait for one of the other two to finish).
    static constexpr uint32_t SMEM_NEED = (RAW0 + NRAW * RAW + 1023) / 1024 * 1024;
    static constexpr uint32_t SMEM = SMEM_NEED > 80 * 1024 ? SMEM_NEED : 80 * 1024;
    // Tensor memory: G buffers at 0 and 64 (Re then Im, S over Re), ACC at
    // 128, Q in the last K2 columns.
    static constexpr uint32_t COL_G = 0, COL_ACC = 128, TMEM_COLS = 256, COL_Q = TMEM_COLS - K2;
    static_assert(2 * (SMEM + 2048) <= 227 * 1024 && 3 * (SMEM + 1024) > 228 * 1024, "two CTAs per SM");
    static_assert(COL_ACC + NB <= COL_Q && V_LBO >= (NB / 8 - 1) * V_SBO + 128 && SLOT % 16 == 0, "layout");
    static_assert(NMATH == 8 * BK && (D == 16 || D == 32) && (!LOADERS || LIT * NLOAD * 2 == BK * D),
                  "item mappings: eight threads per key row");
};

// Wait for a phase parity with the thread suspended (not spinning) until the
// phase completes or a microsecond passes, giving up after `max_cycles`.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* m, uint32_t parity, long long max_cycles) {
    const long long t0 = clock64();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}\n"
            : "=r"(done)
            : "r"(tc::smem_u32(m)), "r"(parity), "r"(1000u)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > max_cycles) return false;
    }
}
__device__ __forceinline__ void mbar_arrive1(uint64_t* m) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(m)) : "memory");
}
// Issued from a converged warp: one elected lane runs the instruction, so the
// operands stay warp-uniform.  D[tmem] (+)= A[tmem] * B[smem]^T, kind::tf32.
__device__ __forceinline__ void mma_ts_warp(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
// The elected lane's commit: the barrier completes once its MMAs are done.
__device__ __forceinline__ void commit_warp(uint64_t* m) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(
            tc::smem_u32(m))
        : "memory");
}
__device__ __forceinline__ void sts4(unsigned char* base, uint32_t off, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(base + off) = make_float4(a, b, c, d);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ float4 lds4(const unsigned char* base, uint32_t off) {
    return *reinterpret_cast<const float4*>(base + off);
}

template <int D>
__global__ void __launch_bounds__(BornW<D>::NT, 2) born_kernel_ws(const float4* __restrict__ q, const float4* __restrict__ k,
                                                                 const float4* __restrict__ v, float2* __restrict__ psi,
                                                                 int T, int H, int nqb, unsigned* status) {
    using bw = BornW<D>;
    constexpr int BK = bw::BK, NR = bw::NR, IT = bw::IT, NRAW = bw::NRAW;
    extern __shared__ __align__(1024) unsigned char smem[];
    // G complete (per buffer), S stored (per buffer, one arrival per math
    // warp), operand slot written (one arrival per staging warp), operand
    // slot read (the value GEMM of the slot's block, and everything before
    // it, complete), drain.
    __shared__ __align__(8) uint64_t mb_g[2], mb_s[2], mb_kv[NR], mb_free[NR], mb_drain;
    __shared__ float s_den[2][bw::BQ];
    __shared__ int s_gave_up;
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = (int)(blockIdx.x / nqb);
    const int qb = nqb - 1 - (int)(blockIdx.x % nqb);  // a head's longest query block first
    const int b = bh / H, h = bh - b * H;
    const int i0 = qb * bw::BQ;
    const int nkb = (T + BK - 1) / BK;
    const int last = min((i0 + bw::BQ - 1) / BK, nkb - 1);  // the key blocks up to the query block's last position
    const size_t tok_stride = (size_t)H * (D / 2);          // float4 between consecutive tokens of a head
    const size_t head0 = ((size_t)b * T * H + h) * (D / 2);

    if (warp == 8) {
        tc::tmem_alloc(&s_tmem, bw::TMEM_COLS);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        s_gave_up = 0;
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&mb_g[i], 1);
            tc::mbar_init(&mb_s[i], 8);
        }
        for (int i = 0; i < NR; ++i) {
            tc::mbar_init(&mb_kv[i], bw::LOADERS ? bw::NLOAD / 32 : 8);
            tc::mbar_init(&mb_free[i], 1);
        }
        tc::mbar_init(&mb_drain, 1);
        tc::mbar_fence_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    bool ok = true;

    if (warp < 8) {
        // Tensor-memory lane L = 32 (warp mod 4) + lane holds query i0 + L; this
        // thread takes key columns 16 ch .. 16 ch + 15 of each block.
        const int L = (warp & 3) * 32 + lane, ch = warp >> 2;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        if constexpr (bw::ONES) {  // rows 2D .. NB - 1 of every value slot: ones, then zeros
            for (int e = tid; e < NR * (bw::NB - 2 * D) * BK; e += bw::NMATH) {
                const int r = e / ((bw::NB - 2 * D) * BK), f = e % ((bw::NB - 2 * D) * BK);
                const int m = 2 * D + f / BK, jj = f % BK;
                sts(smem + r * bw::SLOT + bw::K_BYTES,
                    (jj >> 2) * bw::V_LBO + (m >> 3) * bw::V_SBO + (m & 7) * 16 + (jj & 3) * 4, m == 2 * D ? 1.f : 0.f);
            }
        }
        {  // Q: floats ch D .. ch D + D - 1 of the query row, TF32-rounded
            uint32_t qv[D];
            const bool in = i0 + L < T;
            const float4* src = q + head0 + (size_t)(i0 + L) * tok_stride + ch * (D / 4);
#pragma unroll
            for (int c = 0; c < D / 4; ++c) {
                const float4 x = in ? __ldg(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
                qv[4 * c] = __float_as_uint(rna_tf32(x.x));
                qv[4 * c + 1] = __float_as_uint(rna_tf32(x.y));
                qv[4 * c + 2] = __float_as_uint(rna_tf32(x.z));
                qv[4 * c + 3] = __float_as_uint(rna_tf32(x.w));
            }
#pragma unroll
            for (int cb = 0; cb < D / 16; ++cb)
                tc::tmem_st16(tmem + lane_base + bw::COL_Q + ch * D + 16 * cb,
                              *reinterpret_cast<const uint32_t(*)[16]>(qv + 16 * cb));
            tc::tmem_wait_st();
        }
        // Math staging (width 32): thread tid reads float4 (tid mod 8) + 8 i of
        // key tid / 8 of each block, so eight lanes read one 128-byte row piece.
        const int j = tid >> 3, c0 = tid & 7;
        const float4* kbase = k + head0 + (size_t)j * tok_stride + c0;
        const float4* vbase = v + head0 + (size_t)j * tok_stride + c0;
        auto load = [&](int kb, float4 (&kr)[IT], float4 (&vr)[IT]) {
            const bool in = kb * BK + j < T;
            const size_t o = (size_t)kb * BK * tok_stride;
#pragma unroll
            for (int i = 0; i < IT; ++i) {
                kr[i] = in ? __ldg(kbase + o + 8 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
                vr[i] = in ? __ldg(vbase + o + 8 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        };
        auto write = [&](int kb, const float4 (&kr)[IT], const float4 (&vr)[IT]) {
            unsigned char* sk = smem + (kb % NR) * bw::SLOT;
            unsigned char* sv = sk + bw::K_BYTES;
#pragma unroll
            for (int i = 0; i < IT; ++i) {
                const int c = c0 + 8 * i;  // float4 c = components 2c, 2c + 1
                const float kx = rna_tf32(kr[i].x), ky = rna_tf32(kr[i].y), kz = rna_tf32(kr[i].z),
                            kw = rna_tf32(kr[i].w);
                const uint32_t ko = c * bw::K_LBO + (j & 7) * 16;
                sts4(sk, ko + (j >> 3) * bw::K_SBO, kx, ky, kz, kw);               // row j: (re, im, re, im)
                sts4(sk, ko + ((BK + j) >> 3) * bw::K_SBO, ky, -kx, kw, -kz);     // row BK + j: (im, -re, ...)
                const uint32_t vo = (j >> 2) * bw::V_LBO + (j & 3) * 4;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = 4 * c + e;
                    const float val = e == 0 ? vr[i].x : e == 1 ? vr[i].y : e == 2 ? vr[i].z : vr[i].w;
                    sts(sv, vo + (m >> 3) * bw::V_SBO + (m & 7) * 16, rna_tf32(val));
                }
            }
            tc::fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive1(&mb_kv[kb % NR]);
        };
        float4 ka[IT], va[IT], kb2[IT], vb2[IT];
        if constexpr (!bw::LOADERS) {
            load(0, ka, va);
            write(0, ka, va);
            if (last >= 1) {
                load(1, ka, va);
                write(1, ka, va);
            }
            if (last >= 2) load(2, ka, va);
            if (last >= 3) load(3, kb2, vb2);
        }
        tc::fence_before_sync();
        __syncthreads();  // Q stored

        float den = 0.f;
        auto block = [&](int kb, float4 (&kr)[IT], float4 (&vr)[IT]) {
            const int g = kb & 1;
            ok = mbar_wait_sleep(&mb_g[g], (uint32_t)((kb >> 1) & 1), kBornWait) && ok;
            tc::fence_after_sync();
            uint32_t re[16], im[16];
            const uint32_t col = tmem + lane_base + bw::COL_G + 64 * g + 16 * ch;
            tc::tmem_ld16(col, re);
            tc::tmem_ld16(col + BK, im);
            tc::tmem_wait_ld();
            const int kq = i0 + L - kb * BK - 16 * ch;  // the last key column this query may see
            // With the row of ones the tensor core reads S (truncated to TF32)
            // for the numerator and the sum alike; without it each S is
            // rounded here and summed in this thread.
            if (kq < 15) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const float gr = __uint_as_float(re[jj]), gi = __uint_as_float(im[jj]);
                    float s = fmaf(gr, gr, gi * gi);
                    if (!bw::ONES) s = rna_tf32(s);
                    s = jj <= kq ? s : 0.f;
                    if (!bw::ONES) den += s;
                    re[jj] = __float_as_uint(s);
                }
            } else {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const float gr = __uint_as_float(re[jj]), gi = __uint_as_float(im[jj]);
                    float s = fmaf(gr, gr, gi * gi);
                    if (!bw::ONES) {
                        s = rna_tf32(s);
                        den += s;
                    }
                    re[jj] = __float_as_uint(s);
                }
            }
            tc::tmem_st16(col, re);
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive1(&mb_s[g]);
            if (!bw::LOADERS && kb + 2 <= last) {
                // Block kb + 2 goes into the slot of block kb + 2 - NR.  With
                // four slots that is block kb - 2, free already: G of block
                // kb, complete, was issued after the value GEMM of block kb - 2
                // had completed.  With three it is block kb - 1, whose value
                // GEMM may still be running.
                if (NR == 3 && kb >= 1)
                    ok = mbar_wait_sleep(&mb_free[(kb - 1) % NR], (uint32_t)(((kb - 1) / NR) & 1), kBornWait) && ok;
                write(kb + 2, kr, vr);
                if (kb + 4 <= last) load(kb + 4, kr, vr);
            }
        };
#pragma unroll 1
        for (int kb = 0; kb <= last; kb += 2) {
            block(kb, ka, va);
            if (kb + 1 <= last) block(kb + 1, kb2, vb2);
        }

        // Epilogue: lane L's ACC columns are psi's row (re, im interleaved) times the score sum.
        ok = mbar_wait_sleep(&mb_free[last % NR], (uint32_t)((last / NR) & 1), kBornWait) && ok;
        tc::fence_after_sync();
        float dsum;
        if (bw::ONES) {
            uint32_t sum4[4];
            tc::tmem_ld4(tmem + lane_base + bw::COL_ACC + 2 * D, sum4);
            tc::tmem_wait_ld();
            dsum = __uint_as_float(sum4[0]);
        } else {
            s_den[ch][L] = den;
            asm volatile("bar.sync 1, 256;" ::: "memory");
            dsum = s_den[0][L] + s_den[1][L];
        }
        uint32_t acc[D];
#pragma unroll
        for (int cb = 0; cb < D / 16; ++cb)
            tc::tmem_ld16(tmem + lane_base + bw::COL_ACC + ch * D + 16 * cb, *reinterpret_cast<uint32_t(*)[16]>(acc + 16 * cb));
        tc::tmem_wait_ld();
        if (i0 + L < T) {
            const float inv = dsum != 0.f ? 1.f / dsum : 0.f;
            float4* out = reinterpret_cast<float4*>(psi + ((size_t)((size_t)b * T + i0 + L) * H + h) * D + ch * (D / 2));
#pragma unroll
            for (int m = 0; m < D / 4; ++m)
                out[m] = make_float4(__uint_as_float(acc[4 * m]) * inv, __uint_as_float(acc[4 * m + 1]) * inv,
                                     __uint_as_float(acc[4 * m + 2]) * inv, __uint_as_float(acc[4 * m + 3]) * inv);
        }
    } else if (warp >= 9) {
        if constexpr (bw::LOADERS) {
            // Loader warps: raw key and value rows by cp.async NRAW blocks ahead
            // into the raw slots; each thread then rounds exactly the pieces it
            // copied to TF32 and stores them into the block's operand slot.
            // Item n = lt + NLOAD i is float4 c = n mod (D/2) of key n / (D/2),
            // so eight lanes read one 128-byte row piece.
            const int lt = tid - (bw::NMATH + 32);
            const uint32_t s0 = tc::smem_u32(smem);
            auto copy_block = [&](int kb) {
                if (kb <= last) {
                    const uint32_t rs = s0 + bw::RAW0 + (kb % NRAW) * bw::RAW;
#pragma unroll
                    for (int i = 0; i < bw::LIT; ++i) {
                        const int n = lt + bw::NLOAD * i, j = n / (D / 2), c = n % (D / 2);
                        const bool in = kb * BK + j < T;
                        // past the end: read nothing (the head's first token as the address), write zeros
                        const size_t o = in ? (size_t)(kb * BK + j) * tok_stride + c : (size_t)c;
                        cp_async16(rs + n * 16, k + head0 + o, in ? 16u : 0u);
                        cp_async16(rs + bw::RAW_HALF + n * 16, v + head0 + o, in ? 16u : 0u);
                    }
                }
                cp_async_commit();  // one group per block, empty past the last
            };
            for (int kb = 0; kb < NRAW; ++kb) copy_block(kb);
            __syncthreads();  // Q and the constant rows stored (the math warps' barrier)
#pragma unroll 1
            for (int kb = 0; kb <= last; ++kb) {
                cp_async_wait<NRAW - 1>();  // this thread's copies of block kb have landed
                // Operand slot kb mod NR last held block kb - NR: its value GEMM must be done.
                if (kb >= NR)
                    ok = mbar_wait_sleep(&mb_free[(kb - NR) % NR], (uint32_t)(((kb - NR) / NR) & 1), kBornWait) && ok;
                const unsigned char* rs = smem + bw::RAW0 + (kb % NRAW) * bw::RAW;
                unsigned char* sk = smem + (kb % NR) * bw::SLOT;
                unsigned char* sv = sk + bw::K_BYTES;
#pragma unroll
                for (int i = 0; i < bw::LIT; ++i) {
                    const int n = lt + bw::NLOAD * i, j = n / (D / 2), c = n % (D / 2);
                    const float4 kr = lds4(rs, n * 16), vr = lds4(rs + bw::RAW_HALF, n * 16);
                    const float kx = rna_tf32(kr.x), ky = rna_tf32(kr.y), kz = rna_tf32(kr.z), kw = rna_tf32(kr.w);
                    const uint32_t ko = c * bw::K_LBO + (j & 7) * 16;
                    sts4(sk, ko + (j >> 3) * bw::K_SBO, kx, ky, kz, kw);            // row j: (re, im, re, im)
                    sts4(sk, ko + ((BK + j) >> 3) * bw::K_SBO, ky, -kx, kw, -kz);  // row BK + j: (im, -re, ...)
                    const uint32_t vo = (j >> 2) * bw::V_LBO + (j & 3) * 4;
                    const float vv[4] = {vr.x, vr.y, vr.z, vr.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int m = 4 * c + e;
                        sts(sv, vo + (m >> 3) * bw::V_SBO + (m & 7) * 16, rna_tf32(vv[e]));
                    }
                }
                tc::fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive1(&mb_kv[kb % NR]);
                copy_block(kb + NRAW);  // into the raw slot just read (its values are in registers already)
            }
            cp_async_wait<0>();
        }
    } else {
        __syncthreads();  // Q stored
        {  // the whole warp runs the loop; one elected lane issues
            tc::fence_after_sync();
            const uint32_t ID_G = tc::idesc_tf32(128, 2 * BK), ID_V = tc::idesc_tf32(128, bw::NB);
            constexpr uint64_t K_STEP = (2 * bw::K_LBO) >> 4, V_STEP = (2 * bw::V_LBO) >> 4;
            const uint32_t s0 = tc::smem_u32(smem);
            auto issue_g = [&](int kb) {
                const uint64_t bk = tc::make_desc(s0 + (kb % NR) * bw::SLOT, bw::K_LBO, bw::K_SBO);
                const uint32_t d = tmem + bw::COL_G + 64 * (kb & 1);
#pragma unroll
                for (int ks = 0; ks < bw::K2 / 8; ++ks)
                    mma_ts_warp(d, tmem + bw::COL_Q + 8 * ks, bk + ks * K_STEP, ID_G, ks > 0 ? 1u : 0u);
                commit_warp(&mb_g[kb & 1]);
            };
            auto issue_v = [&](int kb) {
                const uint64_t bv = tc::make_desc(s0 + (kb % NR) * bw::SLOT + bw::K_BYTES, bw::V_LBO, bw::V_SBO);
                const uint32_t a = tmem + bw::COL_G + 64 * (kb & 1);
#pragma unroll
                for (int ks = 0; ks < BK / 8; ++ks)
                    mma_ts_warp(tmem + bw::COL_ACC, a + 8 * ks, bv + ks * V_STEP, ID_V, (kb > 0 || ks > 0) ? 1u : 0u);
                commit_warp(&mb_free[kb % NR]);
            };
            ok = __all_sync(0xffffffffu, mbar_wait_sleep(&mb_kv[0], 0u, kBornWait)) && ok;
            tc::fence_after_sync();
            issue_g(0);
            if (last >= 1) {
                ok = __all_sync(0xffffffffu, mbar_wait_sleep(&mb_kv[1], 0u, kBornWait)) && ok;
                tc::fence_after_sync();
                issue_g(1);
            }
#pragma unroll 1
            for (int kb = 0; kb <= last; ++kb) {
                ok = __all_sync(0xffffffffu, mbar_wait_sleep(&mb_s[kb & 1], (uint32_t)((kb >> 1) & 1), kBornWait)) && ok;
                tc::fence_after_sync();
                issue_v(kb);
                if (kb + 2 <= last) {
                    ok = __all_sync(0xffffffffu, mbar_wait_sleep(&mb_kv[(kb + 2) % NR], (uint32_t)(((kb + 2) / NR) & 1), kBornWait)) && ok;
                    ok = __all_sync(0xffffffffu, mbar_wait_sleep(&mb_free[kb % NR], (uint32_t)((kb / NR) & 1), kBornWait)) && ok;
                    tc::fence_after_sync();
                    issue_g(kb + 2);
                }
            }
        }
    }
    if (!ok) s_gave_up = 1;  // a wait gave up
    __syncthreads();
    if (s_gave_up && warp == 8) {  // the issuing warp: one more commit from its elected lane, waited for
        if (lane == 0 && status) atomicOr(status, kStatusBornMma);
        commit_warp(&mb_drain);
        mbar_wait_sleep(&mb_drain, 0u, kBornWait);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 8) tc::tmem_dealloc(tmem, bw::TMEM_COLS);
}

template <int D>
static cudaError_t launch_born_ws(const BornArgs& a, cudaStream_t st) {
    using bw = BornW<D>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<bool> attr_set[128];
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(born_kernel_ws<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bw::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    const int64_t BH = a.Bz * a.H, nqb = (a.T + bw::BQ - 1) / bw::BQ;
    born_kernel_ws<D><<<(unsigned)(BH * nqb), bw::NT, bw::SMEM, st>>>(
        reinterpret_cast<const float4*>(a.q), reinterpret_cast<const float4*>(a.k), reinterpret_cast<const float4*>(a.v),
        a.psi, (int)a.T, (int)a.H, (int)nqb, status_word());
    return cudaGetLastError();
}

}  // namespace

bool born_supported(int64_t D) { return D == 16 || D == 32; }

cudaError_t launch_born(const BornArgs& a, cudaStream_t st) {
    return a.D == 16 ? launch_born_ws<16>(a, st) : launch_born_ws<32>(a, st);
}

}  // namespace cssd
