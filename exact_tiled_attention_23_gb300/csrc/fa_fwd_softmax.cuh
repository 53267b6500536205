// fa_fwd_softmax.cuh -- the online-softmax step of one query row over one key
// block of 128 (or 64) scores, shared by the tensor-core forward kernels.
//
// One thread owns one query row (one TMEM lane), or one half of a row's keys.
// Per key block it has its kCols raw scores S = q.k in registers (fp32 bits,
// masked entries already -inf) and turns them into P = 2^(S*scale*log2e -
// m_ref), stored as 16-bit pairs in kCols/2 TMEM columns (over the first
// columns of the score tile, or in columns of their own), while keeping the
// running sum l against the same reference m_ref.  This is the
// recurrence of "vectorized-flash-attention-kernel", Core algorithm step 3,
// in base 2.
//
// Two running sums are kept.  l sums the fp32 p and gives the LSE.  l_o sums
// the same p after rounding to the 16-bit type, i.e. exactly the weights the
// tensor core multiplies V by, and normalises O: O = sum(P~ V) / sum(P~) is a
// convex combination of V rows whatever the rounding, so a dominant weight's
// rounding error cancels.  With the lazy reference below the dominant p is
// not 1, and normalising by the fp32 sum instead leaves its relative rounding
// error (up to 2^-8 for bf16) on O: 2.6e-2 on |O| ~ 4 in near one-hot rows.
//
// The reference max is lazy.  The first key block sets it from the row max.
// Later blocks reuse it without scanning for their max as long as the block's
// sum of p stays within a limit (2^64 for bf16 P, 2^15 for fp16 P), which
// bounds every p, so l, P and O stay far from overflow.  A block that exceeds
// the limit, or gives inf/NaN, scans its max, raises m_ref, rescales O and l
// by 2^(m_old - m_new) and recomputes P.  l and O always share m_ref, so the
// result is exact in real arithmetic.
#pragma once

#include "fa_tc_common.cuh"
#include "sm103_ptx.cuh"

#include <cmath>
#include <cstdint>

namespace fa {

// Largest block sum of p kept without a max scan: 2^64.  It bounds every p
// by 2^64, so l <= N * 2^64 and |O| <= N * 2^64 * max|V| stay far below the
// fp32/bf16 limit of ~2^128 for any N < 2^31 and max|V| < 2^30.
constexpr float kLazyLimit = 18446744073709551616.f;
// With fp16 operands P must also fit fp16 (max 65504): every p <= 2^15.
constexpr float kLazyLimitF16 = 32768.f;

// D: number of fp32 O columns in TMEM for this row; kF16: P is fp16 (else
// bf16); kCols: scores per key block (128, or 64 when two threads share a row
// and each keeps its own m_ref, l, l_o and O).
template <int D, bool kF16, int kCols = 128>
struct OnlineRow {
    static_assert(kCols == 64 || kCols == 128, "scores per block");
    static constexpr int kC = kCols / 32;      // 32-score chunks
    float m_ref = -INFINITY;   // reference max of scale*log2e*S: a lower bound of the running max
    float l = 0.f;             // running sum of p against m_ref (fp32 p): the LSE
    float l_o = 0.f;           // running sum of the 16-bit rounded P: O's normaliser

    // Raise m_ref to the block's max; rescale l (and O in TMEM at tO when it
    // already holds earlier blocks) by 2^(m_old - m_new).  before_o_touch()
    // runs, warp-uniformly, just before O is read.
    template <typename Hook>
    __device__ __forceinline__ void raise(const uint32_t (&s)[kC][32], float sl2, bool o_live, uint32_t tO,
                                          Hook &before_o_touch)
    {
        // Eight running maxima: scores 0..7, then 16 per step over
        // 8..kCols-9 (two per 3-input max), then the last 8.
        float mx8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = u2f(s[0][a]);
#pragma unroll
        for (int k = 8; k < kCols - 8; k += 16)
#pragma unroll
            for (int a = 0; a < 8; ++a)
                mx8[a] = ptx::max3(mx8[a], u2f(s[(k + 2 * a) / 32][(k + 2 * a) % 32]),
                                   u2f(s[(k + 2 * a + 1) / 32][(k + 2 * a + 1) % 32]));
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = fmaxf(mx8[a], u2f(s[kC - 1][24 + a]));
        const float mx = fmaxf(ptx::max3(mx8[0], mx8[1], mx8[2]),
                               fmaxf(ptx::max3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float m_new = fmaxf(m_ref, mx * sl2);
        const float alpha = (m_ref == -INFINITY) ? 0.f : ptx::ex2_approx(m_ref - m_new);
        if (o_live && __any_sync(0xffffffffu, alpha != 1.f)) {
            before_o_touch();
            const uint64_t a2 = ptx::pack2(alpha, alpha);
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {       // 16 columns at a time: few registers beside S
                uint32_t o[16];
                ptx::tmem_ld16(tO + c * 16, o);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    float lo, hi;
                    ptx::unpack2(ptx::mul2(ptx::pack2(u2f(o[2 * t]), u2f(o[2 * t + 1])), a2), lo, hi);
                    o[2 * t] = f2u(lo);
                    o[2 * t + 1] = f2u(hi);
                }
                ptx::tmem_st16(tO + c * 16, o);
            }
        }
        l *= alpha;
        l_o *= alpha;
        m_ref = m_new;
    }

    // p = 2^(S*scale*log2e - m_ref): packed FMA, MUFU ex2, packed sums; P
    // goes to the 64 columns at tP as 16-bit pairs.  Returns sum p in `sum`
    // and the sum of the stored (rounded) P in `sum_o`.  pre_store() runs
    // (warp-uniformly) once the first kEarly x 32 scores are done, before the
    // first P store: a kernel whose P columns may still be read by the
    // previous product waits for it there, with that much of the pass done.
    template <int kEarly, typename PreStore>
    __device__ __forceinline__ void exp_pass(const uint32_t (&s)[kC][32], float sl2, uint32_t tP, float &sum,
                                             float &sum_o, PreStore &pre_store) const
    {
        static_assert(kEarly >= 1 && kEarly <= kC, "chunks before the first P store");
        const float mref_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        const uint64_t t2 = ptx::pack2(sl2, sl2);
        const uint64_t nm2 = ptx::pack2(-mref_use, -mref_use);
        uint64_t acc2[4], rnd2[2];
#pragma unroll
        for (int a = 0; a < 4; ++a) acc2[a] = 0ull;
#pragma unroll
        for (int a = 0; a < 2; ++a) rnd2[a] = 0ull;
        uint32_t pk[kC][16];
#pragma unroll
        for (int c = 0; c < kC; ++c) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                float y0, y1;
                ptx::unpack2(ptx::fma2(ptx::pack2(u2f(s[c][2 * t]), u2f(s[c][2 * t + 1])), t2, nm2), y0, y1);
                const float p0 = ptx::ex2_approx(y0);
                const float p1 = ptx::ex2_approx(y1);
                acc2[t & 3] = ptx::add2(acc2[t & 3], ptx::pack2(p0, p1));
                pk[c][t] = ptx::pack16x2<kF16>(p0, p1);
                rnd2[t & 1] = ptx::add2(rnd2[t & 1], ptx::widen16x2<kF16>(pk[c][t]));
            }
            if (c + 1 == kEarly) {
                pre_store();
#pragma unroll
                for (int e = 0; e <= c; ++e) ptx::tmem_st16(tP + e * 16, pk[e]);
            } else if (c >= kEarly) {
                ptx::tmem_st16(tP + c * 16, pk[c]);
            }
        }
        float a0, a1, b0, b1, c0, c1, d0, d1;
        ptx::unpack2(acc2[0], a0, a1);
        ptx::unpack2(acc2[1], b0, b1);
        ptx::unpack2(acc2[2], c0, c1);
        ptx::unpack2(acc2[3], d0, d1);
        sum = ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
        ptx::unpack2(rnd2[0], a0, a1);
        ptx::unpack2(rnd2[1], b0, b1);
        sum_o = (a0 + a1) + (b0 + b1);
    }

    // One key block; P goes to tP.  o_live: O at tO holds earlier blocks.
    // before_o_touch() runs (warp-uniformly) before any access to O, for
    // kernels whose O may still be written by an MMA at that point;
    // before_p_store() before the first store to tP, for kernels whose P
    // columns may still be read by one (both may run more than once).  On
    // return every P store has landed in TMEM.
    // kEarly: chunks of 32 scores exponentiated before before_p_store() and
    // the first P store.
    template <int kEarly = 1, typename Hook, typename PreStore>
    __device__ __forceinline__ void block(const uint32_t (&s)[kC][32], float sl2, bool o_live, uint32_t tP,
                                          uint32_t tO, Hook &&before_o_touch, PreStore &&before_p_store)
    {
        if (__any_sync(0xffffffffu, m_ref == -INFINITY)) raise(s, sl2, o_live, tO, before_o_touch);
        float sum, sum_o;
        exp_pass<kEarly>(s, sl2, tP, sum, sum_o, before_p_store);
        if (__any_sync(0xffffffffu, !(sum <= (kF16 ? kLazyLimitF16 : kLazyLimit)))) {
            raise(s, sl2, o_live, tO, before_o_touch);
            ptx::tmem_wait_st();      // the first pass's P stores land before the new ones
            exp_pass<kEarly>(s, sl2, tP, sum, sum_o, before_p_store);
        }
        ptx::tmem_wait_st();
        l += sum;
        l_o += sum_o;
    }

    template <typename Hook>
    __device__ __forceinline__ void block(const uint32_t (&s)[kC][32], float sl2, bool o_live, uint32_t tP,
                                          uint32_t tO, Hook &&before_o_touch)
    {
        block<1>(s, sl2, o_live, tP, tO, before_o_touch, [] {});
    }
};

}  // namespace fa
