// softmax_tile.cuh -- the per-row online-softmax step on one 128-key tile,
// shared by every fused attention kernel.
//
// One thread owns one query row (= one TMEM lane).  For key tile j it reads
// the fp32 scores S from TMEM, forms log2-domain logits t (scale * log2 e is
// folded into the exponent's multiply-add for the plain score, or applied
// with the score_mod), masks them, takes the row max, lazily rescales the
// running output O and sums when the max has grown by more than
// kRescaleThreshold (2^8), and writes P = 2^(t - m) as bf16 into TMEM for the
// P V product.  This is the running-max / running-sum recurrence of the
// online softmax (Flashlight gist.science summary, "Methodology" item 3; talk
// notes, "Compiler design 2"); keeping a stale reference max m is exact in
// real arithmetic because every term and both sums carry the same factor.
//
// Two sums are kept: `l` adds the exact P (it gives the log-sum-exp), and
// `l_round` adds the bf16-rounded P the tensor core actually multiplies V
// by (it normalises O, so O / l_round is an exact convex combination of V
// rows with those weights).
#pragma once

#include "common.cuh"

namespace fl {

constexpr float kRescaleThreshold = 8.f; // log2 units

struct RowState {
    float m_ref;   // reference max (log2 units) every P of this row is relative to
    float l;       // sum of the exact P
    float l_round; // sum of the bf16-rounded P
};

struct ScoreMod {
    float qk_log2;     // scale * log2(e) (> 0)
    float alibi_c;     // slope_h * log2(e)                 (ALiBi)
    float softcap_in;  // 2 * scale * log2(e) / cap           (softcap)
    float softcap_out; // cap * log2(e)                       (softcap)
    float scale;       // scale                               (expression)
    float b, h;        // batch index and query head          (expression)
};

// Loads the N scores (N a multiple of 16) of this thread's row from TMEM
// columns [tS, tS + N).
template <int N = BN>
__device__ __forceinline__ void load_scores(uint32_t tS, float (&x)[N])
{
    static_assert(N % 16 == 0, "tile width must be a multiple of 16");
    uint32_t raw[N];
#pragma unroll
    for (int c = 0; c < N / 32; ++c)
        ptx::tmem_ld32(tS + 32 * c, raw + 32 * c);
    if constexpr (N % 32 != 0)
        ptx::tmem_ld16(tS + 32 * (N / 32), raw + 32 * (N / 32));
    ptx::tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < N / 16; ++c)
        ptx::reg_fence<16>(raw + 16 * c);
#pragma unroll
    for (int e = 0; e < N; ++e)
        x[e] = __uint_as_float(raw[e]);
}

// Scores -> logits for query row i and keys j0 .. j0 + 127.  For MOD_NONE the
// scores stay unscaled (the scale is applied in the exponent); the other
// score_mods produce log2-domain logits.
template <int MOD, int N = BN>
__device__ __forceinline__ void apply_score_mod(float (&x)[N], const ScoreMod &sm, int i, int j0)
{
    // Both score_mods work on pairs of keys with the packed fp32 instructions
    // (one issue for two scores): fewer instructions in the exponential phase,
    // which one warp per sub-partition runs.
    if constexpr (MOD == MOD_ALIBI) {
        // z - slope |i - j|, in log2 units; j - i of keys 2e and 2e + 1 stepped
        // by 2 (exact in fp32: |j - i| < 2^24)
        const float nc = -sm.alibi_c;
        float dA = static_cast<float>(j0 - i), dB = dA + 1.f;
#pragma unroll
        for (int e = 0; e < N / 2; ++e) {
            ptx::fma2(x[2 * e], x[2 * e + 1], x[2 * e], x[2 * e + 1], sm.qk_log2, sm.qk_log2, nc * fabsf(dA),
                      nc * fabsf(dB));
            ptx::add2(dA, dB, 2.f, 2.f);
        }
    } else if constexpr (MOD == MOD_SOFTCAP) {
        // cap * tanh(z / cap) with tanh(u) = 1 - 2 / (1 + e^(2u)), in log2 units:
        // out (1 - 2 r) as out + (-2 out) r, r = 1 / (1 + 2^(z in))
        const float m2o = -2.f * sm.softcap_out;
#pragma unroll
        for (int e = 0; e < N / 2; ++e) {
            float a0, a1;
            ptx::fma2(a0, a1, x[2 * e], x[2 * e + 1], sm.softcap_in, sm.softcap_in, 0.f, 0.f);
            float d0 = ptx::ex2(a0), d1 = ptx::ex2(a1);
            ptx::add2(d0, d1, 1.f, 1.f);
            const float r0 = ptx::rcp_approx(d0), r1 = ptx::rcp_approx(d1);
            ptx::fma2(x[2 * e], x[2 * e + 1], r0, r1, m2o, m2o, sm.softcap_out, sm.softcap_out);
        }
    } else if constexpr (MOD == MOD_EXPR) {
#ifdef FL_SCORE_EXPR
        // the run-time expression fl_score_expr(score, b, h, q_idx, kv_idx)
        // (defined ahead of this file by the runtime compilation), in log2 units
        // (indices below 2^24 are exact in fp32; j0 + e as one add per score)
        const float fi = static_cast<float>(i), fj0 = static_cast<float>(j0);
#pragma unroll
        for (int e = 0; e < N; ++e)
            x[e] = kLog2e * fl_score_expr(x[e] * sm.scale, sm.b, sm.h, fi, fj0 + static_cast<float>(e));
#endif
    }
}

// Keys outside [row_lo, row_hi) -> -inf (only on tiles that hold masked pairs).
template <int N = BN>
__device__ __forceinline__ void apply_row_mask(float (&x)[N], int j0, int row_lo, int row_hi)
{
    const int a = row_lo - j0, z = row_hi - j0;
#pragma unroll
    for (int e = 0; e < N; ++e)
        if (e < a || e >= z)
            x[e] = kNegInf;
}

// One tile's online-softmax step, in two parts so the caller can overlap the
// exponentials with the P V product of the previous tile:
//   softmax_compute_p: max, rescale decision, P (packed bf16 in registers)
//                      and both sums; O is not touched;
//   rescale_o + store_p: once the previous P V has completed.
// Returns the O rescale factor (1 when no rescale is needed for this warp).
template <int N = BN>
__device__ __forceinline__ float softmax_compute_p(float (&x)[N], float c, RowState &st,
                                                   bool first, uint32_t (&pk)[N / 2],
                                                   bool &rescale)
{
    float mc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        mc[q] = fmaxf(x[2 * q], x[2 * q + 1]);
#pragma unroll
    for (int e = 8; e < N; e += 8) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            mc[q] = ptx::max3(mc[q], x[e + 2 * q], x[e + 2 * q + 1]);
    }
    const float mx = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3])) * c; // c > 0
    float alpha = 1.f;
    rescale = false;
    if (first) {
        st.m_ref = mx;
    } else {
        const bool need = mx > st.m_ref + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
            const float m_new = fmaxf(st.m_ref, mx);
            alpha = (m_new == kNegInf) ? 1.f : ptx::ex2(st.m_ref - m_new);
            st.l *= alpha;
            st.l_round *= alpha;
            st.m_ref = m_new;
            rescale = true;
        }
    }
    const float nmu = (st.m_ref == kNegInf) ? 0.f : -st.m_ref;
    float le[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float lr[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < N / 2; ++e) {
        float a0, a1;
        ptx::fma2(a0, a1, x[2 * e], x[2 * e + 1], c, c, nmu, nmu);
        const float p0 = ptx::ex2(a0);
        const float p1 = ptx::ex2(a1);
        pk[e] = ptx::pack_bf16(p0, p1);
        const int q = 2 * (e & 3);
        ptx::add2(le[q], le[q + 1], p0, p1);
        ptx::add_bf16x2_to_f32(lr[q], lr[q + 1], pk[e]); // the rounded P, widened exactly
    }
    st.l += ((le[0] + le[1]) + (le[2] + le[3])) + ((le[4] + le[5]) + (le[6] + le[7]));
    st.l_round += ((lr[0] + lr[1]) + (lr[2] + lr[3])) + ((lr[4] + lr[5]) + (lr[6] + lr[7]));
    return alpha;
}

// As softmax_compute_p, for kernels whose P V product also produces the sum
// of the rounded P (an extra output column multiplied by ones): only the
// exact sum `l` is kept here; st.l_round is left untouched.
template <int N = BN>
__device__ __forceinline__ float softmax_compute_p_exact_sum(float (&x)[N], float c, RowState &st,
                                                             bool first, uint32_t (&pk)[N / 2],
                                                             bool &rescale)
{
    float mc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        mc[q] = fmaxf(x[2 * q], x[2 * q + 1]);
#pragma unroll
    for (int e = 8; e < N; e += 8) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            mc[q] = ptx::max3(mc[q], x[e + 2 * q], x[e + 2 * q + 1]);
    }
    const float mx = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3])) * c; // c > 0
    float alpha = 1.f;
    rescale = false;
    if (first) {
        st.m_ref = mx;
    } else {
        const bool need = mx > st.m_ref + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
            const float m_new = fmaxf(st.m_ref, mx);
            alpha = (m_new == kNegInf) ? 1.f : ptx::ex2(st.m_ref - m_new);
            st.l *= alpha;
            st.m_ref = m_new;
            rescale = true;
        }
    }
    const float nmu = (st.m_ref == kNegInf) ? 0.f : -st.m_ref;
    float le[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < N / 2; ++e) {
        float a0, a1;
        ptx::fma2(a0, a1, x[2 * e], x[2 * e + 1], c, c, nmu, nmu);
        const float p0 = ptx::ex2(a0);
        const float p1 = ptx::ex2(a1);
        pk[e] = ptx::pack_bf16(p0, p1);
        const int q = 2 * (e & 3);
        ptx::add2(le[q], le[q + 1], p0, p1);
    }
    st.l += ((le[0] + le[1]) + (le[2] + le[3])) + ((le[4] + le[5]) + (le[6] + le[7]));
    return alpha;
}

// O *= alpha over DV fp32 columns at tO (this thread's row).
template <int DV>
__device__ __forceinline__ void rescale_o(uint32_t tO, float alpha)
{
#pragma unroll 1
    for (int k = 0; k < DV / 16; ++k) {
        uint32_t o[16];
        ptx::tmem_ld16(tO + 16 * k, o);
        ptx::tmem_wait_ld();
        ptx::reg_fence<16>(o);
#pragma unroll
        for (int e = 0; e < 16; ++e)
            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        ptx::tmem_st16(tO + 16 * k, o);
    }
}

// P (packed bf16, N / 2 columns) -> TMEM at tP; completes the stores.
template <int N = BN>
__device__ __forceinline__ void store_p(uint32_t tP, const uint32_t (&pk)[N / 2])
{
#pragma unroll
    for (int k = 0; k < N / 32; ++k)
        ptx::tmem_st16(tP + 16 * k, pk + 16 * k);
    if constexpr (N % 32 != 0)
        ptx::tmem_st8(tP + 16 * (N / 32), pk + 16 * (N / 32));
    ptx::tmem_wait_st();
}

// Natural-log LSE of a finished row (from the exact sum).
__device__ __forceinline__ float row_lse(const RowState &st)
{
    return st.l > 0.f ? (st.m_ref + log2f(st.l)) * kLn2 : kNegInf;
}

// 1 / (the normaliser of O), 0 for a row with no allowed key.
__device__ __forceinline__ float row_inv_norm(const RowState &st)
{
    return st.l_round > 0.f ? ptx::rcp_approx(st.l_round) : 0.f; // l_round >= 1: the row max has P >= 1
}

} // namespace fl
