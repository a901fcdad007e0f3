// bwd_standard.cu -- attention backward for the standard kind (MHA / GQA,
// D = Dv = 64, every mask of the forward): dQ, dK, dV from Q, K, V, the forward's O
// and natural-log LSE, and dO.  The pages name training (the backward pass)
// as the next step for the fused kernels (gist.science summary, "Limitations
// and future work"); the gradients are those of
//     O = softmax(scale Q K^T + mask) V:
//     P   = exp(scale q_i k_j - LSE_i)              (recomputed, never stored)
//     dV  = P^T dO
//     dP  = dO V^T
//     dS  = P * (dP - D_i),  D_i = sum_d dO_id O_id   (= sum_j P_ij dP_ij)
//     dQ  = scale dS K,      dK = scale dS^T Q
// with GQA heads summed into their shared K/V head.
//
// Two launches, no atomics (every output element has one writer):
//   bwd_prep_kernel  per query row: D_i, LSE_i * log2 e and the row's allowed
//                    key interval [lo_i, hi_i) into the workspace (padded
//                    rows get LSE +inf, so their P is 0, and the empty
//                    interval [S, S));
//   bwd_fused_kernel one CTA per tile, of two kinds in one grid:
//     dK/dV tiles (bwd_dkdv_body), one per (128-key tile, KV head, batch):
//                    dK and dV accumulate in TMEM over every 64-row query
//                    tile of every query head of the group whose rows allow
//                    a key of the tile;
//     dQ tiles (bwd_dq_body), one per (128-row query tile, query head,
//                    batch): dQ accumulates in TMEM over the 64-key tiles.
// Both tile kinds run on the tcgen05 tensor cores with the same layout of
// roles: a TMA producer warp, one MMA-issuing warp per product chain (an MMA
// returns to its thread only when the tensor core accepts it, so separate
// issuers let independent chains interleave), and two warpgroups of one
// thread per TMEM lane taking alternate tiles for the elementwise step, which
// writes bf16 operands back into TMEM for the next products.  Recomputing S
// and dP in the dQ kernel costs two more of the seven products than an atomic
// dQ accumulation would, and buys determinism and no dQ workspace.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace fl {
namespace {

constexpr uint32_t kTileBytes = kBwdBlock * 64 * 2; // one 64-row tile, 8 KB

__device__ uint32_t g_lib_error_word;

// Query rows [qa, qb) that allow at least one key of [k0, k1) (k0 < k1 <= S).
// Row i allows [lo_i, hi_i) with both bounds non-decreasing in i, so the rows
// are those with hi_i > k0 and lo_i < k1: from the first row whose interval
// reaches k0 to the first row whose interval starts at or after k1.
__device__ __forceinline__ void key_block_query_range(const MaskSpec &m, int b, int k0, int k1, int &qa, int &qb)
{
    qa = 0;
    qb = m.S;
    switch (m.kind) {
    case MASK_NONE:
        break;
    case MASK_CAUSAL:
        qa = k0;
        break;
    case MASK_WINDOW:
        qa = k0;
        qb = min(m.S, k1 - 1 + m.window);
        break;
    case MASK_PREFIX:
        qa = k0 < m.prefix ? 0 : k0;
        break;
    default: { // MASK_DOC: up to the first document start at or after k1
        qa = k0;
        const int32_t *st = m.doc + static_cast<int64_t>(b) * m.doc_stride;
        for (int t = 0; t < m.doc_stride; ++t) {
            const int s0 = __ldg(st + t);
            if (s0 >= k1) {
                qb = min(qb, s0);
                break;
            }
        }
        break;
    }
    }
}

// The score_mod in the backward: the logit (log2 units) of raw score x = q.k
// for query i and key j, and the chain factor dz/du turning dL/dz into dL/du
// (u = scale x): 1 for none and ALiBi (an additive bias), 1 - tanh^2(u / cap)
// for softcap.  tanh(v) = 1 - 2 / (1 + e^(2v)) as in the forward.
struct ModCtx {
    float sl2;     // scale log2 e
    float alibi_c; // slope_h log2 e
    float cap_in;  // 2 scale log2 e / cap
    float cap_out; // cap log2 e
    float scale;   // scale                      (expression)
    float fb, fh;  // batch index and query head (expression)
};

template <int MOD>
__device__ __forceinline__ float mod_logit2(const ModCtx &m, float x, int i, int j, float &chain)
{
    if constexpr (MOD == MOD_SOFTCAP) {
        const float th = 1.f - 2.f * ptx::rcp_approx(1.f + ptx::ex2(x * m.cap_in));
        chain = 1.f - th * th;
        return m.cap_out * th;
    } else if constexpr (MOD == MOD_ALIBI) {
        chain = 1.f;
        return fmaf(x, m.sl2, -m.alibi_c * fabsf(static_cast<float>(i - j)));
    } else if constexpr (MOD == MOD_EXPR) {
#ifdef FL_SCORE_EXPR
        // the run-time expression and its derivative with respect to the
        // score (defined ahead of this file by the runtime compilation)
        const float u = x * m.scale, fi = static_cast<float>(i), fj = static_cast<float>(j);
        chain = fl_score_expr_du(u, m.fb, m.fh, fi, fj);
        return kLog2e * fl_score_expr(u, m.fb, m.fh, fi, fj);
#else
        chain = 1.f;
        return 0.f;
#endif
    } else {
        chain = 1.f;
        return x * m.sl2;
    }
}

__device__ __forceinline__ ModCtx mod_ctx(const BwdParams &p, int b, int h)
{
    ModCtx m;
    m.scale = p.scale;
    m.fb = static_cast<float>(b);
    m.fh = static_cast<float>(h);
    m.sl2 = p.scale * kLog2e;
    const float slope = p.alibi_slopes ? __ldg(p.alibi_slopes + h) : exp2f(p.alibi_exp_coef * static_cast<float>(h + 1));
    m.alibi_c = slope * kLog2e;
    m.cap_in = p.softcap > 0.f ? 2.f * p.scale * kLog2e / p.softcap : 0.f;
    m.cap_out = p.softcap * kLog2e;
    return m;
}

// The exponent arguments (logit - LSE, log2 units) and chain factors of a pair
// of scores x0, x1 with the packed fp32 instructions (one issue for two
// scores: the elementwise step of both tile kinds is issue-bound, and this
// form cut its instructions enough to take the plain-score backward from 448
// to 534 TFLOP/s at S = 2048); dA, dB: i - j of the two pairs (ALiBi; exact in
// fp32), nl0, nl1: -LSE log2 e of their rows.  Run-time expressions keep the
// per-score mod_logit2 above.
template <int MOD>
__device__ __forceinline__ void mod_args2(const ModCtx &m, float x0, float x1, float dA, float dB, float nl0,
                                          float nl1, float &a0, float &a1, float &ch0, float &ch1)
{
    ch0 = ch1 = 1.f;
    if constexpr (MOD == MOD_SOFTCAP) {
        float g0, g1, t0, t1;
        ptx::fma2(g0, g1, x0, x1, m.cap_in, m.cap_in, 0.f, 0.f);
        float e0 = ptx::ex2(g0), e1 = ptx::ex2(g1);
        ptx::add2(e0, e1, 1.f, 1.f);
        const float r0 = ptx::rcp_approx(e0), r1 = ptx::rcp_approx(e1);
        ptx::fma2(t0, t1, r0, r1, -2.f, -2.f, 1.f, 1.f);       // tanh
        ptx::fma2(a0, a1, t0, t1, m.cap_out, m.cap_out, nl0, nl1);
        ptx::fma2(ch0, ch1, -t0, -t1, t0, t1, 1.f, 1.f);      // 1 - tanh^2
    } else if constexpr (MOD == MOD_ALIBI) {
        const float nc = -m.alibi_c;
        ptx::fma2(a0, a1, x0, x1, m.sl2, m.sl2, fmaf(nc, fabsf(dA), nl0), fmaf(nc, fabsf(dB), nl1));
    } else {
        ptx::fma2(a0, a1, x0, x1, m.sl2, m.sl2, nl0, nl1);
    }
}

// ---------------------------------------------------------------- prep

__global__ void __launch_bounds__(128) bwd_prep_kernel(const BwdParams p)
{
    // one thread per (b, h, row of the padded length)
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.S_pad;
    if (idx >= rows)
        return;
    const int i = static_cast<int>(idx % p.S_pad);
    const int64_t bh = idx / p.S_pad;
    const int h = static_cast<int>(bh % p.Hq), b = static_cast<int>(bh / p.Hq);
    // padded rows: P = 0 and the empty key interval [S, S), which keeps both
    // interval bounds non-decreasing over the rows (tile tests rely on it)
    BwdRowStat st{__int_as_float(0x7f800000), 0.f, p.S, p.S};
    if (i < p.S) {
        const uint4 *o4 = reinterpret_cast<const uint4 *>(p.o + b * p.o_sb + i * p.o_ss + h * p.o_sh);
        const uint4 *d4 = reinterpret_cast<const uint4 *>(p.dout + b * p.do_sb + i * p.do_ss + h * p.do_sh);
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 ow = o4[c], dw = d4[c];
            const uint32_t ov[4] = {ow.x, ow.y, ow.z, ow.w}, dv[4] = {dw.x, dw.y, dw.z, dw.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc = fmaf(__uint_as_float(ov[q] << 16), __uint_as_float(dv[q] << 16), acc);
                acc = fmaf(__uint_as_float(ov[q] & 0xFFFF0000u), __uint_as_float(dv[q] & 0xFFFF0000u), acc);
            }
        }
        const float lse = p.lse[b * p.l_sb + h * p.l_sh + i];
        // a row with no allowed key (LSE = -inf) has P = 0 everywhere
        st.lse2 = lse == kNegInf ? __int_as_float(0x7f800000) : lse * kLog2e;
        st.d = acc;
        row_interval(p.mask, b, i, st.lo, st.hi);
    }
    p.ws_stats[idx] = st;
}

// ---------------------------------------------------------------- dQ (tcgen05)
//
// One CTA per (128-row query tile, query head, batch), eight warps:
//   warp 0     TMA producer: the Q and dO tiles once, then the K and V tiles
//              of 64 keys through a kDqStages ring;
//   warps 1-3  MMA issuers (one thread each; warp 1 also owns TMEM): per key
//              tile j, warp 1 issues S(j) = Q K_j^T and warp 2 dP(j) =
//              dO V_j^T into TMEM buffer j % 2 (smem x smem, K-major
//              operands); once the softmax has written dS(j), warp 3 issues
//              dQ += dS(j) K_j (dS from TMEM, K as an MN-major smem operand).
//              A tcgen05.mma returns to its thread only when the tensor core
//              accepts it, so one issuer per chain lets the chains interleave;
//              the S and dP of tile j + 1 run while the softmax works on j;
//   warps 4-11 two warpgroups, one thread per query row (TMEM lane), taking
//              alternate key tiles: dS = P (dP - D) with
//              P = 2^(S scale log2 e - LSE log2 e), packed to bf16 into TMEM;
//              at the end dQ (fp32, TMEM) * scale -> bf16.
// TMEM columns: S[2] at 0 / 64, dP[2] at 128 / 192, dS[2] (bf16 pairs) at
// 256 / 288, dQ at 320.
constexpr int kDqRows = kBwdDqRows, kDqKeys = 64, kDqStages = 4, kDqThreads = kBwdThreads;
constexpr uint32_t kDqTile = kDqRows * 64 * 2;   // Q or dO tile, 16 KB
constexpr uint32_t kColDqS = 0, kColDqP = 128, kColDqDs = 256, kColDq = 320;

struct __align__(1024) DqSmem {
    uint8_t q[kDqTile];
    uint8_t dout[kDqTile];
    uint8_t k[kDqStages][kTileBytes];
    uint8_t v[kDqStages][kTileBytes];
    uint64_t q_full, kv_full[kDqStages], kv_empty[kDqStages];
    uint64_t s_full[2], s_free[2], ds_full[2], dq_done[2], mma_done;
    uint32_t tmem_base;
    uint32_t abort_flag;
};

// dQ of query tile qt of head h, batch b (one CTA; the maps are kernel
// parameters, so their addresses stay in the parameter space).
template <int MOD>
__device__ __forceinline__ void bwd_dq_body(const CUtensorMap &tm_q, const CUtensorMap &tm_do,
                                            const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                            const BwdParams &p, const int qt, const int h, const int b)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = qt * kDqRows;
    const int hk = h / (p.Hq / p.Hk);
    // the key tiles holding an allowed pair of the tile's rows, and the span
    // of keys every row allows (tiles inside it need no mask)
    const TileRange tr = q_block_range<kDqKeys>(p.mask, b, q0);
    const int n_it = max(tr.hi - tr.lo, 0);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    DqSmem &sm = *reinterpret_cast<DqSmem *>(smem_raw + ((1024u - (base & 1023u)) & 1023u));
    auto bar = [](const uint64_t &x) { return ptx::smem_u32(&x); };

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(sm.q_full), 1);
        for (int s = 0; s < kDqStages; ++s) {
            ptx::mbar_init(bar(sm.kv_full[s]), 1);
            ptx::mbar_init(bar(sm.kv_empty[s]), 2); // the dP and the dQ issuer
        }
        for (int u = 0; u < 2; ++u) {
            ptx::mbar_init(bar(sm.s_full[u]), 2);   // the S and the dP issuer
            ptx::mbar_init(bar(sm.s_free[u]), 128);
            ptx::mbar_init(bar(sm.ds_full[u]), 128);
            ptx::mbar_init(bar(sm.dq_done[u]), 1);
        }
        ptx::mbar_init(bar(sm.mma_done), 3);        // every issuer
        sm.abort_flag = 0;
        ptx::fence_mbarrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&sm.tmem_base), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    WaitCtl wc;
    wc.abort_flag = &sm.abort_flag;
    wc.timeout_cycles = p.timeout_ns * 21 / 10;
    wc.err_user = p.err_user;
    wc.err_lib = &g_lib_error_word;
    bool ok = true;

    if (warp == 0) {
        // ---- producer
        int issued = 0;
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(sm.q_full), 2 * kDqTile);
            ptx::tma_load_4d(ptx::smem_u32(sm.q), &tm_q, bar(sm.q_full), 0, q0, h, b);
            ptx::tma_load_4d(ptx::smem_u32(sm.dout), &tm_do, bar(sm.q_full), 0, q0, h, b);
        }
        for (int j = 0; j < n_it; ++j) {
            const int s = j % kDqStages;
            if (j >= kDqStages && !warp_wait(bar(sm.kv_empty[s]), ((j / kDqStages) - 1) & 1, wc, W_KV_EMPTY)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bar(sm.kv_full[s]), 2 * kTileBytes);
                ptx::tma_load_4d(ptx::smem_u32(sm.k[s]), &tm_k, bar(sm.kv_full[s]), 0, (tr.lo + j) * kDqKeys, hk, b);
                ptx::tma_load_4d(ptx::smem_u32(sm.v[s]), &tm_v, bar(sm.kv_full[s]), 0, (tr.lo + j) * kDqKeys, hk, b);
            }
            __syncwarp();
            issued = j + 1;
        }
        if (!ok) {
            // the last copies into each stage, and Q / dO, may still land
            for (int s = 0; s < kDqStages; ++s) {
                const int last = issued - 1 - ((issued - 1 - s) % kDqStages + kDqStages) % kDqStages;
                if (last >= 0)
                    mbar_wait_drain(bar(sm.kv_full[s]), (last / kDqStages) & 1, wc, W_DRAIN);
            }
            mbar_wait_drain(bar(sm.q_full), 0, wc, W_DRAIN);
        }
    } else if (warp <= 3) {
        // ---- MMA issuers, one chain kind per warp so the chains interleave
        // on the tensor core: warp 1 S(j), warp 2 dP(j), warp 3 dQ += dS(j) K
        constexpr uint32_t idesc_s = umma_idesc_bf16(kDqRows, kDqKeys, false);
        constexpr uint32_t idesc_dq = umma_idesc_bf16(kDqRows, 64, true);
        constexpr uint64_t kHiKmaj = umma_desc_hi(16, 1024, kSwizzle128B);
        constexpr uint64_t kHiMN = umma_desc_hi(16, 1024, kSwizzle128B);
        if (warp < 3) {
            const uint32_t a_lo = ptx::smem_u32(warp == 1 ? sm.q : sm.dout) >> 4;
            const uint32_t col = warp == 1 ? kColDqS : kColDqP;
            ok = warp_wait(bar(sm.q_full), 0, wc, W_Q_FULL);
            for (int j = 0; j < n_it && ok; ++j) {
                const int s = j % kDqStages, u = j & 1;
                if (!warp_wait(bar(sm.kv_full[s]), (j / kDqStages) & 1, wc, W_KV_FULL) ||
                    (j >= 2 && !warp_wait(bar(sm.s_free[u]), ((j - 2) >> 1) & 1, wc, W_S_FULL))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if (lane == 0) {
                    // S = Q K^T (warp 1) or dP = dO V^T (warp 2)
                    const uint32_t b_lo = ptx::smem_u32(warp == 1 ? sm.k[s] : sm.v[s]) >> 4;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_ss(tmem + col + 64 * u, kHiKmaj | (a_lo + 2 * kk), kHiKmaj | (b_lo + 2 * kk),
                                    idesc_s, kk > 0 ? 1u : 0u);
                    ptx::mma_commit(bar(sm.s_full[u]));
                    if (warp == 2)
                        ptx::mma_commit(bar(sm.kv_empty[s])); // the last read of V_j
                }
                __syncwarp();
            }
        } else {
            for (int j = 0; j < n_it; ++j) {
                const int s = j % kDqStages, u = j & 1;
                if (!warp_wait(bar(sm.ds_full[u]), (j >> 1) & 1, wc, W_P_FULL)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t k_lo = ptx::smem_u32(sm.k[s]) >> 4;
#pragma unroll
                    for (int kk = 0; kk < kDqKeys / 16; ++kk)
                        ptx::mma_ts(tmem + kColDq, tmem + kColDqDs + 32 * u + 8 * kk, kHiMN | (k_lo + 128 * kk),
                                    idesc_dq, (j > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(bar(sm.dq_done[u]));
                    // the last read of K_j (S(j) completed before dS(j) existed)
                    ptx::mma_commit(bar(sm.kv_empty[s]));
                }
                __syncwarp();
            }
        }
        // every MMA the issuers started has completed before TMEM is read or freed
        if (lane == 0)
            ptx::mma_commit(bar(sm.mma_done));
        __syncwarp();
        mbar_wait_drain(bar(sm.mma_done), 0, wc, W_FINAL);
    } else {
        // ---- softmax warpgroups (warps 4-7 take the even key tiles, 8-11 the
        // odd ones: TMEM buffer u = j % 2 belongs to warpgroup u); a warp
        // reaches TMEM lanes 32 (warp % 4) ..
        const int wg = (warp >> 2) - 1;
        const int r = 32 * (warp & 3) + lane;
        const int row = q0 + r;
        const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        const BwdRowStat st = p.ws_stats[(static_cast<int64_t>(b) * p.Hq + h) * p.S_pad + row];
        const ModCtx mc = mod_ctx(p, b, h);
        for (int j = wg; j < n_it; j += 2) {
            const int u = j & 1;
            if (!warp_wait(bar(sm.s_full[u]), (j >> 1) & 1, wc, W_S_FULL)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint32_t sv[64], pv[64];
            ptx::tmem_ld32(tmem + lane_off + kColDqS + 64 * u, sv);
            ptx::tmem_ld32(tmem + lane_off + kColDqS + 64 * u + 32, sv + 32);
            ptx::tmem_ld32(tmem + lane_off + kColDqP + 64 * u, pv);
            ptx::tmem_ld32(tmem + lane_off + kColDqP + 64 * u + 32, pv + 32);
            ptx::tmem_wait_ld();
            ptx::reg_fence<64>(sv);
            ptx::reg_fence<64>(pv);
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(sm.s_free[u]));
            const int j0 = (tr.lo + j) * kDqKeys;
            const bool edge = !(j0 >= tr.full_lo && j0 + kDqKeys <= tr.full_hi);
            uint32_t ds[32];
            if constexpr (MOD != MOD_EXPR) {
                if constexpr (MOD != MOD_SOFTCAP) {
                    // a removed pair's score -> -inf, so its P is 0 (a softcap
                    // score is bounded: its argument is masked below instead)
                    if (edge) {
#pragma unroll
                        for (int col = 0; col < 64; ++col)
                            if (j0 + col < st.lo || j0 + col >= st.hi)
                                sv[col] = 0xFF800000u;
                    }
                }
                const float nl = -st.lse2, nd = -st.d;
                float dA = static_cast<float>(row - j0), dB = dA - 1.f; // i - j of keys 2c, 2c + 1
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float a0, a1, ch0, ch1, u0, u1, r0, r1;
                    mod_args2<MOD>(mc, __uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1]), dA, dB, nl, nl,
                                   a0, a1, ch0, ch1);
                    if constexpr (MOD == MOD_ALIBI)
                        ptx::add2(dA, dB, -2.f, -2.f);
                    if constexpr (MOD == MOD_SOFTCAP) {
                        if (edge) {
                            if (j0 + 2 * c < st.lo || j0 + 2 * c >= st.hi)
                                a0 = kNegInf;
                            if (j0 + 2 * c + 1 < st.lo || j0 + 2 * c + 1 >= st.hi)
                                a1 = kNegInf;
                        }
                    }
                    const float p0 = ptx::ex2(a0), p1 = ptx::ex2(a1);
                    ptx::fma2(u0, u1, __uint_as_float(pv[2 * c]), __uint_as_float(pv[2 * c + 1]), 1.f, 1.f, nd,
                              nd);
                    if constexpr (MOD == MOD_SOFTCAP)
                        ptx::fma2(u0, u1, u0, u1, ch0, ch1, 0.f, 0.f);
                    ptx::fma2(r0, r1, p0, p1, u0, u1, 0.f, 0.f);
                    ds[c] = ptx::pack_bf16(r0, r1);
                }
            } else
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float d2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = 2 * c + e;
                    float chain;
                    const float t = mod_logit2<MOD>(mc, __uint_as_float(sv[col]), row, j0 + col, chain);
                    const float pr = ptx::ex2(t - st.lse2);
                    float dsv = pr * (__uint_as_float(pv[col]) - st.d) * chain;
                    if constexpr (MOD == MOD_EXPR)
                        dsv = pr > 0.f ? dsv : 0.f; // a removed pair's derivative may be inf or NaN
                    if (edge && (j0 + col < st.lo || j0 + col >= st.hi))
                        dsv = 0.f;
                    d2[e] = dsv;
                }
                ds[c] = ptx::pack_bf16(d2[0], d2[1]);
            }
            // dQ(j - 2) has read dS buffer u
            if (j >= 2 && !warp_wait(bar(sm.dq_done[u]), ((j - 2) >> 1) & 1, wc, W_O_FULL)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            ptx::tmem_st32(tmem + lane_off + kColDqDs + 32 * u, ds);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(sm.ds_full[u]));
        }
        if (ok)
            ok = warp_wait(bar(sm.mma_done), 0, wc, W_FINAL);
        // warpgroup wg writes output columns 32 wg .. 32 wg + 31 of its row;
        // the TMEM load is warp-collective, so every lane takes it (`ok` is
        // warp-uniform) and only the store depends on the row
        if (ok) {
            uint32_t o[32];
            ptx::tc_fence_after();
            ptx::tmem_ld32(tmem + lane_off + kColDq + 32 * wg, o);
            ptx::tmem_wait_ld();
            ptx::reg_fence<32>(o);
            const float f = n_it > 0 ? p.scale : 0.f; // no visited tile: dQ = 0
            uint4 *dst = reinterpret_cast<uint4 *>(p.dq + b * p.dq_sb + static_cast<int64_t>(row) * p.dq_ss +
                                                   h * p.dq_sh + 32 * wg);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    w[q] = ptx::pack_bf16(__uint_as_float(o[8 * c + 2 * q]) * f,
                                          __uint_as_float(o[8 * c + 2 * q + 1]) * f);
                if (row < p.S)
                    dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- dK, dV (tcgen05)
//
// One CTA per (128-key tile, KV head, batch), twelve warps; the key tile is
// the MMA's M side (TMEM lane = key):
//   warp 0     TMA producer: the K and V tiles once, then for every query
//              tile of 64 rows of every query head of the group that holds
//              an allowed pair with the key tile, the Q and dO tiles through a
//              kKvStages ring, with the rows' (LSE log2 e, D) copied by the
//              warp's lanes;
//   warps 1-3  MMA issuers: warp 1 S^T(i) = K Q_i^T, warp 2 dP^T(i) =
//              V dO_i^T into TMEM buffer i % 2; warp 3, once P^T(i) and
//              dS^T(i) are in TMEM, dV += P^T(i) dO_i and dK += dS^T(i) Q_i
//              (TMEM x MN-major smem operands), accumulating over the whole
//              loop;
//   warps 4-11 two warpgroups taking alternate query tiles, one thread per
//              key: P^T = 2^(S^T scale log2 e - LSE log2 e) and
//              dS^T = P^T (dP^T - D), both packed to bf16 into TMEM; at the
//              end warpgroup 0 writes dV and warpgroup 1 scale * dK.
// TMEM columns: S^T[2] at 0 / 64, dP^T[2] at 128 / 192, P^T[2] at 256 / 288,
// dS^T[2] at 320 / 352, dV at 384, dK at 448.
constexpr int kKvKeys = kBwdKvKeys, kKvQ = 64, kKvStages = 4, kKvThreads = kBwdThreads;
constexpr uint32_t kKvTile = kKvKeys * 64 * 2;   // K or V tile, 16 KB
constexpr uint32_t kColTS = 0, kColTP = 128, kColTPb = 256, kColTDs = 320, kColDv = 384, kColDk = 448;

struct __align__(1024) DkvSmem {
    uint8_t k[kKvTile];
    uint8_t v[kKvTile];
    uint8_t q[kKvStages][kTileBytes];
    uint8_t dout[kKvStages][kTileBytes];
    BwdRowStat stats[kKvStages][kKvQ];
    uint64_t kv_full, st_full[kKvStages], st_empty[kKvStages];
    uint64_t s_full[2], s_free[2], pds_full[2], acc_done[2], mma_done;
    uint32_t tmem_base;
    uint32_t abort_flag;
};

// dK and dV of key tile kt of KV head hk, batch b (one CTA).
template <int MOD>
__device__ __forceinline__ void bwd_dkdv_body(const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                              const CUtensorMap &tm_q, const CUtensorMap &tm_do,
                                              const BwdParams &p, const int kt, const int hk, const int b)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k0 = kt * kKvKeys;
    const int G = p.Hq / p.Hk;
    const int nq = p.S_pad / kKvQ;
    // the query tiles whose rows allow a key of this tile (row intervals never
    // decrease with the row, so those rows form one interval)
    int qa, qb;
    key_block_query_range(p.mask, b, k0, min(k0 + kKvKeys, p.S), qa, qb);
    const int qj0 = qa / kKvQ;
    const int n_qt = max((qb + kKvQ - 1) / kKvQ - qj0, 0);
    const int n_it = G * n_qt;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    DkvSmem &sm = *reinterpret_cast<DkvSmem *>(smem_raw + ((1024u - (base & 1023u)) & 1023u));
    auto bar = [](const uint64_t &x) { return ptx::smem_u32(&x); };

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(sm.kv_full), 1);
        for (int s = 0; s < kKvStages; ++s) {
            ptx::mbar_init(bar(sm.st_full[s]), 1);
            ptx::mbar_init(bar(sm.st_empty[s]), 1); // the dV / dK issuer
        }
        for (int u = 0; u < 2; ++u) {
            ptx::mbar_init(bar(sm.s_full[u]), 2);   // the S^T and the dP^T issuer
            ptx::mbar_init(bar(sm.s_free[u]), 128);
            ptx::mbar_init(bar(sm.pds_full[u]), 128);
            ptx::mbar_init(bar(sm.acc_done[u]), 1);
        }
        ptx::mbar_init(bar(sm.mma_done), 3);
        sm.abort_flag = 0;
        ptx::fence_mbarrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&sm.tmem_base), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    WaitCtl wc;
    wc.abort_flag = &sm.abort_flag;
    wc.timeout_cycles = p.timeout_ns * 21 / 10;
    wc.err_user = p.err_user;
    wc.err_lib = &g_lib_error_word;
    bool ok = true;

    if (warp == 0) {
        // ---- producer
        int issued = 0;
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(sm.kv_full), 2 * kKvTile);
            ptx::tma_load_4d(ptx::smem_u32(sm.k), &tm_k, bar(sm.kv_full), 0, k0, hk, b);
            ptx::tma_load_4d(ptx::smem_u32(sm.v), &tm_v, bar(sm.kv_full), 0, k0, hk, b);
        }
        for (int i = 0; i < n_it; ++i) {
            const int s = i % kKvStages;
            const int h = hk * G + i / n_qt, q0 = (qj0 + i % n_qt) * kKvQ;
            if (i >= kKvStages && !warp_wait(bar(sm.st_empty[s]), ((i / kKvStages) - 1) & 1, wc, W_KV_EMPTY)) {
                ok = false;
                break;
            }
            const BwdRowStat *src = p.ws_stats + (static_cast<int64_t>(b) * p.Hq + h) * p.S_pad + q0;
            sm.stats[s][lane] = src[lane];
            sm.stats[s][lane + 32] = src[lane + 32];
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bar(sm.st_full[s]), 2 * kTileBytes);
                ptx::tma_load_4d(ptx::smem_u32(sm.q[s]), &tm_q, bar(sm.st_full[s]), 0, q0, h, b);
                ptx::tma_load_4d(ptx::smem_u32(sm.dout[s]), &tm_do, bar(sm.st_full[s]), 0, q0, h, b);
            }
            __syncwarp();
            issued = i + 1;
        }
        if (!ok) {
            for (int s = 0; s < kKvStages; ++s) {
                const int last = issued - 1 - ((issued - 1 - s) % kKvStages + kKvStages) % kKvStages;
                if (last >= 0)
                    mbar_wait_drain(bar(sm.st_full[s]), (last / kKvStages) & 1, wc, W_DRAIN);
            }
            mbar_wait_drain(bar(sm.kv_full), 0, wc, W_DRAIN);
        }
    } else if (warp <= 3) {
        // ---- MMA issuers
        constexpr uint32_t idesc_s = umma_idesc_bf16(kKvKeys, kKvQ, false);
        constexpr uint32_t idesc_acc = umma_idesc_bf16(kKvKeys, 64, true);
        constexpr uint64_t kHiKmaj = umma_desc_hi(16, 1024, kSwizzle128B);
        constexpr uint64_t kHiMN = umma_desc_hi(16, 1024, kSwizzle128B);
        if (warp < 3) {
            // S^T = K Q_i^T (warp 1) or dP^T = V dO_i^T (warp 2)
            const uint32_t a_lo = ptx::smem_u32(warp == 1 ? sm.k : sm.v) >> 4;
            const uint32_t col = warp == 1 ? kColTS : kColTP;
            ok = warp_wait(bar(sm.kv_full), 0, wc, W_Q_FULL);
            for (int i = 0; i < n_it && ok; ++i) {
                const int s = i % kKvStages, u = i & 1;
                if (!warp_wait(bar(sm.st_full[s]), (i / kKvStages) & 1, wc, W_KV_FULL) ||
                    (i >= 2 && !warp_wait(bar(sm.s_free[u]), ((i - 2) >> 1) & 1, wc, W_S_FULL))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t b_lo = ptx::smem_u32(warp == 1 ? sm.q[s] : sm.dout[s]) >> 4;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_ss(tmem + col + 64 * u, kHiKmaj | (a_lo + 2 * kk), kHiKmaj | (b_lo + 2 * kk),
                                    idesc_s, kk > 0 ? 1u : 0u);
                    ptx::mma_commit(bar(sm.s_full[u]));
                }
                __syncwarp();
            }
        } else {
            for (int i = 0; i < n_it; ++i) {
                const int s = i % kKvStages, u = i & 1;
                if (!warp_wait(bar(sm.pds_full[u]), (i >> 1) & 1, wc, W_P_FULL)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t do_lo = ptx::smem_u32(sm.dout[s]) >> 4, q_lo = ptx::smem_u32(sm.q[s]) >> 4;
#pragma unroll
                    for (int kk = 0; kk < kKvQ / 16; ++kk)
                        ptx::mma_ts(tmem + kColDv, tmem + kColTPb + 32 * u + 8 * kk, kHiMN | (do_lo + 128 * kk),
                                    idesc_acc, (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < kKvQ / 16; ++kk)
                        ptx::mma_ts(tmem + kColDk, tmem + kColTDs + 32 * u + 8 * kk, kHiMN | (q_lo + 128 * kk),
                                    idesc_acc, (i > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(bar(sm.acc_done[u]));
                    // the stage's last readers (S^T(i), dP^T(i) completed before P^T(i) existed)
                    ptx::mma_commit(bar(sm.st_empty[s]));
                }
                __syncwarp();
            }
        }
        if (lane == 0)
            ptx::mma_commit(bar(sm.mma_done));
        __syncwarp();
        mbar_wait_drain(bar(sm.mma_done), 0, wc, W_FINAL);
    } else {
        // ---- two softmax warpgroups (warps 4-7: even i, 8-11: odd i); a warp
        // reaches TMEM lanes 32 (warp % 4) ..
        const int wg = (warp >> 2) - 1;
        const int r = 32 * (warp & 3) + lane;
        const int key = k0 + r;
        const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        for (int i = wg; i < n_it; i += 2) {
            const int s = i % kKvStages, u = i & 1;
            const int q0 = (qj0 + i % n_qt) * kKvQ;
            const ModCtx mc = mod_ctx(p, b, hk * G + i / n_qt);
            // the stage's row statistics (written by the producer warp before
            // it armed st_full) and the tile's S^T, dP^T
            if (!warp_wait(bar(sm.st_full[s]), (i / kKvStages) & 1, wc, W_KV_FULL) ||
                !warp_wait(bar(sm.s_full[u]), (i >> 1) & 1, wc, W_S_FULL)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            // no masked pair in the tile iff its first row allows keys up to the
            // tile's end and its last row allows keys from the tile's start
            const bool edge = !(sm.stats[s][0].hi >= k0 + kKvKeys && sm.stats[s][kKvQ - 1].lo <= k0);
            uint32_t pa[32], da[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t sv[32], pv[32];
                ptx::tmem_ld32(tmem + lane_off + kColTS + 64 * u + 32 * half, sv);
                ptx::tmem_ld32(tmem + lane_off + kColTP + 64 * u + 32 * half, pv);
                ptx::tmem_wait_ld();
                ptx::reg_fence<32>(sv);
                ptx::reg_fence<32>(pv);
                if constexpr (MOD != MOD_EXPR) {
                    if constexpr (MOD != MOD_SOFTCAP) {
                        if (edge) {
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                const BwdRowStat &sc = sm.stats[s][32 * half + c];
                                if (key < sc.lo || key >= sc.hi)
                                    sv[c] = 0xFF800000u; // -inf: P = 0
                            }
                        }
                    }
                    // i - j of query rows 2 c2, 2 c2 + 1 of this half
                    float dA = static_cast<float>(q0 + 32 * half - key), dB = dA + 1.f;
#pragma unroll
                    for (int c2 = 0; c2 < 16; ++c2) {
                        const BwdRowStat s0 = sm.stats[s][32 * half + 2 * c2];
                        const BwdRowStat s1 = sm.stats[s][32 * half + 2 * c2 + 1];
                        float a0, a1, ch0, ch1, u0, u1, r0, r1;
                        mod_args2<MOD>(mc, __uint_as_float(sv[2 * c2]), __uint_as_float(sv[2 * c2 + 1]), dA, dB,
                                       -s0.lse2, -s1.lse2, a0, a1, ch0, ch1);
                        if constexpr (MOD == MOD_ALIBI)
                            ptx::add2(dA, dB, 2.f, 2.f);
                        if constexpr (MOD == MOD_SOFTCAP) {
                            if (edge) {
                                if (key < s0.lo || key >= s0.hi)
                                    a0 = kNegInf;
                                if (key < s1.lo || key >= s1.hi)
                                    a1 = kNegInf;
                            }
                        }
                        const float p0 = ptx::ex2(a0), p1 = ptx::ex2(a1);
                        ptx::fma2(u0, u1, __uint_as_float(pv[2 * c2]), __uint_as_float(pv[2 * c2 + 1]), 1.f, 1.f,
                                  -s0.d, -s1.d);
                        if constexpr (MOD == MOD_SOFTCAP)
                            ptx::fma2(u0, u1, u0, u1, ch0, ch1, 0.f, 0.f);
                        ptx::fma2(r0, r1, p0, p1, u0, u1, 0.f, 0.f);
                        pa[16 * half + c2] = ptx::pack_bf16(p0, p1);
                        da[16 * half + c2] = ptx::pack_bf16(r0, r1);
                    }
                    continue;
                }
#pragma unroll
                for (int c2 = 0; c2 < 16; ++c2) {
                    float pp[2], dd[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int c = 32 * half + 2 * c2 + e;
                        const BwdRowStat st = sm.stats[s][c];
                        float chain;
                        const float t = mod_logit2<MOD>(mc, __uint_as_float(sv[2 * c2 + e]), q0 + c, key, chain);
                        float pr = ptx::ex2(t - st.lse2);
                        if (edge && (key < st.lo || key >= st.hi))
                            pr = 0.f;
                        pp[e] = pr;
                        dd[e] = pr * (__uint_as_float(pv[2 * c2 + e]) - st.d) * chain;
                        if constexpr (MOD == MOD_EXPR)
                            dd[e] = pr > 0.f ? dd[e] : 0.f; // a removed pair's derivative may be inf or NaN
                    }
                    pa[16 * half + c2] = ptx::pack_bf16(pp[0], pp[1]);
                    da[16 * half + c2] = ptx::pack_bf16(dd[0], dd[1]);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(sm.s_free[u]));
            // dV / dK of tile i - 2 have read P^T / dS^T buffer u
            if (i >= 2 && !warp_wait(bar(sm.acc_done[u]), ((i - 2) >> 1) & 1, wc, W_O_FULL)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            ptx::tmem_st32(tmem + lane_off + kColTPb + 32 * u, pa);
            ptx::tmem_st32(tmem + lane_off + kColTDs + 32 * u, da);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(sm.pds_full[u]));
        }
        if (ok)
            ok = warp_wait(bar(sm.mma_done), 0, wc, W_FINAL);
        // warpgroup 0 writes dV, warpgroup 1 scale * dK (the TMEM loads are
        // warp-collective: every lane takes them; only the stores test the key)
        if (ok) {
            ptx::tc_fence_after();
            uint32_t o[64];
            const uint32_t col = wg == 0 ? kColDv : kColDk;
            ptx::tmem_ld32(tmem + lane_off + col, o);
            ptx::tmem_ld32(tmem + lane_off + col + 32, o + 32);
            ptx::tmem_wait_ld();
            ptx::reg_fence<64>(o);
            const float f = n_it > 0 ? (wg == 0 ? 1.f : p.scale) : 0.f; // no visited tile: 0
            __nv_bfloat16 *dst = wg == 0 ? p.dv + b * p.dv_sb + static_cast<int64_t>(key) * p.dv_ss + hk * p.dv_sh
                                         : p.dk + b * p.dk_sb + static_cast<int64_t>(key) * p.dk_ss + hk * p.dk_sh;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    w[q] = ptx::pack_bf16(__uint_as_float(o[8 * c + 2 * q]) * f,
                                          __uint_as_float(o[8 * c + 2 * q + 1]) * f);
                if (key < p.S)
                    reinterpret_cast<uint4 *>(dst)[c] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// more than half an SM's shared memory: one dQ CTA per SM, so that no second
// CTA waits in tcgen05.alloc for the 512 TMEM columns the first one holds
// Both gradients in one launch: blocks [0, n_kv) take the dK/dV tiles (key
// tile fastest, then KV head, then batch), the others the dQ tiles (query
// tile fastest, then head, then batch).  With one CTA per SM, two launches
// each end in a partly filled wave and the second cannot start on the SMs
// the first leaves idle; one grid shares a single last wave.
template <int MOD>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_fused_kernel(const __grid_constant__ CUtensorMap tm_k128, const __grid_constant__ CUtensorMap tm_v128,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_q128, const __grid_constant__ CUtensorMap tm_do128,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const BwdParams p)
{
    const int nkt = (p.S + kKvKeys - 1) / kKvKeys;
    const int n_kv = nkt * p.Hk * p.B;
    int x = static_cast<int>(blockIdx.x);
    if (x < n_kv) {
        const int kt = x % nkt;
        x /= nkt;
        bwd_dkdv_body<MOD>(tm_k128, tm_v128, tm_q, tm_do, p, kt, x % p.Hk, x / p.Hk);
    } else {
        x -= n_kv;
        const int nqt = (p.S + kDqRows - 1) / kDqRows;
        const int qt = x % nqt;
        x /= nqt;
        bwd_dq_body<MOD>(tm_q128, tm_do128, tm_k, tm_v, p, qt, x % p.Hq, x / p.Hq);
    }
}

constexpr size_t kDqSmemBytes = sizeof(DqSmem) + 1024 > 120 * 1024 ? sizeof(DqSmem) + 1024 : 120 * 1024;
constexpr size_t kKvSmemBytes = sizeof(DkvSmem) + 1024 > 120 * 1024 ? sizeof(DkvSmem) + 1024 : 120 * 1024;

} // namespace

#ifndef __CUDACC_RTC__
namespace {

template <int MOD>
cudaError_t launch_bwd_mod(const CUtensorMap &tq, const CUtensorMap &tdo, const CUtensorMap &tk,
                           const CUtensorMap &tv, const CUtensorMap &tq128, const CUtensorMap &tdo128,
                           const CUtensorMap &tk128, const CUtensorMap &tv128, const BwdParams &p,
                           cudaStream_t stream)
{
    const size_t smem = bwd_smem_bytes();
    static bool configured = false; // benign race: the call is idempotent
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(bwd_fused_kernel<MOD>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    bwd_fused_kernel<MOD><<<static_cast<unsigned>(bwd_fused_blocks(p)), kBwdThreads, smem, stream>>>(
        tk128, tv128, tq, tdo, tq128, tdo128, tk, tv, p);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_bwd_prep(const BwdParams &p, cudaStream_t stream)
{
    const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.S_pad;
    bwd_prep_kernel<<<static_cast<unsigned>((rows + 127) / 128), 128, 0, stream>>>(p);
    return cudaGetLastError();
}

size_t bwd_smem_bytes() { return kKvSmemBytes > kDqSmemBytes ? kKvSmemBytes : kDqSmemBytes; }

int64_t bwd_fused_blocks(const BwdParams &p)
{
    return int64_t((p.S + kKvKeys - 1) / kKvKeys) * p.Hk * p.B +
           int64_t((p.S + kDqRows - 1) / kDqRows) * p.Hq * p.B;
}

cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tdo, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tq128, const CUtensorMap &tdo128,
                       const CUtensorMap &tk128, const CUtensorMap &tv128, const BwdParams &p,
                       cudaStream_t stream)
{
    const cudaError_t e = launch_bwd_prep(p, stream);
    if (e != cudaSuccess)
        return e;
    switch (p.score_mod) {
    case MOD_ALIBI:
        return launch_bwd_mod<MOD_ALIBI>(tq, tdo, tk, tv, tq128, tdo128, tk128, tv128, p, stream);
    case MOD_SOFTCAP:
        return launch_bwd_mod<MOD_SOFTCAP>(tq, tdo, tk, tv, tq128, tdo128, tk128, tv128, p, stream);
    default:
        return launch_bwd_mod<MOD_NONE>(tq, tdo, tk, tv, tq128, tdo128, tk128, tv128, p, stream);
    }
}

#endif // !__CUDACC_RTC__

} // namespace fl
