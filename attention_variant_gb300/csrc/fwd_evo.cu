// fwd_evo.cu -- Evoformer MSA gated self-attention forward, c = 32 per head:
//     O = sigmoid(g) * softmax(scale q k^T + b) v
// row-wise (attention over residues for each MSA row, pair bias b[h, i, j]
// shared by every MSA row) and column-wise (attention over MSA rows for each
// residue, no bias).  The pages evaluate both as complex variants template
// systems cannot express (talk notes, "Evaluation: complex variants" and
// "End-to-end: AlphaFold2": Evoformer with 8 heads of dimension 32); here the
// gate is fused into the epilogue and the bias into the online softmax.
//
// Both passes run over a [batch, sequence, head, c] view: the row pass takes
// batch = MSA row and sequence = residue, the column pass the reverse (the
// host swaps the two strides).
//
// Work item = (head h, query block qb, a chunk of batch indices).  The CTA's
// two slots take alternate batch indices of the chunk; a slot's "steps" are
// its (batch index, key tile) pairs in order.  In the row pass the bias rows
// of (h, qb) are loaded once per item into shared memory (128 rows x up to
// 384 keys) and read by every MSA row of the chunk: the pair-bias tile is
// reused across MSA rows instead of being re-read from L2 for each of them.
//
// Warps: 0 TMA producer for both slots (Q double-buffered per slot, K/V
// through one ring per slot, and the bias), 1 issues S = Q K^T for both slots
// (TMEM owner), 2 and 3 issue O += P V for slot 0 and slot 1, 4-7 softmax of
// slot 0, 8-11 softmax of slot 1.  The producer and the S warp walk the steps
// of both slots interleaved (step s of slot 0, then of slot 1), the order in
// which the slots consume them.  Q K^T and P V are issued by different warps
// because a tcgen05.mma returns to its issuing thread only once the tensor
// core has accepted it: one thread issuing both chains of a slot spends most
// of a tile blocked in issue.

// TMEM per slot t: S[t] fp32 at 128 t; O[t] at 256 + 64 t with 48 columns:
// 32 output columns and 16 columns of sum_j P_j (P V multiplies P by V
// extended with a tile of ones, so the tensor core also sums the exact bf16 P
// it used: the normaliser of O); P[t] bf16 pairs at 384 + 64 t.
//
// Per slot and key tile j: softmax waits s_full, copies S out of TMEM and
// arrives s_free (the MMA warp then issues the next Q K^T at once), computes P
// in registers, waits pv_done (the previous P V), rescales O if the reference
// max moved, writes P, arrives p_full (the MMA warp then issues P V).  The
// epilogue of one batch index (O / sum, times the prefetched gate) runs inside
// the first key tile of the slot's next batch index, where the latency of the
// last P V is hidden behind the exponentials.
#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "launch.h"
#include "softmax_tile.cuh"

namespace fl {
namespace {

constexpr int kThreads = 384;
constexpr uint32_t kRegsLaunch = 168;
constexpr uint32_t kRegsSoftmax = 200;
constexpr uint32_t kRegsOther = 104;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther == kThreads * kRegsLaunch,
              "register split must equal the launch allocation");
constexpr uint32_t kTile = BM * 32 * 2;       // one 128 x 32 bf16 tile (8 KB)
constexpr uint32_t kBiasBox = BM * 64 * 2;    // 128 rows x 64 keys of bias (16 KB)
constexpr int kMaxBiasBoxes = 6;              // resident bias covers up to 384 keys
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
constexpr uint32_t kDvExt = 48;               // 32 output columns + 16 sum columns
constexpr uint32_t kColSum = 32;


template <bool BIAS>
struct EvoCfg {
    static constexpr int kStages = BIAS ? 2 : 4; // K/V ring depth per slot
};

template <bool BIAS>
struct __align__(1024) EvoSmem {
    static constexpr int NS = EvoCfg<BIAS>::kStages;
    uint8_t bias[BIAS ? kMaxBiasBoxes : 1][BIAS ? kBiasBox : 1024];
    uint8_t q[2][2][kTile];         // [slot][Q buffer]
    uint8_t k[2][NS][kTile];        // [slot][stage]
    uint8_t v[2][NS][kTile];
    uint8_t ones[kTile];            // bf16 1.0 everywhere: the extra columns of V; it must
                                    // follow every V stage (the descriptor offset is unsigned)
    uint64_t q_full[2][2], q_empty[2][2];
    uint64_t kv_full[2][NS], kv_empty[2][NS];
    uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], o_final[2], s_final;
    uint64_t bias_full, bias_empty;
    uint32_t tmem_base;
    uint32_t abort_flag;
};

__device__ uint32_t g_lib_error_word;

template <bool BIAS>
struct Ctx {
    EvoSmem<BIAS> *sm;
    uint32_t tmem;
    WaitCtl wc;
};

__device__ __forceinline__ uint32_t bar(const uint64_t &b) { return ptx::smem_u32(&b); }

struct EvoItem {
    int h, qb, b0, b1;
};

__device__ __forceinline__ EvoItem decode_evo(const EvoParams &p, int64_t L)
{
    // query blocks fastest, so the items reading the same K/V run together
    EvoItem it;
    it.qb = static_cast<int>(L % p.grid.nq);
    const int64_t rest = L / p.grid.nq;
    it.h = static_cast<int>(rest % p.grid.Hq);
    const int chunk = static_cast<int>(rest / p.grid.Hq);
    it.b0 = chunk * p.chunk;
    it.b1 = min(it.b0 + p.chunk, p.grid.B);
    return it;
}

// Batch indices of slot t in an item: b0 + t, b0 + t + 2, ... < b1.
__device__ __forceinline__ int slot_rows(const EvoItem &it, int t)
{
    return it.b1 - it.b0 > t ? (it.b1 - it.b0 - t + 1) / 2 : 0;
}

// ------------------------------------------------------------------ producer
template <bool BIAS>
__device__ void producer_role(const Ctx<BIAS> &cx, const EvoParams &p, const CUtensorMap *tm_q,
                              const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                              const CUtensorMap *tm_b)
{
    constexpr int NS = EvoCfg<BIAS>::kStages;
    EvoSmem<BIAS> &sm = *cx.sm;
    const uint32_t lane = ptx::lane_id();
    const int nkv = (p.mask.S + BN - 1) / BN;
    const int nbox = (p.mask.S + 63) / 64;
    uint32_t kv_count[2] = {0u, 0u}, q_count[2] = {0u, 0u}, item_count = 0;
    bool ok = true;
    for (int64_t L = blockIdx.x; L < p.n_items && ok; L += gridDim.x, ++item_count) {
        const EvoItem it = decode_evo(p, L);
        if (BIAS) {
            if (item_count > 0) {
                ok = warp_wait(bar(sm.bias_empty), (item_count - 1) & 1, cx.wc, W_BIAS);
                if (!ok)
                    break;
            }
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bar(sm.bias_full), nbox * kBiasBox);
                for (int jb = 0; jb < nbox; ++jb)
                    ptx::tma_load_4d(ptx::smem_u32(sm.bias[jb]), tm_b, bar(sm.bias_full), 64 * jb,
                                     it.qb * BM, it.h, p.bias_rows ? it.b0 / p.bias_rows : 0);
            }
            __syncwarp();
        }
        const int steps[2] = {slot_rows(it, 0) * nkv, slot_rows(it, 1) * nkv};
        const int n_steps = max(steps[0], steps[1]);
        for (int st = 0; st < n_steps && ok; ++st) {
            const int j = st % nkv;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (st >= steps[t])
                    continue;
                const int b = it.b0 + t + 2 * (st / nkv);
                if (j == 0) {
                    const uint32_t qbuf = q_count[t] & 1;
                    if (q_count[t] >= 2) {
                        ok = warp_wait(bar(sm.q_empty[t][qbuf]), ((q_count[t] - 2) >> 1) & 1, cx.wc,
                                       W_Q_EMPTY);
                        if (!ok)
                            break;
                    }
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(bar(sm.q_full[t][qbuf]), kTile);
                        ptx::tma_load_4d(ptx::smem_u32(sm.q[t][qbuf]), tm_q, bar(sm.q_full[t][qbuf]), 0,
                                         it.qb * BM, it.h, b);
                    }
                    __syncwarp();
                    ++q_count[t];
                }
                const uint32_t stage = kv_count[t] % NS;
                ok = warp_wait(bar(sm.kv_empty[t][stage]), ((kv_count[t] / NS) & 1) ^ 1, cx.wc,
                               W_KV_EMPTY);
                if (!ok)
                    break;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(bar(sm.kv_full[t][stage]), 2 * kTile);
                    ptx::tma_load_4d(ptx::smem_u32(sm.k[t][stage]), tm_k, bar(sm.kv_full[t][stage]), 0,
                                     j * BN, it.h, b);
                    ptx::tma_load_4d(ptx::smem_u32(sm.v[t][stage]), tm_v, bar(sm.kv_full[t][stage]), 0,
                                     j * BN, it.h, b);
                }
                __syncwarp();
                ++kv_count[t];
            }
        }
    }
    if (!ok) {
        // wait (bounded, ignoring the abort) for this warp's own loads in flight
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t first = kv_count[t] > NS ? kv_count[t] - NS : 0;
            for (uint32_t idx = first; idx < kv_count[t]; ++idx)
                mbar_wait_drain(bar(sm.kv_full[t][idx % NS]), (idx / NS) & 1, cx.wc, W_DRAIN);
            for (uint32_t n = q_count[t] > 2 ? q_count[t] - 2 : 0; n < q_count[t]; ++n)
                mbar_wait_drain(bar(sm.q_full[t][n & 1]), (n >> 1) & 1, cx.wc, W_DRAIN);
        }
        if (BIAS && item_count > 0)
            mbar_wait_drain(bar(sm.bias_full), (item_count - 1) & 1, cx.wc, W_DRAIN);
    }
}

// ------------------------------------------------------------------ MMA issuers
constexpr uint64_t kHiK = umma_desc_hi(16, 512, kSwizzle64B); // Q, K: K-major, 64-byte rows

// S = Q K^T for both slots, steps interleaved like the producer's.  q_empty
// (one arrival) is committed after a batch index's last S; S(t, s) waits for
// the softmax to have copied S(t, s-1) out of TMEM.
template <bool BIAS>
__device__ void s_role(const Ctx<BIAS> &cx, const EvoParams &p)
{
    constexpr int NS = EvoCfg<BIAS>::kStages;
    EvoSmem<BIAS> &sm = *cx.sm;
    const uint32_t lane = ptx::lane_id();
    constexpr uint32_t idesc_qk = umma_idesc_bf16(BM, BN, false);
    constexpr uint32_t kTileLo = kTile >> 4;
    const int nkv = (p.mask.S + BN - 1) / BN;
    uint32_t kv_count[2] = {0u, 0u}, q_count[2] = {0u, 0u}, issued[2] = {0u, 0u};
    bool ok = true;
    for (int64_t L = blockIdx.x; L < p.n_items && ok; L += gridDim.x) {
        const EvoItem it = decode_evo(p, L);
        const int steps[2] = {slot_rows(it, 0) * nkv, slot_rows(it, 1) * nkv};
        const int n_steps = max(steps[0], steps[1]);
        for (int st = 0; st < n_steps && ok; ++st) {
            const int j = st % nkv;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (st >= steps[t])
                    continue;
                const uint32_t qbuf = q_count[t] & 1;
                if (j == 0) {
                    ok = warp_wait(bar(sm.q_full[t][qbuf]), (q_count[t] >> 1) & 1, cx.wc, W_Q_FULL);
                    if (!ok)
                        break;
                }
                if (issued[t] > 0) {
                    ok = warp_wait(bar(sm.s_free[t]), (issued[t] - 1) & 1, cx.wc, W_S_FULL);
                    if (!ok)
                        break;
                }
                const uint32_t stage = kv_count[t] % NS;
                ok = warp_wait(bar(sm.kv_full[t][stage]), (kv_count[t] / NS) & 1, cx.wc, W_KV_FULL);
                if (!ok)
                    break;
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t qlo = (ptx::smem_u32(sm.q[t][qbuf]) >> 4);
                    const uint32_t klo = (ptx::smem_u32(sm.k[t][0]) >> 4) + stage * kTileLo;
                    const uint32_t tS = cx.tmem + kColS + 128 * t;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        ptx::mma_ss(tS, kHiK | (qlo + 2 * kk), kHiK | (klo + 2 * kk), idesc_qk,
                                    kk > 0 ? 1u : 0u);
                    ptx::mma_commit(bar(sm.s_full[t]));
                    if (j + 1 == nkv)
                        ptx::mma_commit(bar(sm.q_empty[t][qbuf])); // last read of this Q buffer
                }
                __syncwarp();
                ++issued[t];
                ++kv_count[t];
                if (j + 1 == nkv)
                    ++q_count[t];
            }
        }
    }
    // Every MMA this thread issued has completed before TMEM is released.
    if (lane == 0)
        ptx::mma_commit(bar(sm.s_final));
    __syncwarp();
    mbar_wait_drain(bar(sm.s_final), 0, cx.wc, W_FINAL);
}

// O += P [V | 1] for slot t.  S(j) of a step completes before its softmax can
// publish P(j), so the commit after P V also covers the K read: kv_empty has
// one arrival (this warp's).
template <bool BIAS>
__device__ void pv_role(const Ctx<BIAS> &cx, const EvoParams &p, int t)
{
    constexpr int NS = EvoCfg<BIAS>::kStages;
    EvoSmem<BIAS> &sm = *cx.sm;
    const uint32_t lane = ptx::lane_id();
    constexpr uint32_t idesc_pv = umma_idesc_bf16(BM, kDvExt, true);
    constexpr uint32_t kTileLo = kTile >> 4;
    const uint32_t v_lo0 = ptx::smem_u32(sm.v[t][0]) >> 4;
    const uint32_t ones_lo = ptx::smem_u32(sm.ones) >> 4;
    const uint32_t tO = cx.tmem + kColO + 64 * t, tP = cx.tmem + kColP + 64 * t;
    const int nkv = (p.mask.S + BN - 1) / BN;
    uint32_t kv_count = 0, pcount = 0;
    bool ok = true;
    for (int64_t L = blockIdx.x; L < p.n_items && ok; L += gridDim.x) {
        const EvoItem it = decode_evo(p, L);
        const int steps = slot_rows(it, t) * nkv;
        for (int st = 0; st < steps && ok; ++st, ++kv_count) {
            const int j = st % nkv;
            // the softmax has written P(j) and rescaled O: O += P [V_j | 1]
            ok = warp_wait(bar(sm.p_full[t]), pcount & 1, cx.wc, W_P_FULL);
            if (!ok)
                break;
            ++pcount;
            ptx::tc_fence_after();
            if (lane == 0) {
                const uint32_t stage = kv_count % NS;
                const uint32_t vlo = v_lo0 + stage * kTileLo;
                const uint64_t hi_v = umma_desc_hi((ones_lo - vlo) << 4, 512, kSwizzle64B);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    ptx::mma_ts(tO, tP + 8 * kk, hi_v | (vlo + 64 * kk), idesc_pv,
                                (j > 0 || kk > 0) ? 1u : 0u);
                ptx::mma_commit(bar(sm.pv_done[t]));
                ptx::mma_commit(bar(sm.kv_empty[t][stage]));
            }
            __syncwarp();
        }
    }
    const uint32_t b_final = bar(sm.o_final[t]);
    if (lane == 0)
        ptx::mma_commit(b_final);
    __syncwarp();
    mbar_wait_drain(b_final, 0, cx.wc, W_FINAL);
}

// ------------------------------------------------------------------ softmax

struct PendingRow {
    int b, h, qb, i;
    RowState st;
};

__device__ __forceinline__ float tanh_approx(float x)
{
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// sigmoid(g) * O / sum(P) -> bf16 row, LSE, visited-tile count.  O[t] must
// hold the finished output of `pr` (its last P V has completed).
template <bool LSE>
__device__ __forceinline__ void store_row_output(const EvoParams &p, uint32_t tO,
                                                 const PendingRow &pr, int r, int nkv)
{
    uint32_t o[32], sum[1];
    ptx::tmem_ld32(tO, o);
    ptx::tmem_ld1(tO + kColSum, sum);
    ptx::tmem_wait_ld();
    ptx::reg_fence<32>(o);
    ptx::reg_fence<1>(sum);
    const float l_round = __uint_as_float(sum[0]);
    const float inv = l_round > 0.f ? 1.f / l_round : 0.f;
    if (pr.i < p.mask.S) {
        uint4 *d4 = reinterpret_cast<uint4 *>(p.out + pr.b * p.o_sb +
                                              static_cast<int64_t>(pr.i) * p.o_si + pr.h * p.o_sh);
        const uint4 *g4 = reinterpret_cast<const uint4 *>(
            p.gate + pr.b * p.g_sb + static_cast<int64_t>(pr.i) * p.g_si + pr.h * p.g_sh);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
            const uint4 gw = __ldg(g4 + c4); // prefetched into L1 when the row started
            const uint32_t gv[4] = {gw.x, gw.y, gw.z, gw.w};
            uint32_t ov[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                // sigmoid(g) = 1/2 + tanh(g / 2) / 2 (one special-function op)
                const float g0 = __uint_as_float(gv[q] << 16);
                const float g1 = __uint_as_float(gv[q] & 0xFFFF0000u);
                const float s0 = fmaf(0.5f, tanh_approx(0.5f * g0), 0.5f);
                const float s1 = fmaf(0.5f, tanh_approx(0.5f * g1), 0.5f);
                ov[q] = ptx::pack_bf16(__uint_as_float(o[8 * c4 + 2 * q]) * inv * s0,
                                       __uint_as_float(o[8 * c4 + 2 * q + 1]) * inv * s1);
            }
            d4[c4] = make_uint4(ov[0], ov[1], ov[2], ov[3]);
        }
        if (LSE)
            p.lse[pr.b * p.l_sb + pr.h * p.l_sh + pr.i] = row_lse(pr.st);
    }
    if (p.tile_counts && r == 0)
        p.tile_counts[(static_cast<int64_t>(pr.b) * p.grid.Hq + pr.h) * p.grid.nq + pr.qb] = nkv;
}

// Whether the MSA mask keeps key `key` of batch index b (a nonzero entry;
// keys past the sequence count as removed).
__device__ __forceinline__ uint32_t mask_keeps(const EvoParams &p, int b, int key, int S)
{
    if (key >= S)
        return 0u;
    const int64_t off = b * p.km_sb + static_cast<int64_t>(key) * p.km_sk;
    return p.km_f32 ? (__ldg(static_cast<const uint32_t *>(p.kmask) + off) & 0x7FFFFFFFu)
                    : (__ldg(static_cast<const uint16_t *>(p.kmask) + off) & 0x7FFFu);
}

template <bool BIAS, bool LSE, bool KMASK>
__device__ void softmax_role(const Ctx<BIAS> &cx, const EvoParams &p, int t)
{
    EvoSmem<BIAS> &sm = *cx.sm;
    const int r = threadIdx.x & 127;             // row of the query tile = TMEM lane
    const uint32_t wq = (threadIdx.x >> 5) & 3;  // warp's quarter of the lanes
    const uint32_t lane_off = (wq * 32u) << 16;
    const uint32_t tS = cx.tmem + lane_off + kColS + 128 * t;
    const uint32_t tO = cx.tmem + lane_off + kColO + 64 * t;
    const uint32_t tP = cx.tmem + lane_off + kColP + 64 * t;
    const int S = p.mask.S;
    const int nkv = (S + BN - 1) / BN;
    // bias smem: row r of each 64-key box is 128 bytes, 16-byte chunk c stored
    // at position c ^ (r & 7) (the 128-byte swizzle the TMA wrote it with)
    const uint32_t bias_row = ptx::smem_u32(sm.bias[0]) + r * 128;
    uint32_t scount = 0, pvcount = 0, item_count = 0;
    bool pending = false;
    PendingRow prev{};

    for (int64_t L = blockIdx.x; L < p.n_items; L += gridDim.x, ++item_count) {
        const EvoItem it = decode_evo(p, L);
        const int i = it.qb * BM + r;
        const TileRange tr = q_block_range(p.mask, 0, it.qb * BM);
        int row_lo, row_hi;
        row_interval(p.mask, 0, i, row_lo, row_hi);
        if (BIAS && !warp_wait(bar(sm.bias_full), item_count & 1, cx.wc, W_BIAS))
            return;
        for (int b = it.b0 + t; b < it.b1; b += 2) {
            RowState st{kNegInf, 0.f, 0.f};
            for (int j = 0; j < nkv; ++j) {
                // MSA mask of this batch index and key tile: lane l reads keys
                // j0 + 32 w + l (issued before the wait, used after it)
                uint32_t keep[4];
                if constexpr (KMASK) {
                    const int lane = threadIdx.x & 31;
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        keep[w] = mask_keeps(p, b, j * BN + 32 * w + lane, S);
                }
                if (!warp_wait(bar(sm.s_full[t]), scount & 1, cx.wc, W_S_FULL))
                    return;
                ++scount;
                ptx::tc_fence_after();
                float x[BN];
                load_scores(tS, x);
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(sm.s_free[t])); // S[t] may be overwritten
                const int j0 = j * BN;
                float c = p.qk_log2;
                if constexpr (BIAS) {
                    // natural-unit logits scale q.k + b[h, i, j]; log2 e goes
                    // into the exponent
                    c = kLog2e;
#pragma unroll
                    for (int ch = 0; ch < BN / 8; ++ch) {
                        const int box = 2 * j + (ch >> 3), cc = ch & 7;
                        const uint32_t addr =
                            bias_row + box * kBiasBox + ((cc ^ (r & 7)) << 4);
                        uint32_t w0, w1, w2, w3;
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                                     : "r"(addr));
                        const uint32_t wv[4] = {w0, w1, w2, w3};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            x[8 * ch + 2 * q] =
                                fmaf(x[8 * ch + 2 * q], p.qk_scale, __uint_as_float(wv[q] << 16));
                            x[8 * ch + 2 * q + 1] = fmaf(x[8 * ch + 2 * q + 1], p.qk_scale,
                                                         __uint_as_float(wv[q] & 0xFFFF0000u));
                        }
                    }
                }
                if (!((j0 >= tr.full_lo) && (j0 + BN <= tr.full_hi)))
                    apply_row_mask(x, j0, row_lo, row_hi);
                if constexpr (KMASK) {
                    // word w bit l: key j0 + 32 w + l is kept
                    uint32_t bits[4], all = ~0u;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        bits[w] = __ballot_sync(0xffffffffu, keep[w] != 0u);
                        all &= bits[w];
                    }
                    if (all != ~0u) {
#pragma unroll
                        for (int e = 0; e < BN; ++e)
                            if (!((bits[e >> 5] >> (e & 31)) & 1u))
                                x[e] = kNegInf;
                    }
                }
                uint32_t pk[BN / 2];
                bool rescale;
                const float alpha =
                    LSE ? softmax_compute_p_exact_sum(x, c, st, j == 0, pk, rescale)
                        : softmax_compute_p_no_sum(x, c, st, j == 0, pk, rescale);
                if (j > 0 || pending) {
                    // the previous P V of this slot has consumed P[t] and
                    // landed in O[t]
                    if (!warp_wait(bar(sm.pv_done[t]), pvcount & 1, cx.wc, W_O_FULL))
                        return;
                    ++pvcount;
                    ptx::tc_fence_after();
                    if (j > 0) {
                        if (rescale)
                            rescale_o<kDvExt>(tO, alpha);
                    } else {
                        store_row_output<LSE>(p, tO, prev, r, nkv);
                        pending = false;
                    }
                }
                if (j == 0 && i < S) {
                    // bring this row's 64 gate bytes into L1 for its (deferred) epilogue
                    const __nv_bfloat16 *gp =
                        p.gate + b * p.g_sb + static_cast<int64_t>(i) * p.g_si + it.h * p.g_sh;
                    asm volatile("prefetch.global.L1 [%0];" ::"l"(gp));
                }
                store_p(tP, pk);
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(sm.p_full[t]));
            }
            prev.b = b;
            prev.h = it.h;
            prev.qb = it.qb;
            prev.i = i;
            prev.st = st;
            pending = true;
        }
        if (BIAS)
            ptx::mbar_arrive(bar(sm.bias_empty)); // this warpgroup is done with the bias rows
    }
    if (pending) {
        if (!warp_wait(bar(sm.o_final[t]), 0, cx.wc, W_O_FULL))
            return;
        ptx::tc_fence_after();
        store_row_output<LSE>(p, tO, prev, r, nkv);
    }
}

template <bool BIAS, bool LSE, bool KMASK>
__global__ void __launch_bounds__(kThreads, 1)
    evo_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_b,
                   const EvoParams p)
{
    constexpr int NS = EvoCfg<BIAS>::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    EvoSmem<BIAS> *sm = reinterpret_cast<EvoSmem<BIAS> *>(smem_raw + ((1024u - (base & 1023u)) & 1023u));
    const int warp = threadIdx.x >> 5;

    // the ones tile (bf16 1.0 pairs), read by the tensor core through the async proxy
    for (uint32_t w = threadIdx.x; w < kTile / 4; w += kThreads)
        reinterpret_cast<uint32_t *>(sm->ones)[w] = 0x3F803F80u;
    ptx::fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            for (int b = 0; b < 2; ++b) {
                ptx::mbar_init(bar(sm->q_full[t][b]), 1);
                ptx::mbar_init(bar(sm->q_empty[t][b]), 1);
            }
            for (int s = 0; s < NS; ++s) {
                ptx::mbar_init(bar(sm->kv_full[t][s]), 1);
                ptx::mbar_init(bar(sm->kv_empty[t][s]), 1);
            }
            ptx::mbar_init(bar(sm->s_full[t]), 1);
            ptx::mbar_init(bar(sm->s_free[t]), 128);
            ptx::mbar_init(bar(sm->p_full[t]), 128);
            ptx::mbar_init(bar(sm->pv_done[t]), 1);
            ptx::mbar_init(bar(sm->o_final[t]), 1);
        }
        ptx::mbar_init(bar(sm->s_final), 1);
        ptx::mbar_init(bar(sm->bias_full), 1);
        ptx::mbar_init(bar(sm->bias_empty), 256);
        sm->abort_flag = 0;
        ptx::fence_mbarrier_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0 && ptx::lane_id() == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        if (BIAS)
            ptx::prefetch_tensormap(&tm_b);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&sm->tmem_base), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    Ctx<BIAS> cx;
    cx.sm = sm;
    cx.tmem = sm->tmem_base;
    cx.wc.abort_flag = &sm->abort_flag;
    cx.wc.timeout_cycles = p.timeout_ns * 21 / 10; // 2.1 cycles per ns at the maximum clock
    cx.wc.err_user = p.err_user;
    cx.wc.err_lib = &g_lib_error_word;

    // Each branch ends with its own copy of the teardown barrier, so no code
    // runs under both register limits.
    if (warp >= 4) {
        ptx::setmaxnreg_inc<kRegsSoftmax>();
        softmax_role<BIAS, LSE, KMASK>(cx, p, (warp >> 2) - 1);
        ptx::tc_fence_before();
        ptx::named_barrier_sync(1, kThreads);
    } else {
        ptx::setmaxnreg_dec<kRegsOther>();
        if (warp == 0)
            producer_role<BIAS>(cx, p, &tm_q, &tm_k, &tm_v, &tm_b);
        else if (warp == 1)
            s_role<BIAS>(cx, p);
        else
            pv_role<BIAS>(cx, p, warp - 2);
        ptx::tc_fence_before();
        ptx::named_barrier_sync(1, kThreads);
        if (warp == 1) {
            ptx::tc_fence_after();
            ptx::tmem_dealloc(cx.tmem, 512);
        }
    }
}

template <bool BIAS, bool LSE, bool KMASK>
cudaError_t launch_variant(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const CUtensorMap &tb, const EvoParams &p, int grid, cudaStream_t stream)
{
    const size_t smem = sizeof(EvoSmem<BIAS>) + 1024;
    static bool configured = false; // benign race: both calls are idempotent
    if (!configured) {
        cudaFuncAttributes attr;
        cudaError_t e = cudaFuncGetAttributes(&attr, evo_fwd_kernel<BIAS, LSE, KMASK>);
        if (e != cudaSuccess)
            return e;
        // The setmaxnreg split assumes exactly kRegsLaunch registers at launch.
        if (attr.numRegs != static_cast<int>(kRegsLaunch))
            return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(evo_fwd_kernel<BIAS, LSE, KMASK>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    evo_fwd_kernel<BIAS, LSE, KMASK><<<grid, kThreads, smem, stream>>>(tq, tk, tv, tb, p);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_evo(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tb, const EvoParams &p, int grid, cudaStream_t stream)
{
    if (p.kmask) {
        if (p.bias)
            return p.lse ? launch_variant<true, true, true>(tq, tk, tv, tb, p, grid, stream)
                         : launch_variant<true, false, true>(tq, tk, tv, tb, p, grid, stream);
        return p.lse ? launch_variant<false, true, true>(tq, tk, tv, tb, p, grid, stream)
                     : launch_variant<false, false, true>(tq, tk, tv, tb, p, grid, stream);
    }
    if (p.bias)
        return p.lse ? launch_variant<true, true, false>(tq, tk, tv, tb, p, grid, stream)
                     : launch_variant<true, false, false>(tq, tk, tv, tb, p, grid, stream);
    return p.lse ? launch_variant<false, true, false>(tq, tk, tv, tb, p, grid, stream)
                 : launch_variant<false, false, false>(tq, tk, tv, tb, p, grid, stream);
}

int evo_max_bias_keys() { return kMaxBiasBoxes * 64; }

} // namespace fl
