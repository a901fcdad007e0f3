// fwd_diff.cu -- differential attention forward, D = 64, Dv = 64 or 128:
//     O = softmax(scale Q1 K1^T) V - lambda softmax(scale Q2 K2^T) V
// with both softmax streams fused in one kernel and sharing every V tile
// (the pages name differential attention among the variants that template
// systems cannot express: gist.science summary, "Results"; talk notes,
// "Evaluation: complex variants").  Masks: none or causal.
//
// CTA organisation (persistent: one CTA per SM, 384 threads).  A work item is
// one 128-row query block of one (batch, head); its two softmax streams see
// the same key tiles, with K tiles of their own and one shared V tile:
//   warp  0     TMA producer: Q1 and Q2 once per item (double-buffered across
//               items), then per key tile K1, K2 and V through a ring of
//               kStages mbarrier-guarded stages
//   warp  1     issues S_s = Q_s K_s^T for both streams; owns TMEM
//   warps 2, 3  issue O_s += P_s V for stream 0 and stream 1
//   warps 4-7   online softmax of stream 0 (one thread per query row)
//   warps 8-11  online softmax of stream 1
// The softmax warpgroups take turns on the exponential phase (mask, max, P,
// sums), so one stream's exponentials run while the tensor core works on the
// other stream's products.  P has TMEM columns of its own, so a stream's next
// S is issued as soon as its softmax has copied the scores out.
//
// TMEM per stream s (DiffCfg):
//   Dv = 64:  key tiles of 112 keys.  S at 112 s, O at 224 + 80 s (64 output
//             columns and a 16-column block holding sum_j P_j: the P V product
//             multiplies P by V extended with a tile of ones, so O's normaliser
//             is the sum of exactly the rounded P it weighed), P at 384 + 56 s.
//   Dv = 128: key tiles of 80 keys.  S at 80 s, O at 160 + 128 s, P at 416 + 40 s;
//             no room for sum columns, so each thread keeps the sum of its
//             rounded P and the two streams exchange theirs through shared
//             memory for the epilogue.
// Epilogue: when both streams' last P V has landed, warpgroup s writes output
// columns [s Dv / 2, (s + 1) Dv / 2) as O_1 / l_1 - lambda O_2 / l_2 from both
// streams' TMEM, then releases both O for the next item (o_free).
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
constexpr uint32_t kSmemLimit = 232448; // 227 KB per CTA

// Tile shapes, shared-memory sizes and TMEM columns per value head dimension.
template <int DV>
struct DiffCfg {
    static_assert(DV == 64 || DV == 128, "value head dimension");
    static constexpr int kBN = diff_key_tile(DV);       // keys per K/V tile
    static constexpr bool kOnes = DV == 64;              // row sum from the ones columns
    static constexpr int kVHalves = DV / 64;             // 64-column halves of a V row
    static constexpr uint32_t kQBytes = BM * 128;        // one 128 x 64 bf16 Q tile
    static constexpr uint32_t kKBytes = kBN * 128;       // one kBN x 64 bf16 K tile
    static constexpr uint32_t kVHalf = kBN * 128;        // one kBN x 64 half of a V tile
    static constexpr uint32_t kStageBytes = 2 * kKBytes + kVHalves * kVHalf;
    static constexpr uint32_t kOnesBytes = kOnes ? kQBytes : 16;
    // Q buffers, ones tile, row-sum exchange, barriers and the alignment pad
    static constexpr uint32_t kFixed = 4 * kQBytes + kOnesBytes + 2 * BM * 4 + 1024 + 1024;
    static constexpr int kStagesFit = static_cast<int>((kSmemLimit - kFixed) / kStageBytes);
    static constexpr int kStages = kStagesFit > 4 ? 4 : kStagesFit;
    static_assert(kStages >= 2, "K/V ring");
    static constexpr uint32_t kDvExt = kOnes ? DV + 16 : DV; // O columns (with the sum block)
    static constexpr uint32_t kColS = 0, kStrideS = kBN;
    static constexpr uint32_t kColO = 2 * kBN, kStrideO = kDvExt;
    static constexpr uint32_t kColP = kColO + 2 * kDvExt, kStrideP = kBN / 2;
    static_assert(kColP + 2 * kStrideP <= 512, "TMEM budget");
    static_assert(kBN % 16 == 0 && kBN <= 128, "key tile");
    static_assert(kBN * 128 <= kOnesBytes || !kOnes, "ones tile covers a key tile");
};

template <int DV>
struct __align__(1024) DiffSmem {
    using C = DiffCfg<DV>;
    uint8_t q[2][2][C::kQBytes];                  // [Q buffer][stream]
    uint8_t k[C::kStages][2][C::kKBytes];         // [stage][stream]
    uint8_t v[C::kStages][C::kVHalves][C::kVHalf];
    uint8_t ones[C::kOnesBytes];                  // bf16 1.0 everywhere: V's extra columns
                                                  // (Dv = 64; after every V stage)
    float lx[2][BM];                              // Dv = 128: each stream's rounded row sums
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[C::kStages], kv_empty[C::kStages];
    uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
    uint64_t turn[2];                             // exponential-phase token of each warpgroup
    uint64_t o_full[2], o_free, l_full;
    uint64_t final_bar[3];
    uint32_t tmem_base;
    uint32_t abort_flag;
};

__device__ uint32_t g_lib_error_word;

template <int DV>
struct Ctx {
    DiffSmem<DV> *sm;
    uint32_t tmem;
    WaitCtl wc;
};

__device__ __forceinline__ uint32_t bar(const uint64_t &b) { return ptx::smem_u32(&b); }

struct DiffItem {
    int b, h, kvh, qb;
};

__device__ __forceinline__ DiffItem decode(const DiffParams &p, int64_t L)
{
    const int Hx = p.B * p.H;
    int r, hx;
    if (p.lpt) {
        r = p.nq - 1 - static_cast<int>(L / Hx);
        hx = static_cast<int>(L % Hx);
    } else {
        const int64_t per_strip = static_cast<int64_t>(p.group) * p.nq;
        const int strip = static_cast<int>(L / per_strip);
        const int h0 = strip * p.group;
        const int gs = min(p.group, Hx - h0);
        const int w = static_cast<int>(L - strip * per_strip);
        r = w / gs;
        hx = h0 + w % gs;
    }
    DiffItem it;
    it.b = hx / p.H;
    it.h = hx % p.H;
    it.kvh = it.h / p.G;
    it.qb = r;
    return it;
}

// ------------------------------------------------------------------ producer
template <int DV>
__device__ void producer_role(const Ctx<DV> &cx, const DiffParams &p, const CUtensorMap *tm_q,
                              const CUtensorMap *tm_k, const CUtensorMap *tm_v)
{
    using C = DiffCfg<DV>;
    constexpr int NS = C::kStages, kBN = C::kBN;
    DiffSmem<DV> &sm = *cx.sm;
    const uint32_t lane = ptx::lane_id();
    uint32_t kv_count = 0, item_count = 0;
    bool ok = true;
    for (int64_t L = blockIdx.x; L < p.n_items && ok; L += gridDim.x, ++item_count) {
        const DiffItem it = decode(p, L);
        const TileRange tr = q_block_range<kBN>(p.mask, it.b, it.qb * BM);
        const uint32_t qbuf = item_count & 1;
        if (item_count >= 2) {
            ok = warp_wait(bar(sm.q_empty[qbuf]), ((item_count - 2) >> 1) & 1, cx.wc, W_Q_EMPTY);
            if (!ok)
                break;
        }
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(sm.q_full[qbuf]), 2 * C::kQBytes);
            for (int s = 0; s < 2; ++s)
                ptx::tma_load_5d(ptx::smem_u32(sm.q[qbuf][s]), tm_q, bar(sm.q_full[qbuf]), 0, it.qb * BM,
                                 it.h, it.b, s);
        }
        __syncwarp();
        for (int j = tr.lo; j < tr.hi; ++j, ++kv_count) {
            const uint32_t st = kv_count % NS;
            ok = warp_wait(bar(sm.kv_empty[st]), ((kv_count / NS) & 1) ^ 1, cx.wc, W_KV_EMPTY);
            if (!ok)
                break;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bar(sm.kv_full[st]), C::kStageBytes);
                for (int s = 0; s < 2; ++s)
                    ptx::tma_load_5d(ptx::smem_u32(sm.k[st][s]), tm_k, bar(sm.kv_full[st]), 0, j * kBN,
                                     it.kvh, it.b, s);
                for (int hf = 0; hf < C::kVHalves; ++hf)
                    ptx::tma_load_4d(ptx::smem_u32(sm.v[st][hf]), tm_v, bar(sm.kv_full[st]), 64 * hf,
                                     j * kBN, it.kvh, it.b);
            }
            __syncwarp();
        }
    }
    if (!ok) {
        // wait (bounded, ignoring the abort) for this warp's own loads in flight
        const uint32_t first = kv_count > NS ? kv_count - NS : 0;
        for (uint32_t idx = first; idx < kv_count; ++idx)
            mbar_wait_drain(bar(sm.kv_full[idx % NS]), (idx / NS) & 1, cx.wc, W_DRAIN);
        for (uint32_t n = item_count > 2 ? item_count - 2 : 0; n < item_count; ++n)
            mbar_wait_drain(bar(sm.q_full[n & 1]), (n >> 1) & 1, cx.wc, W_DRAIN);
    }
}

// ------------------------------------------------------------------ MMA issuers
//
// S warp: per key tile, S_0 = Q_1 K_{1,j}^T, then S_1 = Q_2 K_{2,j}^T, each
// once its softmax has copied the stream's previous scores out of TMEM
// (s_free).  A K/V stage is released by the two P V warps' commits: S_s(j)
// completes before its softmax can publish P_s(j), so the commit after
// P_s V_j also covers the read of K_{s,j}.  A Q buffer is released by the S
// warp's commit after the item's last S (a commit covers every earlier MMA of
// its thread).
template <int DV>
__device__ void s_role(const Ctx<DV> &cx, const DiffParams &p)
{
    using C = DiffCfg<DV>;
    constexpr int NS = C::kStages, kBN = C::kBN;
    DiffSmem<DV> &sm = *cx.sm;
    const uint32_t lane = ptx::lane_id();
    constexpr uint32_t idesc_qk = umma_idesc_bf16(BM, kBN, false);
    constexpr uint64_t kHiK = umma_desc_hi(16, 1024, kSwizzle128B); // Q, K: K-major, 128-byte rows
    uint32_t kv_count = 0, item_count = 0;
    uint32_t issued[2] = {0u, 0u};
    bool ok = true;
    for (int64_t L = blockIdx.x; L < p.n_items && ok; L += gridDim.x, ++item_count) {
        const DiffItem it = decode(p, L);
        const TileRange tr = q_block_range<kBN>(p.mask, it.b, it.qb * BM);
        const uint32_t qbuf = item_count & 1;
        ok = warp_wait(bar(sm.q_full[qbuf]), (item_count >> 1) & 1, cx.wc, W_Q_FULL);
        for (int j = tr.lo; j < tr.hi && ok; ++j, ++kv_count) {
            const uint32_t st = kv_count % NS;
            ok = warp_wait(bar(sm.kv_full[st]), (kv_count / NS) & 1, cx.wc, W_KV_FULL);
#pragma unroll
            for (int s = 0; s < 2 && ok; ++s) {
                if (issued[s] > 0) {
                    ok = warp_wait(bar(sm.s_free[s]), (issued[s] - 1) & 1, cx.wc, W_S_FULL);
                    if (!ok)
                        break;
                }
                ++issued[s];
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t qlo = ptx::smem_u32(sm.q[qbuf][s]) >> 4;
                    const uint32_t klo = ptx::smem_u32(sm.k[st][s]) >> 4;
                    const uint32_t tS = cx.tmem + C::kColS + C::kStrideS * s;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) // 16 features (32 bytes) per step
                        ptx::mma_ss(tS, kHiK | (qlo + 2 * kk), kHiK | (klo + 2 * kk), idesc_qk,
                                    kk > 0 ? 1u : 0u);
                    ptx::mma_commit(bar(sm.s_full[s]));
                    if (s == 1 && j + 1 == tr.hi)
                        ptx::mma_commit(bar(sm.q_empty[qbuf])); // the item's last read of this Q buffer
                }
                __syncwarp();
            }
        }
    }
    // Every MMA this thread issued has completed before TMEM is released.
    const uint32_t b_final = bar(sm.final_bar[0]);
    if (lane == 0)
        ptx::mma_commit(b_final);
    __syncwarp();
    mbar_wait_drain(b_final, 0, cx.wc, W_FINAL);
}

// P V warp of stream s: O_s += P_s [V_j | 1] (Dv = 64) or O_s += P_s V_j
// (Dv = 128).  An item's first P V (which overwrites O_s) waits until the
// previous item's epilogue has read both streams' O (o_free); the item's last
// commits o_full[s].
template <int DV>
__device__ void pv_role(const Ctx<DV> &cx, const DiffParams &p, int s)
{
    using C = DiffCfg<DV>;
    constexpr int NS = C::kStages, kBN = C::kBN;
    DiffSmem<DV> &sm = *cx.sm;
    const uint32_t lane = ptx::lane_id();
    constexpr uint32_t idesc_pv = umma_idesc_bf16(BM, C::kDvExt, true);
    const uint32_t ones_lo = ptx::smem_u32(sm.ones) >> 4;
    const uint32_t tO = cx.tmem + C::kColO + C::kStrideO * s;
    const uint32_t tP = cx.tmem + C::kColP + C::kStrideP * s;
    uint32_t kv_count = 0, pcount = 0, item_count = 0;
    bool ok = true;
    for (int64_t L = blockIdx.x; L < p.n_items && ok; L += gridDim.x, ++item_count) {
        const DiffItem it = decode(p, L);
        const TileRange tr = q_block_range<kBN>(p.mask, it.b, it.qb * BM);
        for (int j = tr.lo; j < tr.hi && ok; ++j, ++kv_count) {
            ok = warp_wait(bar(sm.p_full[s]), pcount & 1, cx.wc, W_P_FULL);
            if (ok && j == tr.lo && item_count > 0)
                ok = warp_wait(bar(sm.o_free), (item_count - 1) & 1, cx.wc, W_O_FULL);
            if (!ok)
                break;
            ++pcount;
            ptx::tc_fence_after();
            if (lane == 0) {
                const uint32_t st = kv_count % NS;
                const uint32_t vlo = ptx::smem_u32(sm.v[st][0]) >> 4;
                // V's second 64-column block is LBO bytes away: the ones tile
                // (Dv = 64, of which the MMA reads 16 columns) or V's second half
                const uint32_t lbo = C::kOnes ? (ones_lo - vlo) << 4 : C::kVHalf;
                const uint64_t hi_v = umma_desc_hi(lbo, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) // 16 keys (2048 bytes of V) per step
                    ptx::mma_ts(tO, tP + 8 * kk, hi_v | (vlo + 128 * kk), idesc_pv,
                                (j > tr.lo || kk > 0) ? 1u : 0u);
                ptx::mma_commit(bar(sm.pv_done[s]));
                ptx::mma_commit(bar(sm.kv_empty[st])); // this stream is done with stage st
                if (j + 1 == tr.hi)
                    ptx::mma_commit(bar(sm.o_full[s]));
            }
            __syncwarp();
        }
    }
    const uint32_t b_final = bar(sm.final_bar[1 + s]);
    if (lane == 0)
        ptx::mma_commit(b_final);
    __syncwarp();
    mbar_wait_drain(b_final, 0, cx.wc, W_FINAL);
}

// ------------------------------------------------------------------ softmax
//
// Turn k of warpgroup 1 follows warpgroup 0's turn k; turn k > 0 of
// warpgroup 0 follows warpgroup 1's turn k - 1; warpgroup 0's first turn is
// free.  Both streams visit the same key tiles, so both take the same turns.
// Every query block has at least one key tile (masks none and causal).
template <int DV>
__device__ void softmax_role(const Ctx<DV> &cx, const DiffParams &p, int s)
{
    using C = DiffCfg<DV>;
    constexpr int kBN = C::kBN;
    DiffSmem<DV> &sm = *cx.sm;
    const int r = threadIdx.x & 127; // row of the query block = TMEM lane
    const uint32_t lane_off = (((threadIdx.x >> 5) & 3u) * 32u) << 16;
    const uint32_t tS = cx.tmem + lane_off + C::kColS + C::kStrideS * s;
    const uint32_t tP = cx.tmem + lane_off + C::kColP + C::kStrideP * s;
    const uint32_t tO0 = cx.tmem + lane_off + C::kColO;
    const uint32_t tO1 = tO0 + C::kStrideO;
    const uint32_t tOs = s == 0 ? tO0 : tO1;
    const uint32_t b_turn_mine = bar(sm.turn[s]), b_turn_other = bar(sm.turn[s ^ 1]);
    uint32_t scount = 0, pvcount = 0, turns = 0, item_count = 0;

    for (int64_t L = blockIdx.x; L < p.n_items; L += gridDim.x, ++item_count) {
        const DiffItem it = decode(p, L);
        const TileRange tr = q_block_range<kBN>(p.mask, it.b, it.qb * BM);
        const int i = it.qb * BM + r;
        int row_lo, row_hi;
        row_interval(p.mask, it.b, i, row_lo, row_hi);
        const int n_tiles = tr.hi - tr.lo;
        RowState st{kNegInf, 0.f, 0.f};
        for (int kk = 0; kk < n_tiles; ++kk, ++turns) {
            const int j = tr.lo + kk;
            if (!warp_wait(bar(sm.s_full[s]), scount & 1, cx.wc, W_S_FULL))
                return;
            ++scount;
            ptx::tc_fence_after();
            float x[kBN];
            load_scores<kBN>(tS, x);
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(sm.s_free[s])); // S_s may be overwritten
            if (!(s == 0 && turns == 0) &&
                !warp_wait(b_turn_mine, (s == 1 ? turns : turns - 1) & 1, cx.wc, W_TURN))
                return;
            const int j0 = j * kBN;
            if (!((j0 >= tr.full_lo) && (j0 + kBN <= tr.full_hi)))
                apply_row_mask<kBN>(x, j0, row_lo, row_hi);
            uint32_t pk[kBN / 2];
            bool rescale;
            const float alpha = C::kOnes
                                    ? softmax_compute_p_exact_sum<kBN>(x, p.qk_log2, st, kk == 0, pk, rescale)
                                    : softmax_compute_p<kBN>(x, p.qk_log2, st, kk == 0, pk, rescale);
            ptx::mbar_arrive(b_turn_other); // hand the turn over
            if (kk > 0) {
                // the previous tile's P V has consumed P_s and landed in O_s
                if (!warp_wait(bar(sm.pv_done[s]), pvcount & 1, cx.wc, W_O_FULL))
                    return;
                ++pvcount;
                ptx::tc_fence_after();
                if (rescale)
                    rescale_o<C::kDvExt>(tOs, alpha);
            }
            store_p<kBN>(tP, pk);
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(sm.p_full[s]));
        }

        // epilogue: this stream's last P V, then the other stream's (o_full)
        if (!warp_wait(bar(sm.pv_done[s]), pvcount & 1, cx.wc, W_O_FULL))
            return;
        ++pvcount;
        if (p.lse && i < p.mask.S)
            p.lse[s * p.l_s2 + it.b * p.l_sb + it.h * p.l_sh + i] = row_lse(st);
        if (p.tile_counts && s == 0 && r == 0)
            p.tile_counts[(static_cast<int64_t>(it.b) * p.H + it.h) * p.nq + it.qb] = n_tiles;
        if constexpr (!C::kOnes) {
            sm.lx[s][r] = st.l_round;
            ptx::mbar_arrive(bar(sm.l_full));
        }
        if (!warp_wait(bar(sm.o_full[s ^ 1]), item_count & 1, cx.wc, W_O_FULL))
            return;
        float l0, l1;
        if constexpr (C::kOnes) {
            ptx::tc_fence_after();
            uint32_t sum[2];
            ptx::tmem_ld1(tO0 + DV, sum); // the first sum column
            ptx::tmem_ld1(tO1 + DV, sum + 1);
            ptx::tmem_wait_ld();
            ptx::reg_fence<2>(sum);
            l0 = __uint_as_float(sum[0]);
            l1 = __uint_as_float(sum[1]);
        } else {
            if (!warp_wait(bar(sm.l_full), item_count & 1, cx.wc, W_O_FULL))
                return;
            ptx::tc_fence_after();
            l0 = sm.lx[0][r];
            l1 = sm.lx[1][r];
        }
        const float c0 = l0 > 0.f ? ptx::rcp_approx(l0) : 0.f;
        const float c1 = l1 > 0.f ? -p.lambda * ptx::rcp_approx(l1) : 0.f;
        __nv_bfloat16 *dst = p.out + it.b * p.o_sb + static_cast<int64_t>(i) * p.o_ss + it.h * p.o_sh +
                             (DV / 2) * s;
        // 32 of this warpgroup's output columns per round: both streams' TMEM
        // loads under one wait, the row written with 32-byte stores where aligned
#pragma unroll
        for (int c = 0; c < DV / 64; ++c) {
            uint32_t a[32], bb[32];
            ptx::tmem_ld32(tO0 + (DV / 2) * s + 32 * c, a);
            ptx::tmem_ld32(tO1 + (DV / 2) * s + 32 * c, bb);
            ptx::tmem_wait_ld();
            ptx::reg_fence<32>(a);
            ptx::reg_fence<32>(bb);
            if (i < p.mask.S) {
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float y0 = fmaf(__uint_as_float(a[2 * e]), c0, __uint_as_float(bb[2 * e]) * c1);
                    const float y1 =
                        fmaf(__uint_as_float(a[2 * e + 1]), c0, __uint_as_float(bb[2 * e + 1]) * c1);
                    w[e] = ptx::pack_bf16(y0, y1);
                }
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
                if ((reinterpret_cast<uint64_t>(d4) & 31u) == 0u) {
                    ptx::st_global_v8(d4, w);
                    ptx::st_global_v8(d4 + 2, w + 8);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        d4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                }
            }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(sm.o_free)); // both O may be overwritten by the next item
    }
}

template <int DV>
__global__ void __launch_bounds__(kThreads, 1)
    diff_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const DiffParams p)
{
    using C = DiffCfg<DV>;
    constexpr int NS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    DiffSmem<DV> *sm = reinterpret_cast<DiffSmem<DV> *>(smem_raw + ((1024u - (base & 1023u)) & 1023u));
    const int warp = threadIdx.x >> 5;

    // the ones tile (bf16 1.0 pairs), read by the tensor core through the async proxy
    if constexpr (C::kOnes) {
        for (uint32_t w = threadIdx.x; w < C::kOnesBytes / 4; w += kThreads)
            reinterpret_cast<uint32_t *>(sm->ones)[w] = 0x3F803F80u;
        ptx::fence_proxy_async_smem();
    }
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(sm->q_full[b]), 1);
            ptx::mbar_init(bar(sm->q_empty[b]), 1);
        }
        for (int st = 0; st < NS; ++st) {
            ptx::mbar_init(bar(sm->kv_full[st]), 1);
            ptx::mbar_init(bar(sm->kv_empty[st]), 2); // a commit per P V warp
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(bar(sm->s_full[s]), 1);
            ptx::mbar_init(bar(sm->s_free[s]), 128);
            ptx::mbar_init(bar(sm->p_full[s]), 128);
            ptx::mbar_init(bar(sm->pv_done[s]), 1);
            ptx::mbar_init(bar(sm->turn[s]), 128); // arrived by the other warpgroup
            ptx::mbar_init(bar(sm->o_full[s]), 1);
        }
        ptx::mbar_init(bar(sm->o_free), 256);
        ptx::mbar_init(bar(sm->l_full), 256);
        for (int b = 0; b < 3; ++b)
            ptx::mbar_init(bar(sm->final_bar[b]), 1);
        sm->abort_flag = 0;
        ptx::fence_mbarrier_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0 && ptx::lane_id() == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&sm->tmem_base), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    Ctx<DV> cx;
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
        softmax_role<DV>(cx, p, (warp >> 2) - 1);
        ptx::tc_fence_before();
        ptx::named_barrier_sync(1, kThreads);
    } else {
        ptx::setmaxnreg_dec<kRegsOther>();
        if (warp == 0)
            producer_role<DV>(cx, p, &tm_q, &tm_k, &tm_v);
        else if (warp == 1)
            s_role<DV>(cx, p);
        else
            pv_role<DV>(cx, p, warp - 2);
        ptx::tc_fence_before();
        ptx::named_barrier_sync(1, kThreads);
        if (warp == 1) {
            ptx::tc_fence_after();
            ptx::tmem_dealloc(cx.tmem, 512);
        }
    }
}

template <int DV>
cudaError_t launch_dv(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                      const DiffParams &p, int grid, cudaStream_t stream)
{
    // the layout plus the worst-case alignment pad within 227 KB per CTA
    static_assert(sizeof(DiffSmem<DV>) + 1024 <= kSmemLimit, "shared memory per CTA");
    const size_t smem = sizeof(DiffSmem<DV>) + 1024;
    static bool configured = false; // benign race: both calls are idempotent
    if (!configured) {
        cudaFuncAttributes attr;
        cudaError_t e = cudaFuncGetAttributes(&attr, diff_fwd_kernel<DV>);
        if (e != cudaSuccess)
            return e;
        // The setmaxnreg split assumes exactly kRegsLaunch registers at launch.
        if (attr.numRegs != static_cast<int>(kRegsLaunch))
            return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(diff_fwd_kernel<DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    diff_fwd_kernel<DV><<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_diff(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const DiffParams &p, int grid, cudaStream_t stream)
{
    return p.dv == 64 ? launch_dv<64>(tq, tk, tv, p, grid, stream)
                      : launch_dv<128>(tq, tk, tv, p, grid, stream);
}

} // namespace fl
