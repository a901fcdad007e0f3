// fwd_evo.cu -- Evoformer MSA gated self-attention forward, c = 32 per head:
//     O = sigmoid(g) * softmax(scale q k^T + b) v
// row-wise (attention over residues for each MSA row, pair bias b[h, i, j]
// shared by every MSA row) and column-wise (attention over MSA rows for each
// residue, no bias).  The pages evaluate both as complex variants template
// systems cannot express (talk notes, "Evaluation: complex variants" and
// "End-to-end: AlphaFold2": Evoformer with 8 heads of dimension 32); the gate
// is fused into the epilogue and the bias into the online softmax.
//
// The structure is that of the standard kernel (fwd_standard.cu): persistent
// CTAs of 384 threads, two 128-row query tiles ("slots") per work item sharing
// every K/V tile, one TMA producer warp, one MMA warp per slot that issues the
// next Q K^T as soon as its softmax has copied the scores out of TMEM, and two
// softmax warpgroups.  For c = 32 a tile row is 64 bytes, so Q/K/V use the
// 64-byte swizzle, Q K^T takes two 16-deep MMA steps and P V has N = 32.
// Both passes are the same kernel over a [batch, sequence, head, c] view:
// the row pass takes batch = MSA row and sequence = residue, the column pass
// the reverse (the host swaps the two strides).
//
// TMEM per slot t: S[t] fp32 at 128 t, O[t] fp32 (32 columns) at 256 + 32 t,
// P[t] bf16 pairs at 384 + 64 t.
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
constexpr int kStages = 6;
constexpr uint32_t kTileBytes = BM * 32 * 2; // one 128 x 32 bf16 tile
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;

struct __align__(1024) EvoSmem {
    uint8_t q[2][2][kTileBytes]; // [Q buffer][slot]
    uint8_t k[kStages][kTileBytes];
    uint8_t v[kStages][kTileBytes];
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
    uint64_t final_bar[2];
    uint32_t tmem_base;
    uint32_t abort_flag;
};

__device__ uint32_t g_lib_error_word;

struct KernelCtx {
    EvoSmem *sm;
    uint32_t tmem;
    WaitCtl wc;
};

__device__ __forceinline__ uint32_t bar(const uint64_t &b) { return ptx::smem_u32(&b); }

// ------------------------------------------------------------------ producer
__device__ void producer_role(const KernelCtx &cx, const EvoParams &p, const CUtensorMap *tm_q,
                              const CUtensorMap *tm_k, const CUtensorMap *tm_v)
{
    EvoSmem &sm = *cx.sm;
    const uint32_t lane = ptx::lane_id();
    uint32_t kv_count = 0, item_count = 0;
    int64_t dropped = -1;
    bool ok = true;
    for (int64_t L = blockIdx.x; L < p.grid.n_items && ok; L += gridDim.x) {
        const Item it = decode_item(p.grid, L);
        int lo = 1 << 30, hi = 0;
        int nvalid = 0;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (!it.valid[t])
                continue;
            const TileRange r = q_block_range(p.mask, it.b, it.qb[t] * BM);
            lo = min(lo, r.lo);
            hi = max(hi, r.hi);
            ++nvalid;
        }
        const uint32_t qbuf = item_count & 1;
        if (item_count >= 2) {
            ok = warp_wait(bar(sm.q_empty[qbuf]), ((item_count - 2) >> 1) & 1, cx.wc, W_Q_EMPTY);
            if (!ok)
                break;
        }
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(sm.q_full[qbuf]), nvalid * kTileBytes);
#pragma unroll
            for (int t = 0; t < 2; ++t)
                if (it.valid[t])
                    ptx::tma_load_4d(ptx::smem_u32(sm.q[qbuf][t]), tm_q, bar(sm.q_full[qbuf]), 0,
                                     it.qb[t] * BM, it.h[t], it.b);
        }
        __syncwarp();
        for (int j = lo; j < hi; ++j, ++kv_count) {
            const uint32_t s = kv_count % kStages;
            const uint32_t ph = (kv_count / kStages) & 1;
            ok = warp_wait(bar(sm.kv_empty[s]), ph ^ 1, cx.wc, W_KV_EMPTY);
            if (!ok)
                break;
            if (lane == 0) {
                const bool drop = p.inject == 1 && blockIdx.x == 0 && kv_count == 0;
                if (drop) {
                    dropped = kv_count;
                } else {
                    ptx::mbar_arrive_expect_tx(bar(sm.kv_full[s]), 2 * kTileBytes);
                    ptx::tma_load_4d(ptx::smem_u32(sm.k[s]), tm_k, bar(sm.kv_full[s]), 0, j * BN,
                                     it.kvh, it.b);
                    ptx::tma_load_4d(ptx::smem_u32(sm.v[s]), tm_v, bar(sm.kv_full[s]), 0, j * BN,
                                     it.kvh, it.b);
                }
            }
            __syncwarp();
        }
        ++item_count;
    }
    if (!ok) {
        // Drain: wait (bounded, ignoring the abort) for this warp's own loads in
        // flight so that no TMA write lands after the CTA has exited.
        dropped = __shfl_sync(0xffffffffu, dropped, 0);
        const uint32_t first = kv_count > kStages ? kv_count - kStages : 0;
        for (uint32_t idx = first; idx < kv_count; ++idx) {
            if (static_cast<int64_t>(idx) == dropped)
                continue;
            mbar_wait_drain(bar(sm.kv_full[idx % kStages]), (idx / kStages) & 1, cx.wc, W_DRAIN);
        }
        for (uint32_t n = item_count > 2 ? item_count - 2 : 0; n < item_count; ++n)
            mbar_wait_drain(bar(sm.q_full[n & 1]), (n >> 1) & 1, cx.wc, W_DRAIN);
    }
}

// ------------------------------------------------------------------ MMA issuers
//
// Two MMA warps, one per slot, so each slot's S -> softmax -> P V chain moves
// independently and the tensor core interleaves the two.  Each keeps its state
// in registers and builds descriptors as (constant high word) | (14-bit start
// address).  kv_empty and q_empty take one arrival from each warp: a warp
// commits after its last MMA reading the tile (or Q buffer), or -- for a tile
// its slot does not use -- arrives once the tile has landed, which proves the
// stage's previous phase is complete.
__device__ __forceinline__ bool wait_kv_tiles(const KernelCtx &cx, uint32_t bar_kvf0,
                                              uint32_t kv_base, int rel, int &waited)
{
    while (waited <= rel) {
        const uint32_t idx = kv_base + static_cast<uint32_t>(waited);
        if (!warp_wait(bar_kvf0 + (idx % kStages) * static_cast<uint32_t>(sizeof(uint64_t)),
                       (idx / kStages) & 1, cx.wc, W_KV_FULL))
            return false;
        ++waited;
    }
    return true;
}

__device__ void mma_role(const KernelCtx &cx, const EvoParams &p, int t)
{
    EvoSmem &sm = *cx.sm;
    const uint32_t lane = ptx::lane_id();
    constexpr uint32_t idesc_qk = umma_idesc_bf16(BM, BN, false);
    constexpr uint32_t idesc_pv = umma_idesc_bf16(BM, 32, true);
    constexpr uint64_t kHiK = umma_desc_hi(16, 512, kSwizzle64B);           // Q, K: K-major
    constexpr uint64_t kHiV = umma_desc_hi(kTileBytes, 512, kSwizzle64B);   // V: MN-major
    constexpr uint32_t kTileLo = kTileBytes >> 4;
    constexpr uint32_t kBarStride = sizeof(uint64_t);
    const uint32_t q_lo0 = ptx::smem_u32(sm.q[0][t]) >> 4;
    const uint32_t k_lo0 = ptx::smem_u32(sm.k[0]) >> 4;
    const uint32_t v_lo0 = ptx::smem_u32(sm.v[0]) >> 4;
    const uint32_t tS = cx.tmem + kColS + 128 * t, tO = cx.tmem + kColO + 32 * t;
    const uint32_t tP = cx.tmem + kColP + 64 * t;
    const uint32_t b_sfull = bar(sm.s_full[t]), b_sfree = bar(sm.s_free[t]);
    const uint32_t b_pfull = bar(sm.p_full[t]), b_pvdone = bar(sm.pv_done[t]);
    const uint32_t b_kvf0 = bar(sm.kv_full[0]), b_kve0 = bar(sm.kv_empty[0]);

    uint32_t kv_base = 0, item_count = 0, fcount = 0, pcount = 0;
    bool ok = true;
    for (int64_t L = blockIdx.x; L < p.grid.n_items && ok; L += gridDim.x) {
        const Item it = decode_item(p.grid, L);
        int lo = 1 << 30, hi = 0, lot = 0, hit = 0;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (!it.valid[u])
                continue;
            const TileRange r = q_block_range(p.mask, it.b, it.qb[u] * BM);
            lo = min(lo, r.lo);
            hi = max(hi, r.hi);
            if (u == t) {
                lot = r.lo;
                hit = r.hi;
            }
        }
        const bool active = it.valid[t];
        const uint32_t qbuf = item_count & 1;
        const uint32_t b_qe = bar(sm.q_empty[qbuf]);
        ok = warp_wait(bar(sm.q_full[qbuf]), (item_count >> 1) & 1, cx.wc, W_Q_FULL);
        if (!ok)
            break;
        ptx::tc_fence_after();
        const uint32_t qlo = q_lo0 + qbuf * 2 * kTileLo;
        int waited = 0;

        for (int j = lo; j < hi && ok; ++j) {
            const uint32_t stage_j = (kv_base + (j - lo)) % kStages;
            if (!active || j < lot || j >= hit) {
                // tile not used by this slot: release it once it has landed
                if (!(ok = wait_kv_tiles(cx, b_kvf0, kv_base, j - lo, waited)))
                    break;
                if (lane == 0)
                    ptx::mbar_arrive(b_kve0 + stage_j * kBarStride);
                __syncwarp();
                continue;
            }
            if (j == lot) {
                // first S of the item for this slot
                if (!(ok = wait_kv_tiles(cx, b_kvf0, kv_base, j - lo, waited)))
                    break;
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t klo = k_lo0 + stage_j * kTileLo;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        ptx::mma_ss(tS, kHiK | (qlo + 2 * kk), kHiK | (klo + 2 * kk), idesc_qk,
                                    kk > 0 ? 1u : 0u);
                    ptx::mma_commit(b_sfull);
                    if (j + 1 == hit)
                        ptx::mma_commit(b_qe); // last read of this Q buffer
                }
                __syncwarp();
            }
            // the softmax has copied S(j) out of TMEM: issue S(j + 1)
            ok = warp_wait(b_sfree, fcount & 1, cx.wc, W_S_FULL);
            if (!ok)
                break;
            ++fcount;
            if (j + 1 < hit) {
                if (!(ok = wait_kv_tiles(cx, b_kvf0, kv_base, j + 1 - lo, waited)))
                    break;
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t klo = k_lo0 + ((kv_base + (j + 1 - lo)) % kStages) * kTileLo;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        ptx::mma_ss(tS, kHiK | (qlo + 2 * kk), kHiK | (klo + 2 * kk), idesc_qk,
                                    kk > 0 ? 1u : 0u);
                    ptx::mma_commit(b_sfull);
                    if (j + 2 == hit)
                        ptx::mma_commit(b_qe);
                }
                __syncwarp();
            }
            // the softmax has written P(j) and rescaled O: issue P V(j)
            ok = warp_wait(b_pfull, pcount & 1, cx.wc, W_P_FULL);
            if (!ok)
                break;
            ++pcount;
            ptx::tc_fence_after();
            if (lane == 0) {
                const uint32_t vlo = v_lo0 + stage_j * kTileLo;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    ptx::mma_ts(tO, tP + 8 * kk, kHiV | (vlo + 64 * kk), idesc_pv,
                                (j > lot || kk > 0) ? 1u : 0u);
                ptx::mma_commit(b_pvdone);
                ptx::mma_commit(b_kve0 + stage_j * kBarStride); // this slot is done with tile j
            }
            __syncwarp();
        }
        if (!ok)
            break;
        if (!active) {
            if (lane == 0)
                ptx::mbar_arrive(b_qe);
            __syncwarp();
        }
        kv_base += static_cast<uint32_t>(hi - lo);
        ++item_count;
    }
    // Every MMA this thread issued has completed before TMEM is released.
    const uint32_t b_final = bar(sm.final_bar[t]);
    if (lane == 0)
        ptx::mma_commit(b_final);
    __syncwarp();
    mbar_wait_drain(b_final, 0, cx.wc, W_FINAL);
}

// ------------------------------------------------------------------ softmax
template <bool BIAS>
__device__ void softmax_role(const KernelCtx &cx, const EvoParams &p, int t)
{
    EvoSmem &sm = *cx.sm;
    const int r = threadIdx.x & 127;             // row of the query tile = TMEM lane
    const uint32_t wq = (threadIdx.x >> 5) & 3;  // warp's quarter of the lanes
    const uint32_t lane_off = (wq * 32u) << 16;
    const uint32_t tS = cx.tmem + lane_off + kColS + 128 * t;
    const uint32_t tO = cx.tmem + lane_off + kColO + 32 * t;
    const uint32_t tP = cx.tmem + lane_off + kColP + 64 * t;
    const int S = p.mask.S;
    uint32_t scount = 0, pvcount = 0;

    for (int64_t L = blockIdx.x; L < p.grid.n_items; L += gridDim.x) {
        const Item it = decode_item(p.grid, L);
        if (!it.valid[t])
            continue;
        const int b = it.b, h = it.h[t], qb = it.qb[t];
        const int i = qb * BM + r;
        const TileRange tr = q_block_range(p.mask, b, qb * BM);
        int row_lo, row_hi;
        row_interval(p.mask, b, i, row_lo, row_hi);
        const __nv_bfloat16 *brow = nullptr;
        if constexpr (BIAS)
            brow = p.bias + h * p.bias_sh + static_cast<int64_t>(min(i, S - 1)) * p.bias_si;

        RowState st{kNegInf, 0.f, 0.f};
        int ntiles = 0;
        for (int j = tr.lo; j < tr.hi; ++j) {
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
                // natural-unit logits scale q.k + b[h, i, j]; log2 e goes into
                // the exponent.  The bias row segment is read from global
                // memory (it stays in L2: every MSA row reads the same bias).
                c = kLog2e;
#pragma unroll
                for (int ch = 0; ch < BN / 8; ++ch) {
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    const int k0 = j0 + 8 * ch;
                    if (k0 + 8 <= S) {
                        w = __ldg(reinterpret_cast<const uint4 *>(brow + k0));
                    } else if (k0 < S) {
                        uint32_t e4[4] = {0u, 0u, 0u, 0u};
                        for (int e = 0; e < 8 && k0 + e < S; ++e) {
                            const uint32_t bits = __ldg(reinterpret_cast<const unsigned short *>(brow + k0 + e));
                            e4[e >> 1] |= bits << (16 * (e & 1));
                        }
                        w = make_uint4(e4[0], e4[1], e4[2], e4[3]);
                    }
                    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        x[8 * ch + 2 * q] = fmaf(x[8 * ch + 2 * q], p.qk_scale, __uint_as_float(wv[q] << 16));
                        x[8 * ch + 2 * q + 1] =
                            fmaf(x[8 * ch + 2 * q + 1], p.qk_scale, __uint_as_float(wv[q] & 0xFFFF0000u));
                    }
                }
            }
            if (!((j0 >= tr.full_lo) && (j0 + BN <= tr.full_hi)))
                apply_row_mask(x, j0, row_lo, row_hi);
            uint32_t pk[BN / 2];
            bool rescale;
            const float alpha = softmax_compute_p(x, c, st, j == tr.lo, pk, rescale);
            if (j > tr.lo) {
                // the previous tile's P V has consumed P[t] and landed in O[t]
                if (!warp_wait(bar(sm.pv_done[t]), pvcount & 1, cx.wc, W_O_FULL))
                    return;
                ++pvcount;
                ptx::tc_fence_after();
                if (rescale)
                    rescale_o<32>(tO, alpha);
            }
            store_p(tP, pk);
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(sm.p_full[t]));
            ++ntiles;
        }

        // epilogue: sigmoid(g) * O / l -> bf16, LSE
        if (!warp_wait(bar(sm.pv_done[t]), pvcount & 1, cx.wc, W_O_FULL))
            return;
        ++pvcount;
        ptx::tc_fence_after();
        uint32_t o[32];
        ptx::tmem_ld32(tO, o);
        ptx::tmem_wait_ld();
        ptx::reg_fence<32>(o);
        const float inv = row_inv_norm(st);
        if (i < S) {
            const int64_t off = b * p.g_sb + static_cast<int64_t>(i) * p.g_si + h * p.g_sh;
            const uint4 *g4 = reinterpret_cast<const uint4 *>(p.gate + off);
            uint4 *d4 = reinterpret_cast<uint4 *>(p.out + b * p.o_sb + static_cast<int64_t>(i) * p.o_si +
                                                  h * p.o_sh);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const uint4 gw = __ldg(g4 + c4);
                const uint32_t gv[4] = {gw.x, gw.y, gw.z, gw.w};
                uint32_t ov[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // sigmoid(g) = 1 / (1 + 2^(-g log2 e))
                    const float g0 = __uint_as_float(gv[q] << 16);
                    const float g1 = __uint_as_float(gv[q] & 0xFFFF0000u);
                    const float s0 = ptx::rcp_approx(1.f + ptx::ex2(-g0 * kLog2e));
                    const float s1 = ptx::rcp_approx(1.f + ptx::ex2(-g1 * kLog2e));
                    ov[q] = ptx::pack_bf16(__uint_as_float(o[8 * c4 + 2 * q]) * inv * s0,
                                           __uint_as_float(o[8 * c4 + 2 * q + 1]) * inv * s1);
                }
                d4[c4] = make_uint4(ov[0], ov[1], ov[2], ov[3]);
            }
            if (p.lse)
                p.lse[b * p.l_sb + h * p.l_sh + i] = row_lse(st);
        }
        if (p.tile_counts && r == 0)
            p.tile_counts[(static_cast<int64_t>(b) * p.grid.Hq + h) * p.grid.nq + qb] = ntiles;
    }
}

template <bool BIAS>
__global__ void __launch_bounds__(kThreads, 1)
    evo_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const EvoParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    EvoSmem *sm = reinterpret_cast<EvoSmem *>(smem_raw + ((1024u - (base & 1023u)) & 1023u));
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(sm->q_full[b]), 1);
            ptx::mbar_init(bar(sm->q_empty[b]), 2); // one arrival per MMA warp
        }
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar(sm->kv_full[s]), 1);
            ptx::mbar_init(bar(sm->kv_empty[s]), 2); // one arrival per MMA warp
        }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bar(sm->s_full[t]), 1);
            ptx::mbar_init(bar(sm->p_full[t]), 128);
            ptx::mbar_init(bar(sm->s_free[t]), 128);
            ptx::mbar_init(bar(sm->pv_done[t]), 1);
        }
        ptx::mbar_init(bar(sm->final_bar[0]), 1);
        ptx::mbar_init(bar(sm->final_bar[1]), 1);
        sm->abort_flag = 0;
        ptx::fence_mbarrier_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 8 && ptx::lane_id() == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }
    if (warp == 9) {
        ptx::tmem_alloc(ptx::smem_u32(&sm->tmem_base), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    KernelCtx cx;
    cx.sm = sm;
    cx.tmem = sm->tmem_base;
    cx.wc.abort_flag = &sm->abort_flag;
    cx.wc.timeout_cycles = p.timeout_ns * 21 / 10; // 2.1 cycles per ns at the maximum clock
    cx.wc.err_user = p.err_user;
    cx.wc.err_lib = &g_lib_error_word;

    // Each branch ends with its own copy of the teardown barrier, so no code
    // runs under both register limits.
    if (warp < 8) {
        ptx::setmaxnreg_inc<kRegsSoftmax>();
        softmax_role<BIAS>(cx, p, warp >> 2);
        ptx::tc_fence_before();
        ptx::named_barrier_sync(1, kThreads);
    } else {
        ptx::setmaxnreg_dec<kRegsOther>();
        if (warp == 8)
            producer_role(cx, p, &tm_q, &tm_k, &tm_v);
        else if (warp == 9 || warp == 10)
            mma_role(cx, p, warp - 9);
        ptx::tc_fence_before();
        ptx::named_barrier_sync(1, kThreads);
        if (warp == 9) {
            ptx::tc_fence_after();
            ptx::tmem_dealloc(cx.tmem, 512);
        }
    }
}

template <bool BIAS>
cudaError_t launch_bias(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const EvoParams &p, int grid, cudaStream_t stream)
{
    const size_t smem = sizeof(EvoSmem) + 1024;
    static bool configured = false; // benign race: both calls are idempotent
    if (!configured) {
        cudaFuncAttributes attr;
        cudaError_t e = cudaFuncGetAttributes(&attr, evo_fwd_kernel<BIAS>);
        if (e != cudaSuccess)
            return e;
        // The setmaxnreg split assumes exactly kRegsLaunch registers at launch.
        if (attr.numRegs != static_cast<int>(kRegsLaunch))
            return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(evo_fwd_kernel<BIAS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    evo_fwd_kernel<BIAS><<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_evo(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const EvoParams &p, int grid, cudaStream_t stream)
{
    return p.bias ? launch_bias<true>(tq, tk, tv, p, grid, stream)
                  : launch_bias<false>(tq, tk, tv, p, grid, stream);
}

} // namespace fl
