// fwd_diff.cu -- differential attention forward, D = 64, Dv = 64 or 128:
//     O = softmax(scale Q1 K1^T) V - lambda softmax(scale Q2 K2^T) V
// with both softmax streams fused in one kernel and sharing every V tile
// (the pages name differential attention among the variants that template
// systems cannot express: gist.science summary, "Results"; talk notes,
// "Evaluation: complex variants").  Masks: none or causal.
//
// CTA organisation (persistent, 384 threads):
//   warpgroup 0  online softmax of stream 1 (one thread per query row), then
//                output columns [0, Dv / 2)
//   warpgroup 1  online softmax of stream 2, then output columns [Dv / 2, Dv)
//   warp 8       TMA producer (Q1, Q2 once per work item; K1, K2, V per key tile)
//   warp 9       MMA issuer and TMEM owner
// TMEM: S_s at columns 128 s (P_s written over the first 64 of them),
// O_s (Dv fp32 columns) at 256 + 128 s.  V tiles arrive as Dv / 64 halves of
// 64 columns, each the B operand of its own N = 64 P V product.  Per key tile j the MMA thread issues,
// for s = 1, 2: [O_s += P_s V_{j-1}] then S_s = Q_s K_{s,j}^T, so the tensor
// core works on one stream while the other stream's softmax runs.  P_s may
// reuse S_s's columns because tcgen05.mma operations issued by one thread
// execute in order: S_s of tile j is issued after the P V of tile j-1 that
// reads P_s.
#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "launch.h"
#include "softmax_tile.cuh"

namespace fl {
namespace {

constexpr int kThreads = 384;
constexpr int kStages = 2;
constexpr uint32_t kTile = BM * 64 * 2; // 128 x 64 bf16
constexpr uint32_t kRegsLaunch = 168;
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsOther = 72;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther == kThreads * kRegsLaunch,
              "register split must equal the launch allocation");

template <int DV>
struct __align__(1024) DiffSmem {
    static constexpr int kVHalves = DV / 64;
    uint8_t q[2][kTile];
    uint8_t k[kStages][2][kTile];
    uint8_t v[kStages][kVHalves][kTile]; // the 64-column halves of a 128 x Dv V tile
    float lx[2][BM];              // each stream's row sums for the combined epilogue
    uint64_t q_full, q_empty;
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], p_full[2], o_full[2];
    uint64_t l_full, o_free, final_bar;
    uint32_t tmem_base;
    uint32_t abort_flag;
};

__device__ uint32_t g_lib_error_word;

__device__ __forceinline__ uint32_t bar(const uint64_t &b) { return ptx::smem_u32(&b); }

template <int DV>
struct Ctx {
    DiffSmem<DV> *sm;
    uint32_t tmem;
    WaitCtl wc;
};

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

template <int DV>
__device__ void producer_role(const Ctx<DV> &cx, const DiffParams &p, const CUtensorMap *tm_q,
                              const CUtensorMap *tm_k, const CUtensorMap *tm_v)
{
    constexpr int kVHalves = DiffSmem<DV>::kVHalves;
    DiffSmem<DV> &sm = *cx.sm;
    const uint32_t lane = ptx::lane_id();
    uint32_t kv_count = 0, item_count = 0;
    bool ok = true;
    for (int64_t L = blockIdx.x; L < p.n_items && ok; L += gridDim.x) {
        const DiffItem it = decode(p, L);
        const TileRange tr = q_block_range(p.mask, it.b, it.qb * BM);
        if (item_count > 0) {
            ok = warp_wait(bar(sm.q_empty), (item_count - 1) & 1, cx.wc, W_Q_EMPTY);
            if (!ok)
                break;
        }
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(sm.q_full), 2 * kTile);
            for (int s = 0; s < 2; ++s)
                ptx::tma_load_5d(ptx::smem_u32(sm.q[s]), tm_q, bar(sm.q_full), 0, it.qb * BM, it.h,
                                 it.b, s);
        }
        __syncwarp();
        for (int j = tr.lo; j < tr.hi; ++j, ++kv_count) {
            const uint32_t st = kv_count % kStages;
            ok = warp_wait(bar(sm.kv_empty[st]), ((kv_count / kStages) & 1) ^ 1, cx.wc, W_KV_EMPTY);
            if (!ok)
                break;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bar(sm.kv_full[st]), (2 + kVHalves) * kTile);
                for (int s = 0; s < 2; ++s)
                    ptx::tma_load_5d(ptx::smem_u32(sm.k[st][s]), tm_k, bar(sm.kv_full[st]), 0,
                                     j * BN, it.kvh, it.b, s);
                for (int half = 0; half < kVHalves; ++half)
                    ptx::tma_load_4d(ptx::smem_u32(sm.v[st][half]), tm_v, bar(sm.kv_full[st]),
                                     64 * half, j * BN, it.kvh, it.b);
            }
            __syncwarp();
        }
        ++item_count;
    }
    if (!ok) {
        const uint32_t first = kv_count > kStages ? kv_count - kStages : 0;
        for (uint32_t idx = first; idx < kv_count; ++idx)
            mbar_wait_drain(bar(sm.kv_full[idx % kStages]), (idx / kStages) & 1, cx.wc, W_DRAIN);
        if (item_count > 0)
            mbar_wait_drain(bar(sm.q_full), (item_count - 1) & 1, cx.wc, W_DRAIN);
    }
}

template <int DV>
__device__ void mma_role(const Ctx<DV> &cx, const DiffParams &p)
{
    constexpr int kVHalves = DiffSmem<DV>::kVHalves;
    DiffSmem<DV> &sm = *cx.sm;
    const uint32_t lane = ptx::lane_id();
    constexpr uint32_t idesc_qk = umma_idesc_bf16(BM, BN, false);
    constexpr uint32_t idesc_pv = umma_idesc_bf16(BM, 64, true);
    uint32_t kv_count = 0, item_count = 0;
    uint32_t pcount[2] = {0, 0};
    bool ok = true;
    for (int64_t L = blockIdx.x; L < p.n_items && ok; L += gridDim.x) {
        const DiffItem it = decode(p, L);
        const TileRange tr = q_block_range(p.mask, it.b, it.qb * BM);
        ok = warp_wait(bar(sm.q_full), item_count & 1, cx.wc, W_Q_FULL);
        if (!ok)
            break;
        ptx::tc_fence_after();
        uint32_t prev = 0;
        for (int j = tr.lo; j <= tr.hi && ok; ++j) {
            const uint32_t st = kv_count % kStages;
            if (j < tr.hi) {
                ok = warp_wait(bar(sm.kv_full[st]), (kv_count / kStages) & 1, cx.wc, W_KV_FULL);
                if (!ok)
                    break;
                ptx::tc_fence_after();
            }
            for (int s = 0; s < 2; ++s) {
                if (j > tr.lo) {
                    ok = warp_wait(bar(sm.p_full[s]), pcount[s] & 1, cx.wc, W_P_FULL);
                    if (ok && s == 0 && j == tr.lo + 1 && item_count > 0)
                        // the epilogue of the previous item has read O_1 and O_2
                        ok = warp_wait(bar(sm.o_free), (item_count - 1) & 1, cx.wc, W_O_FULL);
                    if (!ok)
                        break;
                    ++pcount[s];
                    ptx::tc_fence_after();
                    if (lane == 0) {
#pragma unroll
                        for (int half = 0; half < kVHalves; ++half) {
                            const uint32_t vb = ptx::smem_u32(sm.v[prev][half]);
#pragma unroll
                            for (int kk = 0; kk < BN / 16; ++kk)
                                ptx::mma_ts(cx.tmem + 256 + 128 * s + 64 * half,
                                            cx.tmem + 128 * s + 8 * kk,
                                            umma_desc(vb + kk * 2048, kTile, 1024, kSwizzle128B),
                                            idesc_pv, (j - 1 > tr.lo || kk > 0) ? 1u : 0u);
                        }
                        if (j == tr.hi)
                            ptx::mma_commit(bar(sm.o_full[s]));
                    }
                    __syncwarp();
                }
                if (j < tr.hi) {
                    if (lane == 0) {
                        const uint32_t qb = ptx::smem_u32(sm.q[s]);
                        const uint32_t kb = ptx::smem_u32(sm.k[st][s]);
#pragma unroll
                        for (int kk = 0; kk < 64 / 16; ++kk)
                            ptx::mma_ss(cx.tmem + 128 * s,
                                        umma_desc(qb + kk * 32, 16, 1024, kSwizzle128B),
                                        umma_desc(kb + kk * 32, 16, 1024, kSwizzle128B), idesc_qk,
                                        kk > 0 ? 1u : 0u);
                        ptx::mma_commit(bar(sm.s_full[s]));
                    }
                    __syncwarp();
                }
            }
            if (!ok)
                break;
            if (lane == 0) {
                if (j > tr.lo)
                    ptx::mma_commit(bar(sm.kv_empty[prev]));
                if (j == tr.hi - 1)
                    ptx::mma_commit(bar(sm.q_empty));
            }
            __syncwarp();
            if (j < tr.hi) {
                prev = st;
                ++kv_count;
            }
        }
        ++item_count;
    }
    if (lane == 0)
        ptx::mma_commit(bar(sm.final_bar));
    __syncwarp();
    mbar_wait_drain(bar(sm.final_bar), 0, cx.wc, W_FINAL);
}

template <int DV>
__device__ void softmax_role(const Ctx<DV> &cx, const DiffParams &p, int s)
{
    DiffSmem<DV> &sm = *cx.sm;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = (((threadIdx.x >> 5) & 3u) * 32u) << 16;
    const uint32_t tS = cx.tmem + lane_off + 128 * s;
    const uint32_t tO[2] = {cx.tmem + lane_off + 256, cx.tmem + lane_off + 384};
    uint32_t scount = 0, icount = 0;
    ScoreMod smod{};
    smod.qk_log2 = p.qk_log2;

    for (int64_t L = blockIdx.x; L < p.n_items; L += gridDim.x, ++icount) {
        const DiffItem it = decode(p, L);
        const TileRange tr = q_block_range(p.mask, it.b, it.qb * BM);
        const int i = it.qb * BM + r;
        int row_lo, row_hi;
        row_interval(p.mask, it.b, i, row_lo, row_hi);
        RowState st{kNegInf, 0.f, 0.f};
        for (int j = tr.lo; j < tr.hi; ++j) {
            if (!warp_wait(bar(sm.s_full[s]), scount & 1, cx.wc, W_S_FULL))
                return;
            ++scount;
            ptx::tc_fence_after();
            float x[BN];
            load_scores(tS, x);
            const int j0 = j * BN;
            apply_score_mod<MOD_NONE>(x, smod, i, j0);
            if (!((j0 >= tr.full_lo) && (j0 + BN <= tr.full_hi)))
                apply_row_mask(x, j0, row_lo, row_hi);
            online_update_and_store_p<DV>(x, p.qk_log2, st, j == tr.lo, tO[s], tS);
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(sm.p_full[s]));
        }

        // epilogue: share l, then this warpgroup writes output columns
        // [Dv / 2 s, Dv / 2 (s + 1))
        sm.lx[s][r] = st.l_round;
        ptx::mbar_arrive(bar(sm.l_full));
        if (p.lse && i < p.mask.S)
            p.lse[s * p.l_s2 + it.b * p.l_sb + it.h * p.l_sh + i] = row_lse(st);
        if (p.tile_counts && s == 0 && r == 0)
            p.tile_counts[(static_cast<int64_t>(it.b) * p.H + it.h) * p.nq + it.qb] = tr.hi - tr.lo;
        if (!warp_wait(bar(sm.o_full[0]), icount & 1, cx.wc, W_O_FULL) ||
            !warp_wait(bar(sm.o_full[1]), icount & 1, cx.wc, W_O_FULL) ||
            !warp_wait(bar(sm.l_full), icount & 1, cx.wc, W_O_FULL))
            return;
        ptx::tc_fence_after();
        const float l0 = sm.lx[0][r], l1 = sm.lx[1][r];
        const float c0 = l0 > 0.f ? 1.f / l0 : 0.f;
        const float c1 = l1 > 0.f ? -p.lambda / l1 : 0.f;
        __nv_bfloat16 *dst = p.out + it.b * p.o_sb + static_cast<int64_t>(i) * p.o_ss +
                             it.h * p.o_sh + (DV / 2) * s;
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
            uint32_t a[16], bb[16];
            ptx::tmem_ld16(tO[0] + (DV / 2) * s + 16 * c, a);
            ptx::tmem_ld16(tO[1] + (DV / 2) * s + 16 * c, bb);
            ptx::tmem_wait_ld();
            ptx::reg_fence<16>(a);
            ptx::reg_fence<16>(bb);
            if (i < p.mask.S) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float y0 = fmaf(__uint_as_float(a[2 * e]), c0, __uint_as_float(bb[2 * e]) * c1);
                    const float y1 =
                        fmaf(__uint_as_float(a[2 * e + 1]), c0, __uint_as_float(bb[2 * e + 1]) * c1);
                    w[e] = ptx::pack_bf16(y0, y1);
                }
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + 16 * c);
                d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
                d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(sm.o_free));
    }
}

template <int DV>
__global__ void __launch_bounds__(kThreads, 1)
    diff_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const DiffParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    DiffSmem<DV> *sm = reinterpret_cast<DiffSmem<DV> *>(smem_raw + ((1024u - (base & 1023u)) & 1023u));
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(sm->q_full), 1);
        ptx::mbar_init(bar(sm->q_empty), 1);
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar(sm->kv_full[s]), 1);
            ptx::mbar_init(bar(sm->kv_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(bar(sm->s_full[s]), 1);
            ptx::mbar_init(bar(sm->p_full[s]), 128);
            ptx::mbar_init(bar(sm->o_full[s]), 1);
        }
        ptx::mbar_init(bar(sm->l_full), 256);
        ptx::mbar_init(bar(sm->o_free), 256);
        ptx::mbar_init(bar(sm->final_bar), 1);
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
    Ctx<DV> cx;
    cx.sm = sm;
    cx.tmem = sm->tmem_base;
    cx.wc.abort_flag = &sm->abort_flag;
    cx.wc.timeout_cycles = p.timeout_ns * 21 / 10; // 2.1 cycles per ns at the maximum clock
    cx.wc.err_user = p.err_user;
    cx.wc.err_lib = &g_lib_error_word;
    if (warp < 8) {
        ptx::setmaxnreg_inc<kRegsSoftmax>();
        softmax_role<DV>(cx, p, warp >> 2);
        ptx::tc_fence_before();
        ptx::named_barrier_sync(1, kThreads);
    } else {
        ptx::setmaxnreg_dec<kRegsOther>();
        if (warp == 8)
            producer_role<DV>(cx, p, &tm_q, &tm_k, &tm_v);
        else if (warp == 9)
            mma_role<DV>(cx, p);
        ptx::tc_fence_before();
        ptx::named_barrier_sync(1, kThreads);
        if (warp == 9) {
            ptx::tc_fence_after();
            ptx::tmem_dealloc(cx.tmem, 512);
        }
    }
}

template <int DV>
cudaError_t launch_dv(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                      const DiffParams &p, int grid, cudaStream_t stream)
{
    const size_t smem = sizeof(DiffSmem<DV>) + 1024;
    static bool configured = false;
    if (!configured) {
        cudaFuncAttributes attr;
        cudaError_t e = cudaFuncGetAttributes(&attr, diff_fwd_kernel<DV>);
        if (e != cudaSuccess)
            return e;
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
