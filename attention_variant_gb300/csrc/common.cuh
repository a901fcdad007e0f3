// common.cuh -- device helpers shared by the fused attention kernels:
// per-row key intervals of the masks, the linearised logical grid, and the
// bounded mbarrier waits every role uses.
#pragma once

#include "rtc_compat.cuh"

#include "fastdiv.h"
#include "ptx.cuh"

namespace fl {

constexpr int BM = 128; // query rows per tile (one TMEM lane per row)
constexpr int BN = 128; // keys per KV tile

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_bit_cast(float, 0x7f800000u); // -infinity

// MOD_EXPR: a score_mod expression compiled into the kernel at run time
enum : int { MOD_NONE = 0, MOD_ALIBI = 1, MOD_SOFTCAP = 2, MOD_EXPR = 3 };
enum : int { MASK_NONE = 0, MASK_CAUSAL = 1, MASK_WINDOW = 2, MASK_PREFIX = 3, MASK_DOC = 4 };

// ---------------------------------------------------------------- masks
//
// Every mask of the workload set allows, for query row i, one contiguous
// interval of keys [lo_i, hi_i):
//   none    [0, S)
//   causal  [0, i + 1)
//   window  [i - W + 1, i + 1)            (j <= i and i - j < W)
//   prefix  [0, max(i + 1, P))            (j <= i or j < P)
//   doc     [docstart(i), i + 1)          (same document and j <= i)
// clipped to [0, S).  lo_i and hi_i never decrease with i, so for a block of
// rows the union of allowed keys is [lo_first, hi_last) and every key tile
// meeting it holds at least one allowed pair; the tile range below is
// therefore minimal, and a tile is free of masked pairs exactly when it lies
// inside [lo_last, hi_first).
struct MaskSpec {
    int kind;
    int S;
    int window;
    int prefix;
    const int32_t *doc; // [B][doc_stride]
    int doc_stride;
};

__device__ __forceinline__ void row_interval(const MaskSpec &m, int b, int i, int &lo, int &hi)
{
    switch (m.kind) {
    case MASK_NONE:
        lo = 0;
        hi = m.S;
        break;
    case MASK_CAUSAL:
        lo = 0;
        hi = min(i + 1, m.S);
        break;
    case MASK_WINDOW:
        lo = max(0, i - m.window + 1);
        hi = min(i + 1, m.S);
        break;
    case MASK_PREFIX:
        lo = 0;
        hi = min(m.S, max(i + 1, m.prefix));
        break;
    default: { // MASK_DOC: the largest document start <= i (row starts at 0)
        const int32_t *st = m.doc + static_cast<int64_t>(b) * m.doc_stride;
        int a = 0, z = m.doc_stride - 1;
        while (a < z) {
            const int mid = (a + z + 1) >> 1;
            if (__ldg(st + mid) <= i)
                a = mid;
            else
                z = mid - 1;
        }
        lo = __ldg(st + a);
        hi = min(i + 1, m.S);
        break;
    }
    }
}

struct TileRange {
    int lo, hi;            // KV tiles [lo, hi) this query block visits
    int full_lo, full_hi;  // a tile [j0, j0 + width) needs no mask iff full_lo <= j0 and
                           // j0 + width <= full_hi
};

// TBN: the kernel's key-tile width (128 unless it says otherwise).
template <int TBN = BN>
__device__ __forceinline__ TileRange q_block_range(const MaskSpec &m, int b, int q0)
{
    const int i_first = q0;
    const int i_last = min(q0 + BM, m.S) - 1;
    int lo_f, hi_f, lo_l, hi_l;
    row_interval(m, b, i_first, lo_f, hi_f);
    row_interval(m, b, i_last, lo_l, hi_l);
    TileRange r;
    r.lo = lo_f / TBN;
    r.hi = (hi_l + TBN - 1) / TBN;
    r.full_lo = lo_l;
    r.full_hi = hi_f;
    return r;
}

// ---------------------------------------------------------------- logical grid
//
// The (query block x head) tile grid is unrolled into one linear index and
// decoded in-kernel (the "logical grid" of the Flashlight pages: talk notes,
// "Compiler design 4").  A CTA runs two query tiles ("slots") that share
// every K/V tile it loads:
//   G == 1 (MHA): the two slots are consecutive query blocks of one head;
//   G >= 2 (GQA): the two slots are two query heads of one KV group at the
//                 same query block.
// Axes: R row positions (query-block pairs for MHA, query blocks for GQA) and
// Hx head positions (b, head) or (b, kv head, head pair).
// Orders:
//   lpt = 1 (causal-family masks): longest work first -- rows descending,
//           heads fastest;
//   lpt = 0: GROUP_M-style strips of `group` head positions; inside a strip
//           heads run fastest, then rows, so concurrently running CTAs share
//           the K/V of at most `group` heads in L2 (talk notes,
//           "Implementation details": L2 cache optimisation).
// The divisions of the decoding use multipliers the host computes once per
// launch (fastdiv.h); the host keeps n_items below 2^31.
struct GridSpec {
    int B, Hq, Hk, G, nq;
    int R, Hx;
    int64_t n_items;
    int lpt;
    int group;      // strip width, at most Hx
    int pair_heads;
    FastDiv div_hx;    // Hx
    FastDiv div_strip; // group * R, the items of one strip
    FastDiv div_group; // group (every strip but a narrower last one)
    FastDiv div_last;  // the last strip's width, Hx - (strips - 1) * group
    FastDiv div_hq;    // Hq
    FastDiv div_pairs; // (G + 1) / 2, the head pairs of a KV group
    FastDiv div_hk;    // Hk
};

struct Item {
    int b, kvh;
    int h[2];
    int qb[2];
    bool valid[2];
};

#ifndef __CUDACC_RTC__
// The work-item grid for B batches, Hq query heads sharing Hk KV heads (G =
// Hq / Hk per KV head) and nq query blocks, in the LPT order or in strips;
// false (nothing set) when the items would number 2^31 or more.
inline bool make_grid_spec(int B, int Hq, int Hk, int nq, bool lpt, GridSpec &g)
{
    const int G = Hq / Hk;
    const int64_t R = G >= 2 ? nq : (nq + 1) / 2;
    const int64_t Hx = G >= 2 ? int64_t(B) * Hk * ((G + 1) / 2) : int64_t(B) * Hq;
    if (R * Hx >= (int64_t(1) << 31))
        return false;
    g.B = B;
    g.Hq = Hq;
    g.Hk = Hk;
    g.G = G;
    g.nq = nq;
    g.pair_heads = G >= 2 ? 1 : 0;
    g.R = int(R);
    g.Hx = int(Hx);
    g.n_items = R * Hx;
    g.lpt = lpt ? 1 : 0;
    g.group = g.Hx < 8 ? g.Hx : 8;
    const int strips = (g.Hx + g.group - 1) / g.group;
    g.div_hx = make_fastdiv(g.Hx);
    g.div_strip = make_fastdiv(g.group * g.R);
    g.div_group = make_fastdiv(g.group);
    g.div_last = make_fastdiv(g.Hx - (strips - 1) * g.group);
    g.div_hq = make_fastdiv(g.Hq);
    g.div_pairs = make_fastdiv((G + 1) / 2);
    g.div_hk = make_fastdiv(g.Hk);
    return true;
}
#endif // !__CUDACC_RTC__

__host__ __device__ __forceinline__ Item decode_item(const GridSpec &g, int64_t L64)
{
    const int L = static_cast<int>(L64); // < n_items < 2^31
    int r, hx;
    if (g.lpt) {
        const int q = fast_div(L, g.div_hx);
        r = g.R - 1 - q;
        hx = L - q * g.Hx;
    } else {
        const int strip = fast_div(L, g.div_strip);
        const int h0 = strip * g.group;
        const int w = L - strip * g.div_strip.d;
        // the strip's width: group, or what is left for the last strip
        const bool full = h0 + g.group <= g.Hx;
        FastDiv gs;
        gs.d = full ? g.div_group.d : g.div_last.d;
        gs.m = full ? g.div_group.m : g.div_last.m;
        gs.p = full ? g.div_group.p : g.div_last.p;
        r = fast_div(w, gs);
        hx = h0 + (w - r * gs.d);
    }
    Item it;
    if (!g.pair_heads) {
        it.b = fast_div(hx, g.div_hq);
        const int h = hx - it.b * g.Hq;
        it.kvh = h;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            it.h[t] = h;
            it.qb[t] = 2 * r + t;
            it.valid[t] = it.qb[t] < g.nq;
        }
    } else {
        const int bk = fast_div(hx, g.div_pairs);
        const int hp = hx - bk * g.div_pairs.d;
        it.b = fast_div(bk, g.div_hk);
        it.kvh = bk - it.b * g.Hk;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int gi = 2 * hp + t;
            it.valid[t] = gi < g.G;
            it.h[t] = it.kvh * g.G + gi;
            it.qb[t] = r;
        }
    }
    return it;
}

// ---------------------------------------------------------------- bounded waits
//
// Every wait on an mbarrier is bounded in wall-clock time.  When a wait runs
// out the thread raises the CTA's abort flag and records FL_DEVERR_TIMEOUT in
// the error word(s); every other wait in the CTA then returns false at once,
// each role leaves its loop, and the CTA reaches its teardown (drain of its
// own copies in flight, TMEM release) instead of hanging.
// A blocked waiter sleeps in hardware for at most this long between checks of
// the abort flag and the timeout (the phase completing wakes it at once).
constexpr uint32_t kWaitSuspendNs = 20000;

struct WaitCtl {
    volatile uint32_t *abort_flag; // shared memory
    uint64_t timeout_cycles;
    uint32_t *err_user;            // may be null
    uint32_t *err_lib;             // the library's own word
};

static __device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                                      const WaitCtl &c, uint32_t where,
                                                      bool honour_abort)
{
    // The bound is kept in SM clock cycles (clock64 is a cheap register read;
    // the global timer is not): timeout_cycles assumes the maximum SM clock,
    // so at lower clocks the wait only lasts longer in wall time.
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_try_wait_sleep(bar, parity, kWaitSuspendNs))
            return true;
        if (honour_abort && *c.abort_flag)
            return false;
        if (static_cast<uint64_t>(clock64() - t0) > c.timeout_cycles) {
            *c.abort_flag = 1u;
            const uint32_t code = 0x1u | ((where & 0xFFu) << 8);
            if (c.err_user)
                atomicOr(c.err_user, code);
            atomicOr(c.err_lib, code);
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl &c,
                                          uint32_t where)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    return mbar_wait_slow(bar, parity, c, where, true);
}

// Whole-warp wait: every lane polls, and the result is made warp-uniform so
// that no lane can leave a role loop alone.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl &c,
                                          uint32_t where)
{
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, c, where));
}

// Wait used while draining after an abort: ignores the abort flag, still bounded.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, const WaitCtl &c,
                                                uint32_t where)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    return mbar_wait_slow(bar, parity, c, where, false);
}

// Where-codes recorded in bits 8..15 of the error word.
enum : uint32_t {
    W_Q_EMPTY = 1, W_KV_EMPTY = 2, W_Q_FULL = 3, W_KV_FULL = 4, W_P_FULL = 5,
    W_S_FULL = 6, W_O_FULL = 7, W_FINAL = 8, W_DRAIN = 9, W_BIAS = 10, W_TURN = 11,
    W_INFO_FULL = 12, W_INFO_EMPTY = 13
};

} // namespace fl
