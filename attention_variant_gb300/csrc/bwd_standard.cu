// bwd_standard.cu -- attention backward for the standard kind (MHA / GQA,
// D = Dv = 64, no mask or causal): dQ, dK, dV from Q, K, V, the forward's O
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
// Three kernels, no atomics (every output element has one writer):
//   bwd_prep_kernel  per query row: D_i and LSE_i * log2 e into the workspace
//                    (padded rows get +inf, so their P is 0);
//   bwd_dkdv_kernel  one CTA per (64-key block, KV head, batch): four warps
//                    own 16 keys each and keep dK and dV in registers while
//                    the CTA walks every query block of every query head of
//                    the group (query blocks wholly before the key block are
//                    skipped under the causal mask);
//   bwd_dq_kernel    one CTA per (128-row query tile, query head, batch) on
//                    the tcgen05 tensor cores: S, dP and the dQ accumulator
//                    in TMEM, dS computed by one thread per query row
//                    (described at the kernel).
// In the dK/dV kernel a producer warp streams the 64-row Q and dO tiles
// (128-byte swizzle) through a 3-stage TMA ring and the consumer warps
// recompute S and P and form the products with warp-level bf16 MMAs
// (m16n8k16, fp32 accumulate) on ldmatrix fragments; P and dS go from
// accumulators straight into A operands.  Recomputing S and dP in the dQ
// kernel costs two more of the seven products than an atomic dQ
// accumulation would, and buys determinism and no dQ workspace.
#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "launch.h"
#include "warp_mma.cuh"

namespace fl {
namespace {

constexpr int kBlk = kBwdBlock;              // rows per tile (queries or keys)
constexpr int kConsumerWarps = 4;            // 16 rows each
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kStages = 3;
constexpr uint32_t kTileBytes = kBlk * 64 * 2; // 8 KB
constexpr uint32_t kStatBytes = kBlk * 8;      // (lse2, D) per row

__device__ uint32_t g_lib_error_word;

__device__ __forceinline__ uint32_t bf16_bits(const __nv_bfloat16 &x)
{
    return static_cast<uint32_t>(__bfloat16_as_ushort(x));
}

// A fragments of 16 consecutive rows (r0 .. r0+15) of a [.., 64] bf16 row
// block in global memory, k-steps 0..3; rows >= n are zero.
__device__ __forceinline__ void load_a_rows(const __nv_bfloat16 *base, int64_t row_stride, int r0, int n,
                                            uint32_t (&a)[4][4])
{
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        a[k][0] = a[k][1] = a[k][2] = a[k][3] = 0u;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = r0 + g + 8 * half;
        if (r >= n)
            continue;
        const __nv_bfloat16 *p = base + r * row_stride;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            a[k][half] = bf16_bits(p[16 * k + 2 * t]) | (bf16_bits(p[16 * k + 2 * t + 1]) << 16);
            a[k][2 + half] = bf16_bits(p[16 * k + 8 + 2 * t]) | (bf16_bits(p[16 * k + 9 + 2 * t]) << 16);
        }
    }
}

// Accumulators (16 rows x 64 columns as eight n-tiles) of one warp -> bf16 A
// fragments over those 64 columns as k (four k-steps).
__device__ __forceinline__ void acc_to_a(const float (&c)[8][4], uint32_t (&a)[4][4])
{
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        a[kk][0] = ptx::pack_bf16(c[2 * kk][0], c[2 * kk][1]);
        a[kk][1] = ptx::pack_bf16(c[2 * kk][2], c[2 * kk][3]);
        a[kk][2] = ptx::pack_bf16(c[2 * kk + 1][0], c[2 * kk + 1][1]);
        a[kk][3] = ptx::pack_bf16(c[2 * kk + 1][2], c[2 * kk + 1][3]);
    }
}

__device__ __forceinline__ void zero(float (&c)[8][4])
{
#pragma unroll
    for (int n = 0; n < 8; ++n)
        c[n][0] = c[n][1] = c[n][2] = c[n][3] = 0.f;
}

// c += A (16 x 64, as k) times the 64 x 64 tile `tile`, read as B with k along
// the tile's rows and n along its columns (P V form).
__device__ __forceinline__ void mma_a_tile_cols(float (&c)[8][4], const uint32_t (&a)[4][4], uint32_t tile)
{
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int u2 = 0; u2 < 4; ++u2) {
            uint32_t b[4];
            wm::ldsm_b_cols(tile, 16 * kk, u2, b);
            wm::mma16816(c[2 * u2], a[kk], b[0], b[1]);
            wm::mma16816(c[2 * u2 + 1], a[kk], b[2], b[3]);
        }
}

// c += A (16 x 64 dims) times tile^T: n along the tile's rows (Q K^T form).
__device__ __forceinline__ void mma_a_tile_rows(float (&c)[8][4], const uint32_t (&a)[4][4], uint32_t tile)
{
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int n2 = 0; n2 < 4; ++n2) {
            uint32_t b[4];
            wm::ldsm_b_rows(tile, 16 * n2, kk, b);
            wm::mma16816(c[2 * n2], a[kk], b[0], b[1]);
            wm::mma16816(c[2 * n2 + 1], a[kk], b[2], b[3]);
        }
}

// Shared memory of both main kernels: the stages' tiles (each 1024-byte
// aligned, as the 128-byte swizzle pattern assumes), the stages' row
// statistics, then the barriers.
struct Ring {
    uint8_t *base;
    uint64_t *full, *empty;
    volatile uint32_t *abort;
    __device__ uint32_t tile(int s, int which) const
    {
        return ptx::smem_u32(base) + (2 * s + which) * kTileBytes;
    }
    __device__ float *stats(int s) const
    {
        return reinterpret_cast<float *>(base + kStages * 2 * kTileBytes + s * kStatBytes);
    }
};

__device__ __forceinline__ Ring make_ring(uint8_t *smem_raw)
{
    const uint32_t b = ptx::smem_u32(smem_raw);
    Ring r;
    r.base = smem_raw + ((1024u - (b & 1023u)) & 1023u);
    r.full = reinterpret_cast<uint64_t *>(r.base + kStages * (2 * kTileBytes + kStatBytes));
    r.empty = r.full + kStages;
    r.abort = reinterpret_cast<volatile uint32_t *>(r.empty + kStages);
    return r;
}

__device__ __forceinline__ void init_ring(const Ring &r)
{
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&r.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&r.empty[s]), kConsumerWarps);
        }
        *r.abort = 0;
        ptx::fence_mbarrier_init();
    }
    __syncthreads();
}

// The last copy issued into each stage may still be landing after a failed
// wait: wait for it (bounded) before the CTA exits.
__device__ __forceinline__ void drain(const Ring &r, int issued, const WaitCtl &wc)
{
    for (int s = 0; s < kStages; ++s) {
        const int last = issued - 1 - ((issued - 1 - s) % kStages + kStages) % kStages;
        if (last >= 0)
            mbar_wait_drain(ptx::smem_u32(&r.full[s]), (last / kStages) & 1, wc, W_DRAIN);
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
    float2 st = make_float2(__int_as_float(0x7f800000), 0.f); // padded: P = 0
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
        st = make_float2(lse == kNegInf ? __int_as_float(0x7f800000) : lse * kLog2e, acc);
    }
    reinterpret_cast<float2 *>(p.ws_stats)[idx] = st;
}

// ---------------------------------------------------------------- dK, dV

__global__ void __launch_bounds__(kThreads, 2)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p)
{
    const int kb = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int k0 = kb * kBlk;
    const int G = p.Hq / p.Hk;
    const int nqb = p.S_pad / kBlk;
    const int qb0 = p.causal ? kb : 0; // query blocks before the key block see none of its keys
    const int n_it = G * (nqb - qb0);

    extern __shared__ uint8_t smem_raw[];
    const Ring ring = make_ring(smem_raw);
    init_ring(ring);
    WaitCtl wc;
    wc.abort_flag = ring.abort;
    wc.timeout_cycles = p.timeout_ns * 21 / 10;
    wc.err_user = p.err_user;
    wc.err_lib = &g_lib_error_word;

    bool ok = true;
    int issued = 0;
    float dk[8][4], dv[8][4];
    zero(dk);
    zero(dv);

    if (warp == kConsumerWarps) {
        // ---- producer: per iteration (head h of the group, query block qb)
        // the Q and dO tiles by TMA and the rows' (lse2, D) by the warp's lanes
        for (int it = 0; it < n_it; ++it) {
            const int s = it % kStages;
            const int h = hk * G + it / (nqb - qb0), qb = qb0 + it % (nqb - qb0);
            if (it >= kStages &&
                !__all_sync(0xffffffffu, mbar_wait(ptx::smem_u32(&ring.empty[s]), ((it / kStages) - 1) & 1, wc,
                                                   W_KV_EMPTY))) {
                ok = false;
                break;
            }
            const float2 *src = reinterpret_cast<const float2 *>(p.ws_stats) +
                                (static_cast<int64_t>(b) * p.Hq + h) * p.S_pad + qb * kBlk;
            float2 *dst = reinterpret_cast<float2 *>(ring.stats(s));
            dst[lane] = src[lane];
            dst[lane + 32] = src[lane + 32];
            __syncwarp();
            if (lane == 0) {
                const uint32_t bar = ptx::smem_u32(&ring.full[s]);
                ptx::mbar_arrive_expect_tx(bar, 2 * kTileBytes);
                ptx::tma_load_4d(ring.tile(s, 0), &tm_q, bar, 0, qb * kBlk, h, b);
                ptx::tma_load_4d(ring.tile(s, 1), &tm_do, bar, 0, qb * kBlk, h, b);
            }
            issued = it + 1;
        }
    } else {
        // ---- consumers: keys k0 + 16 warp .. + 15
        const int key_a = k0 + 16 * warp + g, key_b = key_a + 8;
        uint32_t ka[4][4], va[4][4];
        load_a_rows(p.k + b * p.k_sb + hk * p.k_sh, p.k_ss, k0 + 16 * warp, p.S, ka);
        load_a_rows(p.v + b * p.v_sb + hk * p.v_sh, p.v_ss, k0 + 16 * warp, p.S, va);
        const float sl2 = p.scale * kLog2e;
        for (int it = 0; it < n_it; ++it) {
            const int s = it % kStages;
            const int qb = qb0 + it % (nqb - qb0);
            if (!warp_wait(ptx::smem_u32(&ring.full[s]), (it / kStages) & 1, wc, W_KV_FULL)) {
                ok = false;
                break;
            }
            const uint32_t sq = ring.tile(s, 0), sdo = ring.tile(s, 1);
            const float2 *st = reinterpret_cast<const float2 *>(ring.stats(s));
            const int q0 = qb * kBlk;
            // P^T (keys x queries) = exp2(sl2 K Q^T - lse2)
            float pt[8][4];
            zero(pt);
            mma_a_tile_rows(pt, ka, sq);
            const bool masked = p.causal && q0 < k0 + kBlk; // the diagonal block
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int qc = 8 * n + 2 * t + (e & 1);
                    const float pv = ptx::ex2(fmaf(pt[n][e], sl2, -st[qc].x));
                    const int key = e < 2 ? key_a : key_b;
                    pt[n][e] = (masked && key > q0 + qc) ? 0.f : pv;
                }
            uint32_t pa[4][4];
            acc_to_a(pt, pa);
            // dV += P^T dO
            mma_a_tile_cols(dv, pa, sdo);
            // dP^T = V dO^T, then dS^T = P^T (dP^T - D)
            float dpt[8][4];
            zero(dpt);
            mma_a_tile_rows(dpt, va, sdo);
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int qc = 8 * n + 2 * t + (e & 1);
                    dpt[n][e] = pt[n][e] * (dpt[n][e] - st[qc].y);
                }
            uint32_t dsa[4][4];
            acc_to_a(dpt, dsa);
            // dK += dS^T Q
            mma_a_tile_cols(dk, dsa, sq);
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(ptx::smem_u32(&ring.empty[s]));
        }
    }
    if (!__syncthreads_and(ok)) {
        if (warp == kConsumerWarps && lane == 0)
            drain(ring, issued, wc);
        return; // recorded in the error words; this block's dK, dV stay unwritten
    }
    if (warp < kConsumerWarps) {
        const int key_a = k0 + 16 * warp + g, key_b = key_a + 8;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int key = half ? key_b : key_a;
            if (key >= p.S)
                continue;
            __nv_bfloat16 *pk = p.dk + b * p.dk_sb + key * p.dk_ss + hk * p.dk_sh;
            __nv_bfloat16 *pv = p.dv + b * p.dv_sb + key * p.dv_ss + hk * p.dv_sh;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                *reinterpret_cast<uint32_t *>(pk + 8 * n + 2 * t) =
                    ptx::pack_bf16(dk[n][2 * half] * p.scale, dk[n][2 * half + 1] * p.scale);
                *reinterpret_cast<uint32_t *>(pv + 8 * n + 2 * t) =
                    ptx::pack_bf16(dv[n][2 * half], dv[n][2 * half + 1]);
            }
        }
    }
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
constexpr int kDqRows = 128, kDqKeys = 64, kDqStages = 4, kDqThreads = 384;
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

__global__ void __launch_bounds__(kDqThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const BwdParams p)
{
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = qt * kDqRows;
    const int hk = h / (p.Hq / p.Hk);
    const int nkb = (p.S + kDqKeys - 1) / kDqKeys;
    // causal: key tiles wholly after the last row of the query tile see none
    const int n_it = p.causal ? min(nkb, (q0 + kDqRows + kDqKeys - 1) / kDqKeys) : nkb;

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
                ptx::tma_load_4d(ptx::smem_u32(sm.k[s]), &tm_k, bar(sm.kv_full[s]), 0, j * kDqKeys, hk, b);
                ptx::tma_load_4d(ptx::smem_u32(sm.v[s]), &tm_v, bar(sm.kv_full[s]), 0, j * kDqKeys, hk, b);
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
        const float2 st = reinterpret_cast<const float2 *>(p.ws_stats)[(static_cast<int64_t>(b) * p.Hq + h) * p.S_pad + row];
        const float sl2 = p.scale * kLog2e;
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
            const int j0 = j * kDqKeys;
            const bool edge = j0 + kDqKeys > p.S || (p.causal && j0 + kDqKeys - 1 > q0);
            uint32_t ds[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float d2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = 2 * c + e;
                    const float pr = ptx::ex2(fmaf(__uint_as_float(sv[col]), sl2, -st.x));
                    float dsv = pr * (__uint_as_float(pv[col]) - st.y);
                    if (edge && (j0 + col >= p.S || (p.causal && j0 + col > row)))
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
            uint4 *dst = reinterpret_cast<uint4 *>(p.dq + b * p.dq_sb + static_cast<int64_t>(row) * p.dq_ss +
                                                   h * p.dq_sh + 32 * wg);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    w[q] = ptx::pack_bf16(__uint_as_float(o[8 * c + 2 * q]) * p.scale,
                                          __uint_as_float(o[8 * c + 2 * q + 1]) * p.scale);
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

constexpr size_t kSmemBytes = kStages * (2 * kTileBytes + kStatBytes) + 2 * kStages * 8 + 8 + 1024;
// more than half an SM's shared memory: one dQ CTA per SM, so that no second
// CTA waits in tcgen05.alloc for the 512 TMEM columns the first one holds
constexpr size_t kDqSmemBytes = sizeof(DqSmem) + 1024 > 120 * 1024 ? sizeof(DqSmem) + 1024 : 120 * 1024;

} // namespace

cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tdo, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tq128, const CUtensorMap &tdo128,
                       const BwdParams &p, cudaStream_t stream)
{
    const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.S_pad;
    bwd_prep_kernel<<<static_cast<unsigned>((rows + 127) / 128), 128, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    static bool configured = false; // benign race: the calls are idempotent
    if (!configured) {
        if ((e = cudaFuncSetAttribute(bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kSmemBytes))) != cudaSuccess ||
            (e = cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kDqSmemBytes))) != cudaSuccess)
            return e;
        configured = true;
    }
    const int nb = p.S_pad / kBlk;
    bwd_dkdv_kernel<<<dim3(nb, p.Hk, p.B), kThreads, kSmemBytes, stream>>>(tq, tdo, p);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    bwd_dq_kernel<<<dim3((p.S + kDqRows - 1) / kDqRows, p.Hq, p.B), kDqThreads, kDqSmemBytes, stream>>>(
        tq128, tdo128, tk, tv, p);
    return cudaGetLastError();
}

} // namespace fl
