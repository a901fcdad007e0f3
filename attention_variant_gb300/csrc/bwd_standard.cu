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
//   bwd_dq_kernel    one CTA per (64-row query block, query head, batch):
//                    four warps own 16 query rows each and keep dQ in
//                    registers while the CTA walks the key blocks.
// In both main kernels a producer warp streams the 64-row tiles the loop
// needs (Q and dO, or K and V; 128-byte swizzle) through a 3-stage TMA ring,
// and the consumer warps recompute S and P and form the products with
// warp-level bf16 MMAs (m16n8k16, fp32 accumulate) on ldmatrix fragments;
// P and dS go from accumulators straight into A operands.  Recomputing S in
// the dQ kernel costs two more of the seven products than an atomic dQ
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

// ---------------------------------------------------------------- dQ

__global__ void __launch_bounds__(kThreads, 2)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const BwdParams p)
{
    const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int q0 = qb * kBlk;
    const int hk = h / (p.Hq / p.Hk);
    const int nkb = (p.S + kBlk - 1) / kBlk;
    const int n_it = p.causal ? min(qb + 1, nkb) : nkb; // key blocks past the query block see none

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
    float dq[8][4];
    zero(dq);

    if (warp == kConsumerWarps) {
        if (lane == 0)
            for (int it = 0; it < n_it; ++it) {
                const int s = it % kStages;
                if (it >= kStages &&
                    !mbar_wait(ptx::smem_u32(&ring.empty[s]), ((it / kStages) - 1) & 1, wc, W_KV_EMPTY)) {
                    ok = false;
                    break;
                }
                const uint32_t bar = ptx::smem_u32(&ring.full[s]);
                ptx::mbar_arrive_expect_tx(bar, 2 * kTileBytes);
                ptx::tma_load_4d(ring.tile(s, 0), &tm_k, bar, 0, it * kBlk, hk, b);
                ptx::tma_load_4d(ring.tile(s, 1), &tm_v, bar, 0, it * kBlk, hk, b);
                issued = it + 1;
            }
    } else {
        // ---- consumers: query rows q0 + 16 warp .. + 15
        const int row_a = q0 + 16 * warp + g, row_b = row_a + 8;
        uint32_t qa[4][4], doa[4][4];
        load_a_rows(p.q + b * p.q_sb + h * p.q_sh, p.q_ss, q0 + 16 * warp, p.S, qa);
        load_a_rows(p.dout + b * p.do_sb + h * p.do_sh, p.do_ss, q0 + 16 * warp, p.S, doa);
        const float2 *stats = reinterpret_cast<const float2 *>(p.ws_stats) +
                              (static_cast<int64_t>(b) * p.Hq + h) * p.S_pad;
        const float2 st_a = stats[row_a], st_b = stats[row_b]; // rows < S_pad
        const float sl2 = p.scale * kLog2e;
        for (int it = 0; it < n_it; ++it) {
            const int s = it % kStages;
            if (!warp_wait(ptx::smem_u32(&ring.full[s]), (it / kStages) & 1, wc, W_KV_FULL)) {
                ok = false;
                break;
            }
            const uint32_t sk = ring.tile(s, 0), sv = ring.tile(s, 1);
            const int j0 = it * kBlk;
            // P = exp2(sl2 Q K^T - lse2)
            float pr[8][4];
            zero(pr);
            mma_a_tile_rows(pr, qa, sk);
            const bool edge = j0 + kBlk > p.S || (p.causal && j0 + kBlk > q0);
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = j0 + 8 * n + 2 * t + (e & 1);
                    const int row = e < 2 ? row_a : row_b;
                    const float pv = ptx::ex2(fmaf(pr[n][e], sl2, -(e < 2 ? st_a.x : st_b.x)));
                    pr[n][e] = (edge && (key >= p.S || (p.causal && key > row))) ? 0.f : pv;
                }
            // dP = dO V^T, dS = P (dP - D)
            float dp[8][4];
            zero(dp);
            mma_a_tile_rows(dp, doa, sv);
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dp[n][e] = pr[n][e] * (dp[n][e] - (e < 2 ? st_a.y : st_b.y));
            uint32_t dsa[4][4];
            acc_to_a(dp, dsa);
            // dQ += dS K
            mma_a_tile_cols(dq, dsa, sk);
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(ptx::smem_u32(&ring.empty[s]));
        }
    }
    if (!__syncthreads_and(ok)) {
        if (warp == kConsumerWarps && lane == 0)
            drain(ring, issued, wc);
        return;
    }
    if (warp < kConsumerWarps) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int row = q0 + 16 * warp + g + 8 * half;
            if (row >= p.S)
                continue;
            __nv_bfloat16 *pq = p.dq + b * p.dq_sb + row * p.dq_ss + h * p.dq_sh;
#pragma unroll
            for (int n = 0; n < 8; ++n)
                *reinterpret_cast<uint32_t *>(pq + 8 * n + 2 * t) =
                    ptx::pack_bf16(dq[n][2 * half] * p.scale, dq[n][2 * half + 1] * p.scale);
        }
    }
}

constexpr size_t kSmemBytes = kStages * (2 * kTileBytes + kStatBytes) + 2 * kStages * 8 + 8 + 1024;

} // namespace

cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tdo, const CUtensorMap &tk,
                       const CUtensorMap &tv, const BwdParams &p, cudaStream_t stream)
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
                                      static_cast<int>(kSmemBytes))) != cudaSuccess)
            return e;
        configured = true;
    }
    const int nb = p.S_pad / kBlk;
    bwd_dkdv_kernel<<<dim3(nb, p.Hk, p.B), kThreads, kSmemBytes, stream>>>(tq, tdo, p);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    bwd_dq_kernel<<<dim3(nb, p.Hq, p.B), kThreads, kSmemBytes, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

} // namespace fl
