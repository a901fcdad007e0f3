// fwd_decode.cu -- attention forward for serving with a KV cache (decode):
// a few new query tokens per sequence against a cached, variable-length and
// optionally paged K/V, with the causal (query row s of a sequence of L keys
// sits at position L - Sq + s) and softcap variants the pages serve LLaMA-3.2-1B
// with (talk notes, "End-to-end: LLaMA-3.2-1B (vLLM / Mooncake)").  The result
// is the same softmax(score_mod(scale q k^T) + mask) V as every other kind; the
// online-softmax recurrence is applied across key chunks (gist.science summary,
// "Methodology" item 3).
//
// Decode reads every cached key once and multiplies it by only R = G * Sq
// query rows (G = Hq / Hk query heads per KV head), so it is HBM-bound: the
// design keeps as many K/V bytes in flight as the SM can take and spends as few
// instructions per key as it can.
//   * Split-KV: one CTA per (split of split_chunks * kDecodeChunk keys, KV
//     head, sequence); splits past a sequence's length exit at once.
//   * A producer warp streams the split's chunks of kDecodeChunk keys (K and V,
//     bf16, 128-byte swizzle) into a ring of kStages shared-memory stages by
//     TMA: one box per chunk for a contiguous cache, one per page for a paged
//     one (pages holding no key of the sequence are not loaded).
//   * Four consumer warps share each chunk: warp w owns a group of 16 query
//     rows (rows padded to 16) and a slice of the chunk's keys, and keeps its
//     own online softmax (running max m, sum l, unnormalised O) in registers.
//     Q K^T and P V are warp-level bf16 tensor-core MMAs (m16n8k16, fp32
//     accumulate) on operands fetched from the swizzled stages by ldmatrix; P
//     goes from the score accumulators straight into the A operand of P V.  A
//     warp releases a stage by one arrive; no CTA-wide barrier runs per chunk.
//   * At the end the warps' (m, l, O) meet in shared memory; a split that
//     covers the whole sequence writes bf16 O and the natural-log LSE, other
//     splits write a partial to the workspace and an atomic ticket per
//     (sequence, KV head) makes the last one merge them
//     (O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s) and zero its counter.
// Scores are kept in base 2 (scale * log2 e folded in) inside the kernel.
//
// The tensor cores used are the warp-level ones: the contraction has at most
// 16 rows per warp, below the 64-row minimum of a tcgen05 MMA, and its flops
// are a few percent of what the bytes allow; what the warp-level MMA buys is
// the removal of the per-key CUDA-core dot products, which otherwise bound
// this kernel.
#include <cuda_bf16.h>
#include <algorithm>
#include <cstdint>
#include <mutex>

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "warp_mma.cuh"

namespace fl {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1); // + the producer warp
constexpr int kStages = 3;
constexpr uint32_t kKVBytes = kDecodeChunk * 64 * 2; // one chunk of K (or V), 16 KB
constexpr uint32_t kStageBytes = 2 * kKVBytes;
// block-table entries one split touches at most (pages of 16 keys)
constexpr int kSplitPages = kDecodeMaxSplitChunks * kDecodeChunk / 16;
__device__ uint32_t g_lib_error_word;

using wm::ldsm_x4;
using wm::ldsm_x4_t;
using wm::mma16816;
using wm::swz;

__device__ __forceinline__ uint32_t bf16_bits(const __nv_bfloat16 &x)
{
    return static_cast<uint32_t>(__bfloat16_as_ushort(x));
}

// Thread 0 of the producer: start the loads of chunk c of (b, hk) into stage
// (sk, sv), completing on `bar`.  `pages` holds the block-table entries of the
// split from page `pg_first` on.  A box is always written whole (rows past the
// tensor's end are zero-filled), so the expected bytes count whole boxes.
__device__ __forceinline__ void issue_chunk(const DecodeParams &p, const CUtensorMap *tm_k,
                                            const CUtensorMap *tm_v, int b, int hk, int c, int L,
                                            const int *pages, int pg_first, uint32_t sk, uint32_t sv,
                                            uint32_t bar)
{
    const int k0 = c * kDecodeChunk;
    if (!p.block_table) {
        // one box of min(cache length, kDecodeChunk) rows (p.page holds the
        // cache length for a contiguous cache)
        ptx::mbar_arrive_expect_tx(bar, 2u * 128u * static_cast<uint32_t>(min(p.page, kDecodeChunk)));
        ptx::tma_load_4d(sk, tm_k, bar, 0, k0, hk, b);
        ptx::tma_load_4d(sv, tm_v, bar, 0, k0, hk, b);
    } else if (p.page >= kDecodeChunk) {
        // the chunk is a slice of one page
        const int page = pages[k0 / p.page - pg_first];
        ptx::mbar_arrive_expect_tx(bar, 2 * kKVBytes);
        ptx::tma_load_4d(sk, tm_k, bar, 0, k0 % p.page, hk, page);
        ptx::tma_load_4d(sv, tm_v, bar, 0, k0 % p.page, hk, page);
    } else {
        const int nk = min(kDecodeChunk, L - k0);
        const int pg0 = k0 / p.page, npg = (nk + p.page - 1) / p.page;
        const uint32_t pbytes = static_cast<uint32_t>(p.page) * 128u;
        ptx::mbar_arrive_expect_tx(bar, 2u * pbytes * static_cast<uint32_t>(npg));
        for (int g = 0; g < npg; ++g) {
            const int page = pages[pg0 + g - pg_first];
            ptx::tma_load_4d(sk + g * pbytes, tm_k, bar, 0, 0, hk, page);
            ptx::tma_load_4d(sv + g * pbytes, tm_v, bar, 0, 0, hk, page);
        }
    }
}

// Output row r = s * G + g of (b, hk): head hk * G + g, new token s.
__device__ __forceinline__ void write_row(const DecodeParams &p, int b, int hk, int r, int dp, float o0,
                                          float o1, float m2, float l)
{
    const int s = r / p.G, h = hk * p.G + r % p.G;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat162 ov;
    ov.x = __float2bfloat16(o0 * inv);
    ov.y = __float2bfloat16(o1 * inv);
    *reinterpret_cast<__nv_bfloat162 *>(p.out + b * p.o_sb + s * p.o_ss + h * p.o_sh + 2 * dp) = ov;
    if (dp == 0 && p.lse)
        p.lse[b * p.l_sb + h * p.l_sh + s] = l > 0.f ? (m2 + __log2f(l)) * kLn2 : kNegInf;
}

__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeParams p)
{
    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = min(__ldg(p.kv_lens + b), p.max_kv);
    const int R = p.G * p.Sq;

    if (L <= 0) {
        // an empty cache: the rows have no key (O = 0, LSE = -inf)
        if (split == 0)
            for (int e = tid; e < R * 64; e += kThreads) {
                const int r = e >> 6, d = e & 63;
                const int s = r / p.G, h = hk * p.G + r % p.G;
                p.out[b * p.o_sb + s * p.o_ss + h * p.o_sh + d] = __float2bfloat16(0.f);
                if (d == 0 && p.lse)
                    p.lse[b * p.l_sb + h * p.l_sh + s] = kNegInf;
            }
        return;
    }
    const int split_keys = p.split_chunks * kDecodeChunk;
    const int n_splits = (L + split_keys - 1) / split_keys;
    if (split >= n_splits)
        return;
    const int c_lo = split * p.split_chunks;
    const int n_ch = min(p.split_chunks, (L + kDecodeChunk - 1) / kDecodeChunk - c_lo);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    uint8_t *sm = smem_raw + ((1024u - (base & 1023u)) & 1023u);
    const uint32_t s_stage = ptx::smem_u32(sm);                  // [kStages][K | V]
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    int *s_ticket = reinterpret_cast<int *>(empty + kStages);
    volatile uint32_t *s_abort = reinterpret_cast<volatile uint32_t *>(s_ticket + 1);
    int *s_pages = s_ticket + 2; // [kSplitPages] block-table entries of the split

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&empty[s]), kConsumerWarps);
        }
        *s_abort = 0;
        ptx::fence_mbarrier_init();
    }
    __syncthreads();

    WaitCtl wc;
    wc.abort_flag = s_abort;
    wc.timeout_cycles = p.timeout_ns * 21 / 10;
    wc.err_user = p.err_user;
    wc.err_lib = &g_lib_error_word;

    // rows: group rg of 16 (n_rg4 groups, padded to 1, 2 or 4); the chunk's
    // keys are split into kConsumerWarps / n_rg4 slices
    const int n_rg4 = R <= 16 ? 1 : (R <= 32 ? 2 : 4);
    const int slices = kConsumerWarps / n_rg4;
    const int slice_keys = kDecodeChunk / slices;
    const int g = lane >> 2, t = lane & 3;

    bool ok = true;
    int issued = 0;
    // unnormalised O of rows (g, g + 8) of the warp's group: o[n][0..1] row g,
    // columns 8n + 2t, +1; o[n][2..3] the same for row g + 8
    float o[8][4];
    float m_a = kNegInf, m_b = kNegInf, l_a = 0.f, l_b = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    if (warp == kConsumerWarps) {
        // ---- producer: the split's block-table entries first (one load per
        // lane instead of one dependent load before every chunk's copies)
        const int pg_first = p.block_table ? c_lo * kDecodeChunk / p.page : 0;
        if (p.block_table) {
            const int pg_last = (min(L, (c_lo + n_ch) * kDecodeChunk) - 1) / p.page;
            for (int e = lane; e <= pg_last - pg_first; e += 32)
                s_pages[e] = __ldg(p.block_table + static_cast<int64_t>(b) * p.bt_stride + pg_first + e);
            __syncwarp();
        }
        if (lane == 0)
            for (int i = 0; i < n_ch; ++i) {
                const int s = i % kStages;
                if (i >= kStages &&
                    !mbar_wait(ptx::smem_u32(&empty[s]), ((i / kStages) - 1) & 1, wc, W_KV_EMPTY)) {
                    ok = false;
                    break;
                }
                issue_chunk(p, &tm_k, &tm_v, b, hk, c_lo + i, L, s_pages, pg_first,
                            s_stage + s * kStageBytes, s_stage + s * kStageBytes + kKVBytes,
                            ptx::smem_u32(&full[s]));
                issued = i + 1;
            }
    } else {
        // ---- consumers
        const int rg = warp % n_rg4, ks = warp / n_rg4;
        const int r_a = rg * 16 + g, r_b = r_a + 8;
        const bool active = rg * 16 < R;
        // Q fragments (A operand, rows r_a / r_b, dims 16 k + 2t (+1, +8, +9))
        uint32_t qa[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            qa[k][0] = qa[k][1] = qa[k][2] = qa[k][3] = 0u;
        auto qrow = [&](int r) {
            const int s = r / p.G, h = hk * p.G + r % p.G;
            return p.q + b * p.q_sb + s * p.q_ss + h * p.q_sh;
        };
        if (r_a < R) {
            const __nv_bfloat16 *q = qrow(r_a);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                qa[k][0] = bf16_bits(q[16 * k + 2 * t]) | (bf16_bits(q[16 * k + 2 * t + 1]) << 16);
                qa[k][2] = bf16_bits(q[16 * k + 8 + 2 * t]) | (bf16_bits(q[16 * k + 9 + 2 * t]) << 16);
            }
        }
        if (r_b < R) {
            const __nv_bfloat16 *q = qrow(r_b);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                qa[k][1] = bf16_bits(q[16 * k + 2 * t]) | (bf16_bits(q[16 * k + 2 * t + 1]) << 16);
                qa[k][3] = bf16_bits(q[16 * k + 8 + 2 * t]) | (bf16_bits(q[16 * k + 9 + 2 * t]) << 16);
            }
        }
        // last key each row may see: L - 1, or L - Sq + s under the causal mask
        const int lim_all = p.causal ? L - p.Sq : L - 1; // the tightest of all rows
        const int lim_a = p.causal ? min(L - 1, L - p.Sq + r_a / p.G) : L - 1;
        const int lim_b = p.causal ? min(L - 1, L - p.Sq + r_b / p.G) : L - 1;
        const float sl2 = p.scale * kLog2e;
        const bool capped = p.softcap > 0.f;
        // cap * tanh(u), u = scale * z / cap, as cap (1 - 2 / (1 + e^(2u))), in log2 units
        const float cap_in = capped ? 2.f * p.scale * kLog2e / p.softcap : 0.f;
        const float cap_out = p.softcap * kLog2e;

        for (int i = 0; i < n_ch; ++i) {
            const int s = i % kStages;
            if (!warp_wait(ptx::smem_u32(&full[s]), (i / kStages) & 1, wc, W_KV_FULL)) {
                ok = false;
                break;
            }
            const uint32_t sk = s_stage + s * kStageBytes, sv = sk + kKVBytes;
            const int k0 = (c_lo + i) * kDecodeChunk;
            const int nk = min(kDecodeChunk, L - k0); // valid keys of the chunk
            for (int kb = ks * slice_keys; active && kb < (ks + 1) * slice_keys && kb < nk; kb += 32) {
                // ---- scores of rows (r_a, r_b) against keys kb .. kb + 31
                float sc[4][4];
#pragma unroll
                for (int n = 0; n < 4; ++n)
                    sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
                {
                    const int mi = lane >> 3, ri = lane & 7;
                    const int key = kb + ri + ((mi >> 1) << 3);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t b0, b1, b2, b3, b4, b5, b6, b7;
                        ldsm_x4(sk + swz(key, 2 * k + (mi & 1)), b0, b1, b2, b3);
                        ldsm_x4(sk + swz(key + 16, 2 * k + (mi & 1)), b4, b5, b6, b7);
                        mma16816(sc[0], qa[k], b0, b1);
                        mma16816(sc[1], qa[k], b2, b3);
                        mma16816(sc[2], qa[k], b4, b5);
                        mma16816(sc[3], qa[k], b6, b7);
                    }
                }
#pragma unroll
                for (int n = 0; n < 4; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sc[n][e] = capped ? cap_out * (1.f - 2.f * ptx::rcp_approx(1.f + ptx::ex2(sc[n][e] * cap_in)))
                                          : sc[n][e] * sl2;
                if (k0 + kb + 31 > lim_all) {
                    // keys past the cache or the causal limit of a row
#pragma unroll
                    for (int n = 0; n < 4; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = k0 + kb + 8 * n + 2 * t + (e & 1);
                            if (j > (e < 2 ? lim_a : lim_b))
                                sc[n][e] = kNegInf;
                        }
                }
                // ---- online softmax (rows r_a: e = 0, 1; r_b: e = 2, 3)
                float mx_a = m_a, mx_b = m_b;
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    mx_a = fmaxf(mx_a, fmaxf(sc[n][0], sc[n][1]));
                    mx_b = fmaxf(mx_b, fmaxf(sc[n][2], sc[n][3]));
                }
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
                const float use_a = mx_a == kNegInf ? 0.f : mx_a;
                const float use_b = mx_b == kNegInf ? 0.f : mx_b;
                const float al_a = ptx::ex2(m_a - use_a), al_b = ptx::ex2(m_b - use_b);
                m_a = mx_a;
                m_b = mx_b;
                float sum_a = 0.f, sum_b = 0.f;
                uint32_t pa[2][4]; // P as the A operand of two 16-key steps
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    const float p0 = ptx::ex2(sc[n][0] - use_a), p1 = ptx::ex2(sc[n][1] - use_a);
                    const float p2 = ptx::ex2(sc[n][2] - use_b), p3 = ptx::ex2(sc[n][3] - use_b);
                    sum_a += p0 + p1;
                    sum_b += p2 + p3;
                    pa[n >> 1][(n & 1) * 2] = ptx::pack_bf16(p0, p1);
                    pa[n >> 1][(n & 1) * 2 + 1] = ptx::pack_bf16(p2, p3);
                }
                l_a = fmaf(l_a, al_a, sum_a);
                l_b = fmaf(l_b, al_b, sum_b);
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    o[n][0] *= al_a;
                    o[n][1] *= al_a;
                    o[n][2] *= al_b;
                    o[n][3] *= al_b;
                }
                // ---- O += P V over the two 16-key steps
                {
                    const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int kk = kb + 16 * h;
                        const int key = kk + ri + ((mi & 1) << 3);
                        // keys past the chunk's valid ones hold arbitrary bytes:
                        // their P is 0, but 0 * NaN is not, so their V is zeroed
                        const bool ragged = kk + 16 > nk;
                        const uint32_t lo_ok = kk + 2 * t < nk ? 0xFFFFu : 0u;
                        const uint32_t hi_ok = kk + 2 * t + 1 < nk ? 0xFFFF0000u : 0u;
                        const uint32_t lo8 = kk + 8 + 2 * t < nk ? 0xFFFFu : 0u;
                        const uint32_t hi8 = kk + 9 + 2 * t < nk ? 0xFFFF0000u : 0u;
                        const uint32_t m0 = ragged ? (lo_ok | hi_ok) : 0xFFFFFFFFu;
                        const uint32_t m1 = ragged ? (lo8 | hi8) : 0xFFFFFFFFu;
#pragma unroll
                        for (int d = 0; d < 8; d += 2) {
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4_t(sv + swz(key, d + (mi >> 1)), b0, b1, b2, b3);
                            mma16816(o[d], pa[h], b0 & m0, b1 & m1);
                            mma16816(o[d + 1], pa[h], b2 & m0, b3 & m1);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(ptx::smem_u32(&empty[s]));
        }
        // the row sums are spread over the quad of lanes holding a row
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    }

    // ---- every chunk consumed (or the CTA gave up): the stages are free
    if (!__syncthreads_and(ok)) {
        if (warp == kConsumerWarps && lane == 0)
            for (int s = 0; s < kStages; ++s) {
                // the last chunk issued into stage s may still be landing
                const int last = issued - 1 - ((issued - 1 - s) % kStages + kStages) % kStages;
                if (last >= 0)
                    mbar_wait_drain(ptx::smem_u32(&full[s]), (last / kStages) & 1, wc, W_DRAIN);
            }
        return; // recorded in the error words; this sequence's outputs stay unwritten
    }

    // the warps' partials, [slice][row of 16 n_rg4][64] O and [slice][row] m, l
    const int rows4 = 16 * n_rg4;
    float *w_o = reinterpret_cast<float *>(sm);
    float *w_m = w_o + slices * rows4 * 64;
    float *w_l = w_m + slices * rows4;
    if (warp < kConsumerWarps) {
        const int rg = warp % n_rg4, ks = warp / n_rg4;
        const int r_a = rg * 16 + g, r_b = r_a + 8;
        float *oa = w_o + (ks * rows4 + r_a) * 64, *ob = w_o + (ks * rows4 + r_b) * 64;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            *reinterpret_cast<float2 *>(oa + 8 * n + 2 * t) = make_float2(o[n][0], o[n][1]);
            *reinterpret_cast<float2 *>(ob + 8 * n + 2 * t) = make_float2(o[n][2], o[n][3]);
        }
        if (t == 0) {
            w_m[ks * rows4 + r_a] = m_a;
            w_m[ks * rows4 + r_b] = m_b;
            w_l[ks * rows4 + r_a] = l_a;
            w_l[ks * rows4 + r_b] = l_b;
        }
    }
    __syncthreads();

    const size_t pair = static_cast<size_t>(b) * p.Hk + hk;
    float *po = p.ws_o + (pair * p.max_splits + split) * static_cast<size_t>(R) * 64;
    float *pml = p.ws_ml + (pair * p.max_splits + split) * static_cast<size_t>(R) * 2;
    for (int e = tid; e < R * 32; e += kThreads) {
        const int r = e >> 5, dp = e & 31;
        float M = kNegInf;
        for (int q = 0; q < slices; ++q)
            M = fmaxf(M, w_m[q * rows4 + r]);
        float o0 = 0.f, o1 = 0.f, l = 0.f;
        if (M != kNegInf)
            for (int q = 0; q < slices; ++q) {
                const float w = ptx::ex2(w_m[q * rows4 + r] - M);
                const float2 ov = *reinterpret_cast<const float2 *>(w_o + (q * rows4 + r) * 64 + 2 * dp);
                o0 = fmaf(w, ov.x, o0);
                o1 = fmaf(w, ov.y, o1);
                l = fmaf(w, w_l[q * rows4 + r], l);
            }
        if (n_splits == 1) {
            write_row(p, b, hk, r, dp, o0, o1, M, l);
        } else {
            *reinterpret_cast<float2 *>(po + r * 64 + 2 * dp) = make_float2(o0, o1);
            if (dp == 0)
                *reinterpret_cast<float2 *>(pml + 2 * r) = make_float2(M, l);
        }
    }
    if (n_splits == 1)
        return;

    // ---- the last split of (b, hk) merges every partial
    __threadfence();
    __syncthreads();
    if (tid == 0)
        *s_ticket = atomicAdd(p.ws_cnt + pair, 1);
    __syncthreads();
    if (*s_ticket != n_splits - 1)
        return;
    __threadfence();
    const float *o_all = p.ws_o + pair * p.max_splits * static_cast<size_t>(R) * 64;
    const float *ml_all = p.ws_ml + pair * p.max_splits * static_cast<size_t>(R) * 2;
    for (int e = tid; e < R * 32; e += kThreads) {
        const int r = e >> 5, dp = e & 31;
        float M = kNegInf;
        for (int q = 0; q < n_splits; ++q)
            M = fmaxf(M, __ldcg(ml_all + (static_cast<size_t>(q) * R + r) * 2));
        float o0 = 0.f, o1 = 0.f, l = 0.f;
        if (M != kNegInf)
            for (int q = 0; q < n_splits; ++q) {
                const size_t at = static_cast<size_t>(q) * R + r;
                const float w = ptx::ex2(__ldcg(ml_all + at * 2) - M);
                l = fmaf(w, __ldcg(ml_all + at * 2 + 1), l);
                o0 = fmaf(w, __ldcg(o_all + at * 64 + 2 * dp), o0);
                o1 = fmaf(w, __ldcg(o_all + at * 64 + 2 * dp + 1), o1);
            }
        write_row(p, b, hk, r, dp, o0, o1, M, l);
    }
    if (tid == 0)
        p.ws_cnt[pair] = 0; // ready for the next call
}

} // namespace

// ---- scratch for callers that cannot allocate device memory
//
// fl_attn_decode_static runs the same kernel with its workspace in this
// array instead of caller memory: for callers that cannot call cudaMalloc
// (one that must not take the device-wide synchronisation an allocation or
// a free can cause in a serving loop, or a plug-in that does not own the
// process's device allocator) and have no buffer to hand over.  Every GPU
// that loads this library holds the array until the process exits; every
// call shares it and finds the previous call's contents (the host clears the
// counters, the only part that must start at zero, before each launch), so
// calls that overlap on the GPU race.
namespace {
static __device__ __align__(256) uint8_t g_decode_scratch[kDecodeStaticScratch];

// The array's device address belongs to a CUDA context: a device's primary
// context, a context the caller made current, or the new primary context a
// cudaDeviceReset leads to all hold it at their own address.  Addresses are
// therefore cached per context, under the context's process-unique id (a
// handle value can be reused by a later context; the id cannot).
struct ScratchEntry {
    unsigned long long ctx_id;
    void *ptr;
};
constexpr int kScratchEntries = 64;
std::mutex g_scratch_mutex;
ScratchEntry g_scratch[kScratchEntries];
int g_scratch_used = 0, g_scratch_next = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <class Fn>
Fn driver_fn(const char *name)
{
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return reinterpret_cast<Fn>(f);
}

// Unique id of the calling thread's current context; false when there is
// none yet (the runtime creates the primary context on its first use).
bool current_ctx_id(unsigned long long &id)
{
    static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_current || !get_id)
        return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx)
        return false;
    return get_id(ctx, &id) == CUDA_SUCCESS;
}
} // namespace

// Device address of the scratch array in the current context.  The first call
// in a context looks it up (host code cannot use the array's name as a device
// address); later calls in that context return the cached pointer.
cudaError_t decode_static_scratch(void **ptr)
{
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    unsigned long long id = 0;
    if (current_ctx_id(id))
        for (int n = 0; n < g_scratch_used; ++n)
            if (g_scratch[n].ctx_id == id) {
                *ptr = g_scratch[n].ptr;
                return cudaSuccess;
            }
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch); // makes a context current if none was
    if (e != cudaSuccess)
        return e;
    if (current_ctx_id(id)) {
        ScratchEntry &slot = g_scratch_used < kScratchEntries ? g_scratch[g_scratch_used++]
                                                              : g_scratch[g_scratch_next++ % kScratchEntries];
        slot.ctx_id = id;
        slot.ptr = p;
    }
    *ptr = p;
    return cudaSuccess;
}

size_t decode_smem_bytes(int)
{
    // the stages (reused at the end for the warps' partials: at most 4 x 16
    // rows x 66 floats, 17 KB), the barriers, the ticket and the abort flag,
    // the split's block-table entries, and up to 1 KB of alignment padding
    return kStages * static_cast<size_t>(kStageBytes) + 2 * kStages * 8 + 8 + kSplitPages * 4 + 1024;
}

cudaError_t launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                          cudaStream_t stream)
{
    const size_t smem = decode_smem_bytes(p.G * p.Sq);
    cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    const dim3 grid(p.max_splits, p.Hk, p.B);
    decode_kernel<<<grid, kThreads, smem, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

} // namespace fl
