// fwd_decode.cu -- attention forward for serving with a KV cache (decode):
// a few new query tokens per sequence against a cached, variable-length and
// optionally paged K/V, with the causal (query row s of a sequence of L keys
// sits at position L - Sq + s) and softcap variants the pages serve LLaMA-3.2-1B
// with (talk notes, "End-to-end: LLaMA-3.2-1B (vLLM / Mooncake)").  The result
// is the same softmax(score_mod(scale q k^T) + mask) V as every other kind; the
// online-softmax recurrence is applied across key chunks (gist.science summary,
// "Methodology" item 3).
//
// Decode reads every cached key once and multiplies it by only G * Sq query
// rows (G = Hq / Hk query heads per KV head), so it is HBM-bound and runs on
// the CUDA cores, split over the keys (split-KV):
//   * one CTA per (key chunk of kChunk keys, KV head, sequence); chunks past a
//     sequence's length exit at once;
//   * the chunk's K and V (kChunk x 64 bf16 each) arrive by TMA into shared
//     memory (128-byte swizzle): one box for a contiguous cache, one box per
//     page for a paged one (pages that hold no key of the sequence are not
//     loaded);
//   * each thread scores one key against the R = G * Sq query rows (fp32 dot
//     products), a warp per row reduces the chunk's max m and sum l of
//     e^(z - m), and each warp accumulates P V over 32 of the chunk's keys
//     for every row (a lane per pair of output columns), the
//     warps' sums meeting in shared memory;
//   * the chunk's partial (O, m, l) goes to the workspace; an atomic ticket per
//     (sequence, KV head) makes the last chunk's CTA merge every partial
//     (O = sum_c e^(m_c - M) O_c / sum_c e^(m_c - M) l_c, LSE = M + ln of that
//     sum), write bf16 O and the natural-log LSE, and zero its counter again.
#include <cuda_bf16.h>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace fl {
namespace {

constexpr int kThreads = kDecodeChunk; // one thread per key of a chunk
constexpr uint32_t kKVBytes = kDecodeChunk * 64 * 2; // one chunk of K (or V), 16 KB

__device__ uint32_t g_lib_error_word;

// The K (or V) row of key t of the chunk: 16-byte chunk c at c ^ (t mod 8)
// (the 128-byte swizzle the TMA wrote the rows with).
__device__ __forceinline__ const uint4 *kv_chunk16(const uint8_t *base, int t, int c)
{
    return reinterpret_cast<const uint4 *>(base + t * 128 + ((c ^ (t & 7)) << 4));
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Six CTAs per SM (~35 KB of shared memory each for one new token per
// sequence) keep six chunks' loads in flight per SM.
__global__ void __launch_bounds__(kThreads, 6)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeParams p)
{
    const int c = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = min(p.kv_lens[b], p.max_kv);
    const int n_chunks = (L + kDecodeChunk - 1) / kDecodeChunk;
    const int R = p.G * p.Sq;

    if (L <= 0) {
        // an empty cache: the rows have no key (O = 0, LSE = -inf)
        if (c == 0)
            for (int e = tid; e < R * 64; e += kThreads) {
                const int r = e >> 6, d = e & 63;
                const int s = r / p.G, h = hk * p.G + r % p.G;
                p.out[b * p.o_sb + s * p.o_ss + h * p.o_sh + d] = __float2bfloat16(0.f);
                if (d == 0 && p.lse)
                    p.lse[b * p.l_sb + h * p.l_sh + s] = kNegInf;
            }
        return;
    }
    if (c >= n_chunks)
        return;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    uint8_t *sm = smem_raw + ((1024u - (base & 1023u)) & 1023u);
    uint8_t *sk = sm;                                   // [kDecodeChunk][128 B], swizzled
    uint8_t *sv = sm + kKVBytes;
    float *sq = reinterpret_cast<float *>(sm + 2 * kKVBytes);       // [R][64]
    float *sp = sq + R * 64;                                          // [R][kDecodeChunk]
    float *sml = sp + R * kDecodeChunk;                               // [R][2]: m, l
    uint64_t *bar_kv = reinterpret_cast<uint64_t *>(sml + 2 * R + (((2 * R) & 1) ? 1 : 0) + 2);
    int *s_ticket = reinterpret_cast<int *>(bar_kv + 1);
    volatile uint32_t *s_abort = reinterpret_cast<volatile uint32_t *>(s_ticket + 1);

    const int k0 = c * kDecodeChunk;
    const int nk = min(kDecodeChunk, L - k0); // valid keys of this chunk
    if (tid == 0) {
        ptx::mbar_init(ptx::smem_u32(bar_kv), 1);
        *s_abort = 0;
        ptx::fence_mbarrier_init();
        ptx::fence_proxy_async_smem();
        // loads: one box for a contiguous cache, one per touched page otherwise
        uint32_t bytes = 0;
        if (!p.block_table) {
            bytes = 2 * kKVBytes;
            ptx::mbar_arrive_expect_tx(ptx::smem_u32(bar_kv), bytes);
            ptx::tma_load_4d(ptx::smem_u32(sk), &tm_k, ptx::smem_u32(bar_kv), 0, k0, hk, b);
            ptx::tma_load_4d(ptx::smem_u32(sv), &tm_v, ptx::smem_u32(bar_kv), 0, k0, hk, b);
        } else if (p.page >= kDecodeChunk) {
            // the chunk is a slice of one page
            const int page = __ldg(p.block_table + static_cast<int64_t>(b) * p.bt_stride + k0 / p.page);
            bytes = 2 * kKVBytes;
            ptx::mbar_arrive_expect_tx(ptx::smem_u32(bar_kv), bytes);
            ptx::tma_load_4d(ptx::smem_u32(sk), &tm_k, ptx::smem_u32(bar_kv), 0, k0 % p.page, hk, page);
            ptx::tma_load_4d(ptx::smem_u32(sv), &tm_v, ptx::smem_u32(bar_kv), 0, k0 % p.page, hk, page);
        } else {
            const int pg0 = k0 / p.page, npg = (nk + p.page - 1) / p.page;
            const uint32_t pbytes = static_cast<uint32_t>(p.page) * 128u;
            bytes = 2u * pbytes * static_cast<uint32_t>(npg);
            ptx::mbar_arrive_expect_tx(ptx::smem_u32(bar_kv), bytes);
            for (int g = 0; g < npg; ++g) {
                const int page = __ldg(p.block_table + static_cast<int64_t>(b) * p.bt_stride + pg0 + g);
                ptx::tma_load_4d(ptx::smem_u32(sk + g * pbytes), &tm_k, ptx::smem_u32(bar_kv), 0, 0, hk,
                                 page);
                ptx::tma_load_4d(ptx::smem_u32(sv + g * pbytes), &tm_v, ptx::smem_u32(bar_kv), 0, 0, hk,
                                 page);
            }
        }
    }
    // query rows r = s * G + g (head hk * G + g, new token s), fp32
    for (int e = tid; e < R * 64; e += kThreads) {
        const int r = e >> 6, d = e & 63;
        const int s = r / p.G, h = hk * p.G + r % p.G;
        sq[e] = __bfloat162float(p.q[b * p.q_sb + s * p.q_ss + h * p.q_sh + d]);
    }
    __syncthreads();

    WaitCtl wc;
    wc.abort_flag = s_abort;
    wc.timeout_cycles = p.timeout_ns * 21 / 10;
    wc.err_user = p.err_user;
    wc.err_lib = &g_lib_error_word;
    // block-uniform: every thread leaves, or none (a later __syncthreads needs all)
    if (!__syncthreads_and(mbar_wait_drain(ptx::smem_u32(bar_kv), 0, wc, W_KV_FULL)))
        return; // recorded in the error words; this sequence's outputs stay unwritten

    // ---- scores: thread tid scores key k0 + tid against every row
    const int pos0 = L - p.Sq; // position of new token 0
    if (tid < kDecodeChunk) {
        const bool valid = tid < nk;
        uint32_t kw[32];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
            const uint4 w = *kv_chunk16(sk, tid, q4);
            kw[4 * q4] = w.x;
            kw[4 * q4 + 1] = w.y;
            kw[4 * q4 + 2] = w.z;
            kw[4 * q4 + 3] = w.w;
        }
        const int j = k0 + tid;
        for (int r = 0; r < R; ++r) {
            const float4 *qr = reinterpret_cast<const float4 *>(sq + r * 64);
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) {
                const float4 qv = qr[q4];
                a0 = fmaf(qv.x, bf_lo(kw[2 * q4]), a0);
                a1 = fmaf(qv.y, bf_hi(kw[2 * q4]), a1);
                a0 = fmaf(qv.z, bf_lo(kw[2 * q4 + 1]), a0);
                a1 = fmaf(qv.w, bf_hi(kw[2 * q4 + 1]), a1);
            }
            float z = (a0 + a1) * p.scale;
            if (p.softcap > 0.f)
                z = p.softcap * tanhf(z / p.softcap);
            const bool ok = valid && (!p.causal || j <= pos0 + r / p.G);
            sp[r * kDecodeChunk + tid] = ok ? z : kNegInf;
        }
    }
    __syncthreads();

    // ---- per row: the chunk's max and sum, P = e^(z - m) in place
    for (int r = warp; r < R; r += kThreads / 32) {
        float *row = sp + r * kDecodeChunk;
        float m = kNegInf;
        for (int t = lane; t < kDecodeChunk; t += 32)
            m = fmaxf(m, row[t]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        for (int t = lane; t < kDecodeChunk; t += 32) {
            const float e = m == kNegInf ? 0.f : expf(row[t] - m);
            row[t] = e;
            l += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            sml[2 * r] = m;
            sml[2 * r + 1] = l;
        }
    }
    __syncthreads();

    // ---- partial O: warp w takes keys [32 w, 32 w + 32) of the chunk, lane l
    // the output columns 2l and 2l + 1 of every row; the warps' sums
    // meet in shared memory (the query rows' space, free after the scores)
    for (int e = tid; e < R * 64; e += kThreads)
        sq[e] = 0.f;
    __syncthreads();
    const int dp = lane;
    const int t0 = warp * 32, t1 = min(t0 + 32, nk);
    for (int r0 = 0; r0 < R; r0 += 4) {
        float acc[4][2];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
            acc[rr][0] = acc[rr][1] = 0.f;
        const int nr = min(4, R - r0);
        if (nr == 4) {
            for (int t = t0; t < t1; ++t) {
                const uint32_t vw = reinterpret_cast<const uint32_t *>(kv_chunk16(sv, t, dp >> 2))[dp & 3];
                const float v0 = bf_lo(vw), v1 = bf_hi(vw);
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const float pt = sp[(r0 + rr) * kDecodeChunk + t];
                    acc[rr][0] = fmaf(pt, v0, acc[rr][0]);
                    acc[rr][1] = fmaf(pt, v1, acc[rr][1]);
                }
            }
        } else {
            for (int t = t0; t < t1; ++t) {
                const uint32_t vw = reinterpret_cast<const uint32_t *>(kv_chunk16(sv, t, dp >> 2))[dp & 3];
                const float v0 = bf_lo(vw), v1 = bf_hi(vw);
                for (int rr = 0; rr < nr; ++rr) {
                    const float pt = sp[(r0 + rr) * kDecodeChunk + t];
                    acc[rr][0] = fmaf(pt, v0, acc[rr][0]);
                    acc[rr][1] = fmaf(pt, v1, acc[rr][1]);
                }
            }
        }
        if (t0 < t1)
            for (int rr = 0; rr < nr; ++rr) {
                atomicAdd(sq + (r0 + rr) * 64 + 2 * dp, acc[rr][0]);
                atomicAdd(sq + (r0 + rr) * 64 + 2 * dp + 1, acc[rr][1]);
            }
    }
    __syncthreads();
    const int rg = warp;
    const size_t unit = static_cast<size_t>(b) * p.Hk + hk;
    float *po = p.ws_o + (unit * p.max_chunks + c) * static_cast<size_t>(R) * 64;
    float *pml = p.ws_ml + (unit * p.max_chunks + c) * static_cast<size_t>(R) * 2;
    for (int e = tid; e < R * 64; e += kThreads)
        po[e] = sq[e];
    for (int e = tid; e < 2 * R; e += kThreads)
        pml[e] = sml[e];

    // ---- the last chunk of (b, hk) merges every partial
    __threadfence();
    __syncthreads();
    if (tid == 0)
        *s_ticket = atomicAdd(p.ws_cnt + unit, 1);
    __syncthreads();
    if (*s_ticket != n_chunks - 1)
        return;
    __threadfence();
    const float *o_all = p.ws_o + unit * p.max_chunks * static_cast<size_t>(R) * 64;
    const float *ml_all = p.ws_ml + unit * p.max_chunks * static_cast<size_t>(R) * 2;
    for (int r = rg; r < R; r += kThreads / 32) {
        float M = kNegInf;
        for (int cc = 0; cc < n_chunks; ++cc)
            M = fmaxf(M, __ldcg(ml_all + (static_cast<size_t>(cc) * R + r) * 2));
        float Lsum = 0.f, o0 = 0.f, o1 = 0.f;
        if (M != kNegInf)
            for (int cc = 0; cc < n_chunks; ++cc) {
                const size_t at = static_cast<size_t>(cc) * R + r;
                const float w = expf(__ldcg(ml_all + at * 2) - M);
                Lsum = fmaf(w, __ldcg(ml_all + at * 2 + 1), Lsum);
                o0 = fmaf(w, __ldcg(o_all + at * 64 + 2 * dp), o0);
                o1 = fmaf(w, __ldcg(o_all + at * 64 + 2 * dp + 1), o1);
            }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        const int s = r / p.G, h = hk * p.G + r % p.G;
        __nv_bfloat162 ov;
        ov.x = __float2bfloat16(o0 * inv);
        ov.y = __float2bfloat16(o1 * inv);
        *reinterpret_cast<__nv_bfloat162 *>(p.out + b * p.o_sb + s * p.o_ss + h * p.o_sh + 2 * dp) = ov;
        if (dp == 0 && p.lse)
            p.lse[b * p.l_sb + h * p.l_sh + s] = Lsum > 0.f ? M + logf(Lsum) : kNegInf;
    }
    if (tid == 0)
        p.ws_cnt[unit] = 0; // ready for the next call
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

std::mutex g_scratch_mutex;
void *g_scratch_ptr[64];
}

// Device address of the scratch array on the current device.  The first call
// on a device looks it up (host code cannot use the array's name as a device
// address); later calls return the cached pointer.
cudaError_t decode_static_scratch(void **ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

size_t decode_smem_bytes(int R)
{
    return 2 * static_cast<size_t>(kKVBytes) + static_cast<size_t>(R) * 64 * 4 +
           static_cast<size_t>(R) * kDecodeChunk * 4 + static_cast<size_t>(2 * R + 2) * 4 + 64 + 1024;
}

cudaError_t launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                          cudaStream_t stream)
{
    const int R = p.G * p.Sq;
    const size_t smem = decode_smem_bytes(R);
    cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    const dim3 grid(p.max_chunks, p.Hk, p.B);
    decode_kernel<<<grid, kThreads, smem, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

} // namespace fl
