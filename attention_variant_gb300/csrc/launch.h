// launch.h -- host-side interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Internal to the library.  Under the runtime
// compiler (NVRTC) only the parameter structs are seen.
#pragma once

#include <cuda_bf16.h>
#ifndef __CUDACC_RTC__
#include <cuda.h>
#include <cuda_runtime.h>
#endif

#include "common.cuh"

namespace fl {

// Parameters of the standard (MHA / GQA) kernel.  Strides are in elements.
struct StdParams {
    GridSpec grid;
    MaskSpec mask;
    int head_dim;         // D = Dv: 32, 64 or 128
    int score_mod;
    float qk_log2;        // scale * log2(e)
    float softcap_in;     // 2 * scale * log2(e) / cap
    float softcap_out;    // cap * log2(e)
    float scale;          // scale (the `score` of a score_mod expression is scale * q.k)
    const float *alibi_slopes;
    float alibi_exp_coef; // default slopes: 2^(alibi_exp_coef * (h + 1)), coef = -8 / Hq
    __nv_bfloat16 *out;
    int64_t o_sb, o_ss, o_sh;
    float *lse;
    int64_t l_sb, l_sh;
    int32_t *tile_counts; // [B][Hq][nq] or null
    uint32_t *err_user;
    int inject;
    uint64_t timeout_ns;
};

// Parameters of the differential-attention kernel (D = 64, Dv = 64 or 128).
struct DiffParams {
    int B, H, Hk, G, nq;
    int dv;               // 64 or 128
    int64_t n_items;
    int lpt, group;
    MaskSpec mask;        // none or causal
    float qk_log2;        // scale * log2(e)
    float lambda;
    __nv_bfloat16 *out;   // [B, S, H, Dv]
    int64_t o_sb, o_ss, o_sh;
    float *lse;           // [2, B, H, S] or null
    int64_t l_s2, l_sb, l_sh;
    int32_t *tile_counts; // [B][H][nq] or null
    uint32_t *err_user;
    uint64_t timeout_ns;
};

#ifndef __CUDACC_RTC__
cudaError_t launch_diff(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const DiffParams &p, int grid, cudaStream_t stream);
#endif

// Parameters of the Evoformer kernel (c = 32 or 64) over a [batch, sequence, head, c]
// view: row pass batch = MSA row, sequence = residue; column pass the reverse.
// Work items are (head, query block, chunk of `chunk` batch indices).
struct EvoParams {
    GridSpec grid;          // B, Hq (= heads), nq used
    MaskSpec mask;          // kind NONE; S = length of the attended axis
    int head_dim;           // c: 32 or 64
    int64_t n_items;
    int chunk;
    float qk_log2;          // scale * log2(e)
    float qk_scale;         // scale
    const __nv_bfloat16 *bias; // row pass only (its TMA map is passed separately)
    int bias_rows;          // 0: one bias for every batch index; else a bias per stack of
                            //   bias_rows consecutive batch indices (work items never
                            //   straddle two stacks)
    const __nv_bfloat16 *gate;
    int64_t g_sb, g_si, g_sh;
    __nv_bfloat16 *out;
    int64_t o_sb, o_si, o_sh;
    float *lse;             // [batch, head, sequence] or null
    int64_t l_sb, l_sh;
    int32_t *tile_counts;   // [batch][head][nq] or null
    const void *kmask;      // MSA mask or null: key j of batch index b is removed where
    int64_t km_sb, km_sk;   //   kmask[b * km_sb + j * km_sk] is zero (element strides)
    int km_f32;             //   fp32 entries (else bf16)
    uint32_t *err_user;
    uint64_t timeout_ns;
};

// ---- backward of the standard kind (bwd_standard.cu)
constexpr int kBwdBlock = 64;   // query / key rows per streamed tile
constexpr int kBwdDqRows = 128; // query rows per dQ CTA
constexpr int kBwdKvKeys = 128; // keys per dK / dV CTA
constexpr int kBwdThreads = 384;

// Per query row of the backward's workspace: LSE log2 e, rowsum(dO O) and the
// row's allowed key interval [lo, hi).
struct BwdRowStat {
    float lse2, d;
    int lo, hi;
};

struct BwdParams {
    int B, Hq, Hk, S, S_pad;      // S_pad: S rounded up to 128 (a multiple of kBwdBlock)
    MaskSpec mask;
    float scale;
    int score_mod;                // MOD_NONE, MOD_ALIBI or MOD_SOFTCAP
    float softcap;                // cap (softcap)
    const float *alibi_slopes;    // [Hq] or null: 2^(alibi_exp_coef (h + 1))
    float alibi_exp_coef;
    const __nv_bfloat16 *q, *k, *v, *o, *dout; // element strides (batch, position, head):
    int64_t q_sb, q_ss, q_sh, k_sb, k_ss, k_sh, v_sb, v_ss, v_sh;
    int64_t o_sb, o_ss, o_sh, do_sb, do_ss, do_sh;
    const float *lse;             // [B, Hq, S] natural log
    int64_t l_sb, l_sh;
    __nv_bfloat16 *dq, *dk, *dv;
    int64_t dq_sb, dq_ss, dq_sh, dk_sb, dk_ss, dk_sh, dv_sb, dv_ss, dv_sh;
    BwdRowStat *ws_stats;         // [B][Hq][S_pad]
    uint32_t *err_user;
    uint64_t timeout_ns;
};

// ---- backward of the differential kind (bwd_diff.cu): the combining step
// out[row, 0:64] = sum_p coef[p] in_p[row, 0:64] (fp32 sum of bf16 partials);
// row = (b * S + position) * heads + head of the output view.
struct DiffCombine {
    int64_t rows, S, heads;
    const __nv_bfloat16 *in[2]; // contiguous [rows][64]; in[1] may be null
    float coef[2];
    __nv_bfloat16 *out;         // element strides (batch, position, head); 64 columns contiguous
    int64_t o_sb, o_ss, o_sh;
};

// ---- serving with a KV cache (fwd_decode.cu)
constexpr int kDecodeChunk = 128; // keys per pipeline stage
constexpr int kDecodeMaxSplitChunks = 8; // chunks per CTA (split) at most
constexpr int kDecodeMaxRows = 64; // G * Sq query rows per (sequence, KV head)

struct DecodeParams {
    int B, Hk, G, Sq;
    int max_kv;
    int split_chunks, max_splits; // chunks per split; splits of the longest sequence
    int page;                     // keys per page (paged cache)
    int64_t bt_stride;            // block_table row stride
    const int32_t *kv_lens;       // [B]
    const int32_t *block_table;   // [B][bt_stride] or null (contiguous cache)
    const __nv_bfloat16 *q;       // [B, Sq, Hq, 64] element strides:
    int64_t q_sb, q_ss, q_sh;
    __nv_bfloat16 *out;
    int64_t o_sb, o_ss, o_sh;
    float *lse;                   // [B, Hq, Sq] or null
    int64_t l_sb, l_sh;
    float scale, softcap;         // softcap 0: none
    int causal;
    float *ws_o;                  // [B][Hk][max_splits][R][64]
    float *ws_ml;                 // [B][Hk][max_splits][R][2]: base-2 max, sum
    int *ws_cnt;                  // [B][Hk], zero before the launch
    uint32_t *err_user;
    uint64_t timeout_ns;
};

#ifndef __CUDACC_RTC__
cudaError_t launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                          cudaStream_t stream);
size_t decode_smem_bytes(int R);

// Size of the library's own decode scratch array (fl_attn_decode_static).
constexpr size_t kDecodeStaticScratch = size_t(64) << 20;
cudaError_t decode_static_scratch(void **ptr);

cudaError_t launch_diff_bwd_combine(const DiffCombine &c, int sm_count, cudaStream_t stream);

cudaError_t launch_evo(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tb, const EvoParams &p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_prep(const BwdParams &p, cudaStream_t stream);
// Dynamic shared memory and block count of the fused dK/dV + dQ launch.
size_t bwd_smem_bytes();
int64_t bwd_fused_blocks(const BwdParams &p);
// The main backward kernel specialised for a translated expression `cuda`
// with derivative `grad` (run-time compiled, like launch_standard_expr);
// launch_bwd_prep must have run first on the same stream.
cudaError_t launch_bwd_expr(const CUtensorMap &tq, const CUtensorMap &tdo, const CUtensorMap &tk,
                            const CUtensorMap &tv, const CUtensorMap &tq128, const CUtensorMap &tdo128,
                            const CUtensorMap &tk128, const CUtensorMap &tv128, const BwdParams &p,
                            cudaStream_t stream, const char *cuda, const char *grad, char *err, size_t err_n);
cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tdo, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tq128, const CUtensorMap &tdo128,
                       const CUtensorMap &tk128, const CUtensorMap &tv128, const BwdParams &p,
                       cudaStream_t stream);
#endif

// Keys per K/V tile of the standard kernel for head dimension D (its TMEM
// budget: see fwd_standard.cu), its threads per CTA and the registers per
// thread it must be compiled to.
__host__ __device__ constexpr int std_key_tile(int D) { return D == 128 ? 64 : D == 64 ? 112 : 128; }
constexpr int kStdThreads = 384;
constexpr int kStdRegs = 168;
// Keys per K/V tile of the differential kernel for value head dimension Dv
// (its TMEM budget: see fwd_diff.cu).
__host__ __device__ constexpr int diff_key_tile(int dv) { return dv == 128 ? 80 : 112; }

#ifndef __CUDACC_RTC__
cudaError_t launch_standard(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const StdParams &p, int grid, cudaStream_t stream);
size_t standard_smem_bytes(int head_dim);

// ---- score_mod expressions (score_expr.cu)
// Checks `expr` against the expression grammar of fl_attn.h and writes the
// equivalent fp32 CUDA expression to `cuda` (NUL-terminated, at most `n`
// bytes); false with a message in `err` otherwise.
bool score_expr_translate(const char *expr, char *cuda, size_t n, char *err, size_t err_n);
// The same, also writing the derivative of the expression with respect to
// `score` (forward-mode differentiation through the grammar) to `grad`.
bool score_expr_translate_grad(const char *expr, char *cuda, size_t n, char *grad, size_t grad_n, char *err,
                               size_t err_n);
// Runs the runtime compilation of the standard kernel for the translated
// expression `cuda`, and of the backward kernels for it and its derivative
// `grad` (unless null), without loading them (needs no device).
bool score_expr_compile_only(const char *cuda, const char *grad, char *err, size_t err_n);
// The standard kernel specialised for the translated expression `cuda`:
// compiled at run time on first use (per device and expression), then
// launched like launch_standard.  Errors other than CUDA ones are described
// in `err`.
cudaError_t launch_standard_expr(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const StdParams &p, int grid, cudaStream_t stream, const char *cuda,
                                 char *err, size_t err_n);
#endif

}  // namespace fl
