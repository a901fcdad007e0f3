/*
 * fl_attn.h -- C ABI of the GB300 fused attention-variant forward.
 *
 * One call computes, for every (batch, query head, query row i),
 *
 *     O_i   = sum_j softmax_j( z_ij ) v_j
 *     LSE_i = ln sum_j exp( z_ij )
 *     z_ij  = score_mod( scale * q_i . k_j ) + bias_ij    (or -inf where masked)
 *
 * in a single pass over the keys with an online softmax: a running maximum and
 * a running sum per query row, the sum (and the output accumulator) rescaled
 * whenever the maximum moves, so that no S x S score or probability tensor is
 * ever written to device memory.  This is the fused kernel shape the
 * Flashlight pages describe (gist.science summary, "Methodology" items 2-4:
 * dimension demotion fuses max() into QK^T, the homomorphism
 * e^(x-y) = e^x / e^y turns the two-pass stable softmax into a one-pass
 * online one, and tiling-aware dimension elimination fuses softmax(QK^T)V;
 * talk notes, "Compiler design" 1-4).  The variants are the ones the talk
 * notes evaluate ("Evaluation: FlexAttention-supported variants" and
 * "Evaluation: complex variants"): vanilla, ALiBi, softcap, causal, sliding
 * window, PrefixLM, document mask, MHA and GQA, differential attention, and
 * the AlphaFold Evoformer row- and column-wise gated self-attention with pair
 * bias.  The pages give no formula for these; the ones used are stated at
 * each enum below.
 *
 * Conventions shared by every entry point
 *  - Every tensor is a caller-owned DEVICE buffer of the current CUDA device
 *    (e.g. a torch tensor).  The library never allocates, frees or retains
 *    caller memory.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream).  A returned FL_OK means the work was enqueued.
 *  - Functions never throw.  Argument validation happens before any CUDA
 *    call; a failed validation launches nothing and leaves outputs
 *    untouched.  fl_attn_last_error() then describes the failure.
 *  - The library is thread-safe for concurrent calls on different streams.
 */
#ifndef FL_ATTN_H
#define FL_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FL_ATTN_VERSION 1

typedef struct CUstream_st *fl_stream_t; /* identical to cudaStream_t */

typedef enum {
    FL_OK = 0,
    FL_ERR_INVALID_ARG = 1,    /* null pointer, bad rank/shape/dtype, bad parameter */
    FL_ERR_UNSUPPORTED = 2,    /* valid request outside the compiled kernel set */
    FL_ERR_ALIGNMENT = 3,      /* base pointer or stride not 16-byte aligned */
    FL_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
    FL_ERR_DEVICE_TIMEOUT = 5, /* reported through error_word: a device wait ran out */
    FL_ERR_NO_DEVICE = 6       /* no CUDA device, or not an sm_103 (GB300) device */
} fl_status;

typedef enum { FL_BF16 = 0, FL_F32 = 1 } fl_dtype;

/* A strided view.  sizes/strides are in ELEMENTS, outermost first; the
 * innermost stride must be 1.  All other strides of bf16 tensors must be
 * multiples of 8 elements (16 bytes) and every ptr 16-byte aligned. */
typedef struct {
    void *ptr;
    int32_t dtype; /* fl_dtype */
    int32_t ndim;
    int64_t sizes[5];
    int64_t strides[5];
} fl_tensor;

typedef enum {
    FL_KIND_STANDARD = 0, /* MHA / GQA with score_mod and mask */
    FL_KIND_DIFF = 1,     /* differential attention, two softmax streams, one V */
    FL_KIND_EVO_ROW = 2,  /* Evoformer MSA row-wise gated attention + pair bias */
    FL_KIND_EVO_COL = 3   /* Evoformer MSA column-wise gated attention */
} fl_kind;

typedef enum {
    FL_MOD_NONE = 0,
    FL_MOD_ALIBI = 1,   /* z += -slope_h * |i - j|, slope_h = 2^(-8 (h+1) / Hq) by default */
    FL_MOD_SOFTCAP = 2, /* z = cap * tanh(z / cap) */
    FL_MOD_EXPR = 3     /* z = the expression desc->score_mod_expr (FL_KIND_STANDARD) */
} fl_score_mod;

/*
 * score_mod expressions (FL_MOD_EXPR).  The logit of (query row q_idx, key
 * kv_idx) of batch b and query head h is the value of a user expression over
 *     score   scale * q . k (the scaled dot product)
 *     b, h, q_idx, kv_idx
 * in this grammar (every value fp32; a comparison gives 1 or 0; '/' is the
 * fast division, within 2 ulp; exp and exp2 use the hardware 2^x, relative
 * error about 2^-22; tanh is 1 - 2 / (1 + e^(2x)) on it, absolute error
 * about 1e-7):
 *     expr    := sum [ relop sum ]        relop: < <= > >= == !=  (no chains)
 *     sum     := term { (+ | -) term }
 *     term    := unary { (* | /) unary }
 *     unary   := (- | +) unary | primary
 *     primary := number | score | b | h | q_idx | kv_idx | inf
 *              | tanh(e) | exp(e) | exp2(e) | log(e) | log2(e) | sqrt(e)
 *              | abs(e) | floor(e) | min(e, e) | max(e, e)
 *              | where(c, x, y)           (x where c != 0, else y)
 *              | ( expr )
 * e.g. "20 * tanh(score / 20)" (softcap), "score - 0.5 * abs(q_idx - kv_idx)"
 * (ALiBi with slope 0.5), "where(kv_idx <= q_idx, score, -inf)" (a causal
 * mask written as a score_mod).  -inf removes the pair; the mask in the desc
 * still applies on top.  This is the pages' generic-variant interface: the
 * expression is fused into the same single-pass kernel as the built-in
 * variants (talk notes, "Compiler design" and the comparison with
 * FlexAttention).  The first call with a new expression on a device compiles
 * the kernel for it at run time (NVRTC, about two seconds; the CUDA toolkit's
 * libnvrtc.so.13 and include directory -- $CUDA_HOME, else /usr/local/cuda --
 * must be present, or the call returns FL_ERR_UNSUPPORTED); later calls reuse
 * it.  A string outside the grammar returns FL_ERR_INVALID_ARG.
 */

typedef enum {
    FL_MASK_NONE = 0,
    FL_MASK_CAUSAL = 1, /* key j allowed for query i iff j <= i */
    FL_MASK_WINDOW = 2, /* j <= i and i - j < window */
    FL_MASK_PREFIX = 3, /* j <= i or j < prefix (bidirectional over the first prefix keys) */
    FL_MASK_DOC = 4     /* same document and j <= i */
} fl_mask;

/* Test-only fault injection: the library itself never sets these. */
typedef enum {
    FL_INJECT_NONE = 0,
    FL_INJECT_DROP_KV_LOAD = 1 /* one K/V tile load of CTA 0 is never issued, so the
                                  consumer's bounded wait runs out */
} fl_inject;

/* Bits the kernel ORs into error_word. */
#define FL_DEVERR_TIMEOUT 0x1u        /* a bounded wait ran out; the CTA quit cleanly */
#define FL_DEVERR_WHERE_SHIFT 8       /* bits 8..15: which wait (diagnostic) */

typedef struct {
    int32_t kind;            /* fl_kind */
    int32_t score_mod;       /* fl_score_mod (FL_KIND_STANDARD only) */
    float softcap;           /* cap > 0 for FL_MOD_SOFTCAP */
    int32_t mask;            /* fl_mask (STANDARD and DIFF; DIFF takes NONE or CAUSAL) */
    int32_t window;          /* FL_MASK_WINDOW, >= 1 */
    int32_t prefix;          /* FL_MASK_PREFIX, >= 0 */
    const int32_t *doc_offsets; /* FL_MASK_DOC: device int32 [B][doc_stride]; row b holds the
                                   ascending document starts of batch b (first 0), padded
                                   with S */
    int32_t doc_stride;      /* entries per row of doc_offsets (max documents + 1) */
    int32_t gqa_group;       /* Hq / Hk; 0 derives it from the shapes, else must match */
    float diff_lambda;       /* FL_KIND_DIFF: O = O_1 - lambda O_2 */
    float scale;             /* 0 means 1 / sqrt(D) */
    const float *alibi_slopes; /* device float [Hq], or NULL for 2^(-8 (h+1) / Hq) */
    int32_t *debug_tile_counts; /* NULL, or device int32 [batch][heads][ceil(S/128)]: the
                                   number of key tiles each 128-row query block visited
                                   (key-tile width from fl_attn_tile_shape: 128 for the
                                   standard kind at D = 32, 112 at D = 64, 64 at D = 128; 112 for
                                   the differential kind at Dv = 64, 80 at Dv = 128; 128
                                   for the Evoformer kinds) */
    uint32_t *error_word;    /* NULL, or a device word the kernel ORs FL_DEVERR_* into */
    int32_t debug_inject;    /* fl_inject; 0 in normal use */
    uint32_t wait_timeout_us; /* bound of every device-side wait; 0 means 2,000,000 */
    const char *score_mod_expr; /* FL_MOD_EXPR: the expression (host string), else unused */
} fl_attn_variant_desc;

/*
 * fl_attn_fwd -- fused attention forward.
 *
 * Layouts (sizes in this logical order; any strides subject to the fl_tensor
 * rules), all bf16 except lse (fp32):
 *   FL_KIND_STANDARD  q [B,S,Hq,D]  k [B,S,Hk,D]  v [B,S,Hk,Dv]  out [B,S,Hq,Dv]
 *                     lse [B,Hq,S] or NULL.        bias, gate: NULL.
 *   FL_KIND_DIFF      q [2,B,S,H,D] k [2,B,S,Hk,D] v [B,S,Hk,Dv] out [B,S,H,Dv]
 *                     lse [2,B,H,S] or NULL (one LSE per softmax stream).
 *                     out = softmax(scale Q1 K1^T) V - lambda softmax(scale Q2 K2^T) V.
 *   FL_KIND_EVO_ROW   q,k,v,gate,out [N_seq,N_res,H,c]; bias [H,N_res,N_res];
 *                     attention over residues for each MSA row:
 *                     out = sigmoid(gate) * softmax(scale q k^T + bias) v;
 *                     lse [N_seq,H,N_res] or NULL.
 *   FL_KIND_EVO_COL   q,k,v,gate,out [N_seq,N_res,H,c]; bias NULL;
 *                     attention over MSA rows for each residue (axis 0);
 *                     lse [N_res,H,N_seq] or NULL.
 * lse is natural-log; its innermost stride must be 1.
 *
 * Supported shapes: STANDARD D = Dv in {32, 64, 128}; DIFF D = 64, Dv = 64
 * or 128 with mask none or causal; EVO c = 32 or 64, any N_res (the row pass
 * keeps a query block's bias rows in shared memory for c = 32 and N_res <= 384,
 * and streams them per key tile otherwise).  Other shapes return
 * FL_ERR_UNSUPPORTED.  The bias may be passed with any strides obeying the
 * fl_tensor rules (for example a [N_res,N_res,H] tensor viewed as
 * [H,N_res,N_res]).  Evoformer sequence lengths must keep every stride a
 * multiple of 16 bytes (c = 32 bf16 rows always do; the bias row stride must
 * be a multiple of 8 elements: pad N_res or the bias rows otherwise).
 * STANDARD launches of 2^31 or more work items (pairs of 128-row query
 * blocks per batch and head) also return FL_ERR_UNSUPPORTED.
 *
 * Returns FL_OK when enqueued.  Device-side failures (a wait that ran out)
 * are reported asynchronously through desc->error_word.
 */
fl_status fl_attn_fwd(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                      const fl_tensor *out, const fl_tensor *lse,
                      const fl_attn_variant_desc *desc, const fl_tensor *bias,
                      const fl_tensor *gate, fl_stream_t stream);

/*
 * fl_attn_evoformer -- the Evoformer kinds over a batch of MSA stacks, with an
 * optional MSA mask (AlphaFold2 context: talk notes, "End-to-end: AlphaFold2").
 *
 * desc->kind is FL_KIND_EVO_ROW or FL_KIND_EVO_COL; everything fl_attn_fwd
 * says of those kinds holds per stack.  Shapes (bf16 unless noted):
 *   q, k, v, gate, out  [B, N_seq, N_res, H, c]   (or [N_seq, N_res, H, c]: B = 1)
 *   bias (row pass)     [B, H, N_res, N_res], or [H, N_res, N_res] shared by all stacks
 *   msa_mask            NULL, or [B, N_seq, N_res] / [N_seq, N_res] shared, bf16 or
 *                       fp32: where msa_mask[s, r] is 0 the entry is removed as a key --
 *                       residue r for MSA row s in the row pass, MSA row s for residue
 *                       r in the column pass.  A query row left with no key gives
 *                       O = 0 and LSE = -inf.
 *   lse                 NULL, or [B, N_seq, H, N_res] (row) / [B, N_res, H, N_seq] (col)
 * The stack axis may have any stride that is a positive multiple of 16 bytes.
 * Each stack is one kernel launch on `stream`.  Every argument is validated
 * before the first launch.
 */
fl_status fl_attn_evoformer(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                            const fl_tensor *out, const fl_tensor *lse,
                            const fl_attn_variant_desc *desc, const fl_tensor *bias,
                            const fl_tensor *gate, const fl_tensor *msa_mask, fl_stream_t stream);

/*
 * fl_attn_bwd -- backward of the standard kind: dQ, dK, dV of
 *     O = softmax(scale Q K^T + mask) V
 * given the forward's out and (natural-log) lse and the output gradient
 * dout.  The pages name the backward pass as the fused kernels' next step
 * (gist.science summary, "Limitations and future work").  P is recomputed
 * from Q, K and the LSE; dS = P (dP - D) with D_i = sum_d dout_id out_id.
 *   q, out, dout, dq [B, S, Hq, 64]; k, v, dk, dv [B, S, Hk, 64]; lse [B, Hq, S] fp32
 *   desc: kind FL_KIND_STANDARD, any score_mod (FL_MOD_EXPR included: the
 *   backward kernels are compiled at run time with the expression and its
 *   derivative with respect to `score`, derived through the grammar), any
 *   mask of the standard kind, scale (0: 1/8).  GQA heads are summed into
 *   dk, dv.
 * `workspace`: device memory of at least fl_attn_bwd_workspace_size bytes,
 * 256-byte aligned, owned by the caller, no initialisation needed.  Three
 * kernel launches on `stream`; every output element is written once (no
 * atomics: the result does not depend on scheduling).
 */
fl_status fl_attn_bwd_workspace_size(const fl_tensor *q, const fl_tensor *k,
                                     const fl_attn_variant_desc *desc, size_t *bytes);
fl_status fl_attn_bwd(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                      const fl_tensor *out, const fl_tensor *lse, const fl_tensor *dout,
                      const fl_tensor *dq, const fl_tensor *dk, const fl_tensor *dv,
                      const fl_attn_variant_desc *desc, void *workspace, size_t workspace_bytes,
                      fl_stream_t stream);

/*
 * fl_attn_diff_bwd -- backward of the differential kind: dQ1, dQ2, dK1, dK2
 * and dV of
 *     O = softmax(scale Q1 K1^T + mask) V - lambda softmax(scale Q2 K2^T + mask) V
 * given the forward's per-stream (natural-log) lse and the output gradient
 * dout (the pages name differential attention among the complex variants,
 * gist.science summary, "Results", and the backward as the fused kernels'
 * next step, "Limitations and future work").
 *   q, dq [2, B, S, H, 64]; k, dk [2, B, S, Hk, 64]; v, dv [B, S, Hk, Dv],
 *   Dv 64 or 128; dout [B, S, H, Dv]; lse [2, B, H, S] fp32 (fl_attn_fwd's).
 *   desc: kind FL_KIND_DIFF, mask none or causal, no score_mod, scale (0:
 *   1/8), diff_lambda; GQA heads are summed into dk, dv.
 * Stream t's gradients are those of one softmax attention whose output
 * gradient is c_t dout (c = 1, -lambda); the library recomputes each stream's
 * output from q, k and v and runs the standard backward on it, per 64-column
 * half of V when Dv = 128, then adds the partial gradients with their
 * coefficients in fp32 and rounds once to bf16.
 * `workspace`: device memory of at least fl_attn_diff_bwd_workspace_size
 * bytes, 256-byte aligned, owned by the caller, no initialisation needed.
 * All launches go to `stream`, validation happens before the first one, and
 * every output element is written exactly once (no atomics).
 */
fl_status fl_attn_diff_bwd_workspace_size(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                                          const fl_attn_variant_desc *desc, size_t *bytes);
fl_status fl_attn_diff_bwd(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                           const fl_tensor *lse, const fl_tensor *dout, const fl_tensor *dq,
                           const fl_tensor *dk, const fl_tensor *dv, const fl_attn_variant_desc *desc,
                           void *workspace, size_t workspace_bytes, fl_stream_t stream);

/* Query-block and key-tile sizes the kernel for `desc` uses (for the
 * visited-tile accounting).  `head_dim` is D for the standard and Evoformer
 * kinds and the value head dimension Dv for FL_KIND_DIFF (whose D is 64).
 * Never touches the device. */
fl_status fl_attn_tile_shape(const fl_attn_variant_desc *desc, int32_t head_dim,
                             int32_t *block_m, int32_t *block_n);

/* Checks a score_mod expression against the FL_MOD_EXPR grammar (FL_OK or
 * FL_ERR_INVALID_ARG, with the position in fl_attn_last_error()).  With
 * `compile` 1 it also runs the runtime compilation of the forward kernel for
 * it, with 2 also that of the backward kernels for it and its derivative (no
 * device needed; FL_ERR_UNSUPPORTED without NVRTC). */
fl_status fl_attn_score_expr_check(const char *expr, int32_t compile);

/* Static text for a status code. */
const char *fl_attn_status_string(fl_status status);

/* Detail of the last failure on the calling thread ("" if none). */
const char *fl_attn_last_error(void);

/* FL_ATTN_VERSION of the loaded library. */
int32_t fl_attn_version(void);

/* ------------------------------------------------------------------------
 * Serving with a KV cache (decode).
 *
 * A few new query tokens per sequence attend to that sequence's cached keys
 * and values: the LLaMA-3.2-1B serving workload of the talk notes ("End-to-end:
 * LLaMA-3.2-1B (vLLM / Mooncake)"), whose attention is made causal or
 * softcapped.  out = softmax(score_mod(scale q k^T) + mask) v over the keys
 * 0 .. kv_lens[b] - 1 of sequence b; with `causal`, new token s of a sequence
 * of L cached keys (the new tokens included) sits at position L - Sq + s and
 * sees the keys up to it.
 */
typedef struct {
    int32_t score_mod;          /* FL_MOD_NONE or FL_MOD_SOFTCAP */
    float softcap;              /* FL_MOD_SOFTCAP: the cap (> 0) */
    int32_t causal;             /* 1: decode-causal as above; 0: every cached key */
    float scale;                /* 0 means 1 / sqrt(D) */
    const int32_t *kv_lens;     /* device int32 [B]: cache length of each sequence */
    int32_t max_kv_len;         /* host bound on kv_lens[] (sizes the launch and the workspace);
                                   larger entries are clamped to it */
    const int32_t *block_table; /* NULL: contiguous cache; else device int32
                                   [B][block_table_stride]: page index of each page of a
                                   sequence */
    int32_t block_table_stride; /* entries per row of block_table */
    uint32_t *error_word;       /* NULL, or a device word the kernel ORs FL_DEVERR_* into */
    uint32_t wait_timeout_us;   /* bound of every device-side wait; 0 means 2,000,000 */
} fl_decode_desc;

/*
 * Layouts (bf16 except lse):
 *   q        [B, Sq, Hq, 64]
 *   k_cache, v_cache
 *            contiguous (block_table NULL): [B, S_max, Hk, 64], S_max >= max_kv_len;
 *            paged: [num_pages, page_size, Hk, 64] with page_size in
 *            {16, 32, 64, 128, 256}; key p of sequence b is row p % page_size of
 *            page block_table[b][p / page_size]
 *   out      [B, Sq, Hq, 64]
 *   lse      [B, Hq, Sq] fp32 (natural log) or NULL
 * Hq must be a multiple of Hk, and (Hq / Hk) * Sq <= 64.  The kernel splits
 * every sequence's keys into splits of 128, 256, 512 or 1024 keys (the
 * longest that leaves B * Hk * splits-of-max_kv_len >= 2048, else 128) and
 * merges the splits' partial results through `workspace`: device memory of
 * at least the size
 * fl_attn_decode_workspace_size reports, 256-byte aligned, owned by the
 * caller; its contents need no initialisation (the call clears what must
 * start at zero).  Calls sharing one workspace must not overlap on the GPU.
 */
fl_status fl_attn_decode_workspace_size(const fl_tensor *q, const fl_tensor *k_cache,
                                        const fl_decode_desc *desc, size_t *bytes);

fl_status fl_attn_decode(const fl_tensor *q, const fl_tensor *k_cache, const fl_tensor *v_cache,
                         const fl_tensor *out, const fl_tensor *lse, const fl_decode_desc *desc,
                         void *workspace, size_t workspace_bytes, fl_stream_t stream);

/*
 * fl_attn_decode_static -- fl_attn_decode without a workspace argument, for
 * callers that cannot allocate device memory: for example a serving loop that
 * must not take the device-wide synchronisation a cudaMalloc or cudaFree can
 * cause, or a plug-in that does not own the process's device allocator, and
 * that has no buffer of its own to pass.  (The pages have no counterpart: it
 * is an interface for such callers, not part of the method.)
 *
 * The call allocates nothing.  Its scratch is a static device array of
 * FL_DECODE_STATIC_SCRATCH_BYTES (64 MiB) inside this library, which every GPU
 * that loads the library holds until the process exits; shapes that need more
 * (see fl_attn_decode_workspace_size) return FL_ERR_UNSUPPORTED.  The first
 * call in each CUDA context -- a device's primary context, a context the
 * caller made current, or the new primary context after cudaDeviceReset --
 * looks up the array's device address in that context (which may load the
 * library's device code there): make that first call before any stream
 * capture.  Every call shares the one array and finds the previous
 * call's contents; the call clears what must start at zero, but calls that
 * overlap on the GPU race: issue them on one stream, or order them.
 * Arguments, layouts and results are those of fl_attn_decode.
 */
#define FL_DECODE_STATIC_SCRATCH_BYTES (64u << 20)
fl_status fl_attn_decode_static(const fl_tensor *q, const fl_tensor *k_cache,
                                const fl_tensor *v_cache, const fl_tensor *out,
                                const fl_tensor *lse, const fl_decode_desc *desc,
                                fl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FL_ATTN_H */
