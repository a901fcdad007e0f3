// api.cu -- the C ABI (include/fl_attn.h): argument validation, planning
// (tile grid, work order, TMA descriptors) and dispatch to the kernels.
//
// Validation runs before any CUDA call, so a rejected request touches no
// device state.  The library allocates no device memory: TMA descriptors are
// passed to the kernel as __grid_constant__ parameters.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "fl_attn.h"
#include "launch.h"

namespace {

thread_local char g_last_error[2048];

// Room for a translated score_mod expression (the grammar caps the source at
// 4096 characters; the translation adds parentheses and helper names).
constexpr size_t kExprCudaMax = 16384;

fl_status fail(fl_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

fl_status ok()
{
    g_last_error[0] = '\0';
    return FL_OK;
}

// A validated, normalised copy of an fl_tensor (size-1 axes get the stride a
// packed layout would give them, so arbitrary strides on them are accepted).
struct View {
    void *ptr;
    int ndim;
    int64_t size[5];
    int64_t stride[5];
};

fl_status check_tensor(const fl_tensor *t, const char *name, int ndim, int dtype, View &v)
{
    if (!t)
        return fail(FL_ERR_INVALID_ARG, "%s is NULL", name);
    if (!t->ptr)
        return fail(FL_ERR_INVALID_ARG, "%s->ptr is NULL", name);
    if (t->ndim != ndim)
        return fail(FL_ERR_INVALID_ARG, "%s must have %d dimensions, has %d", name, ndim, t->ndim);
    if (t->dtype != dtype)
        return fail(FL_ERR_INVALID_ARG, "%s must be %s", name, dtype == FL_BF16 ? "bf16" : "fp32");
    v.ptr = t->ptr;
    v.ndim = ndim;
    for (int d = 0; d < ndim; ++d) {
        if (t->sizes[d] < 1 || t->sizes[d] > (int64_t(1) << 31) - 1)
            return fail(FL_ERR_INVALID_ARG, "%s size[%d] = %lld out of range", name, d,
                        (long long)t->sizes[d]);
        v.size[d] = t->sizes[d];
        v.stride[d] = t->strides[d];
    }
    int64_t packed = 1;
    for (int d = ndim - 1; d >= 0; --d) {
        if (v.size[d] == 1)
            v.stride[d] = packed;
        packed *= v.size[d];
    }
    if (v.stride[ndim - 1] != 1)
        return fail(FL_ERR_INVALID_ARG, "%s innermost stride must be 1", name);
    const int elt = dtype == FL_BF16 ? 2 : 4;
    for (int d = 0; d < ndim - 1; ++d) {
        if (v.stride[d] <= 0)
            return fail(FL_ERR_INVALID_ARG, "%s stride[%d] must be positive", name, d);
        if (dtype == FL_BF16 && (v.stride[d] * elt) % 16 != 0)
            return fail(FL_ERR_ALIGNMENT, "%s stride[%d] = %lld elements is not a multiple of 16 bytes",
                        name, d, (long long)v.stride[d]);
        if (v.stride[d] * elt >= (int64_t(1) << 40))
            return fail(FL_ERR_INVALID_ARG, "%s stride[%d] too large", name, d);
    }
    if (reinterpret_cast<uintptr_t>(v.ptr) % (dtype == FL_BF16 ? 16 : 4) != 0)
        return fail(FL_ERR_ALIGNMENT, "%s->ptr is not %d-byte aligned", name,
                    dtype == FL_BF16 ? 16 : 4);
    return FL_OK;
}

bool same(const View &v, std::initializer_list<int64_t> sizes)
{
    int d = 0;
    for (int64_t s : sizes)
        if (v.size[d++] != s)
            return false;
    return true;
}

// ------------------------------------------------------------------ device state

struct DeviceInfo {
    bool ready;
    bool supported;
    int sm_count;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

fl_status device_info(int &dev, DeviceInfo &info)
{
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) {
        cudaGetLastError();
        return fail(FL_ERR_NO_DEVICE, "no CUDA device");
    }
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fail(FL_ERR_NO_DEVICE, "cannot query the current device");
    }
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return fail(FL_ERR_CUDA, "cudaDeviceGetAttribute failed");
        }
        d.supported = (major == 10 && minor == 3);
        d.sm_count = sms;
        d.ready = true;
    }
    info = d;
    if (!info.supported)
        return fail(FL_ERR_NO_DEVICE, "this library is built for sm_103 (GB300) only");
    return FL_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        cudaGetLastError();
    });
    return fn;
}

// A bf16 tensor map over dims (innermost first) with byte strides of dims 1..rank-1.
fl_status make_map(CUtensorMap &map, void *ptr, int rank, const uint64_t *dims,
                   const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swz,
                   const char *what)
{
    auto fn = encode_fn();
    if (!fn)
        return fail(FL_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t gd[5];
    cuuint64_t gs[4];
    cuuint32_t bx[5], es[5];
    for (int d = 0; d < rank; ++d) {
        gd[d] = dims[d];
        bx[d] = box[d];
        es[d] = 1;
    }
    for (int d = 0; d < rank - 1; ++d)
        gs[d] = strides_bytes[d];
    CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, ptr, gd, gs, bx, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FL_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
    return FL_OK;
}

uint64_t timeout_ns(const fl_attn_variant_desc *d)
{
    const uint64_t us = d->wait_timeout_us ? d->wait_timeout_us : 2000000u;
    return us * 1000ull;
}

fl_status check_mask(const fl_attn_variant_desc *d)
{
    switch (d->mask) {
    case FL_MASK_NONE:
    case FL_MASK_CAUSAL:
        return FL_OK;
    case FL_MASK_WINDOW:
        if (d->window < 1)
            return fail(FL_ERR_INVALID_ARG, "window must be >= 1");
        return FL_OK;
    case FL_MASK_PREFIX:
        if (d->prefix < 0)
            return fail(FL_ERR_INVALID_ARG, "prefix must be >= 0");
        return FL_OK;
    case FL_MASK_DOC:
        if (!d->doc_offsets || d->doc_stride < 2)
            return fail(FL_ERR_INVALID_ARG, "doc mask needs doc_offsets and doc_stride >= 2");
        if (reinterpret_cast<uintptr_t>(d->doc_offsets) % 4)
            return fail(FL_ERR_ALIGNMENT, "doc_offsets is not 4-byte aligned");
        return FL_OK;
    default:
        return fail(FL_ERR_INVALID_ARG, "unknown mask %d", d->mask);
    }
}

// ------------------------------------------------------------------ standard

fl_status fwd_standard(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                       const fl_tensor *out, const fl_tensor *lse,
                       const fl_attn_variant_desc *d, const fl_tensor *bias,
                       const fl_tensor *gate, cudaStream_t stream)
{
    View Q, K, V, O, L{};
    fl_status s;
    if ((s = check_tensor(q, "q", 4, FL_BF16, Q)) != FL_OK) return s;
    if ((s = check_tensor(k, "k", 4, FL_BF16, K)) != FL_OK) return s;
    if ((s = check_tensor(v, "v", 4, FL_BF16, V)) != FL_OK) return s;
    if ((s = check_tensor(out, "out", 4, FL_BF16, O)) != FL_OK) return s;
    if (bias || gate)
        return fail(FL_ERR_INVALID_ARG, "bias and gate are only taken by the Evoformer kinds");
    const int64_t B = Q.size[0], S = Q.size[1], Hq = Q.size[2], D = Q.size[3];
    const int64_t Hk = K.size[2], Dv = V.size[3];
    if (!same(K, {B, S, Hk, D}))
        return fail(FL_ERR_INVALID_ARG, "k must be [B, S, Hk, D] matching q");
    if (!same(V, {B, S, Hk, Dv}))
        return fail(FL_ERR_INVALID_ARG, "v must be [B, S, Hk, Dv] matching k");
    if (!same(O, {B, S, Hq, Dv}))
        return fail(FL_ERR_INVALID_ARG, "out must be [B, S, Hq, Dv]");
    if (Hq % Hk != 0)
        return fail(FL_ERR_INVALID_ARG, "Hq (%lld) must be a multiple of Hk (%lld)", (long long)Hq,
                    (long long)Hk);
    const int64_t G = Hq / Hk;
    if (d->gqa_group != 0 && d->gqa_group != G)
        return fail(FL_ERR_INVALID_ARG, "gqa_group %d does not match Hq / Hk = %lld", d->gqa_group,
                    (long long)G);
    if (lse) {
        if ((s = check_tensor(lse, "lse", 3, FL_F32, L)) != FL_OK) return s;
        if (!same(L, {B, Hq, S}))
            return fail(FL_ERR_INVALID_ARG, "lse must be [B, Hq, S]");
    }
    if ((s = check_mask(d)) != FL_OK) return s;
    if (d->score_mod < FL_MOD_NONE || d->score_mod > FL_MOD_EXPR)
        return fail(FL_ERR_INVALID_ARG, "unknown score_mod %d", d->score_mod);
    if (d->score_mod == FL_MOD_SOFTCAP && !(d->softcap > 0.f && std::isfinite(d->softcap)))
        return fail(FL_ERR_INVALID_ARG, "softcap must be positive and finite");
    char expr_cuda[kExprCudaMax];
    if (d->score_mod == FL_MOD_EXPR) {
        char err[256];
        if (!fl::score_expr_translate(d->score_mod_expr, expr_cuda, sizeof expr_cuda, err, sizeof err))
            return fail(FL_ERR_INVALID_ARG, "score_mod_expr: %s", err);
    }
    if (!std::isfinite(d->scale) || d->scale < 0.f)
        return fail(FL_ERR_INVALID_ARG, "scale must be finite and positive (0 selects 1/sqrt(D))");
    if (d->mask == FL_MASK_DOC && d->doc_stride < 2)
        return fail(FL_ERR_INVALID_ARG, "doc_stride must be >= 2");
    if (D != Dv || (D != 32 && D != 64 && D != 128))
        return fail(FL_ERR_UNSUPPORTED, "standard kind supports D = Dv in {32, 64, 128} (got %lld, %lld)",
                    (long long)D, (long long)Dv);
    const int nq = static_cast<int>((S + fl::BM - 1) / fl::BM);
    fl::GridSpec work{};
    if (!fl::make_grid_spec(int(B), int(Hq), int(Hk), nq,
                            d->mask == FL_MASK_CAUSAL || d->mask == FL_MASK_PREFIX || d->mask == FL_MASK_DOC,
                            work))
        return fail(FL_ERR_UNSUPPORTED, "more than 2^31 - 1 work items (B * heads * query tiles)");

    int dev;
    DeviceInfo info;
    if ((s = device_info(dev, info)) != FL_OK) return s;

    CUtensorMap tq, tk, tv;
    // rows of up to 128 bytes per TMA box (D = 128: two boxes per row, the
    // kernel loads both halves); the swizzle is the box row's width
    const uint32_t box_cols = D == 128 ? 64u : uint32_t(D);
    const CUtensorMapSwizzle swz = D == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    const uint32_t box[4] = {box_cols, 128, 1, 1};
    const uint32_t kvbox[4] = {box_cols, uint32_t(fl::std_key_tile(int(D))), 1, 1};
    {
        const uint64_t dims[4] = {uint64_t(D), uint64_t(S), uint64_t(Hq), uint64_t(B)};
        const uint64_t st[3] = {uint64_t(Q.stride[1]) * 2, uint64_t(Q.stride[2]) * 2,
                                uint64_t(Q.stride[0]) * 2};
        if ((s = make_map(tq, Q.ptr, 4, dims, st, box, swz, "q")) != FL_OK)
            return s;
    }
    {
        const uint64_t dims[4] = {uint64_t(D), uint64_t(S), uint64_t(Hk), uint64_t(B)};
        const uint64_t st[3] = {uint64_t(K.stride[1]) * 2, uint64_t(K.stride[2]) * 2,
                                uint64_t(K.stride[0]) * 2};
        if ((s = make_map(tk, K.ptr, 4, dims, st, kvbox, swz, "k")) != FL_OK)
            return s;
    }
    {
        const uint64_t dims[4] = {uint64_t(Dv), uint64_t(S), uint64_t(Hk), uint64_t(B)};
        const uint64_t st[3] = {uint64_t(V.stride[1]) * 2, uint64_t(V.stride[2]) * 2,
                                uint64_t(V.stride[0]) * 2};
        if ((s = make_map(tv, V.ptr, 4, dims, st, kvbox, swz, "v")) != FL_OK)
            return s;
    }

    fl::StdParams p{};
    p.grid = work;
    p.head_dim = int(D);
    p.mask.kind = d->mask;
    p.mask.S = int(S);
    p.mask.window = d->window;
    p.mask.prefix = d->prefix;
    p.mask.doc = d->doc_offsets;
    p.mask.doc_stride = d->doc_stride;
    p.score_mod = d->score_mod;
    const float scale = d->scale != 0.f ? d->scale : 1.0f / std::sqrt(float(D));
    const float log2e = 1.4426950408889634f;
    p.qk_log2 = scale * log2e;
    p.scale = scale;
    if (d->score_mod == FL_MOD_SOFTCAP) {
        p.softcap_in = 2.f * scale * log2e / d->softcap;
        p.softcap_out = d->softcap * log2e;
    }
    p.alibi_slopes = d->alibi_slopes;
    p.alibi_exp_coef = -8.0f / float(Hq);
    p.out = static_cast<__nv_bfloat16 *>(O.ptr);
    p.o_sb = O.stride[0];
    p.o_ss = O.stride[1];
    p.o_sh = O.stride[2];
    if (lse) {
        p.lse = static_cast<float *>(L.ptr);
        p.l_sb = L.stride[0];
        p.l_sh = L.stride[1];
    }
    p.tile_counts = d->debug_tile_counts;
    p.err_user = d->error_word;
    p.inject = d->debug_inject;
    p.timeout_ns = timeout_ns(d);

    const int grid = int(p.grid.n_items < info.sm_count ? p.grid.n_items : info.sm_count);
    if (d->score_mod == FL_MOD_EXPR) {
        char err[1024] = "";
        const cudaError_t e = fl::launch_standard_expr(tq, tk, tv, p, grid, stream, expr_cuda, err,
                                                       sizeof err);
        if (e == cudaErrorInvalidSource)
            return fail(FL_ERR_INVALID_ARG, "score_mod_expr: %s", err);
        if (e == cudaErrorNotSupported)
            return fail(FL_ERR_UNSUPPORTED, "score_mod_expr: %s", err);
        if (e != cudaSuccess)
            return fail(FL_ERR_CUDA, "score_mod_expr kernel: %s%s%s", cudaGetErrorString(e),
                        err[0] ? ": " : "", err);
        return ok();
    }
    cudaError_t e = fl::launch_standard(tq, tk, tv, p, grid, stream);
    if (e != cudaSuccess)
        return fail(FL_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return ok();
}

// ------------------------------------------------------------------ differential

fl_status fwd_diff(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                   const fl_tensor *out, const fl_tensor *lse, const fl_attn_variant_desc *d,
                   const fl_tensor *bias, const fl_tensor *gate, cudaStream_t stream)
{
    View Q, K, V, O, L{};
    fl_status s;
    if ((s = check_tensor(q, "q", 5, FL_BF16, Q)) != FL_OK) return s;
    if ((s = check_tensor(k, "k", 5, FL_BF16, K)) != FL_OK) return s;
    if ((s = check_tensor(v, "v", 4, FL_BF16, V)) != FL_OK) return s;
    if ((s = check_tensor(out, "out", 4, FL_BF16, O)) != FL_OK) return s;
    if (bias || gate)
        return fail(FL_ERR_INVALID_ARG, "bias and gate are only taken by the Evoformer kinds");
    if (Q.size[0] != 2 || K.size[0] != 2)
        return fail(FL_ERR_INVALID_ARG, "q and k need a leading stream axis of size 2");
    const int64_t B = Q.size[1], S = Q.size[2], H = Q.size[3], D = Q.size[4];
    const int64_t Hk = K.size[3], Dv = V.size[3];
    if (!(K.size[1] == B && K.size[2] == S && K.size[4] == D))
        return fail(FL_ERR_INVALID_ARG, "k must be [2, B, S, Hk, D] matching q");
    if (!same(V, {B, S, Hk, Dv}))
        return fail(FL_ERR_INVALID_ARG, "v must be [B, S, Hk, Dv]");
    if (!same(O, {B, S, H, Dv}))
        return fail(FL_ERR_INVALID_ARG, "out must be [B, S, H, Dv]");
    if (H % Hk != 0)
        return fail(FL_ERR_INVALID_ARG, "H must be a multiple of Hk");
    if (d->gqa_group != 0 && d->gqa_group != H / Hk)
        return fail(FL_ERR_INVALID_ARG, "gqa_group does not match H / Hk");
    if (lse) {
        if ((s = check_tensor(lse, "lse", 4, FL_F32, L)) != FL_OK) return s;
        if (!same(L, {2, B, H, S}))
            return fail(FL_ERR_INVALID_ARG, "lse must be [2, B, H, S]");
    }
    if (d->mask != FL_MASK_NONE && d->mask != FL_MASK_CAUSAL)
        return fail(FL_ERR_UNSUPPORTED, "differential attention takes no mask or causal");
    if (d->score_mod != FL_MOD_NONE)
        return fail(FL_ERR_UNSUPPORTED, "differential attention takes no score_mod");
    if (!std::isfinite(d->scale) || d->scale < 0.f || !std::isfinite(d->diff_lambda))
        return fail(FL_ERR_INVALID_ARG, "scale must be finite and positive, diff_lambda finite");
    if (D != 64 || (Dv != 64 && Dv != 128))
        return fail(FL_ERR_UNSUPPORTED, "differential kind supports D = 64, Dv = 64 or 128");

    int dev;
    DeviceInfo info;
    if ((s = device_info(dev, info)) != FL_OK) return s;
    CUtensorMap tq, tk, tv;
    {
        const uint64_t dims[5] = {uint64_t(D), uint64_t(S), uint64_t(H), uint64_t(B), 2};
        const uint64_t st[4] = {uint64_t(Q.stride[2]) * 2, uint64_t(Q.stride[3]) * 2,
                                uint64_t(Q.stride[1]) * 2, uint64_t(Q.stride[0]) * 2};
        const uint32_t box[5] = {64, 128, 1, 1, 1};
        if ((s = make_map(tq, Q.ptr, 5, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B, "q")) != FL_OK)
            return s;
    }
    {
        const uint64_t dims[5] = {uint64_t(D), uint64_t(S), uint64_t(Hk), uint64_t(B), 2};
        const uint64_t st[4] = {uint64_t(K.stride[2]) * 2, uint64_t(K.stride[3]) * 2,
                                uint64_t(K.stride[1]) * 2, uint64_t(K.stride[0]) * 2};
        const uint32_t box[5] = {64, uint32_t(fl::diff_key_tile(int(Dv))), 1, 1, 1};
        if ((s = make_map(tk, K.ptr, 5, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B, "k")) != FL_OK)
            return s;
    }
    {
        const uint64_t dims[4] = {uint64_t(Dv), uint64_t(S), uint64_t(Hk), uint64_t(B)};
        const uint64_t st[3] = {uint64_t(V.stride[1]) * 2, uint64_t(V.stride[2]) * 2,
                                uint64_t(V.stride[0]) * 2};
        const uint32_t box[4] = {64, uint32_t(fl::diff_key_tile(int(Dv))), 1, 1};
        if ((s = make_map(tv, V.ptr, 4, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B, "v")) != FL_OK)
            return s;
    }
    fl::DiffParams p{};
    p.dv = int(Dv);
    p.B = int(B);
    p.H = int(H);
    p.Hk = int(Hk);
    p.G = int(H / Hk);
    p.nq = int((S + fl::BM - 1) / fl::BM);
    p.n_items = int64_t(p.B) * p.H * p.nq;
    p.lpt = d->mask == FL_MASK_CAUSAL;
    p.group = 8;
    p.mask.kind = d->mask;
    p.mask.S = int(S);
    p.qk_log2 = (d->scale != 0.f ? d->scale : 1.0f / std::sqrt(float(D))) * 1.4426950408889634f;
    p.lambda = d->diff_lambda;
    p.out = static_cast<__nv_bfloat16 *>(O.ptr);
    p.o_sb = O.stride[0];
    p.o_ss = O.stride[1];
    p.o_sh = O.stride[2];
    if (lse) {
        p.lse = static_cast<float *>(L.ptr);
        p.l_s2 = L.stride[0];
        p.l_sb = L.stride[1];
        p.l_sh = L.stride[2];
    }
    p.tile_counts = d->debug_tile_counts;
    p.err_user = d->error_word;
    p.timeout_ns = timeout_ns(d);
    const int grid = int(p.n_items < info.sm_count ? p.n_items : info.sm_count);
    cudaError_t e = fl::launch_diff(tq, tk, tv, p, grid, stream);
    if (e != cudaSuccess)
        return fail(FL_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return ok();
}

// ------------------------------------------------------------------ Evoformer

// bias_rows > 0: q, k, v, gate, out (and lse, msa_mask) are a batch of
// stacks folded along the MSA-row axis (bias_rows rows per stack) and bias is
// [stacks, H, N_res, N_res], one per stack.
fl_status fwd_evo(bool row_pass, const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                  const fl_tensor *out, const fl_tensor *lse, const fl_attn_variant_desc *d,
                  const fl_tensor *bias, const fl_tensor *gate, const fl_tensor *msa_mask,
                  cudaStream_t stream, int64_t bias_rows = 0)
{
    View Q, K, V, O, G, Bz{}, L{}, M{};
    fl_status s;
    if ((s = check_tensor(q, "q", 4, FL_BF16, Q)) != FL_OK) return s;
    if ((s = check_tensor(k, "k", 4, FL_BF16, K)) != FL_OK) return s;
    if ((s = check_tensor(v, "v", 4, FL_BF16, V)) != FL_OK) return s;
    if ((s = check_tensor(out, "out", 4, FL_BF16, O)) != FL_OK) return s;
    if ((s = check_tensor(gate, "gate", 4, FL_BF16, G)) != FL_OK) return s;
    const int64_t Ns = Q.size[0], Nr = Q.size[1], H = Q.size[2], C = Q.size[3];
    for (const View *t : {&K, &V, &O, &G})
        if (!same(*t, {Ns, Nr, H, C}))
            return fail(FL_ERR_INVALID_ARG, "q, k, v, gate and out must all be [N_seq, N_res, H, c]");
    if (row_pass && bias_rows > 0) {
        // a per-stack bias as [stacks, H, N_res, N_res], viewed below as
        // (j, i, h, stack) with the rank-3 view's strides in the first axes
        View B4;
        if ((s = check_tensor(bias, "bias", 4, FL_BF16, B4)) != FL_OK) return s;
        if (Ns % bias_rows != 0 || !same(B4, {Ns / bias_rows, H, Nr, Nr}))
            return fail(FL_ERR_INVALID_ARG, "bias must be [B, H, N_res, N_res]");
        Bz.ptr = B4.ptr;
        Bz.ndim = 3;
        for (int a = 0; a < 3; ++a) {
            Bz.size[a] = B4.size[a + 1];
            Bz.stride[a] = B4.stride[a + 1];
        }
        Bz.stride[3] = B4.stride[0];
    } else if (row_pass) {
        if ((s = check_tensor(bias, "bias", 3, FL_BF16, Bz)) != FL_OK) return s;
        if (!same(Bz, {H, Nr, Nr}))
            return fail(FL_ERR_INVALID_ARG, "bias must be [H, N_res, N_res]");
    } else if (bias) {
        return fail(FL_ERR_INVALID_ARG, "the column pass takes no bias");
    }
    const int64_t B = row_pass ? Ns : Nr, S = row_pass ? Nr : Ns;
    if (lse) {
        if ((s = check_tensor(lse, "lse", 3, FL_F32, L)) != FL_OK) return s;
        if (!same(L, {B, H, S}))
            return fail(FL_ERR_INVALID_ARG, row_pass ? "lse must be [N_seq, H, N_res]"
                                                     : "lse must be [N_res, H, N_seq]");
    }
    if (msa_mask) {
        if (msa_mask->dtype != FL_BF16 && msa_mask->dtype != FL_F32)
            return fail(FL_ERR_INVALID_ARG, "msa_mask must be bf16 or fp32");
        if ((s = check_tensor(msa_mask, "msa_mask", 2, msa_mask->dtype, M)) != FL_OK) return s;
        if (!same(M, {Ns, Nr}))
            return fail(FL_ERR_INVALID_ARG, "msa_mask must be [N_seq, N_res]");
    }
    if (d->mask != FL_MASK_NONE || d->score_mod != FL_MOD_NONE)
        return fail(FL_ERR_UNSUPPORTED, "the Evoformer kinds take no mask and no score_mod");
    if (!std::isfinite(d->scale) || d->scale < 0.f)
        return fail(FL_ERR_INVALID_ARG, "scale must be finite and positive (0 selects 1/sqrt(c))");
    if (C != 32 && C != 64)
        return fail(FL_ERR_UNSUPPORTED, "the Evoformer kinds support c = 32 or 64 (got %lld)", (long long)C);

    int dev;
    DeviceInfo info;
    if ((s = device_info(dev, info)) != FL_OK) return s;

    // [batch, sequence, head, c] view: which tensor axis plays batch and sequence
    const int ab = row_pass ? 0 : 1, ai = row_pass ? 1 : 0;
    CUtensorMap tq, tk, tv;
    const uint32_t box[4] = {uint32_t(C), 128, 1, 1};
    const CUtensorMapSwizzle swz = C == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    const View *src[3] = {&Q, &K, &V};
    CUtensorMap *dst[3] = {&tq, &tk, &tv};
    const char *names[3] = {"q", "k", "v"};
    for (int m = 0; m < 3; ++m) {
        const View &T = *src[m];
        const uint64_t dims[4] = {uint64_t(C), uint64_t(S), uint64_t(H), uint64_t(B)};
        const uint64_t st[3] = {uint64_t(T.stride[ai]) * 2, uint64_t(T.stride[2]) * 2,
                                uint64_t(T.stride[ab]) * 2};
        if ((s = make_map(*dst[m], T.ptr, 4, dims, st, box, swz, names[m])) != FL_OK)
            return s;
    }
    CUtensorMap tb;
    std::memset(&tb, 0, sizeof tb);
    if (row_pass) {
        // bias[stack, h, i, j] as (j, i, h, stack); boxes of 64 keys x 128 query
        // rows (kept for a whole work item, or streamed per key tile when
        // N_res > 384 or c = 64)
        const uint64_t stacks = bias_rows > 0 ? uint64_t(Ns / bias_rows) : 1;
        const uint64_t dims[4] = {uint64_t(Nr), uint64_t(Nr), uint64_t(H), stacks};
        const uint64_t st[3] = {uint64_t(Bz.stride[1]) * 2, uint64_t(Bz.stride[0]) * 2,
                                bias_rows > 0 ? uint64_t(Bz.stride[3]) * 2
                                              : uint64_t(Bz.stride[0]) * 2 * uint64_t(H)};
        const uint32_t bbox[4] = {64, 128, 1, 1};
        if ((s = make_map(tb, Bz.ptr, 4, dims, st, bbox, CU_TENSOR_MAP_SWIZZLE_128B, "bias")) != FL_OK)
            return s;
    }
    fl::EvoParams p{};
    p.head_dim = int(C);
    const int nq = int((S + fl::BM - 1) / fl::BM);
    p.grid.B = int(B);
    p.grid.Hq = int(H);
    p.grid.Hk = int(H);
    p.grid.G = 1;
    p.grid.nq = nq;
    // chunk of batch indices per work item: the CTA's two slots run a chunk's
    // batch indices two at a time, so an item costs ceil(chunk / 2) row times
    // plus about half a row time of start-up (the item's bias rows and first
    // Q tiles, loaded once the previous item is done with them); minimise
    // waves x (2 ceil(chunk / 2) + 1) over the SMs, on a tie the smaller chunk
    // (more items to spread over the SMs)
    {
        int64_t best_cost = -1;
        int best_chunk = 1;
        for (int64_t chunk = 1; chunk <= B; ++chunk) {
            if (bias_rows > 0 && bias_rows % chunk != 0)
                continue; // an item's rows share one stack's bias
            const int64_t items = ((B + chunk - 1) / chunk) * H * nq;
            const int64_t waves = (items + info.sm_count - 1) / info.sm_count;
            const int64_t cost = waves * (2 * ((chunk + 1) / 2) + 1);
            if (best_cost < 0 || cost < best_cost) {
                best_cost = cost;
                best_chunk = int(chunk);
            }
        }
        p.chunk = best_chunk;
        p.n_items = ((B + best_chunk - 1) / best_chunk) * H * nq;
    }
    p.mask.kind = FL_MASK_NONE;
    p.mask.S = int(S);
    const float scale = d->scale != 0.f ? d->scale : 1.0f / std::sqrt(float(C));
    p.qk_scale = scale;
    p.qk_log2 = scale * 1.4426950408889634f;
    if (row_pass) {
        p.bias = static_cast<const __nv_bfloat16 *>(Bz.ptr);
        p.bias_rows = int(bias_rows);
    }
    p.gate = static_cast<const __nv_bfloat16 *>(G.ptr);
    p.g_sb = G.stride[ab];
    p.g_si = G.stride[ai];
    p.g_sh = G.stride[2];
    p.out = static_cast<__nv_bfloat16 *>(O.ptr);
    p.o_sb = O.stride[ab];
    p.o_si = O.stride[ai];
    p.o_sh = O.stride[2];
    if (lse) {
        p.lse = static_cast<float *>(L.ptr);
        p.l_sb = L.stride[0];
        p.l_sh = L.stride[1];
    }
    p.tile_counts = d->debug_tile_counts;
    if (msa_mask) {
        // key j of batch index b: row pass b = MSA row, j = residue; column
        // pass b = residue, j = MSA row
        p.kmask = M.ptr;
        p.km_f32 = msa_mask->dtype == FL_F32;
        p.km_sb = M.stride[ab];
        p.km_sk = M.stride[ai];
    }
    p.err_user = d->error_word;
    p.timeout_ns = timeout_ns(d);
    const int grid = int(p.n_items < info.sm_count ? p.n_items : info.sm_count);
    cudaError_t e = fl::launch_evo(tq, tk, tv, tb, p, grid, stream);
    if (e != cudaSuccess)
        return fail(FL_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return ok();
}

// ------------------------------------------------------------------ decode

constexpr size_t kWsAlign = 256;
size_t align_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

struct DecodePlan {
    View Q, K, V;
    int64_t B, Sq, Hq, Hk, P, T;
    int G, R, split_chunks, max_splits;
    size_t o_bytes, ml_bytes, cnt_bytes, total;
};

// Validates the shapes common to the workspace query and the call.
fl_status decode_plan(const fl_tensor *q, const fl_tensor *k_cache, const fl_tensor *v_cache,
                      const fl_decode_desc *d, DecodePlan &pl)
{
    fl_status s;
    if (!d)
        return fail(FL_ERR_INVALID_ARG, "desc is NULL");
    if ((s = check_tensor(q, "q", 4, FL_BF16, pl.Q)) != FL_OK) return s;
    if ((s = check_tensor(k_cache, "k_cache", 4, FL_BF16, pl.K)) != FL_OK) return s;
    if (v_cache) {
        if ((s = check_tensor(v_cache, "v_cache", 4, FL_BF16, pl.V)) != FL_OK) return s;
        if (!same(pl.V, {pl.K.size[0], pl.K.size[1], pl.K.size[2], pl.K.size[3]}))
            return fail(FL_ERR_INVALID_ARG, "v_cache must have the shape of k_cache");
    }
    pl.B = pl.Q.size[0];
    pl.Sq = pl.Q.size[1];
    pl.Hq = pl.Q.size[2];
    pl.P = pl.K.size[0];
    pl.T = pl.K.size[1];
    pl.Hk = pl.K.size[2];
    if (pl.Q.size[3] != 64 || pl.K.size[3] != 64)
        return fail(FL_ERR_UNSUPPORTED, "decode supports head dimension 64");
    if (pl.Hq % pl.Hk != 0)
        return fail(FL_ERR_INVALID_ARG, "Hq (%lld) must be a multiple of Hk (%lld)",
                    (long long)pl.Hq, (long long)pl.Hk);
    pl.G = int(pl.Hq / pl.Hk);
    if (int64_t(pl.G) * pl.Sq > fl::kDecodeMaxRows)
        return fail(FL_ERR_UNSUPPORTED, "(Hq / Hk) * Sq = %lld exceeds %d",
                    (long long)(int64_t(pl.G) * pl.Sq), fl::kDecodeMaxRows);
    pl.R = int(pl.G * pl.Sq);
    if (d->max_kv_len < 1)
        return fail(FL_ERR_INVALID_ARG, "max_kv_len must be >= 1");
    if (d->score_mod != FL_MOD_NONE && d->score_mod != FL_MOD_SOFTCAP)
        return fail(FL_ERR_UNSUPPORTED, "decode supports score_mod none or softcap");
    if (d->score_mod == FL_MOD_SOFTCAP && !(d->softcap > 0.f && std::isfinite(d->softcap)))
        return fail(FL_ERR_INVALID_ARG, "softcap must be positive and finite");
    if (!std::isfinite(d->scale) || d->scale < 0.f)
        return fail(FL_ERR_INVALID_ARG, "scale must be finite and positive (0 selects 1/sqrt(D))");
    if (!d->block_table) {
        if (pl.P != pl.B)
            return fail(FL_ERR_INVALID_ARG, "a contiguous cache is [B, S_max, Hk, 64]");
        if (d->max_kv_len > pl.T)
            return fail(FL_ERR_INVALID_ARG, "max_kv_len %d exceeds the cache length %lld",
                        d->max_kv_len, (long long)pl.T);
    } else {
        if (pl.T != 16 && pl.T != 32 && pl.T != 64 && pl.T != 128 && pl.T != 256)
            return fail(FL_ERR_UNSUPPORTED, "page size %lld: must be 16, 32, 64, 128 or 256",
                        (long long)pl.T);
        if (int64_t(d->block_table_stride) * pl.T < d->max_kv_len)
            return fail(FL_ERR_INVALID_ARG, "block_table_stride %d pages cannot hold %d keys",
                        d->block_table_stride, d->max_kv_len);
        if (reinterpret_cast<uintptr_t>(d->block_table) % 4)
            return fail(FL_ERR_ALIGNMENT, "block_table is not 4-byte aligned");
    }
    // Keys per CTA: the longest split (fewest partials to merge) that still
    // leaves about 2048 CTAs for the longest sequences' work, so that the GPU
    // stays full; a function of the shapes alone, so that the workspace query
    // and the call agree.
    const int64_t max_chunks = (d->max_kv_len + fl::kDecodeChunk - 1) / fl::kDecodeChunk;
    pl.split_chunks = 1;
    for (int sc = fl::kDecodeMaxSplitChunks; sc > 1; sc /= 2)
        if (pl.B * pl.Hk * ((max_chunks + sc - 1) / sc) >= 2048) {
            pl.split_chunks = sc;
            break;
        }
    pl.max_splits = int((max_chunks + pl.split_chunks - 1) / pl.split_chunks);
    const size_t units = size_t(pl.B) * size_t(pl.Hk) * size_t(pl.max_splits) * size_t(pl.R);
    pl.o_bytes = align_up(units * 64 * sizeof(float));
    pl.ml_bytes = align_up(units * 2 * sizeof(float));
    pl.cnt_bytes = align_up(size_t(pl.B) * size_t(pl.Hk) * sizeof(int));
    pl.total = pl.o_bytes + pl.ml_bytes + pl.cnt_bytes;
    return FL_OK;
}

fl_status decode_run(const DecodePlan &pl, const fl_tensor *out, const fl_tensor *lse,
                     const fl_decode_desc *d, void *workspace, cudaStream_t stream)
{
    View O, L{};
    fl_status s;
    if ((s = check_tensor(out, "out", 4, FL_BF16, O)) != FL_OK) return s;
    if (!same(O, {pl.B, pl.Sq, pl.Hq, 64}))
        return fail(FL_ERR_INVALID_ARG, "out must be [B, Sq, Hq, 64]");
    if (lse) {
        if ((s = check_tensor(lse, "lse", 3, FL_F32, L)) != FL_OK) return s;
        if (!same(L, {pl.B, pl.Hq, pl.Sq}))
            return fail(FL_ERR_INVALID_ARG, "lse must be [B, Hq, Sq]");
    }
    if (!d->kv_lens)
        return fail(FL_ERR_INVALID_ARG, "kv_lens is NULL");
    if (reinterpret_cast<uintptr_t>(d->kv_lens) % 4)
        return fail(FL_ERR_ALIGNMENT, "kv_lens is not 4-byte aligned");
    int dev;
    DeviceInfo info;
    if ((s = device_info(dev, info)) != FL_OK) return s;

    CUtensorMap tk, tv;
    const uint32_t box[4] = {64, uint32_t(pl.T < fl::kDecodeChunk ? pl.T : fl::kDecodeChunk), 1, 1};
    const View *src[2] = {&pl.K, &pl.V};
    CUtensorMap *dst[2] = {&tk, &tv};
    const char *names[2] = {"k_cache", "v_cache"};
    for (int m = 0; m < 2; ++m) {
        const View &T = *src[m];
        const uint64_t dims[4] = {64, uint64_t(pl.T), uint64_t(pl.Hk), uint64_t(pl.P)};
        const uint64_t st[3] = {uint64_t(T.stride[1]) * 2, uint64_t(T.stride[2]) * 2,
                                uint64_t(T.stride[0]) * 2};
        if ((s = make_map(*dst[m], T.ptr, 4, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B, names[m])) != FL_OK)
            return s;
    }
    fl::DecodeParams p{};
    p.B = int(pl.B);
    p.Hk = int(pl.Hk);
    p.G = pl.G;
    p.Sq = int(pl.Sq);
    p.max_kv = d->max_kv_len;
    p.split_chunks = pl.split_chunks;
    p.max_splits = pl.max_splits;
    p.page = int(pl.T);
    p.bt_stride = d->block_table_stride;
    p.kv_lens = d->kv_lens;
    p.block_table = d->block_table;
    p.q = static_cast<const __nv_bfloat16 *>(pl.Q.ptr);
    p.q_sb = pl.Q.stride[0];
    p.q_ss = pl.Q.stride[1];
    p.q_sh = pl.Q.stride[2];
    p.out = static_cast<__nv_bfloat16 *>(O.ptr);
    p.o_sb = O.stride[0];
    p.o_ss = O.stride[1];
    p.o_sh = O.stride[2];
    if (lse) {
        p.lse = static_cast<float *>(L.ptr);
        p.l_sb = L.stride[0];
        p.l_sh = L.stride[1];
    }
    p.scale = d->scale != 0.f ? d->scale : 0.125f; // 1 / sqrt(64)
    p.softcap = d->score_mod == FL_MOD_SOFTCAP ? d->softcap : 0.f;
    p.causal = d->causal ? 1 : 0;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.ws_o = reinterpret_cast<float *>(ws);
    p.ws_ml = reinterpret_cast<float *>(ws + pl.o_bytes);
    p.ws_cnt = reinterpret_cast<int *>(ws + pl.o_bytes + pl.ml_bytes);
    p.err_user = d->error_word;
    p.timeout_ns = uint64_t(d->wait_timeout_us ? d->wait_timeout_us : 2000000u) * 1000ull;

    // the per-(sequence, KV head) tickets must start at zero
    cudaError_t e = cudaMemsetAsync(p.ws_cnt, 0, size_t(pl.B) * size_t(pl.Hk) * sizeof(int), stream);
    if (e != cudaSuccess)
        return fail(FL_ERR_CUDA, "clearing the workspace counters failed: %s", cudaGetErrorString(e));
    e = fl::launch_decode(tk, tv, p, stream);
    if (e != cudaSuccess)
        return fail(FL_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return ok();
}

// ------------------------------------------------------------------ backward

struct BwdPlan {
    View Q, K, V;
    int64_t B, S, Hq, Hk, S_pad;
    size_t total;
    std::string expr, expr_grad; // FL_MOD_EXPR: the translated expression and its derivative
};

fl_status bwd_plan(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                   const fl_attn_variant_desc *d, BwdPlan &pl)
{
    fl_status s;
    if (!d)
        return fail(FL_ERR_INVALID_ARG, "desc is NULL");
    if ((s = check_tensor(q, "q", 4, FL_BF16, pl.Q)) != FL_OK) return s;
    if ((s = check_tensor(k, "k", 4, FL_BF16, pl.K)) != FL_OK) return s;
    if (v) {
        if ((s = check_tensor(v, "v", 4, FL_BF16, pl.V)) != FL_OK) return s;
        if (!same(pl.V, {pl.K.size[0], pl.K.size[1], pl.K.size[2], pl.K.size[3]}))
            return fail(FL_ERR_INVALID_ARG, "v must have the shape of k");
    }
    pl.B = pl.Q.size[0];
    pl.S = pl.Q.size[1];
    pl.Hq = pl.Q.size[2];
    pl.Hk = pl.K.size[2];
    if (pl.K.size[0] != pl.B || pl.K.size[1] != pl.S)
        return fail(FL_ERR_INVALID_ARG, "k must be [B, S, Hk, D] matching q");
    if (pl.Q.size[3] != 64 || pl.K.size[3] != 64)
        return fail(FL_ERR_UNSUPPORTED, "the backward supports head dimension 64");
    if (pl.Hq % pl.Hk != 0)
        return fail(FL_ERR_INVALID_ARG, "Hq (%lld) must be a multiple of Hk (%lld)",
                    (long long)pl.Hq, (long long)pl.Hk);
    if (d->kind != FL_KIND_STANDARD)
        return fail(FL_ERR_UNSUPPORTED, "the backward supports the standard kind");
    if (d->score_mod < FL_MOD_NONE || d->score_mod > FL_MOD_EXPR)
        return fail(FL_ERR_INVALID_ARG, "unknown score_mod %d", d->score_mod);
    if (d->score_mod == FL_MOD_EXPR) {
        std::vector<char> v(kExprCudaMax), g(kExprCudaMax);
        char err[256];
        if (!fl::score_expr_translate_grad(d->score_mod_expr, v.data(), v.size(), g.data(), g.size(), err,
                                           sizeof err))
            return fail(FL_ERR_INVALID_ARG, "score_mod_expr: %s", err);
        pl.expr = v.data();
        pl.expr_grad = g.data();
    }
    if (d->score_mod == FL_MOD_SOFTCAP && !(d->softcap > 0.f && std::isfinite(d->softcap)))
        return fail(FL_ERR_INVALID_ARG, "softcap must be positive and finite");
    if ((s = check_mask(d)) != FL_OK)
        return s;
    if (d->gqa_group != 0 && d->gqa_group != pl.Hq / pl.Hk)
        return fail(FL_ERR_INVALID_ARG, "gqa_group does not match Hq / Hk");
    if (!std::isfinite(d->scale) || d->scale < 0.f)
        return fail(FL_ERR_INVALID_ARG, "scale must be finite and positive (0 selects 1/sqrt(D))");
    // padded to the dQ kernel's 128-row query tiles (a multiple of kBwdBlock)
    pl.S_pad = (pl.S + 127) / 128 * 128;
    pl.total = (size_t(pl.B) * size_t(pl.Hq) * size_t(pl.S_pad) * sizeof(fl::BwdRowStat) + 255) / 256 * 256;
    return FL_OK;
}

// ------------------------------------------------------------------ differential backward

// A bf16 [d0, d1, d2, d3] view at `ptr` with the given element strides (the
// innermost one 1), as the library's own entry points take it.
fl_tensor view4(void *ptr, int dtype, const int64_t (&size)[4], const int64_t (&stride)[3])
{
    fl_tensor t{};
    t.ptr = ptr;
    t.dtype = static_cast<fl_dtype>(dtype);
    t.ndim = 4;
    for (int d = 0; d < 4; ++d)
        t.sizes[d] = size[d];
    for (int d = 0; d < 3; ++d)
        t.strides[d] = stride[d];
    t.strides[3] = 1;
    return t;
}

fl_tensor view3(void *ptr, int dtype, const int64_t (&size)[3], const int64_t (&stride)[2])
{
    fl_tensor t{};
    t.ptr = ptr;
    t.dtype = static_cast<fl_dtype>(dtype);
    t.ndim = 3;
    for (int d = 0; d < 3; ++d)
        t.sizes[d] = size[d];
    t.strides[0] = stride[0];
    t.strides[1] = stride[1];
    t.strides[2] = 1;
    return t;
}

// Shapes, the desc the standard kind's kernels run with, and the workspace
// layout of the differential backward: one recomputed O half, the bf16
// partial gradients of every (stream, value half), and the standard
// backward's own workspace (reused by each of its runs).
struct DiffBwdPlan {
    View Q, K, V;
    int64_t B, S, H, Hk, Dv, halves;
    fl_attn_variant_desc sd; // the standard kind's desc for the inner calls
    size_t unit_q, unit_k;   // bytes of one [B, S, H, 64] / [B, S, Hk, 64] bf16 buffer
    size_t off_o, off_dq, off_dk, off_dv, off_ws, ws_bytes, total;
};

fl_status diff_bwd_plan(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                        const fl_attn_variant_desc *d, DiffBwdPlan &pl)
{
    fl_status s;
    if (!d)
        return fail(FL_ERR_INVALID_ARG, "desc is NULL");
    if (d->kind != FL_KIND_DIFF)
        return fail(FL_ERR_INVALID_ARG, "fl_attn_diff_bwd takes FL_KIND_DIFF");
    if ((s = check_tensor(q, "q", 5, FL_BF16, pl.Q)) != FL_OK) return s;
    if ((s = check_tensor(k, "k", 5, FL_BF16, pl.K)) != FL_OK) return s;
    if ((s = check_tensor(v, "v", 4, FL_BF16, pl.V)) != FL_OK) return s;
    if (pl.Q.size[0] != 2 || pl.K.size[0] != 2)
        return fail(FL_ERR_INVALID_ARG, "q and k need a leading stream axis of size 2");
    pl.B = pl.Q.size[1];
    pl.S = pl.Q.size[2];
    pl.H = pl.Q.size[3];
    pl.Hk = pl.K.size[3];
    pl.Dv = pl.V.size[3];
    if (!(pl.K.size[1] == pl.B && pl.K.size[2] == pl.S && pl.K.size[4] == pl.Q.size[4]))
        return fail(FL_ERR_INVALID_ARG, "k must be [2, B, S, Hk, D] matching q");
    if (!same(pl.V, {pl.B, pl.S, pl.Hk, pl.Dv}))
        return fail(FL_ERR_INVALID_ARG, "v must be [B, S, Hk, Dv]");
    if (pl.H % pl.Hk != 0)
        return fail(FL_ERR_INVALID_ARG, "H must be a multiple of Hk");
    if (d->gqa_group != 0 && d->gqa_group != pl.H / pl.Hk)
        return fail(FL_ERR_INVALID_ARG, "gqa_group does not match H / Hk");
    if (pl.Q.size[4] != 64 || (pl.Dv != 64 && pl.Dv != 128))
        return fail(FL_ERR_UNSUPPORTED, "the differential backward supports D = 64, Dv = 64 or 128");
    if (d->mask != FL_MASK_NONE && d->mask != FL_MASK_CAUSAL)
        return fail(FL_ERR_UNSUPPORTED, "differential attention takes no mask or causal");
    if (d->score_mod != FL_MOD_NONE)
        return fail(FL_ERR_UNSUPPORTED, "differential attention takes no score_mod");
    if (!std::isfinite(d->scale) || d->scale < 0.f || !std::isfinite(d->diff_lambda))
        return fail(FL_ERR_INVALID_ARG, "scale must be finite and positive, diff_lambda finite");
    pl.halves = pl.Dv / 64;
    pl.sd = fl_attn_variant_desc{};
    pl.sd.kind = FL_KIND_STANDARD;
    pl.sd.score_mod = FL_MOD_NONE;
    pl.sd.mask = d->mask;
    pl.sd.gqa_group = 0;
    pl.sd.scale = d->scale;
    pl.sd.error_word = d->error_word;
    pl.sd.wait_timeout_us = d->wait_timeout_us;
    const auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    pl.unit_q = up(size_t(pl.B) * pl.S * pl.H * 64 * 2);
    pl.unit_k = up(size_t(pl.B) * pl.S * pl.Hk * 64 * 2);
    pl.off_o = 0;
    pl.off_dq = pl.off_o + pl.unit_q;
    pl.off_dk = pl.off_dq + 2 * pl.halves * pl.unit_q;
    pl.off_dv = pl.off_dk + 2 * pl.halves * pl.unit_k;
    pl.off_ws = pl.off_dv + 2 * pl.halves * pl.unit_k;
    const int64_t S_pad = (pl.S + 127) / 128 * 128; // as the standard backward sizes its own
    pl.ws_bytes = up(size_t(pl.B) * size_t(pl.H) * size_t(S_pad) * sizeof(fl::BwdRowStat));
    pl.total = pl.off_ws + pl.ws_bytes;
    return FL_OK;
}

} // namespace

extern "C" {

fl_status fl_attn_bwd_workspace_size(const fl_tensor *q, const fl_tensor *k,
                                     const fl_attn_variant_desc *desc, size_t *bytes)
{
    if (!bytes)
        return fail(FL_ERR_INVALID_ARG, "bytes is NULL");
    BwdPlan pl;
    const fl_status s = bwd_plan(q, k, nullptr, desc, pl);
    if (s != FL_OK)
        return s;
    *bytes = pl.total;
    return ok();
}

fl_status fl_attn_bwd(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                      const fl_tensor *out, const fl_tensor *lse, const fl_tensor *dout,
                      const fl_tensor *dq, const fl_tensor *dk, const fl_tensor *dv,
                      const fl_attn_variant_desc *desc, void *workspace, size_t workspace_bytes,
                      fl_stream_t stream)
{
    if (!v)
        return fail(FL_ERR_INVALID_ARG, "v is NULL");
    BwdPlan pl;
    fl_status s = bwd_plan(q, k, v, desc, pl);
    if (s != FL_OK)
        return s;
    View O, DO, DQ, DK, DV, L;
    if ((s = check_tensor(out, "out", 4, FL_BF16, O)) != FL_OK) return s;
    if ((s = check_tensor(dout, "dout", 4, FL_BF16, DO)) != FL_OK) return s;
    if ((s = check_tensor(dq, "dq", 4, FL_BF16, DQ)) != FL_OK) return s;
    if ((s = check_tensor(dk, "dk", 4, FL_BF16, DK)) != FL_OK) return s;
    if ((s = check_tensor(dv, "dv", 4, FL_BF16, DV)) != FL_OK) return s;
    if ((s = check_tensor(lse, "lse", 3, FL_F32, L)) != FL_OK) return s;
    for (const View *t : {&O, &DO, &DQ})
        if (!same(*t, {pl.B, pl.S, pl.Hq, 64}))
            return fail(FL_ERR_INVALID_ARG, "out, dout and dq must be [B, S, Hq, 64]");
    for (const View *t : {&DK, &DV})
        if (!same(*t, {pl.B, pl.S, pl.Hk, 64}))
            return fail(FL_ERR_INVALID_ARG, "dk and dv must be [B, S, Hk, 64]");
    if (!same(L, {pl.B, pl.Hq, pl.S}))
        return fail(FL_ERR_INVALID_ARG, "lse must be [B, Hq, S]");
    if (!workspace)
        return fail(FL_ERR_INVALID_ARG, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % kWsAlign)
        return fail(FL_ERR_ALIGNMENT, "workspace is not %zu-byte aligned", kWsAlign);
    if (workspace_bytes < pl.total)
        return fail(FL_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", workspace_bytes, pl.total);
    int dev;
    DeviceInfo info;
    if ((s = device_info(dev, info)) != FL_OK) return s;

    // [64 features, S, heads, B] maps, boxes of 64 rows
    CUtensorMap tq, tdo, tk, tv;
    const uint32_t box[4] = {64, uint32_t(fl::kBwdBlock), 1, 1};
    const View *src[4] = {&pl.Q, &DO, &pl.K, &pl.V};
    CUtensorMap *dst[4] = {&tq, &tdo, &tk, &tv};
    const char *names[4] = {"q", "dout", "k", "v"};
    for (int m = 0; m < 4; ++m) {
        const View &T = *src[m];
        const uint64_t dims[4] = {64, uint64_t(pl.S), uint64_t(T.size[2]), uint64_t(pl.B)};
        const uint64_t st[3] = {uint64_t(T.stride[1]) * 2, uint64_t(T.stride[2]) * 2,
                                uint64_t(T.stride[0]) * 2};
        if ((s = make_map(*dst[m], T.ptr, 4, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B, names[m])) != FL_OK)
            return s;
    }
    fl::BwdParams p{};
    p.B = int(pl.B);
    p.Hq = int(pl.Hq);
    p.Hk = int(pl.Hk);
    p.S = int(pl.S);
    p.S_pad = int(pl.S_pad);
    p.score_mod = desc->score_mod;
    p.softcap = desc->score_mod == FL_MOD_SOFTCAP ? desc->softcap : 0.f;
    p.alibi_slopes = desc->alibi_slopes;
    p.alibi_exp_coef = -8.0f / float(pl.Hq);
    p.mask.kind = desc->mask;
    p.mask.S = int(pl.S);
    p.mask.window = desc->window;
    p.mask.prefix = desc->prefix;
    p.mask.doc = desc->doc_offsets;
    p.mask.doc_stride = desc->doc_stride;
    p.scale = desc->scale != 0.f ? desc->scale : 0.125f; // 1 / sqrt(64)
    auto strides3 = [](const View &t, int64_t &sb, int64_t &ss, int64_t &sh) {
        sb = t.stride[0];
        ss = t.stride[1];
        sh = t.stride[2];
    };
    p.q = static_cast<const __nv_bfloat16 *>(pl.Q.ptr);
    strides3(pl.Q, p.q_sb, p.q_ss, p.q_sh);
    p.k = static_cast<const __nv_bfloat16 *>(pl.K.ptr);
    strides3(pl.K, p.k_sb, p.k_ss, p.k_sh);
    p.v = static_cast<const __nv_bfloat16 *>(pl.V.ptr);
    strides3(pl.V, p.v_sb, p.v_ss, p.v_sh);
    p.o = static_cast<const __nv_bfloat16 *>(O.ptr);
    strides3(O, p.o_sb, p.o_ss, p.o_sh);
    p.dout = static_cast<const __nv_bfloat16 *>(DO.ptr);
    strides3(DO, p.do_sb, p.do_ss, p.do_sh);
    p.lse = static_cast<const float *>(L.ptr);
    p.l_sb = L.stride[0];
    p.l_sh = L.stride[1];
    p.dq = static_cast<__nv_bfloat16 *>(DQ.ptr);
    strides3(DQ, p.dq_sb, p.dq_ss, p.dq_sh);
    p.dk = static_cast<__nv_bfloat16 *>(DK.ptr);
    strides3(DK, p.dk_sb, p.dk_ss, p.dk_sh);
    p.dv = static_cast<__nv_bfloat16 *>(DV.ptr);
    strides3(DV, p.dv_sb, p.dv_ss, p.dv_sh);
    p.ws_stats = static_cast<fl::BwdRowStat *>(workspace);
    p.err_user = desc->error_word;
    p.timeout_ns = timeout_ns(desc);
    // all four again with 128-row boxes (the dQ kernel's query tiles, the
    // dK/dV kernel's key tiles)
    CUtensorMap tq128, tdo128, tk128, tv128;
    CUtensorMap *dst128[4] = {&tq128, &tdo128, &tk128, &tv128};
    const uint32_t box128[4] = {64, 128, 1, 1};
    for (int m = 0; m < 4; ++m) {
        const View &T = *src[m];
        const uint64_t dims[4] = {64, uint64_t(pl.S), uint64_t(T.size[2]), uint64_t(pl.B)};
        const uint64_t st[3] = {uint64_t(T.stride[1]) * 2, uint64_t(T.stride[2]) * 2,
                                uint64_t(T.stride[0]) * 2};
        if ((s = make_map(*dst128[m], T.ptr, 4, dims, st, box128, CU_TENSOR_MAP_SWIZZLE_128B, names[m])) !=
            FL_OK)
            return s;
    }
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (desc->score_mod == FL_MOD_EXPR) {
        cudaError_t e = fl::launch_bwd_prep(p, st);
        char err[1024] = "";
        if (e == cudaSuccess)
            e = fl::launch_bwd_expr(tq, tdo, tk, tv, tq128, tdo128, tk128, tv128, p, st, pl.expr.c_str(),
                                    pl.expr_grad.c_str(), err, sizeof err);
        if (e == cudaErrorInvalidSource)
            return fail(FL_ERR_INVALID_ARG, "score_mod_expr: %s", err);
        if (e == cudaErrorNotSupported)
            return fail(FL_ERR_UNSUPPORTED, "score_mod_expr: %s", err);
        if (e != cudaSuccess)
            return fail(FL_ERR_CUDA, "score_mod_expr backward: %s%s%s", cudaGetErrorString(e), err[0] ? ": " : "",
                        err);
        return ok();
    }
    const cudaError_t e = fl::launch_bwd(tq, tdo, tk, tv, tq128, tdo128, tk128, tv128, p, st);
    if (e != cudaSuccess)
        return fail(FL_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return ok();
}

fl_status fl_attn_diff_bwd_workspace_size(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                                          const fl_attn_variant_desc *desc, size_t *bytes)
{
    if (!bytes)
        return fail(FL_ERR_INVALID_ARG, "bytes is NULL");
    DiffBwdPlan pl;
    const fl_status s = diff_bwd_plan(q, k, v, desc, pl);
    if (s != FL_OK)
        return s;
    *bytes = pl.total;
    return ok();
}

fl_status fl_attn_diff_bwd(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                           const fl_tensor *lse, const fl_tensor *dout, const fl_tensor *dq,
                           const fl_tensor *dk, const fl_tensor *dv, const fl_attn_variant_desc *desc,
                           void *workspace, size_t workspace_bytes, fl_stream_t stream)
{
    DiffBwdPlan pl;
    fl_status s = diff_bwd_plan(q, k, v, desc, pl);
    if (s != FL_OK)
        return s;
    View L, DO, DQ, DK, DV;
    if ((s = check_tensor(lse, "lse", 4, FL_F32, L)) != FL_OK) return s;
    if ((s = check_tensor(dout, "dout", 4, FL_BF16, DO)) != FL_OK) return s;
    if ((s = check_tensor(dq, "dq", 5, FL_BF16, DQ)) != FL_OK) return s;
    if ((s = check_tensor(dk, "dk", 5, FL_BF16, DK)) != FL_OK) return s;
    if ((s = check_tensor(dv, "dv", 4, FL_BF16, DV)) != FL_OK) return s;
    if (!same(L, {2, pl.B, pl.H, pl.S}))
        return fail(FL_ERR_INVALID_ARG, "lse must be [2, B, H, S]");
    if (!same(DO, {pl.B, pl.S, pl.H, pl.Dv}))
        return fail(FL_ERR_INVALID_ARG, "dout must be [B, S, H, Dv]");
    if (!same(DQ, {2, pl.B, pl.S, pl.H, 64}))
        return fail(FL_ERR_INVALID_ARG, "dq must be [2, B, S, H, 64]");
    if (!same(DK, {2, pl.B, pl.S, pl.Hk, 64}))
        return fail(FL_ERR_INVALID_ARG, "dk must be [2, B, S, Hk, 64]");
    if (!same(DV, {pl.B, pl.S, pl.Hk, pl.Dv}))
        return fail(FL_ERR_INVALID_ARG, "dv must be [B, S, Hk, Dv]");
    if (!workspace)
        return fail(FL_ERR_INVALID_ARG, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % kWsAlign)
        return fail(FL_ERR_ALIGNMENT, "workspace is not %zu-byte aligned", kWsAlign);
    if (workspace_bytes < pl.total)
        return fail(FL_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", workspace_bytes, pl.total);
    int dev;
    DeviceInfo info;
    if ((s = device_info(dev, info)) != FL_OK)
        return s;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const auto bf = [](void *base, int64_t elems) {
        return static_cast<void *>(static_cast<__nv_bfloat16 *>(base) + elems);
    };
    const int64_t B = pl.B, S = pl.S, H = pl.H, Hk = pl.Hk;
    const int64_t packed_q[3] = {S * H * 64, H * 64, 64}, packed_k[3] = {S * Hk * 64, Hk * 64, 64};
    const float coef[2] = {1.f, -desc->diff_lambda};
    // The views below only re-address tensors validated above (a stream's
    // slice, a 64-column half, a workspace buffer), so the inner calls cannot
    // fail validation after an earlier one has launched.
    for (int t = 0; t < 2; ++t) {
        const fl_tensor qt = view4(bf(pl.Q.ptr, t * pl.Q.stride[0]), FL_BF16, {B, S, H, 64},
                                   {pl.Q.stride[1], pl.Q.stride[2], pl.Q.stride[3]});
        const fl_tensor kt = view4(bf(pl.K.ptr, t * pl.K.stride[0]), FL_BF16, {B, S, Hk, 64},
                                   {pl.K.stride[1], pl.K.stride[2], pl.K.stride[3]});
        const fl_tensor lt = view3(static_cast<float *>(L.ptr) + t * L.stride[0], FL_F32, {B, H, S},
                                   {L.stride[1], L.stride[2]});
        for (int64_t hv = 0; hv < pl.halves; ++hv) {
            const fl_tensor vh = view4(bf(pl.V.ptr, 64 * hv), FL_BF16, {B, S, Hk, 64},
                                       {pl.V.stride[0], pl.V.stride[1], pl.V.stride[2]});
            const fl_tensor doh = view4(bf(DO.ptr, 64 * hv), FL_BF16, {B, S, H, 64},
                                        {DO.stride[0], DO.stride[1], DO.stride[2]});
            const fl_tensor oh = view4(ws + pl.off_o, FL_BF16, {B, S, H, 64}, packed_q);
            const size_t part = size_t(2 * hv + t); // partial buffers in (half, stream) order
            const fl_tensor gq = view4(ws + pl.off_dq + part * pl.unit_q, FL_BF16, {B, S, H, 64}, packed_q);
            const fl_tensor gk = view4(ws + pl.off_dk + part * pl.unit_k, FL_BF16, {B, S, Hk, 64}, packed_k);
            const fl_tensor gv = view4(ws + pl.off_dv + part * pl.unit_k, FL_BF16, {B, S, Hk, 64}, packed_k);
            // this stream's output over this half of V, then its backward with dO
            if ((s = fwd_standard(&qt, &kt, &vh, &oh, nullptr, &pl.sd, nullptr, nullptr,
                                  reinterpret_cast<cudaStream_t>(stream))) != FL_OK)
                return s;
            if ((s = fl_attn_bwd(&qt, &kt, &vh, &oh, &lt, &doh, &gq, &gk, &gv, &pl.sd, ws + pl.off_ws,
                                 pl.ws_bytes, stream)) != FL_OK)
                return s;
        }
    }
    // dQ_t = c_t sum over halves, dK_t likewise, dV half = sum_t c_t dV_t
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const auto part_ptr = [&](size_t off, size_t unit, int64_t hv, int t) {
        return reinterpret_cast<const __nv_bfloat16 *>(ws + off + size_t(2 * hv + t) * unit);
    };
    for (int t = 0; t < 2; ++t) {
        for (int which = 0; which < 2; ++which) { // dQ, dK
            const View &Out = which == 0 ? DQ : DK;
            const int64_t heads = which == 0 ? H : Hk;
            fl::DiffCombine c{};
            c.rows = B * S * heads;
            c.S = S;
            c.heads = heads;
            for (int64_t hv = 0; hv < pl.halves; ++hv) {
                c.in[hv] = which == 0 ? part_ptr(pl.off_dq, pl.unit_q, hv, t) : part_ptr(pl.off_dk, pl.unit_k, hv, t);
                c.coef[hv] = coef[t];
            }
            c.out = static_cast<__nv_bfloat16 *>(Out.ptr) + t * Out.stride[0];
            c.o_sb = Out.stride[1];
            c.o_ss = Out.stride[2];
            c.o_sh = Out.stride[3];
            const cudaError_t e = fl::launch_diff_bwd_combine(c, info.sm_count, st);
            if (e != cudaSuccess)
                return fail(FL_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
        }
    }
    for (int64_t hv = 0; hv < pl.halves; ++hv) {
        fl::DiffCombine c{};
        c.rows = B * S * Hk;
        c.S = S;
        c.heads = Hk;
        for (int t = 0; t < 2; ++t) {
            c.in[t] = part_ptr(pl.off_dv, pl.unit_k, hv, t);
            c.coef[t] = coef[t];
        }
        c.out = static_cast<__nv_bfloat16 *>(DV.ptr) + 64 * hv;
        c.o_sb = DV.stride[0];
        c.o_ss = DV.stride[1];
        c.o_sh = DV.stride[2];
        const cudaError_t e = fl::launch_diff_bwd_combine(c, info.sm_count, st);
        if (e != cudaSuccess)
            return fail(FL_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    }
    return ok();
}

// Otherwise (the column pass, or strides that do not merge) stacks run one
// launch each: the per-stack tensors are views of the caller's, only the base
// pointer moving by the stack stride, so validating the stack-stride rules and
// the first stack validates them all before anything is launched.
fl_status fl_attn_evoformer(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                            const fl_tensor *out, const fl_tensor *lse,
                            const fl_attn_variant_desc *desc, const fl_tensor *bias,
                            const fl_tensor *gate, const fl_tensor *msa_mask, fl_stream_t stream)
{
    if (!desc)
        return fail(FL_ERR_INVALID_ARG, "desc is NULL");
    if (desc->kind != FL_KIND_EVO_ROW && desc->kind != FL_KIND_EVO_COL)
        return fail(FL_ERR_INVALID_ARG, "fl_attn_evoformer takes FL_KIND_EVO_ROW or FL_KIND_EVO_COL");
    const bool row = desc->kind == FL_KIND_EVO_ROW;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!q)
        return fail(FL_ERR_INVALID_ARG, "q is NULL");
    if (q->ndim == 4)
        return fwd_evo(row, q, k, v, out, lse, desc, bias, gate, msa_mask, st);
    if (q->ndim != 5)
        return fail(FL_ERR_INVALID_ARG, "q must be [N_seq, N_res, H, c] or [B, N_seq, N_res, H, c]");
    const int64_t Bt = q->sizes[0];
    if (Bt < 1)
        return fail(FL_ERR_INVALID_ARG, "batch of stacks must be >= 1");
    // every batched tensor has one more leading axis of size Bt, whose stride
    // keeps the per-stack views aligned; bias and msa_mask may instead have
    // one axis fewer (one tensor shared by every stack)
    struct Arg {
        const fl_tensor *t;
        const char *name;
        int batched_rank;
        bool shared_ok;
    };
    const Arg args[] = {{q, "q", 5, false},       {k, "k", 5, false},
                        {v, "v", 5, false},       {out, "out", 5, false},
                        {gate, "gate", 5, false}, {lse, "lse", 4, false},
                        {bias, "bias", 4, true},  {msa_mask, "msa_mask", 3, true}};
    // The row pass runs as ONE launch over all stacks when each batched
    // tensor's stack stride is N_seq times its MSA-row stride (the stacks then
    // form one longer MSA-row axis), the mask (if any) is per stack, and the
    // bias is shared or per stack (work items then never straddle a stack).
    if (row && Bt > 1) {
        const int64_t Ns = q->sizes[1];
        auto merges = [&](const fl_tensor *t, int rank) {
            return t && t->ndim == rank && t->sizes[0] == Bt && t->strides[0] == Ns * t->strides[1] &&
                   t->sizes[1] == Ns;
        };
        const bool fold = merges(q, 5) && merges(k, 5) && merges(v, 5) && merges(out, 5) &&
                          merges(gate, 5) && (!lse || merges(lse, 4)) &&
                          (!msa_mask || merges(msa_mask, 3)) && bias && (bias->ndim == 3 || bias->ndim == 4);
        if (fold) {
            auto merged = [&](const fl_tensor *t) {
                fl_tensor m = *t;
                m.ndim = t->ndim - 1;
                m.sizes[0] = Bt * Ns;
                m.strides[0] = t->strides[1];
                for (int d = 1; d < m.ndim; ++d) {
                    m.sizes[d] = t->sizes[d + 1];
                    m.strides[d] = t->strides[d + 1];
                }
                return m;
            };
            const fl_tensor fq = merged(q), fk = merged(k), fv = merged(v), fo = merged(out), fg = merged(gate);
            fl_tensor fl{}, fm{};
            if (lse)
                fl = merged(lse);
            if (msa_mask)
                fm = merged(msa_mask);
            return fwd_evo(true, &fq, &fk, &fv, &fo, lse ? &fl : nullptr, desc, bias, &fg,
                           msa_mask ? &fm : nullptr, st, bias->ndim == 4 ? Ns : 0);
        }
    }
    fl_tensor views[8];
    const fl_tensor *per_stack[8];
    bool batched[8];
    for (int a = 0; a < 8; ++a) {
        per_stack[a] = args[a].t;
        batched[a] = false;
        if (!args[a].t)
            continue;
        const fl_tensor &t = *args[a].t;
        if (t.ndim == args[a].batched_rank) {
            if (t.sizes[0] != Bt)
                return fail(FL_ERR_INVALID_ARG, "%s has %lld stacks, q has %lld", args[a].name,
                            (long long)t.sizes[0], (long long)Bt);
            const int elt = t.dtype == FL_F32 ? 4 : 2;
            if (Bt > 1 && (t.strides[0] <= 0 || (t.strides[0] * elt) % 16 != 0))
                return fail(FL_ERR_ALIGNMENT, "%s stack stride must be a positive multiple of 16 bytes",
                            args[a].name);
            views[a] = t;
            views[a].ndim = t.ndim - 1;
            for (int d = 0; d < 4; ++d) {
                views[a].sizes[d] = t.sizes[d + 1];
                views[a].strides[d] = t.strides[d + 1];
            }
            per_stack[a] = &views[a];
            batched[a] = true;
        } else if (!(args[a].shared_ok && t.ndim == args[a].batched_rank - 1)) {
            return fail(FL_ERR_INVALID_ARG, "%s must have %d dimensions%s", args[a].name,
                        args[a].batched_rank, args[a].shared_ok ? " (or one fewer, shared)" : "");
        }
    }
    for (int64_t b = 0; b < Bt; ++b) {
        for (int a = 0; a < 8; ++a)
            if (batched[a]) {
                const fl_tensor &t = *args[a].t;
                const int elt = t.dtype == FL_F32 ? 4 : 2;
                views[a].ptr = static_cast<char *>(t.ptr) + b * t.strides[0] * elt;
            }
        const fl_status s = fwd_evo(row, per_stack[0], per_stack[1], per_stack[2], per_stack[3],
                                    per_stack[5], desc, per_stack[6], per_stack[4], per_stack[7], st);
        if (s != FL_OK)
            return s;
    }
    return ok();
}

fl_status fl_attn_score_expr_check(const char *expr, int32_t compile)
{
    std::vector<char> cuda(kExprCudaMax), grad(kExprCudaMax);
    char err[1024];
    if (!fl::score_expr_translate_grad(expr, cuda.data(), cuda.size(), grad.data(), grad.size(), err, sizeof err))
        return fail(FL_ERR_INVALID_ARG, "score_mod_expr: %s", err);
    if (compile && !fl::score_expr_compile_only(cuda.data(), compile > 1 ? grad.data() : nullptr, err, sizeof err))
        return fail(strstr(err, "not found") ? FL_ERR_UNSUPPORTED : FL_ERR_INVALID_ARG,
                    "score_mod_expr: %s", err);
    return ok();
}

// No workspace argument: the scratch is the library's own static device
// array (fl::decode_static_scratch), looked up on the first call per context.
// Nothing is allocated.
fl_status fl_attn_decode_static(const fl_tensor *q, const fl_tensor *k_cache,
                                const fl_tensor *v_cache, const fl_tensor *out,
                                const fl_tensor *lse, const fl_decode_desc *desc,
                                fl_stream_t stream)
{
    if (!v_cache)
        return fail(FL_ERR_INVALID_ARG, "v_cache is NULL");
    DecodePlan pl;
    fl_status s = decode_plan(q, k_cache, v_cache, desc, pl);
    if (s != FL_OK)
        return s;
    if (pl.total > fl::kDecodeStaticScratch)
        return fail(FL_ERR_UNSUPPORTED,
                    "these shapes need %zu bytes of scratch; the library's static decode scratch "
                    "holds %zu (use fl_attn_decode with a workspace)",
                    pl.total, fl::kDecodeStaticScratch);
    int dev;
    DeviceInfo info;
    if ((s = device_info(dev, info)) != FL_OK)
        return s;
    void *scratch = nullptr;
    const cudaError_t e = fl::decode_static_scratch(&scratch);
    if (e != cudaSuccess)
        return fail(FL_ERR_CUDA, "looking up the static decode scratch failed: %s",
                    cudaGetErrorString(e));
    return decode_run(pl, out, lse, desc, scratch, reinterpret_cast<cudaStream_t>(stream));
}

fl_status fl_attn_decode_workspace_size(const fl_tensor *q, const fl_tensor *k_cache,
                                        const fl_decode_desc *desc, size_t *bytes)
{
    if (!bytes)
        return fail(FL_ERR_INVALID_ARG, "bytes is NULL");
    DecodePlan pl;
    fl_status s = decode_plan(q, k_cache, nullptr, desc, pl);
    if (s != FL_OK)
        return s;
    *bytes = pl.total;
    return ok();
}

fl_status fl_attn_decode(const fl_tensor *q, const fl_tensor *k_cache, const fl_tensor *v_cache,
                         const fl_tensor *out, const fl_tensor *lse, const fl_decode_desc *desc,
                         void *workspace, size_t workspace_bytes, fl_stream_t stream)
{
    if (!v_cache)
        return fail(FL_ERR_INVALID_ARG, "v_cache is NULL");
    DecodePlan pl;
    fl_status s = decode_plan(q, k_cache, v_cache, desc, pl);
    if (s != FL_OK)
        return s;
    if (!workspace)
        return fail(FL_ERR_INVALID_ARG, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % kWsAlign)
        return fail(FL_ERR_ALIGNMENT, "workspace is not %zu-byte aligned", kWsAlign);
    if (workspace_bytes < pl.total)
        return fail(FL_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", workspace_bytes,
                    pl.total);
    return decode_run(pl, out, lse, desc, workspace, reinterpret_cast<cudaStream_t>(stream));
}

fl_status fl_attn_fwd(const fl_tensor *q, const fl_tensor *k, const fl_tensor *v,
                      const fl_tensor *out, const fl_tensor *lse,
                      const fl_attn_variant_desc *desc, const fl_tensor *bias,
                      const fl_tensor *gate, fl_stream_t stream)
{
    if (!desc)
        return fail(FL_ERR_INVALID_ARG, "desc is NULL");
    switch (desc->kind) {
    case FL_KIND_STANDARD:
        return fwd_standard(q, k, v, out, lse, desc, bias, gate, reinterpret_cast<cudaStream_t>(stream));
    case FL_KIND_DIFF:
        return fwd_diff(q, k, v, out, lse, desc, bias, gate, reinterpret_cast<cudaStream_t>(stream));
    case FL_KIND_EVO_ROW:
    case FL_KIND_EVO_COL:
        return fwd_evo(desc->kind == FL_KIND_EVO_ROW, q, k, v, out, lse, desc, bias, gate, nullptr,
                       reinterpret_cast<cudaStream_t>(stream));
    default:
        return fail(FL_ERR_INVALID_ARG, "unknown kind %d", desc->kind);
    }
}

fl_status fl_attn_tile_shape(const fl_attn_variant_desc *desc, int32_t head_dim, int32_t *block_m,
                             int32_t *block_n)
{
    if (!desc || !block_m || !block_n)
        return fail(FL_ERR_INVALID_ARG, "NULL argument");
    switch (desc->kind) {
    case FL_KIND_STANDARD:
        if (head_dim != 32 && head_dim != 64 && head_dim != 128)
            return fail(FL_ERR_UNSUPPORTED, "head_dim %d not supported for kind %d", head_dim,
                        desc->kind);
        break;
    case FL_KIND_DIFF: // head_dim is the value head dimension Dv here (D is 64)
        if (head_dim != 64 && head_dim != 128)
            return fail(FL_ERR_UNSUPPORTED, "value head_dim %d not supported for kind %d", head_dim,
                        desc->kind);
        break;
    case FL_KIND_EVO_ROW:
    case FL_KIND_EVO_COL:
        if (head_dim != 32 && head_dim != 64)
            return fail(FL_ERR_UNSUPPORTED, "head_dim %d not supported for kind %d", head_dim,
                        desc->kind);
        break;
    default:
        return fail(FL_ERR_INVALID_ARG, "unknown kind %d", desc->kind);
    }
    *block_m = fl::BM;
    *block_n = desc->kind == FL_KIND_STANDARD ? fl::std_key_tile(head_dim)
               : desc->kind == FL_KIND_DIFF   ? fl::diff_key_tile(head_dim)
                                              : fl::BN;
    return ok();
}

const char *fl_attn_status_string(fl_status s)
{
    switch (s) {
    case FL_OK: return "FL_OK";
    case FL_ERR_INVALID_ARG: return "FL_ERR_INVALID_ARG: invalid argument";
    case FL_ERR_UNSUPPORTED: return "FL_ERR_UNSUPPORTED: outside the compiled kernel set";
    case FL_ERR_ALIGNMENT: return "FL_ERR_ALIGNMENT: pointer or stride not 16-byte aligned";
    case FL_ERR_CUDA: return "FL_ERR_CUDA: CUDA call failed";
    case FL_ERR_DEVICE_TIMEOUT: return "FL_ERR_DEVICE_TIMEOUT: a device-side wait ran out";
    case FL_ERR_NO_DEVICE: return "FL_ERR_NO_DEVICE: no sm_103 device";
    default: return "unknown fl_status";
    }
}

const char *fl_attn_last_error(void) { return g_last_error; }

int32_t fl_attn_version(void) { return FL_ATTN_VERSION; }

} // extern "C"
