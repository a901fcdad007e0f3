/*
 * fl_oracle.c -- CPU oracle for the fused attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA library never
 * calls it and shares no code, header or table with it.
 *
 * What it computes is the plain definition, in double precision, of the
 * result the fused kernel reaches by an online softmax (Flashlight,
 * gist.science summary, "Methodology" items 2-4: the online softmax is an
 * exact algebraic rewrite of the stable two-pass softmax via
 * e^(x-y) = e^x / e^y; talk notes, "Comparison with FlexAttention":
 * equivalent over the reals).  For every requested query row it
 *
 *   1. forms the whole logit row  z_j = score_mod(scale * q_i . k_j) + bias_ij,
 *      or -inf where the mask forbids the pair (i, j);
 *   2. runs the two-pass stable softmax: m = max_j z_j, l = sum_j e^(z_j - m),
 *      P_j = e^(z_j - m) / l;
 *   3. returns O_i = sum_j P_j v_j and LSE_i = m + ln l (natural log).
 *
 * A row whose every key is masked returns O_i = 0 and LSE_i = -inf.
 *
 * Inputs are bf16 bit patterns, widened exactly to double.  Nothing is
 * blocked, fused or reordered beyond the definition above.
 *
 * Variant definitions (score_mod and masks), taken from the workload
 * statement that accompanies the pages (the pages name the variants in the
 * talk notes, "Evaluation: FlexAttention-supported variants", but give no
 * formulas):
 *   ALiBi    z += -slope_h * |i - j|,  slope_h = 2^(-8 (h + 1) / H), h 0-based
 *   softcap  z  = cap * tanh(z / cap)
 *   causal   key j allowed iff j <= i
 *   window   allowed iff j <= i and i - j < W
 *   prefix   allowed iff j <= i or j < P   (bidirectional over the first P)
 *   document allowed iff doc(i) == doc(j) and j <= i
 *   KV length  allowed iff j < kv_len[b]            (a cache of kv_len[b] keys)
 *   decode     allowed iff j < kv_len[b] and j <= kv_len[b] - Sq + i
 *              (the Sq query rows are the last Sq positions of a sequence of
 *              kv_len[b] tokens: serving with a KV cache, talk notes,
 *              "End-to-end: LLaMA-3.2-1B (vLLM / Mooncake)", causal variant)
 *   key mask (any of the above, and)  key j of batch element b allowed only if
 *              key_mask[b][j] != 0  (the Evoformer MSA mask: a masked residue or
 *              sequence is removed as a key; AlphaFold2 context, talk notes,
 *              "End-to-end: AlphaFold2")
 * Query head h reads key/value head h / (Hq / Hk) (contiguous GQA groups).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define FL_ORACLE_MOD_NONE 0
#define FL_ORACLE_MOD_ALIBI 1
#define FL_ORACLE_MOD_SOFTCAP 2

#define FL_ORACLE_MASK_NONE 0
#define FL_ORACLE_MASK_CAUSAL 1
#define FL_ORACLE_MASK_WINDOW 2
#define FL_ORACLE_MASK_PREFIX 3
#define FL_ORACLE_MASK_DOC 4
#define FL_ORACLE_MASK_KVLEN 5
#define FL_ORACLE_MASK_DECODE 6

typedef struct {
    int32_t B, Hq, Hk, Sq, Sk, D, Dv;
    /* element strides of the (batch, position, head) axes; features contiguous */
    int64_t q_stride[3];
    int64_t k_stride[3];
    int64_t v_stride[3];
    int32_t score_mod;
    double softcap;
    const double *alibi_slopes; /* [Hq], or NULL for 2^(-8 (h+1) / Hq) */
    int32_t mask;
    int32_t window;
    int32_t prefix;
    const int32_t *doc_offsets; /* [B][doc_stride] ascending starts, padded with Sk */
    int32_t doc_stride;
    double scale;               /* 0 means 1 / sqrt(D) */
    const uint16_t *bias;       /* NULL, or bias[h, i, j] with the strides below */
    int64_t bias_stride[3];
    const int32_t *kv_len;      /* [B] cache lengths (KV-length and decode masks) */
    const uint8_t *key_mask;    /* NULL, or key_mask[b, j] with the strides below */
    int64_t key_mask_stride[2];
} fl_oracle_problem;

static double widen_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Index of the document holding position x: the number of document starts
 * at or before x, minus one. */
static int32_t doc_of(const int32_t *starts, int32_t n, int32_t x)
{
    int32_t d = -1;
    for (int32_t t = 0; t < n; ++t)
        if (starts[t] <= x)
            d = t;
    return d;
}

static int allowed(const fl_oracle_problem *p, int32_t b, int64_t i, int64_t j)
{
    if (p->key_mask && !p->key_mask[b * p->key_mask_stride[0] + j * p->key_mask_stride[1]])
        return 0;
    switch (p->mask) {
    case FL_ORACLE_MASK_NONE:
        return 1;
    case FL_ORACLE_MASK_CAUSAL:
        return j <= i;
    case FL_ORACLE_MASK_WINDOW:
        return j <= i && i - j < p->window;
    case FL_ORACLE_MASK_PREFIX:
        return j <= i || j < p->prefix;
    case FL_ORACLE_MASK_DOC: {
        const int32_t *starts = p->doc_offsets + (int64_t)b * p->doc_stride;
        return j <= i && doc_of(starts, p->doc_stride, (int32_t)i) ==
                             doc_of(starts, p->doc_stride, (int32_t)j);
    }
    case FL_ORACLE_MASK_KVLEN:
        return j < p->kv_len[b];
    case FL_ORACLE_MASK_DECODE:
        return j < p->kv_len[b] && j <= (int64_t)p->kv_len[b] - p->Sq + i;
    default:
        return 0;
    }
}

static double alibi_slope(const fl_oracle_problem *p, int32_t h)
{
    if (p->alibi_slopes)
        return p->alibi_slopes[h];
    return pow(2.0, -8.0 * (double)(h + 1) / (double)p->Hq);
}

/* One query row (b, h, i): writes Dv outputs and the log-sum-exp. */
static void one_row(const fl_oracle_problem *p, const uint16_t *q, const uint16_t *k,
                    const uint16_t *v, int32_t b, int32_t h, int64_t i, double *z,
                    double *o, double *lse)
{
    const int32_t group = p->Hq / p->Hk;
    const int32_t hk = h / group;
    const double scale = p->scale != 0.0 ? p->scale : 1.0 / sqrt((double)p->D);
    const uint16_t *qi = q + b * p->q_stride[0] + i * p->q_stride[1] + h * p->q_stride[2];

    /* step 1: the whole logit row */
    for (int64_t j = 0; j < p->Sk; ++j) {
        if (!allowed(p, b, i, j)) {
            z[j] = -INFINITY;
            continue;
        }
        const uint16_t *kj = k + b * p->k_stride[0] + j * p->k_stride[1] + hk * p->k_stride[2];
        double dot = 0.0;
        for (int32_t d = 0; d < p->D; ++d)
            dot += widen_bf16(qi[d]) * widen_bf16(kj[d]);
        double x = scale * dot;
        if (p->score_mod == FL_ORACLE_MOD_ALIBI)
            x += -alibi_slope(p, h) * fabs((double)(i - j));
        else if (p->score_mod == FL_ORACLE_MOD_SOFTCAP)
            x = p->softcap * tanh(x / p->softcap);
        if (p->bias)
            x += widen_bf16(p->bias[h * p->bias_stride[0] + i * p->bias_stride[1] +
                                    j * p->bias_stride[2]]);
        z[j] = x;
    }

    /* step 2: two-pass stable softmax */
    double m = -INFINITY;
    for (int64_t j = 0; j < p->Sk; ++j)
        if (z[j] > m)
            m = z[j];
    for (int32_t d = 0; d < p->Dv; ++d)
        o[d] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < p->Sk; ++j)
        l += exp(z[j] - m);

    /* step 3: P V and the log-sum-exp */
    for (int64_t j = 0; j < p->Sk; ++j) {
        if (z[j] == -INFINITY)
            continue;
        const double pj = exp(z[j] - m) / l;
        const uint16_t *vj = v + b * p->v_stride[0] + j * p->v_stride[1] + hk * p->v_stride[2];
        for (int32_t d = 0; d < p->Dv; ++d)
            o[d] += pj * widen_bf16(vj[d]);
    }
    *lse = m + log(l);
}

/*
 * rows == NULL: every row; out is [B][Sq][Hq][Dv], lse is [B][Hq][Sq].
 * rows != NULL: n_rows triples (b, h, i); out is [n_rows][Dv], lse [n_rows].
 * Returns 0, or -1 on an invalid problem.
 */
int fl_oracle_attention(const fl_oracle_problem *p, const uint16_t *q, const uint16_t *k,
                        const uint16_t *v, const int64_t *rows, int64_t n_rows, double *out,
                        double *lse, int nthreads)
{
    if (!p || !q || !k || !v || !out || !lse || p->Hk <= 0 || p->Hq % p->Hk != 0 ||
        p->D <= 0 || p->Dv <= 0 || p->Sk < 0 || p->Sq < 0)
        return -1;
    if (p->mask == FL_ORACLE_MASK_DOC && (!p->doc_offsets || p->doc_stride <= 0))
        return -1;
    if (p->mask == FL_ORACLE_MASK_KVLEN || p->mask == FL_ORACLE_MASK_DECODE) {
        if (!p->kv_len)
            return -1;
        for (int32_t b = 0; b < p->B; ++b)
            if (p->kv_len[b] < 0 || p->kv_len[b] > p->Sk ||
                (p->mask == FL_ORACLE_MASK_DECODE && p->kv_len[b] < p->Sq))
                return -1;
    }
    if (rows) {
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[3 * r] < 0 || rows[3 * r] >= p->B || rows[3 * r + 1] < 0 ||
                rows[3 * r + 1] >= p->Hq || rows[3 * r + 2] < 0 || rows[3 * r + 2] >= p->Sq)
                return -1;
    }
    const int64_t total = rows ? n_rows : (int64_t)p->B * p->Hq * p->Sq;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)(p->Sk > 0 ? p->Sk : 1));
        if (!z) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < total; ++r) {
            if (!z)
                continue;
            int32_t b, h;
            int64_t i;
            double *o, *l;
            if (rows) {
                b = (int32_t)rows[3 * r];
                h = (int32_t)rows[3 * r + 1];
                i = rows[3 * r + 2];
                o = out + r * p->Dv;
                l = lse + r;
            } else {
                /* r enumerates (b, h, i) with i fastest */
                i = r % p->Sq;
                h = (int32_t)((r / p->Sq) % p->Hq);
                b = (int32_t)(r / ((int64_t)p->Sq * p->Hq));
                o = out + (((int64_t)b * p->Sq + i) * p->Hq + h) * p->Dv;
                l = lse + ((int64_t)b * p->Hq + h) * p->Sq + i;
            }
            one_row(p, q, k, v, b, h, i, z, o, l);
        }
        free(z);
    }
    return failed ? -1 : 0;
}

/* Threads the oracle would use for nthreads == 0. */
int fl_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
