/*
 * fp64 CPU oracle for paged-KV GQA/MQA verify attention.
 *
 * TEST INFRASTRUCTURE.  Only the tests, __graft_entry__.smoke() and the
 * benchmark's CPU-baseline / reference arm may load this library.  It shares
 * no code, header or constant with the CUDA path.
 *
 * What it computes is the plain definition, evaluated in double precision:
 *
 *   for request b, query token t < L_b and query head qh (KV head h = qh / G):
 *     K_b, V_b  = the request's cached keys / values gathered in position
 *                 order through its page table, decoded and multiplied by the
 *                 per-tensor k_scale / v_scale;
 *     s_j       = sm_scale * <Q[t, qh], K_b[j, h]> + M_b[t, j]
 *     lse       = ln sum_j exp(s_j)            (max-shifted for range only)
 *     out       = sum_j exp(s_j - lse) * V_b[j, h]
 *
 * with M_b an explicit dense [L_b, kv_len_b] additive mask (0 or -inf).
 * Sources, by page:
 *  - "flashmap 0.1.0 - flashmap/sglang/verify_attention.py": the split-KV
 *    verify kernel's docstring and its two branches define the row map
 *    (query head h*G + g shares KV head h), the visible set (the whole prefix
 *    plus the draft columns the tree mask or causality allows), the scales
 *    (k_scale on the logits, v_scale on the values) and the natural-log LSE;
 *    its merge kernel defines how splits recombine (oracle_merge_partials).
 *  - vLLM PR #2401 "Support MQA/GQA in prefill stage by using FlashAttention":
 *    GQA as MHA on K/V expanded per query head.
 *  - FlashInfer PR #286 "Separate Q and KV dtypes for decode",
 *    begin_forward's parameters: the page table (indptr, indices,
 *    last_page_len, page_size).
 *  - FlashInfer issue #152 "How to implement a tree attention": custom
 *    (tree) masks, -inf (or -5e4) where masked and 0 elsewhere.
 *
 * Readings where the sources leave a step open: drafts are appended to the
 * pages before attention, so the queries are the last L_b positions of the kv
 * range; the mask is each request's L_b x L_b block, bit-packed LSB-first at
 * bit offset mask_indptr[b], bit 1 = visible, the prefix always visible; with
 * no mask the draft columns are causal (u <= t); a fully masked row has
 * lse = -inf and out = 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_EINVAL -1
#define OR_ENOMEM -2

/* bf16: the upper 16 bits of an IEEE-754 binary32. */
double oracle_decode_bf16(uint16_t bits) {
    union { uint32_t u; float f; } x;
    x.u = ((uint32_t)bits) << 16;
    return (double)x.f;
}

/* fp8 e4m3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinity. */
double oracle_decode_e4m3(uint8_t bits) {
    int sign = bits >> 7;
    int e = (bits >> 3) & 15;
    int m = bits & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

/* fp8-e4m3 code of a binary32 value, on the grid oracle_decode_e4m3 defines
 * (subnormals m * 2^-9, m = 0..7; normals (8 + m) * 2^(e - 10), e = 1..15):
 * the nearest grid value, a tie going to the code whose last mantissa bit is
 * 0 (round to nearest even); finite overflow and infinities saturate to
 * +-448, the largest finite value ("satfinite"); NaN gives the NaN code
 * 0x7F. */
static uint8_t encode_e4m3_value(double x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; 8 * 2^-9 = 2^-6 is code 0x08 */
        double m = nearbyint(ldexp(a, 9));
        return sign | (uint8_t)m;
    }
    int ex;
    (void)frexp(a, &ex);              /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                   /* 2^e <= a < 2^(e+1), e in [-6, 8] */
    double m = nearbyint(ldexp(a, 3 - e));   /* in [8, 16] */
    if (m == 16.0) {
        m = 8.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && m > 14.0)) return sign | 0x7E;
    return sign | (uint8_t)(((e + 7) << 3) | ((int)m - 8));
}

uint8_t oracle_encode_e4m3_satfinite(float x) { return encode_e4m3_value((double)x); }

/* bf16 bits of the value nearest to x (ties to the even code): 8 significant
 * bits, exponents down to 2^-126 with subnormals at multiples of 2^-133,
 * overflow to infinity (binary32's exponent range). */
uint16_t oracle_encode_bf16(double x) {
    union { float f; uint32_t u; } v;
    if (isnan(x)) return 0x7FC0;
    double a = fabs(x);
    double r;
    if (a == 0.0 || isinf(a)) {
        r = a;
    } else {
        int ex;
        (void)frexp(a, &ex);
        int e = ex - 1;
        if (e < -126) e = -126;
        double m = nearbyint(ldexp(a, 7 - e));
        r = ldexp(m, e - 7);
        /* the largest finite bf16 is (2 - 2^-7) * 2^127; a tie above it rounds up */
        if (r >= ldexp(1.0, 128)) r = INFINITY;
    }
    v.f = (float)r;                   /* exact: r is on the bf16 grid */
    uint16_t bits = (uint16_t)(v.u >> 16);
    return signbit(x) ? (uint16_t)(bits | 0x8000) : bits;
}

/* LLaMA-style rotary position embedding of one d-vector in place ("rotate
 * half": element i pairs with i + d/2): for i < d/2, with angle
 * a_i = pos / scale * theta^(-2i/d),
 *   y_i = x_i cos a_i - x_{i+d/2} sin a_i,  y_{i+d/2} = x_{i+d/2} cos a_i + x_i sin a_i.
 * FlashInfer PR #286 names it ROPE_LLAMA (rope_theta, rope_scale); FlashInfer
 * issue #152 asks for it at each draft's tree position. */
void oracle_rope_vec(double* x, int d, double pos, double theta, double scale) {
    int half = d / 2;
    for (int i = 0; i < half; ++i) {
        double a = pos / scale * pow(theta, -2.0 * i / d);
        double c = cos(a), sn = sin(a);
        double x0 = x[i], x1 = x[i + half];
        x[i] = x0 * c - x1 * sn;
        x[i + half] = x1 * c + x0 * sn;
    }
}

/* The binary32 quotient x / scale, correctly rounded: the quotient of two
 * binary32 values computed in binary64 and rounded once more to binary32
 * equals the correctly rounded binary32 quotient, because 53 >= 2 * 24 + 2
 * (double rounding is innocuous for division at that precision; Figueroa,
 * "When is double rounding innocuous?", SIGNUM 1995). */
float oracle_div_f32(float x, float scale) {
    return (float)((double)x / (double)scale);
}

/* A query row as the e4m3 tensor-core path takes it: with amax = max |q_i|,
 * inv = 448 / amax and qsc = amax / 448 (binary32 divisions), each element
 * is stored as the e4m3 code of the binary32 product q_i * inv (round to
 * nearest even, saturating), and the row stands for codes * qsc.  An all-zero
 * row keeps scale 1.  Writes the codes and returns qsc. */
float oracle_quantize_q_e4m3(const double* q, int d, uint8_t* codes) {
    float amax = 0.0f;
    for (int e = 0; e < d; ++e) {
        float a = (float)fabs(q[e]);
        if (a > amax) amax = a;
    }
    float inv = amax > 0.0f ? oracle_div_f32(448.0f, amax) : 1.0f;
    float qsc = amax > 0.0f ? oracle_div_f32(amax, 448.0f) : 1.0f;
    for (int e = 0; e < d; ++e) {
        /* the binary32 product: exact in binary64 (24 + 24 bits), rounded once */
        float x = (float)((double)(float)q[e] * (double)inv);
        codes[e] = oracle_encode_e4m3_satfinite(x);
    }
    return qsc;
}

static double decode_kv(const void* base, int64_t idx, int kv_fp8) {
    if (kv_fp8) return oracle_decode_e4m3(((const uint8_t*)base)[idx]);
    return oracle_decode_bf16(((const uint16_t*)base)[idx]);
}

/* kv_len of request b from FlashInfer's page table: (pages - 1) * page_size
 * + last_page_len, and 0 for a request with no pages. */
int64_t oracle_kv_len(const int32_t* kv_indptr, const int32_t* last_page_len, int b,
                      int page_size) {
    int64_t n = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
    if (n <= 0) return 0;
    return (n - 1) * page_size + last_page_len[b];
}

static int check_tables(const int32_t* kv_indptr, const int32_t* kv_indices,
                        const int32_t* last_page_len, const int32_t* qo_indptr, int batch,
                        int page_size, int num_pages) {
    if (batch < 0 || page_size <= 0) return OR_EINVAL;
    if (kv_indptr[0] != 0 || qo_indptr[0] != 0) return OR_EINVAL;
    for (int b = 0; b < batch; ++b) {
        int32_t np = kv_indptr[b + 1] - kv_indptr[b];
        int32_t nq = qo_indptr[b + 1] - qo_indptr[b];
        if (np < 0 || nq < 0) return OR_EINVAL;
        if (np > 0 && (last_page_len[b] < 1 || last_page_len[b] > page_size)) return OR_EINVAL;
        if (oracle_kv_len(kv_indptr, last_page_len, b, page_size) < nq) return OR_EINVAL;
        for (int32_t p = kv_indptr[b]; p < kv_indptr[b + 1]; ++p)
            if (kv_indices[p] < 0 || kv_indices[p] >= num_pages) return OR_EINVAL;
    }
    return OR_OK;
}

/*
 * Dense attention for one head: rows x keys, explicit additive mask.
 * out[r][e] = sum_j softmax_j(scale * Q[r].K[j] + M[r][j]) * V[j][e],
 * lse[r] = ln sum_j exp(scale * Q[r].K[j] + M[r][j]).
 * Q row stride q_ld, K / V row stride kv_ld (in doubles).  A row whose every
 * entry is masked gets lse = -inf and out = 0.  The _dv form takes values of
 * dv elements (sglang's value head size, which may differ from the key's d)
 * and separate K and V row strides; out rows then hold dv elements.
 */
void oracle_dense_attention_dv(int n_rows, int n_keys, int d, int dv, const double* Q,
                               int64_t q_ld, const double* K, int64_t k_ld, const double* V,
                               int64_t v_ld, const double* M, double scale, double* out,
                               double* lse, double* s_scratch) {
    for (int r = 0; r < n_rows; ++r) {
        const double* qr = Q + (int64_t)r * q_ld;
        double mx = -INFINITY;
        for (int j = 0; j < n_keys; ++j) {
            const double* kj = K + (int64_t)j * k_ld;
            double dot = 0.0;
            for (int e = 0; e < d; ++e) dot += qr[e] * kj[e];
            double s = scale * dot + M[(int64_t)r * n_keys + j];
            s_scratch[j] = s;
            if (s > mx) mx = s;
        }
        double* o = out + (int64_t)r * dv;
        for (int e = 0; e < dv; ++e) o[e] = 0.0;
        if (mx == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int j = 0; j < n_keys; ++j) sum += exp(s_scratch[j] - mx);
        double l = mx + log(sum);
        lse[r] = l;
        for (int j = 0; j < n_keys; ++j) {
            double p = exp(s_scratch[j] - l);
            if (p == 0.0) continue;
            const double* vj = V + (int64_t)j * v_ld;
            for (int e = 0; e < dv; ++e) o[e] += p * vj[e];
        }
    }
}

void oracle_dense_attention(int n_rows, int n_keys, int d, const double* Q, int64_t q_ld,
                            const double* K, const double* V, int64_t kv_ld,
                            const double* M, double scale, double* out, double* lse,
                            double* s_scratch) {
    oracle_dense_attention_dv(n_rows, n_keys, d, d, Q, q_ld, K, kv_ld, V, kv_ld, M, scale, out,
                              lse, s_scratch);
}

/* Row index of (page, head, slot) in a cache of the given layout: HND
 * [pages][h_kv][P][d] or NHD [pages][P][h_kv][d] (FlashInfer PR #286's
 * kv_layout). */
static int64_t cache_row(int layout, int64_t page, int h, int64_t slot, int h_kv, int page_size) {
    if (layout == 1) return (page * page_size + slot) * h_kv + h;
    return (page * h_kv + h) * page_size + slot;
}

/* Gather request b's K into [kv_len][h_kv][d] and V into [kv_len][h_kv][dv]
 * doubles (decoded and scaled), walking its pages in order and stopping at
 * kv_len; the V cache's rows hold dv elements. */
static void gather_request(const void* k_cache, const void* v_cache, int kv_fp8, int layout,
                           const int32_t* kv_indptr, const int32_t* kv_indices, int b,
                           int64_t kv_len, int h_kv, int d, int dv, int page_size,
                           double k_scale, double v_scale, double* K, double* V) {
    for (int64_t j = 0; j < kv_len; ++j) {
        int32_t page = kv_indices[kv_indptr[b] + j / page_size];
        int64_t slot = j % page_size;
        for (int h = 0; h < h_kv; ++h) {
            int64_t row = cache_row(layout, page, h, slot, h_kv, page_size);
            for (int e = 0; e < d; ++e)
                K[(j * h_kv + h) * d + e] = decode_kv(k_cache, row * d + e, kv_fp8) * k_scale;
            for (int e = 0; e < dv; ++e)
                V[(j * h_kv + h) * dv + e] = decode_kv(v_cache, row * dv + e, kv_fp8) * v_scale;
        }
    }
}

static int mask_bit(const uint8_t* mask, int64_t bit) {
    return (mask[bit >> 3] >> (bit & 7)) & 1;
}

/* Request b's explicit [L][kv_len] additive mask.  Layout 0 (each request's
 * L x L draft block, as flashmap's QLEN_ONLY custom mask): prefix columns 0;
 * draft column prefix + u is 0 when visible to token t (mask bit (t, u) at
 * mask_indptr[b] + t * L + u, or u <= t with no mask) and -inf otherwise.
 * Layout 1 (flashmap's full custom mask: L rows of kv_len bits): column j is
 * 0 iff bit mask_indptr[b] + t * kv_len + j is set, prefix columns included. */
static void build_mask(const uint8_t* mask, const int32_t* mask_indptr, int mask_layout, int b,
                       int64_t L, int64_t kv_len, double* M) {
    int64_t prefix = kv_len - L;
    for (int64_t t = 0; t < L; ++t) {
        for (int64_t j = 0; j < kv_len; ++j) {
            int visible;
            if (mask && mask_layout == 1) {
                visible = mask_bit(mask, (int64_t)mask_indptr[b] + t * kv_len + j);
            } else if (j < prefix) {
                visible = 1;
            } else {
                int64_t u = j - prefix;
                if (mask) visible = mask_bit(mask, (int64_t)mask_indptr[b] + t * L + u);
                else visible = (u <= t);
            }
            M[t * kv_len + j] = visible ? 0.0 : -INFINITY;
        }
    }
}

typedef struct {
    /* shared, read-only */
    const uint16_t* q;
    const double* K;
    const double* V;
    const double* M;
    int64_t kv_len, L, qo_start;
    int h_q, h_kv, d, dv, group;
    double sm_scale;
    const int32_t* q_pos;  /* NULL: no rotary embedding of the queries */
    int q_fp8;             /* 1: the row is replaced by its e4m3 quantisation */
    double rope_theta, rope_scale;
    const int64_t* rows;   /* flat row ids token*h_q+head of this request */
    const int64_t* dest;   /* where each row's result goes */
    int64_t n_rows;
    double* out;
    double* lse;
    /* per thread */
    int64_t lo, hi;
    int status;
} job_t;

static void* run_rows(void* arg) {
    job_t* jb = (job_t*)arg;
    double* s = (double*)malloc(sizeof(double) * (size_t)(jb->kv_len > 0 ? jb->kv_len : 1));
    double* qrow = (double*)malloc(sizeof(double) * (size_t)jb->d);
    if (!s || !qrow) {
        free(s);
        free(qrow);
        jb->status = OR_ENOMEM;
        return NULL;
    }
    for (int64_t i = jb->lo; i < jb->hi; ++i) {
        int64_t flat = jb->rows[i];
        int64_t tok = flat / jb->h_q;
        int qh = (int)(flat % jb->h_q);
        int h = qh / jb->group;
        int64_t t = tok - jb->qo_start;
        for (int e = 0; e < jb->d; ++e)
            qrow[e] = oracle_decode_bf16(jb->q[flat * jb->d + e]);
        if (jb->q_pos) {
            /* RoPE maps the bf16 query tensor to a bf16 query tensor: the
             * rotated row is rounded once to bf16 (nearest even) before the
             * dot products, as the rotated queries the pages' kernels feed
             * to their bf16 matrix units are */
            oracle_rope_vec(qrow, jb->d, (double)jb->q_pos[tok], jb->rope_theta, jb->rope_scale);
            for (int e = 0; e < jb->d; ++e)
                qrow[e] = oracle_decode_bf16(oracle_encode_bf16(qrow[e]));
        }
        if (jb->q_fp8) {
            uint8_t codes[1024];
            double qsc = (double)oracle_quantize_q_e4m3(qrow, jb->d, codes);
            for (int e = 0; e < jb->d; ++e) qrow[e] = oracle_decode_e4m3(codes[e]) * qsc;
        }
        /* One query row against the request's keys of KV head h: K/V rows are
         * [j][h][:] so the row stride is h_kv * d and the base is offset by h. */
        oracle_dense_attention_dv(1, (int)jb->kv_len, jb->d, jb->dv, qrow, jb->d,
                                  jb->K + (int64_t)h * jb->d, (int64_t)jb->h_kv * jb->d,
                                  jb->V + (int64_t)h * jb->dv, (int64_t)jb->h_kv * jb->dv,
                                  jb->M + t * jb->kv_len, jb->sm_scale,
                                  jb->out + jb->dest[i] * jb->dv, jb->lse + jb->dest[i], s);
    }
    free(s);
    free(qrow);
    return NULL;
}

/*
 * The whole verify attention of a batch, or of a selection of output rows.
 *  q        [total_qo, h_q, d] bf16 bits
 *  k_cache, v_cache bf16 (kv_fp8 = 0) or fp8-e4m3 (kv_fp8 = 1) bit patterns
 *           in the HND (kv_layout 0: [num_pages, h_kv, page_size, d]) or NHD
 *           (kv_layout 1: [num_pages, page_size, h_kv, d]) layout; the cache
 *           holds keys as stored (rotated by the append when RoPE is used)
 *  mask_layout: 0 = each request's L x L draft block, 1 = L rows of kv_len
 *           bits (see build_mask)
 *  q_pos    NULL, or [total_qo] positions: each query row is rotated by
 *           oracle_rope_vec at its token's position (rope_theta, rope_scale)
 *           and rounded to bf16 (the query dtype) before the dot products
 *  q_fp8    1: each query row (after any rotation) is replaced by its e4m3
 *           quantisation (oracle_quantize_q_e4m3: codes times the row scale),
 *           the operand of the e4m3 tensor-core path
 *  dv       elements of a value row (v_cache rows and out rows), which may
 *           differ from the key's d
 *  sel / n_sel: flat row ids token * h_q + head to compute (NULL = all rows,
 *           in flat order); out [n, dv] and lse [n] follow the selection order.
 *  nthreads: worker threads (>= 1).
 * Returns 0, or a negative code on an inconsistent page table.
 */
int oracle_verify_attn_dv(const uint16_t* q, const void* k_cache, const void* v_cache,
                          int kv_fp8, int kv_layout, const int32_t* kv_indptr,
                          const int32_t* kv_indices, const int32_t* last_page_len,
                          const int32_t* qo_indptr, const uint8_t* mask,
                          const int32_t* mask_indptr, int mask_layout, const int32_t* q_pos,
                          double rope_theta, double rope_scale, int q_fp8, int batch, int h_q,
                          int h_kv, int d, int dv, int page_size, int num_pages, double sm_scale,
                          double k_scale, double v_scale, const int32_t* sel, int64_t n_sel,
                          double* out, double* lse, int nthreads) {
    if (h_kv <= 0 || h_q <= 0 || h_q % h_kv != 0 || d <= 0 || dv <= 0 || nthreads < 1)
        return OR_EINVAL;
    if (q_fp8 && d > 1024) return OR_EINVAL;
    if ((kv_layout != 0 && kv_layout != 1) || (mask_layout != 0 && mask_layout != 1))
        return OR_EINVAL;
    if (q_pos && !(rope_theta > 0.0 && rope_scale > 0.0)) return OR_EINVAL;
    int rc = check_tables(kv_indptr, kv_indices, last_page_len, qo_indptr, batch, page_size,
                          num_pages);
    if (rc) return rc;
    if (mask) {
        if (!mask_indptr) return OR_EINVAL;
        for (int b = 0; b < batch; ++b) {
            int64_t L = qo_indptr[b + 1] - qo_indptr[b];
            int64_t cols = mask_layout == 1 ? oracle_kv_len(kv_indptr, last_page_len, b, page_size) : L;
            if ((int64_t)mask_indptr[b + 1] - mask_indptr[b] != L * cols) return OR_EINVAL;
        }
    }
    int64_t total_qo = qo_indptr[batch];
    int64_t n_all = total_qo * h_q;
    if (!sel) n_sel = n_all;
    for (int64_t i = 0; i < n_sel; ++i) {
        int64_t r = sel ? sel[i] : i;
        if (r < 0 || r >= n_all) return OR_EINVAL;
    }
    int group = h_q / h_kv;

    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_sel > 0 ? n_sel : 1));
    int64_t* dest = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_sel > 0 ? n_sel : 1));
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    job_t* jobs = (job_t*)malloc(sizeof(job_t) * (size_t)nthreads);
    if (!rows || !dest || !th || !jobs) {
        free(rows); free(dest); free(th); free(jobs);
        return OR_ENOMEM;
    }
    int status = OR_OK;
    for (int b = 0; b < batch && status == OR_OK; ++b) {
        int64_t qo0 = qo_indptr[b], qo1 = qo_indptr[b + 1];
        int64_t L = qo1 - qo0;
        /* this request's selected rows */
        int64_t nr = 0;
        for (int64_t i = 0; i < n_sel; ++i) {
            int64_t r = sel ? sel[i] : i;
            int64_t tok = r / h_q;
            if (tok >= qo0 && tok < qo1) {
                rows[nr] = r;
                dest[nr] = i;
                ++nr;
            }
        }
        if (nr == 0) continue;
        int64_t kv_len = oracle_kv_len(kv_indptr, last_page_len, b, page_size);
        size_t kv_rows = (size_t)(kv_len > 0 ? kv_len : 1) * (size_t)h_kv;
        double* K = (double*)malloc(sizeof(double) * kv_rows * (size_t)d);
        double* V = (double*)malloc(sizeof(double) * kv_rows * (size_t)dv);
        double* M = (double*)malloc(sizeof(double) * (size_t)(L * (kv_len > 0 ? kv_len : 1)));
        if (!K || !V || !M) {
            free(K); free(V); free(M);
            status = OR_ENOMEM;
            break;
        }
        gather_request(k_cache, v_cache, kv_fp8, kv_layout, kv_indptr, kv_indices, b, kv_len,
                       h_kv, d, dv, page_size, k_scale, v_scale, K, V);
        build_mask(mask, mask_indptr, mask_layout, b, L, kv_len, M);
        int nt = nthreads;
        if (nt > nr) nt = (int)nr;
        for (int i = 0; i < nt; ++i) {
            job_t* jb = &jobs[i];
            jb->q = q; jb->K = K; jb->V = V; jb->M = M;
            jb->kv_len = kv_len; jb->L = L; jb->qo_start = qo0;
            jb->h_q = h_q; jb->h_kv = h_kv; jb->d = d; jb->dv = dv; jb->group = group;
            jb->sm_scale = sm_scale; jb->rows = rows; jb->dest = dest; jb->n_rows = nr;
            jb->q_pos = q_pos; jb->rope_theta = rope_theta; jb->rope_scale = rope_scale;
            jb->q_fp8 = q_fp8;
            jb->out = out; jb->lse = lse;
            jb->lo = nr * i / nt; jb->hi = nr * (i + 1) / nt;
            jb->status = OR_OK;
        }
        for (int i = 1; i < nt; ++i) pthread_create(&th[i], NULL, run_rows, &jobs[i]);
        run_rows(&jobs[0]);
        for (int i = 1; i < nt; ++i) pthread_join(th[i], NULL);
        for (int i = 0; i < nt; ++i)
            if (jobs[i].status) status = jobs[i].status;
        free(K); free(V); free(M);
    }
    free(rows); free(dest); free(th); free(jobs);
    return status;
}

/* oracle_verify_attn_dv with values of the key's width (dv = d). */
int oracle_verify_attn_ex(const uint16_t* q, const void* k_cache, const void* v_cache,
                          int kv_fp8, int kv_layout, const int32_t* kv_indptr,
                          const int32_t* kv_indices, const int32_t* last_page_len,
                          const int32_t* qo_indptr, const uint8_t* mask,
                          const int32_t* mask_indptr, int mask_layout, const int32_t* q_pos,
                          double rope_theta, double rope_scale, int q_fp8, int batch, int h_q,
                          int h_kv, int d, int page_size, int num_pages, double sm_scale,
                          double k_scale, double v_scale, const int32_t* sel, int64_t n_sel,
                          double* out, double* lse, int nthreads) {
    return oracle_verify_attn_dv(q, k_cache, v_cache, kv_fp8, kv_layout, kv_indptr, kv_indices,
                                 last_page_len, qo_indptr, mask, mask_indptr, mask_layout, q_pos,
                                 rope_theta, rope_scale, q_fp8, batch, h_q, h_kv, d, d, page_size,
                                 num_pages, sm_scale, k_scale, v_scale, sel, n_sel, out, lse,
                                 nthreads);
}

/* oracle_verify_attn_ex for an HND cache, each request's L x L mask block and
 * no rotary embedding. */
int oracle_verify_attn(const uint16_t* q, const void* k_cache, const void* v_cache, int kv_fp8,
                       const int32_t* kv_indptr, const int32_t* kv_indices,
                       const int32_t* last_page_len, const int32_t* qo_indptr,
                       const uint8_t* mask, const int32_t* mask_indptr, int batch, int h_q,
                       int h_kv, int d, int page_size, int num_pages, double sm_scale,
                       double k_scale, double v_scale, const int32_t* sel, int64_t n_sel,
                       double* out, double* lse, int nthreads) {
    return oracle_verify_attn_ex(q, k_cache, v_cache, kv_fp8, 0, kv_indptr, kv_indices,
                                 last_page_len, qo_indptr, mask, mask_indptr, 0, NULL, 0.0, 0.0, 0,
                                 batch, h_q, h_kv, d, page_size, num_pages, sm_scale, k_scale,
                                 v_scale, sel, n_sel, out, lse, nthreads);
}

/*
 * Attention of one (request, query head, token) row restricted to the key
 * positions [lo, hi) of the request: the unnormalised pieces a split-KV
 * program produces ("flashmap ... verify_attention.py", the partial kernel's
 * per-split output: normalised partial out and its LSE).  Used to pin the
 * merge rule; masked positions follow the same explicit mask.
 */
int oracle_attn_range(const uint16_t* q, const void* k_cache, const void* v_cache, int kv_fp8,
                      const int32_t* kv_indptr, const int32_t* kv_indices,
                      const int32_t* last_page_len, const int32_t* qo_indptr,
                      const uint8_t* mask, const int32_t* mask_indptr, int batch, int h_q,
                      int h_kv, int d, int page_size, int num_pages, double sm_scale,
                      double k_scale, double v_scale, int b, int64_t t, int qh, int64_t lo,
                      int64_t hi, double* out, double* lse) {
    int rc = check_tables(kv_indptr, kv_indices, last_page_len, qo_indptr, batch, page_size,
                          num_pages);
    if (rc) return rc;
    if (b < 0 || b >= batch || qh < 0 || qh >= h_q || h_q % h_kv) return OR_EINVAL;
    int64_t L = qo_indptr[b + 1] - qo_indptr[b];
    int64_t kv_len = oracle_kv_len(kv_indptr, last_page_len, b, page_size);
    if (t < 0 || t >= L || lo < 0 || hi > kv_len || lo > hi) return OR_EINVAL;
    size_t kv_elems = (size_t)(kv_len > 0 ? kv_len : 1) * (size_t)h_kv * (size_t)d;
    double* K = (double*)malloc(sizeof(double) * kv_elems);
    double* V = (double*)malloc(sizeof(double) * kv_elems);
    double* M = (double*)malloc(sizeof(double) * (size_t)(L * (kv_len > 0 ? kv_len : 1)));
    double* s = (double*)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
    double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
    if (!K || !V || !M || !s || !qrow) {
        free(K); free(V); free(M); free(s); free(qrow);
        return OR_ENOMEM;
    }
    gather_request(k_cache, v_cache, kv_fp8, 0, kv_indptr, kv_indices, b, kv_len, h_kv, d, d,
                   page_size, k_scale, v_scale, K, V);
    build_mask(mask, mask_indptr, 0, b, L, kv_len, M);
    int64_t tok = qo_indptr[b] + t;
    for (int e = 0; e < d; ++e) qrow[e] = oracle_decode_bf16(q[(tok * h_q + qh) * d + e]);
    int h = qh / (h_q / h_kv);
    oracle_dense_attention(1, (int)(hi - lo), d, qrow, d, K + (lo * h_kv + h) * d,
                           V + (lo * h_kv + h) * d, (int64_t)h_kv * d, M + t * kv_len + lo,
                           sm_scale, out, lse, s);
    free(K); free(V); free(M); free(s); free(qrow);
    return OR_OK;
}

/*
 * Merge of n_parts partial results of the same rows by their log-sum-exp
 * ("flashmap ... verify_attention.py", the merge kernel): with m = max lse_s,
 * out = sum_s e^(lse_s - m) out_s / sum_s e^(lse_s - m) and
 * lse = m + ln sum_s e^(lse_s - m); parts with lse = -inf carry no mass; if
 * every part is empty, out = 0 and lse = -inf.
 * outs [n_parts][n_rows][d], lses [n_parts][n_rows].
 */
void oracle_merge_partials(int n_parts, int n_rows, int d, const double* outs,
                           const double* lses, double* out, double* lse) {
    for (int r = 0; r < n_rows; ++r) {
        double m = -INFINITY;
        for (int s = 0; s < n_parts; ++s) {
            double l = lses[(int64_t)s * n_rows + r];
            if (l > m) m = l;
        }
        double* o = out + (int64_t)r * d;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double den = 0.0;
        for (int s = 0; s < n_parts; ++s) {
            double l = lses[(int64_t)s * n_rows + r];
            if (l == -INFINITY) continue;
            double w = exp(l - m);
            den += w;
            const double* os = outs + ((int64_t)s * n_rows + r) * d;
            for (int e = 0; e < d; ++e) o[e] += w * os[e];
        }
        for (int e = 0; e < d; ++e) o[e] /= den;
        lse[r] = m + log(den);
    }
}

/*
 * Host scatter of new tokens into the paged cache (the "append first" step:
 * vLLM PR #1679 caches every draft's keys and values before attention).
 * For request b and new token i < n_b = append_indptr[b+1] - append_indptr[b],
 * the position is pos = kv_len_b - n_b + i; its row is slot pos % page_size
 * of page kv_indices[kv_indptr[b] + pos / page_size].  The bytes of
 * k_new[append_indptr[b] + i, h, :] are copied unchanged (elem_bytes per
 * element) to k_cache[page, h, slot, :]; likewise for V.
 */
/*
 * Quantising append: the walk of oracle_paged_kv_append, with bf16 new rows
 * and an fp8-e4m3 cache; element x of a K row is stored as
 * oracle_encode_e4m3_satfinite(oracle_div_f32(x, k_scale)) (likewise V with
 * v_scale): the per-tensor scale of FlashInfer PR #286's fp8 cache
 * (dequantised value = stored * scale), rounded to nearest even, saturated.
 */
int oracle_paged_kv_append_quant(const uint16_t* k_new, const uint16_t* v_new, float k_scale,
                                 float v_scale, const int32_t* append_indptr,
                                 const int32_t* kv_indptr, const int32_t* kv_indices,
                                 const int32_t* last_page_len, int batch, int h_kv, int d,
                                 int page_size, int num_pages, uint8_t* k_cache,
                                 uint8_t* v_cache) {
    if (batch < 0 || h_kv <= 0 || d <= 0 || page_size <= 0) return OR_EINVAL;
    if (!(k_scale > 0.0f) || !(v_scale > 0.0f)) return OR_EINVAL;
    for (int b = 0; b < batch; ++b) {
        int64_t n = (int64_t)append_indptr[b + 1] - append_indptr[b];
        int64_t kv_len = oracle_kv_len(kv_indptr, last_page_len, b, page_size);
        if (n < 0 || n > kv_len) return OR_EINVAL;
        for (int64_t i = 0; i < n; ++i) {
            int64_t pos = kv_len - n + i;
            int64_t pidx = (int64_t)kv_indptr[b] + pos / page_size;
            if (pidx >= kv_indptr[b + 1]) return OR_EINVAL;
            int32_t page = kv_indices[pidx];
            if (page < 0 || page >= num_pages) return OR_EINVAL;
            int64_t slot = pos % page_size;
            int64_t tok = (int64_t)append_indptr[b] + i;
            for (int h = 0; h < h_kv; ++h) {
                size_t dst = (((size_t)page * h_kv + h) * page_size + slot) * (size_t)d;
                size_t src = ((size_t)tok * h_kv + h) * (size_t)d;
                for (int e = 0; e < d; ++e) {
                    float xk = (float)oracle_decode_bf16(k_new[src + e]);
                    float xv = (float)oracle_decode_bf16(v_new[src + e]);
                    k_cache[dst + e] = oracle_encode_e4m3_satfinite(oracle_div_f32(xk, k_scale));
                    v_cache[dst + e] = oracle_encode_e4m3_satfinite(oracle_div_f32(xv, v_scale));
                }
            }
        }
    }
    return OR_OK;
}

/*
 * The append with options, as the library's extended append defines it:
 *  - layout 0 / 1: HND or NHD destination rows (cache_row);
 *  - quantize: bf16 new rows into an fp8-e4m3 cache; without positions each
 *    element is stored exactly as oracle_paged_kv_append_quant stores it;
 *  - positions (nullable, [total_new]): each new K row is first rotated by
 *    oracle_rope_vec at its token's position, in fp64, then rounded once to
 *    the cache dtype: bf16 to nearest even, or e4m3 to nearest even with
 *    saturation (after the division by k_scale when quantizing; an fp8 row
 *    copied without quantizing is rotated in its stored units).  V rows are
 *    never rotated.
 * Without quantize or positions this is oracle_paged_kv_append's bit copy.
 * V rows (new and cached) hold dv elements, K rows d.
 */
int oracle_paged_kv_append_dv(const void* k_new, const void* v_new, int cache_fp8, int quantize,
                              float k_scale, float v_scale, int layout, const int32_t* positions,
                              double theta, double rope_scale, const int32_t* append_indptr,
                              const int32_t* kv_indptr, const int32_t* kv_indices,
                              const int32_t* last_page_len, int batch, int h_kv, int d, int dv,
                              int page_size, int num_pages, void* k_cache, void* v_cache) {
    if (batch < 0 || h_kv <= 0 || d <= 0 || dv <= 0 || page_size <= 0) return OR_EINVAL;
    if (layout != 0 && layout != 1) return OR_EINVAL;
    if (quantize && (!cache_fp8 || !(k_scale > 0.0f) || !(v_scale > 0.0f))) return OR_EINVAL;
    if (positions && !(theta > 0.0 && rope_scale > 0.0)) return OR_EINVAL;
    const int src_bf16 = quantize || !cache_fp8;
    double* row = (double*)malloc(sizeof(double) * (size_t)d);
    if (!row) return OR_ENOMEM;
    for (int b = 0; b < batch; ++b) {
        int64_t n = (int64_t)append_indptr[b + 1] - append_indptr[b];
        int64_t kv_len = oracle_kv_len(kv_indptr, last_page_len, b, page_size);
        if (n < 0 || n > kv_len) { free(row); return OR_EINVAL; }
        for (int64_t i = 0; i < n; ++i) {
            int64_t pos = kv_len - n + i;
            int64_t pidx = (int64_t)kv_indptr[b] + pos / page_size;
            if (pidx >= kv_indptr[b + 1]) { free(row); return OR_EINVAL; }
            int32_t page = kv_indices[pidx];
            if (page < 0 || page >= num_pages) { free(row); return OR_EINVAL; }
            int64_t slot = pos % page_size;
            int64_t tok = (int64_t)append_indptr[b] + i;
            for (int h = 0; h < h_kv; ++h) {
                size_t crow = (size_t)cache_row(layout, page, h, slot, h_kv, page_size);
                for (int kv = 0; kv < 2; ++kv) {
                    const int w = kv ? dv : d;  /* elements of this row */
                    size_t dst = crow * (size_t)w;
                    size_t src = ((size_t)tok * h_kv + h) * (size_t)w;
                    const void* in = kv ? v_new : k_new;
                    void* cache = kv ? v_cache : k_cache;
                    const float scale = kv ? v_scale : k_scale;
                    const int rotate = positions && kv == 0;
                    if (!rotate) {
                        for (int e = 0; e < w; ++e) {
                            if (quantize) {
                                float x = (float)oracle_decode_bf16(((const uint16_t*)in)[src + e]);
                                ((uint8_t*)cache)[dst + e] =
                                    oracle_encode_e4m3_satfinite(oracle_div_f32(x, scale));
                            } else if (cache_fp8) {
                                ((uint8_t*)cache)[dst + e] = ((const uint8_t*)in)[src + e];
                            } else {
                                ((uint16_t*)cache)[dst + e] = ((const uint16_t*)in)[src + e];
                            }
                        }
                        continue;
                    }
                    for (int e = 0; e < d; ++e)
                        row[e] = src_bf16 ? oracle_decode_bf16(((const uint16_t*)in)[src + e])
                                          : oracle_decode_e4m3(((const uint8_t*)in)[src + e]);
                    oracle_rope_vec(row, d, (double)positions[tok], theta, rope_scale);
                    for (int e = 0; e < d; ++e) {
                        if (!cache_fp8)
                            ((uint16_t*)cache)[dst + e] = oracle_encode_bf16(row[e]);
                        else
                            ((uint8_t*)cache)[dst + e] =
                                encode_e4m3_value(quantize ? row[e] / (double)scale : row[e]);
                    }
                }
            }
        }
    }
    free(row);
    return OR_OK;
}

/* oracle_paged_kv_append_dv with value rows of the key's width (dv = d). */
int oracle_paged_kv_append_ex(const void* k_new, const void* v_new, int cache_fp8, int quantize,
                              float k_scale, float v_scale, int layout, const int32_t* positions,
                              double theta, double rope_scale, const int32_t* append_indptr,
                              const int32_t* kv_indptr, const int32_t* kv_indices,
                              const int32_t* last_page_len, int batch, int h_kv, int d,
                              int page_size, int num_pages, void* k_cache, void* v_cache) {
    return oracle_paged_kv_append_dv(k_new, v_new, cache_fp8, quantize, k_scale, v_scale, layout,
                                     positions, theta, rope_scale, append_indptr, kv_indptr,
                                     kv_indices, last_page_len, batch, h_kv, d, d, page_size,
                                     num_pages, k_cache, v_cache);
}

int oracle_paged_kv_append(const void* k_new, const void* v_new, int elem_bytes,
                           const int32_t* append_indptr, const int32_t* kv_indptr,
                           const int32_t* kv_indices, const int32_t* last_page_len, int batch,
                           int h_kv, int d, int page_size, int num_pages, void* k_cache,
                           void* v_cache) {
    if (batch < 0 || h_kv <= 0 || d <= 0 || page_size <= 0 || elem_bytes <= 0) return OR_EINVAL;
    size_t row = (size_t)d * (size_t)elem_bytes;
    for (int b = 0; b < batch; ++b) {
        int64_t n = (int64_t)append_indptr[b + 1] - append_indptr[b];
        int64_t kv_len = oracle_kv_len(kv_indptr, last_page_len, b, page_size);
        if (n < 0 || n > kv_len) return OR_EINVAL;
        for (int64_t i = 0; i < n; ++i) {
            int64_t pos = kv_len - n + i;
            int64_t pidx = (int64_t)kv_indptr[b] + pos / page_size;
            if (pidx >= kv_indptr[b + 1]) return OR_EINVAL;
            int32_t page = kv_indices[pidx];
            if (page < 0 || page >= num_pages) return OR_EINVAL;
            int64_t slot = pos % page_size;
            int64_t tok = (int64_t)append_indptr[b] + i;
            for (int h = 0; h < h_kv; ++h) {
                size_t dst = ((((size_t)page * h_kv + h) * page_size + slot)) * row;
                size_t src = ((size_t)tok * h_kv + h) * row;
                memcpy((char*)k_cache + dst, (const char*)k_new + src, row);
                memcpy((char*)v_cache + dst, (const char*)v_new + src, row);
            }
        }
    }
    return OR_OK;
}
