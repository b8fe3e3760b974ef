/*
 * oracle.c -- plain, slow, float64 CPU restatement of extend attention over a
 * page-size-1 KV pool, decode attention, merge_state, the unified KV-index
 * build, the KV-index gather from the request-to-token table and the KV
 * write into the pool, for bf16 pools and for fp8 (e4m3 / e5m2) pools with
 * per-tensor k_scale / v_scale, and the expansion of paged KV indices (page
 * size > 1) into per-token pool slots.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file.  It exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark have an obviously correct answer to compare
 * the CUDA kernels against.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * Sources (the web pages this method is taken from):
 *   [EXT]  sglang extend_attention.py (diff 0.5.3rc2 -> 0.5.4.post1):
 *          _fwd_kernel_unified, extend_attention_fwd_unified,
 *          extend_attention_fwd, redundant_attention,
 *          _copy_unified_indices_kernel, build_unified_kv_indices.
 *   [FI]   sglang flashinfer_backend.py: forward_extend (ragged + paged +
 *          merge_state split), forward_decode, the sliding-window index
 *          updaters, create_flashinfer_kv_indices_triton, set_kv_buffer.
 *   [CPU]  sglang cpu_graph_runner.py: the MLA K/V layout (V is the first
 *          kv_lora_rank dims of K) in the qkv_proj_with_rope fake.
 *
 * Every floating-point step runs in double on the exact bf16 input values.
 * Loops are in the order sequence -> head -> query -> key, with no tiling,
 * no online softmax and no reordering beyond the definition:
 *
 *   s_j   = sm_scale * sum_d q[d] * k_j[d]                ([EXT] QK, scale)
 *   s_j   = cap * tanh(s_j / cap)           if cap > 0     ([EXT] logit cap)
 *   vis_j = (j <= qpos) && (W <= 0 || qpos - j <= W)       ([EXT] causal
 *           mask on the extend part; sliding-window mask)
 *   m     = max_{vis} s_j ;  l = sum_{vis} exp(s_j - m)
 *   o     = sum_{vis} exp(s_j - m) v_j / l ;  lse = m + log(l)
 *
 * where a sequence's keys are its P prefix keys followed by its E extend keys,
 * and extend query i sits at position qpos = P + i.
 *
 * Optional, as in [EXT] _fwd_kernel_unified:
 *   custom mask: a byte per (extend row i, key j) of sequence b at
 *     custom_mask[mask_indptr[b] + i * T_b + j]; when given it replaces the
 *     causal term, the window still applies ([EXT] "Apply custom mask",
 *     "IS_CAUSAL and not USE_CUSTOM_MASK");
 *   sink: a logit per query head that adds exp(sink - m) to the softmax
 *     denominator and nothing to o ([EXT] "Handle sink tokens"):
 *       l = sum_{vis} exp(s_j - m) + exp(sink - m), lse = m + log(l)
 *     (m is any reference point; here the max over the visible s_j and
 *     the sink).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double (bf16 is the top half of an IEEE float). */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * fp8 codes of the pool ([FI] kv_cache_dtype float8_e4m3fn / float8_e5m2,
 * with k_scale / v_scale): the value of a code, from the formats'
 * definitions.
 *   e4m3fn: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
 *           subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities.
 *   e5m2:   sign, 5 exponent bits (bias 15), 2 mantissa bits; exponent 0 is
 *           subnormal (m/4 * 2^-14); exponent 31 is inf (m = 0) or NaN.
 */
enum { KV_BF16 = 0, KV_E4M3 = 1, KV_E5M2 = 2 };

double oracle_fp8_value(uint8_t code, int fmt)
{
    int sign = code >> 7;
    int e, m;
    double v;
    if (fmt == KV_E4M3) {
        e = (code >> 3) & 15;
        m = code & 7;
        if (e == 15 && m == 7)
            return NAN;
        v = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    } else {
        e = (code >> 2) & 31;
        m = code & 3;
        if (e == 31)
            return m == 0 ? (sign ? -INFINITY : INFINITY) : NAN;
        v = e == 0 ? ldexp(m / 4.0, -14) : ldexp(1.0 + m / 4.0, e - 15);
    }
    return sign ? -v : v;
}

/*
 * The code of an fp32 value: the nearest finite code, ties to the code
 * with an even mantissa (round to nearest even), values past the largest
 * finite magnitude saturate to it (448 for e4m3, 57344 for e5m2).  The sign
 * is kept, so a negative value that rounds to zero gives -0.  Written as a
 * search over the 128 non-negative codes.
 */
uint8_t oracle_fp8_code(float x, int fmt)
{
    int neg = signbit(x) != 0;
    double a = fabs((double)x);
    int best = 0;
    double best_d = INFINITY;
    /* past the largest finite code: that code (the distances below would
     * lose their precision there) */
    int top = fmt == KV_E4M3 ? 0x7e : 0x7b;
    if (a >= oracle_fp8_value((uint8_t)top, fmt))
        return (uint8_t)(top | (neg ? 0x80 : 0));
    for (int c = 0; c < 128; ++c) {
        double v = oracle_fp8_value((uint8_t)c, fmt);
        if (isnan(v) || isinf(v))
            continue;
        double d = fabs(v - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(best | (neg ? 0x80 : 0));
}

/* One key or value row: bf16 elements, or fp8 codes times the row's scale. */
typedef struct {
    const void *p;
    int fmt;
    double scale;
} kv_row;

static double row_elem(kv_row r, int d)
{
    if (r.fmt == KV_BF16)
        return bf16_to_double(((const uint16_t *)r.p)[d]);
    return oracle_fp8_value(((const uint8_t *)r.p)[d], r.fmt) * r.scale;
}

/* Row (slot, h) of a pool whose element size follows its format. */
static kv_row pool_row(const void *buf, int fmt, double scale, long slot,
                       long ss, long hs, int hk)
{
    kv_row r;
    long off = slot * ss + (long)hk * hs;
    r.p = fmt == KV_BF16 ? (const void *)((const uint16_t *)buf + off)
                         : (const void *)((const uint8_t *)buf + off);
    r.fmt = fmt;
    r.scale = scale;
    return r;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Attention of one query row over one sequence's key list.
 *   krow[j], vrow[j]: the j-th key / value row of the sequence (position j).
 *   qpos: the query's position in the sequence.  window <= 0: no window.
 *   s: scratch of n_keys doubles.
 * Writes o[0..lv) and *lse.  A query that sees no key (cannot happen for a
 * valid extend or decode query, which always sees itself) gets o = 0 and
 * lse = -inf.
 */
static void attend_one_query(const uint16_t *q, int lq, int lv, long n_keys,
                             const kv_row *krow, const kv_row *vrow, long qpos,
                             long window, double sm_scale, double logit_cap,
                             const uint8_t *mask_row, const double *sink,
                             double *s, double *o, double *lse)
{
    double m = -INFINITY;
    for (long j = 0; j < n_keys; ++j) {
        int visible = (j <= qpos) && (window <= 0 || qpos - j <= window);
        if (mask_row)
            visible = (mask_row[j] != 0) && (window <= 0 || qpos - j <= window);
        if (!visible) {
            s[j] = -INFINITY;
            continue;
        }
        double dot = 0.0;
        for (int d = 0; d < lq; ++d)
            dot += bf16_to_double(q[d]) * row_elem(krow[j], d);
        double sj = sm_scale * dot;
        if (logit_cap > 0.0)
            sj = logit_cap * tanh(sj / logit_cap);
        s[j] = sj;
        if (sj > m)
            m = sj;
    }
    if (sink && *sink > m)
        m = *sink;
    for (int d = 0; d < lv; ++d)
        o[d] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (long j = 0; j < n_keys; ++j) {
        if (s[j] == -INFINITY)
            continue;
        double p = exp(s[j] - m);
        l += p;
        for (int d = 0; d < lv; ++d)
            o[d] += p * row_elem(vrow[j], d);
    }
    if (sink)
        l += exp(*sink - m);
    for (int d = 0; d < lv; ++d)
        o[d] /= l;
    *lse = m + log(l);
}

/* Index b of the sequence whose extend rows [qo_indptr[b], qo_indptr[b+1])
 * contain token t, or -1. */
static int sequence_of_token(const int32_t *qo_indptr, int batch, long t)
{
    for (int b = 0; b < batch; ++b)
        if (t >= qo_indptr[b] && t < qo_indptr[b + 1])
            return b;
    return -1;
}

/*
 * Extend attention, two-stage form ([EXT] extend_attention_fwd and its
 * _fwd_kernel): prefix K/V come from the pool through
 * kv_indices[kv_indptr[b] .. kv_indptr[b+1]), extend K/V are the contiguous
 * rows k_extend/v_extend[qo_indptr[b] .. qo_indptr[b+1]).
 *
 * Layouts (element strides; the last dim is contiguous):
 *   q_extend [n_tokens, hq, lq] contiguous
 *   k_extend row (t, h) at k_ext + t*k_ext_ts + h*k_ext_hs  (lq elements)
 *   v_extend row (t, h) at v_ext + t*v_ext_ts + h*v_ext_hs  (lv elements)
 *   k_buffer row (slot, h) at k_buf + slot*k_buf_ss + h*k_buf_hs
 *   v_buffer row (slot, h) at v_buf + slot*v_buf_ss + h*v_buf_hs
 * kv_fmt: the pool's element format (KV_BF16, or fp8 KV_E4M3 / KV_E5M2 whose
 *   keys read code * k_scale and values code * v_scale; [FI] forward with
 *   k_scale / v_scale); k_extend / v_extend are always bf16.
 * rows: NULL -> every (token, head) and o_out is [n_tokens, hq, lv],
 *       lse_out [n_tokens, hq];
 *       else rows[r] = token*hq + head for r < n_rows, and o_out is
 *       [n_rows, lv], lse_out [n_rows].
 * Returns 0, or -1 on an argument error.
 */
int oracle_extend_attention(
    const uint16_t *q_extend, const uint16_t *k_ext, long k_ext_ts,
    long k_ext_hs, const uint16_t *v_ext, long v_ext_ts, long v_ext_hs,
    const void *k_buf, long k_buf_ss, long k_buf_hs, const void *v_buf,
    long v_buf_ss, long v_buf_hs, int kv_fmt, double k_scale, double v_scale,
    const int32_t *qo_indptr,
    const int32_t *kv_indptr, const int32_t *kv_indices, int batch, int hq,
    int hkv, int lq, int lv, double sm_scale, double logit_cap,
    long sliding_window, const uint8_t *custom_mask, const int32_t *mask_indptr,
    const double *sinks, const int64_t *rows, long n_rows, double *o_out,
    double *lse_out)
{
    if (batch < 0 || hkv <= 0 || hq % hkv != 0 || (custom_mask && !mask_indptr))
        return -1;
    int group = hq / hkv; /* [EXT] kv_group_num: q heads per kv head */
    long n_tokens = batch > 0 ? qo_indptr[batch] : 0;
    long total = rows ? n_rows : n_tokens * hq;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 4) reduction(| : bad)
    for (long r = 0; r < total; ++r) {
        long row = rows ? rows[r] : r;
        long t = row / hq;
        int h = (int)(row % hq);
        int b = sequence_of_token(qo_indptr, batch, t);
        if (b < 0) {
            bad = 1;
            continue;
        }
        int hk = h / group;
        long p_len = kv_indptr[b + 1] - kv_indptr[b];
        long e_len = qo_indptr[b + 1] - qo_indptr[b];
        long n_keys = p_len + e_len;
        kv_row *krow = malloc(sizeof(*krow) * (size_t)(n_keys + 1));
        kv_row *vrow = malloc(sizeof(*vrow) * (size_t)(n_keys + 1));
        double *s = malloc(sizeof(double) * (size_t)(n_keys + 1));
        /* Key j of sequence b: prefix keys through the page table, then the
         * sequence's own extend tokens. */
        for (long j = 0; j < p_len; ++j) {
            long slot = kv_indices[kv_indptr[b] + j];
            krow[j] = pool_row(k_buf, kv_fmt, k_scale, slot, k_buf_ss, k_buf_hs, hk);
            vrow[j] = pool_row(v_buf, kv_fmt, v_scale, slot, v_buf_ss, v_buf_hs, hk);
        }
        for (long e = 0; e < e_len; ++e) {
            long te = qo_indptr[b] + e;
            krow[p_len + e] = pool_row(k_ext, KV_BF16, 1.0, te, k_ext_ts, k_ext_hs, hk);
            vrow[p_len + e] = pool_row(v_ext, KV_BF16, 1.0, te, v_ext_ts, v_ext_hs, hk);
        }
        long i = t - qo_indptr[b];
        const uint8_t *mask_row =
            custom_mask ? custom_mask + mask_indptr[b] + i * n_keys : NULL;
        attend_one_query(q_extend + (t * hq + h) * (long)lq, lq, lv, n_keys,
                         krow, vrow, p_len + i, sliding_window, sm_scale,
                         logit_cap, mask_row, sinks ? sinks + h : NULL, s,
                         o_out + r * (long)lv, lse_out + r);
        free(krow);
        free(vrow);
        free(s);
    }
    return bad ? -1 : 0;
}

/*
 * Extend attention, unified form ([EXT] extend_attention_fwd_unified and
 * _fwd_kernel_unified): every key of sequence b, prefix and extend alike, is
 * pool slot kv_indices[kv_indptr[b] + j]; the first prefix_lens[b] of them are
 * the prefix.  Extend query i sits at position prefix_lens[b] + i.  The window
 * start position is 0 for every sequence (the launcher's default).
 * q [n_tokens, hq, lq] contiguous; rows / outputs as in
 * oracle_extend_attention.
 */
int oracle_extend_attention_unified(
    const uint16_t *q, const void *k_buf, long k_buf_ss, long k_buf_hs,
    const void *v_buf, long v_buf_ss, long v_buf_hs, int kv_fmt,
    double k_scale, double v_scale, const int32_t *qo_indptr,
    const int32_t *kv_indptr, const int64_t *kv_indices, const int32_t *prefix_lens, int batch, int hq,
    int hkv, int lq, int lv, double sm_scale, double logit_cap,
    long sliding_window, const uint8_t *custom_mask, const int32_t *mask_indptr,
    const double *sinks, const int64_t *rows, long n_rows, double *o_out,
    double *lse_out)
{
    if (batch < 0 || hkv <= 0 || hq % hkv != 0 || (custom_mask && !mask_indptr))
        return -1;
    int group = hq / hkv;
    long n_tokens = batch > 0 ? qo_indptr[batch] : 0;
    long total = rows ? n_rows : n_tokens * hq;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 4) reduction(| : bad)
    for (long r = 0; r < total; ++r) {
        long row = rows ? rows[r] : r;
        long t = row / hq;
        int h = (int)(row % hq);
        int b = sequence_of_token(qo_indptr, batch, t);
        if (b < 0) {
            bad = 1;
            continue;
        }
        int hk = h / group;
        long n_keys = kv_indptr[b + 1] - kv_indptr[b];
        kv_row *krow = malloc(sizeof(*krow) * (size_t)(n_keys + 1));
        kv_row *vrow = malloc(sizeof(*vrow) * (size_t)(n_keys + 1));
        double *s = malloc(sizeof(double) * (size_t)(n_keys + 1));
        for (long j = 0; j < n_keys; ++j) {
            long slot = (long)kv_indices[kv_indptr[b] + j];
            krow[j] = pool_row(k_buf, kv_fmt, k_scale, slot, k_buf_ss, k_buf_hs, hk);
            vrow[j] = pool_row(v_buf, kv_fmt, v_scale, slot, v_buf_ss, v_buf_hs, hk);
        }
        long i = t - qo_indptr[b];
        const uint8_t *mask_row =
            custom_mask ? custom_mask + mask_indptr[b] + i * n_keys : NULL;
        attend_one_query(q + (t * hq + h) * (long)lq, lq, lv, n_keys, krow,
                         vrow, (long)prefix_lens[b] + i, sliding_window,
                         sm_scale, logit_cap, mask_row, sinks ? sinks + h : NULL,
                         s, o_out + r * (long)lv, lse_out + r);
        free(krow);
        free(vrow);
        free(s);
    }
    return bad ? -1 : 0;
}

/*
 * Decode attention ([FI] forward_decode): one query per sequence; the
 * sequence's K/V, the current token's included, are all in the pool at
 * kv_indices[kv_indptr[b] .. kv_indptr[b+1]).  The query sits at the last
 * position T_b - 1, so with a window W > 0 it sees the last W + 1 keys ([FI]
 * sliding-window decode updater keeps min(seq_len, W + 1) keys).
 * q [batch, hq, lq] contiguous; o_out [batch, hq, lv]; lse_out [batch, hq].
 * A sequence with T_b = 0 gets o = 0, lse = -inf.
 */
int oracle_decode_attention(const uint16_t *q, const void *k_buf,
                            long k_buf_ss, long k_buf_hs, const void *v_buf,
                            long v_buf_ss, long v_buf_hs, int kv_fmt,
                            double k_scale, double v_scale,
                            const int32_t *kv_indptr, const int32_t *kv_indices,
                            int batch, int hq, int hkv, int lq, int lv,
                            double sm_scale, double logit_cap,
                            long sliding_window, double *o_out,
                            double *lse_out)
{
    if (batch < 0 || hkv <= 0 || hq % hkv != 0)
        return -1;
    int group = hq / hkv;
    long total = (long)batch * hq;

#pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < total; ++r) {
        int b = (int)(r / hq);
        int h = (int)(r % hq);
        int hk = h / group;
        long n_keys = kv_indptr[b + 1] - kv_indptr[b];
        kv_row *krow = malloc(sizeof(*krow) * (size_t)(n_keys + 1));
        kv_row *vrow = malloc(sizeof(*vrow) * (size_t)(n_keys + 1));
        double *s = malloc(sizeof(double) * (size_t)(n_keys + 1));
        for (long j = 0; j < n_keys; ++j) {
            long slot = kv_indices[kv_indptr[b] + j];
            krow[j] = pool_row(k_buf, kv_fmt, k_scale, slot, k_buf_ss, k_buf_hs, hk);
            vrow[j] = pool_row(v_buf, kv_fmt, v_scale, slot, v_buf_ss, v_buf_hs, hk);
        }
        attend_one_query(q + r * (long)lq, lq, lv, n_keys, krow, vrow,
                         n_keys - 1, sliding_window, sm_scale, logit_cap, NULL,
                         NULL, s, o_out + r * (long)lv, lse_out + r);
        free(krow);
        free(vrow);
        free(s);
    }
    return 0;
}

/*
 * merge_state ([FI] forward_extend, ragged + paged split): two partial
 * attention states (v_a, s_a) and (v_b, s_b) of the same queries over
 * disjoint key sets, with s the natural-log sum of exp of the scaled (and
 * capped) logits, combine into the state over the union:
 *   s = log(exp(s_a) + exp(s_b))
 *   v = exp(s_a - s) * v_a + exp(s_b - s) * v_b
 * A side with s = -inf holds no key and has weight 0; both -inf gives v = 0,
 * s = -inf.
 * v_* [n, h, dv] bf16; s_* [n, h] fp32; outputs double.
 */
void oracle_merge_state(const uint16_t *v_a, const float *s_a,
                        const uint16_t *v_b, const float *s_b, long n, int h,
                        int dv, double *v_out, double *s_out)
{
    long total = n * (long)h;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < total; ++r) {
        double sa = s_a[r], sb = s_b[r];
        if (sa == -INFINITY && sb == -INFINITY) {
            for (int d = 0; d < dv; ++d)
                v_out[r * dv + d] = 0.0;
            s_out[r] = -INFINITY;
            continue;
        }
        double m = sa > sb ? sa : sb;
        double s = m + log(exp(sa - m) + exp(sb - m));
        double wa = exp(sa - s), wb = exp(sb - s);
        for (int d = 0; d < dv; ++d)
            v_out[r * dv + d] = wa * bf16_to_double(v_a[r * dv + d]) +
                                wb * bf16_to_double(v_b[r * dv + d]);
        s_out[r] = s;
    }
}

/*
 * Unified KV-index build ([EXT] build_unified_kv_indices and
 * _copy_unified_indices_kernel):
 *   prefix_lens[b]            = prefix_kv_indptr[b+1] - prefix_kv_indptr[b]
 *   unified_kv_indptr[0]      = 0
 *   unified_kv_indptr[b+1]    = unified_kv_indptr[b] + prefix_lens[b]
 *                               + extend_seq_lens[b]
 *   unified_kv_indices[unified_kv_indptr[b] + j]
 *       = prefix_kv_indices[prefix_kv_indptr[b] + j]           j < P_b
 *       = extend_kv_indices[extend_start_loc[b] + j - P_b]     P_b <= j < T_b
 * Entries of unified_kv_indices past unified_kv_indptr[bs] are not written.
 */
void oracle_build_unified_kv_indices(
    const int32_t *prefix_kv_indptr, const int32_t *prefix_kv_indices,
    const int32_t *extend_start_loc, const int32_t *extend_seq_lens,
    const int32_t *extend_kv_indices, int bs, int32_t *unified_kv_indptr,
    int64_t *unified_kv_indices, int32_t *prefix_lens)
{
    unified_kv_indptr[0] = 0;
    for (int b = 0; b < bs; ++b) {
        prefix_lens[b] = prefix_kv_indptr[b + 1] - prefix_kv_indptr[b];
        unified_kv_indptr[b + 1] =
            unified_kv_indptr[b] + prefix_lens[b] + extend_seq_lens[b];
    }
    for (int b = 0; b < bs; ++b) {
        long dst = unified_kv_indptr[b];
        for (long j = 0; j < prefix_lens[b]; ++j)
            unified_kv_indices[dst + j] =
                prefix_kv_indices[prefix_kv_indptr[b] + j];
        for (long e = 0; e < extend_seq_lens[b]; ++e)
            unified_kv_indices[dst + prefix_lens[b] + e] =
                extend_kv_indices[extend_start_loc[b] + e];
    }
}

/*
 * KV-index gather from the request-to-token table ([FI]
 * create_flashinfer_kv_indices_triton, with the indptr its callers build in
 * the decode and prefill index updaters):
 *   kv_indptr[0]   = 0
 *   kv_indptr[b+1] = kv_indptr[b] + paged_kernel_lens[b]
 *   kv_indices[kv_indptr[b] + j]
 *       = req_to_token[req_pool_indices[b] * stride + kv_start[b] + j]
 *   for j < paged_kernel_lens[b], with kv_start[b] = kv_start_idx[b], or 0
 *   when kv_start_idx is NULL.  Lengths and starts are taken as 32-bit, as the
 *   gather does.  Entries past kv_indptr[bs] are not written.
 */
void oracle_create_kv_indices(
    const int32_t *req_to_token, long stride, const int64_t *req_pool_indices,
    const int64_t *paged_kernel_lens, const int64_t *kv_start_idx, int bs,
    int32_t *kv_indptr, int32_t *kv_indices)
{
    kv_indptr[0] = 0;
    for (int b = 0; b < bs; ++b)
        kv_indptr[b + 1] = kv_indptr[b] + (int32_t)paged_kernel_lens[b];
    for (int b = 0; b < bs; ++b) {
        long row = (long)req_pool_indices[b] * stride;
        long start = kv_start_idx ? (long)(int32_t)kv_start_idx[b] : 0;
        for (long j = 0; j < (long)(int32_t)paged_kernel_lens[b]; ++j)
            kv_indices[kv_indptr[b] + j] = req_to_token[row + start + j];
    }
}

/*
 * KV write into the pool ([FI] forward_extend / forward_decode,
 * token_to_kv_pool.set_kv_buffer(layer, cache_loc, k, v, ...)): token t's
 * rows go to pool slot cache_loc[t], every KV head:
 *   k_buf[cache_loc[t], h, :lk] = k[t, h, :lk]
 *   v_buf[cache_loc[t], h, :lv] = v[t, h, :lv]     (skipped when v is NULL:
 *                                                    the MLA pool holds K only)
 * The pool is bf16 like the inputs, so the write is a copy of the bit
 * patterns.  Slots not named in cache_loc keep their contents.
 */
void oracle_set_kv_buffer(
    const uint16_t *k, long k_ts, long k_hs, const uint16_t *v, long v_ts,
    long v_hs, const int64_t *cache_loc, long n_tokens, int hkv, int lk,
    int lv, uint16_t *k_buf, long k_buf_ss, long k_buf_hs, uint16_t *v_buf,
    long v_buf_ss, long v_buf_hs)
{
    for (long t = 0; t < n_tokens; ++t) {
        long slot = (long)cache_loc[t];
        for (int h = 0; h < hkv; ++h) {
            for (int d = 0; d < lk; ++d)
                k_buf[slot * k_buf_ss + (long)h * k_buf_hs + d] =
                    k[t * k_ts + (long)h * k_hs + d];
            if (v)
                for (int d = 0; d < lv; ++d)
                    v_buf[slot * v_buf_ss + (long)h * v_buf_hs + d] =
                        v[t * v_ts + (long)h * v_hs + d];
        }
    }
}

/*
 * KV write into an fp8 pool ([FI] set_kv_buffer(layer, cache_loc, k, v,
 * k_scale, v_scale) with kv_cache_dtype fp8): each element is divided by its
 * scale in fp32 and stored as the nearest fp8 code (oracle_fp8_code):
 *   k_buf[cache_loc[t], h, d] = code((float)k[t, h, d] / (float)k_scale)
 *   v_buf[cache_loc[t], h, d] = code((float)v[t, h, d] / (float)v_scale)
 * v may be NULL (K-only pool).  Slots not in cache_loc keep their codes.
 */
void oracle_set_kv_buffer_fp8(
    const uint16_t *k, long k_ts, long k_hs, const uint16_t *v, long v_ts,
    long v_hs, const int64_t *cache_loc, long n_tokens, int hkv, int lk,
    int lv, float k_scale, float v_scale, int fmt, uint8_t *k_buf,
    long k_buf_ss, long k_buf_hs, uint8_t *v_buf, long v_buf_ss,
    long v_buf_hs)
{
    for (long t = 0; t < n_tokens; ++t) {
        long slot = (long)cache_loc[t];
        for (int h = 0; h < hkv; ++h) {
            for (int d = 0; d < lk; ++d) {
                float x = (float)bf16_to_double(k[t * k_ts + (long)h * k_hs + d]);
                k_buf[slot * k_buf_ss + (long)h * k_buf_hs + d] =
                    oracle_fp8_code(x / k_scale, fmt);
            }
            if (v)
                for (int d = 0; d < lv; ++d) {
                    float x = (float)bf16_to_double(v[t * v_ts + (long)h * v_hs + d]);
                    v_buf[slot * v_buf_ss + (long)h * v_buf_hs + d] =
                        oracle_fp8_code(x / v_scale, fmt);
                }
        }
    }
}

/*
 * Paged KV indices to per-token pool slots ([FI] the paged KV format of the
 * wrappers' plan: indptr over pages, indices of pages, last_page_len, and
 * page_size; the pool viewed as [pages, page_size, ...], so key j of
 * sequence b sits in page kv_indices[kv_indptr[b] + j / page_size] at
 * offset j % page_size):
 *   pages_b            = kv_indptr[b+1] - kv_indptr[b]
 *   T_b                = pages_b > 0 ? (pages_b - 1) * page_size
 *                                      + kv_last_page_len[b] : 0
 *   token_indptr[b+1]  = token_indptr[b] + T_b          (token_indptr[0] = 0)
 *   token_indices[token_indptr[b] + j]
 *       = kv_indices[kv_indptr[b] + j / page_size] * page_size
 *         + j % page_size                                  (j < T_b)
 */
void oracle_expand_paged_kv_indices(
    const int32_t *kv_indptr, const int32_t *kv_indices,
    const int32_t *kv_last_page_len, int page_size, int bs,
    int32_t *token_indptr, int32_t *token_indices)
{
    token_indptr[0] = 0;
    for (int b = 0; b < bs; ++b) {
        long pages = kv_indptr[b + 1] - kv_indptr[b];
        long t = pages > 0 ? (pages - 1) * page_size + kv_last_page_len[b] : 0;
        token_indptr[b + 1] = token_indptr[b] + (int32_t)t;
    }
    for (int b = 0; b < bs; ++b) {
        long t = token_indptr[b + 1] - token_indptr[b];
        for (long j = 0; j < t; ++j)
            token_indices[token_indptr[b] + j] =
                kv_indices[kv_indptr[b] + j / page_size] * page_size +
                (int32_t)(j % page_size);
    }
}
