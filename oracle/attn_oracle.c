/*
 * attn_oracle.c -- plain fp64 CPU oracle for varlen / paged causal attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant
 * with the CUDA library: it is a separate restatement of what the pages
 * define, written for a reader to check by eye, not for speed.
 *
 * Sources (page title, section):
 *  - "vLLM 中 Attention Kernel 如何并行处理多个请求" (www.2kiu.com):
 *      sec. 1 and 5   packed requests, local positions, block-diagonal mask
 *      sec. 10        bottom-right aligned mask q_abs = context_len + q_local
 *      sec. 11        paged address: block_table[r][pos / bs] * bs + pos % bs
 *  - "FlashAttention deep dive" (gaoleia.github.io):
 *      "flash_attn_varlen_func 参数说明"  softmax_scale multiplies Q K^T
 *      "KV Cache 更新"                    reshape_and_cache_flash via slot_mapping
 *      "合并算法"                          log-sum-exp merge of two states
 *      "FA3 的 FP8 支持"                   float8_e4m3fn KV cache
 *
 * Every value is read in its storage type and widened exactly to double
 * (bf16, fp16 and e4m3 all embed exactly in double); all arithmetic after
 * that is fp64.  Softmax is taken in two passes (max, then sum), i.e. the
 * textbook definition, not the online recurrence.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* storage type codes used by this oracle's own interface */
#define ORC_BF16 0
#define ORC_FP16 1
#define ORC_E4M3 2
#define ORC_FP32 3

#define ORC_OK 0
#define ORC_EINVAL 1       /* bad sizes / dtype */
#define ORC_EBLOCK 2       /* block id out of [0, num_blocks) */
#define ORC_ESLOT 3        /* slot out of [0, num_blocks * block_size) */

/* ---------------------------------------------------------------- decoding */

/* bf16: the upper 16 bits of an IEEE binary32. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
static double fp16_to_double(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return s ? -v : v;
}

/* float8 e4m3 "fn" variant: 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 is NaN, largest finite 448. */
double oracle_e4m3_to_double(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                  /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);        /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* Round an fp32 value to e4m3: nearest representable value, ties to the
 * even mantissa, magnitudes beyond 448 saturate to +-448 (the "satfinite"
 * convention), NaN maps to the NaN code.  The two scaled quantities fed to
 * nearbyint() below are exact in double, so the default rounding mode
 * (round-half-even) performs exactly one correct rounding. */
uint8_t oracle_e4m3_from_float(float xf) {
    double x = (double)xf;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (isnan(x))
        return (uint8_t)(sign | 0x7F);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: grid step 2^-9; m == 8 is the smallest normal */
        double m = nearbyint(a * 512.0);
        return (uint8_t)(sign | (uint8_t)m);
    }
    int k;
    double f = frexp(a, &k);            /* a = f * 2^k, f in [0.5, 1) */
    int E = k - 1;                      /* a = (2f) * 2^E, 2f in [1, 2) */
    double mant = nearbyint((2.0 * f - 1.0) * 8.0);
    if (mant >= 8.0) {                  /* rounded up to the next binade */
        mant = 0.0;
        E += 1;
    }
    if (E > 8 || (E == 8 && mant > 6.0))   /* beyond 448 after rounding */
        return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | (uint8_t)(((E + 7) << 3) | (int)mant));
}

static double load_elem(const void *base, int64_t idx, int dtype) {
    switch (dtype) {
    case ORC_BF16: return bf16_to_double(((const uint16_t *)base)[idx]);
    case ORC_FP16: return fp16_to_double(((const uint16_t *)base)[idx]);
    case ORC_E4M3: return oracle_e4m3_to_double(((const uint8_t *)base)[idx]);
    case ORC_FP32: return (double)((const float *)base)[idx];
    default: return NAN;
    }
}

static int elem_bytes(int dtype) {
    switch (dtype) {
    case ORC_BF16: case ORC_FP16: return 2;
    case ORC_E4M3: return 1;
    case ORC_FP32: return 4;
    default: return 0;
    }
}

/* ------------------------------------------------------------- attention */

/*
 * out[t, h, :] = sum_j softmax_j(scale * q[t,h,:] . K_j) V_j   over the keys
 * visible to packed query token t, for every query head h.
 *
 * Request r owns packed tokens [cu_seqlens_q[r], cu_seqlens_q[r+1]) and
 * kv_len = seqused_k[r] keys.  Its i-th query token sits at absolute
 * position ctx + i, ctx = kv_len - q_len (bottom-right alignment of the
 * causal mask).  Key j (0 <= j < kv_len) is visible iff !causal or
 * j <= ctx + i.  Query head h reads KV head h / (Hq / Hkv).
 *
 * Key j of request r lives at physical block block_table[r*bt_stride + j/bs],
 * row j % bs, so K_j[g, d] = k_cache[((phys*bs + j%bs)*Hkv + g)*D + d].
 * FP8 caches are widened and multiplied by k_scale / v_scale.
 *
 * rows: optional list of packed token indices to evaluate (n_rows of them);
 * NULL means all tokens 0 .. cu_seqlens_q[B]-1.  out is [n, Hq, D] and lse
 * is [n, Hq] (natural log), n = number of evaluated tokens.  A query with
 * no visible key gets out = 0 and lse = -inf.
 */
/*
 * Variants named in the argument table of "FlashAttention deep dive"
 * (flash_attn_varlen_func: window_size, softcap, s_aux) and in its table of
 * supported variants (sliding window = local attention, soft cap on the
 * logits, attention sinks).  The page names them without formulas; this
 * oracle takes the plain readings:
 *   window (left, right): query i of a request sits at p = ctx + i and sees
 *     keys j with p - left <= j <= p + right (a negative bound is
 *     unlimited), on top of the causal rule j <= p and of j < kv_len;
 *   softcap c > 0: each scaled logit s becomes c * tanh(s / c);
 *   q_scale: q is stored scaled ("FlashAttention deep dive", FA3 FP8
 *     support: q_descale beside k/v_descale), its value is code * q_scale;
 *   sinks: query head h has a logit z_h that joins the softmax
 *     normalisation with a zero value vector:
 *       out = sum_j e^{s_j} V_j / (e^{z_h} + sum_j e^{s_j}),
 *       lse = log(e^{z_h} + sum_j e^{s_j}).
 */
int oracle_attention_ext(const void *q, int q_dtype, int64_t q_stride_tok,
                         const void *k_cache, const void *v_cache, int kv_dtype,
                         double k_scale, double v_scale,
                         const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                         const int32_t *block_table, int64_t bt_stride,
                         int B, int Hq, int Hkv, int D, int bs, int num_blocks,
                         double softmax_scale, int causal,
                         int64_t window_left, int64_t window_right, double softcap,
                         const double *sinks, double q_scale,
                         const int64_t *rows, int64_t n_rows,
                         double *out, double *lse, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || bs <= 0 ||
        num_blocks < 0 || elem_bytes(q_dtype) == 0 || elem_bytes(kv_dtype) == 0)
        return ORC_EINVAL;
    const int G = Hq / Hkv;
    const int64_t T = cu_seqlens_q[B];
    const int64_t n = rows ? n_rows : T;
    int status = ORC_OK;

#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel
    {
        int64_t cap = 0;
        double *s = NULL;
        double *qv = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t w = 0; w < n * Hq; ++w) {
            const int64_t oi = w / Hq;                 /* output row */
            const int h = (int)(w % Hq);
            const int64_t t = rows ? rows[oi] : oi;    /* packed token */
            double *o = out + (oi * Hq + h) * D;
            if (t < 0 || t >= T) {
#pragma omp atomic write
                status = ORC_EINVAL;
                continue;
            }
            int r = 0;                                  /* owning request */
            while (!(cu_seqlens_q[r] <= t && t < cu_seqlens_q[r + 1]))
                ++r;
            const int64_t q_len = cu_seqlens_q[r + 1] - cu_seqlens_q[r];
            const int64_t kv_len = seqused_k[r];
            const int64_t i = t - cu_seqlens_q[r];
            const int64_t ctx = kv_len - q_len;
            const int g = h / G;
            int64_t last = kv_len - 1;                  /* last visible key */
            if (causal && ctx + i < last)
                last = ctx + i;
            if (window_right >= 0 && ctx + i + window_right < last)
                last = ctx + i + window_right;
            int64_t first = 0;                          /* first visible key */
            if (window_left >= 0 && ctx + i - window_left > first)
                first = ctx + i - window_left;
            const int64_t nvis = last + 1 > 0 ? last + 1 : 0;   /* keys 0 .. last: s[] indexed by j */
            if (nvis > cap) {
                free(s);
                cap = nvis;
                s = (double *)malloc(sizeof(double) * (size_t)cap);
            }
            const int64_t q_off = t * q_stride_tok + (int64_t)h * D;
            for (int d = 0; d < D; ++d)
                qv[d] = load_elem(q, q_off + d, q_dtype) * q_scale;
            int bad = 0;
            double M = -INFINITY;
            for (int64_t j = first; j < nvis; ++j) {
                const int32_t phys = block_table[r * bt_stride + j / bs];
                if (phys < 0 || phys >= num_blocks) { bad = 1; break; }
                const int64_t k_off = (((int64_t)phys * bs + j % bs) * Hkv + g) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += qv[d] * (load_elem(k_cache, k_off + d, kv_dtype) * k_scale);
                s[j] = softmax_scale * dot;
                if (softcap > 0.0)
                    s[j] = softcap * tanh(s[j] / softcap);
                if (s[j] > M) M = s[j];
            }
            if (bad) {
#pragma omp atomic write
                status = ORC_EBLOCK;
                continue;
            }
            const double z = sinks ? sinks[h] : -INFINITY;     /* sink logit */
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (nvis <= first && z == -INFINITY) {      /* no visible key and no sink */
                lse[oi * Hq + h] = -INFINITY;
                continue;
            }
            if (z > M) M = z;
            double L = z == -INFINITY ? 0.0 : exp(z - M);      /* the sink's share, value 0 */
            for (int64_t j = first; j < nvis; ++j) {
                const double e = exp(s[j] - M);
                L += e;
                const int32_t phys = block_table[r * bt_stride + j / bs];
                const int64_t v_off = (((int64_t)phys * bs + j % bs) * Hkv + g) * D;
                for (int d = 0; d < D; ++d)
                    o[d] += e * (load_elem(v_cache, v_off + d, kv_dtype) * v_scale);
            }
            for (int d = 0; d < D; ++d) o[d] /= L;
            lse[oi * Hq + h] = M + log(L);
        }
        free(s);
        free(qv);
    }
    return status;
}

/* Plain attention: no window, no soft cap, no sink. */
int oracle_attention(const void *q, int q_dtype, int64_t q_stride_tok,
                     const void *k_cache, const void *v_cache, int kv_dtype,
                     double k_scale, double v_scale,
                     const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                     const int32_t *block_table, int64_t bt_stride,
                     int B, int Hq, int Hkv, int D, int bs, int num_blocks,
                     double softmax_scale, int causal,
                     const int64_t *rows, int64_t n_rows,
                     double *out, double *lse, int nthreads) {
    return oracle_attention_ext(q, q_dtype, q_stride_tok, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                                cu_seqlens_q, seqused_k, block_table, bt_stride, B, Hq, Hkv, D, bs,
                                num_blocks, softmax_scale, causal, -1, -1, 0.0, NULL, 1.0, rows, n_rows, out,
                                lse, nthreads);
}

/* ------------------------------------------------------------------ merge */

/*
 * Merge two attention states over disjoint key sets (the cascade merge and
 * the split-KV reduction are the same operation):
 *   lse = log(exp(lse1) + exp(lse2)),
 *   out = exp(lse1 - lse) * o1 + exp(lse2 - lse) * o2.
 * The larger lse is factored out before exponentiating.  A side with
 * lse = -inf covers no key and gets weight 0; both -inf gives out 0,
 * lse -inf.
 */
void oracle_merge_states(int64_t n, int D, const double *o1, const double *lse1,
                         const double *o2, const double *lse2,
                         double *out, double *lse) {
    for (int64_t i = 0; i < n; ++i) {
        const double a = lse1[i], b = lse2[i];
        if (a == -INFINITY && b == -INFINITY) {
            for (int d = 0; d < D; ++d) out[i * D + d] = 0.0;
            lse[i] = -INFINITY;
            continue;
        }
        const double mx = a > b ? a : b;
        const double l = mx + log(exp(a - mx) + exp(b - mx));
        const double w1 = exp(a - l), w2 = exp(b - l);
        for (int d = 0; d < D; ++d)
            out[i * D + d] = w1 * o1[i * D + d] + w2 * o2[i * D + d];
        lse[i] = l;
    }
}

/* --------------------------------------------------------------- KV write */

/*
 * Scatter new K/V rows into the paged cache through slot_mapping:
 * token t goes to block slot[t] / bs, row slot[t] % bs; slot < 0 means
 * "no slot" (padding) and the token is skipped.  key/value are [T, Hkv, D]
 * with token stride src_stride_tok (elements).  When the cache type equals
 * the source type the bytes are copied; for an e4m3 cache each value is
 * divided by its per-tensor scale in fp32 and rounded to e4m3 (nearest,
 * ties to even, saturating at +-448).
 */
int oracle_kv_write(const void *key, const void *value, int src_dtype,
                    int64_t src_stride_tok, void *k_cache, void *v_cache,
                    int kv_dtype, const int64_t *slot_mapping, int64_t T,
                    int Hkv, int D, int bs, int num_blocks,
                    float k_scale, float v_scale) {
    const int sb = elem_bytes(src_dtype), cb = elem_bytes(kv_dtype);
    if (sb == 0 || cb == 0 || (kv_dtype != src_dtype && kv_dtype != ORC_E4M3))
        return ORC_EINVAL;
    for (int64_t t = 0; t < T; ++t)
        if (slot_mapping[t] >= (int64_t)num_blocks * bs)
            return ORC_ESLOT;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        const int64_t blk = slot / bs, row = slot % bs;
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                const int64_t src = t * src_stride_tok + (int64_t)h * D + d;
                const int64_t dst = ((blk * bs + row) * Hkv + h) * D + d;
                if (kv_dtype == src_dtype) {
                    memcpy((char *)k_cache + dst * cb, (const char *)key + src * sb, (size_t)cb);
                    memcpy((char *)v_cache + dst * cb, (const char *)value + src * sb, (size_t)cb);
                } else {
                    const float kx = (float)load_elem(key, src, src_dtype);
                    const float vx = (float)load_elem(value, src, src_dtype);
                    ((uint8_t *)k_cache)[dst] = oracle_e4m3_from_float(kx / k_scale);
                    ((uint8_t *)v_cache)[dst] = oracle_e4m3_from_float(vx / v_scale);
                }
            }
        }
    }
    return ORC_OK;
}
