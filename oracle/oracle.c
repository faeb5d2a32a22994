/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for causal
 * grouped-query flash attention with attention sinks + a recent window and an
 * fp32 or Q4_0 KV cache.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
 * baseline load this library. The product path never links or calls it, and it
 * shares no code, header or table with the CUDA path.
 *
 * Sources (page title, then section):
 *   [A]  "attention.cu" (Foundry cuda_kernels): file header (sliding window
 *        with sinks), "4-bit KV cache (Q4_0 blocks)", fc_kvq4_is_fp16,
 *        fc_kvq4_quant_block, fc_kvq4_dequant_elem, fc_attn_tile_in_window,
 *        fc_attn_flash_prefill_q4 (fp16 shadow read rule, ring liveness),
 *        "Decode-mode flash attention" (fc_attn_dec_plan, the combine).
 *   [B]  "vt/ops.h" (vllm-cpp-sys): vt::Attention (dense causal GQA
 *        definition, q head h reads kv head h/(Hq/Hkv)), MergeAttnStates.
 *   [C]  "qwen38_batched.rs": bq_attn (two-pass global-max decode attention).
 *
 * Attention is computed as its definition in fp64 with a two-pass global max
 * ([B] vt::Attention, [C] bq_attn):
 *     s_j = scale * sum_e q[e] * k_j[e]          for j in S(p)
 *     out = sum_j exp(s_j - m) v_j / sum_j exp(s_j - m),   m = max_j s_j
 * where S(p) is the attended key set of the query at position p ([A] header).
 *
 * The Q4_0 quantiser follows [A] fc_kvq4_quant_block step by step in fp32, the
 * precision that page fixes; fp16 conversion is round-to-nearest-even done
 * by bit manipulation.
 *
 * Built with -ffp-contract=off and without fast-math so every float
 * operation is one IEEE single-precision operation.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define ORACLE_Q4_BLK 32
#define ORACLE_Q4_BLK_BYTES 18
#define ORACLE_RING_ROWS 256 /* [A] 4-bit KV cache: the recent ring holds 256 rows */

/* ------------------------------------------------------------------ fp16 */

/* fp32 -> binary16, round to nearest, ties to even ([A] fc_attn_kv_append_q4
 * mirrors rows with __float2half, which rounds to nearest even). Overflow
 * gives +-inf, fp16 subnormals are produced, NaN maps to the quiet NaN
 * sign|0x7e00. */
uint16_t oracle_f16_rne(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    const uint32_t sign = (x >> 16) & 0x8000u;
    const uint32_t bexp = (x >> 23) & 0xffu;
    const uint32_t man = x & 0x7fffffu;
    if (bexp == 0xffu)
        return (uint16_t)(sign | (man ? 0x7e00u : 0x7c00u));
    if (bexp == 0)            /* fp32 zero or subnormal: below 2^-126, rounds to 0 */
        return (uint16_t)sign;
    const int E = (int)bexp - 127;
    if (E > 15)
        return (uint16_t)(sign | 0x7c00u);
    const uint32_t sig = man | 0x800000u; /* 24-bit significand, value sig * 2^(E-23) */
    if (E >= -14) {
        uint32_t h = ((uint32_t)(E + 15) << 10) | ((sig >> 13) & 0x3ffu);
        const uint32_t rem = sig & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u)))
            h += 1u; /* a carry into the exponent is the correct next value (or inf) */
        return (uint16_t)(sign | h);
    }
    /* fp16 subnormal: units of 2^-24, count = sig * 2^(E+1) = sig >> s */
    const int s = -(E + 1); /* >= 14 */
    if (s > 31)
        return (uint16_t)sign;
    uint32_t qv = sig >> s;
    const uint32_t rem = sig & ((1u << s) - 1u);
    const uint32_t half = 1u << (s - 1);
    if (rem > half || (rem == half && (qv & 1u)))
        qv += 1u;
    return (uint16_t)(sign | qv);
}

/* binary16 bits -> exact value as double. */
double oracle_f16_to_f64(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int bexp = (h >> 10) & 0x1f;
    const int man = h & 0x3ff;
    double v;
    if (bexp == 0x1f)
        v = man ? NAN : INFINITY;
    else if (bexp == 0)
        v = ldexp((double)man, -24);
    else
        v = ldexp((double)(man | 0x400), bexp - 25);
    return sign ? -v : v;
}

void oracle_f16_rne_array(const float *x, int64_t count, uint16_t *out) {
    for (int64_t i = 0; i < count; i++)
        out[i] = oracle_f16_rne(x[i]);
}

void oracle_f16_to_f64_array(const uint16_t *h, int64_t count, double *out) {
    for (int64_t i = 0; i < count; i++)
        out[i] = oracle_f16_to_f64(h[i]);
}

/* ---------------------------------------------------------- fp8 e4m3fn */

/* fp8 e4m3fn ("vt/ops.h" fp8 KV cache: 1-byte fp8-e4m3fn pages): 1 sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
 * subnormals m * 2^-9; there is no infinity, S.1111.111 is NaN, so the
 * largest finite magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_f64(uint8_t c) {
    const int sign = (c >> 7) & 1;
    const int e = (c >> 3) & 0xf;
    const int m = c & 7;
    double v;
    if (e == 0xf && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

/* float -> e4m3fn, round to nearest, ties to even, magnitudes past 448
 * (and infinities) saturate to +-448 ("vt/ops.h": fp8_e4m3(clamp(x, -448,
 * 448)), the hardware conversion with saturation to finite); NaN gives 0x7f. */
uint8_t oracle_e4m3_rne_sat(float f) {
    if (isnan(f))
        return 0x7f;
    const uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint8_t)(sign | 0x7e);
    int e2;
    (void)frexp(a, &e2); /* a = fr * 2^e2, fr in [0.5, 1): floor(log2 a) = e2 - 1 */
    int e = e2 - 1;
    if (e < -6) {
        /* subnormal grid: multiples of 2^-9; q = 8 is the smallest normal */
        const double t = ldexp(a, 9);
        double q = floor(t);
        const double r = t - q;
        if (r > 0.5 || (r == 0.5 && fmod(q, 2.0) == 1.0))
            q += 1.0;
        return (uint8_t)(sign | (uint8_t)q);
    }
    if (e > 8)
        return (uint8_t)(sign | 0x7e);
    /* normal: a = q * 2^(e-3) with q in [8, 16) */
    const double t = ldexp(a, 3 - e);
    double q = floor(t);
    const double r = t - q;
    if (r > 0.5 || (r == 0.5 && fmod(q, 2.0) == 1.0))
        q += 1.0;
    if (q == 16.0) {
        q = 8.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && q > 14.0))
        return (uint8_t)(sign | 0x7e); /* past 448: saturate */
    return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | ((int)q - 8)));
}

/* The fp8 KV store of "vt/ops.h" (ReshapeAndCacheFp8): each element as
 * Quantize(x / scale), the division one float operation. */
void oracle_e4m3_store_array(const float *x, int64_t count, float scale, uint8_t *out) {
    for (int64_t i = 0; i < count; i++) {
        const float t = x[i] / scale;
        out[i] = oracle_e4m3_rne_sat(t);
    }
}

/* The fp8 KV read: Dequant(fp8) * scale, one float multiplication. */
void oracle_e4m3_load_array(const uint8_t *q, int64_t count, float scale, double *out) {
    for (int64_t i = 0; i < count; i++) {
        const float v = (float)oracle_e4m3_to_f64(q[i]);
        const float w = v * scale;
        out[i] = (double)w;
    }
}

/* ------------------------------------------------------------------ Q4_0 */

/* Round to nearest integer, ties to even, with the saturating conversion of
 * a float to a signed 32-bit integer: NaN -> 0, out of range -> INT32_MIN /
 * INT32_MAX. (Reading of [A] fc_kvq4_quant_block "(int)rintf(x * id)": the
 * conversion order convert -> +8 -> clamp is stated to be part of the output.)
 * Done in double, where every float and every half-integer is exact. */
static int32_t oracle_cvt_rni_s32(float t) {
    if (isnan(t))
        return 0;
    const double td = (double)t;
    if (td >= 2147483648.0)
        return INT32_MAX;
    if (td <= -2147483648.0)
        return INT32_MIN;
    double r = floor(td);
    const double frac = td - r; /* exact: |td| < 2^31 */
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    return (int32_t)r;
}

/* Code of one element: convert, add 8 with 32-bit wrap-around, clamp to [0,15]. */
static int oracle_q4_code(float t) {
    const int32_t qv = oracle_cvt_rni_s32(t);
    const int32_t c = (int32_t)((uint32_t)qv + 8u);
    if (c < 0)
        return 0;
    if (c > 15)
        return 15;
    return (int)c;
}

/* Quantise one block of 32 floats into 18 bytes ([A] "4-bit KV cache (Q4_0
 * blocks)" and fc_kvq4_quant_block):
 *   amax = fmaxf fold of |x_j| from +0.0
 *   d    = amax / -8        (scale stored negative)
 *   id   = d != 0 ? 1 / d : 0
 *   code_j = clamp(rni(x_j * id) + 8, 0, 15)
 *   bytes 0..1 = binary16(d) little-endian; byte 2+j = code_j | code_{j+16} << 4 */
void oracle_q4_encode_block(const float *x, uint8_t *b) {
    float amax = 0.0f;
    for (int j = 0; j < ORACLE_Q4_BLK; j++)
        amax = fmaxf(amax, fabsf(x[j]));
    const float d = amax / -8.0f;
    const float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    const uint16_t dh = oracle_f16_rne(d);
    b[0] = (uint8_t)(dh & 0xffu);
    b[1] = (uint8_t)(dh >> 8);
    for (int j = 0; j < ORACLE_Q4_BLK / 2; j++) {
        const float t_lo = x[j] * id;
        const float t_hi = x[j + ORACLE_Q4_BLK / 2] * id;
        b[2 + j] = (uint8_t)(oracle_q4_code(t_lo) | (oracle_q4_code(t_hi) << 4));
    }
}

/* Decode one 18-byte block to 32 exact values (c - 8) * d ([A]
 * fc_kvq4_dequant_elem). */
void oracle_q4_decode_block(const uint8_t *b, double *out) {
    const uint16_t dh = (uint16_t)(b[0] | (b[1] << 8));
    const double d = oracle_f16_to_f64(dh);
    for (int j = 0; j < ORACLE_Q4_BLK / 2; j++) {
        out[j] = (double)((b[2 + j] & 0xf) - 8) * d;
        out[j + ORACLE_Q4_BLK / 2] = (double)(((b[2 + j] >> 4) & 0xf) - 8) * d;
    }
}

/* Rows of head_dim floats (head_dim % 32 == 0) -> rows of head_dim/32 blocks. */
void oracle_q4_encode_rows(const float *x, int64_t rows, int head_dim, uint8_t *out) {
    const int nb = head_dim / ORACLE_Q4_BLK;
    for (int64_t r = 0; r < rows; r++)
        for (int b = 0; b < nb; b++)
            oracle_q4_encode_block(x + r * head_dim + b * ORACLE_Q4_BLK,
                                   out + (r * nb + b) * ORACLE_Q4_BLK_BYTES);
}

void oracle_q4_decode_rows(const uint8_t *in, int64_t rows, int head_dim, double *out) {
    const int nb = head_dim / ORACLE_Q4_BLK;
    for (int64_t r = 0; r < rows; r++)
        for (int b = 0; b < nb; b++)
            oracle_q4_decode_block(in + (r * nb + b) * ORACLE_Q4_BLK_BYTES,
                                   out + r * head_dim + b * ORACLE_Q4_BLK);
}

/* ------------------------------------------------------ visibility rules */

/* Is key j in the attended set of the query at position p? ([A] file header:
 * with win > 0 the query attends [0, sink) U [p - win + 1, p]; with win <= 0
 * it attends every key j <= p.) Causality always applies. */
int oracle_visible(int p, int j, int sink, int win) {
    if (j < 0 || j > p)
        return 0;
    if (win <= 0)
        return 1;
    return (j < sink) || (j >= p - win + 1);
}

/* Tile map by brute force for n queries at positions pos0 .. pos0+n-1 over
 * keys 0 .. pos0+n-1: map[qt][kt] = 1 iff some query row t in
 * [qt*bq, min(n, qt*bq+bq)), at position pos0 + t, sees some key j in
 * [kt*bk, min(L, kt*bk+bk)), L = pos0 + n. */
void oracle_tile_map(int pos0, int n, int bq, int bk, int sink, int win, uint8_t *map) {
    const int L = pos0 + n;
    const int nqt = (n + bq - 1) / bq, nkt = (L + bk - 1) / bk;
    for (int qt = 0; qt < nqt; qt++)
        for (int kt = 0; kt < nkt; kt++) {
            int any = 0;
            for (int t = qt * bq; t < n && t < qt * bq + bq && !any; t++)
                for (int j = kt * bk; j < L && j < kt * bk + bk; j++)
                    if (oracle_visible(pos0 + t, j, sink, win)) {
                        any = 1;
                        break;
                    }
            map[(int64_t)qt * nkt + kt] = (uint8_t)any;
        }
}

/* Which copy of key s a query at position p reads from a Q4_0 cache whose
 * last appended row is L-1 ([A] fc_kvq4_is_fp16 and the ring liveness floor
 * of fc_attn_flash_prefill_q4): the fp16 shadow iff s is a shadow sink row, or
 * it lies in the shadow window of p and its ring slot still holds it. */
int oracle_reads_fp16(int p, int s, int L, int shadow_sink, int shadow_win) {
    if (s < shadow_sink)
        return 1;
    return shadow_win > 0 && s > p - shadow_win && s > L - 1 - ORACLE_RING_ROWS;
}

/* --------------------------------------------------------------- attention */

/* Value of element e of key s (kv head g) seen by the query at position p.
 * body: [L][Hkv][hd] doubles (fp32 widened, or Q4_0 decoded);
 * f16:  [L][Hkv][hd] doubles (fp16 shadow copy) or NULL for an fp32 cache. */
static const double *oracle_key_row(const double *body, const double *f16, int p, int s, int g,
                                    int L, int Hkv, int hd, int shadow_sink, int shadow_win) {
    const int64_t off = ((int64_t)s * Hkv + g) * hd;
    if (f16 && oracle_reads_fp16(p, s, L, shadow_sink, shadow_win))
        return f16 + off;
    return body + off;
}

/* out[r][h][:] for query rows r at positions qpos[r] (q: [nq][Hq][hd] float),
 * and, when lse is not NULL, lse[r][h] = log(sum_j exp(s_j)) = m + log(sum_j
 * exp(s_j - m)), the log-sum-exp of the row's scores ([B] MergeAttnStates
 * consumes it). Returns 0, or -1 if a position is out of range, -2 if a query
 * has no visible key (impossible: p always sees itself). */
int oracle_attention(const float *q, const int *qpos, int nq, int Hq, int Hkv, int hd, int L,
                     const double *kbody, const double *vbody, const double *kf16,
                     const double *vf16, int shadow_sink, int shadow_win, int sink, int win,
                     double scale, double *out, double *lse) {
    if (Hkv <= 0 || Hq % Hkv != 0)
        return -1;
    const int G = Hq / Hkv;
    int status = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t rh = 0; rh < (int64_t)nq * Hq; rh++) {
        const int r = (int)(rh / Hq), h = (int)(rh % Hq);
        const int p = qpos[r];
        double *o = out + rh * hd;
        if (p < 0 || p >= L) {
#pragma omp atomic write
            status = -1;
            continue;
        }
        const int g = h / G; /* [B] vt::Attention: q head h reads kv head h / (Hq/Hkv) */
        const float *qr = q + rh * hd;
        double *sc = (double *)malloc(sizeof(double) * (size_t)(p + 1));
        /* pass 1: scores and the global max */
        double m = -INFINITY;
        for (int j = 0; j <= p; j++) {
            if (!oracle_visible(p, j, sink, win))
                continue;
            const double *kr = oracle_key_row(kbody, kf16, p, j, g, L, Hkv, hd, shadow_sink,
                                              shadow_win);
            double dot = 0.0;
            for (int e = 0; e < hd; e++)
                dot += (double)qr[e] * kr[e];
            sc[j] = scale * dot;
            if (sc[j] > m)
                m = sc[j];
        }
        if (m == -INFINITY) {
#pragma omp atomic write
            status = -2;
            free(sc);
            continue;
        }
        /* pass 2: weights, denominator and the weighted sum of V */
        for (int e = 0; e < hd; e++)
            o[e] = 0.0;
        double den = 0.0;
        for (int j = 0; j <= p; j++) {
            if (!oracle_visible(p, j, sink, win))
                continue;
            const double w = exp(sc[j] - m);
            den += w;
            const double *vr = oracle_key_row(vbody, vf16, p, j, g, L, Hkv, hd, shadow_sink,
                                              shadow_win);
            for (int e = 0; e < hd; e++)
                o[e] += w * vr[e];
        }
        for (int e = 0; e < hd; e++)
            o[e] /= den;
        if (lse)
            lse[rh] = m + log(den);
        free(sc);
    }
    return status;
}

/* [B] MergeAttnStates: two attention results over disjoint key sets, each with
 * its log-sum-exp, combined into the result over the union. Per token t and
 * head h (outputs [T][H][D], lses [H][T]):
 *   - tokens t >= with_context (when with_context >= 0) take the suffix output
 *     and its lse unchanged;
 *   - an lse of +inf counts as -inf;
 *   - if both lses are -inf (no key on either side) the output is the prefix
 *     output and the lse is -inf;
 *   - otherwise m = max(lp, ls), wp = exp(lp - m), ws = exp(ls - m),
 *     out = prefix * wp/(wp+ws) + suffix * ws/(wp+ws), lse = log(wp+ws) + m.
 * Inputs are float (the tensors' type), arithmetic fp64. */
void oracle_merge_attn_states(const float *prefix, const float *prefix_lse, const float *suffix,
                              const float *suffix_lse, int T, int H, int D, int with_context,
                              double *out, double *out_lse) {
    for (int t = 0; t < T; t++)
        for (int h = 0; h < H; h++) {
            const int64_t row = ((int64_t)t * H + h) * D;
            const int64_t li = (int64_t)h * T + t;
            if (with_context >= 0 && t >= with_context) {
                for (int d = 0; d < D; d++)
                    out[row + d] = suffix[row + d];
                out_lse[li] = suffix_lse[li];
                continue;
            }
            double lp = prefix_lse[li], ls = suffix_lse[li];
            if (lp == INFINITY)
                lp = -INFINITY;
            if (ls == INFINITY)
                ls = -INFINITY;
            const double m = lp > ls ? lp : ls;
            if (m == -INFINITY) {
                for (int d = 0; d < D; d++)
                    out[row + d] = prefix[row + d];
                out_lse[li] = -INFINITY;
                continue;
            }
            const double wp = exp(lp - m), ws = exp(ls - m), tot = wp + ws;
            for (int d = 0; d < D; d++)
                out[row + d] = prefix[row + d] * (wp / tot) + suffix[row + d] * (ws / tot);
            out_lse[li] = log(tot) + m;
        }
}

/* -------------------------------------------------- split-KV decode + merge */

/* Split plan of [A] "Decode-mode flash attention" (fc_attn_dec_plan): about
 * kps keys per split, between 1 and cap splits, split length rounded up to a
 * multiple of 16; returns the number of non-empty splits. */
int oracle_dec_plan(int seq_len, int kps, int cap, int *split_len_out) {
    int ns = (seq_len + kps - 1) / kps;
    if (ns < 1)
        ns = 1;
    if (ns > cap)
        ns = cap;
    int split_len = (seq_len + ns - 1) / ns;
    split_len = (split_len + 15) / 16 * 16;
    *split_len_out = split_len;
    return (seq_len + split_len - 1) / split_len;
}

/* Unnormalised partial over keys [k_lo, k_hi) of one query (position p) for
 * every q head: m = max s_j, l = sum exp(s_j - m), acc = sum exp(s_j - m) v_j
 * over the visible keys of the range; an empty range gives m = -inf, l = 0,
 * acc = 0 ([A] "Multi-user decode attention": empty partials).
 * m, l: [Hq]; acc: [Hq][hd]. */
void oracle_partial(const float *q, int p, int k_lo, int k_hi, int Hq, int Hkv, int hd, int L,
                    const double *kbody, const double *vbody, const double *kf16,
                    const double *vf16, int shadow_sink, int shadow_win, int sink, int win,
                    double scale, double *m_out, double *l_out, double *acc_out) {
    const int G = Hq / Hkv;
    for (int h = 0; h < Hq; h++) {
        const int g = h / G;
        const float *qr = q + (int64_t)h * hd;
        double *acc = acc_out + (int64_t)h * hd;
        double m = -INFINITY;
        for (int j = k_lo; j < k_hi; j++) {
            if (!oracle_visible(p, j, sink, win))
                continue;
            const double *kr = oracle_key_row(kbody, kf16, p, j, g, L, Hkv, hd, shadow_sink,
                                              shadow_win);
            double dot = 0.0;
            for (int e = 0; e < hd; e++)
                dot += (double)qr[e] * kr[e];
            if (scale * dot > m)
                m = scale * dot;
        }
        for (int e = 0; e < hd; e++)
            acc[e] = 0.0;
        double l = 0.0;
        if (m != -INFINITY) {
            for (int j = k_lo; j < k_hi; j++) {
                if (!oracle_visible(p, j, sink, win))
                    continue;
                const double *kr = oracle_key_row(kbody, kf16, p, j, g, L, Hkv, hd,
                                                  shadow_sink, shadow_win);
                double dot = 0.0;
                for (int e = 0; e < hd; e++)
                    dot += (double)qr[e] * kr[e];
                const double w = exp(scale * dot - m);
                l += w;
                const double *vr = oracle_key_row(vbody, vf16, p, j, g, L, Hkv, hd,
                                                  shadow_sink, shadow_win);
                for (int e = 0; e < hd; e++)
                    acc[e] += w * vr[e];
            }
        }
        m_out[h] = m;
        l_out[h] = l;
    }
}

/* Log-sum-exp merge of ns partials of one head, in ascending split order
 * ([A] fc_attn_flash_decode_combine; [B] deterministic ascending merge):
 *   M = max m_s, w_s = exp(m_s - M) (0 for an empty split),
 *   out = sum w_s acc_s / sum w_s l_s.
 * m, l: [ns]; acc: [ns][hd]. Returns -1 if every split is empty. */
int oracle_combine(const double *m, const double *l, const double *acc, int ns, int hd,
                   double *out) {
    double M = -INFINITY;
    for (int s = 0; s < ns; s++)
        if (m[s] > M)
            M = m[s];
    if (M == -INFINITY)
        return -1;
    double den = 0.0;
    for (int e = 0; e < hd; e++)
        out[e] = 0.0;
    for (int s = 0; s < ns; s++) {
        if (m[s] == -INFINITY)
            continue;
        const double w = exp(m[s] - M);
        den += w * l[s];
        for (int e = 0; e < hd; e++)
            out[e] += w * acc[(int64_t)s * hd + e];
    }
    for (int e = 0; e < hd; e++)
        out[e] /= den;
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
