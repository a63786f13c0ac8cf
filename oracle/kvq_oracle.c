/*
 * kvq_oracle.c -- plain, slow, fp64 CPU oracle for decode attention over a
 * quantized KV cache.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the benchmark's CPU-baseline leg may call it; the product path never does.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes, and where each rule comes from:
 *  - K is kept as an 8-bit payload plus one fp16 scale per 32 elements
 *    ("Flash Attention for llama.cpp on RDNA3", first paragraph: only the
 *    8-bit K payload and fp16 scales are stored).  The scale is absmax/127
 *    rounded to fp16; codes are x/s rounded half away from zero, clamped to
 *    [-127, 127].
 *  - V is q8_0 (same rule as K) or q4_0 (scale d = absmax/8 rounded to fp16,
 *    code q = round(x/d) + 8 clamped to [0, 15], value (q-8)*d) -- the V
 *    formats of the VRAM and KLD tables of the same page.
 *  - Q is quantized with the K rule, so QK^T is a sum over 32-blocks of exact
 *    integer dot products I_b, each scaled by sq_b*sk_b ("integer-native
 *    pipeline", BitLLM summary, "How to use": the MatMul stays in the integer
 *    domain, casts are deferred).
 *  - Attention is textbook softmax attention over those dequantized tensors,
 *    evaluated two-pass (max, then sum) in fp64.
 *  - F16 K variant ("Flash Attention for llama.cpp on RDNA3", title and KLD
 *    tables: F16 K with q4_0 V): K is kept as the fp16 values themselves and
 *    Q is not quantized, so the score is sm_scale * sum_j q_j * k_j over the
 *    fp16 values (orc_decode_seq_f16k).
 *
 * Byte layouts emitted (and read back) by this file:
 *  - K codes: int8 [n_kv_heads][n_tok][head_dim] (4 per 32-bit word,
 *    little-endian: byte i of word w is element 4w+i).
 *  - F16 K: fp16 bit patterns [n_kv_heads][n_tok][head_dim].
 *  - K / V scales: fp16 bit patterns [n_kv_heads][n_tok][head_dim/32].
 *  - V q8_0 codes: int8 [n_kv_heads][n_tok][head_dim].
 *  - V q4_0 codes: uint8 [n_kv_heads][n_tok][head_dim/2]; in each 32-block,
 *    byte j holds element j in its low nibble and element j+16 in its high
 *    nibble.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_QBLK 32
#define ORC_VT_Q4_0 0
#define ORC_VT_Q8_0 1

/* ---------------------------------------------------------------- fp16 -- */

/* IEEE-754 binary16 -> double (exact). */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24);               /* subnormal: man * 2^-24 */
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + man), ex - 25);  /* (1.man) * 2^(ex-15) */
    return sign ? -v : v;
}

/* double -> IEEE-754 binary16, round to nearest, ties to even. */
uint16_t orc_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x))
        return 0x7e00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: integer multiple of 2^-24; 1024 lands on the
         * smallest normal, whose encoding is the same integer */
        double m = nearbyint(ldexp(a, 24));
        return sign | (uint16_t)m;
    }
    int e2;
    double f = frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                    /* a = (2f) * 2^e, 2f in [1, 2) */
    double m = nearbyint(f * 2048.0);  /* 11-bit significand, exact scaling */
    if (m == 2048.0) {
        m = 1024.0;
        e += 1;
    }
    if (e > 15)
        return sign | 0x7c00;          /* overflow -> inf */
    return sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)m - 1024);
}

/* ------------------------------------------------------------ quantizers -- */

static double orc_absmax(const uint16_t *x, int n)
{
    double a = 0.0;
    for (int i = 0; i < n; ++i) {
        double v = fabs(orc_f16_to_f64(x[i]));
        if (v > a)
            a = v;
    }
    return a;
}

/* One 32-element block -> int8 codes + fp16 scale (K, Q and q8_0 V rule). */
void orc_quant_i8_block(const uint16_t *x, int8_t *codes, uint16_t *scale)
{
    double a = orc_absmax(x, ORC_QBLK);
    uint16_t s16 = orc_f64_to_f16(a / 127.0);
    double s = orc_f16_to_f64(s16);
    *scale = s16;
    for (int i = 0; i < ORC_QBLK; ++i) {
        if (s == 0.0) {
            codes[i] = 0;
            continue;
        }
        double c = round(orc_f16_to_f64(x[i]) / s);   /* half away from zero */
        if (c > 127.0) c = 127.0;
        if (c < -127.0) c = -127.0;
        codes[i] = (int8_t)c;
    }
}

/* One 32-element block -> q4_0: 16 packed bytes + fp16 scale. */
void orc_quant_q4_0_block(const uint16_t *x, uint8_t *packed, uint16_t *scale)
{
    double a = orc_absmax(x, ORC_QBLK);
    uint16_t d16 = orc_f64_to_f16(a / 8.0);
    double d = orc_f16_to_f64(d16);
    int q[ORC_QBLK];
    *scale = d16;
    for (int i = 0; i < ORC_QBLK; ++i) {
        if (d == 0.0) {
            q[i] = 8;
            continue;
        }
        double c = round(orc_f16_to_f64(x[i]) / d) + 8.0;
        if (c > 15.0) c = 15.0;
        if (c < 0.0) c = 0.0;
        q[i] = (int)c;
    }
    for (int j = 0; j < ORC_QBLK / 2; ++j)
        packed[j] = (uint8_t)((q[j] & 0xf) | ((q[j + 16] & 0xf) << 4));
}

/* Dequantized value of element j of one V block. */
static double orc_v_deq(int v_type, const uint8_t *vq_blk, double scale, int j)
{
    if (v_type == ORC_VT_Q4_0) {
        uint8_t byte = vq_blk[j % 16];
        int q = (j < 16) ? (byte & 0xf) : (byte >> 4);
        return (double)(q - 8) * scale;
    }
    return (double)((const int8_t *)vq_blk)[j] * scale;
}

/*
 * Quantize n_tok new tokens of K and V (fp16 bits, token-major
 * [n_tok][n_kv_heads][head_dim]) into the head-major cache layout described at
 * the top of this file.
 */
int orc_quantize_kv(int n_tok, int n_kv_heads, int head_dim, int v_type,
                    const uint16_t *k16, const uint16_t *v16,
                    int8_t *kq, uint16_t *ks, uint8_t *vq, uint16_t *vs)
{
    if (head_dim % ORC_QBLK || (v_type != ORC_VT_Q4_0 && v_type != ORC_VT_Q8_0))
        return 1;
    int nb = head_dim / ORC_QBLK;
    int vbytes = (v_type == ORC_VT_Q4_0) ? head_dim / 2 : head_dim;
    int vblk = (v_type == ORC_VT_Q4_0) ? 16 : 32;
    for (int t = 0; t < n_tok; ++t)
        for (int h = 0; h < n_kv_heads; ++h) {
            const uint16_t *kx = k16 + ((size_t)t * n_kv_heads + h) * head_dim;
            const uint16_t *vx = v16 + ((size_t)t * n_kv_heads + h) * head_dim;
            size_t row = (size_t)h * n_tok + t;
            for (int b = 0; b < nb; ++b) {
                orc_quant_i8_block(kx + b * ORC_QBLK, kq + row * head_dim + b * ORC_QBLK,
                                   ks + row * nb + b);
                if (v_type == ORC_VT_Q4_0)
                    orc_quant_q4_0_block(vx + b * ORC_QBLK, vq + row * vbytes + b * vblk,
                                         vs + row * nb + b);
                else
                    orc_quant_i8_block(vx + b * ORC_QBLK,
                                       (int8_t *)(vq + row * vbytes + b * vblk),
                                       vs + row * nb + b);
            }
        }
    return 0;
}

/*
 * Softmax over the scores s[0..n-1] of one row (two passes: max, then sum)
 * and the weighted sum of the dequantized V rows of kv head h into o
 * (head_dim values, zeroed by the caller).  Returns lse = m + ln(sum).
 */
static double orc_attend(int n, const double *s, int L, int h, int head_dim, int v_type,
                         const uint8_t *vq, const uint16_t *vs, double *o)
{
    int nb = head_dim / ORC_QBLK;
    int vbytes = (v_type == ORC_VT_Q4_0) ? head_dim / 2 : head_dim;
    int vblk = (v_type == ORC_VT_Q4_0) ? 16 : 32;
    double m = -INFINITY;
    for (int t = 0; t < n; ++t)
        if (s[t] > m)
            m = s[t];
    double z = 0.0;
    for (int t = 0; t < n; ++t) {
        double p = exp(s[t] - m);
        size_t row = (size_t)h * L + t;
        z += p;
        for (int b = 0; b < nb; ++b) {
            const uint8_t *vb = vq + row * vbytes + b * vblk;
            double d = orc_f16_to_f64(vs[row * nb + b]);
            for (int j = 0; j < ORC_QBLK; ++j)
                o[b * ORC_QBLK + j] += p * orc_v_deq(v_type, vb, d, j);
        }
    }
    for (int j = 0; j < head_dim; ++j)
        o[j] /= z;
    return m + log(z);
}

/*
 * Decode attention for ONE sequence of length L whose quantized cache is held
 * in the layout above with n_tok = L (positions 0..L-1).
 *
 *  q16      fp16 bits [t_q][n_q_heads][head_dim]; the t_q query tokens are the
 *           last t_q positions of the sequence.
 *  head_map [n_q_heads] kv head of each query head.
 *  causal   if nonzero, query token i sees positions 0 .. L - t_q + i;
 *           otherwise every query token sees 0 .. L-1.
 *  out      fp64 [t_q][n_q_heads][head_dim]; lse fp64 [t_q][n_q_heads]
 *           (natural log of sum_t exp(score_t), score including sm_scale).
 *           A row that sees no position gets out = 0 and lse = -inf.
 *  q_codes / q_scales / scores: optional (NULL to skip) -- the Q codes
 *           [t_q][n_q_heads][head_dim], Q scales [t_q][n_q_heads][head_dim/32]
 *           and the exact per-block integer dots I [t_q][n_q_heads][L][nb]
 *           (positions a row does not see are left untouched).
 *  row_mask optional [t_q*n_q_heads]: rows with 0 are skipped.
 */
int orc_decode_seq(int L, int n_kv_heads, int head_dim, int v_type,
                   const int8_t *kq, const uint16_t *ks,
                   const uint8_t *vq, const uint16_t *vs,
                   int t_q, int n_q_heads, const int32_t *head_map, int causal,
                   double sm_scale, const uint16_t *q16,
                   double *out, double *lse,
                   int8_t *q_codes, uint16_t *q_scales, int64_t *scores,
                   const uint8_t *row_mask, int n_threads)
{
    if (head_dim % ORC_QBLK || head_dim > 1024 || L < 0 || t_q < 1)
        return 1;
    int nb = head_dim / ORC_QBLK;
    int n_rows = t_q * n_q_heads;
    for (int h = 0; h < n_q_heads; ++h)
        if (head_map[h] < 0 || head_map[h] >= n_kv_heads)
            return 2;
    if (n_threads < 1)
        n_threads = 1;

#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
    for (int r = 0; r < n_rows; ++r) {
        if (row_mask && !row_mask[r])
            continue;
        int i = r / n_q_heads;
        int hq = r % n_q_heads;
        int h = head_map[hq];
        int8_t qc[1024];
        double sq[32];
        uint16_t sq16[32];
        const uint16_t *qx = q16 + (size_t)r * head_dim;
        for (int b = 0; b < nb; ++b) {
            orc_quant_i8_block(qx + b * ORC_QBLK, qc + b * ORC_QBLK, &sq16[b]);
            sq[b] = orc_f16_to_f64(sq16[b]);
        }
        if (q_codes)
            memcpy(q_codes + (size_t)r * head_dim, qc, head_dim);
        if (q_scales)
            memcpy(q_scales + (size_t)r * nb, sq16, nb * sizeof(uint16_t));

        int last = causal ? L - t_q + i : L - 1;   /* inclusive */
        double *o = out + (size_t)r * head_dim;
        for (int j = 0; j < head_dim; ++j)
            o[j] = 0.0;
        if (last < 0) {
            lse[r] = -INFINITY;
            continue;
        }
        int n = last + 1;
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        /* scores */
        for (int t = 0; t < n; ++t) {
            size_t row = (size_t)h * L + t;
            const int8_t *kc = kq + row * head_dim;
            double acc = 0.0;
            for (int b = 0; b < nb; ++b) {
                int64_t I = 0;
                for (int j = 0; j < ORC_QBLK; ++j)
                    I += (int64_t)qc[b * ORC_QBLK + j] * (int64_t)kc[b * ORC_QBLK + j];
                if (scores)
                    scores[((size_t)r * L + t) * nb + b] = I;
                acc += (double)I * sq[b] * orc_f16_to_f64(ks[row * nb + b]);
            }
            s[t] = sm_scale * acc;
        }
        lse[r] = orc_attend(n, s, L, h, head_dim, v_type, vq, vs, o);
        free(s);
    }
    return 0;
}

/*
 * The same decode attention with K kept as fp16 values (k16: fp16 bits
 * [n_kv_heads][L][head_dim]) and Q not quantized: the score of position t is
 * sm_scale * sum_j q_j * k_tj over the fp16 values, in fp64.  V, the causal
 * tail, out and lse as in orc_decode_seq.
 */
int orc_decode_seq_f16k(int L, int n_kv_heads, int head_dim, int v_type, const uint16_t *k16,
                        const uint8_t *vq, const uint16_t *vs,
                        int t_q, int n_q_heads, const int32_t *head_map, int causal,
                        double sm_scale, const uint16_t *q16, double *out, double *lse,
                        const uint8_t *row_mask, int n_threads)
{
    if (head_dim % ORC_QBLK || head_dim > 1024 || L < 0 || t_q < 1)
        return 1;
    int n_rows = t_q * n_q_heads;
    for (int h = 0; h < n_q_heads; ++h)
        if (head_map[h] < 0 || head_map[h] >= n_kv_heads)
            return 2;
    if (n_threads < 1)
        n_threads = 1;

#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
    for (int r = 0; r < n_rows; ++r) {
        if (row_mask && !row_mask[r])
            continue;
        int i = r / n_q_heads;
        int h = head_map[r % n_q_heads];
        double qv[1024];
        const uint16_t *qx = q16 + (size_t)r * head_dim;
        for (int j = 0; j < head_dim; ++j)
            qv[j] = orc_f16_to_f64(qx[j]);
        int last = causal ? L - t_q + i : L - 1;   /* inclusive */
        double *o = out + (size_t)r * head_dim;
        for (int j = 0; j < head_dim; ++j)
            o[j] = 0.0;
        if (last < 0) {
            lse[r] = -INFINITY;
            continue;
        }
        int n = last + 1;
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        for (int t = 0; t < n; ++t) {
            const uint16_t *kx = k16 + ((size_t)h * L + t) * head_dim;
            double acc = 0.0;
            for (int j = 0; j < head_dim; ++j)
                acc += qv[j] * orc_f16_to_f64(kx[j]);
            s[t] = sm_scale * acc;
        }
        lse[r] = orc_attend(n, s, L, h, head_dim, v_type, vq, vs, o);
        free(s);
    }
    return 0;
}
