/*
 * gqa_oracle.c -- plain, slow, fp64 CPU oracle for one GQA decode step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, and where the pages define it:
 *
 *  - oracle_gqa_decode: grouped-query attention for the new token(s) of each sequence,
 *    "分组查询注意力 (GQA)", section 技术原理, steps 2-4 and the attention
 *    equation softmax(Q_group K_g^T / sqrt(d_k)) V_g. Query head h uses KV head
 *    g = h / (H/K) (the [K, H/K] reshape of step 2; the head mapping j = i // 4
 *    of the KV-cache essay's GQA section is the H/K = 4 case). The softmax is
 *    the plain definition: subtract the maximum score, exponentiate, divide by
 *    the sum. The cache is dense [B, S_max, K, d] (the [batch, seq,
 *    num_kv_heads, head_dim] index of "LLM 推理性能优化实战", section 7.3).
 *    An empty context (length 0) yields a zero output (reading: the pages never
 *    decode an empty sequence).
 *    Two widenings of the same definition, each only a change of the attended
 *    token range:
 *      * T >= 1 new tokens per sequence (speculative verification, "LLM 推理性能
 *        优化实战" section 14.2; chunked prefill mixed with decode, section
 *        11.7): the T queries of sequence b sit at positions lens[b]-T .. lens[b]-1
 *        (lens counts the new tokens) and query i attends positions
 *        0 .. lens[b]-T+i, causal among the new tokens. A query whose position
 *        is negative (lens[b] < T) attends nothing and yields zeros.
 *      * a sliding window W > 0 (section 6.4.1: only the most recent N tokens
 *        are attended): each query attends the last W positions up to and
 *        including its own. W = 0 is full attention.
 *
 *  - oracle_quantize_int8: symmetric int8 quantisation with one scale per
 *    (token, kv-head) row ("LLM 推理性能优化实战", section 15.1: symmetric range
 *    [-127, 127]; sections 15.2 and 15.5: per-token scales for the KV cache).
 *    The pages leave rounding and scale precision open; the reading used here:
 *      amax = max_i |x_i|                     (fp32)
 *      s    = fp16_rne(min(amax / 127, 65504)) (fp32 IEEE division, then RNE)
 *      q_i  = 0 if s == 0 else clamp(rint(x_i / s), -127, 127)
 *    with fp32 IEEE division and round-half-to-even. Dequantisation is q_i * s
 *    evaluated exactly in fp64.
 *
 *  - oracle_quantize_int4: the INT4 KV cache of "LLM 推理性能优化实战" section
 *    15.5 (KV quantised to INT4; section 15.3 lists INT4 among the low-precision
 *    formats) with the same symmetric per-(token, kv-head) rule, range [-7, 7]:
 *      s = fp16_rne(min(amax / 7, 65504)),  q_i = clamp(rint(x_i / s), -7, 7).
 *    (Reading: the symmetric range of section 15.1 narrowed to four bits, -8
 *    unused so the range stays symmetric.) Two codes share a byte, element 2j
 *    in the low nibble, as two's-complement nibbles.
 *
 *  - oracle_quantize_int4_channels: the KIVI-style K cache named in "LLM 推理性能
 *    优化实战" section 15.5 (K quantised per channel, V per token, both to
 *    INT4; section 15.2 describes per-channel quantisation as one scale per
 *    channel). Reading: a channel's group is the tokens one 16-token cache block
 *    holds for one kv-head (the unit the paged cache stores), with the same
 *    symmetric rule as the per-token codes, applied down each channel:
 *      amax_i = max over the block's n present tokens t of |x[t][i]|,
 *      s_i = fp16_rne(min(amax_i / 7, 65504)),  q[t][i] = clamp(rint(x[t][i] / s_i), -7, 7).
 *    A block that is still filling is quantised over the tokens it holds so
 *    far, and again, from the unquantised values, each time a token joins it.
 *
 *  - oracle_quantize_fp8 / oracle_f32_to_e4m3 / oracle_e4m3_to_f64: the FP8
 *    (E4M3) KV cache named among the KV quantisation options of "LLM 推理性能优化实战"
 *    section 15.5 (FP8 E4M3/E5M2 for long-tailed K/V): per-(token, kv-head) fp16
 *    scale s = fp16_rne(min(amax/448, 65504)), codes = nearest-even e4m3 of x/s,
 *    saturated to +-448. Decoding is exact in fp64.
 *
 *  - oracle_f32_to_f16_bits / oracle_f16_bits_to_f32: IEEE 754 binary16
 *    conversion with round-to-nearest-even, written from the format's
 *    definition (1 sign, 5 exponent, 10 fraction bits, bias 15).
 *
 * Build: plain C99, -O2 -fno-fast-math -ffp-contract=off, pthreads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------- */
/* IEEE binary16 conversions                                                 */
/* ------------------------------------------------------------------------- */

uint16_t oracle_f32_to_f16_bits(float f)
{
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7fffffffu;

    if (ax >= 0x7f800000u)                       /* inf or NaN */
        return (uint16_t)(sign | 0x7c00u | (ax > 0x7f800000u ? 0x0200u : 0u));

    int32_t e32 = (int32_t)(ax >> 23);           /* biased fp32 exponent */
    uint32_t frac = ax & 0x007fffffu;
    if (e32 == 0)                                /* fp32 subnormal: far below fp16 range */
        return sign;
    uint32_t mant = frac | 0x00800000u;          /* 24-bit significand, value = mant * 2^(e32-150) */
    int32_t e16 = e32 - 127 + 15;                /* biased fp16 exponent if normal */

    if (e16 >= 31)                               /* at or above 2^16: overflow */
        return (uint16_t)(sign | 0x7c00u);

    if (e16 <= 0) {
        /* fp16 subnormal: value / 2^-24 = mant * 2^(e32 - 126); shift right by 126 - e32 */
        int32_t shift = 126 - e32;               /* >= 14 here */
        if (shift > 24)
            return sign;                         /* below half the smallest subnormal */
        uint32_t q = mant >> shift;
        uint32_t rem = mant & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        if (rem > half || (rem == half && (q & 1u)))
            q += 1u;                             /* may carry into the smallest normal: still correct */
        return (uint16_t)(sign | q);
    }

    /* normal: keep 10 of the 23 fraction bits, round to nearest even */
    uint32_t q = ((uint32_t)e16 << 10) | (frac >> 13);
    uint32_t rem = frac & 0x1fffu;
    if (rem > 0x1000u || (rem == 0x1000u && (q & 1u)))
        q += 1u;                                 /* carry may reach the exponent, or inf at 65520 */
    return (uint16_t)(sign | q);
}

float oracle_f16_bits_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1fu;
    uint32_t frac = h & 0x3ffu;
    float out;
    if (e == 0) {
        /* zero or subnormal: frac * 2^-24, exact in fp32 */
        out = (float)frac * (1.0f / 16777216.0f);
        if (sign) out = -out;
        return out;
    }
    uint32_t bits;
    if (e == 31)
        bits = sign | 0x7f800000u | (frac << 13);
    else
        bits = sign | ((e - 15 + 127) << 23) | (frac << 13);
    memcpy(&out, &bits, sizeof out);
    return out;
}

/* ------------------------------------------------------------------------- */
/* int8 KV quantisation, one scale per row                                   */
/* ------------------------------------------------------------------------- */

/* Symmetric integer quantisation to [-qmax, qmax] of `groups` groups of
 * `members` values with one fp16 scale per group (the rule above, with 127
 * replaced by qmax). Member m of group g sits at x[g*gstride + m*mstride], and
 * its code goes to the same index of `codes`. Rows of a [rows, d] array are
 * (groups = rows, gstride = d, members = d, mstride = 1); its channels are
 * (groups = d, gstride = 1, members = rows, mstride = d). */
static void quantize_symmetric(const float *x, int64_t groups, int64_t gstride, int32_t members,
                               int64_t mstride, float qmax, int8_t *codes, uint16_t *scale_bits)
{
    for (int64_t g = 0; g < groups; ++g) {
        const int64_t base = g * gstride;
        float amax = 0.0f;
        for (int32_t m = 0; m < members; ++m) {
            float a = fabsf(x[base + m * mstride]);
            if (a > amax) amax = a;
        }
        volatile float s32 = amax / qmax;        /* IEEE fp32 division */
        float s = s32;
        if (s > 65504.0f) s = 65504.0f;
        uint16_t sb = oracle_f32_to_f16_bits(s);
        float sf = oracle_f16_bits_to_f32(sb);
        scale_bits[g] = sb;
        for (int32_t m = 0; m < members; ++m) {
            int32_t q = 0;
            if (sf != 0.0f) {
                volatile float t = x[base + m * mstride] / sf;   /* IEEE fp32 division */
                float rq = rintf(t);             /* round half to even (default mode) */
                if (rq > qmax) rq = qmax;
                if (rq < -qmax) rq = -qmax;
                q = (int32_t)rq;
            }
            codes[base + m * mstride] = (int8_t)q;
        }
    }
}

void oracle_quantize_int8(const float *x, int64_t rows, int32_t d,
                          int8_t *codes, uint16_t *scale_bits)
{
    quantize_symmetric(x, rows, d, d, 1, 127.0f, codes, scale_bits);
}

/* Codes in [-7, 7], one per int8 (packing two per byte is the caller's). */
void oracle_quantize_int4(const float *x, int64_t rows, int32_t d,
                          int8_t *codes, uint16_t *scale_bits)
{
    quantize_symmetric(x, rows, d, d, 1, 7.0f, codes, scale_bits);
}

/* One block's [n, d] K values -> codes [n, d] in [-7, 7] and d channel scales. */
void oracle_quantize_int4_channels(const float *x, int32_t n, int32_t d,
                                   int8_t *codes, uint16_t *scale_bits)
{
    quantize_symmetric(x, d, 1, n, d, 7.0f, codes, scale_bits);
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 (the "fn" variant: no infinities, max 448) and its quantisation  */
/* ------------------------------------------------------------------------- */

/* Value of an e4m3 code: sign bit, 4 exponent bits (bias 7), 3 fraction bits;
 * exponent 0 is subnormal (2^-6 * f/8); code S.1111.111 is NaN. */
double oracle_e4m3_to_f64(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 15, f = code & 7;
    if (e == 15 && f == 7) return NAN;
    double v = e == 0 ? ldexp(f / 8.0, -6) : ldexp(1.0 + f / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest e4m3 code to a finite float, ties to the even code, magnitudes
 * beyond 448 saturated to 448 (the reading of "round to nearest even,
 * saturate to finite"). Brute force over the 127 non-negative finite codes. */
uint8_t oracle_f32_to_e4m3(float x)
{
    double a = fabs((double)x);
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 0x7e; ++c) {
        double d = fabs(oracle_e4m3_to_f64((uint8_t)c) - a);
        if (d < bd || (d == bd && (c & 1) == 0)) { bd = d; best = c; }
    }
    if (a >= 448.0) best = 0x7e;
    return (uint8_t)(best | (signbit(x) ? 0x80 : 0));
}

/* Per-row FP8 quantisation with an fp16 scale (same rule as int8 with the
 * code range of e4m3):
 *   s = fp16_rne(min(amax / 448, 65504)); code_i = s == 0 ? 0 : e4m3(x_i / s). */
void oracle_quantize_fp8(const float *x, int64_t rows, int32_t d, uint8_t *codes,
                         uint16_t *scale_bits)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * (int64_t)d;
        float amax = 0.0f;
        for (int32_t i = 0; i < d; ++i) {
            float a = fabsf(xr[i]);
            if (a > amax) amax = a;
        }
        volatile float s32 = amax / 448.0f;
        float s = s32;
        if (s > 65504.0f) s = 65504.0f;
        uint16_t sb = oracle_f32_to_f16_bits(s);
        float sf = oracle_f16_bits_to_f32(sb);
        scale_bits[r] = sb;
        for (int32_t i = 0; i < d; ++i) {
            uint8_t c = 0;
            if (sf != 0.0f) {
                volatile float t = xr[i] / sf;
                c = oracle_f32_to_e4m3(t);
            }
            codes[r * (int64_t)d + i] = c;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* GQA decode attention, fp64                                                */
/* ------------------------------------------------------------------------- */

typedef struct {
    const double *q, *k, *v;
    const int32_t *lens;
    int32_t B, T, H, K, d, S_max, window;
    double scale;
    double *out;
    int64_t next;              /* next (b, i, h) work item, shared */
    pthread_mutex_t lock;
} decode_job;

/* One (b, i, h) output row (query i of sequence b, head h), straight from the
 * definition over the attended positions [lo, hi). */
static void decode_one(const decode_job *J, int32_t b, int32_t i, int32_t h, double *s)
{
    const int32_t G = J->H / J->K;
    const int32_t g = h / G;                     /* query head h reads KV head h / (H/K) */
    const int32_t d = J->d, K = J->K;
    const int64_t row = ((int64_t)b * J->T + i) * J->H + h;
    const double *qh = J->q + row * d;
    double *o = J->out + row * d;

    for (int32_t e = 0; e < d; ++e) o[e] = 0.0;
    const int32_t hi = J->lens[b] - J->T + i + 1;          /* own position + 1 */
    if (hi <= 0) return;
    const int32_t lo = (J->window > 0 && hi > J->window) ? hi - J->window : 0;

    /* scores s_t = scale * <q_h, k_{t,g}> */
    double mx = -INFINITY;
    for (int32_t t = lo; t < hi; ++t) {
        const double *kt = J->k + (((int64_t)b * J->S_max + t) * K + g) * d;
        double acc = 0.0;
        for (int32_t e = 0; e < d; ++e) acc += qh[e] * kt[e];
        s[t] = J->scale * acc;
        if (s[t] > mx) mx = s[t];
    }
    /* softmax weights and the weighted sum of values */
    double denom = 0.0;
    for (int32_t t = lo; t < hi; ++t) {
        double w = exp(s[t] - mx);
        denom += w;
        const double *vt = J->v + (((int64_t)b * J->S_max + t) * K + g) * d;
        for (int32_t e = 0; e < d; ++e) o[e] += w * vt[e];
    }
    for (int32_t e = 0; e < d; ++e) o[e] /= denom;
}

static void *decode_worker(void *arg)
{
    decode_job *J = (decode_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->S_max > 0 ? J->S_max : 1));
    if (!s) return (void *)1;
    const int64_t total = (int64_t)J->B * J->T * J->H;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t it = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (it >= total) break;
        const int64_t bi = it / J->H;
        decode_one(J, (int32_t)(bi / J->T), (int32_t)(bi % J->T), (int32_t)(it % J->H), s);
    }
    free(s);
    return NULL;
}

int oracle_num_cpus(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* q [B,T,H,d], k/v [B,S_max,K,d], lens [B] (new tokens included), out
 * [B,T,H,d]; all fp64, host memory. window 0 = full attention. nthreads <= 0
 * uses every online CPU. Returns 0, or -1 on bad arguments, -2 when a thread
 * or buffer could not be created. */
int oracle_gqa_decode(const double *q, const double *k, const double *v,
                      const int32_t *lens, int32_t B, int32_t T, int32_t H, int32_t K,
                      int32_t d, int32_t S_max, int32_t window, double scale, double *out,
                      int32_t nthreads)
{
    if (B < 0 || T <= 0 || H <= 0 || K <= 0 || d <= 0 || S_max < 0 || H % K != 0 || window < 0)
        return -1;
    for (int32_t b = 0; b < B; ++b)
        if (lens[b] < 0 || lens[b] > S_max) return -1;
    decode_job J = {q, k, v, lens, B, T, H, K, d, S_max, window, scale, out, 0,
                    PTHREAD_MUTEX_INITIALIZER};
    int32_t nt = nthreads > 0 ? nthreads : oracle_num_cpus();
    int64_t items = (int64_t)B * T * H;
    if (nt > items) nt = (int32_t)(items > 0 ? items : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!th) return -2;
    /* workers pull items until none are left, so any number of started
       threads completes the whole job */
    int32_t started = 0, rc = 0;
    for (; started < nt; ++started)
        if (pthread_create(&th[started], NULL, decode_worker, &J) != 0) break;
    for (int32_t i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret) rc = -2;
    }
    if (started == 0) {                          /* no thread could start: run inline */
        void *ret = decode_worker(&J);
        rc = ret ? -2 : 0;
    }
    free(th);
    pthread_mutex_destroy(&J.lock);
    return rc;
}
