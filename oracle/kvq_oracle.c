/*
 * kvq_oracle.c -- plain, slow, single-threaded CPU oracle for the low-bit KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library.  It shares no
 * code, header, table or helper with the CUDA path (bit_kv_cache_gb300/csrc).
 *
 * What it computes, and where the pages define it:
 *   - min-max asymmetric quantization of one group: scale = (max-min)/(2^b-1),
 *     code = clamp(round((x-min)/scale), 0, 2^b-1), dequant = code*scale+min
 *     (KIVI notes "KV Cache 量化算子：KIVI", Step 1, the quant_kcache listing; the
 *     step is written (max-min)/2^N in the prose, the listing and the rest of
 *     the page use 2^b-1, which is taken here);
 *   - keys per channel over groups of G tokens, values per token over groups of
 *     Gv channels (same page, Step 1);
 *   - pack_tensor: 32/b codes per int32, element j of a word at bit b*j, least
 *     significant first (same page, Step 2; the worked example "logical column
 *     19 -> word 1, shift 6" in Step 4);
 *   - Kitty's channel-wise precision boost: per page, score_d = sum_t |k_{t,d}|,
 *     the top n_boost channels quantized at 4 bits and the rest at 2 bits; the
 *     page is stored as a dense low 2-bit plane for all channels, a compact high
 *     2-bit plane for the boosted channels and a per-channel boost index with
 *     sentinel n_boost+1 ("Kitty: Accurate and Efficient 2-Bit KV Cache
 *     Quantization ...", Sec. 3.2 and Sec. 4.1, Algorithm 1);
 *   - decode attention softmax(q . K^T / sqrt(d)) . V over the dequantized cache
 *     ("BitDecoding", Sec. II, Fig. 2 caption), accumulated in fp64;
 *   - pre-RoPE keys ("KVQuant 完全拆解", mechanism two): the cache holds keys
 *     before the rotary position embedding; attention dequantizes key t, rotates
 *     channel pair (2i, 2i+1) by the angle t * theta_i, theta_i = base^(-2i/d)
 *     (i = 0 .. d/2-1, the page's R_{theta,m} with its 1-based index shifted), and
 *     only then takes the dot product with the (already rotated) query.  t is the
 *     token's 0-based position in the sequence (sink, packed, residual order).
 *
 * Precision (the pages leave it open; this is the reading taken): min/max are
 * exact fp16 comparisons, the scale is computed in fp32 then rounded to fp16,
 * the code is computed in fp32 with IEEE division and round-half-to-even,
 * a zero (or fp16-underflowing) scale gives code 0, a -0.0 minimum (or maximum)
 * is taken as +0.0, so the stored min and scale never carry a negative zero.  Dequantization and attention use fp64.
 *
 * Build: cc -O2 -fno-fast-math -ffp-contract=off -shared -fPIC.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary32, written from the format definition.      */
/* ------------------------------------------------------------------------ */

float kvq_or_h2f(uint16_t h)
{
    unsigned e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);                    /* zero / subnormal */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(m | 0x400u), (int)e - 25); /* normal */
    return (h & 0x8000u) ? -v : v;
}

uint16_t kvq_or_f2h(float f)
{
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    float a = fabsf(f);
    if (isnan(f))
        return (uint16_t)(sign | 0x7e00u);
    if (isinf(f))
        return (uint16_t)(sign | 0x7c00u);
    if (a < ldexpf(1.0f, -14)) {
        /* subnormal grid of 2^-24; the scaling is exact, rintf rounds half to even.
           A result of 1024 is the bit pattern of the smallest normal, 2^-14. */
        float m = rintf(a * ldexpf(1.0f, 24));
        return (uint16_t)(sign | (uint16_t)m);
    }
    int e;
    frexpf(a, &e);
    e -= 1;                                 /* 2^e <= a < 2^(e+1) */
    float m = rintf(ldexpf(a, 10 - e));     /* significand on an 11-bit grid */
    if (m == 2048.0f) {
        m = 1024.0f;
        e += 1;
    }
    if (e > 15)
        return (uint16_t)(sign | 0x7c00u);  /* overflow to infinity */
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(m - 1024.0f));
}

/* ------------------------------------------------------------------------ */
/* The quantizer of one group.                                              */
/* ------------------------------------------------------------------------ */

/* Quantize n fp16 values x[i*stride] with max_int = 2^b - 1.
 * Writes the fp16 scale and min and one code per element. */
void kvq_or_quant_group(const uint16_t *x, long stride, int n, int max_int,
                        uint16_t *scale_out, uint16_t *min_out, uint8_t *codes)
{
    float mn = kvq_or_h2f(x[0]), mx = mn;
    for (int i = 1; i < n; i++) {
        float v = kvq_or_h2f(x[(long)i * stride]);
        if (v < mn)
            mn = v;
        if (v > mx)
            mx = v;
    }
    if (mn == 0.0f)
        mn = 0.0f;                      /* store -0.0 as +0.0 */
    if (mx == 0.0f)
        mx = 0.0f;                      /* so an all-zero group has scale +0.0 */
    float range = mx - mn;              /* fp32, round to nearest */
    float s32 = range / (float)max_int; /* fp32 IEEE division */
    uint16_t s16 = kvq_or_f2h(s32);     /* scale kept in fp16 */
    float s = kvq_or_h2f(s16);
    *scale_out = s16;
    *min_out = kvq_or_f2h(mn);
    for (int i = 0; i < n; i++) {
        if (s == 0.0f) {                /* zero range or underflowed scale */
            codes[i] = 0;
            continue;
        }
        float d = kvq_or_h2f(x[(long)i * stride]) - mn;
        float v = d / s;
        float r = rintf(v);             /* round half to even */
        if (r < 0.0f)
            r = 0.0f;
        if (r > (float)max_int)
            r = (float)max_int;
        codes[i] = (uint8_t)r;
    }
}

/* ------------------------------------------------------------------------ */
/* KIVI keys: per channel, groups of G tokens, packed along tokens.         */
/* ------------------------------------------------------------------------ */

/* k:       fp16 [U][L][D] (U = B*H_kv units), quantize tokens [t0, t0+T).
 * codes:   int32 [U][T/fpi][D]  -- pack_tensor along the token axis
 * meta:    fp16  [U][T/G][D][2] -- (scale, min) per channel per group */
void kvq_or_quant_k(const uint16_t *k, int U, long L, int D, int G, int bits,
                    long t0, long T, int32_t *codes, uint16_t *meta)
{
    int fpi = 32 / bits, max_int = (1 << bits) - 1;
    long n_words = T / fpi;
    uint8_t *c = (uint8_t *)malloc((size_t)G);
    for (int u = 0; u < U; u++) {
        const uint16_t *ku = k + (long)u * L * D;
        int32_t *cu = codes + (long)u * n_words * D;
        memset(cu, 0, sizeof(int32_t) * (size_t)(n_words * D));
        for (long grp = 0; grp < T / G; grp++) {
            for (int d = 0; d < D; d++) {
                uint16_t *mt = meta + (((long)u * (T / G) + grp) * D + d) * 2;
                kvq_or_quant_group(ku + (t0 + grp * G) * D + d, D, G, max_int,
                                   &mt[0], &mt[1], c);
                for (int i = 0; i < G; i++) {
                    long tau = grp * G + i;  /* token index within the packed region */
                    uint32_t w = (uint32_t)cu[(tau / fpi) * D + d];
                    w |= (uint32_t)c[i] << (bits * (tau % fpi));
                    cu[(tau / fpi) * D + d] = (int32_t)w;
                }
            }
        }
    }
    free(c);
}

/* ------------------------------------------------------------------------ */
/* Values: per token, groups of Gv channels, packed along channels.         */
/* ------------------------------------------------------------------------ */

/* v:       fp16 [U][L][D], quantize tokens [t0, t0+T).
 * codes:   int32 [U][T][D/fpi]  -- pack_tensor along the channel axis
 * meta:    fp16  [U][T][D/Gv][2] */
void kvq_or_quant_v(const uint16_t *v, int U, long L, int D, int Gv, int bits,
                    long t0, long T, int32_t *codes, uint16_t *meta)
{
    int fpi = 32 / bits, max_int = (1 << bits) - 1;
    uint8_t *c = (uint8_t *)malloc((size_t)Gv);
    for (int u = 0; u < U; u++) {
        for (long tau = 0; tau < T; tau++) {
            const uint16_t *row = v + ((long)u * L + t0 + tau) * D;
            int32_t *cw = codes + ((long)u * T + tau) * (D / fpi);
            memset(cw, 0, sizeof(int32_t) * (size_t)(D / fpi));
            for (int gv = 0; gv < D / Gv; gv++) {
                uint16_t *mt = meta + (((long)u * T + tau) * (D / Gv) + gv) * 2;
                kvq_or_quant_group(row + gv * Gv, 1, Gv, max_int, &mt[0], &mt[1], c);
                for (int i = 0; i < Gv; i++) {
                    int d = gv * Gv + i;
                    uint32_t w = (uint32_t)cw[d / fpi];
                    w |= (uint32_t)c[i] << (bits * (d % fpi));
                    cw[d / fpi] = (int32_t)w;
                }
            }
        }
    }
    free(c);
}

/* ------------------------------------------------------------------------ */
/* Kitty keys: per page of G tokens, top-n_boost channels at 4 bits.        */
/* ------------------------------------------------------------------------ */

/* |x| * 2^24 as an exact integer (every finite fp16 magnitude is a multiple of 2^-24). */
static int64_t abs_units(uint16_t h)
{
    unsigned e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    if (e == 0)
        return (int64_t)m;
    return (int64_t)(m | 0x400u) << (e - 1);
}

/* Channel importance of one page: score_d = sum_t |k_{t,d}| (the 1/T of the mean
 * does not change the ranking), exact in units of 2^-24.  Boosted channels are
 * the n_boost largest scores; equal scores go to the lower channel index. */
void kvq_or_kitty_select(const uint16_t *page, int G, int D, int n_boost,
                         int64_t *score, uint8_t *bidx)
{
    for (int d = 0; d < D; d++) {
        score[d] = 0;
        for (int t = 0; t < G; t++)
            score[d] += abs_units(page[(long)t * D + d]);
    }
    int slot = 0;
    for (int d = 0; d < D; d++) {
        int rank = 0;
        for (int e = 0; e < D; e++)
            if (score[e] > score[d] || (score[e] == score[d] && e < d))
                rank++;
        /* slots in ascending channel order; sentinel n_boost+1 when not boosted */
        bidx[d] = (uint8_t)(rank < n_boost ? slot++ : n_boost + 1);
    }
}

/* k:      fp16 [U][L][D], quantize tokens [t0, t0+T) in pages of G tokens.
 * lo:     int32 [U][T/16][D]        low 2 bits of every channel, packed along tokens
 * hi:     int32 [U][T/16][n_boost]  high 2 bits of the boosted channels, slot order
 * bidx:   uint8 [U][T/G][D]         channel -> slot, or n_boost+1
 * meta:   fp16  [U][T/G][D][2] */
void kvq_or_quant_k_kitty(const uint16_t *k, int U, long L, int D, int G, int n_boost,
                          long t0, long T, int32_t *lo, int32_t *hi, uint8_t *bidx,
                          uint16_t *meta)
{
    long nw = T / 16;
    uint8_t *c = (uint8_t *)malloc((size_t)G);
    int64_t *score = (int64_t *)malloc(sizeof(int64_t) * (size_t)D);
    for (int u = 0; u < U; u++) {
        const uint16_t *ku = k + (long)u * L * D;
        int32_t *lu = lo + (long)u * nw * D;
        int32_t *hu = hi + (long)u * nw * n_boost;
        memset(lu, 0, sizeof(int32_t) * (size_t)(nw * D));
        if (n_boost)
            memset(hu, 0, sizeof(int32_t) * (size_t)(nw * n_boost));
        for (long grp = 0; grp < T / G; grp++) {
            const uint16_t *page = ku + (t0 + grp * G) * D;
            uint8_t *bi = bidx + ((long)u * (T / G) + grp) * D;
            kvq_or_kitty_select(page, G, D, n_boost, score, bi);
            for (int d = 0; d < D; d++) {
                int boosted = bi[d] < n_boost;   /* slot index (0-based) */
                uint16_t *mt = meta + (((long)u * (T / G) + grp) * D + d) * 2;
                kvq_or_quant_group(page + d, D, G, boosted ? 15 : 3, &mt[0], &mt[1], c);
                for (int i = 0; i < G; i++) {
                    long tau = grp * G + i;
                    uint32_t w = (uint32_t)lu[(tau / 16) * D + d];
                    lu[(tau / 16) * D + d] = (int32_t)(w | ((uint32_t)(c[i] & 3u) << (2 * (tau % 16))));
                    if (boosted) {
                        long at = (tau / 16) * n_boost + bi[d];
                        uint32_t h = (uint32_t)hu[at];
                        hu[at] = (int32_t)(h | ((uint32_t)(c[i] >> 2) << (2 * (tau % 16))));
                    }
                }
            }
        }
    }
    free(score);
    free(c);
}

/* ------------------------------------------------------------------------ */
/* Dequantization to fp64 token rows and fp64 attention.                    */
/* ------------------------------------------------------------------------ */

/* One (b, h_kv) sequence of the cache, in the oracle's own layouts.
 * Logical token order: [sink | K packed | K residual] for keys and
 * [sink | V packed | V residual (KIVI) or Q-buffer (Kitty) | local (Kitty)]
 * for values; both orders cover the same L tokens. */
typedef struct {
    int D, G, bits, Gv, n_boost, kitty, vbits;   /* bits: keys, vbits: values */
    long n_sink, T_k, n_kres, T_v, n_vres, n_local, local_head, local_cap;
    const uint16_t *k_sink, *v_sink;   /* [n_sink][D] */
    const int32_t *k_codes;            /* [T_k/fpi][D] (Kitty: low plane, fpi 16) */
    const int32_t *k_hi;               /* [T_k/16][n_boost] */
    const uint8_t *k_bidx;             /* [T_k/G][D] */
    const uint16_t *k_meta;            /* [T_k/G][D][2] */
    const uint16_t *k_res;             /* [n_kres][D] */
    const int32_t *v_codes;            /* [T_v][D/fpi] */
    const uint16_t *v_meta;            /* [T_v][D/Gv][2] */
    const uint16_t *v_res;             /* [n_vres][D] */
    const uint16_t *v_local;           /* [local_cap][D] ring, oldest at local_head */
    double rope_base;                  /* > 0: keys are stored before RoPE with this base */
} kvq_or_seq;

long kvq_or_seq_len(const kvq_or_seq *s)
{
    return s->n_sink + s->T_k + s->n_kres;
}

/* Dequantized keys and values of every token, in logical order, as fp64
 * (dequant = code*scale + min, evaluated in fp64). */
void kvq_or_seq_rows(const kvq_or_seq *s, double *Kh, double *Vh)
{
    int D = s->D;
    long L = kvq_or_seq_len(s);
    int kfpi = s->kitty ? 16 : 32 / s->bits, kbits = s->kitty ? 2 : s->bits;
    int vfpi = 32 / s->vbits, vbits = s->vbits, vmask = (1 << vbits) - 1;
    for (long t = 0; t < L; t++) {
        double *kr = Kh + t * D, *vr = Vh + t * D;
        /* keys */
        if (t < s->n_sink) {
            for (int d = 0; d < D; d++)
                kr[d] = kvq_or_h2f(s->k_sink[t * D + d]);
        } else if (t < s->n_sink + s->T_k) {
            long tau = t - s->n_sink, grp = tau / s->G;
            for (int d = 0; d < D; d++) {
                uint32_t w = (uint32_t)s->k_codes[(tau / kfpi) * D + d];
                int code = (int)((w >> (kbits * (tau % kfpi))) & ((1u << kbits) - 1));
                if (s->kitty && s->n_boost) {
                    int slot = s->k_bidx[grp * D + d];
                    if (slot < s->n_boost) {
                        uint32_t h = (uint32_t)s->k_hi[(tau / 16) * s->n_boost + slot];
                        code |= (int)((h >> (2 * (tau % 16))) & 3u) << 2;
                    }
                }
                const uint16_t *mt = s->k_meta + (grp * D + d) * 2;
                kr[d] = (double)code * (double)kvq_or_h2f(mt[0]) + (double)kvq_or_h2f(mt[1]);
            }
        } else {
            long r = t - s->n_sink - s->T_k;
            for (int d = 0; d < D; d++)
                kr[d] = kvq_or_h2f(s->k_res[r * D + d]);
        }
        /* values */
        if (t < s->n_sink) {
            for (int d = 0; d < D; d++)
                vr[d] = kvq_or_h2f(s->v_sink[t * D + d]);
        } else if (t < s->n_sink + s->T_v) {
            long tau = t - s->n_sink;
            for (int d = 0; d < D; d++) {
                uint32_t w = (uint32_t)s->v_codes[tau * (D / vfpi) + d / vfpi];
                int code = (int)((w >> (vbits * (d % vfpi))) & (uint32_t)vmask);
                const uint16_t *mt = s->v_meta + (tau * (D / s->Gv) + d / s->Gv) * 2;
                vr[d] = (double)code * (double)kvq_or_h2f(mt[0]) + (double)kvq_or_h2f(mt[1]);
            }
        } else if (t < s->n_sink + s->T_v + s->n_vres) {
            long r = t - s->n_sink - s->T_v;
            for (int d = 0; d < D; d++)
                vr[d] = kvq_or_h2f(s->v_res[r * D + d]);
        } else {
            long r = t - s->n_sink - s->T_v - s->n_vres;       /* age rank, oldest first */
            long slot = (s->local_head + r) % s->local_cap;
            for (int d = 0; d < D; d++)
                vr[d] = kvq_or_h2f(s->v_local[slot * D + d]);
        }
    }
}

/* out[h][d] = sum_t softmax_t(q_h . K_t / sqrt(D)) V_t[d] for h < n_heads, in fp64
 * (max-subtracted softmax).  q: [n_heads][D] fp64, K, V: [L][D] fp64. */
void kvq_or_attend(const double *q, int n_heads, const double *K, const double *V,
                   long L, int D, double *out)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double inv = 1.0 / sqrt((double)D);
    for (int h = 0; h < n_heads; h++) {
        const double *qh = q + (long)h * D;
        double m = -INFINITY;
        for (long t = 0; t < L; t++) {
            double acc = 0.0;
            for (int d = 0; d < D; d++)
                acc += qh[d] * K[t * D + d];
            z[t] = acc * inv;
            if (z[t] > m)
                m = z[t];
        }
        double l = 0.0;
        for (long t = 0; t < L; t++) {
            z[t] = exp(z[t] - m);
            l += z[t];
        }
        for (int d = 0; d < D; d++) {
            double acc = 0.0;
            for (long t = 0; t < L; t++)
                acc += z[t] * V[t * D + d];
            out[(long)h * D + d] = acc / l;
        }
    }
    free(z);
}

/* RoPE of rows [0, L) of K [L][D] in place, row i at position t0 + i: channel pair
 * (2j, 2j+1) turns by the angle (t0 + i) * base^(-2j/D) (KVQuant notes, mechanism
 * two; fp64 throughout). */
void kvq_or_rope(double *K, long L, int D, double base, long t0)
{
    for (long i = 0; i < L; i++) {
        double *k = K + i * D;
        double pos = (double)(t0 + i);
        for (int j = 0; j < D / 2; j++) {
            double theta = pow(base, -2.0 * (double)j / (double)D);
            double c = cos(pos * theta), sn = sin(pos * theta);
            double a = k[2 * j], b = k[2 * j + 1];
            k[2 * j] = a * c - b * sn;
            k[2 * j + 1] = a * sn + b * c;
        }
    }
}

/* Convenience: attention of the g query heads that share one (b, h_kv) sequence.
 * q16: fp16 [g][D]; out: fp64 [g][D]; scratch sized internally. */
int kvq_or_seq_attend(const kvq_or_seq *s, const uint16_t *q16, int g, double *out)
{
    long L = kvq_or_seq_len(s);
    int D = s->D;
    double *Kh = (double *)malloc(sizeof(double) * (size_t)(L * D + 1));
    double *Vh = (double *)malloc(sizeof(double) * (size_t)(L * D + 1));
    double *q = (double *)malloc(sizeof(double) * (size_t)(g * D));
    if (!Kh || !Vh || !q) {
        free(Kh);
        free(Vh);
        free(q);
        return -1;
    }
    for (long i = 0; i < (long)g * D; i++)
        q[i] = kvq_or_h2f(q16[i]);
    kvq_or_seq_rows(s, Kh, Vh);
    if (s->rope_base > 0.0)
        kvq_or_rope(Kh, L, D, s->rope_base, 0);
    kvq_or_attend(q, g, Kh, Vh, L, D, out);
    free(Kh);
    free(Vh);
    free(q);
    return 0;
}

/* Array forms of the fp16 conversions (used by the oracle's own tests). */
void kvq_or_h2f_array(const uint16_t *h, float *f, long n)
{
    for (long i = 0; i < n; i++)
        f[i] = kvq_or_h2f(h[i]);
}

void kvq_or_f2h_array(const float *f, uint16_t *h, long n)
{
    for (long i = 0; i < n; i++)
        h[i] = kvq_or_f2h(f[i]);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 pages (BitDecoding notes, Sec. V-D: Blackwell's native low-precision  */
/* formats mxfp4 / nvfp4; the pages name the formats only).  Reading taken:    */
/* elements are e2m1 (1 sign, 2 exponent bits, bias 1, 1 mantissa bit: the    */
/* magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6); every block of 16 elements along   */
/* the dimension a product contracts (channels of a key, tokens of a value)   */
/* has an e4m3 scale (4 exponent bits, bias 7, 3 mantissa bits, largest 448); */
/* each page (G tokens of one sequence) has an fp32 scale S.  In fp32 with    */
/* IEEE operations:                                                           */
/*   S = amax(page) / 2688 (= 6 * 448);                                       */
/*   s = e4m3( amax(block) / 6 / S ), rounded to nearest even, saturating;    */
/*   d = s * S;  code = e2m1( x / d ), nearest even, saturating at 6, signed;  */
/*   an all-zero page has S = 0, and a zero d gives code 0;                   */
/* dequant x^ = e2m1(code) * s * S.                                           */
/* ------------------------------------------------------------------------ */

/* Value of a small float code with ebits exponent bits (bias), mbits mantissa bits
 * and a sign bit above them; exponent field 0 is subnormal. */
double kvq_or_small_float_value(int code, int ebits, int mbits, int bias)
{
    int mag = code & ((1 << (ebits + mbits)) - 1);
    int sign = (code >> (ebits + mbits)) & 1;
    int e = mag >> mbits, m = mag & ((1 << mbits) - 1);
    double v = e == 0 ? ldexp((double)m, 1 - bias - mbits)
                      : ldexp(1.0 + ldexp((double)m, -mbits), e - bias);
    return sign ? -v : v;
}

/* Code of the representable value nearest to x (ties to the even code), with
 * magnitudes above the largest finite value `maxv` taken as maxv (saturation).
 * Written from the format: for each exponent field e the values are spaced by
 * 2^(max(e,1) - bias - mbits), so x is rounded on that grid in its binade. */
int kvq_or_small_float_code(double x, int ebits, int mbits, int bias, double maxv)
{
    int sign = signbit(x) ? 1 : 0;
    double a = fabs(x);
    if (a >= maxv)
        a = maxv;
    /* the binade: largest e with 2^(e - bias) <= a (normal), else subnormal */
    int emax_field = (1 << ebits) - 1, e = 0;
    for (int f = emax_field; f >= 1; f--) {
        if (a >= ldexp(1.0, f - bias)) {
            e = f;
            break;
        }
    }
    double q = ldexp(1.0, (e > 0 ? e : 1) - bias - mbits);  /* spacing in this binade */
    double n = a / q;                                         /* exact: q is a power of 2 */
    double r = floor(n);
    double frac = n - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    /* r counts spacings from 0 (subnormal) or from 2^(e-bias) (normal) */
    int mag;
    if (e == 0) {
        mag = (int)r;  /* may carry into the first normal code: r == 2^mbits */
    } else {
        long steps = (long)r - (1L << mbits);  /* mantissa, may carry into the next binade */
        mag = (e << mbits) + (int)steps;
    }
    int magmax = (1 << (ebits + mbits)) - 1;
    if (mag > magmax)
        mag = magmax;
    return (sign << (ebits + mbits)) | mag;
}

static double fp32_div(double a, double b) { return (double)((float)a / (float)b); }

static int e2m1_code(float x) { return kvq_or_small_float_code((double)x, 2, 1, 1, 6.0); }
static int e4m3_code(float x) { return kvq_or_small_float_code((double)x, 4, 3, 7, 448.0); }
static float e4m3_value(int c) { return (float)kvq_or_small_float_value(c, 4, 3, 7); }
double kvq_or_e2m1_value(int c) { return kvq_or_small_float_value(c, 2, 1, 1); }

/* One NVFP4 block of n elements x[0], x[stride], ...: its scale code and its codes
 * (code i into codes[i]).  S: the page scale. */
static void nvfp4_block(const float *x, long stride, int n, float S, uint8_t *scale, uint8_t *codes)
{
    float amax = 0.0f;
    for (int i = 0; i < n; i++) {
        float a = fabsf(x[i * stride]);
        if (a > amax)
            amax = a;
    }
    if (S == 0.0f) {
        *scale = 0;
        for (int i = 0; i < n; i++)
            codes[i] = 0;
        return;
    }
    float sb = (float)fp32_div(fp32_div(amax, 6.0), S);
    int sc = e4m3_code(sb);
    *scale = (uint8_t)sc;
    volatile float d = e4m3_value(sc) * S;   /* fp32 product, rounded once */
    for (int i = 0; i < n; i++) {
        if (d == 0.0f) {
            codes[i] = 0;
            continue;
        }
        volatile float r = x[i * stride] / d;
        codes[i] = (uint8_t)e2m1_code(r);
    }
}

static float page_scale(const uint16_t *x, long n)
{
    float amax = 0.0f;
    for (long i = 0; i < n; i++) {
        float a = fabsf(kvq_or_h2f(x[i]));
        if (a > amax)
            amax = a;
    }
    return (float)fp32_div(amax, 2688.0);
}

/* Keys: page k [G][D] fp16 -> codes [G][D/2] (channel 2i low nibble, 2i+1 high),
 * scales [G][D/16] (blocks of 16 channels of a token), *S. */
void kvq_or_nvfp4_page_k(const uint16_t *k, int G, int D, uint8_t *codes, uint8_t *scales, float *S_out)
{
    float S = page_scale(k, (long)G * D);
    float x[16];
    uint8_t c[16];
    for (int t = 0; t < G; t++) {
        for (int b = 0; b < D / 16; b++) {
            for (int i = 0; i < 16; i++)
                x[i] = kvq_or_h2f(k[(long)t * D + 16 * b + i]);
            nvfp4_block(x, 1, 16, S, &scales[(long)t * (D / 16) + b], c);
            for (int i = 0; i < 8; i++)
                codes[(long)t * (D / 2) + 8 * b + i] = (uint8_t)(c[2 * i] | (c[2 * i + 1] << 4));
        }
    }
    *S_out = S;
}

/* Values: page v [G][D] fp16 -> codes [G][D/2] (token-major, as keys), scales
 * [G/16][D] (blocks of 16 tokens of a channel), *S. */
void kvq_or_nvfp4_page_v(const uint16_t *v, int G, int D, uint8_t *codes, uint8_t *scales, float *S_out)
{
    float S = page_scale(v, (long)G * D);
    float x[16];
    uint8_t c[16];
    memset(codes, 0, (size_t)G * D / 2);
    for (int tb = 0; tb < G / 16; tb++) {
        for (int ch = 0; ch < D; ch++) {
            for (int i = 0; i < 16; i++)
                x[i] = kvq_or_h2f(v[(long)(16 * tb + i) * D + ch]);
            nvfp4_block(x, 1, 16, S, &scales[(long)tb * D + ch], c);
            for (int i = 0; i < 16; i++)
                codes[(long)(16 * tb + i) * (D / 2) + ch / 2] |= (uint8_t)(c[i] << (4 * (ch & 1)));
        }
    }
    *S_out = S;
}

/* Dequantized page [G][D] fp64 of either layout (value_blocks: blocks run along tokens). */
void kvq_or_nvfp4_dequant(const uint8_t *codes, const uint8_t *scales, float S, int G, int D, int value_blocks,
                          double *out)
{
    for (int t = 0; t < G; t++) {
        for (int ch = 0; ch < D; ch++) {
            int c = (codes[(long)t * (D / 2) + ch / 2] >> (4 * (ch & 1))) & 15;
            int sc = value_blocks ? scales[(long)(t / 16) * D + ch] : scales[(long)t * (D / 16) + ch / 16];
            out[(long)t * D + ch] = kvq_or_e2m1_value(c) * (double)e4m3_value(sc) * (double)S;
        }
    }
}
