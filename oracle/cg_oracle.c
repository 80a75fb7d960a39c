/*
 * cg_oracle.c -- CPU oracle of the CacheGen KV-cache codec.
 *
 * TEST INFRASTRUCTURE ONLY (see cg_oracle.h).  Plain single-threaded C99
 * plus the compiler's 128-bit integers; built with -O2 -ffp-contract=off.
 *
 * Parity status of each function is recorded in its comment: "pinned by"
 * names the independent facts that tests check it against.
 */
#include "cg_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------
 * binary16 <-> binary32, from the IEEE 754 definition of binary16:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent 0 is
 * subnormal (value m*2^-24), exponent 31 is Inf/NaN.
 * Pinned by: exhaustive comparison with numpy's float16 conversion.
 * ---------------------------------------------------------------------- */
float orc_f16_to_f32(uint16_t h)
{
    int sign = h >> 15;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(m + 1024), e - 25);
    return sign ? -v : v;
}

uint16_t orc_f32_to_f16_rn(float f)
{
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    float a = fabsf(f);
    if (isnan(f))
        return sign | 0x7E00;
    if (a >= 65520.0f) /* halfway between 65504 and 2^16 rounds to even: Inf */
        return sign | 0x7C00;
    if (a < 0x1p-14f) {
        /* subnormal: value = m * 2^-24, m = RN(a * 2^24); m = 1024 gives
         * the smallest normal, whose encoding is the same integer. */
        float m = nearbyintf(a * 16777216.0f);
        return sign | (uint16_t)m;
    }
    int e;
    frexpf(a, &e); /* a in [2^(e-1), 2^e) */
    int E = e - 1;
    float m = nearbyintf(ldexpf(a, 10 - E)); /* in [1024, 2048] */
    if (m == 2048.0f) {
        m = 1024.0f;
        E += 1;
    }
    if (E > 15)
        return sign | 0x7C00;
    return (uint16_t)(sign | ((E + 15) << 10) | ((int)m - 1024));
}

static int f16_finite(uint16_t h) { return ((h >> 10) & 31) != 31; }

/* fp16 value times 2^24, which is always an integer of magnitude < 2^40. */
static int64_t f16_scaled_int(uint16_t h)
{
    int e = (h >> 10) & 31;
    int64_t m = h & 1023;
    int64_t v = (e == 0) ? m : ((m + 1024) << (e - 1));
    return (h >> 15) ? -v : v;
}

/* ------------------------------------------------------------------------
 * Step 1 -- per-(layer, K/V, channel) statistics.  The pages ask for
 * "per layer and channel" sensitivity statistics (gptget summary,
 * Methodology) and tables built "based on calibration profiling" (Guide,
 * pillar 3); they do not say which statistic.  Reading adopted: the
 * population standard deviation of the channel's values over all S tokens:
 *     var = (1/S) * sum_t (x_t - mu)^2 ,  mu = (1/S) * sum_t x_t,
 * evaluated exactly.  With X_t = x_t * 2^24 (an integer for every fp16)
 *     var = (S*sum X^2 - (sum X)^2) / S^2 * 2^-48 ,
 * whose numerator is an exact integer.  Rounding: numerator and S^2 each
 * to binary64, one binary64 division, exact scaling by 2^-48, binary64
 * sqrt, then binary32.
 * Pinned by: closed forms (constant -> 0, +-a -> a, two values -> |a-b|/2),
 * numpy.std in binary64 to within one binary32 ulp, and an independent
 * big-integer evaluation in the tests.
 * ---------------------------------------------------------------------- */
float orc_channel_sigma(const uint16_t *x, int64_t S, int64_t stride)
{
    __int128 T = 0;
    unsigned __int128 Q = 0;
    for (int64_t t = 0; t < S; t++) {
        int64_t X = f16_scaled_int(x[t * stride]);
        T += X;
        unsigned __int128 a = (unsigned __int128)(X < 0 ? -X : X);
        Q += a * a;
    }
    unsigned __int128 absT = (unsigned __int128)(T < 0 ? -T : T);
    unsigned __int128 num = (unsigned __int128)S * Q - absT * absT;
    double var = (double)num / (double)((uint64_t)S * (uint64_t)S);
    var = var * 0x1p-48;
    return (float)sqrt(var);
}

/* ------------------------------------------------------------------------
 * Step 2 -- the delta quantization step.  The pages give layer-adaptive
 * precision ("finer in early layers, coarser in deep ones", Guide pillar
 * 1) and per-chunk compression levels (gptget summary, Methodology).  The
 * step for level base b and layer multiplier m is b*m*sigma, floored at
 * 2^-12 so a constant channel still has a finite reciprocal; the
 * quantizer multiplies by the stored reciprocal.
 * Pinned by: direct arithmetic cases in the tests.
 * ---------------------------------------------------------------------- */
void orc_step(float base, float mult, float sigma, float *step, float *recip)
{
    float bm = base * mult;
    float st = bm * sigma;
    if (!(st >= ORC_STEP_MIN))
        st = ORC_STEP_MIN;
    *step = st;
    *recip = 1.0f / st;
}

/* ------------------------------------------------------------------------
 * Step 3/4 -- anchors.  "The first token of each chunk is designated as
 * the Anchor Token ... quantized and stored with high precision" (Guide,
 * pillar 2; the guide's "chunk of size W" is the anchor group here).  The
 * anchor is stored as int8 with a per-(chunk, layer, K/V, channel) absmax
 * scale: s = absmax/127, a_q = clamp(RN(x * 127/absmax), -127, 127),
 * a_hat = a_q * s.  absmax = 0 gives s = 0 (every anchor decodes to 0).
 * Pinned by: G = 1 reduces the codec to textbook per-channel int8 absmax
 * quantization, checked against an independent restatement; the anchor
 * error bound |fp16(a_hat) - x| <= s/2 (1+2^-20) + half an fp16 ulp.
 * ---------------------------------------------------------------------- */
void orc_anchor_scale(float absmax, float *s, float *inv)
{
    if (absmax == 0.0f) {
        *s = 0.0f;
        *inv = 0.0f;
        return;
    }
    *s = absmax / 127.0f;
    *inv = 127.0f / absmax;
}

int32_t orc_anchor_code(float x, float s, float inv, float *ahat)
{
    float v = x * inv;
    float r = nearbyintf(v);
    int32_t a = (int32_t)r;
    if (a > 127)
        a = 127;
    if (a < -127)
        a = -127;
    *ahat = (float)a * s;
    return a;
}

/* ------------------------------------------------------------------------
 * Step 5 -- deltas.  "Delta_t = K_t - K_anchor" (Guide, pillar 2).  The
 * guide's own sketch takes the delta of already-quantized tokens; the
 * decoder only knows the dequantized anchor, so the delta is taken
 * against a_hat (closed loop) and quantized with the stored reciprocal:
 *     q = RN((x - a_hat) * recip).
 * Symbols: q+127 when |q| <= R, else the escape symbol 255 with q sent raw.
 * Pinned by: the per-element bound |x_hat - x| <= step/2 (1+2^-20) plus
 * half an fp16 ulp, checked exhaustively over every finite fp16 x.
 * ---------------------------------------------------------------------- */
int32_t orc_delta_code(float x, float ahat, float recip)
{
    float dlt = x - ahat;
    float v = dlt * recip;
    return (int32_t)nearbyintf(v);
}

int32_t orc_symbol(int32_t q, int32_t R)
{
    if (q >= -R && q <= R)
        return q + 127;
    return ORC_ESC;
}

/* Step 10 -- reconstruction: x_hat = fma(q, step, a_hat), clamped to the
 * finite fp16 range, rounded to fp16 (Guide Step 2 decode_sequence adds
 * the delta back to the anchor; Step 1 dequantize multiplies by the
 * scale). */
uint16_t orc_reconstruct(int32_t q, float step, float ahat)
{
    float v = fmaf((float)q, step, ahat);
    if (v > 65504.0f)
        v = 65504.0f;
    if (v < -65504.0f)
        v = -65504.0f;
    return orc_f32_to_f16_rn(v);
}

/* ------------------------------------------------------------------------
 * Step 7 -- frequency normalisation to a total of M = 2^16 (16-bit CDF
 * tables; pillar 3 of the Guide builds "empirical probability frequency
 * tables").  Every one of the 256 symbols keeps a frequency of at least 1
 * so that any value can be coded:
 *     f_s = 1 + floor(n_s * (M - 256) / N),
 * the remainder M - sum f goes to the most frequent symbol (lowest index
 * on ties; symbol 127, q = 0, when N = 0); cdf_s = sum_{i<s} f_i.
 * Pinned by: sum f = M, f >= 1, |f_s - n_s M/N| <= 1 + 256 n_s/N.
 * ---------------------------------------------------------------------- */
void orc_normalize(const uint64_t n[256], uint32_t f[256], uint32_t cdf[257])
{
    uint64_t N = 0;
    for (int s = 0; s < 256; s++)
        N += n[s];
    uint64_t sum = 0;
    for (int s = 0; s < 256; s++) {
        f[s] = 1 + (N ? (uint32_t)((n[s] * (uint64_t)(ORC_M - ORC_NSYM)) / N) : 0);
        sum += f[s];
    }
    int arg = 127;
    if (N) {
        arg = 0;
        for (int s = 1; s < 256; s++)
            if (n[s] > n[arg])
                arg = s;
    }
    f[arg] += (uint32_t)(ORC_M - sum);
    cdf[0] = 0;
    for (int s = 0; s < 256; s++)
        cdf[s + 1] = cdf[s] + f[s];
}

/* ------------------------------------------------------------------------
 * Step 8/9 -- the range coder.  The pages name arithmetic coding (Guide,
 * pillar 3; gptget Methodology); the coder adopted is rANS (Duda, 2013,
 * "Asymmetric numeral systems"), range variant: 32-bit state in
 * [2^16, 2^32), 16-bit output words, M = 2^16.
 *   encode s:  if x >= f_s * 2^16 { emit x & 0xFFFF; x >>= 16 }
 *              x = floor(x / f_s) * 2^16 + (x mod f_s) + cdf_s
 *   decode:    slot = x & 0xFFFF; s: cdf_s <= slot < cdf_s + f_s
 *              x = f_s * (x >> 16) + slot - cdf_s
 *              if x < 2^16 { x = (x << 16) | next word }
 * One stream interleaves d lanes (one per channel of the head); all
 * lanes share a single word sequence.  Decode order: token ascending,
 * lane ascending, and per lane [renorm word][escape low][escape high].
 * The encoder runs the exact reverse order (token descending, lane
 * descending, per lane: escape high, escape low, renorm word) from the
 * initial state 2^16 and the word sequence is then reversed.
 * Pinned by: brute-force round trip of every sequence of length <= 4 over
 * small tables, final state = 2^16, and the code-length bound
 * |8*bytes - sum -log2(f/M)| <= 16 d.
 * ---------------------------------------------------------------------- */
int64_t orc_rans_encode(int64_t n, int32_t d, const uint8_t *sym,
                        const int32_t *qv, const uint32_t *f,
                        const uint32_t *cdf, uint32_t *state_out,
                        uint16_t *words_out)
{
    uint32_t *x = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(d > 0 ? d : 1));
    for (int32_t j = 0; j < d; j++)
        x[j] = ORC_RANS_L;
    int64_t nw = 0; /* words in encoder (reverse) order */
    for (int64_t t = n - 1; t >= 0; t--) {
        for (int32_t j = d - 1; j >= 0; j--) {
            uint32_t s = sym[t * d + j];
            if (s == ORC_ESC) {
                uint32_t q = (uint32_t)qv[t * d + j];
                words_out[nw++] = (uint16_t)(q >> 16);
                words_out[nw++] = (uint16_t)(q & 0xFFFF);
            }
            uint32_t fs = f[(size_t)j * 256 + s];
            uint32_t cs = cdf[(size_t)j * 257 + s];
            if ((uint64_t)x[j] >= ((uint64_t)fs << 16)) {
                words_out[nw++] = (uint16_t)(x[j] & 0xFFFF);
                x[j] >>= 16;
            }
            x[j] = ((x[j] / fs) << 16) + (x[j] % fs) + cs;
        }
    }
    for (int64_t i = 0; i < nw / 2; i++) { /* reverse into decode order */
        uint16_t tmp = words_out[i];
        words_out[i] = words_out[nw - 1 - i];
        words_out[nw - 1 - i] = tmp;
    }
    for (int32_t j = 0; j < d; j++)
        state_out[j] = x[j];
    free(x);
    return nw;
}

int orc_rans_decode(int64_t n, int32_t d, const uint32_t *state,
                    const uint16_t *words, int64_t n_words, int64_t n_esc,
                    const uint32_t *f, const uint32_t *cdf, uint8_t *sym_out,
                    int32_t *q_out)
{
    int rc = ORC_OK;
    uint32_t *x = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(d > 0 ? d : 1));
    for (int32_t j = 0; j < d; j++) {
        x[j] = state[j];
        if (x[j] < ORC_RANS_L)
            rc = ORC_ERR_CORRUPT;
    }
    int64_t p = 0, esc = 0;
    for (int64_t t = 0; t < n && rc == ORC_OK; t++) {
        for (int32_t j = 0; j < d; j++) {
            const uint32_t *fj = f + (size_t)j * 256;
            const uint32_t *cj = cdf + (size_t)j * 257;
            uint32_t slot = x[j] & 0xFFFF;
            uint32_t s = 0; /* the symbol whose range holds the slot */
            while (s < 255 && cj[s + 1] <= slot)
                s++;
            x[j] = fj[s] * (x[j] >> 16) + slot - cj[s];
            if (x[j] < ORC_RANS_L) {
                if (p >= n_words) {
                    rc = ORC_ERR_CORRUPT;
                    break;
                }
                x[j] = (x[j] << 16) | words[p++];
            }
            int32_t q;
            if (s == ORC_ESC) {
                if (p + 2 > n_words) {
                    rc = ORC_ERR_CORRUPT;
                    break;
                }
                q = (int32_t)((uint32_t)words[p] | ((uint32_t)words[p + 1] << 16));
                p += 2;
                esc++;
            } else {
                q = (int32_t)s - 127;
            }
            sym_out[t * d + j] = (uint8_t)s;
            q_out[t * d + j] = q;
        }
    }
    if (rc == ORC_OK) {
        for (int32_t j = 0; j < d; j++)
            if (x[j] != ORC_RANS_L)
                rc = ORC_ERR_CORRUPT;
        if (p != n_words || esc != n_esc)
            rc = ORC_ERR_CORRUPT;
    }
    free(x);
    return rc;
}

/* ------------------------------------------------------------------------
 * Byte formats.  Little-endian; every section starts on 16 bytes; padding
 * is zero.
 *
 * Tables blob: 64-byte header {"CGTB", u32 version=1, u32 L, H, d,
 * n_levels, R, u32 0, f32 level_base[8]}, then f32 step[NL][L][2][H*d],
 * f32 recip[same], u16 cdf[NL][L][2][H*d][256].
 *
 * Container: 64-byte header {"CGKV", u32 version=1, u32 L, H, d, C, G, R,
 * u64 S, u32 n_levels, u32 n_chunks, u64 total_bytes, u32 0, u32 0}, then
 * u64 chunk_off[n_chunks] (absolute).  Chunk k: 16-byte header {u16 level,
 * u16 0, u32 t0, u32 n_tok, u32 n_groups}, f32 s[L][2][H][d], i8
 * anchors[L][2][H][n_groups][d], u32 stream_off[L][2][H] (from the chunk
 * start), then the streams in (l, kv, h) order.  Stream: {u32 n_words,
 * u32 n_esc, u32 n_delta, u32 0}, u32 state[d], u16 words[n_words].
 * ---------------------------------------------------------------------- */
static uint64_t pad16(uint64_t v) { return (v + 15) & ~(uint64_t)15; }

static void put32(uint8_t *p, uint32_t v) { memcpy(p, &v, 4); }
static void put64(uint8_t *p, uint64_t v) { memcpy(p, &v, 8); }
static uint32_t get32(const uint8_t *p)
{
    uint32_t v;
    memcpy(&v, p, 4);
    return v;
}
static uint64_t get64(const uint8_t *p)
{
    uint64_t v;
    memcpy(&v, p, 8);
    return v;
}

static int64_t n_chunks_of(const orc_dims *dm) { return (dm->S + dm->C - 1) / dm->C; }
static int64_t chunk_ntok(const orc_dims *dm, int64_t k)
{
    int64_t t0 = k * dm->C;
    int64_t n = dm->S - t0;
    return n < dm->C ? n : dm->C;
}
static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

static int dims_ok(const orc_dims *dm)
{
    return dm->L >= 1 && dm->H >= 1 && dm->d >= 1 && dm->C >= 1 && dm->G >= 1 &&
           dm->S >= 1 && dm->S <= ((int64_t)1 << 22) && dm->R >= 0 && dm->R <= 127;
}

size_t orc_tables_bytes(const orc_dims *dm, int32_t n_levels)
{
    uint64_t nc = (uint64_t)n_levels * dm->L * 2 * dm->H * dm->d;
    return (size_t)(64 + 2 * pad16(4 * nc) + 512 * nc);
}

static float tier_mult(int32_t l, int32_t L)
{
    int64_t tier = (3 * (int64_t)l) / L;
    return tier == 0 ? 0.5f : (tier == 1 ? 1.0f : 2.0f);
}

/* The head's symbols at one level, used by both the fit and the encoder. */
typedef struct {
    int64_t n_groups, n_delta;
    float *s;        /* [d]            */
    int8_t *anc;     /* [n_groups][d]  */
    uint8_t *sym;    /* [n_delta][d]   */
    int32_t *q;      /* [n_delta][d]   */
} chunk_syms;

/* Quantize chunk k of one head: anchors, deltas, symbols. */
static int quantize_chunk(const orc_dims *dm, const uint16_t *head, int64_t k,
                          const float *recip, chunk_syms *cs)
{
    const int32_t d = dm->d;
    const int64_t t0 = k * dm->C, ntok = chunk_ntok(dm, k);
    const int64_t ng = ceil_div(ntok, dm->G);
    cs->n_groups = ng;
    cs->n_delta = ntok - ng;
    float *inv = (float *)malloc(sizeof(float) * (size_t)d);
    float *ahat = (float *)malloc(sizeof(float) * (size_t)d);
    int rc = ORC_OK;
    for (int64_t t = t0; t < t0 + ntok; t++)
        for (int32_t j = 0; j < d; j++)
            if (!f16_finite(head[t * d + j]))
                rc = ORC_ERR_NONFINITE;
    for (int32_t j = 0; j < d && rc == ORC_OK; j++) {
        float amax = 0.0f;
        for (int64_t g = 0; g < ng; g++) {
            float v = fabsf(orc_f16_to_f32(head[(t0 + g * dm->G) * d + j]));
            if (v > amax)
                amax = v;
        }
        orc_anchor_scale(amax, &cs->s[j], &inv[j]);
    }
    int64_t di = 0;
    for (int64_t g = 0; g < ng && rc == ORC_OK; g++) {
        int64_t ta = t0 + g * dm->G;
        for (int32_t j = 0; j < d; j++)
            cs->anc[g * d + j] = (int8_t)orc_anchor_code(
                orc_f16_to_f32(head[ta * d + j]), cs->s[j], inv[j], &ahat[j]);
        for (int64_t t = ta + 1; t < ta + dm->G && t < t0 + ntok; t++, di++)
            for (int32_t j = 0; j < d; j++) {
                int32_t q = orc_delta_code(orc_f16_to_f32(head[t * d + j]), ahat[j],
                                           recip[j]);
                cs->q[di * d + j] = q;
                cs->sym[di * d + j] = (uint8_t)orc_symbol(q, dm->R);
            }
    }
    free(inv);
    free(ahat);
    return rc;
}

static void chunk_syms_alloc(const orc_dims *dm, chunk_syms *cs)
{
    int64_t ntok = dm->C < dm->S ? dm->C : dm->S;
    cs->s = (float *)malloc(sizeof(float) * (size_t)dm->d);
    cs->anc = (int8_t *)malloc((size_t)(ntok * dm->d));
    cs->sym = (uint8_t *)malloc((size_t)(ntok * dm->d));
    cs->q = (int32_t *)malloc(sizeof(int32_t) * (size_t)(ntok * dm->d));
}
static void chunk_syms_free(chunk_syms *cs)
{
    free(cs->s);
    free(cs->anc);
    free(cs->sym);
    free(cs->q);
}

int orc_fit_head(const orc_dims *dm, float base, float mult,
                 const uint16_t *head, float *step, float *recip, uint16_t *cdf)
{
    if (!dims_ok(dm))
        return ORC_ERR_INVALID_ARG;
    const int32_t d = dm->d;
    for (int64_t i = 0; i < dm->S * d; i++)
        if (!f16_finite(head[i]))
            return ORC_ERR_NONFINITE;
    for (int32_t j = 0; j < d; j++)
        orc_step(base, mult, orc_channel_sigma(head + j, dm->S, d), &step[j], &recip[j]);
    uint64_t *n = (uint64_t *)calloc((size_t)d * 256, sizeof(uint64_t));
    chunk_syms cs;
    chunk_syms_alloc(dm, &cs);
    int rc = ORC_OK;
    for (int64_t k = 0; k < n_chunks_of(dm) && rc == ORC_OK; k++) {
        rc = quantize_chunk(dm, head, k, recip, &cs);
        for (int64_t i = 0; i < cs.n_delta * d && rc == ORC_OK; i++)
            n[(i % d) * 256 + cs.sym[i]]++;
    }
    uint32_t f[256], c[257];
    for (int32_t j = 0; j < d; j++) {
        orc_normalize(n + (size_t)j * 256, f, c);
        for (int s = 0; s < 256; s++)
            cdf[(size_t)j * 256 + s] = (uint16_t)c[s];
    }
    chunk_syms_free(&cs);
    free(n);
    return rc;
}

int orc_fit_tables(const orc_dims *dm, int32_t n_levels, const float *level_base,
                   const float *layer_mult, const uint16_t *kv, uint8_t *tables)
{
    if (!dims_ok(dm) || n_levels < 1 || n_levels > ORC_MAX_LEVELS)
        return ORC_ERR_INVALID_ARG;
    const int64_t HD = (int64_t)dm->H * dm->d;
    const uint64_t nc = (uint64_t)n_levels * dm->L * 2 * HD;
    memset(tables, 0, orc_tables_bytes(dm, n_levels));
    memcpy(tables, "CGTB", 4);
    put32(tables + 4, 1);
    put32(tables + 8, (uint32_t)dm->L);
    put32(tables + 12, (uint32_t)dm->H);
    put32(tables + 16, (uint32_t)dm->d);
    put32(tables + 20, (uint32_t)n_levels);
    put32(tables + 24, (uint32_t)dm->R);
    for (int i = 0; i < n_levels; i++)
        memcpy(tables + 32 + 4 * i, &level_base[i], 4);
    float *stepv = (float *)(tables + 64);
    float *recipv = (float *)(tables + 64 + pad16(4 * nc));
    uint16_t *cdfv = (uint16_t *)(tables + 64 + 2 * pad16(4 * nc));
    for (int32_t lv = 0; lv < n_levels; lv++)
        for (int32_t l = 0; l < dm->L; l++)
            for (int32_t kvi = 0; kvi < 2; kvi++) {
                float m = layer_mult ? layer_mult[l * 2 + kvi] : tier_mult(l, dm->L);
                for (int32_t h = 0; h < dm->H; h++) {
                    const uint16_t *head = kv + (((int64_t)l * 2 + kvi) * dm->H + h) * dm->S * dm->d;
                    int64_t c0 = (((int64_t)lv * dm->L + l) * 2 + kvi) * HD + (int64_t)h * dm->d;
                    int rc = orc_fit_head(dm, level_base[lv], m, head, stepv + c0,
                                          recipv + c0, cdfv + c0 * 256);
                    if (rc != ORC_OK)
                        return rc;
                }
            }
    return ORC_OK;
}

/* Expand a u16 CDF row into (f, cdf) with cdf[256] = M.  Returns 0 if the
 * row is not a valid CDF (cdf[0] = 0, strictly increasing, below M). */
static int expand_cdf(const uint16_t *c16, uint32_t *f, uint32_t *c)
{
    if (c16[0] != 0)
        return 0;
    for (int s = 0; s < 256; s++)
        c[s] = c16[s];
    c[256] = ORC_M;
    for (int s = 0; s < 256; s++) {
        if (c[s + 1] <= c[s])
            return 0;
        f[s] = c[s + 1] - c[s];
    }
    return 1;
}

int64_t orc_encode_stream(const orc_dims *dm, const uint16_t *head, int64_t k,
                          const float *step, const float *recip,
                          const uint16_t *cdf, float *s_out, int8_t *anchors_out,
                          uint8_t *blk, int64_t blk_cap, uint64_t *symcount,
                          orc_stats *st)
{
    (void)step;
    const int32_t d = dm->d;
    uint32_t *f = (uint32_t *)malloc(sizeof(uint32_t) * 256 * (size_t)d);
    uint32_t *c = (uint32_t *)malloc(sizeof(uint32_t) * 257 * (size_t)d);
    for (int32_t j = 0; j < d; j++)
        if (!expand_cdf(cdf + (size_t)j * 256, f + (size_t)j * 256, c + (size_t)j * 257)) {
            free(f);
            free(c);
            return -ORC_ERR_INVALID_ARG;
        }
    chunk_syms cs;
    chunk_syms_alloc(dm, &cs);
    int rc = quantize_chunk(dm, head, k, recip, &cs);
    int64_t ret = -rc;
    if (rc == ORC_OK) {
        uint16_t *w = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(3 * cs.n_delta * d + 1));
        uint32_t *state = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)d);
        int64_t nw = orc_rans_encode(cs.n_delta, d, cs.sym, cs.q, f, c, state, w);
        uint64_t n_esc = 0;
        for (int64_t i = 0; i < cs.n_delta * d; i++)
            n_esc += cs.sym[i] == ORC_ESC;
        int64_t len = (int64_t)pad16(16 + 4 * (uint64_t)d + 2 * (uint64_t)nw);
        if (len > blk_cap) {
            ret = -ORC_ERR_CAPACITY;
        } else {
            memset(blk, 0, (size_t)len);
            put32(blk, (uint32_t)nw);
            put32(blk + 4, (uint32_t)n_esc);
            put32(blk + 8, (uint32_t)cs.n_delta);
            for (int32_t j = 0; j < d; j++)
                put32(blk + 16 + 4 * j, state[j]);
            memcpy(blk + 16 + 4 * d, w, 2 * (size_t)nw);
            memcpy(s_out, cs.s, sizeof(float) * (size_t)d);
            memcpy(anchors_out, cs.anc, (size_t)(cs.n_groups * d));
            if (symcount)
                for (int64_t i = 0; i < cs.n_delta * d; i++)
                    symcount[(i % d) * 256 + cs.sym[i]]++;
            if (st) {
                st->n_symbols += (uint64_t)(cs.n_delta * d);
                st->n_esc += n_esc;
                st->n_words += (uint64_t)nw;
                st->state_bytes += 4 * (uint64_t)d;
                st->pad_bytes += (uint64_t)len - (16 + 4 * (uint64_t)d + 2 * (uint64_t)nw);
                st->fixed_bytes += 16;
            }
            ret = len;
        }
        free(w);
        free(state);
    }
    chunk_syms_free(&cs);
    free(f);
    free(c);
    return ret;
}

/* Size of chunk k's fixed part (header, scales, anchors, stream index). */
static uint64_t chunk_fixed_bytes(const orc_dims *dm, int64_t k)
{
    uint64_t nstr = (uint64_t)dm->L * 2 * dm->H;
    uint64_t ng = (uint64_t)ceil_div(chunk_ntok(dm, k), dm->G);
    return 16 + pad16(4 * nstr * dm->d) + pad16(nstr * ng * dm->d) + pad16(4 * nstr);
}

uint64_t orc_encode_bound(const orc_dims *dm)
{
    /* words: at most one renorm word per symbol plus two per escape */
    int64_t nk = n_chunks_of(dm);
    uint64_t total = pad16(64 + 8 * (uint64_t)nk);
    for (int64_t k = 0; k < nk; k++) {
        int64_t ntok = chunk_ntok(dm, k);
        int64_t nd = ntok - ceil_div(ntok, dm->G);
        total += chunk_fixed_bytes(dm, k);
        total += (uint64_t)dm->L * 2 * dm->H *
                 pad16(16 + 4 * (uint64_t)dm->d + 6 * (uint64_t)nd * dm->d);
    }
    return total;
}

/* Bits the coded symbols of one table carry at their own empirical
 * frequencies: sum_s n_s log2(N / n_s) over the 256 symbols (escape
 * included).  Summed over the tables it is the first term of the entropy
 * bound a container is measured against: the size an ideal coder would
 * reach with the empirical symbol distribution of each (layer, channel)
 * table (Guide, pillar 3, "Distribution-Aware Arithmetic Coding"). */
double orc_table_entropy(const uint64_t *n)
{
    uint64_t N = 0;
    for (int s = 0; s < 256; s++)
        N += n[s];
    double h = 0.0;
    for (int s = 0; s < 256; s++)
        if (n[s])
            h += (double)n[s] * log2((double)N / (double)n[s]);
    return h;
}

/* Information-bearing structure of a container outside its streams, as
 * the entropy bound counts it (no padding): the header and chunk index, and
 * per chunk its header, scales, anchors and stream offsets.  Stream headers
 * (16 bytes each) are counted by orc_encode_stream. */
uint64_t orc_container_fixed_bytes(const orc_dims *dm)
{
    const int64_t nk = n_chunks_of(dm), nstr = (int64_t)dm->L * 2 * dm->H, d = dm->d;
    uint64_t fixed = 64 + 8 * (uint64_t)nk;
    for (int64_t k = 0; k < nk; k++) {
        int64_t ng = ceil_div(chunk_ntok(dm, k), dm->G);
        fixed += 16 + 4 * (uint64_t)nstr * d + (uint64_t)(nstr * ng * d) + 4 * (uint64_t)nstr;
    }
    return fixed;
}

int orc_encode(const orc_dims *dm, int32_t n_levels, const uint8_t *tables,
               const uint16_t *kv, const uint8_t *chunk_level, uint8_t *out,
               uint64_t cap, uint64_t *out_bytes, orc_stats *st)
{
    if (!dims_ok(dm) || n_levels < 1 || n_levels > ORC_MAX_LEVELS)
        return ORC_ERR_INVALID_ARG;
    if (memcmp(tables, "CGTB", 4) != 0 || get32(tables + 8) != (uint32_t)dm->L ||
        get32(tables + 12) != (uint32_t)dm->H || get32(tables + 16) != (uint32_t)dm->d ||
        get32(tables + 20) != (uint32_t)n_levels || get32(tables + 24) != (uint32_t)dm->R)
        return ORC_ERR_INVALID_ARG;
    const int32_t d = dm->d;
    const int64_t HD = (int64_t)dm->H * d, nk = n_chunks_of(dm);
    const int64_t nstr = (int64_t)dm->L * 2 * dm->H;
    const uint64_t nc = (uint64_t)n_levels * dm->L * 2 * HD;
    const float *stepv = (const float *)(tables + 64);
    const float *recipv = (const float *)(tables + 64 + pad16(4 * nc));
    const uint16_t *cdfv = (const uint16_t *)(tables + 64 + 2 * pad16(4 * nc));
    for (int64_t k = 0; k < nk; k++)
        if (chunk_level[k] >= n_levels)
            return ORC_ERR_INVALID_ARG;

    orc_stats local;
    memset(&local, 0, sizeof local);
    uint64_t *cnt = (uint64_t *)calloc((size_t)nc * 256, sizeof(uint64_t));
    uint64_t pos = pad16(64 + 8 * (uint64_t)nk);
    if (pos > cap) {
        free(cnt);
        return ORC_ERR_CAPACITY;
    }
    memset(out, 0, (size_t)pos);
    int rc = ORC_OK;
    for (int64_t k = 0; k < nk && rc == ORC_OK; k++) {
        const int64_t ntok = chunk_ntok(dm, k), ng = ceil_div(ntok, dm->G);
        const uint64_t base = pos, fixed = chunk_fixed_bytes(dm, k);
        if (base + fixed > cap) {
            rc = ORC_ERR_CAPACITY;
            break;
        }
        memset(out + base, 0, (size_t)fixed);
        put64(out + 64 + 8 * k, base);
        uint8_t *ch = out + base;
        uint16_t lvl = chunk_level[k];
        memcpy(ch, &lvl, 2);
        put32(ch + 4, (uint32_t)(k * dm->C));
        put32(ch + 8, (uint32_t)ntok);
        put32(ch + 12, (uint32_t)ng);
        float *sv = (float *)(ch + 16);
        int8_t *av = (int8_t *)(ch + 16 + pad16(4 * (uint64_t)nstr * d));
        uint8_t *offv = ch + 16 + pad16(4 * (uint64_t)nstr * d) + pad16((uint64_t)(nstr * ng * d));
        pos = base + fixed;
        for (int64_t si = 0; si < nstr && rc == ORC_OK; si++) {
            const int64_t l = si / (2 * dm->H), kvi = (si / dm->H) % 2, h = si % dm->H;
            const uint16_t *head = kv + si * dm->S * d;
            const int64_t c0 = ((lvl * (int64_t)dm->L + l) * 2 + kvi) * HD + h * d;
            put32(offv + 4 * si, (uint32_t)(pos - base));
            int64_t len = orc_encode_stream(dm, head, k, stepv + c0, recipv + c0,
                                            cdfv + c0 * 256, sv + si * d, av + si * ng * d,
                                            out + pos, (int64_t)(cap - pos), cnt + c0 * 256,
                                            &local);
            if (len < 0)
                rc = (int)-len;
            else
                pos += (uint64_t)len;
        }
    }
    if (rc == ORC_OK) {
        memcpy(out, "CGKV", 4);
        put32(out + 4, 1);
        put32(out + 8, (uint32_t)dm->L);
        put32(out + 12, (uint32_t)dm->H);
        put32(out + 16, (uint32_t)dm->d);
        put32(out + 20, (uint32_t)dm->C);
        put32(out + 24, (uint32_t)dm->G);
        put32(out + 28, (uint32_t)dm->R);
        put64(out + 32, (uint64_t)dm->S);
        put32(out + 40, (uint32_t)n_levels);
        put32(out + 44, (uint32_t)nk);
        put64(out + 48, pos);
        *out_bytes = pos;
        if (st) {
            double h = 0.0;
            for (uint64_t i = 0; i < nc; i++)
                h += orc_table_entropy(cnt + i * 256);
            local.entropy_bits = h;
            local.fixed_bytes += orc_container_fixed_bytes(dm);
            local.pad_bytes = pos - local.fixed_bytes - local.state_bytes - 2 * local.n_words;
            *st = local;
        }
    }
    free(cnt);
    return rc;
}

int orc_decode_stream(const orc_dims *dm, const uint8_t *blk, uint64_t blk_len,
                      int64_t k, const float *step, const uint16_t *cdf,
                      const float *s, const int8_t *anchors, uint16_t *head)
{
    const int32_t d = dm->d;
    const int64_t t0 = k * dm->C, ntok = chunk_ntok(dm, k), ng = ceil_div(ntok, dm->G);
    const int64_t nd = ntok - ng;
    if (blk_len < 16 + 4 * (uint64_t)d)
        return ORC_ERR_CORRUPT;
    uint64_t nw = get32(blk), ne = get32(blk + 4);
    if (get32(blk + 8) != (uint32_t)nd || get32(blk + 12) != 0)
        return ORC_ERR_CORRUPT;
    if (16 + 4 * (uint64_t)d + 2 * nw > blk_len)
        return ORC_ERR_CORRUPT;
    uint32_t *f = (uint32_t *)malloc(sizeof(uint32_t) * 256 * (size_t)d);
    uint32_t *c = (uint32_t *)malloc(sizeof(uint32_t) * 257 * (size_t)d);
    uint32_t *state = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)d);
    uint16_t *w = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(nw + 1));
    uint8_t *sym = (uint8_t *)malloc((size_t)(nd * d + 1));
    int32_t *q = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nd * d + 1));
    int rc = ORC_OK;
    for (int32_t j = 0; j < d && rc == ORC_OK; j++)
        if (!expand_cdf(cdf + (size_t)j * 256, f + (size_t)j * 256, c + (size_t)j * 257))
            rc = ORC_ERR_CORRUPT;
    if (rc == ORC_OK) {
        for (int32_t j = 0; j < d; j++)
            state[j] = get32(blk + 16 + 4 * j);
        memcpy(w, blk + 16 + 4 * d, 2 * (size_t)nw);
        rc = orc_rans_decode(nd, d, state, w, (int64_t)nw, (int64_t)ne, f, c, sym, q);
    }
    if (rc == ORC_OK) {
        float *ahat = (float *)malloc(sizeof(float) * (size_t)d);
        int64_t di = 0;
        for (int64_t g = 0; g < ng; g++) {
            int64_t ta = t0 + g * dm->G;
            for (int32_t j = 0; j < d; j++) {
                ahat[j] = (float)anchors[g * d + j] * s[j];
                head[ta * d + j] = orc_f32_to_f16_rn(ahat[j]);
            }
            for (int64_t t = ta + 1; t < ta + dm->G && t < t0 + ntok; t++, di++)
                for (int32_t j = 0; j < d; j++)
                    head[t * d + j] = orc_reconstruct(q[di * d + j], step[j], ahat[j]);
        }
        free(ahat);
    }
    free(f);
    free(c);
    free(state);
    free(w);
    free(sym);
    free(q);
    return rc;
}

int orc_decode(const uint8_t *tables, size_t tables_bytes, const uint8_t *buf,
               uint64_t bytes, int64_t k0, int64_t k1, uint16_t *kv)
{
    if (bytes < 64 || memcmp(buf, "CGKV", 4) != 0 || get32(buf + 4) != 1)
        return ORC_ERR_CORRUPT;
    orc_dims dm;
    dm.L = (int32_t)get32(buf + 8);
    dm.H = (int32_t)get32(buf + 12);
    dm.d = (int32_t)get32(buf + 16);
    dm.C = (int32_t)get32(buf + 20);
    dm.G = (int32_t)get32(buf + 24);
    dm.R = (int32_t)get32(buf + 28);
    dm.S = (int64_t)get64(buf + 32);
    const int32_t nl = (int32_t)get32(buf + 40);
    const int64_t nk = get32(buf + 44);
    if (!dims_ok(&dm) || nl < 1 || nl > ORC_MAX_LEVELS || nk != n_chunks_of(&dm) ||
        get64(buf + 48) != bytes)
        return ORC_ERR_CORRUPT;
    if (tables_bytes < 64 || tables_bytes != orc_tables_bytes(&dm, nl) ||
        memcmp(tables, "CGTB", 4) != 0 || get32(tables + 8) != (uint32_t)dm.L ||
        get32(tables + 12) != (uint32_t)dm.H || get32(tables + 16) != (uint32_t)dm.d ||
        get32(tables + 20) != (uint32_t)nl)
        return ORC_ERR_INVALID_ARG;
    if (k0 < 0 || k1 > nk || k0 > k1)
        return ORC_ERR_INVALID_ARG;
    const int32_t d = dm.d;
    const int64_t HD = (int64_t)dm.H * d, nstr = (int64_t)dm.L * 2 * dm.H;
    const uint64_t nc = (uint64_t)nl * dm.L * 2 * HD;
    const float *stepv = (const float *)(tables + 64);
    const uint16_t *cdfv = (const uint16_t *)(tables + 64 + 2 * pad16(4 * nc));
    if (pad16(64 + 8 * (uint64_t)nk) > bytes)
        return ORC_ERR_CORRUPT;
    for (int64_t k = k0; k < k1; k++) {
        uint64_t base = get64(buf + 64 + 8 * k);
        uint64_t end = (k + 1 < nk) ? get64(buf + 64 + 8 * (k + 1)) : bytes;
        uint64_t fixed = chunk_fixed_bytes(&dm, k);
        if ((base & 15) || end > bytes || base + fixed > end)
            return ORC_ERR_CORRUPT;
        const uint8_t *ch = buf + base;
        uint16_t lvl;
        memcpy(&lvl, ch, 2);
        const int64_t ntok = chunk_ntok(&dm, k), ng = ceil_div(ntok, dm.G);
        if (lvl >= nl || ch[2] || ch[3] || get32(ch + 4) != (uint32_t)(k * dm.C) ||
            get32(ch + 8) != (uint32_t)ntok || get32(ch + 12) != (uint32_t)ng)
            return ORC_ERR_CORRUPT;
        const float *sv = (const float *)(ch + 16);
        const int8_t *av = (const int8_t *)(ch + 16 + pad16(4 * (uint64_t)nstr * d));
        const uint8_t *offv = ch + 16 + pad16(4 * (uint64_t)nstr * d) + pad16((uint64_t)(nstr * ng * d));
        for (int64_t si = 0; si < nstr; si++) {
            uint64_t so = get32(offv + 4 * si);
            uint64_t se = (si + 1 < nstr) ? get32(offv + 4 * (si + 1)) : end - base;
            if ((so & 15) || so < fixed || se < so || base + se > end)
                return ORC_ERR_CORRUPT;
            const int64_t l = si / (2 * dm.H), kvi = (si / dm.H) % 2, h = si % dm.H;
            const int64_t c0 = ((lvl * (int64_t)dm.L + l) * 2 + kvi) * HD + h * d;
            int rc = orc_decode_stream(&dm, ch + so, se - so, k, stepv + c0, cdfv + c0 * 256,
                                       sv + si * d, av + si * ng * d, kv + si * dm.S * d);
            if (rc != ORC_OK)
                return rc;
        }
    }
    return ORC_OK;
}
