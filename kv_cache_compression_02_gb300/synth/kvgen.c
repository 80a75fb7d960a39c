/*
 * kvgen.c -- seeded synthetic KV-cache generator.
 *
 * Produces fp16 tensors laid out [L][2][H][S][d] whose channels follow an
 * AR(1) process over tokens with Laplace or Student-t(3) innovations, a
 * lognormal(0,1) scale per channel and a few outlier channels per (layer,
 * K/V) tensor scaled up.  It stands in for the KV caches of the Llama-
 * shaped models the CacheGen pages evaluate on, which are not available.
 *
 * It holds none of the codec's arithmetic: it only makes inputs.  Both the
 * CPU oracle's tests and the GPU path consume its output.
 *
 * Randomness: counter-based SplitMix64 (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014): the n-th output
 * of a stream with key k is mix64(k + (n+1)*0x9E3779B97F4A7C15).  Every
 * draw is addressed by (seed, purpose, layer, K/V, channel, token), so any
 * head can be generated alone and any thread count gives the same bits.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t L, H, d;
    int32_t innov;        /* 0: Laplace, 1: Student-t(3)                     */
    int64_t S;
    uint64_t seed;
    double rho_lo, rho_hi; /* rho per channel: rho_lo if equal, else U(lo,hi) */
    double outlier_frac;  /* used when n_outliers < 0                         */
    double outlier_scale;
    int32_t n_outliers;   /* outlier channels per (layer, K/V) tensor         */
    int32_t pad_;
} kvgen_spec;

static const uint64_t GOLDEN = 0x9E3779B97F4A7C15ULL;

static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}
static uint64_t draw(uint64_t key, uint64_t n) { return mix64(key + (n + 1) * GOLDEN); }
static double unif(uint64_t r) { return ((double)(r >> 11) + 0.5) * 0x1p-53; } /* (0,1) */

enum { P_RHO = 1, P_SCALE = 2, P_OUTLIER = 3, P_LEVEL = 4, P_INNOV = 5 };

static uint64_t key_of(uint64_t seed, uint64_t purpose, int64_t a, int64_t b, int64_t c)
{
    uint64_t k = draw(seed ^ 0x6B76676B76676B76ULL, purpose);
    k = draw(k, (uint64_t)a);
    k = draw(k, (uint64_t)b);
    return draw(k, (uint64_t)c);
}

/* Unit-variance innovations. */
static double laplace_unit(uint64_t key, int64_t t)
{
    const double b = 0.70710678118654752440; /* 1/sqrt(2) */
    double u = unif(draw(key, (uint64_t)t));
    return u < 0.5 ? b * log(2.0 * u) : -b * log(2.0 * (1.0 - u));
}
/* Student-t with 3 degrees of freedom by Bailey's polar method (Math. Comp.
 * 62, 1994), divided by sqrt(3) for unit variance. */
static double t3_unit(uint64_t key, int64_t t)
{
    for (uint64_t j = 0; j < 64; j++) {
        double u1 = 2.0 * unif(draw(key, (uint64_t)t * 128 + 2 * j)) - 1.0;
        double u2 = 2.0 * unif(draw(key, (uint64_t)t * 128 + 2 * j + 1)) - 1.0;
        double w = u1 * u1 + u2 * u2;
        if (w > 0.0 && w < 1.0) {
            double c = cbrt(w);
            return u1 * sqrt(3.0 * (1.0 / (c * c) - 1.0) / w) / 1.7320508075688772935;
        }
    }
    return 0.0;
}

/* binary64 -> binary16, round to nearest even (the generator's own). */
static uint16_t to_f16(double v)
{
    uint16_t sign = v < 0 ? 0x8000 : 0;
    double a = fabs(v);
    if (a >= 65520.0)
        return sign | 0x7C00;
    if (a < 0x1p-14)
        return sign | (uint16_t)nearbyint(a * 0x1p24);
    int e;
    frexp(a, &e);
    int E = e - 1;
    double m = nearbyint(ldexp(a, 10 - E));
    if (m == 2048.0) {
        m = 1024.0;
        E++;
    }
    if (E > 15)
        return sign | 0x7C00;
    return (uint16_t)(sign | ((E + 15) << 10) | ((int)m - 1024));
}

static int32_t outlier_count(const kvgen_spec *sp)
{
    if (sp->n_outliers >= 0)
        return sp->n_outliers;
    return (int32_t)llround(sp->outlier_frac * (double)sp->H * sp->d);
}

/* Channel parameters: rho and scale (outliers included). */
void kvgen_channel(const kvgen_spec *sp, int32_t l, int32_t kv, int32_t c, double *rho,
                   double *scale)
{
    uint64_t kr = key_of(sp->seed, P_RHO, l, kv, c);
    *rho = sp->rho_lo == sp->rho_hi ? sp->rho_lo
                                    : sp->rho_lo + (sp->rho_hi - sp->rho_lo) * unif(draw(kr, 0));
    uint64_t ks = key_of(sp->seed, P_SCALE, l, kv, c);
    double u1 = unif(draw(ks, 0)), u2 = unif(draw(ks, 1));
    double n01 = sqrt(-2.0 * log(u1)) * cos(6.283185307179586477 * u2); /* Box-Muller */
    double s = exp(n01);
    /* outliers: partial Fisher-Yates over the tensor's H*d channels */
    int32_t n = sp->H * sp->d, k = outlier_count(sp);
    if (k > n)
        k = n;
    if (k > 0) {
        int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
        for (int32_t i = 0; i < n; i++)
            perm[i] = i;
        uint64_t ko = key_of(sp->seed, P_OUTLIER, l, kv, 0);
        for (int32_t i = 0; i < k; i++) {
            int32_t j = i + (int32_t)(draw(ko, (uint64_t)i) % (uint64_t)(n - i));
            int32_t tmp = perm[i];
            perm[i] = perm[j];
            perm[j] = tmp;
            if (perm[i] == c)
                s *= sp->outlier_scale;
        }
        free(perm);
    }
    *scale = s;
}

/* One head (l, kv, h) into out[S][d]. */
void kvgen_head(const kvgen_spec *sp, int32_t l, int32_t kv, int32_t h, uint16_t *out)
{
    const int32_t d = sp->d;
    double *z = (double *)malloc(sizeof(double) * (size_t)d);
    double *rho = (double *)malloc(sizeof(double) * (size_t)d);
    double *cr = (double *)malloc(sizeof(double) * (size_t)d);
    double *sc = (double *)malloc(sizeof(double) * (size_t)d);
    uint64_t *key = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)d);
    for (int32_t j = 0; j < d; j++) {
        int32_t c = h * d + j;
        kvgen_channel(sp, l, kv, c, &rho[j], &sc[j]);
        cr[j] = sqrt(1.0 - rho[j] * rho[j]);
        key[j] = key_of(sp->seed, P_INNOV, l, kv, c);
    }
    for (int64_t t = 0; t < sp->S; t++) {
        for (int32_t j = 0; j < d; j++) {
            double e = sp->innov ? t3_unit(key[j], t) : laplace_unit(key[j], t);
            z[j] = t == 0 ? e : rho[j] * z[j] + cr[j] * e;
            double v = sc[j] * z[j];
            if (v > 65504.0)
                v = 65504.0;
            if (v < -65504.0)
                v = -65504.0;
            out[t * d + j] = to_f16(v);
        }
    }
    free(z);
    free(rho);
    free(cr);
    free(sc);
    free(key);
}

typedef struct {
    const kvgen_spec *sp;
    uint16_t *out;
    int64_t next, n_heads;
    pthread_mutex_t mu;
} job_t;

static void *worker(void *arg)
{
    job_t *jb = (job_t *)arg;
    for (;;) {
        pthread_mutex_lock(&jb->mu);
        int64_t i = jb->next++;
        pthread_mutex_unlock(&jb->mu);
        if (i >= jb->n_heads)
            break;
        const kvgen_spec *sp = jb->sp;
        int32_t h = (int32_t)(i % sp->H), kv = (int32_t)((i / sp->H) % 2),
                l = (int32_t)(i / (2 * sp->H));
        kvgen_head(sp, l, kv, h, jb->out + i * sp->S * sp->d);
    }
    return NULL;
}

/* The whole tensor, heads [h0, h1) of the flattened (l, kv, h) order. */
void kvgen_range(const kvgen_spec *sp, int64_t h0, int64_t h1, uint16_t *out, int32_t threads)
{
    job_t jb;
    jb.sp = sp;
    jb.out = out - h0 * sp->S * sp->d;
    jb.next = h0;
    jb.n_heads = h1;
    pthread_mutex_init(&jb.mu, NULL);
    if (threads < 1)
        threads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    for (int32_t i = 0; i < threads; i++)
        pthread_create(&th[i], NULL, worker, &jb);
    for (int32_t i = 0; i < threads; i++)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&jb.mu);
}

/* Per-chunk compression levels drawn uniformly from n_levels. */
void kvgen_chunk_levels(uint64_t seed, int64_t n_chunks, int32_t n_levels, uint8_t *out)
{
    uint64_t k = key_of(seed, P_LEVEL, 0, 0, 0);
    for (int64_t i = 0; i < n_chunks; i++)
        out[i] = (uint8_t)(draw(k, (uint64_t)i) % (uint64_t)n_levels);
}
