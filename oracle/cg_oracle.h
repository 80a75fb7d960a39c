/*
 * cg_oracle.h -- plain, slow, single-threaded CPU oracle for the CacheGen
 * KV-cache codec (anchor/delta quantization + per-(layer, K/V, channel)
 * range coding).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this code: only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg may use it.  It shares no source, header,
 * table or helper with the CUDA library; the two meet only in the byte
 * format both write.
 *
 * Sources (CacheGen, SIGCOMM'24, as restated by the pages this build reads):
 *   - "Guide to CacheGen" (aifetchly blog), pillar 2 "Anchor-Based Delta
 *     Encoding" and its Step 2 sketch: first token of each group is the
 *     anchor, the other tokens are deltas against it; decode adds back.
 *   - same page, pillar 3 "Distribution-Aware Arithmetic Coding": per-layer
 *     frequency tables, probable symbols cost fractions of a bit.
 *   - same page, pillar 1 "Layer Sensitivity Disparity": finer steps early,
 *     coarser late.
 *   - gptget.net summary of arXiv 2310.07240, "Methodology": chunks with
 *     per-chunk compression levels; delta coding plus arithmetic coding;
 *     per layer and channel sensitivity.
 * Where the pages leave a step open the reading adopted is written beside
 * the function that takes it.
 *
 * Every floating-point step is IEEE binary32 round-to-nearest-even with no
 * contraction (compile with -ffp-contract=off); sigma is exact integer
 * arithmetic rounded to binary64 and then binary32.
 */
#ifndef CG_ORACLE_H
#define CG_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    ORC_OK = 0,
    ORC_ERR_INVALID_ARG = 1,
    ORC_ERR_NONFINITE = 2,
    ORC_ERR_CAPACITY = 3,
    ORC_ERR_CORRUPT = 4
};

#define ORC_M_BITS 16
#define ORC_M (1u << ORC_M_BITS)     /* total frequency of every table      */
#define ORC_NSYM 256                 /* alphabet: q+127 for |q|<=R, and ESC */
#define ORC_ESC 255
#define ORC_RANS_L (1u << 16)        /* lower bound of the 32-bit state     */
#define ORC_STEP_MIN 0x1p-12f        /* floor of the delta step             */
#define ORC_MAX_LEVELS 8

typedef struct {
    int32_t L, H, d; /* layers, KV heads, head dim                         */
    int32_t C;       /* tokens per chunk                                   */
    int32_t G;       /* tokens per anchor group                            */
    int32_t R;       /* alphabet radius (|q| <= R coded directly), 0..127  */
    int64_t S;       /* tokens                                             */
} orc_dims;

typedef struct {
    double entropy_bits; /* sum over tables of n'_s*log2(N'/n'_s)          */
    uint64_t n_symbols;  /* delta symbols coded                            */
    uint64_t n_esc;      /* escapes coded                                  */
    uint64_t n_words;    /* 16-bit words written                           */
    uint64_t fixed_bytes;/* headers, index, scales, anchors                */
    uint64_t state_bytes;/* rANS flush (4 bytes per lane per stream)       */
    uint64_t pad_bytes;  /* alignment padding                              */
} orc_stats;

/* ---- binary16 helpers, written from the IEEE 754 format ---------------- */
float orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_f16_rn(float f);

/* ---- the method's steps ------------------------------------------------ */
float orc_channel_sigma(const uint16_t *x, int64_t S, int64_t stride);
void orc_step(float base, float mult, float sigma, float *step, float *recip);
void orc_anchor_scale(float absmax, float *s, float *inv);
int32_t orc_anchor_code(float x, float s, float inv, float *ahat);
int32_t orc_delta_code(float x, float ahat, float recip);
int32_t orc_symbol(int32_t q, int32_t R);
void orc_normalize(const uint64_t n[256], uint32_t f[256], uint32_t cdf[257]);
uint16_t orc_reconstruct(int32_t q, float step, float ahat);

/* rANS over one stream of n_tok_delta tokens x d interleaved lanes.
 * sym/qv: [n][d] symbol index and quantized value; f/cdf: [d][256]/[d][257].
 * words_out must hold 3*n*d entries.  Returns the number of words. */
int64_t orc_rans_encode(int64_t n, int32_t d, const uint8_t *sym,
                        const int32_t *qv, const uint32_t *f,
                        const uint32_t *cdf, uint32_t *state_out,
                        uint16_t *words_out);
/* Exact inverse.  Returns ORC_OK or ORC_ERR_CORRUPT. */
int orc_rans_decode(int64_t n, int32_t d, const uint32_t *state,
                    const uint16_t *words, int64_t n_words, int64_t n_esc,
                    const uint32_t *f, const uint32_t *cdf, uint8_t *sym_out,
                    int32_t *q_out);

/* ---- container-level codec -------------------------------------------- */
size_t orc_tables_bytes(const orc_dims *dm, int32_t n_levels);
/* layer_mult: [L][2] multipliers, or NULL for tiers {0.5,1,2}[floor(3l/L)] */
int orc_fit_tables(const orc_dims *dm, int32_t n_levels,
                   const float *level_base, const float *layer_mult,
                   const uint16_t *kv, uint8_t *tables);
/* Fit one head (level, l, kv, h) from that head's [S][d] slice. */
int orc_fit_head(const orc_dims *dm, float base, float mult,
                 const uint16_t *head, float *step, float *recip,
                 uint16_t *cdf);

/* Encode one stream (chunk k of one head) given that head's [S][d] slice
 * and its tables at the chunk's level.  Writes the stream block (header,
 * states, words, padding) to blk (capacity blk_cap), the chunk's anchor
 * scales s[d] and int8 anchors [n_groups][d].  Returns the block size, or
 * a negative ORC_ERR_* code.  symcount[d][256] (may be NULL) accumulates
 * the coded symbol counts. */
int64_t orc_encode_stream(const orc_dims *dm, const uint16_t *head,
                          int64_t k, const float *step, const float *recip,
                          const uint16_t *cdf, float *s_out,
                          int8_t *anchors_out, uint8_t *blk, int64_t blk_cap,
                          uint64_t *symcount, orc_stats *st);

uint64_t orc_encode_bound(const orc_dims *dm);
/* sum_s n_s log2(N/n_s) of one table's 256 symbol counts (bits). */
double orc_table_entropy(const uint64_t *counts);
/* Header, chunk index and per-chunk fixed parts of a container, unpadded
 * (the structural bytes of the entropy bound, stream headers excluded). */
uint64_t orc_container_fixed_bytes(const orc_dims *dm);

int orc_encode(const orc_dims *dm, int32_t n_levels, const uint8_t *tables,
               const uint16_t *kv, const uint8_t *chunk_level, uint8_t *out,
               uint64_t cap, uint64_t *out_bytes, orc_stats *st);
/* Decode chunks [k0, k1) of a container into kv ([L,2,H,S,d] fp16). */
int orc_decode(const uint8_t *tables, size_t tables_bytes, const uint8_t *buf,
               uint64_t bytes, int64_t k0, int64_t k1, uint16_t *kv);
/* Decode one stream block of chunk k of one head into head ([S][d]). */
int orc_decode_stream(const orc_dims *dm, const uint8_t *blk, uint64_t blk_len,
                      int64_t k, const float *step, const uint16_t *cdf,
                      const float *s, const int8_t *anchors, uint16_t *head);

#ifdef __cplusplus
}
#endif
#endif
