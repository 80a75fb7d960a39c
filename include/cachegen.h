/*
 * cachegen.h -- C ABI of libcachegen.so, a GB300 (sm_103a) implementation
 * of the data-parallel hot path of the CacheGen KV-cache codec.
 *
 * What the codec computes (CacheGen, SIGCOMM'24, as the pages restate it):
 *   - "Anchor-Based Delta Encoding" (Guide to CacheGen, pillar 2): tokens
 *     are split into groups; the first token of each group is an anchor
 *     kept at high precision (here int8 with a per-chunk, per-channel
 *     absmax scale); the others are deltas against the anchor.
 *   - "Layer Sensitivity Disparity" (Guide, pillar 1) and "layer-specific
 *     compression levels" (gptget summary, Methodology): deltas are
 *     quantized with a step b_level * m_layer * sigma_channel.
 *   - "Distribution-Aware Arithmetic Coding" (Guide, pillar 3; gptget
 *     Methodology, delta + arithmetic coding): quantized deltas are range
 *     coded (rANS, 16-bit words, 2^16 total frequency) with one frequency
 *     table per (level, layer, K/V, channel).
 *   - Chunks with per-chunk compression levels, streamed and decoded in
 *     step with transmission (gptget Methodology; Guide pillar 4
 *     "Overlapped Streaming Decoder Pipeline").
 *
 * Conventions for every call:
 *   - KV tensors are fp16, laid out [L][2][H][S][d] (layer, K=0/V=1, KV
 *     head, token, head dim), contiguous, d innermost, 16-byte aligned.
 *   - Pointers named *_dev are device pointers allocated by the caller;
 *     the library allocates nothing and keeps no state between calls.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *     compute calls are asynchronous on it; argument errors are returned
 *     synchronously before anything is enqueued.
 *   - Errors found on the device (non-finite input, a container or table
 *     that fails validation, an output that does not fit) set bits of a
 *     status word at the start of the caller's workspace; each call clears
 *     it first.  Read it with cg_read_status() after synchronising.
 *     Nothing traps or aborts; after an error the affected outputs are
 *     unspecified, the CUDA context stays usable.
 *   - GPU limits: 8 <= d <= 128 with d a multiple of 8; 1 <= G; 1 <= C;
 *     1 <= S <= 2^22 (exact 128-bit channel moments); 1 <= n_levels <= 8; 0 <= alphabet_radius <= 127.
 *
 * Byte formats (little-endian, every section 16-byte aligned, padding 0):
 *   tables:    64-byte header {"CGTB", u32 1, u32 L, H, d, n_levels, R, 0,
 *              f32 level_base[8]}, f32 step[NL][L][2][H*d], f32
 *              recip[NL][L][2][H*d], u16 cdf[NL][L][2][H*d][256].
 *   container: 64-byte header {"CGKV", u32 1, u32 L, H, d, C, G, R, u64 S,
 *              u32 n_levels, u32 n_chunks, u64 total_bytes, 0, 0},
 *              u64 chunk_off[n_chunks]; per chunk k: {u16 level, u16 0,
 *              u32 t0, u32 n_tok, u32 n_groups}, f32 s[L][2][H][d], i8
 *              anchors[L][2][H][n_groups][d], u32 stream_off[L][2][H]
 *              (from the chunk start), then one stream per (l, kv, h):
 *              {u32 n_words, u32 n_esc, u32 n_delta, u32 0}, u32
 *              state[d], u16 words[n_words] (decode order: token
 *              ascending, lane ascending; per lane the renormalisation
 *              word, then an escape's low and high halves).
 */
#ifndef CACHEGEN_H
#define CACHEGEN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CG_OK = 0,
    CG_ERR_INVALID_ARG = 1, /* bad dims/params/pointer/size (synchronous;
                               also a bad page-table entry found on the
                               device by cg_decode_paged)                  */
    CG_ERR_NONFINITE = 2,   /* an input element is Inf or NaN              */
    CG_ERR_CAPACITY = 3,    /* output or workspace too small              */
    CG_ERR_CORRUPT = 4,     /* container or tables failed validation      */
    CG_ERR_CUDA = 5,        /* a CUDA launch or copy failed               */
    CG_ERR_TIMEOUT = 6      /* a bulk copy of cg_fit_tables' moment pass
                               did not land within its bounded wait: the
                               memory system failed, and the copy may still
                               land later in shared memory given to other
                               work, so treat the CUDA context as unusable */
} cg_status;

typedef struct {
    int32_t L;        /* layers                                          */
    int32_t H;        /* KV heads per layer                              */
    int32_t d;        /* head dim = rANS lanes per stream                */
    int32_t C;        /* tokens per chunk (streaming / level unit)       */
    int32_t G;        /* tokens per anchor group (first = anchor)        */
    int32_t reserved; /* must be 0                                       */
    int64_t S;        /* tokens                                          */
} cg_dims;

typedef struct {
    int32_t n_levels;         /* compression levels, 1..8                  */
    float level_base[8];      /* base step b_level (x sigma x multiplier)  */
    const float *layer_mult;  /* host [L][2] multipliers (K, V); NULL =    */
                              /* 0.5 / 1 / 2 for the first/middle/last     */
                              /* third of the layers                       */
    int32_t alphabet_radius;  /* R: |q| <= R coded directly, else escape   */
} cg_params;

enum { CG_OP_FIT = 0, CG_OP_ENCODE = 1, CG_OP_DECODE = 2, CG_OP_ASSEMBLE = 3 };

/* Size in bytes of the tables blob for (dims, params): the per-(level,
 * layer, K/V, channel) quantisation steps and 16-bit CDF tables that the
 * encoder and decoder share (Guide to CacheGen, pillar 3: frequency tables
 * per layer and head from calibration profiling; gptget summary of arXiv
 * 2310.07240, Methodology: per-layer/channel statistics).  0 on bad input. */
size_t cg_tables_bytes(const cg_dims *dims, const cg_params *params);

/* Workspace bytes needed by operation `op` (CG_OP_*).  0 on bad input.
 * Encode needs about the fp16 size of the KV (word scratch for the chunk
 * streams the pages' encoder produces: gptget summary, Methodology, chunked
 * bitstreams); fit and decode need a few bytes per chunk and channel.  The
 * caller allocates it; the library allocates nothing. */
size_t cg_workspace_bytes(const cg_dims *dims, const cg_params *params, int op);

/* Largest container cg_encode can produce for these dims (the container
 * format above: the chunked bitstream with its stream-offset index that the
 * pages' encoder emits, gptget summary, Methodology).  With the full
 * alphabet (alphabet_radius 127) every stream holds at most one 16-bit word
 * per delta symbol, escapes included: a stream that would need more (more
 * than its raw fp16 size) is rejected with CG_ERR_CAPACITY.  So the bound
 * is about the fp16 size of the KV plus anchors and headers.  With a
 * smaller radius, where most symbols may escape, the limit is three words
 * per symbol.  An output of this size only overflows along with that
 * error. */
cg_status cg_encode_bound(const cg_dims *dims, const cg_params *params, uint64_t *max_bytes);

/* Fit the tables (Guide to CacheGen, pillar 3, "Distribution-Aware
 * Arithmetic Coding": empirical frequency tables for each layer and head
 * from calibration profiling; gptget summary of arXiv 2310.07240,
 * Methodology: statistics per layer and channel; pillar 1, "Layer
 * Sensitivity Disparity": coarser steps in deeper layers).  Computed here:
 * per (layer, K/V, channel) sigma over all S tokens (exact
 * integer moments, rounded once), step = max(b*m*sigma, 2^-12) and its
 * reciprocal per level, and per (level, layer, K/V, channel) the 256-bin
 * histogram of the delta symbols over all chunks, normalised to 16-bit
 * frequencies (f_s = 1 + floor(n_s*65280/N), remainder to the most
 * frequent symbol) and stored as CDFs.
 *   kv_dev:     fp16 [L][2][H][S][d], read only.
 *   tables_dev: cg_tables_bytes() bytes, written.
 *   ws_dev:     cg_workspace_bytes(CG_OP_FIT) bytes, 256-byte aligned.
 * Device errors: CG_ERR_NONFINITE. */
cg_status cg_fit_tables(const cg_dims *dims, const cg_params *params, const void *kv_dev,
                        void *tables_dev, void *ws_dev, size_t ws_bytes, void *stream);

/* Encode kv into a container (format above): per chunk and head, int8
 * anchor tokens with the other tokens delta-coded against them (Guide to
 * CacheGen, pillar 2, "Anchor-Based Delta Encoding"), deltas quantised with
 * the layer-adaptive step (pillar 1) and range coded with the per-channel
 * tables (pillar 3; gptget summary, Methodology: delta encoding plus
 * arithmetic coding into compact bitstreams); chunk k at level
 * chunk_level_host[k] (host array of n_chunks bytes, < n_levels).
 *   out_dev:       out_capacity bytes; on success the first *out_bytes_dev
 *                  bytes are the container (bit-identical to the oracle's).
 *   out_bytes_dev: device u64, written with the container size (also when
 *                  it exceeds out_capacity, so the caller can retry).
 *   ws_dev:        cg_workspace_bytes(CG_OP_ENCODE) bytes.
 * Device errors: CG_ERR_NONFINITE; CG_ERR_CAPACITY when the container does
 * not fit in out_capacity (nothing is written) or when one stream's words
 * exceed the per-symbol limit described at cg_encode_bound. */
cg_status cg_encode(const cg_dims *dims, const cg_params *params, const void *tables_dev,
                    const void *kv_dev, const uint8_t *chunk_level_host, void *out_dev,
                    uint64_t out_capacity, uint64_t *out_bytes_dev, void *ws_dev,
                    size_t ws_bytes, void *stream);

/* The container cg_encode would make for levels chunk_level_host, built
 * from containers of the same KV encoded at one level each (with the same
 * tables): chunk k is copied verbatim from level_containers[chunk_level_host[k]],
 * behind a new header and chunk index.  A serving system can encode a
 * context once per level and assemble any level choice (e.g. from
 * cg_plan_levels) with device copies only (gptget summary of arXiv
 * 2310.07240, Methodology: compression adjusted to the bandwidth while
 * chunks stream).
 *   level_containers: host array of n_levels device pointers (16-byte
 *                     aligned; may be NULL for levels no chunk uses);
 *   level_bytes:      host array of their sizes;
 *   out_dev, out_capacity, out_bytes_dev: as for cg_encode (the size is
 *                     written even when it exceeds out_capacity);
 *   ws_dev:           cg_workspace_bytes(CG_OP_ASSEMBLE) bytes.
 * Device errors: CG_ERR_CORRUPT (a source header, index entry or chunk
 * header that does not match dims/params and the requested level),
 * CG_ERR_CAPACITY (nothing written).  The result is bit-identical to
 * cg_encode's for the same levels. */
cg_status cg_assemble(const cg_dims *dims, const cg_params *params, const void *const *level_containers,
                      const uint64_t *level_bytes, const uint8_t *chunk_level_host, void *out_dev,
                      uint64_t out_capacity, uint64_t *out_bytes_dev, void *ws_dev, size_t ws_bytes,
                      void *stream);

/* Decode chunks [chunk_begin, chunk_end) of a container into the full KV
 * buffer kv_dev (fp16 [L][2][H][S][d]; only those chunks' tokens are
 * written): the range decode, anchor + dequantised delta per token, that
 * turns the received bitstream back into KV "in real time, synchronized
 * with transmission" (gptget summary of arXiv 2310.07240, Methodology;
 * Guide to CacheGen, Step 2 decode_sequence and pillar 4, chunk i decoded
 * while chunk i+1 is in flight).  chunk_end = -1 means all chunks.  dims/params must be the
 * ones the container was made with (the kernel checks them against the
 * container header).  The container must be bitstream_bytes long and the
 * caller must keep it and the tables alive until the stream reaches the
 * decode.  ws_dev: cg_workspace_bytes(CG_OP_DECODE) bytes.
 * Host-resident buffers: bitstream_dev and kv_dev (here and in
 * cg_decode_layers) may be pinned host memory mapped into the device's
 * address space (cudaHostAlloc, or cudaHostRegister with
 * cudaHostRegisterMapped), passed as the device address cg_host_mapped
 * returns.  The decoder then reads the container
 * and writes the tokens across the host link itself, with no staging copy
 * (the receiver of a streamed context decodes as the bytes arrive: Guide to
 * CacheGen, pillar 4).  Tables and workspace stay in device memory.
 * Device errors: CG_ERR_CORRUPT (header/offset/table mismatch, a stream
 * whose lanes do not end in the initial state, or whose word or escape
 * count disagrees with its header); decoding never reads outside the
 * container. */
cg_status cg_decode(const cg_dims *dims, const cg_params *params, const void *tables_dev,
                    const void *bitstream_dev, uint64_t bitstream_bytes, int32_t chunk_begin,
                    int32_t chunk_end, void *kv_dev, void *ws_dev, size_t ws_bytes, void *stream);

/* cg_decode restricted to layers [layer_begin, layer_end) (layer_end = -1:
 * to the last layer): only those layers' tokens of the chosen chunks are
 * written.  Decoding the layers in groups, in layer order, with an event
 * recorded after each group lets a consumer start on the first layers
 * while the later ones are still being decoded (Guide to CacheGen, pillar
 * 4: layers stream in execution order, layer 0 first, so generation can
 * begin once layer 0 is decoded).  Values are bit-identical to cg_decode's; arguments
 * and errors are as for cg_decode, plus CG_ERR_INVALID_ARG for a layer
 * range outside [0, L]. */
cg_status cg_decode_layers(const cg_dims *dims, const cg_params *params, const void *tables_dev,
                           const void *bitstream_dev, uint64_t bitstream_bytes, int32_t chunk_begin,
                           int32_t chunk_end, int32_t layer_begin, int32_t layer_end, void *kv_dev,
                           void *ws_dev, size_t ws_bytes, void *stream);

/* cg_decode into a paged KV cache instead of the contiguous buffer: the
 * cache is split into blocks of block_tokens tokens, and a block table maps
 * each logical block of the sequence to a physical block of a page pool
 * (the block-table cache layout of paged-attention servers).  The Guide to
 * CacheGen's deployment notes (integrating with PagedAttention: direct
 * paged buffer injection) ask the decompressor to write reconstructed
 * tokens straight into the server's block-table pages; this call does.
 *   pools_dev:       device array of 2*L pointers; pools_dev[2*l + kv] is
 *                    the page pool of layer l, K (kv = 0) or V (kv = 1):
 *                    fp16 [n_blocks][H][block_tokens][d], 16-byte aligned.
 *   block_table_dev: device int32 array of ceil(S / block_tokens) entries;
 *                    token t of the sequence goes to row t % block_tokens
 *                    of block block_table_dev[t / block_tokens], which must
 *                    lie in [0, n_blocks).  The same table serves every
 *                    layer and K/V; distinct tokens must map to distinct
 *                    rows (the library does not check this).
 *   block_tokens, n_blocks: both >= 1.
 * Everything else (chunk range, workspace, errors) is as for cg_decode:
 * only the chosen chunks' tokens are written, every value is bit-identical
 * to cg_decode's.  A block id out of range, or a null or misaligned pool
 * pointer, is found on the device: those rows are not written and the
 * status reads CG_ERR_INVALID_ARG (after CG_ERR_CORRUPT, which wins). */
cg_status cg_decode_paged(const cg_dims *dims, const cg_params *params, const void *tables_dev,
                          const void *bitstream_dev, uint64_t bitstream_bytes, int32_t chunk_begin,
                          int32_t chunk_end, void *const *pools_dev, const int32_t *block_table_dev,
                          int32_t block_tokens, int32_t n_blocks, void *ws_dev, size_t ws_bytes,
                          void *stream);

/* cg_decode without a workspace argument, for callers that cannot
 * allocate device memory: allocator-free embedded runtimes, or a serving
 * loop whose device memory is all owned by its own pool and may not grow.
 * (No counterpart in the CacheGen pages; it is a deployment convenience.)
 * Arguments and results are those of cg_decode (the same argument checks);
 * the decode workspace instead lives in a 64 KiB device array inside the
 * library, held by every GPU that loads it until exit, which limits the
 * container to 2040 chunks (CG_ERR_CAPACITY beyond).
 *   status_ws: if not NULL, receives the device address of that array;
 *              pass it to cg_read_status() after synchronising.
 * The first call on each device looks the array's address up and keeps it
 * for the life of the process; after cudaDeviceReset the kept address is
 * stale, so do not call this entry point again in that process.  All calls share the array and it
 * keeps the last call's contents: each call clears the status first, and
 * calls that overlap on the GPU race on it, so serialise them.  It calls no
 * allocating routine. */
cg_status cg_decode_noalloc(const cg_dims *dims, const cg_params *params, const void *tables_dev,
                            const void *bitstream_dev, uint64_t bitstream_bytes,
                            int32_t chunk_begin, int32_t chunk_end, void *kv_dev, void *stream,
                            const void **status_ws);

/* ---- Bandwidth-adaptive streaming (host only, no GPU) ------------------
 * CacheGen adapts each chunk's compression level to the bandwidth the link
 * offers while the context streams (gptget summary of arXiv 2310.07240,
 * Methodology; the paper's abstract: raise the compression level when
 * bandwidth drops, to keep the loading delay low).  The pages give no
 * formula; the rule below is the plainest one they support.
 *
 * A link is a piecewise-constant bandwidth trace: step i lasts `seconds`
 * at `bytes_per_s`, starting where step i-1 ended (time 0 for step 0); the
 * last step lasts forever and must have a positive rate. */
typedef struct {
    double seconds;
    double bytes_per_s;
} cg_link_step;

/* Chooses a level per chunk.  Chunks are sent in order, back to back.
 * Before chunk k the bandwidth estimate is the throughput observed while
 * sending chunk k-1 (initial_bytes_per_s for chunk 0); the level is the
 * first l (levels ordered finest first) with
 *     sum_{j>=k} chunk_bytes[j][l] / estimate <= deadline_s - now - decode_s[n-1],
 * else the last (coarsest) level.  Chunk k's decode starts when its bytes
 * have arrived and chunk k-1's decode has ended and lasts decode_s[k].
 *   chunk_bytes:  host u64 [n_chunks][n_levels], chunk k's bytes at level l
 *                 (e.g. from containers encoded at each level).
 *   decode_s:     host double [n_chunks], >= 0.
 *   levels_out:   host u8 [n_chunks].
 *   timeline_out: host double [n_chunks][3] = (send start, arrival,
 *                 decode end), or NULL.
 *   total_s_out:  when the last decode ends.
 * Arithmetic is IEEE double in a fixed order; byte sums are exact.
 * Errors: CG_ERR_INVALID_ARG (1 <= n_levels <= 8, n_chunks >= 1, finite
 * non-negative durations and rates, positive initial estimate). */
cg_status cg_plan_levels(int32_t n_chunks, int32_t n_levels, const uint64_t *chunk_bytes,
                         const cg_link_step *trace, int32_t n_steps, double initial_bytes_per_s,
                         double deadline_s, const double *decode_s, uint8_t *levels_out,
                         double *timeline_out, double *total_s_out);

/* The same link and decode model for given levels (e.g. one fixed level,
 * for comparison): fills timeline_out (or NULL) and total_s_out. */
cg_status cg_simulate_stream(int32_t n_chunks, int32_t n_levels, const uint64_t *chunk_bytes,
                             const cg_link_step *trace, int32_t n_steps, const uint8_t *levels,
                             const double *decode_s, double *timeline_out, double *total_s_out);

/* The entropy bound of a container whose chunks are all coded at `level`
 * with the tables of the last cg_fit_tables that used ws_fit_dev (whose
 * histograms count exactly those symbols when the same KV is encoded):
 * sum over the level's (layer, K/V, channel) tables of n_s log2(N / n_s)
 * bits, / 8, plus 4 bytes per escape, plus the container's information-
 * bearing structure (headers, chunk index, scales, anchors, stream offsets
 * and stream headers, without padding).  It is the size an ideal coder of
 * each table's empirical distribution would reach (Guide to CacheGen,
 * pillar 3, "Distribution-Aware Arithmetic Coding"), the measure the
 * container is held to within 1%.  The per-table terms are summed on the
 * host in double (log2 evaluated in fp32 on the device).  Blocking: it reads
 * the workspace after synchronising with the device.
 * Errors: CG_ERR_INVALID_ARG (bad dims/params, level out of range, NULL),
 * CG_ERR_CUDA. */
cg_status cg_entropy_bound(const cg_dims *dims, const cg_params *params, const void *ws_fit_dev, int32_t level,
                           double *bound_bytes);

/* Status of the last call that used this workspace (blocking read of the
 * device status word; synchronise the call's stream first).  It reports the
 * device-side checks of the container format above (no passage of the pages
 * covers error reporting; this is the library's own contract). */
cg_status cg_read_status(const void *ws_dev);

/* The device address of host memory that is pinned and mapped into the
 * device's address space (a helper for the host-resident decode that lets
 * the decoder read a streamed container as it lands, Guide to CacheGen,
 * pillar 4; the pages have no call of their own for it) (cudaHostAlloc, or cudaHostRegister with
 * cudaHostRegisterMapped), for the host-resident decode described at
 * cg_decode.  *dev_ptr receives it (NULL on error).  Errors:
 * CG_ERR_INVALID_ARG when host_ptr is not in page-locked host memory
 * (device, managed and pageable memory are refused) or a pointer is NULL.
 * Host only; it launches nothing. */
cg_status cg_host_mapped(const void *host_ptr, void **dev_ptr);

/* Human-readable name of a status code (static string; part of the
 * library's own error contract, no counterpart in the pages). */
const char *cg_status_str(cg_status status);

/* Library ABI version (1): the version of this header and of the tables
 * and container formats above (no counterpart in the pages). */
int32_t cg_version(void);

#ifdef __cplusplus
}
#endif
#endif
