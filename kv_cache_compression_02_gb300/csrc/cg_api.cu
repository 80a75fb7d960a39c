// cg_api.cu -- the C-ABI entry points of libcachegen.so (declared and
// documented in include/cachegen.h): argument checks, workspace layout,
// host->device copies of the small per-call parameters, kernel launches.
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <vector>

#include "cachegen.h"
#include "cg_args.h"
#include "cg_kernels.cuh"

using namespace cg;

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

cg_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CG_OK : CG_ERR_CUDA; }

}  // namespace

// The decode entry points: chunks [k0, k1) of layers [l0, l1) (l1 = -1: to
// the last layer) into kv_dev, or into the paged cache *po when po is set.
static cg_status decode_common(const cg_dims *dims, const cg_params *params, const void *tables_dev,
                        const void *bitstream_dev, uint64_t bitstream_bytes, int32_t chunk_begin,
                        int32_t chunk_end, int32_t l0, int32_t l1, void *kv_dev, const PagedOut *po,
                        void *ws_dev, size_t ws_bytes, void *stream) {
  Layout lo;
  if (!layout_of(dims, params, lo) || !tables_dev || !bitstream_dev || (!po && !kv_dev) || !ws_dev)
    return CG_ERR_INVALID_ARG;
  if (!aligned(tables_dev, 16) || !aligned(bitstream_dev, 16) || !aligned(kv_dev, 16) ||
      !aligned(ws_dev, 256))
    return CG_ERR_INVALID_ARG;
  if (chunk_end < 0) chunk_end = lo.n_chunks;
  if (chunk_begin < 0 || chunk_begin > chunk_end || chunk_end > lo.n_chunks) return CG_ERR_INVALID_ARG;
  if (l1 < 0) l1 = lo.L;
  if (l0 < 0 || l0 > l1 || l1 > lo.L) return CG_ERR_INVALID_ARG;
  const DecWs w = dec_ws(lo);
  if (ws_bytes < w.bytes || bitstream_bytes < lo.hdr_bytes) return CG_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(ws_dev);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e == cudaSuccess && chunk_begin < chunk_end && l0 < l1)
    e = launch_decode(lo, static_cast<const uint8_t *>(tables_dev), static_cast<const uint8_t *>(bitstream_dev),
                      bitstream_bytes, chunk_begin, chunk_end, static_cast<uint16_t *>(kv_dev), ws, st, po, l0, l1);
  return cuda_status(e);
}

extern "C" {

int32_t cg_version(void) { return 1; }

const char *cg_status_str(cg_status s) {
  switch (s) {
    case CG_OK: return "CG_OK";
    case CG_ERR_INVALID_ARG: return "CG_ERR_INVALID_ARG";
    case CG_ERR_NONFINITE: return "CG_ERR_NONFINITE";
    case CG_ERR_CAPACITY: return "CG_ERR_CAPACITY";
    case CG_ERR_CORRUPT: return "CG_ERR_CORRUPT";
    case CG_ERR_CUDA: return "CG_ERR_CUDA";
    case CG_ERR_TIMEOUT: return "CG_ERR_TIMEOUT";
  }
  return "CG_ERR_UNKNOWN";
}

size_t cg_tables_bytes(const cg_dims *dims, const cg_params *params) {
  Layout lo;
  return layout_of(dims, params, lo) ? size_t(lo.tb_bytes) : 0;
}

size_t cg_workspace_bytes(const cg_dims *dims, const cg_params *params, int op) {
  Layout lo;
  if (!layout_of(dims, params, lo)) return 0;
  switch (op) {
    case CG_OP_FIT: return size_t(fit_ws(lo).bytes);
    case CG_OP_ENCODE: return size_t(enc_ws(lo).bytes);
    case CG_OP_DECODE: return size_t(dec_ws(lo).bytes);
    case CG_OP_ASSEMBLE: return size_t(assemble_workspace_bytes(lo));
  }
  return 0;
}

cg_status cg_encode_bound(const cg_dims *dims, const cg_params *params, uint64_t *max_bytes) {
  Layout lo;
  if (!layout_of(dims, params, lo) || !max_bytes) return CG_ERR_INVALID_ARG;
  uint64_t total = lo.hdr_bytes;
  for (int64_t k = 0; k < lo.n_chunks; k++)
    total += chunk_fixed(lo, k) +
             uint64_t(lo.nstr) * pad16(16 + 4 * uint64_t(lo.d) +
                                       2 * words_per_symbol(lo) * uint64_t(chunk_nd(lo, k)) * lo.d);
  *max_bytes = total;
  return CG_OK;
}

cg_status cg_fit_tables(const cg_dims *dims, const cg_params *params, const void *kv_dev,
                        void *tables_dev, void *ws_dev, size_t ws_bytes, void *stream) {
  Layout lo;
  if (!layout_of(dims, params, lo) || !kv_dev || !tables_dev || !ws_dev) return CG_ERR_INVALID_ARG;
  if (!aligned(kv_dev, 16) || !aligned(tables_dev, 16) || !aligned(ws_dev, 256)) return CG_ERR_INVALID_ARG;
  const FitWs w = fit_ws(lo);
  if (ws_bytes < w.bytes) return CG_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(ws_dev);
  uint8_t *tb = static_cast<uint8_t *>(tables_dev);

  std::vector<float> mult(2 * size_t(lo.L));
  for (int l = 0; l < lo.L; l++)
    for (int kv = 0; kv < 2; kv++) {
      const int tier = int((3 * int64_t(l)) / lo.L);
      mult[2 * l + kv] = params->layer_mult ? params->layer_mult[2 * l + kv]
                                            : (tier == 0 ? 0.5f : tier == 1 ? 1.0f : 2.0f);
    }
  Bases bases;
  for (int i = 0; i < kMaxLevels; i++) bases.b[i] = i < lo.n_levels ? params->level_base[i] : 0.0f;
  const uint64_t nc = uint64_t(lo.n_levels) * lo.L * 2 * lo.hd;
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ws + w.mult, mult.data(), 4 * mult.size(), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && lo.tb_recip > lo.tb_step + 4 * nc)
    e = cudaMemsetAsync(tb + lo.tb_step + 4 * nc, 0, lo.tb_recip - lo.tb_step - 4 * nc, st);
  if (e == cudaSuccess && lo.tb_cdf > lo.tb_recip + 4 * nc)
    e = cudaMemsetAsync(tb + lo.tb_recip + 4 * nc, 0, lo.tb_cdf - lo.tb_recip - 4 * nc, st);
  uint32_t *status = reinterpret_cast<uint32_t *>(ws + w.status);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws + w.moments, 0, w.bytes - w.moments, st);
  if (e == cudaSuccess)
    e = launch_stats(lo, static_cast<const uint16_t *>(kv_dev), tb,
                     reinterpret_cast<const float *>(ws + w.mult), bases, status,
                     reinterpret_cast<uint64_t *>(ws + w.moments), reinterpret_cast<uint32_t *>(ws + w.done), st);
  float2 *scale = reinterpret_cast<float2 *>(ws + w.scale);
  if (e == cudaSuccess)
    e = launch_anchor_scales(lo, static_cast<const uint16_t *>(kv_dev), scale, nullptr, status, st);
  if (e == cudaSuccess)
    e = launch_hist(lo, static_cast<const uint16_t *>(kv_dev), scale, tb, reinterpret_cast<double *>(ws + w.ent_bits),
                    reinterpret_cast<uint32_t *>(ws + w.ent_esc), reinterpret_cast<uint32_t *>(ws + w.pair_hist),
                    reinterpret_cast<uint32_t *>(ws + w.pair_done), st);
  return cuda_status(e);
}

cg_status cg_encode(const cg_dims *dims, const cg_params *params, const void *tables_dev,
                    const void *kv_dev, const uint8_t *chunk_level_host, void *out_dev,
                    uint64_t out_capacity, uint64_t *out_bytes_dev, void *ws_dev, size_t ws_bytes,
                    void *stream) {
  Layout lo;
  if (!layout_of(dims, params, lo) || !tables_dev || !kv_dev || !chunk_level_host || !out_dev ||
      !out_bytes_dev || !ws_dev)
    return CG_ERR_INVALID_ARG;
  if (!aligned(kv_dev, 16) || !aligned(tables_dev, 16) || !aligned(out_dev, 16) ||
      !aligned(out_bytes_dev, 8) || !aligned(ws_dev, 256))
    return CG_ERR_INVALID_ARG;
  const EncWs w = enc_ws(lo);
  if (ws_bytes < w.bytes || out_capacity < lo.hdr_bytes) return CG_ERR_INVALID_ARG;
  // per-level chunk lists, then the raw levels
  const size_t nk = size_t(lo.n_chunks);
  std::vector<uint8_t> meta(4 * kMaxLevels * (1 + nk) + nk, 0);
  int32_t *count = reinterpret_cast<int32_t *>(meta.data());
  int32_t *list = count + kMaxLevels;
  uint8_t *lv8 = meta.data() + 4 * kMaxLevels * (1 + nk);
  int teams = 0, live_levels = 0;
  for (size_t k = 0; k < nk; k++) {
    const int lv = chunk_level_host[k];
    if (lv >= lo.n_levels) return CG_ERR_INVALID_ARG;
    list[lv * nk + count[lv]] = int32_t(k);
    if (count[lv]++ == 0) live_levels++;
    if (count[lv] > teams) teams = count[lv];
    lv8[k] = uint8_t(lv);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(ws_dev);
  const uint16_t *kv = static_cast<const uint16_t *>(kv_dev);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ws + w.levels, meta.data(), meta.size(), cudaMemcpyHostToDevice, st);
  uint32_t *status = reinterpret_cast<uint32_t *>(ws + w.status);
  if (e == cudaSuccess) e = launch_anchor_scales(lo, kv, nullptr, ws + w.chunks, status, st);
  if (e == cudaSuccess) e = launch_encode(lo, w, static_cast<const uint8_t *>(tables_dev), kv, ws, teams, live_levels, st);
  if (e == cudaSuccess)
    e = launch_scan_compact(lo, w, ws, static_cast<uint8_t *>(out_dev), out_capacity, out_bytes_dev, st);
  return cuda_status(e);
}

cg_status cg_decode(const cg_dims *dims, const cg_params *params, const void *tables_dev,
                    const void *bitstream_dev, uint64_t bitstream_bytes, int32_t chunk_begin,
                    int32_t chunk_end, void *kv_dev, void *ws_dev, size_t ws_bytes, void *stream) {
  return decode_common(dims, params, tables_dev, bitstream_dev, bitstream_bytes, chunk_begin, chunk_end, 0, -1,
                       kv_dev, nullptr, ws_dev, ws_bytes, stream);
}

cg_status cg_decode_layers(const cg_dims *dims, const cg_params *params, const void *tables_dev,
                           const void *bitstream_dev, uint64_t bitstream_bytes, int32_t chunk_begin,
                           int32_t chunk_end, int32_t layer_begin, int32_t layer_end, void *kv_dev,
                           void *ws_dev, size_t ws_bytes, void *stream) {
  return decode_common(dims, params, tables_dev, bitstream_dev, bitstream_bytes, chunk_begin, chunk_end,
                       layer_begin, layer_end, kv_dev, nullptr, ws_dev, ws_bytes, stream);
}

cg_status cg_decode_paged(const cg_dims *dims, const cg_params *params, const void *tables_dev,
                          const void *bitstream_dev, uint64_t bitstream_bytes, int32_t chunk_begin,
                          int32_t chunk_end, void *const *pools_dev, const int32_t *block_table_dev,
                          int32_t block_tokens, int32_t n_blocks, void *ws_dev, size_t ws_bytes,
                          void *stream) {
  if (!pools_dev || !block_table_dev || block_tokens < 1 || n_blocks < 1 || !aligned(pools_dev, 8) ||
      !aligned(block_table_dev, 4))
    return CG_ERR_INVALID_ARG;
  const PagedOut po{reinterpret_cast<uint16_t *const *>(pools_dev), block_table_dev, block_tokens, n_blocks};
  return decode_common(dims, params, tables_dev, bitstream_dev, bitstream_bytes, chunk_begin, chunk_end, 0, -1,
                       nullptr, &po, ws_dev, ws_bytes, stream);
}

cg_status cg_entropy_bound(const cg_dims *dims, const cg_params *params, const void *ws_fit_dev, int32_t level,
                           double *bound_bytes) {
  Layout lo;
  if (!layout_of(dims, params, lo) || !ws_fit_dev || !bound_bytes || level < 0 || level >= lo.n_levels)
    return CG_ERR_INVALID_ARG;
  *bound_bytes = 0.0;
  const FitWs w = fit_ws(lo);
  const uint64_t per = uint64_t(lo.L) * 2 * lo.hd;  // tables of one level
  std::vector<double> bits(per);
  std::vector<uint32_t> esc(per);
  const uint8_t *ws = static_cast<const uint8_t *>(ws_fit_dev);
  if (cudaMemcpy(bits.data(), ws + w.ent_bits + 8 * uint64_t(level) * per, 8 * per, cudaMemcpyDeviceToHost) !=
          cudaSuccess ||
      cudaMemcpy(esc.data(), ws + w.ent_esc + 4 * uint64_t(level) * per, 4 * per, cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return CG_ERR_CUDA;
  double h = 0.0;
  uint64_t n_esc = 0;
  for (uint64_t t = 0; t < per; t++) {
    h += bits[t];
    n_esc += esc[t];
  }
  // structure that carries information: the header and chunk index; per chunk
  // its header, scales, anchors and stream offsets; per stream its header
  uint64_t fixed = 64 + 8 * uint64_t(lo.n_chunks);
  for (int64_t k = 0; k < lo.n_chunks; k++)
    fixed += 16 + 4 * uint64_t(lo.nstr) * lo.d + uint64_t(lo.nstr) * chunk_ng(lo, k) * lo.d + 4 * uint64_t(lo.nstr) +
             16 * uint64_t(lo.nstr);
  *bound_bytes = h / 8.0 + 4.0 * double(n_esc) + double(fixed);
  return CG_OK;
}

cg_status cg_read_status(const void *ws_dev) {
  if (!ws_dev) return CG_ERR_INVALID_ARG;
  uint32_t bits = 0;
  if (cudaMemcpy(&bits, ws_dev, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return CG_ERR_CUDA;
  if (bits & kStCorrupt) return CG_ERR_CORRUPT;
  if (bits & kStNonfinite) return CG_ERR_NONFINITE;
  if (bits & kStCapacity) return CG_ERR_CAPACITY;
  if (bits & kStTimeout) return CG_ERR_TIMEOUT;
  if (bits & kStBadArg) return CG_ERR_INVALID_ARG;
  return CG_OK;
}

cg_status cg_host_mapped(const void *host_ptr, void **dev_ptr) {
  if (!dev_ptr) return CG_ERR_INVALID_ARG;
  *dev_ptr = nullptr;
  if (!host_ptr) return CG_ERR_INVALID_ARG;
  // only page-locked host memory qualifies (device, managed and ordinary
  // pageable memory are refused); its device address may differ from the
  // host one where the platform has no unified addressing
  cudaPointerAttributes a{};
  void *d = nullptr;
  if (cudaPointerGetAttributes(&a, host_ptr) != cudaSuccess || a.type != cudaMemoryTypeHost ||
      cudaHostGetDevicePointer(&d, const_cast<void *>(host_ptr), 0) != cudaSuccess || !d) {
    (void)cudaGetLastError();  // an argument error, not a sticky one
    return CG_ERR_INVALID_ARG;
  }
  *dev_ptr = d;
  return CG_OK;
}

}  // extern "C"
