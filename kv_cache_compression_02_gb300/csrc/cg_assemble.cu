// cg_assemble.cu -- a mixed-level container out of single-level ones.
//
// CacheGen encodes a context at several compression levels and, while it
// streams, picks each chunk's level from the bandwidth at hand (gptget
// summary of arXiv 2310.07240, Methodology: "dynamically adjusting
// compression according to bandwidth conditions").  A chunk's bytes depend
// only on its own tokens and its level's tables, and every offset inside a
// chunk is relative to the chunk, so a container for any level choice is
// the chosen chunks copied verbatim behind a new header and chunk index --
// byte for byte what cg_encode makes for those levels.  Two kernels:
//
//   k_assemble_plan  one thread validates each source container's header,
//                    and each chosen chunk's index entry and header, then
//                    lays the chunks out and writes the new header and
//                    index (nothing is written when a check fails or the
//                    result does not fit).
//   k_assemble_copy  16-byte copies of the chunks, a CTA row per chunk.
#include <vector>

#include "cachegen.h"
#include "cg_layout.cuh"

namespace cg {
namespace {

struct AsmSrc {
  const uint8_t *p[kMaxLevels];
  uint64_t bytes[kMaxLevels];
};

// Workspace: status at 0; per chunk {u64 src offset, u64 size, u64 dst offset}
// at 256; then the chunk levels (u8).
struct AsmWs {
  uint64_t plan, levels, bytes;
};
AsmWs asm_ws(const Layout &lo) {
  AsmWs w;
  w.plan = 256;
  w.levels = w.plan + 24 * uint64_t(lo.n_chunks);
  w.bytes = pad256(w.levels + uint64_t(lo.n_chunks));
  return w;
}

__device__ __forceinline__ uint32_t ld32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint64_t ld64(const uint8_t *p) { return *reinterpret_cast<const uint64_t *>(p); }

__global__ void k_assemble_plan(Layout lo, AsmSrc src, uint8_t *out, uint64_t cap, uint64_t *out_bytes,
                                uint8_t *ws, AsmWs w) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  uint32_t *status = reinterpret_cast<uint32_t *>(ws);
  uint64_t *plan = reinterpret_cast<uint64_t *>(ws + w.plan);
  const uint8_t *lv8 = ws + w.levels;
  bool ok = true;
  uint32_t checked = 0;  // source containers whose header passed
  uint64_t pos = lo.hdr_bytes;
  for (int k = 0; ok && k < lo.n_chunks; k++) {
    const int lv = lv8[k];
    const uint8_t *s = src.p[lv];
    const uint64_t sb = src.bytes[lv];
    if (!((checked >> lv) & 1u)) {
      ok = sb >= lo.hdr_bytes && ld32(s) == 0x564B4743u && ld32(s + 4) == 1 && ld32(s + 8) == uint32_t(lo.L) &&
           ld32(s + 12) == uint32_t(lo.H) && ld32(s + 16) == uint32_t(lo.d) && ld32(s + 20) == uint32_t(lo.C) &&
           ld32(s + 24) == uint32_t(lo.G) && ld32(s + 28) == uint32_t(lo.R) && ld64(s + 32) == uint64_t(lo.S) &&
           ld32(s + 40) == uint32_t(lo.n_levels) && ld32(s + 44) == uint32_t(lo.n_chunks) && ld64(s + 48) == sb;
      checked |= 1u << lv;
      if (!ok) break;
    }
    const uint64_t off = ld64(s + 64 + 8 * uint64_t(k));
    const uint64_t end = k + 1 < lo.n_chunks ? ld64(s + 64 + 8 * uint64_t(k + 1)) : sb;
    ok = !(off & 15) && !(end & 15) && off >= lo.hdr_bytes && end >= off && end <= sb &&
         end - off >= chunk_fixed(lo, k) && ld32(s + off) == uint32_t(lv);  // the chunk header's level
    plan[3 * k + 0] = off;
    plan[3 * k + 1] = end - off;
    plan[3 * k + 2] = pos;
    pos += end - off;
  }
  *out_bytes = pos;
  if (!ok) {
    atomicOr(status, kStCorrupt);
    return;
  }
  if (pos > cap) {
    atomicOr(status, kStCapacity);
    return;
  }
  // header: the first chunk's source header with the new total; then the index
  const uint8_t *h0 = src.p[lv8[0]];
  for (int b = 0; b < 64; b += 8) *reinterpret_cast<uint64_t *>(out + b) = ld64(h0 + b);
  *reinterpret_cast<uint64_t *>(out + 48) = pos;
  for (uint64_t b = 64; b < lo.hdr_bytes; b += 8) {
    const uint64_t k = (b - 64) / 8;
    *reinterpret_cast<uint64_t *>(out + b) = k < uint64_t(lo.n_chunks) ? plan[3 * k + 2] : 0;
  }
}

__global__ void __launch_bounds__(256) k_assemble_copy(Layout lo, AsmSrc src, uint8_t *out, const uint8_t *ws,
                                                       AsmWs w) {
  const uint32_t status = *reinterpret_cast<const uint32_t *>(ws);
  if (status & (kStCorrupt | kStCapacity)) return;
  const int k = blockIdx.x;
  const uint64_t *plan = reinterpret_cast<const uint64_t *>(ws + w.plan);
  const uint4 *s = reinterpret_cast<const uint4 *>(src.p[ws[w.levels + k]] + plan[3 * k + 0]);
  uint4 *d = reinterpret_cast<uint4 *>(out + plan[3 * k + 2]);
  const uint64_t n = plan[3 * k + 1] / 16;
  for (uint64_t u = uint64_t(blockIdx.y) * blockDim.x + threadIdx.x; u < n; u += uint64_t(gridDim.y) * blockDim.x)
    d[u] = __ldg(s + u);
}

bool layout_ok(const cg_dims *dm, const cg_params *pr, Layout &lo) {
  return dm && pr && dm->reserved == 0 &&
         make_layout(lo, dm->L, dm->H, dm->d, dm->C, dm->G, dm->S, pr->alphabet_radius, pr->n_levels);
}

}  // namespace

uint64_t assemble_workspace_bytes(const Layout &lo) { return asm_ws(lo).bytes; }

}  // namespace cg

extern "C" cg_status cg_assemble(const cg_dims *dims, const cg_params *params,
                                 const void *const *level_containers, const uint64_t *level_bytes,
                                 const uint8_t *chunk_level_host, void *out_dev, uint64_t out_capacity,
                                 uint64_t *out_bytes_dev, void *ws_dev, size_t ws_bytes, void *stream) {
  using namespace cg;
  Layout lo;
  if (!layout_ok(dims, params, lo) || !level_containers || !level_bytes || !chunk_level_host || !out_dev ||
      !out_bytes_dev || !ws_dev)
    return CG_ERR_INVALID_ARG;
  auto al = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  if (!al(out_dev, 16) || !al(out_bytes_dev, 8) || !al(ws_dev, 256)) return CG_ERR_INVALID_ARG;
  const AsmWs w = asm_ws(lo);
  if (ws_bytes < w.bytes || out_capacity < lo.hdr_bytes) return CG_ERR_INVALID_ARG;
  AsmSrc src{};
  std::vector<uint8_t> lv(size_t(lo.n_chunks));
  for (int k = 0; k < lo.n_chunks; k++) {
    const int l = chunk_level_host[k];
    if (l >= lo.n_levels) return CG_ERR_INVALID_ARG;
    const void *p = level_containers[l];
    if (!p || !al(p, 16) || level_bytes[l] < lo.hdr_bytes) return CG_ERR_INVALID_ARG;
    src.p[l] = static_cast<const uint8_t *>(p);
    src.bytes[l] = level_bytes[l];
    lv[size_t(k)] = uint8_t(l);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(ws_dev);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ws + w.levels, lv.data(), lv.size(), cudaMemcpyHostToDevice, st);
  uint8_t *out = static_cast<uint8_t *>(out_dev);
  if (e == cudaSuccess) {
    k_assemble_plan<<<1, 32, 0, st>>>(lo, src, out, out_capacity, out_bytes_dev, ws, w);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    k_assemble_copy<<<dim3(lo.n_chunks, 64), 256, 0, st>>>(lo, src, out, ws, w);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? CG_OK : CG_ERR_CUDA;
}
