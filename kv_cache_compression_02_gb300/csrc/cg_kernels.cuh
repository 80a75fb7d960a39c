// cg_kernels.cuh -- host-side launchers of the codec's kernels (one per
// translation unit), called by the C-ABI entry points in cg_api.cu.
#pragma once

#include <cuda_runtime.h>

#include "cg_layout.cuh"

namespace cg {

struct Bases {
  float b[kMaxLevels];
};

// cg_fit.cu
// moments, done: zeroed workspace ([nstr][d][4] u64 and [nstr] u32) where the
// CTAs that share a head add up their sums
cudaError_t launch_stats(const Layout &lo, const uint16_t *kv, uint8_t *tables, const float *mult,
                         Bases bases, uint32_t *status, uint64_t *moments, uint32_t *done, cudaStream_t st);
cudaError_t launch_anchor_scales(const Layout &lo, const uint16_t *kv, float2 *scale_out,
                                 uint8_t *chunk_scratch, uint32_t *status, cudaStream_t st);
// pair_hist, pair_done: zeroed workspace ([kHistPairsMax][d][257] and
// [kHistPairsMax] u32) where the two CTAs of a shared (level, head) meet
cudaError_t launch_hist(const Layout &lo, const uint16_t *kv, const float2 *scale,
                        uint8_t *tables, double *ent_bits, uint32_t *ent_esc, uint32_t *pair_hist,
                        uint32_t *pair_done, cudaStream_t st);

// cg_encode.cu
// teams: the most chunks a level holds; live_levels: the levels holding any
cudaError_t launch_encode(const Layout &lo, const EncWs &w, const uint8_t *tables,
                          const uint16_t *kv, uint8_t *ws, int teams, int live_levels, cudaStream_t st);
cudaError_t launch_scan_compact(const Layout &lo, const EncWs &w, uint8_t *ws, uint8_t *out,
                                uint64_t cap, uint64_t *out_bytes, cudaStream_t st);

// cg_assemble.cu
uint64_t assemble_workspace_bytes(const Layout &lo);

// cg_decode.cu
// A paged KV cache: the pool of layer l, K/V kv is fp16
// [n_blocks][H][bt][d] at pools[2 l + kv]; token t of the sequence is row
// t mod bt of block table[t / bt].
struct PagedOut {
  uint16_t *const *pools;
  const int32_t *table;
  int32_t bt, n_blocks;
};
// Decodes chunks [k0, k1) of layers [l0, l1) into the contiguous kv buffer,
// or into the paged cache po when po is not null (kv is then unused).
cudaError_t launch_decode(const Layout &lo, const uint8_t *tables, const uint8_t *buf,
                          uint64_t bytes, int32_t k0, int32_t k1, uint16_t *kv, uint8_t *ws,
                          cudaStream_t st, const PagedOut *po, int32_t l0, int32_t l1);

}  // namespace cg
