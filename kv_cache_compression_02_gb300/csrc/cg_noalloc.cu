// cg_noalloc.cu -- cg_decode_noalloc: the decoder for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all: allocator-free embedded
// runtimes, or a serving loop that has handed the whole device to its own
// memory pool and may not grow it.  They own their inputs and outputs but
// cannot provide the small decode workspace (status word and per-level
// chunk lists) that cg_decode takes.  This entry point runs the same decode
// kernels with that workspace in a file-scope device array instead.
//
// The array is kNoallocScratchBytes (64 KiB) in every GPU that loads the
// library, held until the process exits.  All calls share it and it keeps
// the last call's contents; each call clears the status block first, and
// calls that overlap on the GPU race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "cachegen.h"
#include "cg_args.h"
#include "cg_kernels.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = 64 * 1024;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device and kept for the life of the process (host code only sees a
// stand-in symbol, not a device address; a cudaDeviceReset makes the kept
// address stale).
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" cg_status cg_decode_noalloc(const cg_dims *dims, const cg_params *params,
                                       const void *tables_dev, const void *bitstream_dev,
                                       uint64_t bitstream_bytes, int32_t chunk_begin,
                                       int32_t chunk_end, void *kv_dev, void *stream,
                                       const void **status_ws) {
  cg::Layout lo;
  if (!cg::layout_of(dims, params, lo) || !tables_dev || !bitstream_dev || !kv_dev)
    return CG_ERR_INVALID_ARG;
  if (!aligned16(tables_dev) || !aligned16(bitstream_dev) || !aligned16(kv_dev))
    return CG_ERR_INVALID_ARG;
  if (chunk_end < 0) chunk_end = lo.n_chunks;
  if (chunk_begin < 0 || chunk_begin > chunk_end || chunk_end > lo.n_chunks) return CG_ERR_INVALID_ARG;
  if (bitstream_bytes < lo.hdr_bytes) return CG_ERR_INVALID_ARG;
  if (cg::dec_ws(lo).bytes > kNoallocScratchBytes) return CG_ERR_CAPACITY;  // too many chunks
  void *ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return CG_ERR_CUDA;
  if (status_ws) *status_ws = ws;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);  // the status block starts at zero
  if (e == cudaSuccess && chunk_begin < chunk_end)
    e = cg::launch_decode(lo, static_cast<const uint8_t *>(tables_dev),
                          static_cast<const uint8_t *>(bitstream_dev), bitstream_bytes, chunk_begin,
                          chunk_end, static_cast<uint16_t *>(kv_dev), static_cast<uint8_t *>(ws), st,
                          nullptr, 0, lo.L);
  return e == cudaSuccess ? CG_OK : CG_ERR_CUDA;
}
