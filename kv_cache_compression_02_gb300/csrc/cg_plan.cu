// cg_plan.cu -- the bandwidth-adaptive level controller (host code only).
//
// CacheGen streams a context chunk by chunk and "dynamically adjusts
// compression according to bandwidth conditions" (gptget summary of arXiv
// 2310.07240, Methodology); it "adapts the compression level of different
// parts of a KV cache to cope with changes in available bandwidth, in order
// to maintain low context-loading delay", raising the compression level
// when bandwidth drops (the paper's abstract).  The pages give no formula.
// The rule implemented here is the plainest one they support:
//
//   Chunks are sent in order over one link, back to back.  Before chunk k
//   the controller takes, as the bandwidth estimate, the throughput it
//   observed while sending chunk k-1 (a given initial estimate for chunk
//   0), and picks the first level l (levels ordered finest to coarsest)
//   for which sending chunks k..n-1 all at level l at that estimate would
//   leave the last chunk's decode time before the deadline:
//       sum_{j>=k} bytes[j][l] / estimate  <=  deadline - now - decode[n-1].
//   If no level does, the coarsest one.  Chunk k's decode starts once its
//   bytes have arrived and chunk k-1's decode has ended.
//
// The link is a piecewise-constant bandwidth trace.  All arithmetic is
// IEEE double in a fixed order (the oracle repeats it operation for
// operation), and byte sums are exact 64-bit integers.
#include <cmath>
#include <vector>

#include "cachegen.h"

namespace {

// Time at which `bytes` bytes, sent from time t0 on, have all arrived.
double arrival(const cg_link_step *tr, int32_t n, double t0, double bytes) {
  if (!(bytes > 0.0)) return t0;
  double t = t0, rem = bytes, step_start = 0.0;
  for (int32_t i = 0; i < n; i++) {
    const bool last = i + 1 == n;
    const double step_end = last ? INFINITY : step_start + tr[i].seconds;
    if (t < step_end) {
      const double r = tr[i].bytes_per_s;
      const double cap = last ? INFINITY : r * (step_end - t);  // bytes the rest of step i carries
      if (rem <= cap) return t + rem / r;
      rem -= cap;
      t = step_end;
    }
    step_start = step_end;
  }
  return INFINITY;  // not reached: the last step has a positive rate
}

bool valid_trace(const cg_link_step *tr, int32_t n) {
  if (!tr || n < 1) return false;
  for (int32_t i = 0; i < n; i++)
    if (!(tr[i].seconds >= 0.0) || !std::isfinite(tr[i].seconds) || !(tr[i].bytes_per_s >= 0.0) ||
        !std::isfinite(tr[i].bytes_per_s))
      return false;
  return tr[n - 1].bytes_per_s > 0.0;
}

// Sends chunks with the given levels (choose = false) or chooses them
// (choose = true); fills levels, the timeline and the total time.
cg_status run(int32_t n_chunks, int32_t n_levels, const uint64_t *chunk_bytes, const cg_link_step *trace,
              int32_t n_steps, double initial_bytes_per_s, double deadline_s, const double *decode_s,
              bool choose, uint8_t *levels, double *timeline_out, double *total_s_out) {
  if (n_chunks < 1 || n_levels < 1 || n_levels > 8 || !chunk_bytes || !decode_s || !levels || !total_s_out ||
      !valid_trace(trace, n_steps))
    return CG_ERR_INVALID_ARG;
  for (int32_t k = 0; k < n_chunks; k++)
    if (!(decode_s[k] >= 0.0) || !std::isfinite(decode_s[k])) return CG_ERR_INVALID_ARG;
  if (choose) {
    if (!(initial_bytes_per_s > 0.0) || !std::isfinite(initial_bytes_per_s) || std::isnan(deadline_s))
      return CG_ERR_INVALID_ARG;
  } else {
    for (int32_t k = 0; k < n_chunks; k++)
      if (levels[k] >= n_levels) return CG_ERR_INVALID_ARG;
  }
  // suffix sums of the chunk sizes per level
  std::vector<uint64_t> suffix(size_t(n_chunks + 1) * n_levels, 0);
  for (int32_t k = n_chunks - 1; k >= 0; k--)
    for (int32_t l = 0; l < n_levels; l++)
      suffix[size_t(k) * n_levels + l] = suffix[size_t(k + 1) * n_levels + l] + chunk_bytes[size_t(k) * n_levels + l];
  double now = 0.0, estimate = initial_bytes_per_s, dec_end = 0.0;
  const double tail = decode_s[n_chunks - 1];
  for (int32_t k = 0; k < n_chunks; k++) {
    int32_t lv = levels[k];
    if (choose) {
      const double budget = deadline_s - now - tail;
      lv = n_levels - 1;
      for (int32_t l = 0; l < n_levels; l++) {
        const double need = double(suffix[size_t(k) * n_levels + l]) / estimate;
        if (need <= budget) {
          lv = l;
          break;
        }
      }
      levels[k] = uint8_t(lv);
    }
    const double bytes = double(chunk_bytes[size_t(k) * n_levels + lv]);
    const double start = now;
    now = arrival(trace, n_steps, start, bytes);
    if (now > start) estimate = bytes / (now - start);
    const double dstart = now > dec_end ? now : dec_end;
    dec_end = dstart + decode_s[k];
    if (timeline_out) {
      timeline_out[3 * k + 0] = start;
      timeline_out[3 * k + 1] = now;
      timeline_out[3 * k + 2] = dec_end;
    }
  }
  *total_s_out = dec_end;
  return CG_OK;
}

}  // namespace

extern "C" {

cg_status cg_plan_levels(int32_t n_chunks, int32_t n_levels, const uint64_t *chunk_bytes,
                         const cg_link_step *trace, int32_t n_steps, double initial_bytes_per_s,
                         double deadline_s, const double *decode_s, uint8_t *levels_out, double *timeline_out,
                         double *total_s_out) {
  return run(n_chunks, n_levels, chunk_bytes, trace, n_steps, initial_bytes_per_s, deadline_s, decode_s, true,
             levels_out, timeline_out, total_s_out);
}

cg_status cg_simulate_stream(int32_t n_chunks, int32_t n_levels, const uint64_t *chunk_bytes,
                             const cg_link_step *trace, int32_t n_steps, const uint8_t *levels,
                             const double *decode_s, double *timeline_out, double *total_s_out) {
  if (!levels) return CG_ERR_INVALID_ARG;
  std::vector<uint8_t> lv(levels, levels + (n_chunks > 0 ? n_chunks : 0));
  return run(n_chunks, n_levels, chunk_bytes, trace, n_steps, 1.0, 0.0, decode_s, false, lv.data(), timeline_out,
             total_s_out);
}

}  // extern "C"
