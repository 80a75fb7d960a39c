// cg_fit.cu -- fitting the per-(level, layer, K/V, channel) tables.
//
// The CacheGen pages build "empirical probability frequency tables for each
// layer and head based on calibration profiling" (Guide to CacheGen, pillar
// 3) and tune compression "by layer and channel sensitivity" (gptget
// summary of arXiv 2310.07240, Methodology).  Three kernels:
//   k_stats   sigma per channel from exact integer moments, then the step
//             b*m*sigma (floored at 2^-12) and its reciprocal per level;
//   k_anchor  per (chunk, head) the absmax of the anchor tokens -> scale s
//             and 127/absmax (also used by the encoder, which additionally
//             writes the int8 anchors);
//   k_hist    per (level, head) the 256-bin histogram of the delta symbols
//             over all chunks in shared memory, then the normalisation to
//             16-bit frequencies and the CDF, one warp per channel.
// All three are HBM-streaming kernels (no contraction, no tensor cores).
#include <cuda_fp16.h>

#include <algorithm>

#include "cg_kernels.cuh"

namespace cg {
namespace {

__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t half_bits(const uint4 &v, int i) {
  uint32_t w = (i < 2) ? v.x : (i < 4) ? v.y : (i < 6) ? v.z : v.w;
  return uint16_t((i & 1) ? (w >> 16) : (w & 0xFFFF));
}

// unsigned 128-bit integer to binary64, round to nearest even.  The top 64
// bits (with the leading one at bit 63) carry the rounding; any nonzero bit
// below them is folded into the lowest bit as a sticky bit, which lies
// below the rounding position of a 53-bit significand.
__device__ __forceinline__ double u128_to_double_rn(unsigned __int128 v) {
  uint64_t hi = uint64_t(v >> 64);
  if (hi == 0) return __ull2double_rn(uint64_t(v));
  int sh = 64 - __clzll(hi);  // 1..64
  uint64_t top = uint64_t(v >> sh);
  uint64_t below = uint64_t(v) & ((sh == 64) ? ~0ull : ((1ull << sh) - 1));
  top |= (below != 0) ? 1ull : 0ull;
  return __dmul_rn(__ull2double_rn(top), __longlong_as_double(int64_t(1023 + sh) << 52));
}

// ---------------------------------------------------------------- k_stats
// One CTA per head; each thread owns 4 channels and sums a strided subset of
// the tokens.  An fp16 value is X = M * 2^E (times 2^-24) with M < 2^11 and
// E <= 30, so X < 2^41; a 64-entry table gives 2^E and M's implicit bit for
// each sign and exponent field (the sign carried by the signed 2^E, so the
// signed sum needs no separate sign handling).  Most of the work is
// 32x32->64 multiply-adds, which run on the FMA pipe beside the integer ALU:
//   sum X    += M * (+-2^E)                      (signed, 64-bit)
//   X = a 2^21 + b (a < 2^20, b < 2^21):
//   sum X^2  = 2^42 sum a^2 + 2^22 sum ab + sum b^2
// Each of the three partial sums takes terms below 2^42, so 2^18 tokens
// per thread (S <= 2^22) keep it below 2^60.  Integer sums are
// order-free, so the reduction order does not matter for the result.
// A head's tiles may be shared by `parts` CTAs (so that the last wave of
// CTAs is not left to a few SMs): each adds its sums to the head's moments
// with 64-bit atomics (sum X^2 as a 128-bit value, the carry out of the low
// word added to the high word), and the last to finish computes sigma.
constexpr int kStatsThreads = 512;

struct Moments {
  int64_t T;
  uint64_t A2, AB, B2;
};

// Each sum is one 32x32->64 multiply-add with its 64-bit accumulator as the
// addend; AB sums a*b, and the reduction doubles it (2^22 instead of 2^21).
__device__ __forceinline__ void acc_moments(uint32_t h, const uint4 *ptab, Moments &m) {
  const uint4 pe = ptab[h >> 10];  // (+-2^E with h's sign, 2^E, the implicit bit of M)
  const uint32_t M = (h & 1023u) | pe.z;
  uint64_t X;
  asm("mul.wide.u32 %0, %1, %2;" : "=l"(X) : "r"(M), "r"(pe.y));
  asm("mad.wide.s32 %0, %1, %2, %0;" : "+l"(m.T) : "r"(M), "r"(pe.x));
  const uint32_t xl = uint32_t(X), xh = uint32_t(X >> 32);
  const uint32_t a = __funnelshift_r(xl, xh, 21), b = xl & 0x1FFFFFu;  // X = a 2^21 + b
  asm("mad.wide.u32 %0, %1, %1, %0;" : "+l"(m.A2) : "r"(a));
  asm("mad.wide.u32 %0, %1, %2, %0;" : "+l"(m.AB) : "r"(a), "r"(b));
  asm("mad.wide.u32 %0, %1, %1, %0;" : "+l"(m.B2) : "r"(b));
}

// The head's rows stream through shared memory in 16 KB tiles, four in
// flight: one thread issues each tile as a bulk asynchronous copy that
// completes on the tile's mbarrier, so the loads need no registers and the
// next tiles land while this one is summed.
constexpr uint32_t kStatsTile = 16384, kStatsStages = 4;
constexpr uint32_t kWaitLimit = 1u << 22;  // try_wait rounds before a wait gives up

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase) {
  for (uint32_t it = 0; it < kWaitLimit; it++) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(phase)
        : "memory");
    if (done) return true;
  }
  return false;
}

__global__ void __launch_bounds__(kStatsThreads, 2)
k_stats(Layout lo, const uint16_t *__restrict__ kv, uint8_t *__restrict__ tables,
        const float *__restrict__ mult, Bases bases, uint32_t *status, unsigned long long *moments,
        uint32_t *done, int parts) {
  extern __shared__ __align__(128) unsigned char smem[];  // kStatsStages tiles, then the reduction
  __shared__ __align__(8) uint64_t bars[kStatsStages];
  __shared__ uint4 ptab[64];  // per sign and exponent field: (+-2^max(e-1, 0), 2^max(e-1, 0), e ? 1024 : 0)
  __shared__ int s_timeout, s_last;
  if (threadIdx.x < 64) {
    const uint32_t e = threadIdx.x & 31u, p = e ? 1u << (e - 1) : 1u;
    ptab[threadIdx.x] = make_uint4(threadIdx.x & 32u ? uint32_t(-int32_t(p)) : p, p, e ? 1024u : 0u, 0u);
  }
  const int si = int(blockIdx.x) / parts, part = int(blockIdx.x) % parts;
  const int tpr = lo.d / 4;                 // threads per token row
  const int rows = kStatsThreads / tpr;     // token rows summed side by side
  const int col = threadIdx.x % tpr, row = threadIdx.x / tpr;
  const uint32_t row_bytes = 2u * uint32_t(lo.d);
  const uint8_t *head = reinterpret_cast<const uint8_t *>(kv + uint64_t(si) * lo.S * lo.d);
  const uint64_t head_bytes = uint64_t(lo.S) * row_bytes;  // a multiple of 16
  const uint64_t ntiles = (head_bytes + kStatsTile - 1) / kStatsTile;
  const uint64_t t0 = ntiles * uint64_t(part) / uint64_t(parts), t1 = ntiles * uint64_t(part + 1) / uint64_t(parts);

  auto issue = [&](uint64_t t) {  // tile t into stage (t - t0) % kStatsStages
    const uint32_t st = uint32_t((t - t0) % kStatsStages);
    const uint64_t left = head_bytes - t * kStatsTile;
    const uint32_t bytes = uint32_t(left < kStatsTile ? left : kStatsTile);
    const uint32_t bar = smem_addr(&bars[st]);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem + st * kStatsTile)),
        "l"(head + t * kStatsTile), "r"(bytes), "r"(bar)
        : "memory");
  };
  if (threadIdx.x == 0) {
    s_timeout = 0;
    for (uint32_t st = 0; st < kStatsStages; st++)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bars[st])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (uint64_t t = t0; t < t1 && t < t0 + kStatsStages; t++) issue(t);
  }
  __syncthreads();

  Moments mo[4];
#pragma unroll
  for (int i = 0; i < 4; i++) mo[i] = Moments{0, 0, 0, 0};
  uint32_t bad = 0;  // bit 15 of a half: an all-ones exponent (Inf or NaN) was seen
  uint64_t t = t0;
  for (; t < t1; t++) {
    const uint32_t st = uint32_t((t - t0) % kStatsStages);
    if (!mbar_wait(smem_addr(&bars[st]), uint32_t((t - t0) / kStatsStages) & 1u)) s_timeout = 1;
    __syncthreads();  // every thread knows whether the tile landed
    if (s_timeout) break;
    const uint8_t *tile = smem + st * kStatsTile;
    const uint64_t left = head_bytes - t * kStatsTile;
    const uint32_t nr = uint32_t(left < kStatsTile ? left : kStatsTile) / row_bytes;
    for (uint32_t r = row; r < nr; r += rows) {
      const uint2 vv = *reinterpret_cast<const uint2 *>(tile + r * row_bytes + 8 * col);
      const uint32_t hw[4] = {vv.x & 0xFFFFu, vv.x >> 16, vv.y & 0xFFFFu, vv.y >> 16};
      bad |= ((vv.x & 0x7C007C00u) + 0x04000400u) | ((vv.y & 0x7C007C00u) + 0x04000400u);
#pragma unroll
      for (int i = 0; i < 4; i++) acc_moments(hw[i], ptab, mo[i]);  // a non-finite value only spoils a flagged result
    }
    __syncthreads();  // the stage has been read: it can take the next tile
    if (threadIdx.x == 0 && t + kStatsStages < t1) issue(t + kStatsStages);
  }
  // A copy that has not landed after 2^22 try_wait rounds: every tile is an
  // in-bounds, 16-byte aligned read of the caller's kv, which completes
  // unless the memory system itself has failed.  The CTA sets the TIMEOUT
  // bit, waits (bounded again) for each copy it still has in flight and
  // returns.  A copy still in flight after that cannot be cancelled: it may
  // land later in shared memory the SM has since given to another CTA, so
  // CG_ERR_TIMEOUT tells the caller that the context can no longer be
  // trusted (the header says so), not merely that the tables are invalid.
  if (s_timeout) {
    if (threadIdx.x == 0) {
      atomicOr(status, kStTimeout);
      for (uint64_t u = t; u < t1 && u < t + kStatsStages; u++)
        mbar_wait(smem_addr(&bars[(u - t0) % kStatsStages]), uint32_t((u - t0) / kStatsStages) & 1u);
    }
    return;
  }
  if (bad & 0x80008000u) atomicOr(status, kStNonfinite);

  int64_t *sT = reinterpret_cast<int64_t *>(smem);  // [rows][d] each
  uint64_t *sA2 = reinterpret_cast<uint64_t *>(sT + rows * lo.d);
  uint64_t *sAB = sA2 + rows * lo.d;
  uint64_t *sB2 = sAB + rows * lo.d;
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const int c = row * lo.d + 4 * col + i;
    sT[c] = mo[i].T;
    sA2[c] = mo[i].A2;
    sAB[c] = mo[i].AB;
    sB2[c] = mo[i].B2;
  }
  __syncthreads();
  __int128 Ts = 0;
  unsigned __int128 Qs = 0;
  if (threadIdx.x < lo.d) {
    const int c = threadIdx.x;
    for (int r = 0; r < rows; r++) {
      Ts += sT[r * lo.d + c];
      Qs += ((unsigned __int128)sA2[r * lo.d + c] << 42) + ((unsigned __int128)sAB[r * lo.d + c] << 22) +
            (unsigned __int128)sB2[r * lo.d + c];
    }
  }
  if (parts > 1) {  // add to the head's moments; the last CTA of the head goes on with their totals
    unsigned long long *m = moments + (uint64_t(si) * lo.d + threadIdx.x) * 4;
    if (threadIdx.x < lo.d) {
      atomicAdd(&m[0], (unsigned long long)(int64_t)Ts);  // |sum X| < 2^62: two's complement
      const unsigned long long ql = (unsigned long long)Qs, qh = (unsigned long long)(Qs >> 64);
      const unsigned long long old = atomicAdd(&m[1], ql);
      const unsigned long long carry = (old + ql < old) ? 1ull : 0ull;
      if (qh + carry) atomicAdd(&m[2], qh + carry);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&done[si], 1u) == uint32_t(parts - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x < lo.d) {
      Ts = (int64_t)atomicAdd(&m[0], 0ull);
      Qs = ((unsigned __int128)atomicAdd(&m[2], 0ull) << 64) | atomicAdd(&m[1], 0ull);
    }
  }
  if (threadIdx.x < lo.d) {
    const int c = threadIdx.x;
    unsigned __int128 aT = (unsigned __int128)(Ts < 0 ? -Ts : Ts);
    unsigned __int128 num = (unsigned __int128)(uint64_t)lo.S * Qs - aT * aT;
    double var = __ddiv_rn(u128_to_double_rn(num),
                           __ull2double_rn(uint64_t(lo.S) * uint64_t(lo.S)));
    var = __dmul_rn(var, 0x1p-48);
    float sigma = __double2float_rn(__dsqrt_rn(var));

    const int h = si % lo.H, kvi = (si / lo.H) % 2, l = si / (2 * lo.H);
    const float m = mult[l * 2 + kvi];
    float *stepv = reinterpret_cast<float *>(tables + lo.tb_step);
    float *recipv = reinterpret_cast<float *>(tables + lo.tb_recip);
    for (int lv = 0; lv < lo.n_levels; lv++) {
      float st = __fmul_rn(__fmul_rn(bases.b[lv], m), sigma);
      if (!(st >= 0x1p-12f)) st = 0x1p-12f;
      uint64_t ix = tab_index(lo, lv, l, kvi, h * lo.d + c);
      stepv[ix] = st;
      recipv[ix] = __fdiv_rn(1.0f, st);
    }
  }
  if (si == 0 && threadIdx.x == 0) {  // tables header (by the one CTA of head 0 that gets here)
    uint32_t *hd = reinterpret_cast<uint32_t *>(tables);
    hd[0] = 0x42544743u;  // "CGTB"
    hd[1] = 1;
    hd[2] = lo.L;
    hd[3] = lo.H;
    hd[4] = lo.d;
    hd[5] = lo.n_levels;
    hd[6] = lo.R;
    hd[7] = 0;
    float *fb = reinterpret_cast<float *>(tables + 32);
    for (int i = 0; i < kMaxLevels; i++) fb[i] = i < lo.n_levels ? bases.b[i] : 0.0f;
  }
}

// ---------------------------------------------------------------- k_anchor
// One CTA per (chunk, head).  Fit mode writes (s, 127/absmax) per channel;
// encode mode writes s and the int8 anchors into the chunk's fixed-part
// scratch, laid out exactly as in the container.
constexpr int kAnchorThreads = 256;

__global__ void __launch_bounds__(kAnchorThreads)
k_anchor(Layout lo, const uint16_t *__restrict__ kv, float2 *__restrict__ scale_out,
         uint8_t *__restrict__ chunk_scratch, uint32_t *status) {
  __shared__ float s_max[kAnchorThreads * 8];
  __shared__ float s_inv[128];
  const int k = blockIdx.x, si = blockIdx.y;
  const int tpr = lo.d / 8, rows = kAnchorThreads / tpr;
  const int col = threadIdx.x % tpr, row = threadIdx.x / tpr;
  const int ng = chunk_ng(lo, k);
  const int64_t t0 = int64_t(k) * lo.C;
  const uint16_t *head = kv + uint64_t(si) * lo.S * lo.d + 8 * col;

  float amax[8];
#pragma unroll
  for (int i = 0; i < 8; i++) amax[i] = 0.0f;
  bool bad = false;
  for (int g = row; g < ng; g += rows) {
    uint4 v = ld_nc_v4(head + (t0 + int64_t(g) * lo.G) * lo.d);
#pragma unroll
    for (int i = 0; i < 8; i++) {
      uint16_t h = half_bits(v, i);
      if (((h >> 10) & 31u) == 31u) { bad = true; continue; }
      amax[i] = fmaxf(amax[i], fabsf(__half2float(__ushort_as_half(h))));
    }
  }
  if (bad) atomicOr(status, kStNonfinite);
#pragma unroll
  for (int i = 0; i < 8; i++) s_max[row * lo.d + 8 * col + i] = amax[i];
  __syncthreads();
  if (threadIdx.x < lo.d) {
    const int c = threadIdx.x;
    float a = 0.0f;
    for (int r = 0; r < rows; r++) a = fmaxf(a, s_max[r * lo.d + c]);
    float s = 0.0f, inv = 0.0f;
    if (a != 0.0f) {
      s = __fdiv_rn(a, 127.0f);
      inv = __fdiv_rn(127.0f, a);
    }
    if (scale_out) scale_out[(uint64_t(k) * lo.nstr + si) * lo.d + c] = make_float2(s, inv);
    s_inv[c] = inv;
    if (chunk_scratch) {
      float *sv = reinterpret_cast<float *>(chunk_scratch + uint64_t(k) * lo.fixed_full + lo.sec_s);
      sv[uint64_t(si) * lo.d + c] = s;
    }
  }
  if (!chunk_scratch) return;
  __syncthreads();
  int8_t *anc = reinterpret_cast<int8_t *>(chunk_scratch + uint64_t(k) * lo.fixed_full + lo.sec_anc);
  for (int g = row; g < ng; g += rows) {
    uint4 v = ld_nc_v4(head + (t0 + int64_t(g) * lo.G) * lo.d);
    uint32_t packed[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 8; i++) {
      float x = __half2float(__ushort_as_half(half_bits(v, i)));
      int a = __float2int_rn(__fmul_rn(x, s_inv[8 * col + i]));
      a = max(-127, min(127, a));
      packed[i / 4] |= (uint32_t(a) & 0xFFu) << (8 * (i % 4));
    }
    *reinterpret_cast<uint2 *>(anc + (uint64_t(si) * ng + g) * lo.d + 8 * col) =
        make_uint2(packed[0], packed[1]);
  }
}

// ---------------------------------------------------------------- k_hist
// One CTA per (level, head).  A team of d/4 threads (four channels each)
// takes one anchor group at a time: it rebuilds a_hat from the chunk's
// scale, quantizes the group's deltas and counts the symbols into a shared
// histogram of d rows of 257 counts.  Then one warp per channel normalises
// its counts and records, for the entropy bound of a container coded with
// this level, the bits its symbols carry at their own frequencies,
// sum_s n_s log2(N / n_s) (log2 in fp32, summed in fp64), and its escapes.
// Grid rows from split0 on come in pairs (the last wave's heads): the two
// CTAs of a pair count the first and the second half of the head's groups,
// add their histograms into the pair's in the workspace, and the one that
// finishes last normalises the sum (integer counts: exact in any order).
constexpr int kHistThreads = 1024;

__global__ void __launch_bounds__(kHistThreads)
k_hist(Layout lo, const uint16_t *__restrict__ kv, const float2 *__restrict__ scale,
       uint8_t *__restrict__ tables, double *__restrict__ ent_bits, uint32_t *__restrict__ ent_esc,
       uint32_t *pair_hist, uint32_t *pair_done, int split0) {
  extern __shared__ __align__(16) uint32_t hist[];  // [d][257]
  __shared__ int s_last;
  const int lv = blockIdx.x;
  int si = blockIdx.y, part = 0, nparts = 1, pair = 0;
  if (si >= split0) {
    const int j = int(blockIdx.y) - split0;
    si = split0 + j / 2;
    part = j & 1;
    nparts = 2;
    pair = (j / 2) * int(gridDim.x) + lv;  // below kHistPairsMax (the launcher's bound)
  }
  const int h = si % lo.H, kvi = (si / lo.H) % 2, l = si / (2 * lo.H);
  for (int i = threadIdx.x; i < lo.d * 257; i += blockDim.x) hist[i] = 0;
  __syncthreads();

  // four channels per thread (one 8-byte load per token); channel 4 col + i
  // counts into histogram row i * (d/4) + col, so with the odd row stride
  // the threads of a warp counting the same symbol hit different banks
  const int tpr = lo.d / 4, teams = kHistThreads / tpr;
  const int col = threadIdx.x % tpr, team = threadIdx.x / tpr;
  const int c0 = 4 * col;
  const float4 r4 = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(tables + lo.tb_recip) +
                                                       tab_index(lo, lv, l, kvi, h * lo.d + c0));
  const float rc[4] = {r4.x, r4.y, r4.z, r4.w};
  uint32_t *hrow[4];
#pragma unroll
  for (int i = 0; i < 4; i++) hrow[i] = hist + (i * tpr + col) * 257;
  const uint2 *head = reinterpret_cast<const uint2 *>(kv + uint64_t(si) * lo.S * lo.d + c0);
  const int64_t n_groups = int64_t(lo.n_chunks - 1) * lo.ng_full + lo.ng_last;
  const int64_t g_lo = n_groups * part / nparts, g_hi = n_groups * (part + 1) / nparts;
  const uint32_t R = uint32_t(lo.R);

  for (int64_t gi = g_lo + team; gi < g_hi; gi += teams) {
    const int k = int(gi / lo.ng_full), g = int(gi % lo.ng_full);
    const int64_t t0 = int64_t(k) * lo.C;
    const int64_t ta = t0 + int64_t(g) * lo.G;
    const int te = int(min(ta + lo.G, t0 + chunk_ntok(lo, k)) - ta);  // rows of the group
    const float4 *sp = reinterpret_cast<const float4 *>(scale + (uint64_t(k) * lo.nstr + si) * lo.d + c0);
    const uint2 *grow = head + ta * tpr;
    // the scales, the anchor row and the first nine delta rows are loaded
    // together: one memory round trip for a group of up to ten tokens
    const float4 s01 = sp[0], s23 = sp[1];  // (s, 127/absmax) of the four channels
    const uint2 wa = __ldg(grow);
    uint2 w9[9];
#pragma unroll
    for (int u = 0; u < 9; u++) w9[u] = 1 + u < te ? __ldg(grow + (1 + u) * tpr) : make_uint2(0, 0);
    const float sc[4] = {s01.x, s01.z, s23.x, s23.z}, inv[4] = {s01.y, s01.w, s23.y, s23.w};
    const uint32_t ha[4] = {wa.x & 0xFFFFu, wa.x >> 16, wa.y & 0xFFFFu, wa.y >> 16};
    float ah[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const int a = max(-127, min(127, __float2int_rn(__fmul_rn(__half2float(__ushort_as_half(uint16_t(ha[i]))), inv[i]))));
      ah[i] = __fmul_rn(float(a), sc[i]);
    }
#define CG_COUNT_ROW(W)                                                                                   \
  {                                                                                                       \
    const uint32_t hw[4] = {(W).x & 0xFFFFu, (W).x >> 16, (W).y & 0xFFFFu, (W).y >> 16};                 \
    _Pragma("unroll") for (int i = 0; i < 4; i++) {                                                       \
      const int q =                                                                                       \
          __float2int_rn(__fmul_rn(__fsub_rn(__half2float(__ushort_as_half(uint16_t(hw[i]))), ah[i]), rc[i])); \
      const int sym = uint32_t(q) + R <= 2 * R ? q + 127 : kEsc; /* |q| <= R as one unsigned compare */  \
      atomicAdd(&hrow[i][sym], 1u);                                                                       \
    }                                                                                                     \
  }
#pragma unroll
    for (int u = 0; u < 9; u++)
      if (1 + u < te) CG_COUNT_ROW(w9[u])
    for (int tb = 10; tb < te; tb += 8) {  // groups of more than ten tokens: 8 more rows in flight at a time
      uint2 w8[8];
#pragma unroll
      for (int u = 0; u < 8; u++) w8[u] = tb + u < te ? __ldg(grow + (tb + u) * tpr) : make_uint2(0, 0);
#pragma unroll
      for (int u = 0; u < 8; u++)
        if (tb + u < te) CG_COUNT_ROW(w8[u])
    }
#undef CG_COUNT_ROW
  }
  __syncthreads();
  if (nparts > 1) {
    uint32_t *gh = pair_hist + uint64_t(pair) * lo.d * 257;
    for (int i = threadIdx.x; i < lo.d * 257; i += blockDim.x)
      if (hist[i]) atomicAdd(&gh[i], hist[i]);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&pair_done[pair], 1u) == 1u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int i = threadIdx.x; i < lo.d * 257; i += blockDim.x) hist[i] = __ldcg(&gh[i]);
    __syncthreads();
  }

  // normalisation: one warp per channel, 8 symbols per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  uint16_t *cdfv = reinterpret_cast<uint16_t *>(tables + lo.tb_cdf);
  for (int c = warp; c < lo.d; c += nwarps) {
    uint32_t n[8];
    uint32_t nsum = 0, best = 0;
    int bests = 8 * lane;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      n[i] = hist[((c & 3) * (lo.d / 4) + (c >> 2)) * 257 + 8 * lane + i];
      nsum += n[i];
      if (n[i] > best) { best = n[i]; bests = 8 * lane + i; }
    }
    uint32_t N = nsum;
#pragma unroll
    for (int o = 16; o; o >>= 1) N += __shfl_xor_sync(0xffffffffu, N, o);
    // argmax with the lowest symbol on ties
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      uint32_t ob = __shfl_xor_sync(0xffffffffu, best, o);
      int os = __shfl_xor_sync(0xffffffffu, bests, o);
      if (ob > best || (ob == best && os < bests)) { best = ob; bests = os; }
    }
    const int arg = N ? bests : 127;
    uint32_t f[8], fsum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      f[i] = 1u + (N ? uint32_t((uint64_t(n[i]) * (kM - 256u)) / N) : 0u);
      fsum += f[i];
    }
    uint32_t F = fsum;
#pragma unroll
    for (int o = 16; o; o >>= 1) F += __shfl_xor_sync(0xffffffffu, F, o);
    if (arg >= 8 * lane && arg < 8 * lane + 8) {
      f[arg - 8 * lane] += kM - F;
      fsum += kM - F;
    }
    uint32_t incl = fsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    uint32_t run = incl - fsum;
    uint32_t packed[4];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      uint32_t c_a = run;
      run += f[i];
      uint32_t c_b = run;
      run += f[i + 1];
      packed[i / 2] = (c_a & 0xFFFFu) | (c_b << 16);
    }
    uint64_t ix = tab_index(lo, lv, l, kvi, h * lo.d + c);
    *reinterpret_cast<uint4 *>(cdfv + ix * 256 + 8 * lane) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
    double bits = 0.0;  // sum over the lane's symbols of n log2(N / n)
#pragma unroll
    for (int i = 0; i < 8; i++)
      if (n[i]) bits += double(n[i]) * double(log2f(float(N) / float(n[i])));
#pragma unroll
    for (int o = 16; o; o >>= 1) bits += __shfl_xor_sync(0xffffffffu, bits, o);
    if (lane == 31) {  // lane 31 holds symbols 248..255: n[7] counts the escapes
      ent_bits[ix] = bits;
      ent_esc[ix] = n[7];
    }
  }
}

}  // namespace

// parts per head: the number (1 to 8, at least a tile each) with the least
// estimated time, in tiles: ceil(heads * parts / wave) waves of CTAs, each
// ceil(tiles / parts) tiles plus about three tiles' worth for the copies'
// start and the reduction at the end (a CTA's fixed cost, measured on the
// 70B and 7B workloads: 64-tile heads gain nothing from parts).
cudaError_t launch_stats(const Layout &lo, const uint16_t *kv, uint8_t *tables, const float *mult,
                         Bases bases, uint32_t *status, uint64_t *moments, uint32_t *done, cudaStream_t st) {
  const int rows = kStatsThreads / (lo.d / 4);
  const size_t smem = std::max(size_t(kStatsStages) * kStatsTile, size_t(rows) * lo.d * 32);
  cudaError_t e = cudaFuncSetAttribute(k_stats, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_stats, kStatsThreads, smem);
  if (e != cudaSuccess) return e;
  const int64_t wave = int64_t(sms) * per_sm;
  const uint64_t ntiles = (uint64_t(lo.S) * 2 * lo.d + kStatsTile - 1) / kStatsTile;
  int parts = 1;
  if (wave > 0) {
    uint64_t best = 0;
    for (int p = 1; p <= 8 && uint64_t(p) <= ntiles; p++) {
      const uint64_t waves = uint64_t((int64_t(lo.nstr) * p + wave - 1) / wave);
      const uint64_t cost = waves * ((ntiles + p - 1) / p + 3);
      if (p == 1 || cost < best) {
        best = cost;
        parts = p;
      }
    }
  }
  k_stats<<<unsigned(lo.nstr) * unsigned(parts), kStatsThreads, smem, st>>>(
      lo, kv, tables, mult, bases, status, reinterpret_cast<unsigned long long *>(moments), done, parts);
  return cudaGetLastError();
}

cudaError_t launch_anchor_scales(const Layout &lo, const uint16_t *kv, float2 *scale_out,
                                 uint8_t *chunk_scratch, uint32_t *status, cudaStream_t st) {
  dim3 grid(lo.n_chunks, lo.nstr);
  k_anchor<<<grid, kAnchorThreads, 0, st>>>(lo, kv, scale_out, chunk_scratch, status);
  return cudaGetLastError();
}

// The last wave, as for the decoder: when the CTAs past the last full wave,
// doubled, still run side by side (and the pairs fit the workspace), their
// (level, head) units take two CTAs each.
cudaError_t launch_hist(const Layout &lo, const uint16_t *kv, const float2 *scale,
                        uint8_t *tables, double *ent_bits, uint32_t *ent_esc, uint32_t *pair_hist,
                        uint32_t *pair_done, cudaStream_t st) {
  const size_t smem = size_t(lo.d) * 257 * 4;
  cudaError_t e = cudaFuncSetAttribute(k_hist, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_hist, kHistThreads, smem);
  if (e != cudaSuccess) return e;
  const int wave = sms * per_sm, live = lo.nstr * lo.n_levels, rest = wave > 0 ? live % wave : 0;
  int split = 0;
  if (rest > 0) {
    const int r = min((rest + lo.n_levels - 1) / lo.n_levels, lo.nstr);
    if (2 * r * lo.n_levels <= wave && r * lo.n_levels <= kHistPairsMax) split = r;
  }
  dim3 grid(lo.n_levels, lo.nstr + split);
  k_hist<<<grid, kHistThreads, smem, st>>>(lo, kv, scale, tables, ent_bits, ent_esc, pair_hist, pair_done,
                                           lo.nstr - split);
  return cudaGetLastError();
}

}  // namespace cg
