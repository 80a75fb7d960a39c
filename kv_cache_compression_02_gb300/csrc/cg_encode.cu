// cg_encode.cu -- the parallel range-coder encoder.
//
// CacheGen "encodes large tensors into compact bitstreams" with delta coding
// plus arithmetic coding (gptget summary of arXiv 2310.07240, Methodology;
// Guide to CacheGen, pillars 2-3).  Here every (chunk, layer, K/V, head) is
// one rANS stream whose d lanes (channels) share one 16-bit word sequence.
//
//   k_encode          one CTA per (level, head); a team of d/4 threads
//                     encodes one chunk's stream, 4 lanes per thread, in
//                     reverse token order, the next rows loaded while the
//                     current ones are coded.  Per token the team orders its
//                     words with a shuffle scan (lanes descending) and stages
//                     them in a shared-memory ring; each full block of 256
//                     words goes backwards into the stream's scratch slot
//                     with 16-byte stores, so the scratch ends up in decode
//                     order.
//   k_scan_chunks     per chunk: exclusive scan of the padded stream sizes.
//   k_scan_total      chunk offsets and the container size.
//   k_compact_fixed   container header, chunk headers, scales, anchors and
//                     the stream index, copied into place.
//   k_compact_stream  stream headers, states and words copied into place.
// No kernel waits on another CTA; the scan is split into two launches.
#include <cuda_fp16.h>

#include "cg_kernels.cuh"

namespace cg {
namespace {

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// One rANS encode step after renormalisation (x < f * 2^16):
//   x' = floor(x / f) * 2^16 + (x mod f) + cdf.
// The quotient (< 2^16) is estimated in fp32 as x * rcp(f) - 1/4: the
// estimate's error is below 2^-6, so after the offset it lies strictly
// between x/f - 0.27 and x/f - 0.23 and truncates to the quotient or one
// less; one exact correction step finishes it.
__device__ __forceinline__ uint32_t rans_put(uint32_t x, uint32_t f, uint32_t c) {
  uint32_t q = __float2uint_rz(__fmaf_rz(__uint2float_rz(x), rcp_approx(float(f)), -0.25f));
  uint32_t r = x - q * f;
  if (r >= f) {
    q += 1;
    r -= f;
  }
  return (q << 16) + r + c;
}

template <int T>
__device__ __forceinline__ uint32_t team_mask() {
  const int lane = threadIdx.x & 31;
  return T == 32 ? 0xffffffffu : (((1u << T) - 1u) << (lane & ~(T - 1)));
}

constexpr int kLpt = kLanesPerThread;

// Words staged per team before they go to the scratch slot.  A token adds at
// most 12 words per thread (384 per team), and at most 255 wait in a partly
// filled block, so 1024 slots never overwrite a word not yet stored.
constexpr uint32_t kWordRing = 1024;

// Block blk of 256 words (encoder order 256 blk ..) from the ring to the
// scratch slot, whose words [cap - 256 (blk + 1), cap - 256 blk) it fills,
// 16 bytes per store; units below u0 are skipped.
__device__ __forceinline__ void flush_block(const uint16_t *ring, uint16_t *wout, int64_t cap, uint32_t blk,
                                            uint32_t u0, int i, int T) {
  const uint4 *src = reinterpret_cast<const uint4 *>(ring + (kWordRing - 256) - 256 * (blk & 3));
  uint4 *dst = reinterpret_cast<uint4 *>(wout + cap - 256 * (int64_t(blk) + 1));
  for (uint32_t u = u0 + i; u < 32; u += T) dst[u] = src[u];
}

// ---------------------------------------------------------------- k_encode
template <int T>
__global__ void __launch_bounds__(max_threads<T>())
k_encode(Layout lo, EncWs w, const uint8_t *__restrict__ tables, const uint16_t *__restrict__ kv,
         uint8_t *ws) {
  extern __shared__ __align__(16) uint32_t etab[];  // [256][4][T] : cdf | f << 16, then the word rings
  const int lv = blockIdx.x, si = blockIdx.y;
  const int h = si % lo.H, kvi = (si / lo.H) % 2, l = si / (2 * lo.H);
  const int32_t *counts = reinterpret_cast<const int32_t *>(ws + w.levels);
  const int32_t *lists = counts + kMaxLevels;
  const int cnt = counts[lv];
  if (cnt == 0) return;
  uint32_t *status = reinterpret_cast<uint32_t *>(ws + w.status);

  const uint16_t *cdf = reinterpret_cast<const uint16_t *>(tables + lo.tb_cdf) +
                        tab_index(lo, lv, l, kvi, h * lo.d) * 256;
  for (int e = threadIdx.x; e < lo.d * 256; e += blockDim.x) {
    const int c = e >> 8, s = e & 255;
    const uint32_t c0 = cdf[c * 256 + s];
    const uint32_t c1 = s < 255 ? cdf[c * 256 + s + 1] : kM;
    etab[(s * kLpt + (c % kLpt)) * T + c / kLpt] = c0 | ((c1 - c0) << 16);
  }
  __syncthreads();

  const int team = threadIdx.x / T, i = threadIdx.x % T, nteams = blockDim.x / T;
  uint16_t *ring = reinterpret_cast<uint16_t *>(etab + 256 * lo.d) + team * kWordRing;
  const uint32_t tm = team_mask<T>();
  const float4 rc4 = *reinterpret_cast<const float4 *>(
      reinterpret_cast<const float *>(tables + lo.tb_recip) + tab_index(lo, lv, l, kvi, h * lo.d + kLpt * i));
  const float rc[4] = {rc4.x, rc4.y, rc4.z, rc4.w};
  const int R = lo.R;

  for (int idx = team; idx < cnt; idx += nteams) {
    const int k = lists[lv * lo.n_chunks + idx];
    const int ng = chunk_ng(lo, k), ntok = chunk_ntok(lo, k);
    const int64_t t0 = int64_t(k) * lo.C;
    const uint8_t *chunk = ws + w.chunks + uint64_t(k) * lo.fixed_full;
    const float4 s4 = *reinterpret_cast<const float4 *>(chunk + lo.sec_s + (uint64_t(si) * lo.d + kLpt * i) * 4);
    const float sc[4] = {s4.x, s4.y, s4.z, s4.w};
    const uint8_t *anc = chunk + lo.sec_anc + uint64_t(si) * ng * lo.d + kLpt * i;
    const uint16_t *xin = kv + (uint64_t(si) * lo.S + t0) * lo.d + kLpt * i;
    const uint64_t sidx = uint64_t(k) * lo.nstr + si;
    uint16_t *wout = reinterpret_cast<uint16_t *>(ws + w.words) + sidx * w.words_cap;
    const int64_t cap = int64_t(w.words_cap);

    uint32_t x[4] = {kRansL, kRansL, kRansL, kRansL};
    int64_t E = 0;      // words emitted so far (encoder order)
    uint32_t nesc = 0;
    uint32_t badm = 0;  // bit 15 of a half set: an all-ones exponent was seen
    bool overflow = false;
    // tokens in reverse order, kAhead rows per batch, the next batch loaded
    // while this one is encoded; anchor rows are loaded and skipped
    constexpr int kAhead = 2;
    int t = ntok - 1;
    int g = t / lo.G, r = t - g * lo.G;  // group of t and t's place in it
    uint32_t a4 = *reinterpret_cast<const uint32_t *>(anc + uint64_t(g) * lo.d);
    uint32_t a4n = g > 0 ? *reinterpret_cast<const uint32_t *>(anc + uint64_t(g - 1) * lo.d) : 0u;
    float ah[4];
#pragma unroll
    for (int j = 0; j < 4; j++) ah[j] = __fmul_rn(float(int8_t(a4 >> (8 * j))), sc[j]);
    uint2 cur[kAhead], nxt[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; u++)
      cur[u] = t - u >= 0 ? __ldg(reinterpret_cast<const uint2 *>(xin + int64_t(t - u) * lo.d)) : make_uint2(0, 0);
    while (t >= 1 && !overflow) {
#pragma unroll
      for (int u = 0; u < kAhead; u++) {
        const int tn = t - kAhead - u;
        nxt[u] = tn >= 0 ? __ldg(reinterpret_cast<const uint2 *>(xin + int64_t(tn) * lo.d)) : make_uint2(0, 0);
      }
#pragma unroll
      for (int u = 0; u < kAhead; u++) {
        if (t < 1 || overflow) break;
        if (r == 0) {  // the anchor token of group g: on to group g - 1
          g--;
          r = lo.G - 1;
          a4 = a4n;
          if (g > 0) a4n = *reinterpret_cast<const uint32_t *>(anc + uint64_t(g - 1) * lo.d);
#pragma unroll
          for (int j = 0; j < 4; j++) ah[j] = __fmul_rn(float(int8_t(a4 >> (8 * j))), sc[j]);
          t--;
          continue;
        }
        const uint2 raw = cur[u];
        badm |= ((raw.x & 0x7C007C00u) + 0x04000400u) | ((raw.y & 0x7C007C00u) + 0x04000400u);
        const uint32_t hw[4] = {raw.x & 0xFFFFu, raw.x >> 16, raw.y & 0xFFFFu, raw.y >> 16};
        uint32_t word[4], qv[4];
        bool esc[4], ren[4];
        int cntw = 0;
#pragma unroll
        for (int j = 3; j >= 0; j--) {
          const float xv = __half2float(__ushort_as_half(uint16_t(hw[j])));
          const int q = __float2int_rn(__fmul_rn(__fsub_rn(xv, ah[j]), rc[j]));
          esc[j] = uint32_t(q) + uint32_t(R) > uint32_t(2 * R);  // |q| > R, in unsigned arithmetic
          const int sym = esc[j] ? kEsc : q + 127;
          const uint32_t e = etab[(sym * kLpt + j) * T + i];
          const uint32_t f = e >> 16, c = e & 0xFFFFu;
          ren[j] = x[j] >= (f << 16);
          word[j] = x[j] & 0xFFFFu;
          const uint32_t xr = ren[j] ? (x[j] >> 16) : x[j];
          x[j] = rans_put(xr, f, c);
          qv[j] = uint32_t(q);
          cntw += (esc[j] ? 2 : 0) + (ren[j] ? 1 : 0);
        }
        // emission order: lanes descending, i.e. threads descending
        int suf = cntw;
#pragma unroll
        for (int o = 1; o < T; o <<= 1) {
          const int v = __shfl_down_sync(tm, suf, o, T);
          if (i + o < T) suf += v;
        }
        const int tot = __shfl_sync(tm, suf, 0, T);
        if (E + tot > cap) {
          overflow = true;
          break;
        }
        // word e of the stream (encoder order) goes to ring slot ~e mod the
        // ring size, so a block of 256 words sits in the ring in the order it
        // takes at the end of the scratch slot (which is filled backwards)
        uint32_t e = uint32_t(E) + uint32_t(suf - cntw);
        if (esc[0] | esc[1] | esc[2] | esc[3]) {  // escapes (rare): the raw q follows the word
#pragma unroll
          for (int j = 3; j >= 0; j--) {
            if (esc[j]) {
              ring[~e & (kWordRing - 1)] = uint16_t(qv[j] >> 16);
              ring[~(e + 1) & (kWordRing - 1)] = uint16_t(qv[j] & 0xFFFFu);
              e += 2;
              nesc++;
            }
            if (ren[j]) {
              ring[~e & (kWordRing - 1)] = uint16_t(word[j]);
              e += 1;
            }
          }
        } else {
#pragma unroll
          for (int j = 3; j >= 0; j--) {
            if (ren[j]) {
              ring[~e & (kWordRing - 1)] = uint16_t(word[j]);
              e += 1;
            }
          }
        }
        const uint32_t e0 = uint32_t(E), e1 = e0 + uint32_t(tot);
        if ((e1 >> 8) != (e0 >> 8)) {  // blocks completed: 16-byte stores into the slot
          __syncwarp(tm);
          for (uint32_t blk = e0 >> 8; blk < (e1 >> 8); blk++) flush_block(ring, wout, cap, blk, 0, i, T);
          __syncwarp(tm);  // the block's reads are done before its slots take new words
        }
        E += tot;
        t--;
        r--;
      }
#pragma unroll
      for (int u = 0; u < kAhead; u++) cur[u] = nxt[u];
    }
    const bool bad = (badm & 0x80008000u) != 0;
    if (!overflow && (E & 255)) {  // the last, partial block: only units that hold its words
      __syncwarp(tm);
      const uint32_t blk = uint32_t(E) >> 8;
      flush_block(ring, wout, cap, blk, (256 * (blk + 1) - uint32_t(E)) / 8, i, T);
    }
    if (bad) atomicOr(status, kStNonfinite);
    if (overflow) {
      if (i == 0) atomicOr(status, kStCapacity);
      continue;
    }
#pragma unroll
    for (int o = T / 2; o; o >>= 1) nesc += __shfl_xor_sync(tm, nesc, o, T);
    if (i == 0)
      reinterpret_cast<uint2 *>(ws + w.info)[sidx] = make_uint2(uint32_t(E), nesc);
    reinterpret_cast<uint4 *>(ws + w.states)[(sidx * lo.d) / 4 + i] = make_uint4(x[0], x[1], x[2], x[3]);
  }
}

// ---------------------------------------------------------------- d = 128
// k_encode for d = 128 (the models' head dim) with the token loop cut down
// to what a symbol needs: tokens run in reverse over the groups (the anchor
// rows are not coded), the next row loaded while the current one is coded;
// each lane quantises, looks up (cdf, f) and takes one rANS step without a
// branch; one warp vote per token sends a token with an escape to the
// general path; the suffix shuffle scan uses the shuffle's own range
// predicate; a thread's words go to their ring slots from one prefix.
constexpr int kEncTeams128 = 24;

// Inclusive suffix scan step over the warp: v += (value of lane i + O, when
// there is one).
template <int O>
__device__ __forceinline__ uint32_t suffix_step(uint32_t v) {
  asm("{\n\t.reg .pred p;\n\t.reg .u32 t;\n\t"
      "shfl.sync.down.b32 t|p, %0, %1, 31, -1;\n\t"
      "@p add.u32 %0, %0, t;\n\t}"
      : "+r"(v) : "n"(O));
  return v;
}

// Grid rows from split0 on come in pairs: the two CTAs of a pair code the
// even and the odd entries of the same head's chunk list.
__global__ void __launch_bounds__(kEncTeams128 * 32, 1)
k_enc128(Layout lo, EncWs w, const uint8_t *__restrict__ tables, const uint16_t *__restrict__ kv, uint8_t *ws,
         int split0) {
  constexpr int T = 32;
  extern __shared__ __align__(16) uint32_t etab[];  // [256][4][32] : cdf | f << 16, then the word rings
  const int lv = blockIdx.x;
  int si = blockIdx.y, part = 0, nparts = 1;
  if (si >= split0) {
    si = split0 + (int(blockIdx.y) - split0) / 2;
    part = (int(blockIdx.y) - split0) & 1;
    nparts = 2;
  }
  const int h = si % lo.H, kvi = (si / lo.H) % 2, l = si / (2 * lo.H);
  const int32_t *counts = reinterpret_cast<const int32_t *>(ws + w.levels);
  const int32_t *lists = counts + kMaxLevels;
  const int cnt = counts[lv];
  if (cnt <= part) return;
  uint32_t *status = reinterpret_cast<uint32_t *>(ws + w.status);

  const uint16_t *cdf = reinterpret_cast<const uint16_t *>(tables + lo.tb_cdf) +
                        tab_index(lo, lv, l, kvi, h * lo.d) * 256;
  for (int e = threadIdx.x; e < 128 * 256; e += blockDim.x) {
    const int c = e >> 8, s = e & 255;
    const uint32_t c0 = cdf[c * 256 + s];
    const uint32_t c1 = s < 255 ? cdf[c * 256 + s + 1] : kM;
    etab[(s * kLpt + (c % kLpt)) * T + c / kLpt] = c0 | ((c1 - c0) << 16);
  }
  __syncthreads();

  const int team = threadIdx.x >> 5, nteams = blockDim.x >> 5;
  const uint32_t i = threadIdx.x & 31;
  uint16_t *ring = reinterpret_cast<uint16_t *>(etab + 256 * 128) + team * kWordRing;
  const uint32_t *et = etab + i;  // thread i's entries: et[(sym * 4 + j) * 32]
  const float4 rc4 = *reinterpret_cast<const float4 *>(
      reinterpret_cast<const float *>(tables + lo.tb_recip) + tab_index(lo, lv, l, kvi, h * lo.d + kLpt * i));
  const float rc[4] = {rc4.x, rc4.y, rc4.z, rc4.w};
  const int R = lo.R;

  for (int idx = part + nparts * team; idx < cnt; idx += nparts * nteams) {
    const int k = lists[lv * lo.n_chunks + idx];
    const int ng = chunk_ng(lo, k), ntok = chunk_ntok(lo, k);
    const int64_t t0 = int64_t(k) * lo.C;
    const uint8_t *chunk = ws + w.chunks + uint64_t(k) * lo.fixed_full;
    const float4 s4 = *reinterpret_cast<const float4 *>(chunk + lo.sec_s + (uint64_t(si) * lo.d + kLpt * i) * 4);
    const float sc[4] = {s4.x, s4.y, s4.z, s4.w};
    const uint8_t *anc = chunk + lo.sec_anc + uint64_t(si) * ng * lo.d + kLpt * i;
    const uint16_t *xin = kv + (uint64_t(si) * lo.S + t0) * lo.d + kLpt * i;
    const uint64_t sidx = uint64_t(k) * lo.nstr + si;
    uint16_t *wout = reinterpret_cast<uint16_t *>(ws + w.words) + sidx * w.words_cap;
    const int64_t cap = int64_t(w.words_cap);

    uint32_t x[4] = {kRansL, kRansL, kRansL, kRansL};
    int64_t E = 0;  // words emitted so far (encoder order)
    uint32_t nesc = 0, badm = 0;
    bool overflow = false;
    // the first token coded: the chunk's last delta token (none when every
    // token is an anchor)
    int g = ng - 1;
    int tt = min(lo.G, ntok - g * lo.G) - 1;  // its place in group g
    if (tt < 1 && g > 0) {
      g--;
      tt = lo.G - 1;
    }
    uint2 cur = tt >= 1 ? __ldg(reinterpret_cast<const uint2 *>(xin + int64_t(g * lo.G + tt) * lo.d))
                        : make_uint2(0, 0);
    for (; g >= 0 && tt >= 1 && !overflow; g--, tt = lo.G - 1) {
      const uint32_t a4 = *reinterpret_cast<const uint32_t *>(anc + uint64_t(g) * lo.d);
      float ah[4];
#pragma unroll
      for (int j = 0; j < 4; j++) ah[j] = __fmul_rn(float(int8_t(a4 >> (8 * j))), sc[j]);
      for (; tt >= 1; tt--) {
        // the next token coded: t - 1, or across this group's anchor t - 2
        const int t = g * lo.G + tt;
        const int tn = tt > 1 ? t - 1 : t - 2;
        const uint2 raw = cur;
        if (tn >= 1) cur = __ldg(reinterpret_cast<const uint2 *>(xin + int64_t(tn) * lo.d));
        badm |= ((raw.x & 0x7C007C00u) + 0x04000400u) | ((raw.y & 0x7C007C00u) + 0x04000400u);
        const uint32_t hw[4] = {raw.x & 0xFFFFu, raw.x >> 16, raw.y & 0xFFFFu, raw.y >> 16};
        uint32_t word[4], qv[4];
        bool esc[4], ren[4];
        uint32_t cntw = 0;
#pragma unroll
        for (int j = 3; j >= 0; j--) {
          const float xv = __half2float(__ushort_as_half(uint16_t(hw[j])));
          const int q = __float2int_rn(__fmul_rn(__fsub_rn(xv, ah[j]), rc[j]));
          esc[j] = uint32_t(q) + uint32_t(R) > uint32_t(2 * R);  // |q| > R, in unsigned arithmetic
          const int sym = esc[j] ? kEsc : q + 127;
          const uint32_t e = et[(sym * kLpt + j) * T];
          const uint32_t f = e >> 16, c = e & 0xFFFFu;
          ren[j] = x[j] >= (f << 16);
          word[j] = x[j] & 0xFFFFu;
          x[j] = rans_put(ren[j] ? (x[j] >> 16) : x[j], f, c);
          qv[j] = uint32_t(q);
          cntw += ren[j] ? 1u : 0u;
        }
        const bool esc_warp = __any_sync(0xffffffffu, esc[0] | esc[1] | esc[2] | esc[3]);
        if (esc_warp) cntw += 2 * ((esc[0] ? 1u : 0u) + (esc[1] ? 1u : 0u) + (esc[2] ? 1u : 0u) + (esc[3] ? 1u : 0u));
        // emission order: lanes descending, i.e. threads descending
        uint32_t suf = suffix_step<1>(cntw);
        suf = suffix_step<2>(suf);
        suf = suffix_step<4>(suf);
        suf = suffix_step<8>(suf);
        suf = suffix_step<16>(suf);
        const uint32_t tot = __shfl_sync(0xffffffffu, suf, 0);
        if (E + tot > cap) {
          overflow = true;
          break;
        }
        // word e of the stream (encoder order) goes to ring slot ~e mod the
        // ring size, so a block of 256 words sits in the ring in the order it
        // takes at the end of the scratch slot (which is filled backwards)
        const uint32_t e0 = uint32_t(E), e = e0 + suf - cntw;
        if (!esc_warp) {
          const uint32_t p2 = e + (ren[3] ? 1u : 0u), p1 = p2 + (ren[2] ? 1u : 0u), p0 = p1 + (ren[1] ? 1u : 0u);
          if (ren[3]) ring[~e & (kWordRing - 1)] = uint16_t(word[3]);
          if (ren[2]) ring[~p2 & (kWordRing - 1)] = uint16_t(word[2]);
          if (ren[1]) ring[~p1 & (kWordRing - 1)] = uint16_t(word[1]);
          if (ren[0]) ring[~p0 & (kWordRing - 1)] = uint16_t(word[0]);
        } else {  // escapes: the raw q follows the word (decode order: word, low half, high half)
          uint32_t ee = e;
#pragma unroll
          for (int j = 3; j >= 0; j--) {
            if (esc[j]) {
              ring[~ee & (kWordRing - 1)] = uint16_t(qv[j] >> 16);
              ring[~(ee + 1) & (kWordRing - 1)] = uint16_t(qv[j] & 0xFFFFu);
              ee += 2;
              nesc++;
            }
            if (ren[j]) {
              ring[~ee & (kWordRing - 1)] = uint16_t(word[j]);
              ee += 1;
            }
          }
        }
        const uint32_t e1 = e0 + tot;
        if ((e1 >> 8) != (e0 >> 8)) {  // blocks completed: 16-byte stores into the slot
          __syncwarp();
          for (uint32_t blk = e0 >> 8; blk < (e1 >> 8); blk++) flush_block(ring, wout, cap, blk, 0, int(i), T);
          __syncwarp();  // the block's reads are done before its slots take new words
        }
        E += tot;
      }
    }
    const bool bad = (badm & 0x80008000u) != 0;
    if (!overflow && (E & 255)) {  // the last, partial block: only units that hold its words
      __syncwarp();
      const uint32_t blk = uint32_t(E) >> 8;
      flush_block(ring, wout, cap, blk, (256 * (blk + 1) - uint32_t(E)) / 8, int(i), T);
    }
    if (bad) atomicOr(status, kStNonfinite);
    if (overflow) {
      if (i == 0) atomicOr(status, kStCapacity);
      continue;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) nesc += __shfl_xor_sync(0xffffffffu, nesc, o);
    if (i == 0) reinterpret_cast<uint2 *>(ws + w.info)[sidx] = make_uint2(uint32_t(E), nesc);
    reinterpret_cast<uint4 *>(ws + w.states)[(sidx * lo.d) / 4 + i] = make_uint4(x[0], x[1], x[2], x[3]);
  }
}

// The last wave, as for the decoder: when the CTAs past the last full wave
// of the GPU, doubled, still run side by side, their heads take two CTAs each.
cudaError_t launch_encode_128(const Layout &lo, const EncWs &w, const uint8_t *tables, const uint16_t *kv,
                              uint8_t *ws, int teams, int live_levels, cudaStream_t st) {
  if (teams > kEncTeams128) teams = kEncTeams128;
  const size_t smem = size_t(256) * 128 * 4 + size_t(teams) * kWordRing * 2;
  cudaError_t e = cudaFuncSetAttribute(k_enc128, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_enc128, teams * 32, smem);
  if (e != cudaSuccess) return e;
  const int wave = sms * per_sm, live = lo.nstr * live_levels, rest = wave > 0 ? live % wave : 0;
  int split = 0;
  if (rest > 0 && teams >= 2) {
    const int r = min((rest + live_levels - 1) / live_levels, lo.nstr);
    if (2 * r * live_levels <= wave) split = r;
  }
  dim3 grid(lo.n_levels, lo.nstr + split);
  k_enc128<<<grid, teams * 32, smem, st>>>(lo, w, tables, kv, ws, lo.nstr - split);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- scans
constexpr int kScanThreads = 1024;

__device__ uint64_t block_excl_scan(uint64_t v, uint64_t *total, uint64_t *sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint64_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint64_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sm[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint64_t s = lane < nw ? sm[lane] : 0;
    uint64_t si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint64_t t = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += t;
    }
    sm[32 + lane] = si - s;
    if (lane == 31) sm[64] = si;
  }
  __syncthreads();
  const uint64_t r = sm[32 + warp] + incl - v;
  *total = sm[64];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kScanThreads)
k_scan_chunks(Layout lo, EncWs w, uint8_t *ws) {
  __shared__ uint64_t sm[72];
  const int k = blockIdx.x;
  const uint2 *info = reinterpret_cast<const uint2 *>(ws + w.info) + uint64_t(k) * lo.nstr;
  uint32_t *soff = reinterpret_cast<uint32_t *>(ws + w.soff) + uint64_t(k) * lo.nstr;
  uint64_t rel = chunk_fixed(lo, k);
  for (int base = 0; base < lo.nstr; base += kScanThreads) {
    const int s = base + threadIdx.x;
    const uint64_t sz = s < lo.nstr ? pad16(16 + 4 * uint64_t(lo.d) + 2 * uint64_t(info[s].x)) : 0;
    uint64_t tot;
    const uint64_t ex = block_excl_scan(sz, &tot, sm);
    if (s < lo.nstr) soff[s] = uint32_t(rel + ex);
    rel += tot;
  }
  if (threadIdx.x == 0) reinterpret_cast<uint64_t *>(ws + w.coff)[k] = rel;  // chunk size for now
}

__global__ void __launch_bounds__(kScanThreads)
k_scan_total(Layout lo, EncWs w, uint8_t *ws, uint64_t cap, uint64_t *out_bytes) {
  __shared__ uint64_t sm[72];
  uint64_t *coff = reinterpret_cast<uint64_t *>(ws + w.coff);
  uint64_t pos = lo.hdr_bytes;
  for (int base = 0; base < lo.n_chunks; base += kScanThreads) {
    const int k = base + threadIdx.x;
    const uint64_t sz = k < lo.n_chunks ? coff[k] : 0;
    uint64_t tot;
    const uint64_t ex = block_excl_scan(sz, &tot, sm);
    if (k < lo.n_chunks) coff[k] = pos + ex;
    pos += tot;
  }
  if (threadIdx.x == 0) {
    coff[lo.n_chunks] = pos;
    *out_bytes = pos;
    if (pos > cap) atomicOr(reinterpret_cast<uint32_t *>(ws + w.status), kStCapacity);
  }
}

// ---------------------------------------------------------------- compaction
// Fixed parts of all chunks, 16 bytes per thread per step: the chunk
// header, the scales and anchors from the scratch (which has the container's
// layout), the stream index, and zero padding.  Block 0 also writes the
// container header and the chunk index.
__global__ void __launch_bounds__(256)
k_compact_fixed(Layout lo, EncWs w, const uint8_t *__restrict__ ws, uint8_t *__restrict__ out) {
  if (*reinterpret_cast<const uint32_t *>(ws + w.status) & (kStCapacity | kStNonfinite)) return;
  const uint64_t *coff = reinterpret_cast<const uint64_t *>(ws + w.coff);
  const uint8_t *lv8 = ws + w.levels + 4 * kMaxLevels * (1 + uint64_t(lo.n_chunks));
  if (blockIdx.x == 0) {
    for (uint64_t b = 64 + threadIdx.x * 8; b < lo.hdr_bytes; b += blockDim.x * 8) {
      const uint64_t kk = (b - 64) / 8;
      *reinterpret_cast<uint64_t *>(out + b) = kk < uint64_t(lo.n_chunks) ? coff[kk] : 0;
    }
    if (threadIdx.x == 0) {
      uint32_t *hd = reinterpret_cast<uint32_t *>(out);
      hd[0] = 0x564B4743u;  // "CGKV"
      hd[1] = 1;
      hd[2] = lo.L;
      hd[3] = lo.H;
      hd[4] = lo.d;
      hd[5] = lo.C;
      hd[6] = lo.G;
      hd[7] = lo.R;
      *reinterpret_cast<uint64_t *>(out + 32) = uint64_t(lo.S);
      hd[10] = lo.n_levels;
      hd[11] = lo.n_chunks;
      *reinterpret_cast<uint64_t *>(out + 48) = coff[lo.n_chunks];
      hd[14] = 0;
      hd[15] = 0;
    }
  }
  const uint64_t upc = lo.fixed_full / 16;  // 16-byte units per chunk slot
  const uint64_t total = upc * uint64_t(lo.n_chunks);
  const uint32_t *soff_all = reinterpret_cast<const uint32_t *>(ws + w.soff);
  for (uint64_t u = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += uint64_t(gridDim.x) * blockDim.x) {
    const int k = int(u / upc);
    const uint64_t off = (u - uint64_t(k) * upc) * 16;
    if (off >= chunk_fixed(lo, k)) continue;
    const uint64_t ng = chunk_ng(lo, k);
    const uint64_t a_end = lo.sec_anc + uint64_t(lo.nstr) * ng * lo.d;
    const uint64_t o_beg = chunk_sec_off(lo, k);
    uint32_t v[4];
    if (off == 0) {
      v[0] = lv8[k];
      v[1] = uint32_t(int64_t(k) * lo.C);
      v[2] = uint32_t(chunk_ntok(lo, k));
      v[3] = uint32_t(ng);
    } else if (off < o_beg) {  // scales, anchors (the scale section has no padding)
      const uint4 q = *reinterpret_cast<const uint4 *>(ws + w.chunks + uint64_t(k) * lo.fixed_full + off);
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
#pragma unroll
      for (int c = 0; c < 4; c++)
        if (off >= lo.sec_anc && off + 4 * c >= a_end) v[c] = 0;
    } else {  // stream index
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const uint64_t wi = (off - o_beg) / 4 + c;
        v[c] = wi < uint64_t(lo.nstr) ? soff_all[uint64_t(k) * lo.nstr + wi] : 0u;
      }
    }
    *reinterpret_cast<uint4 *>(out + coff[k] + off) = make_uint4(v[0], v[1], v[2], v[3]);
  }
}

// Stream blocks: header, states, then the words copied 16 bytes at a time.
// The scratch words of a stream end on a 16-byte boundary but start anywhere
// (2-byte steps), so each 16-byte output is assembled from two aligned
// 16-byte loads with a funnel shift; bytes past the last word are zero.
template <int OFS, int SH>
__device__ __forceinline__ uint4 shifted16(const uint4 &a, const uint4 &b) {
  const uint32_t q[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t r[4];
#pragma unroll
  for (int k = 0; k < 4; k++) r[k] = SH ? __funnelshift_r(q[k + OFS], q[k + OFS + 1], SH) : q[k + OFS];
  return make_uint4(r[0], r[1], r[2], r[3]);
}

template <int OFS, int SH>
__device__ void copy_words(uint8_t *dst, const uint8_t *src_aligned, uint64_t nbytes, uint64_t nout) {
  for (uint64_t o = threadIdx.x * 16ull; o < nout; o += blockDim.x * 16ull) {
    const uint4 a = *reinterpret_cast<const uint4 *>(src_aligned + o);
    const uint4 b = *reinterpret_cast<const uint4 *>(src_aligned + o + 16);
    uint4 v = shifted16<OFS, SH>(a, b);
    if (o + 16 > nbytes) {  // last piece: zero the padding
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const uint64_t bo = o + 4 * k;
        if (bo >= nbytes) w[k] = 0;
        else if (bo + 4 > nbytes) w[k] &= 0xFFFFu;  // one 2-byte word left in this 4-byte slot
      }
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint4 *>(dst + o) = v;
  }
}

__global__ void __launch_bounds__(128)
k_compact_stream(Layout lo, EncWs w, const uint8_t *__restrict__ ws, uint8_t *__restrict__ out) {
  if (*reinterpret_cast<const uint32_t *>(ws + w.status) & (kStCapacity | kStNonfinite)) return;
  const uint64_t ns = uint64_t(lo.n_chunks) * lo.nstr;
  for (uint64_t sidx = blockIdx.x; sidx < ns; sidx += gridDim.x) {
    const int k = int(sidx / lo.nstr);
    const uint64_t base = reinterpret_cast<const uint64_t *>(ws + w.coff)[k] +
                          reinterpret_cast<const uint32_t *>(ws + w.soff)[sidx];
    const uint2 inf = reinterpret_cast<const uint2 *>(ws + w.info)[sidx];
    uint8_t *blk = out + base;
    if (threadIdx.x == 0)
      *reinterpret_cast<uint4 *>(blk) = make_uint4(inf.x, inf.y, uint32_t(chunk_nd(lo, k)), 0u);
    const uint4 *st = reinterpret_cast<const uint4 *>(ws + w.states + 4 * sidx * lo.d);
    uint4 *sd = reinterpret_cast<uint4 *>(blk + 16);
    for (int j = threadIdx.x; j < lo.d / 4; j += blockDim.x) sd[j] = st[j];
    // words: scratch bytes [so, so + 2 n_words) of this stream's slot
    const uint8_t *slot = ws + w.words + 2 * sidx * w.words_cap;
    const uint64_t so = 2 * (w.words_cap - inf.x);
    const uint64_t nbytes = 2 * uint64_t(inf.x);
    const uint64_t nout = pad16(16 + 4 * uint64_t(lo.d) + nbytes) - 16 - 4 * uint64_t(lo.d);
    const uint8_t *src = slot + (so & ~uint64_t(15));
    uint8_t *dst = blk + 16 + 4 * lo.d;
    switch (so & 15) {  // the same for the whole stream: no divergence
      case 0: copy_words<0, 0>(dst, src, nbytes, nout); break;
      case 2: copy_words<0, 16>(dst, src, nbytes, nout); break;
      case 4: copy_words<1, 0>(dst, src, nbytes, nout); break;
      case 6: copy_words<1, 16>(dst, src, nbytes, nout); break;
      case 8: copy_words<2, 0>(dst, src, nbytes, nout); break;
      case 10: copy_words<2, 16>(dst, src, nbytes, nout); break;
      case 12: copy_words<3, 0>(dst, src, nbytes, nout); break;
      default: copy_words<3, 16>(dst, src, nbytes, nout); break;
    }
  }
}

template <int T>
cudaError_t launch_encode_t(const Layout &lo, const EncWs &w, const uint8_t *tables,
                            const uint16_t *kv, uint8_t *ws, int teams, cudaStream_t st) {
  if (teams > max_threads<T>() / T) teams = max_threads<T>() / T;
  const size_t smem = size_t(256) * lo.d * 4 + size_t(teams) * kWordRing * 2;
  cudaError_t e = cudaFuncSetAttribute(k_encode<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(lo.n_levels, lo.nstr);
  k_encode<T><<<grid, teams * T, smem, st>>>(lo, w, tables, kv, ws);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_encode(const Layout &lo, const EncWs &w, const uint8_t *tables,
                          const uint16_t *kv, uint8_t *ws, int teams, int live_levels, cudaStream_t st) {
  if (teams < 1) return cudaSuccess;
  switch (lo.d / kLpt) {
    case 2: return launch_encode_t<2>(lo, w, tables, kv, ws, teams, st);
    case 4: return launch_encode_t<4>(lo, w, tables, kv, ws, teams, st);
    case 8: return launch_encode_t<8>(lo, w, tables, kv, ws, teams, st);
    case 16: return launch_encode_t<16>(lo, w, tables, kv, ws, teams, st);
    case 32: return launch_encode_128(lo, w, tables, kv, ws, teams, live_levels, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_scan_compact(const Layout &lo, const EncWs &w, uint8_t *ws, uint8_t *out,
                                uint64_t cap, uint64_t *out_bytes, cudaStream_t st) {
  k_scan_chunks<<<lo.n_chunks, kScanThreads, 0, st>>>(lo, w, ws);
  k_scan_total<<<1, kScanThreads, 0, st>>>(lo, w, ws, cap, out_bytes);
  {
    const uint64_t units = (lo.fixed_full / 16) * uint64_t(lo.n_chunks);
    const uint64_t blocks = (units + 255) / 256;
    k_compact_fixed<<<unsigned(blocks < 4096 ? (blocks ? blocks : 1) : 4096), 256, 0, st>>>(lo, w, ws, out);
  }
  const uint64_t ns = uint64_t(lo.n_chunks) * lo.nstr;
  const unsigned grid = unsigned(ns < 65536 ? ns : 65536);
  k_compact_stream<<<grid, 128, 0, st>>>(lo, w, ws, out);
  return cudaGetLastError();
}

}  // namespace cg
