// cg_decode.cu -- the streaming decoder.
//
// CacheGen's receiver decodes the bitstream "in real time, synchronized
// with transmission" (gptget summary of arXiv 2310.07240, Methodology; Guide
// to CacheGen, pillar 4) and rebuilds each token as anchor + delta (Guide,
// Step 2 decode_sequence; Step 1 dequantize).  The kernels:
//
//   k_decode_index  one thread checks the container header against the
//                   caller's dims and the tables header, validates the
//                   chunk index and headers of [k0, k1) and lists the chunks
//                   of each level.
//   k_decode        (d < 128) one CTA per (level, head) holds that head's d
//                   frequency tables in shared memory, laid out so that
//                   thread i of a team only ever touches bank i (no bank
//                   conflicts however the symbols fall); each team of d/4
//                   threads decodes one chunk's stream, 4 rANS lanes per
//                   thread.  Per token: a bucket lookup (slot >> 7) plus one
//                   carry finds the symbol, a shuffle scan over the team
//                   orders the word reads, the fused dequantisation
//                   fma(q, step, a_hat) is clamped, converted to fp16 and
//                   stored 8 bytes per thread (a team writes one token row).
//   k_dec128        (d = 128) the same with a warp per chunk stream and
//                   tables laid out for a short token loop; for ranges with
//                   a few chunks per level (MID) with u8 pair tables, so
//                   that two CTAs share an SM.
//   k_thin128       (d = 128, chunk ranges that give each (level, head) only
//                   a few chunks) four warps per stream, one lane per
//                   thread, for a short dependency chain per token.
//
// Every read of the container is bounded by the stream's own header, which
// is itself checked against the stream index; a stream whose lanes do not
// return to the initial state 2^16, or whose word/escape counts disagree,
// sets the CORRUPT bit.  Nothing waits on another CTA.
#include <cuda_fp16.h>

#include <type_traits>

#include "cg_kernels.cuh"

namespace cg {
namespace {

constexpr int kLpt = kLanesPerThread;

__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint64_t ld_u64(const uint8_t *p) { return *reinterpret_cast<const uint64_t *>(p); }

// Two fp32 values to packed fp16 (lo in the low half), round to nearest
// even, saturating to +-65504 instead of overflowing to infinity: the same
// result as clamping to the finite fp16 range and then rounding.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 16-byte asynchronous global->shared copy that reads only src_bytes (0..16)
// and zero-fills the rest, so a copy never reads past the stream's words.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc, uint32_t src_bytes) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gsrc), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Words staged per team: a ring of kRing words in two halves, followed by
// a copy of its first kMirror words, so that a thread's (up to four) words
// can be read from one base index without wrapping.
constexpr uint32_t kRing = 512, kHalf = 256, kMirror = 16;
// Symbol-search buckets: slot >> kBucketShift, kBuckets of them.
constexpr uint32_t kBucketShift = 7, kBuckets = 1u << (16 - kBucketShift), kBucketSlots = 1u << kBucketShift;
constexpr uint32_t kCdfRows = 258;  // cdf_0 .. cdf_255, cdf_255 again, padding

// ---------------------------------------------------------------- index
__global__ void k_decode_index(Layout lo, const uint8_t *__restrict__ tables,
                               const uint8_t *__restrict__ buf, uint64_t bytes, int32_t k0,
                               int32_t k1, uint8_t *ws) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  uint32_t *status = reinterpret_cast<uint32_t *>(ws);
  int32_t *count = reinterpret_cast<int32_t *>(ws + 64);
  int32_t *list = reinterpret_cast<int32_t *>(ws + 256);
  for (int i = 0; i < kMaxLevels; i++) count[i] = 0;
  bool ok = bytes >= lo.hdr_bytes && ld_u32(buf) == 0x564B4743u && ld_u32(buf + 4) == 1 &&
            ld_u32(buf + 8) == uint32_t(lo.L) && ld_u32(buf + 12) == uint32_t(lo.H) &&
            ld_u32(buf + 16) == uint32_t(lo.d) && ld_u32(buf + 20) == uint32_t(lo.C) &&
            ld_u32(buf + 24) == uint32_t(lo.G) && ld_u32(buf + 28) == uint32_t(lo.R) &&
            ld_u64(buf + 32) == uint64_t(lo.S) && ld_u32(buf + 40) == uint32_t(lo.n_levels) &&
            ld_u32(buf + 44) == uint32_t(lo.n_chunks) && ld_u64(buf + 48) == bytes;
  ok = ok && ld_u32(tables) == 0x42544743u && ld_u32(tables + 4) == 1 &&
       ld_u32(tables + 8) == uint32_t(lo.L) && ld_u32(tables + 12) == uint32_t(lo.H) &&
       ld_u32(tables + 16) == uint32_t(lo.d) && ld_u32(tables + 20) == uint32_t(lo.n_levels);
  for (int k = k0; ok && k < k1; k++) {
    const uint64_t base = ld_u64(buf + 64 + 8 * uint64_t(k));
    const uint64_t end = (k + 1 < lo.n_chunks) ? ld_u64(buf + 64 + 8 * uint64_t(k + 1)) : bytes;
    if ((base & 15) || base < lo.hdr_bytes || end > bytes || end < base ||
        end - base < chunk_fixed(lo, k)) {
      ok = false;
      break;
    }
    const uint8_t *ch = buf + base;
    const uint32_t w0 = ld_u32(ch);
    const uint32_t lv = w0 & 0xFFFFu;
    if ((w0 >> 16) != 0 || lv >= uint32_t(lo.n_levels) || ld_u32(ch + 4) != uint32_t(int64_t(k) * lo.C) ||
        ld_u32(ch + 8) != uint32_t(chunk_ntok(lo, k)) || ld_u32(ch + 12) != uint32_t(chunk_ng(lo, k))) {
      ok = false;
      break;
    }
    list[lv * lo.n_chunks + count[lv]] = k;
    count[lv]++;
  }
  if (!ok) {
    atomicOr(status, kStCorrupt);
    for (int i = 0; i < kMaxLevels; i++) count[i] = 0;
  }
}

template <int T>
__device__ __forceinline__ uint32_t team_mask() {
  const int lane = threadIdx.x & 31;
  return T == 32 ? 0xffffffffu : (((1u << T) - 1u) << (lane & ~(T - 1)));
}

// Row tib of physical block b in a paged cache, at thread i's lanes; ok is
// false (and the row must not be written) when the block id is out of
// range or the pool pointer is null or misaligned.
__device__ __forceinline__ uint16_t *paged_row(const PagedOut &po, uint16_t *pool, int32_t b, int tib,
                                               int h, const Layout &lo, int i, bool &ok) {
  ok = b >= 0 && b < po.n_blocks && pool != nullptr && (reinterpret_cast<uintptr_t>(pool) & 15) == 0;
  return pool + ((uint64_t(ok ? b : 0) * lo.H + h) * po.bt + tib) * lo.d + kLpt * i;
}

// ---------------------------------------------------------------- tables
// A head's d frequency tables in shared memory, laid out so that thread i
// of a team of T threads (lanes 4i..4i+3) only ever touches bank i: u16
// position p of a table row holds the channel 4 ti + j with
// p = (j >> 1) * 2T + 2 ti + (j & 1).
template <int T>
__device__ __forceinline__ int chan_of(int p) {
  const int r = p % (2 * T);
  return 4 * (r >> 1) + 2 * (p / (2 * T)) + (r & 1);
}

// The d cdf columns (global, [d][256] u16) -> cdfc rows 0..255 (position p
// of a row of kRow entries holding channel chan(p)), row 256 repeating
// cdf_255 (so that f_255, the escape, reads as 0) and a zero row 257.  A
// thread takes 8 rows of one position (one 16-byte load); neighbouring
// threads store neighbouring positions of a row.  A column that does not
// start at 0 or does not strictly increase sets *bad.
template <int kRow, typename Chan>
__device__ __forceinline__ void build_cdf_rows(const uint16_t *cdf, uint16_t *cdfc, int *bad, Chan chan) {
  for (int e = threadIdx.x; e < 32 * kRow; e += blockDim.x) {
    const int p = e % kRow, s0 = 8 * (e / kRow);
    const uint16_t *src = cdf + chan(p) * 256 + s0;
    const uint4 v = *reinterpret_cast<const uint4 *>(src);
    const uint32_t nx = s0 + 8 < 256 ? uint32_t(src[8]) : kM;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    bool b = s0 == 0 && (w[0] & 0xFFFFu) != 0;
#pragma unroll
    for (int q = 0; q < 8; q++) {
      const uint32_t c0 = (w[q >> 1] >> (16 * (q & 1))) & 0xFFFFu;
      const uint32_t c1 = q < 7 ? (w[(q + 1) >> 1] >> (16 * ((q + 1) & 1))) & 0xFFFFu : nx;
      b |= c1 <= c0;
      cdfc[(s0 + q) * kRow + p] = uint16_t(c0);
      if (s0 + q == 255) cdfc[256 * kRow + p] = uint16_t(c0);
    }
    if (b) *bad = 1;
  }
  for (int p = threadIdx.x; p < kRow; p += blockDim.x) cdfc[257 * kRow + p] = 0;
}

// The same for the position order of k_decode's tables (thread i of a team
// of T on lanes 4i..4i+3, bank i).
template <int T>
__device__ __forceinline__ void build_cdf_columns(const uint16_t *cdf, uint16_t *cdfc, int *bad) {
  build_cdf_rows<kLpt * T>(cdf, cdfc, bad, [](int p) { return chan_of<T>(p); });
}

// First symbol of the neighbouring pair (sa, sa + 1) holding most of the
// slots [slot0, slot0 + width) of column colp (row stride kRow), where s is
// the symbol at slot0.
template <int kRow>
__device__ __forceinline__ uint32_t densest_pair(const uint16_t *colp, uint32_t s, uint32_t slot0,
                                                 uint32_t width) {
  uint32_t sa = s, t = s, beg = slot0, prev = 0, best = 0;
  for (;;) {
    const uint32_t nt = t < 255 ? uint32_t(colp[(t + 1) * kRow]) : kM;
    const uint32_t cnt = min(nt, slot0 + width) - beg;  // in-bucket slots of t
    if (t > s && prev + cnt > best) {
      best = prev + cnt;
      sa = t - 1;
    }
    if (t == 255 || nt >= slot0 + width) break;
    prev = cnt;
    beg = nt;
    t++;
  }
  return sa;
}

// Full bucket entries: lut16 [512 buckets][row] u16 = sa << 8 | (255 - last
// offset of sa in the 128-slot bucket).  A thread walks 64 buckets of the
// two positions of one 32-bit word, carrying the current symbol from bucket
// to bucket.
template <int T>
__device__ __forceinline__ void build_lut16(uint16_t *lut16, const uint16_t *cdfc) {
  constexpr int kRow = kLpt * T;
  for (int e = threadIdx.x; e < 8 * 2 * T; e += blockDim.x) {
    const int wd = e % (2 * T), b0 = 64 * (e / (2 * T));
#pragma unroll
    for (int hpos = 0; hpos < 2; hpos++) {
      const uint16_t *colp = cdfc + 2 * wd + hpos;
      uint32_t s = 0;  // largest s with cdf_s <= 128 b0 (cdf_0 = 0)
#pragma unroll
      for (uint32_t stp = 128; stp; stp >>= 1)
        if (s + stp <= 255 && colp[(s + stp) * kRow] <= kBucketSlots * b0) s += stp;
      for (int bb = 0; bb < 64; bb++) {
        const uint32_t slot0 = kBucketSlots * (b0 + bb);
        while (s < 255 && colp[(s + 1) * kRow] <= slot0) s++;
        const uint32_t sa = densest_pair<kRow>(colp, s, slot0, kBucketSlots);
        const uint32_t nxt = sa < 255 ? uint32_t(colp[(sa + 1) * kRow]) : kM;
        const uint32_t bnd = min(nxt - slot0, kBucketSlots) - 1;  // last slot of sa in the bucket
        lut16[(b0 + bb) * kRow + 2 * wd + hpos] = uint16_t((sa << 8) | (255 - bnd));
      }
    }
  }
}

// ---------------------------------------------------------------- decode
// Shared memory per CTA (d lanes, T = d/4 threads per team), 119 KB at d = 64
// with 22 teams:
//   lut16 [512 buckets][4 lanes x T] u16 : sa << 8 | (255 - last offset of sa
//                                          in the 128-slot bucket), where
//                                          (sa, sa + 1) is the neighbouring
//                                          pair holding most of the bucket
//   cdfc  [258 rows][4 lanes x T] u16    : cdf_s for s < 256; row 256 repeats
//                                          cdf_255; row 257 is padding
//   rings [teams][512 + 16] u16          : the staged words of each team
// Thread i of a team owns lanes 4i..4i+3; within a row its two 32-bit words
// (lanes 0-1 and 2-3) sit at word index i and T + i, so with T = 32 every
// access of thread i to lut16 or cdfc hits bank i, whatever the symbols.
// PAGED: token rows go to the paged cache po instead of kv.
template <int T, bool PAGED>
__global__ void __launch_bounds__(max_threads<T>())
k_decode(Layout lo, const uint8_t *__restrict__ tables, const uint8_t *__restrict__ buf,
         uint16_t *__restrict__ kv, uint8_t *ws, PagedOut po, int si_lo, int si_hi) {
  extern __shared__ __align__(16) uint32_t smem[];
  uint16_t *lut16 = reinterpret_cast<uint16_t *>(smem);  // [kBuckets][2][T][2]
  uint16_t *cdfc = lut16 + kBuckets * kLpt * T;          // [kCdfRows][2][T][2]
  uint16_t *rings = cdfc + kCdfRows * kLpt * T;          // [teams][kRing + kMirror] words
  __shared__ int s_bad;

  const int lv = blockIdx.x, si = blockIdx.y;
  if (si < si_lo || si >= si_hi) return;  // outside the requested layers
  const int cnt = reinterpret_cast<const int32_t *>(ws + 64)[lv];
  if (cnt == 0) return;
  const int32_t *list = reinterpret_cast<const int32_t *>(ws + 256) + lv * lo.n_chunks;
  uint32_t *status = reinterpret_cast<uint32_t *>(ws);
  const int h = si % lo.H, kvi = (si / lo.H) % 2, l = si / (2 * lo.H);

  // ---- tables -> shared memory
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const uint16_t *cdf = reinterpret_cast<const uint16_t *>(tables + lo.tb_cdf) +
                        tab_index(lo, lv, l, kvi, h * lo.d) * 256;
  build_cdf_columns<T>(cdf, cdfc, &s_bad);
  __syncthreads();
  build_lut16<T>(lut16, cdfc);
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) atomicOr(status, kStCorrupt);
    return;
  }

  const int team = threadIdx.x / T, i = threadIdx.x % T, nteams = blockDim.x / T;
  const uint32_t tm = team_mask<T>();
  const float4 st4 = *reinterpret_cast<const float4 *>(
      reinterpret_cast<const float *>(tables + lo.tb_step) + tab_index(lo, lv, l, kvi, h * lo.d + kLpt * i));
  const float step[4] = {st4.x, st4.y, st4.z, st4.w};
  // thread i's entries: u16 index row * (4T) + (j>>1)*2T + 2i + (j&1); with
  // T = 32 a row is 256 bytes, so the bucket row of state x is x & 0xFF00.
  const uint16_t *lt = lut16 + 2 * i;
  const uint16_t *ct = cdfc + 2 * i;

  for (int idx = team; idx < cnt; idx += nteams) {
    const int k = list[idx];
    const int ng = chunk_ng(lo, k), ntok = chunk_ntok(lo, k), nd = chunk_nd(lo, k);
    const uint64_t base = ld_u64(buf + 64 + 8 * uint64_t(k));
    const uint64_t cend = (k + 1 < lo.n_chunks) ? ld_u64(buf + 64 + 8 * uint64_t(k + 1))
                                                 : ld_u64(buf + 48);
    const uint8_t *chunk = buf + base;
    const uint64_t fixed = chunk_fixed(lo, k);
    const uint32_t *soffv = reinterpret_cast<const uint32_t *>(chunk + chunk_sec_off(lo, k));
    const uint64_t so = soffv[si];
    const uint64_t se = (si + 1 < lo.nstr) ? uint64_t(soffv[si + 1]) : (cend - base);
    bool ok = !(so & 15) && so >= fixed && se >= so && base + se <= cend &&
              se - so >= 16 + 4 * uint64_t(lo.d);
    const uint8_t *blk = chunk + so;
    uint32_t nw = 0, ne = 0;
    if (ok) {
      const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
      nw = hdr.x;
      ne = hdr.y;
      ok = hdr.z == uint32_t(nd) && hdr.w == 0 &&
           16 + 4 * uint64_t(lo.d) + 2 * uint64_t(nw) <= se - so;
    }
    if (!ok) {
      if (i == 0) atomicOr(status, kStCorrupt);
      continue;
    }
    const uint4 xs = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * i);
    uint32_t x[4] = {xs.x, xs.y, xs.z, xs.w};
    const uint16_t *__restrict__ words = reinterpret_cast<const uint16_t *>(blk + 16 + 4 * lo.d);
    // stage the first kRing words (two halves) of the stream in the ring
    uint16_t *ring = rings + team * (kRing + kMirror);
    const uint32_t wbytes = 2 * nw;
    auto load_half = [&](uint32_t w0) {  // words [w0, w0 + kHalf) -> ring half
      for (uint32_t o = 16 * i; o < 2 * kHalf; o += 16 * T) {
        const uint32_t b = 2 * w0 + o;  // byte offset in the word array
        const uint32_t n = b < wbytes ? min(16u, wbytes - b) : 0u;
        cp_async16(ring + ((w0 + o / 2) & (kRing - 1)), reinterpret_cast<const uint8_t *>(words) + (n ? b : 0), n);
      }
      if ((w0 & (kRing - 1)) == 0 && 16 * uint32_t(i) < 2 * kMirror) {  // the mirror of ring[0, kMirror)
        const uint32_t b = 2 * w0 + 16 * i;
        const uint32_t n = b < wbytes ? min(16u, wbytes - b) : 0u;
        cp_async16(ring + kRing + 8 * i, reinterpret_cast<const uint8_t *>(words) + (n ? b : 0), n);
      }
      cp_async_commit();
    };
    __syncwarp(tm);  // the previous stream's reads of this ring are done
    load_half(0);
    load_half(kHalf);
    uint32_t rbase = 0;  // the ring holds words [rbase, rbase + kRing)
    uint32_t ready = 0;  // words [rbase, ready) have landed and are visible to the team
    uint32_t lim = 0;    // p + tot <= lim: no check, refill or wait needed
    const float4 s4 = *reinterpret_cast<const float4 *>(chunk + lo.sec_s + (uint64_t(si) * lo.d + kLpt * i) * 4);
    const float sc[4] = {s4.x, s4.y, s4.z, s4.w};
    const uint8_t *anc = chunk + lo.sec_anc + uint64_t(si) * ng * lo.d + kLpt * i;
    uint32_t p = 0, nesc = 0;
    bool broken = false;

    // output row of the team's current token
    uint16_t *orow;
    bool row_ok = true, bad_row = false;
    [[maybe_unused]] uint16_t *pool = nullptr;
    [[maybe_unused]] int64_t lblk = 0, lblk_end = 0;  // logical block; one past the chunk's last
    [[maybe_unused]] int left = 0;                    // rows left in the current block
    [[maybe_unused]] int32_t bnext = 0;               // block id of logical block lblk + 1, loaded a block ahead
    if constexpr (PAGED) {
      pool = po.pools[l * 2 + kvi];
      const int64_t t0 = int64_t(k) * lo.C;
      lblk = t0 / po.bt;
      lblk_end = (t0 + ntok - 1) / po.bt + 1;
      const int tib = int(t0 - lblk * po.bt);
      left = po.bt - tib;
      orow = paged_row(po, pool, po.table[lblk], tib, h, lo, i, row_ok);
      bad_row = !row_ok;
      if (lblk + 1 < lblk_end) bnext = po.table[lblk + 1];
    } else {
      orow = kv + (uint64_t(si) * lo.S + uint64_t(k) * lo.C) * lo.d + kLpt * i;
    }
    auto next_row = [&]() {
      if constexpr (PAGED) {
        if (--left == 0) {  // the block is full: the next one, if the chunk reaches it
          left = po.bt;
          if (++lblk < lblk_end) {
            orow = paged_row(po, pool, bnext, 0, h, lo, i, row_ok);
            bad_row |= !row_ok;
            if (lblk + 1 < lblk_end) bnext = po.table[lblk + 1];
          }
        } else {
          orow += lo.d;
        }
      } else {
        orow += lo.d;
      }
    };
    uint32_t a4n = *reinterpret_cast<const uint32_t *>(anc);  // next group's anchors, loaded ahead
    for (int g = 0; g < ng && !broken; g++) {
      const uint32_t a4 = a4n;
      if (g + 1 < ng) a4n = *reinterpret_cast<const uint32_t *>(anc + uint64_t(g + 1) * lo.d);
      float ah[4];
#pragma unroll
      for (int j = 0; j < 4; j++) ah[j] = __fmul_rn(float(int8_t(a4 >> (8 * j))), sc[j]);
      if (!PAGED || row_ok)
        *reinterpret_cast<uint2 *>(orow) = make_uint2(pack_f16x2(ah[0], ah[1]), pack_f16x2(ah[2], ah[3]));
      next_row();
      const int nt = min(lo.G, ntok - g * lo.G) - 1;  // delta tokens in this group
      for (int tt = 0; tt < nt; tt++, next_row()) {
        // ---- symbol search.  The bucket entry of slot >> 7 holds a symbol
        // sa and the last in-bucket offset of sa's range, so one carry picks
        // sa or sa + 1.  A lane whose slot falls outside that pair (buckets
        // holding 3+ symbols, the distribution tails) or whose symbol is the
        // escape (its frequency reads as 0) is marked slow and resolved below.
        uint32_t sy[4], ff[4], rr[4];
        bool sl[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const int cj = (j >> 1) * T * 2 + (j & 1);
          const uint32_t b = (x[j] >> kBucketShift) & (kBuckets - 1);
          const uint32_t lu = lt[b * (kLpt * T) + cj];
          // carry out of the low byte adds one when the slot is past s0's part of the bucket
          const uint32_t sj = ((x[j] & (kBucketSlots - 1)) + lu) >> 8;
          const uint32_t c0 = ct[sj * (kLpt * T) + cj];
          const uint32_t c1 = ct[(sj + 1) * (kLpt * T) + cj];
          ff[j] = c1 - c0;
          rr[j] = (x[j] & 0xFFFFu) - c0;  // wraps above 0xFFFF when the slot is below sa
          sy[j] = sj;
          sl[j] = rr[j] >= ff[j];
        }
        // Slow lanes: about 1% of lanes.  Symbol 255 is the escape, whose
        // raw value follows in the words.
        uint32_t escm = 0;
        if (sl[0] | sl[1] | sl[2] | sl[3]) {
          // a binary search in the lane's own table column, between the
          // previous bucket's pair and the chosen pair when the slot is below
          // it, else between the pair and the next bucket's pair
#pragma unroll
          for (int j = 0; j < 4; j++) {
            if (sl[j]) {
              const int cj = (j >> 1) * T * 2 + (j & 1);
              const uint32_t slot = x[j] & 0xFFFFu;
              uint32_t lo = sy[j], hi = lo;
              const uint32_t b = slot >> kBucketShift;
              if (rr[j] > 0xFFFFu) {  // below the pair: down to the previous bucket's pair
                hi = lo - 1;
                lo = b > 0 ? (lt[(b - 1) * (kLpt * T) + cj] >> 8) : 0u;
              } else if (lo < 255) {  // above the pair (255: the escape symbol, already found)
                lo += 1;  // cdf_lo <= slot is known
                hi = b + 1 < kBuckets ? (lt[(b + 1) * (kLpt * T) + cj] >> 8) : 255u;
              }
              while (lo < hi) {
                const uint32_t mid = (lo + hi + 1) >> 1;
                if (ct[mid * (kLpt * T) + cj] <= slot) lo = mid;
                else hi = mid - 1;
              }
              const uint32_t c0 = ct[lo * (kLpt * T) + cj];
              const uint32_t c1 = lo < 255 ? uint32_t(ct[(lo + 1) * (kLpt * T) + cj]) : kM;
              sy[j] = lo;
              ff[j] = c1 - c0;
              rr[j] = slot - c0;
              escm |= lo == uint32_t(kEsc) ? (1u << j) : 0u;
            }
          }
        }
        bool nd4[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
          x[j] = ff[j] * (x[j] >> 16) + rr[j];
          nd4[j] = x[j] < kRansL;
        }
        const int cntw = int(nd4[0]) + int(nd4[1]) + int(nd4[2]) + int(nd4[3]) + 2 * __popc(escm);  // 0..12 words
        // ---- word positions: team-wide exclusive scan of the word counts
        int incl = cntw;
#pragma unroll
        for (int o = 1; o < T; o <<= 1) {
          const int v = __shfl_up_sync(tm, incl, o, T);
          if (i >= o) incl += v;
        }
        const uint32_t tot = uint32_t(__shfl_sync(tm, incl, T - 1, T));
        const uint32_t excl = uint32_t(incl - cntw);
        uint32_t pos = p + excl;
        bool in_ring = true;
        if (p + tot > lim) {  // past the words known to be staged, or a refill may be due
        if (p + tot > nw) {
          broken = true;
          break;
        }
        // make words [p, p + tot) available in the ring
        if (p >= rbase + kHalf) {
          __syncwarp(tm);  // every thread's reads of the consumed half are done
          do {  // first half consumed: refill it with the next words
            load_half(rbase + kRing);
            rbase += kHalf;
          } while (p >= rbase + kHalf);
        }
        in_ring = p + tot <= rbase + kRing;
        if (p + tot > ready) {  // words past what is known to have landed
          if (p + tot <= rbase + kHalf) {
            cp_async_wait_prev();
            ready = rbase + kHalf;
          } else {
            cp_async_wait_all();
            ready = rbase + kRing;
          }
          __syncwarp(tm);
        }
        lim = min(nw, min(ready, rbase + kHalf));
        }
        p += tot;
        float v[4];
        if (in_ring) {
        if (escm == 0) {
          // the thread's words are consecutive from pos: read four (the
          // mirror covers reads past the ring's end; unneeded ones are
          // ignored) and give lane j word number nd_0 + .. + nd_(j-1)
          const uint16_t *rp = ring + (pos & (kRing - 1));
          const uint32_t w0 = rp[0], w1 = rp[1], w2 = rp[2], w3 = rp[3];
          const uint32_t a1 = nd4[0] ? w1 : w0, a2 = nd4[0] ? w2 : w1, a3 = nd4[0] ? w3 : w2;
          const uint32_t b2 = nd4[1] ? a2 : a1, b3 = nd4[1] ? a3 : a2;
          const uint32_t wl[4] = {w0, a1, b2, nd4[2] ? b3 : b2};
#pragma unroll
          for (int j = 0; j < 4; j++) {
            x[j] = nd4[j] ? __byte_perm(wl[j], x[j], 0x5410) : x[j];  // x<<16 | w
            // q = sy - 127 as an exact fp32 (|q| < 2^22): (1.5*2^23 + sy) - (1.5*2^23 + 127)
            const float qf = __int_as_float(0x4B400000 + int(sy[j])) - 12583039.0f;
            v[j] = __fmaf_rn(qf, step[j], ah[j]);
          }
        } else {  // escapes: the raw q follows the lane's renormalisation word
#pragma unroll
          for (int j = 0; j < 4; j++) {
            if (nd4[j]) x[j] = __byte_perm(uint32_t(ring[pos++ & (kRing - 1)]), x[j], 0x5410);
            if ((escm >> j) & 1u) {
              const int q = int(uint32_t(ring[pos & (kRing - 1)]) | (uint32_t(ring[(pos + 1) & (kRing - 1)]) << 16));
              pos += 2;
              nesc++;
              v[j] = __fmaf_rn(__int2float_rn(q), step[j], ah[j]);
            } else {
              const float qf = __int_as_float(0x4B400000 + int(sy[j])) - 12583039.0f;
              v[j] = __fmaf_rn(qf, step[j], ah[j]);
            }
          }
        }
        } else {  // a burst longer than the ring: straight from memory
        if (escm == 0) {
#pragma unroll
          for (int j = 0; j < 4; j++) {
            if (nd4[j]) x[j] = __byte_perm(uint32_t(words[pos++]), x[j], 0x5410);  // x<<16 | w
            // q = sy - 127 as an exact fp32 (|q| < 2^22): (1.5*2^23 + sy) - (1.5*2^23 + 127)
            const float qf = __int_as_float(0x4B400000 + int(sy[j])) - 12583039.0f;
            v[j] = __fmaf_rn(qf, step[j], ah[j]);
          }
        } else {  // escapes: the raw q follows the lane's renormalisation word
#pragma unroll
          for (int j = 0; j < 4; j++) {
            if (nd4[j]) x[j] = __byte_perm(uint32_t(words[pos++]), x[j], 0x5410);
            if ((escm >> j) & 1u) {
              const int q = int(uint32_t(words[pos]) | (uint32_t(words[pos + 1]) << 16));
              pos += 2;
              nesc++;
              v[j] = __fmaf_rn(__int2float_rn(q), step[j], ah[j]);
            } else {
              const float qf = __int_as_float(0x4B400000 + int(sy[j])) - 12583039.0f;
              v[j] = __fmaf_rn(qf, step[j], ah[j]);
            }
          }
        }
        }
        if (!PAGED || row_ok)
          *reinterpret_cast<uint2 *>(orow) = make_uint2(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]));
      }
    }
    cp_async_wait_all();
    if (PAGED && bad_row) atomicOr(status, kStBadArg);
#pragma unroll
    for (int o = T / 2; o; o >>= 1) nesc += __shfl_xor_sync(tm, nesc, o, T);
    const bool lanes_ok = x[0] == kRansL && x[1] == kRansL && x[2] == kRansL && x[3] == kRansL;
    if (broken || !lanes_ok || p != nw || nesc != ne) atomicOr(status, kStCorrupt);
  }
}

// ---------------------------------------------------------------- d = 128
// The decoder for d = 128 (the models' head dim).  One CTA per (level,
// head), a warp per chunk stream, thread i on lanes 4i..4i+3, as k_decode,
// with tables laid out for a short token loop:
//   - main  [256 buckets][128] u16: for the 256-slot bucket slot >> 8, the
//           first symbol sa of the neighbouring pair holding most of it and
//           the last offset of sa's range in it (sa << 8 | 255 - offset),
//           so one carry out of the low byte picks sa or sa + 1;
//   - fine  [256][128] u16, the same entries for 16-slot buckets over the
//           two ends of the slot range, [0, 2048) and [63488, 65536): the
//           distribution tails, where a 256-slot bucket holds many narrow
//           symbols;
//   - cdfc  [258][128] u16 as k_decode's (row 256 repeats cdf_255).
// Each table row holds the 128 channels with thread i's lanes at byte 4i
// of each 128-byte half (bank i), addressed by 32-bit byte offsets.  For a
// lane with state x the main entry's row is x & 0xFF00; a main entry of a
// tail bucket is 0xFFFF, and the lane takes the fine entry at row
// (x << 4) & 0xFF00 instead (bits 4..11 of the slot: rows 0..127 for the low
// end, 128..255 for the high end); both entries are loaded and one selected,
// which keeps the warp off a divergent branch.  The carry out of (x & 255) + entry gives
// t with t & 0xFF00 = symbol * 256: the symbol's cdf row offset and, OR-ed
// into the bits of 2^15, the exact fp32 2^15 + symbol.  A lane whose slot
// still falls outside the pair (about 0.1% on the 70B-shaped workload), or
// whose symbol is the escape, is resolved by a binary search of its cdf
// column; one warp vote per token guards that path.  Words are staged per warp in a
// ring of two halves: the token that crosses into the second half waits for
// it and, after its reads, refills the consumed half.
constexpr uint32_t kMainOff = 0;                        // main [256][128] u16
constexpr uint32_t kFineOff = 256 * 256;                // fine [256][128] u16
constexpr uint32_t kCdfOff = 2 * 256 * 256;             // cdfc [258][128] u16
constexpr uint32_t kRingOff = kCdfOff + kCdfRows * 256; // rings [teams][kRing + kMirror] u16
constexpr uint32_t kRingStride = kRing + kMirror;       // words per warp ring
constexpr uint32_t kTail = 2048;                        // slots covered by the fine table at each end
constexpr int kTeams128Max = 24;
// MID (ranges with a few chunks per level): u8 pair tables as k_thin128's,
// in this kernel's column order (lane 4 i + j at byte 4 i + j, bank i), so
// that two CTAs of eight teams share an SM.
constexpr uint32_t kMidFine = 0;                       // fine [64][128] u8: 32-slot buckets, 1024-slot tails
constexpr uint32_t kMidMain = kMidFine + 64 * 128;     // main [248][128] u8: 256-slot buckets of [1024, 64512)
constexpr uint32_t kMidCdf = kMidMain + 248 * 128;     // cdfc [258][128] u16
constexpr uint32_t kMidRing = kMidCdf + kCdfRows * 256;
constexpr int kMidTeams = 8;
template <bool MID>
__host__ __device__ constexpr uint32_t cdf_off() { return MID ? kMidCdf : kCdfOff; }
template <bool MID>
__host__ __device__ constexpr uint32_t ring_off() { return MID ? kMidRing : kRingOff; }

// byte offset of lane j of thread 0 in a table row (thread i adds 4 i)
template <int J>
__device__ __forceinline__ constexpr uint32_t colb() { return (J >> 1) * 128 + (J & 1) * 2; }

__device__ __forceinline__ uint32_t lds16(const uint8_t *sm, uint32_t off) {
  return *reinterpret_cast<const uint16_t *>(sm + off);
}

// Inclusive warp scan step: v += (value of lane i - O, when there is one).
template <int O>
__device__ __forceinline__ uint32_t scan_step(uint32_t v) {
  asm("{\n\t.reg .pred p;\n\t.reg .u32 t;\n\t"
      "shfl.sync.up.b32 t|p, %0, %1, 0, -1;\n\t"
      "@p add.u32 %0, %0, t;\n\t}"
      : "+r"(v) : "n"(O));
  return v;
}

// Bucket entries for the d = 128 tables (cdf rows of 128 u16 positions).  A
// thread takes kG consecutive buckets of one position, positions fastest so
// that a warp's threads read different banks: a binary search of the
// position's cdf column for the symbol at the first bucket's first slot, then
// per bucket a walk over the symbols it holds for the first symbol sa of the
// neighbouring pair holding most of its `width` slots, carrying the symbol at
// the bucket's end to the next bucket.  emit(b, p, sa, nxt, slot0) writes the
// entry of bucket b (first slot slot0) at position p; nxt = cdf_(sa+1) (M for
// sa = 255).
template <typename Emit>
__device__ __forceinline__ void build_buckets(const uint16_t *cdfc, int nb, uint32_t width, uint32_t base,
                                              Emit emit) {
  constexpr int kRowU = 128, kG = 8;
  const int n = (nb + kG - 1) / kG * kRowU;
  for (int e = threadIdx.x; e < n; e += int(blockDim.x)) {
    const uint32_t p = e % kRowU, b0 = e / kRowU * kG;
    const uint16_t *colp = cdfc + p;
    uint32_t slot0 = base + width * b0;
    uint32_t s = 0;  // largest s with cdf_s <= slot0 (cdf_0 = 0)
#pragma unroll
    for (uint32_t stp = 128; stp; stp >>= 1)
      if (s + stp <= 255 && colp[(s + stp) * kRowU] <= slot0) s += stp;
    uint32_t cs1 = s < 255 ? uint32_t(colp[(s + 1) * kRowU]) : kM;  // cdf_(s+1)
    for (uint32_t b = b0; b < b0 + kG && int(b) < nb; b++) {
      const uint32_t end = slot0 + width;
      uint32_t t = s, nt = cs1, beg = slot0, prev = 0, best = 0, sa = s, nxt = cs1;
      for (;;) {
        const uint32_t cnt = min(nt, end) - beg;  // in-bucket slots of t
        if (t > s && prev + cnt > best) {
          best = prev + cnt;
          sa = t - 1;
          nxt = beg;  // cdf_t
        }
        if (t == 255 || nt >= end) break;
        prev = cnt;
        beg = nt;
        t++;
        nt = t < 255 ? uint32_t(colp[(t + 1) * kRowU]) : kM;
      }
      emit(b, p, sa, nxt, slot0);
      // the next bucket's first symbol: t, or past the symbols ending at `end`
      s = t;
      cs1 = nt;
      while (s < 255 && cs1 <= end) {
        s++;
        cs1 = s < 255 ? uint32_t(colp[(s + 1) * kRowU]) : kM;
      }
      slot0 = end;
    }
  }
}

// Pair entries for nb consecutive buckets of `width` slots (a power of two
// up to 256) from slot `base`: entry b at position p is sa << 8 | (255 - the
// last offset of sa's range in the bucket - bias).  For 16-slot buckets bias
// is the bucket's offset in its 256-slot bucket (16 (b mod 16)), so that the
// carry out of (x & 255) + entry is the same test as for the main table.
// Buckets below flag_lo or from flag_hi get 0xFFFF instead, without a search
// (a tail bucket of 256 slots can hold hundreds of one-slot symbols).
__device__ __forceinline__ void build_pairs(uint16_t *lut, const uint16_t *cdfc, int nb, uint32_t width,
                                            uint32_t base, int flag_lo, int flag_hi) {
  for (int e = threadIdx.x; e < nb * 128; e += blockDim.x)
    if (e / 128 < flag_lo || e / 128 >= flag_hi) lut[e] = 0xFFFFu;
  build_buckets(cdfc, flag_hi - flag_lo, width, base + width * uint32_t(flag_lo),
                [&](uint32_t b, uint32_t p, uint32_t sa, uint32_t nxt, uint32_t slot0) {
                  const uint32_t bb = b + uint32_t(flag_lo);           // the bucket in the table
                  const uint32_t bnd = min(nxt - slot0, width) - 1;  // last offset of sa in the bucket
                  const uint32_t bias = width < 256 ? width * (bb & (256 / width - 1)) : 0u;
                  lut[bb * 128 + p] = uint16_t((sa << 8) | (255 - bnd - bias));
                });
}

// Slow lane J (a slot outside the pair its bucket entry names, or the
// escape symbol, whose frequency reads as 0): a binary search of the lane's
// cdf column.  Replaces the lane's frequency, offset in range and symbol
// row (symbol << 8); marks an escape in escm.
template <int J, uint32_t CDF>
__device__ __forceinline__ void slow128(const uint8_t *sm, uint32_t i4, uint32_t x, uint32_t &ff, uint32_t &rr,
                                        uint32_t &ro, uint32_t &escm) {
  const uint32_t col = i4 + colb<J>();
  const uint32_t slot = x & 0xFFFFu;
  uint32_t s = 0;  // largest s with cdf_s <= slot (cdf_0 = 0)
#pragma unroll
  for (uint32_t stp = 128; stp; stp >>= 1)
    if (lds16(sm, CDF + ((s + stp) << 8) + col) <= slot) s += stp;
  const uint32_t c0 = lds16(sm, CDF + (s << 8) + col);
  const uint32_t c1 = s < 255 ? lds16(sm, CDF + ((s + 1) << 8) + col) : kM;
  ff = c1 - c0;
  rr = slot - c0;
  ro = s << 8;
  if (s == uint32_t(kEsc)) escm |= 1u << J;
}

// cmin, cmax: the CTA decodes its level only if the level holds that many
// chunks in the range (the launches for the other counts take the rest).
// Grid rows from split0 on come in pairs: the two CTAs of a pair decode the
// even and the odd entries of the same head's chunk list.
template <bool PAGED, bool MID>
__global__ void __launch_bounds__(MID ? kMidTeams * 32 : kTeams128Max * 32, MID ? 2 : 1)
k_dec128(Layout lo, const uint8_t *__restrict__ tables, const uint8_t *__restrict__ buf,
         uint16_t *__restrict__ kv, uint8_t *ws, PagedOut po, int si_lo, int si_hi, int cmin, int cmax,
         int split0) {
  constexpr int T = 32;
  extern __shared__ __align__(16) uint8_t smb[];
  __shared__ int s_bad;
  uint16_t *cdfc = reinterpret_cast<uint16_t *>(smb + cdf_off<MID>());

  const int lv = blockIdx.x;
  int si = blockIdx.y, part = 0, nparts = 1;
  if (si >= split0) {
    si = split0 + (int(blockIdx.y) - split0) / 2;
    part = (int(blockIdx.y) - split0) & 1;
    nparts = 2;
  }
  if (si < si_lo || si >= si_hi) return;  // outside the requested layers
  const int cnt = reinterpret_cast<const int32_t *>(ws + 64)[lv];
  const int nteams = blockDim.x >> 5, first = int(blockIdx.z) * nteams;  // this CTA's entries of the list
  if (cnt < cmin || cnt > cmax || part + nparts * first >= cnt) return;
  const int32_t *list = reinterpret_cast<const int32_t *>(ws + 256) + lv * lo.n_chunks;
  uint32_t *status = reinterpret_cast<uint32_t *>(ws);
  const int h = si % lo.H, kvi = (si / lo.H) % 2, l = si / (2 * lo.H);

  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const uint16_t *cdf = reinterpret_cast<const uint16_t *>(tables + lo.tb_cdf) +
                        tab_index(lo, lv, l, kvi, h * lo.d) * 256;
  build_cdf_columns<T>(cdf, cdfc, &s_bad);
  __syncthreads();
  if constexpr (MID) {
    // the lane at cdf position p owns byte chan_of(p) of a u8 row
    const auto sa8 = [&](uint8_t *lut) {
      return [lut](uint32_t b, uint32_t p, uint32_t sa, uint32_t, uint32_t) {
        lut[b * 128 + chan_of<T>(int(p))] = uint8_t(min(sa, 254u));
      };
    };
    build_buckets(cdfc, 248, 256, 1024, sa8(smb + kMidMain));
    build_buckets(cdfc, 32, 32, 0, sa8(smb + kMidFine));
    build_buckets(cdfc, 32, 32, kM - 1024, sa8(smb + kMidFine + 32 * 128));
  } else {
    // main entries of the tail buckets (the first and last 8) point to the fine table
    build_pairs(reinterpret_cast<uint16_t *>(smb + kMainOff), cdfc, 256, 256, 0, kTail / 256, 256 - kTail / 256);
    build_pairs(reinterpret_cast<uint16_t *>(smb + kFineOff), cdfc, 128, 16, 0, 0, 128);
    build_pairs(reinterpret_cast<uint16_t *>(smb + kFineOff) + 128 * 128, cdfc, 128, 16, kM - kTail, 0, 128);
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) atomicOr(status, kStCorrupt);
    return;
  }

  const int team = threadIdx.x >> 5;
  const uint32_t i = threadIdx.x & 31, i4 = 4 * i;
  const float4 st4 = *reinterpret_cast<const float4 *>(
      reinterpret_cast<const float *>(tables + lo.tb_step) + tab_index(lo, lv, l, kvi, h * lo.d + i4));
  const float step[4] = {st4.x, st4.y, st4.z, st4.w};
  uint16_t *ring = reinterpret_cast<uint16_t *>(smb + ring_off<MID>()) + team * kRingStride;

  for (int idx = part + nparts * (first + team); idx < cnt; idx += nparts * nteams * int(gridDim.z)) {
    const int k = list[idx];
    const int ng = chunk_ng(lo, k), ntok = chunk_ntok(lo, k), nd = chunk_nd(lo, k);
    const uint64_t base = ld_u64(buf + 64 + 8 * uint64_t(k));
    const uint64_t cend = (k + 1 < lo.n_chunks) ? ld_u64(buf + 64 + 8 * uint64_t(k + 1)) : ld_u64(buf + 48);
    const uint8_t *chunk = buf + base;
    const uint32_t *soffv = reinterpret_cast<const uint32_t *>(chunk + chunk_sec_off(lo, k));
    const uint64_t so = soffv[si];
    const uint64_t se = (si + 1 < lo.nstr) ? uint64_t(soffv[si + 1]) : (cend - base);
    bool ok = !(so & 15) && so >= chunk_fixed(lo, k) && se >= so && base + se <= cend &&
              se - so >= 16 + 4 * uint64_t(lo.d);
    const uint8_t *blk = chunk + so;
    uint32_t nw = 0, ne = 0;
    if (ok) {
      const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
      nw = hdr.x;
      ne = hdr.y;
      ok = hdr.z == uint32_t(nd) && hdr.w == 0 && 16 + 4 * uint64_t(lo.d) + 2 * uint64_t(nw) <= se - so;
    }
    if (!ok) {
      if (i == 0) atomicOr(status, kStCorrupt);
      continue;
    }
    const uint4 xs = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * i);
    uint32_t x[4] = {xs.x, xs.y, xs.z, xs.w};
    const uint16_t *__restrict__ words = reinterpret_cast<const uint16_t *>(blk + 16 + 4 * lo.d);
    const uint32_t wbytes = 2 * nw;
    auto load_half = [&](uint32_t w0) {  // words [w0, w0 + kHalf) -> ring half, zero past the end
      for (uint32_t o = 16 * i; o < 2 * kHalf; o += 16 * T) {
        const uint32_t b = 2 * w0 + o;
        const uint32_t n = b < wbytes ? min(16u, wbytes - b) : 0u;
        cp_async16(ring + ((w0 + o / 2) & (kRing - 1)), reinterpret_cast<const uint8_t *>(words) + (n ? b : 0), n);
      }
      if ((w0 & (kRing - 1)) == 0 && 16 * i < 2 * kMirror) {  // the mirror of ring[0, kMirror)
        const uint32_t b = 2 * w0 + 16 * i;
        const uint32_t n = b < wbytes ? min(16u, wbytes - b) : 0u;
        cp_async16(ring + kRing + 8 * i, reinterpret_cast<const uint8_t *>(words) + (n ? b : 0), n);
      }
      cp_async_commit();
    };
    __syncwarp();  // the previous stream's reads of this ring are done
    load_half(0);
    load_half(kHalf);
    // the ring holds words [rbase, rbase + kRing); words below lim (<= nw)
    // are known to have landed
    uint32_t rbase = 0, lim = 0, p = 0, nesc = 0;
    const float4 s4 = *reinterpret_cast<const float4 *>(chunk + lo.sec_s + (uint64_t(si) * lo.d + i4) * 4);
    const float sc[4] = {s4.x, s4.y, s4.z, s4.w};
    const uint8_t *anc = chunk + lo.sec_anc + uint64_t(si) * ng * lo.d + i4;
    bool broken = false;

    // output row of the current token
    uint16_t *orow;
    bool row_ok = true, bad_row = false;
    [[maybe_unused]] uint16_t *pool = nullptr;
    [[maybe_unused]] int64_t lblk = 0, lblk_end = 0;
    [[maybe_unused]] int left = 0;
    [[maybe_unused]] int32_t bnext = 0;
    if constexpr (PAGED) {
      pool = po.pools[l * 2 + kvi];
      const int64_t t0 = int64_t(k) * lo.C;
      lblk = t0 / po.bt;
      lblk_end = (t0 + ntok - 1) / po.bt + 1;
      const int tib = int(t0 - lblk * po.bt);
      left = po.bt - tib;
      orow = paged_row(po, pool, po.table[lblk], tib, h, lo, int(i), row_ok);
      bad_row = !row_ok;
      if (lblk + 1 < lblk_end) bnext = po.table[lblk + 1];
    } else {
      orow = kv + (uint64_t(si) * lo.S + uint64_t(k) * lo.C) * lo.d + i4;
    }
    auto next_row = [&]() {
      if constexpr (PAGED) {
        if (--left == 0) {
          left = po.bt;
          if (++lblk < lblk_end) {
            orow = paged_row(po, pool, bnext, 0, h, lo, int(i), row_ok);
            bad_row |= !row_ok;
            if (lblk + 1 < lblk_end) bnext = po.table[lblk + 1];
          }
        } else {
          orow += lo.d;
        }
      } else {
        orow += lo.d;
      }
    };
    auto store_row = [&](float v0, float v1, float v2, float v3) {
      if (!PAGED || row_ok) *reinterpret_cast<uint2 *>(orow) = make_uint2(pack_f16x2(v0, v1), pack_f16x2(v2, v3));
    };

    uint32_t a4n = *reinterpret_cast<const uint32_t *>(anc);  // next group's anchors, loaded ahead
    for (int g = 0; g < ng && !broken; g++) {
      const uint32_t a4 = a4n;
      if (g + 1 < ng) a4n = *reinterpret_cast<const uint32_t *>(anc + uint64_t(g + 1) * lo.d);
      float ah[4];
#pragma unroll
      for (int j = 0; j < 4; j++) ah[j] = __fmul_rn(float(int8_t(a4 >> (8 * j))), sc[j]);
      store_row(ah[0], ah[1], ah[2], ah[3]);
      next_row();
      const int nt = min(lo.G, ntok - g * lo.G) - 1;  // delta tokens in this group
      for (int tt = 0; tt < nt; tt++) {
        // ---- symbol search in the main table
        uint32_t ff[4], rr[4], ro[4];
        bool sl[4];
#define CG_LOOKUP(J)                                                                   \
  {                                                                                    \
    const uint32_t xx = x[J];                                                          \
    uint32_t lu = lds16(smb, kMainOff + colb<J>() + ((xx & 0xFF00u) | i4));            \
    const uint32_t lf = lds16(smb, kFineOff + colb<J>() + (((xx << 4) & 0xFF00u) | i4)); \
    lu = lu >= 0xFF00u ? lf : lu;                                                      \
    const uint32_t t = (xx & 0xFFu) + lu;                                              \
    const uint32_t r = (t & 0xFF00u) | i4;                                    \
    const uint32_t c0 = lds16(smb, kCdfOff + colb<J>() + r);                  \
    const uint32_t c1 = lds16(smb, kCdfOff + 256 + colb<J>() + r);            \
    ff[J] = c1 - c0;                                                          \
    rr[J] = (xx - c0) & 0xFFFFu;                                              \
    ro[J] = t & 0xFF00u;                                                      \
    sl[J] = rr[J] >= ff[J];                                                   \
  }
// MID: the pair's first symbol sa from the u8 tables (the fine one at the
// 1024-slot tails; the main row of a tail slot falls on the fine table or
// the cdf rows, in bounds, and is not used), then cdf_sa, cdf_sa+1 and
// cdf_sa+2 pick sa or sa + 1.
#define CG_LOOKUP_MID(J)                                                               \
  {                                                                                    \
    const uint32_t xx = x[J];                                                          \
    const uint32_t slot = xx & 0xFFFFu;                                                \
    const uint32_t sm8 = smb[kMidMain - 4 * 128 + i4 + J + ((xx >> 1) & 0x7F80u)];     \
    const uint32_t sf8 = smb[kMidFine + i4 + J + ((xx << 2) & 0x1F80u)];               \
    const uint32_t sa = ((slot + 1024u) & 0xFFFFu) < 2048u ? sf8 : sm8;                \
    const uint32_t r = (sa << 8) | i4;                                                 \
    const uint32_t c0 = lds16(smb, kMidCdf + colb<J>() + r);                           \
    const uint32_t c1 = lds16(smb, kMidCdf + 256 + colb<J>() + r);                     \
    const uint32_t c2 = lds16(smb, kMidCdf + 512 + colb<J>() + r);                     \
    const bool up = slot >= c1;                                                        \
    const uint32_t clo = up ? c1 : c0;                                                 \
    ff[J] = (up ? c2 : c1) - clo;                                                      \
    rr[J] = slot - clo;                                                                \
    ro[J] = (sa + (up ? 1u : 0u)) << 8;                                                \
    sl[J] = rr[J] >= ff[J];                                                            \
  }
        if constexpr (MID) {
          CG_LOOKUP_MID(0)
          CG_LOOKUP_MID(1)
          CG_LOOKUP_MID(2)
          CG_LOOKUP_MID(3)
        } else {
          CG_LOOKUP(0)
          CG_LOOKUP(1)
          CG_LOOKUP(2)
          CG_LOOKUP(3)
        }
#undef CG_LOOKUP
#undef CG_LOOKUP_MID
        uint32_t escm = 0, cntw = 0;
        bool esc_warp = false;
        if (__any_sync(0xffffffffu, sl[0] | sl[1] | sl[2] | sl[3])) {
          if (sl[0]) slow128<0, cdf_off<MID>()>(smb, i4, x[0], ff[0], rr[0], ro[0], escm);
          if (sl[1]) slow128<1, cdf_off<MID>()>(smb, i4, x[1], ff[1], rr[1], ro[1], escm);
          if (sl[2]) slow128<2, cdf_off<MID>()>(smb, i4, x[2], ff[2], rr[2], ro[2], escm);
          if (sl[3]) slow128<3, cdf_off<MID>()>(smb, i4, x[3], ff[3], rr[3], ro[3], escm);
          cntw = 2 * __popc(escm);  // an escape's raw value takes two words
          esc_warp = __any_sync(0xffffffffu, escm != 0);
        }
        // ---- state update, word counts, word positions
        bool ndf[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
          x[j] = ff[j] * (x[j] >> 16) + rr[j];
          ndf[j] = x[j] < kRansL;
          cntw += ndf[j] ? 1u : 0u;
        }
        uint32_t incl = scan_step<1>(cntw);
        incl = scan_step<2>(incl);
        incl = scan_step<4>(incl);
        incl = scan_step<8>(incl);
        incl = scan_step<16>(incl);
        const uint32_t pn = p + __shfl_sync(0xffffffffu, incl, 31);
        uint32_t pos = p + incl - cntw;
        float v[4];
        // the thread's words are consecutive from pos: read four from the
        // ring (the mirror covers reads past its end; unneeded ones are
        // ignored) and give lane j word number nd_0 + .. + nd_(j-1)
        const auto ring_words = [&]() {
          const uint16_t *rp = ring + (pos & (kRing - 1));
          const uint32_t w0 = rp[0], w1 = rp[1], w2 = rp[2], w3 = rp[3];
          const uint32_t a1 = ndf[0] ? w1 : w0, a2 = ndf[0] ? w2 : w1, a3 = ndf[0] ? w3 : w2;
          const uint32_t b2 = ndf[1] ? a2 : a1, b3 = ndf[1] ? a3 : a2;
          const uint32_t wl[4] = {w0, a1, b2, ndf[2] ? b3 : b2};
#pragma unroll
          for (int j = 0; j < 4; j++) {
            if (ndf[j]) x[j] = __byte_perm(wl[j], x[j], 0x5410);  // x<<16 | w
            // q = symbol - 127 exactly: (2^15 + symbol) - (2^15 + 127)
            v[j] = __fmaf_rn(__int_as_float(ro[j] | 0x47000000u) - 32895.0f, step[j], ah[j]);
          }
        };
        if (pn > lim || esc_warp) {  // (warp-uniform)
          // ---- rare token: its words reach past those known to have
          // landed (or past the stream's end), or an escape's raw value is
          // among them
          if (pn > nw) {
            broken = true;
            break;
          }
          cp_async_wait_all();  // every word issued so far has landed
          __syncwarp();
          if (!esc_warp) {
            ring_words();
          } else {
            // escapes: the raw q follows the lane's renormalisation word;
            // read the words from the container itself
#pragma unroll
            for (int j = 0; j < 4; j++) {
              if (ndf[j]) x[j] = __byte_perm(uint32_t(words[pos++]), x[j], 0x5410);
              if ((escm >> j) & 1u) {
                const int q = int(uint32_t(words[pos]) | (uint32_t(words[pos + 1]) << 16));
                pos += 2;
                nesc++;
                v[j] = __fmaf_rn(__int2float_rn(q), step[j], ah[j]);
              } else {
                v[j] = __fmaf_rn(__int_as_float(ro[j] | 0x47000000u) - 32895.0f, step[j], ah[j]);
              }
            }
          }
          uint32_t nref = 0;
          if (pn > rbase + kHalf) {  // the first half is consumed: refill it with the next words
            __syncwarp();            // every thread's reads of it are done
            do {
              load_half(rbase + kRing);
              rbase += kHalf;
              nref++;
            } while (pn > rbase + kHalf);
          }
          // all but the refill just issued have landed; after two refills
          // (a token of more than kHalf words, possible only with many
          // escapes) the first of them has not, and the next token waits
          lim = min(nw, nref > 1 ? rbase : rbase + kHalf);
        } else {
          ring_words();
        }
        p = pn;
        store_row(v[0], v[1], v[2], v[3]);
        next_row();
      }
    }
    cp_async_wait_all();
    if (PAGED && bad_row) atomicOr(status, kStBadArg);
#pragma unroll
    for (int o = 16; o; o >>= 1) nesc += __shfl_xor_sync(0xffffffffu, nesc, o);
    const bool lanes_ok = x[0] == kRansL && x[1] == kRansL && x[2] == kRansL && x[3] == kRansL;
    if (broken || !lanes_ok || p != nw || nesc != ne) atomicOr(status, kStCorrupt);
  }
}

// ---------------------------------------------------------------- thin ranges
// The d = 128 decoder for chunk ranges that leave each (level, head) only a
// chunk or two (a streamed chunk group of a mixed-level container).  With a
// warp per stream such a CTA leaves its SM nearly idle, and a token costs
// the warp's whole dependency chain (some 200 instructions).  Here a stream
// is decoded by a team of four warps, one rANS lane per thread (lane 32 w + t
// on thread t of the team's warp w), and a CTA holds four teams, one chunk
// each.  Per token each warp finds its lanes' symbols and counts its words
// with a ballot (and one for escapes when a lane of the warp took the
// search); the four warp totals meet in shared memory behind one named
// barrier of the team.  The tables take 104 KB, so that two CTAs (eight
// streams, the most that the registers allow) share an SM:
//   fine [64][128] u8   : for 32-slot buckets over [0, 1024) (rows 0..31) and
//                         [64512, 65536) (rows 32..63), the distribution
//                         tails, the first symbol sa (at most 254) of the
//                         neighbouring pair holding most of the bucket;
//   main [248][128] u8  : the same for the 256-slot bucket (slot >> 8) - 4
//                         of the slots [1024, 64512);
//   cdf  [258][128] u16 : cdf_s of lane 32 w + t at row s (row 256 repeats
//                         cdf_255, row 257 is padding).
// A lane loads cdf_sa, cdf_sa+1 and cdf_sa+2 and takes sa or sa + 1; a slot
// outside the pair, or the escape (whose frequency then reads as 0), is
// resolved by a binary search of the lane's cdf column.  The rows are laid
// out so that lane 32 w + t (thread t of the team's warp w) only ever
// touches bank t, whatever rows its warp reads: its u8 entries are byte
// 4 t + w of a row, its cdf entries u16 position 2 t + 64 (w >> 1) + (w & 1)
// (byte 4 t + 128 (w >> 1) + 2 (w & 1)).  Words are staged per team in a ring of two
// halves that the team's first warp refills; a token whose words reach past
// those known to have landed waits for them, behind one more barrier.
constexpr int kThinTeams = 4;                                   // teams (streams) per CTA, 128 threads each
constexpr int kThinPerLevel = 4;                                // thin launches: levels of at most this many chunks
constexpr int kMidPerLevel = 8;                                 // MID launches (k_dec128 with u8 tables): at most this
constexpr uint32_t kThinTail = 1024;                            // slots with fine buckets, at each end
constexpr uint32_t kThinMainRows = (kM - 2 * kThinTail) / 256;  // 248
constexpr uint32_t kThinFineRows = 2 * kThinTail / 32;          // 64
constexpr uint32_t kThinFine = 0;
constexpr uint32_t kThinMain = kThinFine + kThinFineRows * 128;
constexpr uint32_t kThinCdf = kThinMain + kThinMainRows * 128;
constexpr uint32_t kThinRing = kThinCdf + kCdfRows * 256;  // rings [teams][kRing] u16, then word counts [teams][2][4] u32
__host__ __device__ constexpr uint32_t thin_smem(int teams) { return kThinRing + uint32_t(teams) * (kRing * 2 + 32); }
static_assert(thin_smem(kThinTeams) + 64 + 1024 <= 233472 / 2, "two thin CTAs must share an SM");
static_assert(kMidRing + kMidTeams * kRingStride * 2 + 64 + 1024 <= 233472 / 2, "two MID CTAs must share an SM");

// The thin tables' column of lane 32 w + t: u16 position p = 2 t + 64 (w >> 1)
// + (w & 1) of a cdf row, and the lane and u8 byte of position p.
__device__ __forceinline__ int thin_lane(int p) { return 32 * (((p >> 6) << 1) | (p & 1)) + ((p >> 1) & 31); }
__device__ __forceinline__ uint32_t thin_byte(uint32_t p) { return 4 * ((p >> 1) & 31) + (((p >> 6) << 1) | (p & 1)); }

// First symbols of the densest neighbouring pairs, as u8 (at most 254), for
// nb buckets of `width` slots from slot `base`, at each lane's byte of a
// 128-byte row.
__device__ __forceinline__ void build_sa8(uint8_t *lut, const uint16_t *cdfr, int nb, uint32_t width,
                                          uint32_t base) {
  build_buckets(cdfr, nb, width, base, [&](uint32_t b, uint32_t p, uint32_t sa, uint32_t, uint32_t) {
    lut[b * 128 + thin_byte(p)] = uint8_t(min(sa, 254u));
  });
}

__device__ __forceinline__ void team_bar(uint32_t id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

template <bool PAGED>
__global__ void __launch_bounds__(kThinTeams * 128, 2)
k_thin128(Layout lo, const uint8_t *__restrict__ tables, const uint8_t *__restrict__ buf,
          uint16_t *__restrict__ kv, uint8_t *ws, PagedOut po, int si_lo, int si_hi, int cmin, int cmax) {
  extern __shared__ __align__(16) uint8_t smb[];
  __shared__ int s_bad;
  __shared__ uint32_t s_nesc[kThinTeams];
  uint16_t *cdfr = reinterpret_cast<uint16_t *>(smb + kThinCdf);
  const int nteams = int(blockDim.x >> 7);

  const int lv = blockIdx.x, si = blockIdx.y;
  if (si < si_lo || si >= si_hi) return;  // outside the requested layers
  const int cnt = reinterpret_cast<const int32_t *>(ws + 64)[lv];
  const int first = int(blockIdx.z) * nteams;  // this CTA's entries of the level's chunk list
  if (cnt < cmin || cnt > cmax || first >= cnt) return;  // (cmin, cmax: as for k_dec128)
  const int32_t *list = reinterpret_cast<const int32_t *>(ws + 256) + lv * lo.n_chunks;
  uint32_t *status = reinterpret_cast<uint32_t *>(ws);
  const int h = si % lo.H, kvi = (si / lo.H) % 2, l = si / (2 * lo.H);

  if (threadIdx.x < kThinTeams) s_nesc[threadIdx.x] = 0;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const uint16_t *cdf = reinterpret_cast<const uint16_t *>(tables + lo.tb_cdf) +
                        tab_index(lo, lv, l, kvi, h * lo.d) * 256;
  build_cdf_rows<128>(cdf, cdfr, &s_bad, [](int p) { return thin_lane(p); });
  __syncthreads();
  build_sa8(smb + kThinMain, cdfr, kThinMainRows, 256, kThinTail);
  build_sa8(smb + kThinFine, cdfr, kThinFineRows / 2, 32, 0);
  build_sa8(smb + kThinFine + (kThinFineRows / 2) * 128, cdfr, kThinFineRows / 2, 32, kM - kThinTail);
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) atomicOr(status, kStCorrupt);
    return;
  }

  // From here on the teams are independent: each syncs on its own barrier.
  const int team = threadIdx.x >> 7;
  const int idx = first + team;
  if (idx >= cnt) return;  // a team without a chunk
  const uint32_t ell = threadIdx.x & 127, wt = ell >> 5, lane = ell & 31, bar_id = 1 + team;
  uint32_t ltm;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(ltm));
  // the earlier warps' word counts, as masks on the exchanged counts
  const uint32_t m1 = wt > 0 ? 0xFFFFu : 0u, m2 = wt > 1 ? 0xFFFFu : 0u, m3 = wt > 2 ? 0xFFFFu : 0u;
  const float stp = reinterpret_cast<const float *>(tables + lo.tb_step)[tab_index(lo, lv, l, kvi, h * lo.d + ell)];
  uint16_t *ring = reinterpret_cast<uint16_t *>(smb + kThinRing) + team * kRing;
  uint32_t *xch = reinterpret_cast<uint32_t *>(smb + kThinRing + nteams * kRing * 2) + team * 8;
  // byte offsets of this lane's column in the main table (row 0 = the bucket
  // of slot 0; rows below 8 and above 247 fall on the neighbouring tables
  // and are never used), the fine table and the cdf rows: bank `lane`
  const uint32_t mcol = kThinMain - (kThinTail / 256) * 128 + 4 * lane + wt, fcol = kThinFine + 4 * lane + wt,
                 ccol = kThinCdf + 4 * lane + 128 * (wt >> 1) + 2 * (wt & 1);

  const int k = list[idx];
  const int ng = chunk_ng(lo, k), ntok = chunk_ntok(lo, k), nd = chunk_nd(lo, k);
  const uint64_t base = ld_u64(buf + 64 + 8 * uint64_t(k));
  const uint64_t cend = (k + 1 < lo.n_chunks) ? ld_u64(buf + 64 + 8 * uint64_t(k + 1)) : ld_u64(buf + 48);
  const uint8_t *chunk = buf + base;
  const uint32_t *soffv = reinterpret_cast<const uint32_t *>(chunk + chunk_sec_off(lo, k));
  const uint64_t so = soffv[si];
  const uint64_t se = (si + 1 < lo.nstr) ? uint64_t(soffv[si + 1]) : (cend - base);
  bool ok = !(so & 15) && so >= chunk_fixed(lo, k) && se >= so && base + se <= cend &&
            se - so >= 16 + 4 * uint64_t(lo.d);
  const uint8_t *blk = chunk + so;
  uint32_t nw = 0, ne = 0;
  if (ok) {
    const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
    nw = hdr.x;
    ne = hdr.y;
    ok = hdr.z == uint32_t(nd) && hdr.w == 0 && 16 + 4 * uint64_t(lo.d) + 2 * uint64_t(nw) <= se - so;
  }
  if (!ok) {  // (the same for every thread of the team)
    if (ell == 0) atomicOr(status, kStCorrupt);
    return;
  }
  uint32_t x = reinterpret_cast<const uint32_t *>(blk + 16)[ell];
  const uint16_t *__restrict__ words = reinterpret_cast<const uint16_t *>(blk + 16 + 4 * lo.d);
  const uint32_t wbytes = 2 * nw;
  auto load_half = [&](uint32_t w0) {  // (first warp) words [w0, w0 + kHalf) -> ring half, zero past the end
    const uint32_t b = 2 * w0 + 16 * lane;
    const uint32_t n = b < wbytes ? min(16u, wbytes - b) : 0u;
    cp_async16(ring + ((w0 + 8 * lane) & (kRing - 1)), reinterpret_cast<const uint8_t *>(words) + (n ? b : 0), n);
    cp_async_commit();
  };
  if (wt == 0) {
    load_half(0);
    load_half(kHalf);
  }
  // the ring holds words [rbase, rbase + kRing); words below lim (<= nw)
  // are known to have landed.  All of these are the same across the team.
  uint32_t rbase = 0, lim = 0, p = 0, par = 0, nesc = 0;
  const float sc = reinterpret_cast<const float *>(chunk + lo.sec_s)[uint64_t(si) * lo.d + ell];
  const int8_t *anc = reinterpret_cast<const int8_t *>(chunk + lo.sec_anc) + uint64_t(si) * ng * lo.d + ell;
  bool broken = false;

  // output row of the current token (this thread's lane in it)
  uint16_t *orow;
  bool row_ok = true, bad_row = false;
  [[maybe_unused]] uint16_t *pool = nullptr;
  [[maybe_unused]] int64_t lblk = 0, lblk_end = 0;
  [[maybe_unused]] int left = 0;
  [[maybe_unused]] int32_t bnext = 0;
  if constexpr (PAGED) {
    pool = po.pools[l * 2 + kvi];
    const int64_t t0 = int64_t(k) * lo.C;
    lblk = t0 / po.bt;
    lblk_end = (t0 + ntok - 1) / po.bt + 1;
    const int tib = int(t0 - lblk * po.bt);
    left = po.bt - tib;
    orow = paged_row(po, pool, po.table[lblk], tib, h, lo, 0, row_ok) + ell;
    bad_row = !row_ok;
    if (lblk + 1 < lblk_end) bnext = po.table[lblk + 1];
  } else {
    orow = kv + (uint64_t(si) * lo.S + uint64_t(k) * lo.C) * lo.d + ell;
  }
  auto next_row = [&]() {
    if constexpr (PAGED) {
      if (--left == 0) {
        left = po.bt;
        if (++lblk < lblk_end) {
          orow = paged_row(po, pool, bnext, 0, h, lo, 0, row_ok) + ell;
          bad_row |= !row_ok;
          if (lblk + 1 < lblk_end) bnext = po.table[lblk + 1];
        }
      } else {
        orow += lo.d;
      }
    } else {
      orow += lo.d;
    }
  };
  auto store = [&](float v) {
    if (!PAGED || row_ok) *orow = uint16_t(pack_f16x2(v, 0.0f) & 0xFFFFu);
  };

  int8_t an = anc[0];  // next group's anchor, loaded ahead
  for (int g = 0; g < ng && !broken; g++) {
    const float ah = __fmul_rn(float(an), sc);
    if (g + 1 < ng) an = anc[uint64_t(g + 1) * lo.d];
    store(ah);
    next_row();
    const int nt = min(lo.G, ntok - g * lo.G) - 1;  // delta tokens in this group
    for (int tt = 0; tt < nt; tt++) {
      // ---- symbol: the pair of the lane's bucket (fine at the tails)
      const uint32_t slot = x & 0xFFFFu;
      const uint32_t sm8 = smb[mcol + ((x >> 1) & 0x7F80u)];  // row slot >> 8
      const uint32_t sf8 = smb[fcol + ((x << 2) & 0x1F80u)];  // row (slot >> 5) & 63: both tails
      const uint32_t sa = ((slot + kThinTail) & 0xFFFFu) < 2 * kThinTail ? sf8 : sm8;
      const uint32_t cb = ccol + sa * 256;
      const uint32_t c0 = lds16(smb, cb), c1 = lds16(smb, cb + 256), c2 = lds16(smb, cb + 512);
      const bool up = slot >= c1;
      const uint32_t clo = up ? c1 : c0;
      uint32_t f = (up ? c2 : c1) - clo, rr = slot - clo, s = sa + (up ? 1u : 0u);
      uint32_t be = 0;  // lanes of the warp with an escape
      if (__any_sync(0xffffffffu, rr >= f)) {
        if (rr >= f) {  // outside the pair, or the escape: a binary search of the lane's column
          uint32_t t = 0;  // largest t with cdf_t <= slot (cdf_0 = 0)
#pragma unroll
          for (uint32_t st = 128; st; st >>= 1)
            if (lds16(smb, ccol + (t + st) * 256) <= slot) t += st;
          const uint32_t a0 = lds16(smb, ccol + t * 256);
          const uint32_t a1 = t < 255 ? lds16(smb, ccol + (t + 1) * 256) : kM;
          f = a1 - a0;
          rr = slot - a0;
          s = t;
        }
        be = __ballot_sync(0xffffffffu, s == uint32_t(kEsc));
      }
      x = f * (x >> 16) + rr;
      const bool ndw = x < kRansL;
      // ---- word positions: lane order within the warp, warp order within
      // the team; an escape's raw value takes two more words
      const uint32_t bn = __ballot_sync(0xffffffffu, ndw);
      xch[par * 4 + wt] = (__popc(bn) + 2 * __popc(be)) | (be ? 0x10000u : 0u);
      team_bar(bar_id);
      const uint4 xv = *reinterpret_cast<const uint4 *>(xch + par * 4);
      par ^= 1;
      const uint32_t sum = xv.x + xv.y + xv.z + xv.w;
      const uint32_t pn = p + (sum & 0xFFFFu);
      const uint32_t pos = p + (xv.x & m1) + (xv.y & m2) + (xv.z & m3) + __popc(bn & ltm) + 2 * __popc(be & ltm);
      float v;
      if (pn > lim || sum > 0xFFFFu) {  // (the same across the team)
        // ---- rare token: its words reach past those known to have landed
        // (or past the stream's end), or an escape's raw value is among them
        if (pn > nw) {
          broken = true;
          break;
        }
        if (wt == 0) cp_async_wait_all();  // every word issued so far has landed ...
        team_bar(bar_id);                  // ... and is visible to the team
        if (sum <= 0xFFFFu) {
          const uint32_t w = ring[pos & (kRing - 1)];
          if (ndw) x = __byte_perm(w, x, 0x5410);  // x<<16 | w
          v = __fmaf_rn(__int_as_float(0x4B400000 + int(s)) - 12583039.0f, stp, ah);
        } else {  // escapes: the raw q follows the lane's renormalisation word; read from the container
          const uint32_t q0 = pos + (ndw ? 1u : 0u);
          if (ndw) x = __byte_perm(uint32_t(words[pos]), x, 0x5410);
          if (s == uint32_t(kEsc)) {
            const int q = int(uint32_t(words[q0]) | (uint32_t(words[q0 + 1]) << 16));
            nesc++;
            v = __fmaf_rn(__int2float_rn(q), stp, ah);
          } else {
            v = __fmaf_rn(__int_as_float(0x4B400000 + int(s)) - 12583039.0f, stp, ah);
          }
        }
        uint32_t nref = 0;
        if (pn > rbase + kHalf) {  // the first half is consumed: refill it with the next words
          team_bar(bar_id);        // every lane's reads of it are done
          do {
            if (wt == 0) load_half(rbase + kRing);
            rbase += kHalf;
            nref++;
          } while (pn > rbase + kHalf);
        }
        // all but the refill just issued have landed (after two, the next token waits)
        lim = min(nw, nref > 1 ? rbase : rbase + kHalf);
      } else {
        const uint32_t w = ring[pos & (kRing - 1)];
        if (ndw) x = __byte_perm(w, x, 0x5410);  // x<<16 | w
        // q = s - 127 as an exact fp32: (1.5*2^23 + s) - (1.5*2^23 + 127)
        v = __fmaf_rn(__int_as_float(0x4B400000 + int(s)) - 12583039.0f, stp, ah);
      }
      p = pn;
      store(v);
      next_row();
    }
  }
  if (wt == 0) cp_async_wait_all();  // no copy may land after the CTA has gone
  if (PAGED && bad_row) atomicOr(status, kStBadArg);
#pragma unroll
  for (int o = 16; o; o >>= 1) nesc += __shfl_xor_sync(0xffffffffu, nesc, o);
  if (lane == 0 && nesc) atomicAdd(&s_nesc[team], nesc);
  team_bar(bar_id);
  if (x != kRansL || (ell == 0 && (broken || p != nw || s_nesc[team] != ne))) atomicOr(status, kStCorrupt);
}

template <int T, bool PAGED>
cudaError_t launch_decode_tpb(const Layout &lo, const uint8_t *tables, const uint8_t *buf, uint16_t *kv,
                              uint8_t *ws, int teams, cudaStream_t st, const PagedOut &po, int l0, int l1) {
  const size_t smem = size_t(kBuckets + kCdfRows) * lo.d * 2 + size_t(teams) * (kRing + kMirror) * 2;
  cudaError_t e = cudaFuncSetAttribute(k_decode<T, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(lo.n_levels, l1 * 2 * lo.H);  // CTAs below layer l0 return at once
  k_decode<T, PAGED>
      <<<grid, teams * T, smem, st>>>(lo, tables, buf, kv, ws, po, l0 * 2 * lo.H, l1 * 2 * lo.H);
  return cudaGetLastError();
}

// d = 128, full tables: k_dec128 with a warp per chunk of the CTA's level
// (at least 16 warps, so that the table build is spread wide; warps without
// a chunk only build).
template <bool PAGED>
cudaError_t launch_decode_128(const Layout &lo, const uint8_t *tables, const uint8_t *buf, uint16_t *kv,
                              uint8_t *ws, int chunks, cudaStream_t st, const PagedOut &po, int l0, int l1,
                              int cmin, int cmax) {
  const int teams = chunks > kTeams128Max ? kTeams128Max : (chunks < 16 ? 16 : chunks);
  const size_t smem = kRingOff + size_t(teams) * kRingStride * 2;
  cudaError_t e = cudaFuncSetAttribute(k_dec128<PAGED, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  // The last wave: when the CTAs past the last full wave of the GPU could be
  // doubled and still run side by side, their heads take two CTAs each, so
  // that the wave takes about half a CTA's time instead of a whole one.  (Each
  // level is counted as live; the CTAs of a level in another band return at
  // once, and the split then only shifts where the waves fall.)
  const int rows = l1 * 2 * lo.H, live = (l1 - l0) * 2 * lo.H * lo.n_levels;
  int split = 0, dev = 0, sms = 0, per_sm = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_dec128<PAGED, false>, teams * 32, smem);
  if (e != cudaSuccess) return e;
  const int wave = sms * per_sm, rest = wave > 0 ? live % wave : 0;
  if (rest > 0 && chunks >= 2) {
    const int r = min((rest + lo.n_levels - 1) / lo.n_levels, l1 - l0 > 0 ? (l1 - l0) * 2 * lo.H : 0);
    if (2 * r * lo.n_levels <= wave) split = r;
  }
  dim3 grid(lo.n_levels, rows + split);  // CTAs below layer l0 return at once
  k_dec128<PAGED, false><<<grid, teams * 32, smem, st>>>(lo, tables, buf, kv, ws, po, l0 * 2 * lo.H, l1 * 2 * lo.H,
                                                         cmin, cmax, rows - split);
  return cudaGetLastError();
}

// d = 128, ranges with a few chunks per level: k_dec128 with the u8 pair
// tables, a CTA per (level, head, eight of the level's chunks), two CTAs per
// SM; CTAs past the level's chunk count return at once.
template <bool PAGED>
cudaError_t launch_decode_mid(const Layout &lo, const uint8_t *tables, const uint8_t *buf, uint16_t *kv,
                              uint8_t *ws, int chunks, cudaStream_t st, const PagedOut &po, int l0, int l1,
                              int cmin, int cmax) {
  const size_t smem = kMidRing + size_t(kMidTeams) * kRingStride * 2;
  cudaError_t e = cudaFuncSetAttribute(k_dec128<PAGED, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e == cudaSuccess)  // all of the SM's unified memory as shared memory, so two CTAs fit
    e = cudaFuncSetAttribute(k_dec128<PAGED, true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             int(cudaSharedmemCarveoutMaxShared));
  if (e != cudaSuccess) return e;
  dim3 grid(lo.n_levels, l1 * 2 * lo.H, (min(chunks, cmax) + kMidTeams - 1) / kMidTeams);
  k_dec128<PAGED, true><<<grid, kMidTeams * 32, smem, st>>>(lo, tables, buf, kv, ws, po, l0 * 2 * lo.H,
                                                             l1 * 2 * lo.H, cmin, cmax, int(grid.y));
  return cudaGetLastError();
}

// Thin ranges: a CTA per (level, head, four of the level's chunks), two
// CTAs per SM; CTAs past the level's chunk count return at once.
template <bool PAGED>
cudaError_t launch_decode_thin(const Layout &lo, const uint8_t *tables, const uint8_t *buf, uint16_t *kv,
                               uint8_t *ws, int chunks, cudaStream_t st, const PagedOut &po, int l0, int l1,
                               int cmin, int cmax) {
  const int smem = int(thin_smem(kThinTeams));
  cudaError_t e = cudaFuncSetAttribute(k_thin128<PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)  // all of the SM's unified memory as shared memory, so two CTAs fit
    e = cudaFuncSetAttribute(k_thin128<PAGED>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             int(cudaSharedmemCarveoutMaxShared));
  if (e != cudaSuccess) return e;
  dim3 grid(lo.n_levels, l1 * 2 * lo.H, (min(chunks, cmax) + kThinTeams - 1) / kThinTeams);
  k_thin128<PAGED><<<grid, kThinTeams * 128, smem, st>>>(lo, tables, buf, kv, ws, po, l0 * 2 * lo.H,
                                                          l1 * 2 * lo.H, cmin, cmax);
  return cudaGetLastError();
}

// chunks: the chunks in the range.  d = 128: each level goes to the kernel
// measured best for the chunks it holds in the range (crossovers on the 70B
// and 128K workloads), which only the device knows (k_decode_index counts
// them): at most four, the thin-range kernel (four warps per stream, a short
// token); five to eight, k_dec128 with the u8 pair tables and eight warps
// per CTA, two CTAs per SM; more, k_dec128 with its full tables and a warp
// per chunk of the level.  One launch per band that the range can reach;
// a CTA whose level is in another band returns at once.  Other d: k_decode,
// a team per chunk of the CTA's level, and at least 512 threads so that the
// table build is spread wide (teams without a chunk only build).
template <int T, bool PAGED>
cudaError_t launch_decode_tp(const Layout &lo, const uint8_t *tables, const uint8_t *buf,
                             uint16_t *kv, uint8_t *ws, int chunks, cudaStream_t st, const PagedOut &po,
                             int l0, int l1) {
  if constexpr (T == 32) {
    cudaError_t e = cudaSuccess;
    if (chunks > kMidPerLevel)
      e = launch_decode_128<PAGED>(lo, tables, buf, kv, ws, chunks, st, po, l0, l1, kMidPerLevel + 1, chunks);
    if (e == cudaSuccess && chunks > kThinPerLevel)
      e = launch_decode_mid<PAGED>(lo, tables, buf, kv, ws, chunks, st, po, l0, l1, kThinPerLevel + 1, kMidPerLevel);
    if (e == cudaSuccess)
      e = launch_decode_thin<PAGED>(lo, tables, buf, kv, ws, chunks, st, po, l0, l1, 1, kThinPerLevel);
    return e;
  } else {
    constexpr int kTeamsMax = max_threads<T>() / T, kTeamsMin = (512 / T < kTeamsMax) ? 512 / T : kTeamsMax;
    const int teams = chunks > kTeamsMax ? kTeamsMax : (chunks < kTeamsMin ? kTeamsMin : chunks);
    return launch_decode_tpb<T, PAGED>(lo, tables, buf, kv, ws, teams, st, po, l0, l1);
  }
}

template <int T>
cudaError_t launch_decode_t(const Layout &lo, const uint8_t *tables, const uint8_t *buf,
                            uint16_t *kv, uint8_t *ws, int teams, cudaStream_t st, const PagedOut *po,
                            int l0, int l1) {
  if (po) return launch_decode_tp<T, true>(lo, tables, buf, kv, ws, teams, st, *po, l0, l1);
  return launch_decode_tp<T, false>(lo, tables, buf, kv, ws, teams, st, PagedOut{nullptr, nullptr, 1, 0}, l0, l1);
}

}  // namespace

cudaError_t launch_decode(const Layout &lo, const uint8_t *tables, const uint8_t *buf,
                          uint64_t bytes, int32_t k0, int32_t k1, uint16_t *kv, uint8_t *ws,
                          cudaStream_t st, const PagedOut *po, int32_t l0, int32_t l1) {
  k_decode_index<<<1, 32, 0, st>>>(lo, tables, buf, bytes, k0, k1, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int teams = k1 - k0;
  if (teams < 1) return cudaSuccess;
  switch (lo.d / kLpt) {
    case 2: return launch_decode_t<2>(lo, tables, buf, kv, ws, teams, st, po, l0, l1);
    case 4: return launch_decode_t<4>(lo, tables, buf, kv, ws, teams, st, po, l0, l1);
    case 8: return launch_decode_t<8>(lo, tables, buf, kv, ws, teams, st, po, l0, l1);
    case 16: return launch_decode_t<16>(lo, tables, buf, kv, ws, teams, st, po, l0, l1);
    case 32: return launch_decode_t<32>(lo, tables, buf, kv, ws, teams, st, po, l0, l1);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cg
