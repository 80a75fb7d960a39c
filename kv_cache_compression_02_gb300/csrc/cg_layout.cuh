// cg_layout.cuh -- byte layout of the tables blob, the container and the
// workspaces, shared by the kernels and the host entry points of
// libcachegen.so.  The formats themselves are described in cachegen.h.
#pragma once

#include <cstdint>

namespace cg {

constexpr uint32_t kM = 1u << 16;      // total frequency of a table
constexpr uint32_t kRansL = 1u << 16;  // lower bound of the rANS state
constexpr int kEsc = 255;              // escape symbol
constexpr int kMaxLevels = 8;
constexpr int kLanesPerThread = 4;     // rANS lanes (channels) per thread
constexpr int kMaxTeams = 32;          // streams coded at once per CTA (T < 32)
// threads per CTA of the coding kernels for teams of T threads; 768 at
// T = 32 leaves 80 registers per thread
template <int T>
constexpr int max_threads() { return T == 32 ? 768 : kMaxTeams * T; }

// status bits in the first word of every workspace
constexpr uint32_t kStNonfinite = 1u;
constexpr uint32_t kStCapacity = 2u;
constexpr uint32_t kStCorrupt = 4u;
constexpr uint32_t kStTimeout = 8u;
constexpr uint32_t kStBadArg = 16u;    // an argument read on the device was invalid

__host__ __device__ inline uint64_t pad16(uint64_t v) { return (v + 15) & ~uint64_t(15); }
__host__ __device__ inline uint64_t pad256(uint64_t v) { return (v + 255) & ~uint64_t(255); }

struct Layout {
  int32_t L, H, d, C, G, R, n_levels;
  int32_t nstr;      // streams per chunk = L*2*H
  int32_t n_chunks;
  int32_t hd;        // H*d
  int64_t S;
  int32_t ntok_last, ng_full, ng_last, nd_full, nd_last;
  // tables blob
  uint64_t tb_step, tb_recip, tb_cdf, tb_bytes;
  // container
  uint64_t hdr_bytes;                 // header + chunk index, padded
  uint64_t sec_s, sec_anc;            // chunk-relative section offsets
  uint64_t sec_off_full, sec_off_last;
  uint64_t fixed_full, fixed_last;    // chunk fixed part sizes
};

__host__ __device__ inline int32_t chunk_ntok(const Layout &lo, int64_t k) {
  return k == lo.n_chunks - 1 ? lo.ntok_last : lo.C;
}
__host__ __device__ inline int32_t chunk_ng(const Layout &lo, int64_t k) {
  return k == lo.n_chunks - 1 ? lo.ng_last : lo.ng_full;
}
__host__ __device__ inline int32_t chunk_nd(const Layout &lo, int64_t k) {
  return k == lo.n_chunks - 1 ? lo.nd_last : lo.nd_full;
}
__host__ __device__ inline uint64_t chunk_fixed(const Layout &lo, int64_t k) {
  return k == lo.n_chunks - 1 ? lo.fixed_last : lo.fixed_full;
}
__host__ __device__ inline uint64_t chunk_sec_off(const Layout &lo, int64_t k) {
  return k == lo.n_chunks - 1 ? lo.sec_off_last : lo.sec_off_full;
}
// table index of (level, layer, kv, channel)
__host__ __device__ inline uint64_t tab_index(const Layout &lo, int lv, int l, int kv, int c) {
  return ((uint64_t(lv) * lo.L + l) * 2 + kv) * uint64_t(lo.hd) + c;
}

inline bool make_layout(Layout &lo, int32_t L, int32_t H, int32_t d, int32_t C, int32_t G,
                        int64_t S, int32_t R, int32_t n_levels) {
  if (L < 1 || H < 1 || d < 8 || d > 128 || (d % 8) != 0 || C < 1 || G < 1 || S < 1 ||
      S > (int64_t(1) << 22) || R < 0 || R > 127 || n_levels < 1 || n_levels > kMaxLevels)
    return false;
  lo.L = L; lo.H = H; lo.d = d; lo.C = C; lo.G = G; lo.S = S; lo.R = R; lo.n_levels = n_levels;
  lo.hd = H * d;
  lo.nstr = L * 2 * H;
  int64_t nk = (S + C - 1) / C;
  if (nk > (1 << 24)) return false;
  lo.n_chunks = int32_t(nk);
  lo.ntok_last = int32_t(S - (nk - 1) * int64_t(C));
  int32_t ntok_full = nk > 1 ? C : lo.ntok_last;
  lo.ng_full = (ntok_full + G - 1) / G;
  lo.ng_last = (lo.ntok_last + G - 1) / G;
  lo.nd_full = ntok_full - lo.ng_full;
  lo.nd_last = lo.ntok_last - lo.ng_last;
  uint64_t nc = uint64_t(n_levels) * L * 2 * lo.hd;
  lo.tb_step = 64;
  lo.tb_recip = lo.tb_step + pad16(4 * nc);
  lo.tb_cdf = lo.tb_recip + pad16(4 * nc);
  lo.tb_bytes = lo.tb_cdf + 512 * nc;
  lo.hdr_bytes = pad16(64 + 8 * uint64_t(nk));
  lo.sec_s = 16;
  lo.sec_anc = 16 + pad16(4 * uint64_t(lo.nstr) * d);
  lo.sec_off_full = lo.sec_anc + pad16(uint64_t(lo.nstr) * lo.ng_full * d);
  lo.sec_off_last = lo.sec_anc + pad16(uint64_t(lo.nstr) * lo.ng_last * d);
  lo.fixed_full = lo.sec_off_full + pad16(4 * uint64_t(lo.nstr));
  lo.fixed_last = lo.sec_off_last + pad16(4 * uint64_t(lo.nstr));
  // worst-case chunk (every symbol an escape with a renorm word) must keep
  // stream offsets within u32
  uint64_t worst = lo.fixed_full + uint64_t(lo.nstr) * pad16(16 + 4 * uint64_t(d) +
                                                              6 * uint64_t(lo.nd_full) * d);
  if (worst >= (uint64_t(1) << 32)) return false;
  return true;
}

// Word slots a stream may use per delta symbol.  With the full alphabet
// (R = 127) escapes are rare and a stream that needs more than one 16-bit
// word per symbol expands its raw fp16 size, which the encoder rejects;
// with a smaller alphabet most symbols may escape (3 words each).
__host__ __device__ inline uint64_t words_per_symbol(const Layout &lo) { return lo.R < 127 ? 3 : 1; }

// ---- workspaces ----------------------------------------------------------
// Every workspace starts with a 256-byte status block.
// Histogram pairs: (level, head) pairs of the histogram pass's last wave
// that two CTAs share, at most this many.
constexpr int kHistPairsMax = 96;
struct FitWs {
  uint64_t status, mult, scale, ent_bits, ent_esc, moments, done, pair_hist, pair_done, bytes;  // offsets
};
inline FitWs fit_ws(const Layout &lo) {
  FitWs w;
  const uint64_t nc = uint64_t(lo.n_levels) * lo.L * 2 * lo.hd;  // tables
  w.status = 0;
  w.mult = 256;                                                   // f32 [L][2]
  w.scale = pad256(w.mult + 8 * uint64_t(lo.L));                  // f32x2 [nk][nstr*d]
  w.ent_bits = pad256(w.scale + 8 * uint64_t(lo.n_chunks) * lo.nstr * lo.d);  // f64 [tables]
  w.ent_esc = pad256(w.ent_bits + 8 * nc);                        // u32 [tables]
  w.moments = pad256(w.ent_esc + 4 * nc);                         // u64 [nstr][d][4]: sum X, sum X^2 (lo, hi)
  w.done = pad256(w.moments + 32 * uint64_t(lo.nstr) * lo.d);     // u32 [nstr]: parts of a head summed
  w.pair_hist = pad256(w.done + 4 * uint64_t(lo.nstr));           // u32 [kHistPairsMax][d][257]
  w.pair_done = pad256(w.pair_hist + 4 * uint64_t(kHistPairsMax) * lo.d * 257);  // u32 [kHistPairsMax]
  w.bytes = pad256(w.pair_done + 4 * uint64_t(kHistPairsMax));
  return w;
}

struct EncWs {
  uint64_t status, levels, chunks, info, states, soff, coff, words, bytes;
  uint64_t words_cap;  // u16 slots per stream
};
inline EncWs enc_ws(const Layout &lo) {
  EncWs w;
  const uint64_t ns = uint64_t(lo.n_chunks) * lo.nstr;
  w.status = 0;
  // i32 count[8], i32 list[8][nk], u8 level[nk]
  w.levels = 256;
  w.chunks = pad256(w.levels + 4 * uint64_t(kMaxLevels) * (1 + uint64_t(lo.n_chunks)) +
                    uint64_t(lo.n_chunks));                         // fixed part per chunk
  w.info = pad256(w.chunks + uint64_t(lo.n_chunks) * lo.fixed_full);  // u32x2 [ns]
  w.states = pad256(w.info + 8 * ns);                              // u32 [ns][d]
  w.soff = pad256(w.states + 4 * ns * lo.d);                       // u32 [ns]
  w.coff = pad256(w.soff + 4 * ns);                                // u64 [nk] + total
  w.words_cap = uint64_t(lo.nd_full) * lo.d * words_per_symbol(lo);
  w.words = pad256(w.coff + 8 * (uint64_t(lo.n_chunks) + 1));      // u16 [ns][cap]
  w.bytes = pad256(w.words + 2 * ns * w.words_cap + 32);  // 16-byte reads may run 32 bytes past the last slot
  return w;
}

struct DecWs {
  uint64_t status, count, list, bytes;
};
inline DecWs dec_ws(const Layout &lo) {
  DecWs w;
  w.status = 0;
  w.count = 64;                                                    // i32 [8]
  w.list = 256;                                                    // i32 [8][nk]
  w.bytes = pad256(w.list + 4 * uint64_t(kMaxLevels) * lo.n_chunks);
  return w;
}

}  // namespace cg
