// cg_decode.cu -- the streaming decoder.
//
// CacheGen's receiver decodes the bitstream "in real time, synchronized
// with transmission" (gptget summary of arXiv 2310.07240, Methodology; Guide
// to CacheGen, pillar 4) and rebuilds each token as anchor + delta (Guide,
// Step 2 decode_sequence; Step 1 dequantize).  Two kernels:
//
//   k_decode_index  one thread checks the container header against the
//                   caller's dims and the tables header, validates the
//                   chunk index and headers of [k0, k1) and lists the chunks
//                   of each level.
//   k_decode        one CTA per (level, head) holds that head's d frequency
//                   tables in shared memory, laid out so that thread i of a
//                   team only ever touches bank i (no bank conflicts however
//                   the symbols fall); each team of d/4 threads decodes one
//                   chunk's stream, 4 rANS lanes per thread.  Per token: a
//                   bucket lookup (slot >> 8) plus a forward check finds the
//                   symbol, a shuffle scan over the team orders the word
//                   reads, the fused dequantisation fma(q, step, a_hat) is
//                   clamped, converted to fp16 and stored 8 bytes per thread
//                   (a team writes one 256-byte token row).
//
// Every read of the container is bounded by the stream's own header, which
// is itself checked against the stream index; a stream whose lanes do not
// return to the initial state 2^16, or whose word/escape counts disagree,
// sets the CORRUPT bit.  Nothing waits on another CTA.
#include <cuda_fp16.h>

#include "cg_kernels.cuh"

namespace cg {
namespace {

constexpr int kLpt = kLanesPerThread;

__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint64_t ld_u64(const uint8_t *p) { return *reinterpret_cast<const uint64_t *>(p); }

__device__ __forceinline__ uint16_t ld_word(const uint16_t *p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

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

// ---------------------------------------------------------------- decode
// Shared memory per CTA (d lanes, T = d/4 threads per team):
//   etab [257][4][T] u32 : cdf_s | f_s << 16   (s = 256 is a zero sentinel)
//   lut  [256][T][4] u8  : first symbol whose range holds slot b*256
// Thread i of a team owns lanes 4i..4i+3; its entries sit at word index
// (row * T + i), so with T = 32 every access of thread i hits bank i.
template <int T>
__global__ void __launch_bounds__(kMaxTeams * T)
k_decode(Layout lo, const uint8_t *__restrict__ tables, const uint8_t *__restrict__ buf,
         uint16_t *__restrict__ kv, uint8_t *ws) {
  extern __shared__ __align__(16) uint32_t smem[];
  uint32_t *etab = smem;
  uint8_t *lut = reinterpret_cast<uint8_t *>(smem + 257 * kLpt * T);
  __shared__ int s_bad;

  const int lv = blockIdx.x, si = blockIdx.y;
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
  for (int e = threadIdx.x; e < lo.d * 256; e += blockDim.x) {
    const int c = e >> 8, s = e & 255;
    const uint32_t c0 = cdf[c * 256 + s];
    const uint32_t c1 = s < 255 ? cdf[c * 256 + s + 1] : kM;
    if (c1 <= c0 || (s == 0 && c0 != 0)) s_bad = 1;
    const int j = c % kLpt, ti = c / kLpt;
    etab[(s * kLpt + j) * T + ti] = c0 | ((c1 - c0) << 16);
    if (s == 0) etab[(256 * kLpt + j) * T + ti] = 0;
    for (uint32_t b = (c0 + 255) >> 8; b <= ((c1 - 1) >> 8) && c1 > c0; b++)
      lut[(b * T + ti) * kLpt + j] = uint8_t(s);
  }
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
  const uint32_t *et = etab + i;                 // + (s*4 + j) * T
  const uint8_t *lt = lut + i * kLpt;            // + b * T * 4 + j

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
    const uint16_t *words = reinterpret_cast<const uint16_t *>(blk + 16 + 4 * lo.d);
    const float4 s4 = *reinterpret_cast<const float4 *>(chunk + lo.sec_s + (uint64_t(si) * lo.d + kLpt * i) * 4);
    const float sc[4] = {s4.x, s4.y, s4.z, s4.w};
    const uint8_t *anc = chunk + lo.sec_anc + uint64_t(si) * ng * lo.d + kLpt * i;
    uint16_t *out = kv + (uint64_t(si) * lo.S + uint64_t(k) * lo.C) * lo.d + kLpt * i;
    uint32_t p = 0, nesc = 0;
    bool broken = false;

    for (int g = 0; g < ng && !broken; g++) {
      const uint32_t a4 = *reinterpret_cast<const uint32_t *>(anc + uint64_t(g) * lo.d);
      float ah[4];
#pragma unroll
      for (int j = 0; j < 4; j++) ah[j] = __fmul_rn(float(int8_t(a4 >> (8 * j))), sc[j]);
      {
        __half2 h01 = __floats2half2_rn(ah[0], ah[1]);
        __half2 h23 = __floats2half2_rn(ah[2], ah[3]);
        *reinterpret_cast<uint2 *>(out + uint64_t(g) * lo.G * lo.d) =
            make_uint2(*reinterpret_cast<uint32_t *>(&h01), *reinterpret_cast<uint32_t *>(&h23));
      }
      const int tend = min(g * lo.G + lo.G, ntok);
      for (int tr = g * lo.G + 1; tr < tend; tr++) {
        uint32_t sym[4], need[4];
        int cntw = 0;
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const uint32_t slot = x[j] & 0xFFFFu;
          uint32_t s = lt[(slot >> 8) * (T * kLpt) + j];
          uint32_t e = et[(s * kLpt + j) * T];
          const uint32_t e1 = et[((s + 1) * kLpt + j) * T];
          uint32_t r = slot - (e & 0xFFFFu);
          if (r >= (e >> 16)) {
            r -= e >> 16;
            s += 1;
            e = e1;
            while (r >= (e >> 16) && s < 255) {  // bucket holding 3+ symbols
              r -= e >> 16;
              s += 1;
              e = et[(s * kLpt + j) * T];
            }
          }
          x[j] = (e >> 16) * (x[j] >> 16) + r;
          sym[j] = s;
          need[j] = x[j] < kRansL ? 1u : 0u;
          cntw += int(need[j]) + (s == kEsc ? 2 : 0);
        }
        int incl = cntw;
#pragma unroll
        for (int o = 1; o < T; o <<= 1) {
          const int v = __shfl_up_sync(tm, incl, o, T);
          if (i >= o) incl += v;
        }
        const uint32_t tot = uint32_t(__shfl_sync(tm, incl, T - 1, T));
        if (p + tot > nw) {
          broken = true;
          break;
        }
        uint32_t pos = p + uint32_t(incl - cntw);
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
          if (need[j]) x[j] = (x[j] << 16) | ld_word(words + pos++);
          int q;
          if (sym[j] == kEsc) {
            q = int(uint32_t(ld_word(words + pos)) | (uint32_t(ld_word(words + pos + 1)) << 16));
            pos += 2;
            nesc++;
          } else {
            q = int(sym[j]) - 127;
          }
          float y = __fmaf_rn(__int2float_rn(q), step[j], ah[j]);
          v[j] = fminf(fmaxf(y, -65504.0f), 65504.0f);
        }
        p += tot;
        __half2 h01 = __floats2half2_rn(v[0], v[1]);
        __half2 h23 = __floats2half2_rn(v[2], v[3]);
        *reinterpret_cast<uint2 *>(out + uint64_t(tr) * lo.d) =
            make_uint2(*reinterpret_cast<uint32_t *>(&h01), *reinterpret_cast<uint32_t *>(&h23));
      }
    }
#pragma unroll
    for (int o = T / 2; o; o >>= 1) nesc += __shfl_xor_sync(tm, nesc, o, T);
    const bool lanes_ok = x[0] == kRansL && x[1] == kRansL && x[2] == kRansL && x[3] == kRansL;
    if (broken || !lanes_ok || p != nw || nesc != ne) atomicOr(status, kStCorrupt);
  }
}

template <int T>
cudaError_t launch_decode_t(const Layout &lo, const uint8_t *tables, const uint8_t *buf,
                            uint16_t *kv, uint8_t *ws, int teams, cudaStream_t st) {
  const size_t smem = size_t(257) * lo.d * 4 + size_t(256) * lo.d;
  cudaError_t e = cudaFuncSetAttribute(k_decode<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(lo.n_levels, lo.nstr);
  k_decode<T><<<grid, teams * T, smem, st>>>(lo, tables, buf, kv, ws);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const Layout &lo, const uint8_t *tables, const uint8_t *buf,
                          uint64_t bytes, int32_t k0, int32_t k1, uint16_t *kv, uint8_t *ws,
                          cudaStream_t st) {
  k_decode_index<<<1, 32, 0, st>>>(lo, tables, buf, bytes, k0, k1, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int teams = k1 - k0;
  if (teams > kMaxTeams) teams = kMaxTeams;
  if (teams < 1) return cudaSuccess;
  switch (lo.d / kLpt) {
    case 2: return launch_decode_t<2>(lo, tables, buf, kv, ws, teams, st);
    case 4: return launch_decode_t<4>(lo, tables, buf, kv, ws, teams, st);
    case 8: return launch_decode_t<8>(lo, tables, buf, kv, ws, teams, st);
    case 16: return launch_decode_t<16>(lo, tables, buf, kv, ws, teams, st);
    case 32: return launch_decode_t<32>(lo, tables, buf, kv, ws, teams, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cg
