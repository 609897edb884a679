// Verify attention over the k8v4 paged cache: n_q (2..8) queries per sequence,
// each with its own visible length (the per-query step arrays of the hybrid-KV
// pull request's "Tests" section), split-K over the cells with the same
// partial/combine scheme as decode.
//
// GB300 design.  The n_q queries of a sequence read the same cells, so each
// 32-cell tile is dequantised ONCE per CTA into shared memory and then read by
// every query warp with ldmatrix:
//   * producer warps convert: K codes -> fp16 (exact), and V nibbles -> the
//     two fp16 terms of c * d (|c| <= 8 has 3 significant bits and d 11, so
//     the product has at most 14 bits and hi + lo = c * d exactly);
//   * warp i < n_q then runs query i over the tile on warp-level tensor-core
//     MMAs: S = K q (two accumulators per 128-lane half, K scales applied
//     after the MMA), online softmax in the log2 domain, and O += (c d) p with
//     p split into two fp16 terms.
// Warps n_q..7 are producers: while the query warps run tile t they copy and
// dequantise tile t + 1 into the other buffer (with n_q = 8 every warp does both).
// Scaling: a cell whose largest V scale reaches 4096 would push c * d past the
// fp16 range, so its d is halved e times (e <= 4, exact unless d is tiny) and
// its p is doubled e times; p carries 2^10 throughout, so the MMA accumulates
// o = 2^10 sum p c d.  One barrier per tile: the converted tiles are double
// buffered, and each producer thread dequantises exactly the bytes its own
// cp.async copies brought in (so the copy wait needs no barrier).
#include <algorithm>

#include "k8v4_common.cuh"

namespace k8v4 {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 256;       // 8 warps: warps < n_q run a query each, the rest convert
constexpr int kTile = 32;           // cells per iteration (two 16-cell MMA sub-tiles)
constexpr int kRawStages = 3;
constexpr int kPStride = 260;       // floats per partial row: o[256], m, l, 2 pad

struct Raw {                        // one tile as copied from the cache (K8V4 format, head g)
  static constexpr int kK = 0;                           // [32][256] int8 codes
  static constexpr int kV = kK + kTile * 256;            // [32][8 blocks][16] nibbles
  static constexpr int kKs = kV + kTile * 128;           // [32][2] f32 K scales
  static constexpr int kVs = kKs + kTile * 8;            // [32][8 threads] 4 B: the fp16 pair holding d
  static constexpr int kBytes = kVs + kTile * 8 * 4;
};
struct Conv {                       // one tile dequantised; rows of 512 B, 16-B chunks swizzled
  static constexpr int kK = 0;                           // [32][256] fp16 K codes
  static constexpr int kV = kK + kTile * 512;            // [2 terms][32][256] fp16 c * d (hi, lo)
  static constexpr int kPs = kV + 2 * kTile * 512;       // [32] f32: 2^(10 + e) per cell
  static constexpr int kKs = kPs + kTile * 4;            // [32][2] f32 K scales
  static constexpr int kBytes = kKs + kTile * 8;
};
constexpr int kSmem = kRawStages * Raw::kBytes + 2 * Conv::kBytes;

// chunk position inside a 512-B row: XOR with the row's low bits spreads the
// eight rows an ldmatrix phase reads; XOR with chunk bits 3..4 spreads the
// eight chunks a quarter-warp of converters writes into one row
__device__ __forceinline__ int sw(int row, int chunk) { return chunk ^ (row & 7) ^ ((chunk >> 3) & 3); }

struct VerifyParams {
  CacheView C;
  const void* q;
  const int32_t* pt;
  int64_t max_pages;
  const int32_t* steps;
  int n_seqs, n_q, max_seq_len, cells_per_split, splits;
  float sm_scale_log2;
  float* ws;
  int* status;
};

__device__ __forceinline__ void mma_f16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<const __half2*>(&u); }

// four int8 codes -> fp16x2 {c0, c1}, {c2, c3}, exact: 0x64XX is 1024 + XX
__device__ __forceinline__ void codes_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;            // c + 128
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  lo = h2u(__hsub2(u2h(prmt(u, 0x64646464u, 0x4140u)), bias));
  hi = h2u(__hsub2(u2h(prmt(u, 0x64646464u, 0x4342u)), bias));
}
// the low nibbles of bytes 0 and 2 of r -> fp16x2 (n - 8); the high nibbles -> (n - 8); exact
__device__ __forceinline__ __half2 nib_lo(uint32_t r) {
  const uint32_t x = (r & 0x000f000fu) | 0x64006400u;                          // 1024 + n
  return __hsub2(u2h(x), __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408)));
}
__device__ __forceinline__ __half2 nib_hi(uint32_t r) {
  const uint32_t x = (r & 0x00f000f0u) | 0x64006400u;                          // 1024 + 16 n
  // (1024 + 16 n) / 16 - 72 = n - 8: one exact fused multiply-add
  return __hfma2(u2h(x), __halves2half2(__ushort_as_half(0x2c00), __ushort_as_half(0x2c00)),
                 __halves2half2(__ushort_as_half(0xd480), __ushort_as_half(0xd480)));
}
// c (fp16x2) times d -> the two fp16 terms of the exact product
__device__ __forceinline__ void split_prod(__half2 c, __half2 d, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __hmul2(c, d);
  hi = h2u(h);
  lo = h2u(__hfma2(c, d, __hneg2(h)));
}

template <bool QF32>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(const VerifyParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int r0 = lane >> 2, c = lane & 3;
  const CacheView& C = p.C;
  const int HQ = C.H * kGqa;
  const int nq = p.n_q;
  const bool qw = warp < nq;                   // this warp runs query `warp`

  // ---- visible counts (device values, clipped to the host bound)
  int n_max = 0, n_vis = 0;
  for (int i = 0; i < nq; ++i) {
    int v = p.steps[static_cast<int64_t>(b) * nq + i];
    if (v < 0 || v > p.max_seq_len) {
      if (tid == 0 && split == 0 && g == 0) record_status(p.status, K8V4_ERANGE);
      v = v < 0 ? 0 : p.max_seq_len;
    }
    n_max = max(n_max, v);
    if (i == warp) n_vis = v;
  }
  const int c_begin = split * p.cells_per_split;
  const int c_stop = c_begin + p.cells_per_split;
  const int c_end = min(c_stop, n_max);
  const int n_it = c_end > c_begin ? (c_end - c_begin + kTile - 1) / kTile : 0;
  const int lim = min(n_vis, c_stop);          // this query's cells in this split end here

  // ---- q fragments (B operand of S = K q): lane holds head r0, dims
  // 16 ks + 2c + {0, 1} (register 0) and 16 ks + 8 + 2c + {0, 1} (register 1)
  uint32_t qf[16][2];
  uint32_t qf_lo[QF32 ? 16 : 1][2];
  float f0 = 0.0f, f1 = 0.0f;
  if (qw) {
    const int64_t qrow = ((static_cast<int64_t>(b) * nq + warp) * HQ + g * kGqa + r0) * kD;
    float qv[16][4];
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      const int64_t e0 = qrow + 16 * ks + 2 * c;
      if (QF32) {
        const float2 a = *reinterpret_cast<const float2*>(static_cast<const float*>(p.q) + e0);
        const float2 bb = *reinterpret_cast<const float2*>(static_cast<const float*>(p.q) + e0 + 8);
        qv[ks][0] = a.x; qv[ks][1] = a.y; qv[ks][2] = bb.x; qv[ks][3] = bb.y;
      } else {
        const uint32_t a = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.q) + e0);
        const uint32_t bb = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.q) + e0 + 8);
        qv[ks][0] = __uint_as_float(a << 16); qv[ks][1] = __uint_as_float(a & 0xffff0000u);
        qv[ks][2] = __uint_as_float(bb << 16); qv[ks][3] = __uint_as_float(bb & 0xffff0000u);
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int ks = 0; ks < 16; ++ks)
#pragma unroll
      for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qv[ks][e]));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    int ex = amax > 0.0f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127 : 0;
    int sh = 14 - ex;                               // amax * 2^sh in [2^14, 2^15)
    sh = max(-100, min(100, sh));
    const float up = ldexpf(1.0f, sh);
    const float fscale = p.sm_scale_log2 * ldexpf(1.0f, -sh);   // per head: sm_scale * log2(e) / 2^sh
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = __fmul_rn(qv[ks][e], up);
      const __half2 h0 = __floats2half2_rn(v[0], v[1]), h1 = __floats2half2_rn(v[2], v[3]);
      qf[ks][0] = h2u(h0);
      qf[ks][1] = h2u(h1);
      if (QF32) {
        const float2 a = __half22float2(h0), bb = __half22float2(h1);
        qf_lo[ks % (QF32 ? 16 : 1)][0] = h2u(__floats2half2_rn(v[0] - a.x, v[1] - a.y));
        qf_lo[ks % (QF32 ? 16 : 1)][1] = h2u(__floats2half2_rn(v[2] - bb.x, v[3] - bb.y));
      }
    }
    // score factors for the heads of the C layout (2c, 2c+1): held by lanes 4h
    f0 = __shfl_sync(kFull, fscale, 8 * c);
    f1 = __shfl_sync(kFull, fscale, 8 * c + 4);
  }

  float o[16][4];
#pragma unroll
  for (int mt = 0; mt < 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;

  // ---- producers: task i (0..255) of a tile is cell i / 8, K chunks i % 8 and
  // i % 8 + 8 (dims 16 kp .. and 128 + 16 kp ..) and V block i % 8; a producer
  // thread copies and dequantises tasks ptid, ptid + NP, ... of every tile
  const bool prod = nq == kThreads / 32 || warp >= nq;
  const int NP = nq == kThreads / 32 ? kThreads : kThreads - 32 * nq;     // producer threads (multiple of 32)
  const int ptid = nq == kThreads / 32 ? tid : tid - 32 * nq;
  const uint32_t raw_s = smem_u32(smem);
  const uint32_t conv_s = raw_s + kRawStages * Raw::kBytes;
  const int32_t* pt_row = p.pt + static_cast<int64_t>(b) * p.max_pages;
  const int H = C.H;
  // page ids of the two sub-tiles of the next tile to copy (read one tile ahead)
  auto page_of = [&](int t, int u) -> int64_t {
    const int cell = c_begin + kTile * t + 16 * u;
    const int lp = cell / C.P;
    return (cell < c_end && lp < p.max_pages) ? pt_row[lp] : -1;
  };
  int64_t nxt_pg0 = -1, nxt_pg1 = -1;
  if (prod && n_it > 0) { nxt_pg0 = page_of(0, 0); nxt_pg1 = page_of(0, 1); }
  auto issue = [&](int t) {
    const uint32_t s = raw_s + (t % kRawStages) * Raw::kBytes;
    for (int i = ptid; i < kTile * 8; i += NP) {
      const int jc = i >> 3, kp = i & 7, u = jc >> 4;
      const int cell = c_begin + kTile * t + jc;
      if (c_begin + kTile * t + 16 * u >= c_end) continue;            // sub-tile past every query's end
      const int64_t page = u ? nxt_pg1 : nxt_pg0;
      if (page < 0 || page >= C.n_pages) {
        record_status(p.status, K8V4_ERANGE);
        continue;
      }
      const uint8_t* base = C.pages + page * C.page_bytes;
      const int64_t row = static_cast<int64_t>(cell % C.P) * H + g;
      cp_async16(s + Raw::kK + jc * 256 + 16 * kp, base + row * 256 + 16 * kp);
      cp_async16(s + Raw::kK + jc * 256 + 16 * (kp + 8), base + row * 256 + 16 * (kp + 8));
      cp_async16(s + Raw::kV + jc * 128 + 16 * kp, base + C.v_off() + row * 128 + 16 * kp);
      cp_async4(s + Raw::kVs + (jc * 8 + kp) * 4, base + C.vs_off() + row * 16 + 4 * (kp >> 1));
      if (kp == 0) cp_async8(s + Raw::kKs + jc * 8, base + C.ks_off() + row * 8);
    }
    if (t + 1 < n_it) { nxt_pg0 = page_of(t + 1, 0); nxt_pg1 = page_of(t + 1, 1); }
  };
  // dequantise this thread's tasks of tile t (copies complete) into conv[t & 1]
  auto convert = [&](int t) {
    const uint32_t rs = raw_s + (t % kRawStages) * Raw::kBytes;
    const uint32_t cs = conv_s + (t & 1) * Conv::kBytes;
    const int tile0 = c_begin + kTile * t;
    for (int i = ptid; i < kTile * 8; i += NP) {             // warp-uniform trip count (256 % NP == 0 mod 32)
      const int jc = i >> 3, kp = i & 7;
      const bool live = tile0 + jc < c_end;                 // cells past every query's end are zeroed
      const uint32_t krow = cs + Conv::kK + jc * 512;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kc = kp + 8 * h;                          // raw chunk: dims 16 kc .. 16 kc + 15
        uint4 lo4 = make_uint4(0, 0, 0, 0), hi4 = make_uint4(0, 0, 0, 0);
        if (live) {
          const uint4 w = lds128(rs + Raw::kK + jc * 256 + 16 * kc);
          codes_to_f16(w.x, lo4.x, lo4.y);
          codes_to_f16(w.y, lo4.z, lo4.w);
          codes_to_f16(w.z, hi4.x, hi4.y);
          codes_to_f16(w.w, hi4.z, hi4.w);
        }
        sts128(krow + 16 * sw(jc, 2 * kc), lo4);
        sts128(krow + 16 * sw(jc, 2 * kc + 1), hi4);
      }
      if (kp == 0) {
        float2 k2 = make_float2(0.0f, 0.0f);
        if (live) k2 = *reinterpret_cast<const float2*>(smem + (rs - raw_s) + Raw::kKs + 8 * jc);
        *reinterpret_cast<float2*>(smem + (cs - raw_s) + Conv::kKs + 8 * jc) = k2;
      }
      // V block kp of cell jc: byte i holds dims 32 kp + i (low nibble) and
      // 32 kp + 16 + i (high nibble)
      const uint32_t dw = *reinterpret_cast<const uint32_t*>(smem + (rs - raw_s) + Raw::kVs + (jc * 8 + kp) * 4);
      const uint32_t dbits = live ? ((kp & 1) ? (dw >> 16) : (dw & 0xffffu)) : 0u;
      // e: halvings that keep 8 |d| below 2^15 for every block of the cell (the
      // cell's eight tasks sit in eight consecutive lanes)
      uint32_t mag = dbits & 0x7fffu;
      mag = max(mag, __shfl_xor_sync(kFull, mag, 1));
      mag = max(mag, __shfl_xor_sync(kFull, mag, 2));
      mag = max(mag, __shfl_xor_sync(kFull, mag, 4));
      const int e = max(0, static_cast<int>(mag >> 10) - 26);                    // |d| >= 4096 -> e >= 1
      __half dh = __ushort_as_half(static_cast<unsigned short>(dbits));
      if (e > 0) dh = __hmul(dh, __ushort_as_half(static_cast<unsigned short>((15 - e) << 10)));   // d / 2^e
      const __half2 d2 = __halves2half2(dh, dh);
      if (kp == 0) *reinterpret_cast<float*>(smem + (cs - raw_s) + Conv::kPs + 4 * jc) = ldexpf(1.0f, 10 + e);
      uint4 nb = make_uint4(0, 0, 0, 0);
      if (live) nb = lds128(rs + Raw::kV + jc * 128 + 16 * kp);
      const uint32_t wv[4] = {nb.x, nb.y, nb.z, nb.w};
      uint32_t ahi[16], alo[16];          // [pair]: pairs 0..7 low nibbles (dims 2i, 2i+1), 8..15 high
#pragma unroll
      for (int w4 = 0; w4 < 4; ++w4) {
        const uint32_t s01 = prmt(wv[w4], 0u, 0x4140u);      // bytes 4 w4, 4 w4 + 1 -> halves
        const uint32_t s23 = prmt(wv[w4], 0u, 0x4342u);      // bytes 4 w4 + 2, 4 w4 + 3
        split_prod(nib_lo(s01), d2, ahi[2 * w4], alo[2 * w4]);
        split_prod(nib_lo(s23), d2, ahi[2 * w4 + 1], alo[2 * w4 + 1]);
        split_prod(nib_hi(s01), d2, ahi[8 + 2 * w4], alo[8 + 2 * w4]);
        split_prod(nib_hi(s23), d2, ahi[8 + 2 * w4 + 1], alo[8 + 2 * w4 + 1]);
      }
      const uint32_t vrow = cs + Conv::kV + jc * 512;
#pragma unroll
      for (int k = 0; k < 4; ++k) {                          // chunk 4 kp + k: dims 32 kp + 8k ..
        const int ch = sw(jc, 4 * kp + k);
        sts128(vrow + 16 * ch, make_uint4(ahi[4 * k], ahi[4 * k + 1], ahi[4 * k + 2], ahi[4 * k + 3]));
        sts128(vrow + kTile * 512 + 16 * ch, make_uint4(alo[4 * k], alo[4 * k + 1], alo[4 * k + 2], alo[4 * k + 3]));
      }
    }
  };

  if (prod) {
#pragma unroll 1
    for (int s = 0; s < kRawStages - 1; ++s) {
      if (s < n_it) issue(s);
      cp_async_commit();
    }
    cp_async_wait<kRawStages - 2>();
    if (n_it > 0) convert(0);
  }
  __syncthreads();
#pragma unroll 1
  for (int t = 0; t < n_it; ++t) {
    if (prod) {
      // tile t + 1 into the other buffer while the query warps read tile t
      if (t + kRawStages - 1 < n_it) issue(t + kRawStages - 1);
      cp_async_commit();
      cp_async_wait<kRawStages - 2>();
      if (t + 1 < n_it) convert(t + 1);
    }
    if (qw) {
      const uint32_t cs = conv_s + (t & 1) * Conv::kBytes;
      const int tile0 = c_begin + kTile * t;
#pragma unroll 1
      for (int u = 0; u < 2; ++u) {
        const int cell0 = tile0 + 16 * u;
        if (cell0 >= lim) break;                               // nothing visible for this query
        // ---- S = K q over the sub-tile; two accumulators per half
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
        const int arow = 16 * u + (lane & 7) + 8 * ((lane >> 3) & 1);     // cell row this lane addresses
        const uint32_t kbase = cs + Conv::kK + arow * 512;
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          uint32_t a[4];
          ldsm_x4(a, kbase + 16 * sw(arow, 2 * ks + (lane >> 4)));
          float* dst = acc[2 * (ks >> 3) + (ks & 1)];
          mma_f16(dst, a, qf[ks][0], qf[ks][1]);
          if (QF32) mma_f16(dst, a, qf_lo[ks % (QF32 ? 16 : 1)][0], qf_lo[ks % (QF32 ? 16 : 1)][1]);
        }
        const float2 kA = *reinterpret_cast<const float2*>(smem + (cs - raw_s) + Conv::kKs + 8 * (16 * u + r0));
        const float2 kB = *reinterpret_cast<const float2*>(smem + (cs - raw_s) + Conv::kKs + 8 * (16 * u + r0 + 8));
        const bool vA = cell0 + r0 < lim, vB = cell0 + r0 + 8 < lim;
        float sc[4];
        sc[0] = vA ? (kA.x * (acc[0][0] + acc[1][0]) + kA.y * (acc[2][0] + acc[3][0])) * f0 : -INFINITY;
        sc[1] = vA ? (kA.x * (acc[0][1] + acc[1][1]) + kA.y * (acc[2][1] + acc[3][1])) * f1 : -INFINITY;
        sc[2] = vB ? (kB.x * (acc[0][2] + acc[1][2]) + kB.y * (acc[2][2] + acc[3][2])) * f0 : -INFINITY;
        sc[3] = vB ? (kB.x * (acc[0][3] + acc[1][3]) + kB.y * (acc[2][3] + acc[3][3])) * f1 : -INFINITY;

        // ---- online softmax (heads 2c, 2c+1)
        float t0 = fmaxf(sc[0], sc[2]), t1 = fmaxf(sc[1], sc[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          t0 = fmaxf(t0, __shfl_xor_sync(kFull, t0, off));
          t1 = fmaxf(t1, __shfl_xor_sync(kFull, t1, off));
        }
        const float mn0 = fmaxf(m0, t0), mn1 = fmaxf(m1, t1);   // finite: cell0 is visible
        const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
        float pr[4];
        pr[0] = exp2f(sc[0] - mn0);
        pr[1] = exp2f(sc[1] - mn1);
        pr[2] = exp2f(sc[2] - mn0);
        pr[3] = exp2f(sc[3] - mn1);
        l0 = l0 * al0 + (pr[0] + pr[2]);
        l1 = l1 * al1 + (pr[1] + pr[3]);
        m0 = mn0;
        m1 = mn1;
        if (__any_sync(kFull, al0 != 1.0f || al1 != 1.0f)) {
#pragma unroll
          for (int mt = 0; mt < 16; ++mt) {
            o[mt][0] *= al0; o[mt][1] *= al1; o[mt][2] *= al0; o[mt][3] *= al1;
          }
        }
        // ---- p to the B layout (lane: head r0, cells 2c, 2c+1, 2c+8, 2c+9), times
        // the cell's 2^(10 + e), as two fp16 terms
        float P[4];
        {
          const uint32_t u0 = __float_as_uint(pr[0]), u1 = __float_as_uint(pr[1]);
          const uint32_t u2 = __float_as_uint(pr[2]), u3 = __float_as_uint(pr[3]);
          const uint32_t th0 = movmatrix_t(prmt(u0, u1, 0x7632u)), tl0 = movmatrix_t(prmt(u0, u1, 0x5410u));
          const uint32_t th1 = movmatrix_t(prmt(u2, u3, 0x7632u)), tl1 = movmatrix_t(prmt(u2, u3, 0x5410u));
          P[0] = __uint_as_float(prmt(tl0, th0, 0x5410u));
          P[1] = __uint_as_float(prmt(tl0, th0, 0x7632u));
          P[2] = __uint_as_float(prmt(tl1, th1, 0x5410u));
          P[3] = __uint_as_float(prmt(tl1, th1, 0x7632u));
        }
        const float* psc = reinterpret_cast<const float*>(smem + (cs - raw_s) + Conv::kPs) + 16 * u;
        const float2 s01 = *reinterpret_cast<const float2*>(psc + 2 * c);
        const float2 s23 = *reinterpret_cast<const float2*>(psc + 2 * c + 8);
        const float x0 = P[0] * s01.x, x1 = P[1] * s01.y, x2 = P[2] * s23.x, x3 = P[3] * s23.y;
        const __half2 bh01 = __floats2half2_rn(x0, x1), bh23 = __floats2half2_rn(x2, x3);
        const float2 g01 = __half22float2(bh01), g23 = __half22float2(bh23);
        const uint32_t bh[2] = {h2u(bh01), h2u(bh23)};
        const uint32_t bl[2] = {h2u(__floats2half2_rn(x0 - g01.x, x1 - g01.y)),
                                h2u(__floats2half2_rn(x2 - g23.x, x3 - g23.y))};

        // ---- O += (c d) p: A = 16 dims x 16 cells of each fp16 term (ldmatrix.trans);
        // four m-tiles at a time so that no accumulator sees back-to-back MMAs
        const int vrow = 16 * u + (lane & 7) + 8 * (lane >> 4);          // cell row this lane addresses
        const uint32_t vbase = cs + Conv::kV + vrow * 512;
#pragma unroll
        for (int mg = 0; mg < 16; mg += 4) {
          uint32_t ah[4][4], al[4][4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int ch = sw(vrow, 2 * (mg + k) + ((lane >> 3) & 1));
            ldsm_x4_t(ah[k], vbase + 16 * ch);
            ldsm_x4_t(al[k], vbase + kTile * 512 + 16 * ch);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_f16(o[mg + k], ah[k], bh[0], bh[1]);
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_f16(o[mg + k], al[k], bh[0], bh[1]);
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_f16(o[mg + k], ah[k], bl[0], bl[1]);
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_f16(o[mg + k], al[k], bl[0], bl[1]);
        }
      }
    }
    __syncthreads();                      // tile t read, tile t + 1 converted
  }
  cp_async_wait<0>();

  // ---- finish: row sums across the 8 lanes of each head; un-rotate and write (o, m, l)
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, off);
    l1 += __shfl_xor_sync(kFull, l1, off);
  }
  __syncthreads();
  float* mo = reinterpret_cast<float*>(smem);                 // [n_q][8 heads][256], then m, l [n_q][8][2]
  float* ml = mo + nq * kGqa * kD;
  if (qw) {
    float* mine = mo + warp * kGqa * kD;
#pragma unroll
    for (int mt = 0; mt < 16; ++mt) {
      const int d0 = 16 * mt + r0;
      mine[(2 * c) * kD + d0] = o[mt][0] * 0x1p-10f;
      mine[(2 * c + 1) * kD + d0] = o[mt][1] * 0x1p-10f;
      mine[(2 * c) * kD + d0 + 8] = o[mt][2] * 0x1p-10f;
      mine[(2 * c + 1) * kD + d0 + 8] = o[mt][3] * 0x1p-10f;
    }
    if (r0 == 0) {
      ml[(warp * kGqa + 2 * c) * 2] = m0;
      ml[(warp * kGqa + 2 * c) * 2 + 1] = l0;
      ml[(warp * kGqa + 2 * c + 1) * 2] = m1;
      ml[(warp * kGqa + 2 * c + 1) * 2 + 1] = l1;
    }
  }
  __syncthreads();
  // one warp per output row (query, head): out = (H / 16) o on the lane's dims 8 lane ..
  for (int rr = warp; rr < nq * kGqa; rr += kThreads / 32) {
    const float* src = mo + rr * kD + 8 * lane;
    const float4 xa = *reinterpret_cast<const float4*>(src);
    const float4 xb = *reinterpret_cast<const float4*>(src + 4);
    float v[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
    for (int hh = 1; hh < 8; hh <<= 1) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (e & hh) continue;
        const float a = v[e], bb = v[e + hh];
        v[e] = a + bb;
        v[e + hh] = a - bb;
      }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float tt = __shfl_xor_sync(kFull, v[e], m);
        v[e] = upper ? tt - v[e] : v[e] + tt;
      }
    }
    const int q2 = rr >> 3, h = rr & 7;
    float* dst = p.ws + ((((static_cast<int64_t>(b) * p.splits + split) * nq + q2) * HQ) + g * kGqa + h) * kPStride;
    reinterpret_cast<float4*>(dst + 8 * lane)[0] = make_float4(v[0] * 0.0625f, v[1] * 0.0625f, v[2] * 0.0625f, v[3] * 0.0625f);
    reinterpret_cast<float4*>(dst + 8 * lane)[1] = make_float4(v[4] * 0.0625f, v[5] * 0.0625f, v[6] * 0.0625f, v[7] * 0.0625f);
    if (lane == 0) {
      dst[256] = ml[rr * 2];
      dst[257] = ml[rr * 2 + 1];
    }
  }
  // the combine kernel may start once every partial of this grid is written
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

AttendPlan plan_verify(const CacheView& C, int n_seqs, int n_q, int max_seq_len, int num_sms) {
  AttendPlan pl{};
  pl.n_q = n_q;
  pl.n_groups = 1;
  pl.warps = kThreads / 32;
  const int tiles = std::max(1, (max_seq_len + kTile - 1) / kTile);
  // about four CTAs per SM over the grid (one resident at a time): sequences of
  // unequal length leave some splits empty, and the short CTAs fill the gaps
  const int64_t pairs = static_cast<int64_t>(C.H) * n_seqs;
  const int64_t target = 4ll * num_sms;
  int64_t splits = (target + pairs - 1) / pairs;
  splits = std::max<int64_t>(1, std::min<int64_t>(splits, std::max(1, tiles / 2)));
  const int tps = static_cast<int>((tiles + splits - 1) / splits);
  pl.cells_per_split = kTile * tps;
  pl.splits = (tiles + tps - 1) / tps;
  pl.ws_bytes = static_cast<size_t>(n_seqs) * pl.splits * n_q * C.H * kGqa * kPStride * sizeof(float);
  return pl;
}

int launch_verify(const Launch& L, const CacheView& C, const AttendPlan& plan, const void* q, int q_dtype,
                  const int32_t* pt, int64_t max_pages, const int32_t* steps, int n_seqs, int max_seq_len,
                  float sm_scale, float* out, void* ws) {
  if (n_seqs == 0) return K8V4_OK;
  VerifyParams p;
  p.C = C;
  p.q = q;
  p.pt = pt;
  p.max_pages = max_pages;
  p.steps = steps;
  p.n_seqs = n_seqs;
  p.n_q = plan.n_q;
  p.max_seq_len = max_seq_len;
  p.cells_per_split = plan.cells_per_split;
  p.splits = plan.splits;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.ws = static_cast<float*>(ws);
  p.status = L.status;
  auto kern = q_dtype == K8V4_F32 ? verify_kernel<true> : verify_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return K8V4_ECUDA;
  kern<<<dim3(plan.splits, C.H, n_seqs), kThreads, kSmem, L.stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return K8V4_ECUDA;
  return launch_combine(L, p.ws, plan.splits, n_seqs, plan.n_q, C.H, out);
}

}  // namespace k8v4
