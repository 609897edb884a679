// Device helpers shared by the append kernel and the fused decode step: the
// loads of a 256-element row, the exact rotation y = RN((H x) / 16), the int8
// and q4_0 quantisers, and the per-warp append of one (token, head) row (K and
// V of the k8v4, INT8 and Q4 formats).  A
// row is held 8 elements per lane (element 8 * lane + r); each function works
// on one warp.
//
// Follows the hybrid-KV pull request "--kv k8v4: hybrid KV cache -- INT8 K +
// Hadamard-rotated Q4_0 V (816 B/cell)", sections "What" and "How".
#pragma once

#include "k8v4_common.cuh"

namespace k8v4 {
namespace {

constexpr unsigned kQFull = 0xffffffffu;

// ------------------------------------------------------------------ loads
template <bool BF16>
__device__ __forceinline__ void load8(const void* base, int64_t elem, float x[8]) {
  if (BF16) {
    const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
    const float4 a = p[0], b = p[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

// ------------------------------------------------------------------ rounding helpers
// rint_even(RN(x / d)) for |x / d| <= 128.  The product with the correctly
// rounded reciprocal is within 2^-16 of x / d and of its fp32 rounding; only when
// it lies within 1e-4 of a half-integer can the two round differently, and then
// the IEEE quotient is computed.
__device__ __forceinline__ float rint_quot(float x, float d, float rcp) {
  const float qa = __fmul_rn(x, rcp);
  float r = rintf(qa);
  if (fabsf(__fsub_rn(qa, r)) > 0.4999f) r = rintf(__fdiv_rn(x, d));
  return r;
}

// RN_fp32(m * 2^e) (sign given separately), ties to even; `sticky` says that
// non-zero bits exist below the last bit of m.  Covers normal, subnormal and
// overflowing results.
__device__ float round_u64(unsigned long long m, int e, bool sticky, bool neg) {
  if (m == 0) return neg ? -0.0f : 0.0f;
  const int nb = 64 - __clzll(static_cast<long long>(m));
  int lsb = nb - 1 + e - 23;            // exponent of the result's last bit
  if (lsb < -149) lsb = -149;
  const int sh = lsb - e;               // bits of m below that bit
  unsigned long long q;
  if (sh <= 0) {
    q = m << (-sh);                     // exact: m has at most 24 bits here
  } else if (sh > 64) {
    q = 0;                              // below half of the smallest subnormal
  } else {
    const unsigned long long rem = sh == 64 ? m : (m & ((1ull << sh) - 1ull));
    q = sh == 64 ? 0ull : (m >> sh);
    const unsigned long long half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (sticky || (q & 1ull)))) ++q;
  }
  if (q >> 24) { q >>= 1; ++lsb; }
  uint32_t bits;
  if (q >= (1ull << 23)) {
    const int ef = lsb + 23 + 127;
    bits = ef >= 255 ? 0x7f800000u : ((static_cast<uint32_t>(ef) << 23) | static_cast<uint32_t>(q & 0x7fffffull));
  } else {
    bits = static_cast<uint32_t>(q);    // subnormal or zero (lsb == -149)
  }
  return __uint_as_float(bits | (neg ? 0x80000000u : 0u));
}

// One output of the exact rotation by a multi-limb sum: y_i = RN((sum_j
// H[i][j] x_j) / 16).  The sum is kept in units of 2^-149 in 32-bit limbs held in
// int64 (no carries needed for 256 additions).
__device__ float exact_rot_elem(const float* xs, int i) {
  long long acc[10];
#pragma unroll
  for (int l = 0; l < 10; ++l) acc[l] = 0;
  for (int j = 0; j < kD; ++j) {
    const uint32_t u = __float_as_uint(xs[j]);
    const uint32_t ef = (u >> 23) & 0xffu, fr = u & 0x7fffffu;
    const uint32_t m = ef ? (fr | 0x800000u) : fr;
    if (!m) continue;
    const int k = ef ? static_cast<int>(ef) - 1 : 0;
    const bool neg = ((u >> 31) ^ (__popc(i & j) & 1)) != 0;
    const unsigned long long w = static_cast<unsigned long long>(m) << (k & 31);
    const long long lo = static_cast<long long>(w & 0xffffffffull), hi = static_cast<long long>(w >> 32);
    const int li = k >> 5;
    if (neg) { acc[li] -= lo; acc[li + 1] -= hi; }
    else { acc[li] += lo; acc[li + 1] += hi; }
  }
  auto normalise = [&]() {
    for (int l = 0; l < 9; ++l) {
      const long long c = acc[l] >> 32;   // floor division
      acc[l] -= static_cast<long long>(static_cast<unsigned long long>(c) << 32);
      acc[l + 1] += c;
    }
  };
  normalise();
  const bool neg = acc[9] < 0;
  if (neg) {
    for (int l = 0; l < 10; ++l) acc[l] = -acc[l];
    normalise();
  }
  int t = 9;
  while (t >= 0 && acc[t] == 0) --t;
  if (t < 0) return 0.0f;
  // top 64-bit window: limbs t and t-1; everything below is sticky
  const unsigned long long W = (static_cast<unsigned long long>(acc[t]) << 32) |
                               (t > 0 ? static_cast<unsigned long long>(acc[t - 1]) : 0ull);
  bool sticky = false;
  for (int l = 0; l < t - 1; ++l) sticky |= acc[l] != 0;
  // acc * 2^-149 / 16, W's last bit weighs 2^(32 (t - 1) - 153)
  return round_u64(W, 32 * (t - 1) - 153, sticky, neg);
}

// Exact rotation of the 256-vector held 8 per lane (element 8 * lane + r).
// `ts` is this warp's shared scratch of kRotScratch int64 (the fast path's
// re-dealing; its first 1 KB also stages the floats of the slow path).
constexpr int kRotScratch = 256 + 32;
__device__ void rotate_exact(float x[8], int lane, long long* ts) {
  float* xs = reinterpret_cast<float*>(ts);
  uint32_t M[8];
  int E[8];
  int lo = 1 << 30, hi = -(1 << 30);
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const uint32_t u = __float_as_uint(x[r]);
    const uint32_t ef = (u >> 23) & 0xffu, fr = u & 0x7fffffu;
    uint32_t m = ef ? (fr | 0x800000u) : fr;
    int e = ef ? static_cast<int>(ef) - 150 : -149;
    if (m) {
      const int tz = __ffs(m) - 1;
      m >>= tz;
      e += tz;
      lo = min(lo, e);
      hi = max(hi, e + 32 - __clz(m));
    }
    M[r] = m;
    E[r] = e;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(kQFull, lo, o));
    hi = max(hi, __shfl_xor_sync(kQFull, hi, o));
  }
  if (lo > hi) {                         // all zero
#pragma unroll
    for (int r = 0; r < 8; ++r) x[r] = 0.0f;
    return;
  }
  if (hi - lo <= 54) {
    // int64 fixed point with last bit 2^lo: |v| < 2^54, sums of 256 stay < 2^62
    long long v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const long long a = M[r] ? static_cast<long long>(static_cast<unsigned long long>(M[r]) << (E[r] - lo)) : 0ll;
      v[r] = (__float_as_uint(x[r]) >> 31) ? -a : a;
    }
    // The eight butterfly stages (one per index bit, in any order) all run
    // in-lane: the warp re-deals the 256 sums through shared memory so that the
    // three register bits r cover index bits {0,1,2}, then {3,4,7}, then {5,6}:
    //   layout 1: i = 8 lane + r
    //   layout 2: i = (lane & 7) | (r & 3) << 3 | (lane >> 3) << 5 | (r >> 2) << 7
    //   layout 3: i = (r >> 2) | (lane & 15) << 1 | (r & 3) << 5 | (lane >> 4) << 7
    // Element i sits at ts[i + i / 8] (one pad slot per eight spreads the banks).
    auto stages = [&](int nbits) {
#pragma unroll
      for (int h = 1; h < 8; h <<= 1) {
        if (h >= (1 << nbits)) break;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (r & h) continue;
          const long long a = v[r], b = v[r + h];
          v[r] = a + b;
          v[r + h] = a - b;
        }
      }
    };
    auto pos = [](int i) { return i + (i >> 3); };
    const int l1 = pos(8 * lane);
    const int l2 = pos((lane & 7) | ((lane >> 3) << 5));
    const int l3 = pos(((lane & 15) << 1) | ((lane >> 4) << 7));
    stages(3);
#pragma unroll
    for (int r = 0; r < 8; ++r) ts[l1 + r] = v[r];
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 8; ++r) v[r] = ts[l2 + pos(((r & 3) << 3) | ((r >> 2) << 7))];
    stages(3);
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 8; ++r) ts[l2 + pos(((r & 3) << 3) | ((r >> 2) << 7))] = v[r];
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 8; ++r) v[r] = ts[l3 + pos((r >> 2) | ((r & 3) << 5))];
    stages(2);
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 8; ++r) ts[l3 + pos((r >> 2) | ((r & 3) << 5))] = v[r];
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 8; ++r) v[r] = ts[l1 + r];
    __syncwarp();
    // RN(s * 2^(lo - 4)): the correctly rounded int64 -> fp32 conversion, then an
    // exact power-of-two scaling by the exponent field while the result stays
    // normal (or overflows to infinity, as the direct rounding would); a result
    // in the subnormal range takes the direct rounding (fewer than 24 bits)
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const long long s = v[r];
      const float f = __ll2float_rn(s);
      const uint32_t fb = __float_as_uint(f);
      const int ef = static_cast<int>((fb >> 23) & 0xffu) + lo - 4;
      if (s == 0) {
        x[r] = 0.0f;
      } else if (ef >= 255) {
        x[r] = __uint_as_float((fb & 0x80000000u) | 0x7f800000u);
      } else if (ef >= 1) {
        x[r] = __uint_as_float((fb & 0x807fffffu) | (static_cast<uint32_t>(ef) << 23));
      } else {
        const unsigned long long mag = s < 0 ? 0ull - static_cast<unsigned long long>(s) : static_cast<unsigned long long>(s);
        x[r] = round_u64(mag, lo - 4, false, s < 0);
      }
    }
    return;
  }
  // slow path: exact multi-limb sums
#pragma unroll
  for (int r = 0; r < 8; ++r) xs[8 * lane + r] = x[r];
  __syncwarp();
#pragma unroll 1
  for (int r = 0; r < 8; ++r) x[r] = exact_rot_elem(xs, 8 * lane + r);
  __syncwarp();
}

// ------------------------------------------------------------------ quantisers
// int8 over a 128-lane half held by 16 lanes (lanes 0-15: half 0, 16-31: half
// 1).  Returns the half's scale; codes packed little-endian into two words.
__device__ __forceinline__ float quant_int8_half(const float x[8], uint2& packed) {
  float a = 0.0f;
#pragma unroll
  for (int r = 0; r < 8; ++r) a = fmaxf(a, fabsf(x[r]));
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(kQFull, a, o));
  const float s = __fdiv_rn(a, 127.0f);
  uint32_t w[2] = {0u, 0u};
  if (s != 0.0f) {
    const bool tiny = s < 0x1p-125f;     // reciprocal could overflow
    const float rcp = tiny ? 0.0f : __frcp_rn(s);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float c = tiny ? rintf(__fdiv_rn(x[r], s)) : rint_quot(x[r], s, rcp);
      c = fminf(fmaxf(c, -127.0f), 127.0f);
      w[r >> 2] |= (static_cast<uint32_t>(static_cast<int>(c)) & 0xffu) << (8 * (r & 3));
    }
  }
  packed = make_uint2(w[0], w[1]);
  return s;
}

// Stores of the row routines: every value goes to page `a` and, when `b` is
// not null, to the same offset of page `b` (the host mirror of a streamed cache
// and its resident device slot hold the same bytes)
template <typename T>
__device__ __forceinline__ void st2(uint8_t* a, uint8_t* b, int64_t off, T v) {
  *reinterpret_cast<T*>(a + off) = v;
  if (b != nullptr) *reinterpret_cast<T*>(b + off) = v;
}

// Q4_0 of the rotated vector (element 8 * lane + r; block = lane / 4).  Writes the
// block's 16 nibble bytes (lanes 4b, 4b+1, 8 bytes each) at q_off and its fp16
// scale (lane 4b) at s_off of page a (and page b)
__device__ __forceinline__ void quant_q4_store(const float y[8], int lane, uint8_t* a, uint8_t* b, int64_t q_off,
                                               int64_t s_off) {
  uint32_t best = __float_as_uint(y[0]) & 0x7fffffffu;
  int bi = 0;
#pragma unroll
  for (int r = 1; r < 8; ++r) {
    const uint32_t a = __float_as_uint(y[r]) & 0x7fffffffu;
    if (a > best) { best = a; bi = r; }  // first index wins ties
  }
  const int idx = 8 * lane + bi;
  unsigned long long key = (static_cast<unsigned long long>(best) << 32) |
                           (static_cast<unsigned long long>(255 - idx) << 1) |
                           static_cast<unsigned long long>(__float_as_uint(y[bi]) >> 31);
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    const unsigned long long other = __shfl_xor_sync(kQFull, key, o);
    key = other > key ? other : key;
  }
  const float m = __uint_as_float(static_cast<uint32_t>(key >> 32) | (static_cast<uint32_t>(key & 1ull) << 31));
  const __half dh = __float2half_rn(__fmul_rn(m, -0.125f));   // m / -8, exact scaling
  const float d = __half2float(dh);
  uint32_t packed = 0x88888888u;
  if (d != 0.0f) {
    const float rcp = __frcp_rn(d);
    packed = 0u;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float c = rint_quot(y[r], d, rcp) + 8.0f;
      c = fminf(fmaxf(c, 0.0f), 15.0f);
      packed |= static_cast<uint32_t>(static_cast<int>(c)) << (4 * r);
    }
  }
  const uint32_t high = __shfl_xor_sync(kQFull, packed, 2);  // codes j + 16 of the block
  const int blk = lane >> 2;
  if ((lane & 2) == 0) {
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint32_t byte = ((packed >> (4 * r)) & 0xfu) | (((high >> (4 * r)) & 0xfu) << 4);
      out[r >> 2] |= byte << (8 * (r & 3));
    }
    st2(a, b, q_off + 16 * blk + 8 * (lane & 1), make_uint2(out[0], out[1]));
  }
  if ((lane & 3) == 0) st2(a, b, s_off + 2 * blk, dh);
}

// ------------------------------------------------------------------ row appends
// K row of (token, head) r: int8 codes + two fp32 scales, or, in the Q4 format,
// rotated q4_0 like V; ts is this warp's kRotScratch int64 of shared scratch
// for the rotation (Q4 only).  Written to page `base` and, when base2 is not
// null, to page base2 as well.
template <bool BF16, int FMT>
__device__ __forceinline__ void append_k_row(const CacheView& C, uint8_t* base, int64_t r, const void* k, int64_t elem,
                                             int lane, long long* ts, uint8_t* base2 = nullptr) {
  float x[8];
  load8<BF16>(k, elem, x);
  if (FMT == K8V4_FORMAT_Q4) {
    rotate_exact(x, lane, ts);
    quant_q4_store(x, lane, base, base2, r * 128, C.ks_off() + r * 16);
    return;
  }
  uint2 kc;
  const float s = quant_int8_half(x, kc);
  const float s_hi = __shfl_xor_sync(kQFull, s, 16);
  st2(base, base2, r * 256 + 8 * lane, kc);
  if (lane == 0) st2(base, base2, C.ks_off() + r * 8, make_float2(s, s_hi));
}
// V row: rotated q4_0 (k8v4 and Q4) or int8 (the INT8 comparison format)
template <bool BF16, int FMT>
__device__ __forceinline__ void append_v_row(const CacheView& C, uint8_t* base, int64_t r, const void* v, int64_t elem,
                                             int lane, long long* ts, uint8_t* base2 = nullptr) {
  float x[8];
  load8<BF16>(v, elem, x);
  if (FMT != K8V4_FORMAT_INT8) {
    rotate_exact(x, lane, ts);
    quant_q4_store(x, lane, base, base2, C.v_off() + r * 128, C.vs_off() + r * 16);
  } else {
    uint2 vc;
    const float sv = quant_int8_half(x, vc);
    const float sv_hi = __shfl_xor_sync(kQFull, sv, 16);
    st2(base, base2, C.v_off() + r * 256 + 8 * lane, vc);
    if (lane == 0) st2(base, base2, C.vs_off() + r * 8, make_float2(sv, sv_hi));
  }
}

}  // namespace
}  // namespace k8v4
