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


// ------------------------------------------------------------------ bf16 rows, fast paths
// The bulk append of bf16 K/V rows.  Same bytes as the routines above (the
// pull request's "What" and "How": int8 K with IEEE quotients, V rotated
// exactly and quantised to q4_0), with fewer instructions for the common row:
//
//  * quotients: q = x * rcp with rcp = rcp.approx(s) (at most 1 ulp off 1/s)
//    lies within 3.1e-5 of RN(x / s) for |x / s| <= 127.5, so rint(q) equals
//    rint(RN(x / s)) unless q is within 1e-4 of a half-integer; such values
//    (about 1 in 5,000) are redone with the IEEE division.  rint is taken by
//    adding 1.5 * 2^23 (whose ulp is 1), which leaves the integer in the low
//    mantissa bits;
//  * rotation: a bf16 value is m * 2^(E - 134) with m < 2^8 (E its exponent
//    field), so every element of a row is an integer multiple of 2^lo, lo =
//    Emin - 134 (Emin: the smallest element's exponent field).  No partial sum
//    of the 256-point transform exceeds the row's L1 norm; when that norm is at
//    most 2^30 units of 2^lo the transform runs exactly in int32 on the integers
//    x / 2^lo, and y = RN(s * 2^(lo - 4)) is the int32 -> fp32 conversion scaled
//    by a power of two (exact: the result is normal).  Other rows (exact zeros,
//    subnormals, a norm too large for the smallest element's grain, inf/NaN)
//    take the int64/multi-limb rotation above.

__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t vmin_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
// 8 bf16 (element 8 * lane + r: word k holds r = 2k low, 2k + 1 high) -> fp32
__device__ __forceinline__ void bf16x8_to_f32(const uint4 raw, float x[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
// the low bytes of four words, packed little-endian
__device__ __forceinline__ uint32_t low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return prmt(prmt(a, b, 0x0040u), prmt(c, d, 0x0040u), 0x5410u);
}

constexpr float kRintMagic = 12582912.0f;        // 1.5 * 2^23
constexpr float kQuotientSlack = 0.4999f;         // |q - rint(q)| above this: redo with the IEEE quotient

// The general quantisers on a bf16 row, out of line (rare rows; keeps the fast
// loop small in the instruction cache)
__device__ __noinline__ void int8_row_general(const uint4 raw, int lane, uint8_t* a, uint8_t* b, int64_t code_off,
                                              int64_t scale_off) {
  float x[8];
  bf16x8_to_f32(raw, x);
  uint2 kc;
  const float s = quant_int8_half(x, kc);
  const float s_hi = __shfl_xor_sync(kQFull, s, 16);
  st2(a, b, code_off + 8 * lane, kc);
  if (lane == 0) st2(a, b, scale_off, make_float2(s, s_hi));
}
__device__ __noinline__ void rot_q4_row_general(const uint4 raw, int lane, long long* ts, uint8_t* a, uint8_t* b,
                                                int64_t q_off, int64_t s_off) {
  float x[8];
  bf16x8_to_f32(raw, x);
  __syncwarp();
  rotate_exact(x, lane, ts);
  quant_q4_store(x, lane, a, b, q_off, s_off);
  __syncwarp();
}

// RN(M / 127) for the 128 significands M = 128..255 of a bf16 value, the int8
// scale s = RN(amax / 127) of amax = M * 2^(E - 134) being that entry scaled by
// 2^(E - 134) (exact while s is normal).  Filled once per CTA.
__device__ __forceinline__ void fill_int8_scale_table(float* tab) {
  for (int i = threadIdx.x; i < 128; i += blockDim.x) tab[i] = __fdiv_rn(static_cast<float>(128 + i), 127.0f);
}

// int8 of a bf16 row (two 128-element halves, lanes 0-15 and 16-31): codes at
// code_off + 8 * lane, the two fp32 scales at scale_off
__device__ __forceinline__ void int8_row_bf16(const uint4 raw, int lane, const float* tab, uint8_t* a, uint8_t* b,
                                              int64_t code_off, int64_t scale_off) {
  uint32_t m = vmax_u16x2(vmax_u16x2(raw.x & 0x7fff7fffu, raw.y & 0x7fff7fffu),
                          vmax_u16x2(raw.z & 0x7fff7fffu, raw.w & 0x7fff7fffu));
  m = vmax_u16x2(m, prmt(m, 0u, 0x1032u));
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) m = vmax_u16x2(m, __shfl_xor_sync(kQFull, m, o));
  const uint32_t a16 = m & 0xffffu;                  // |largest| of this half, bf16 bits
  const uint32_t e16 = a16 >> 7;                     // its exponent field
  // s normal and at least 2^-125 needs E >= 10; a zero half gives s = 0
  if (__any_sync(kQFull, a16 >= 0x7f80u || (a16 != 0u && e16 < 10u))) {
    int8_row_general(raw, lane, a, b, code_off, scale_off);
    return;
  }
  const float s = a16 == 0u ? 0.0f
                            : __uint_as_float(__float_as_uint(tab[a16 & 0x7fu]) + ((e16 - 134u + 0u) << 23));
  float x[8];
  bf16x8_to_f32(raw, x);
  const float rcp = s != 0.0f ? rcp_approx(s) : 0.0f;
  uint32_t t[8];
  float worst = 0.0f;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const float q = __fmul_rn(x[r], rcp);
    const float tf = __fadd_rn(q, kRintMagic);
    worst = fmaxf(worst, fabsf(__fsub_rn(q, __fsub_rn(tf, kRintMagic))));
    t[r] = __float_as_uint(tf);
  }
  if (__any_sync(kQFull, worst > kQuotientSlack)) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float q = __fmul_rn(x[r], rcp);
      if (fabsf(__fsub_rn(q, __fsub_rn(__uint_as_float(t[r]), kRintMagic))) > kQuotientSlack)
        t[r] = __float_as_uint(__fadd_rn(rintf(__fdiv_rn(x[r], s)), kRintMagic));
    }
  }
  // |code| <= 127: the low byte of the biased word is the two's-complement code
  st2(a, b, code_off + 8 * lane, make_uint2(low_bytes(t[0], t[1], t[2], t[3]), low_bytes(t[4], t[5], t[6], t[7])));
  const float s_hi = __shfl_xor_sync(kQFull, s, 16);
  if (lane == 0) st2(a, b, scale_off, make_float2(s, s_hi));
}

// Shared-memory word of transform index i for the int32 re-dealing: i with bits
// 2-4 flipped when bit 5 is set.  All three access patterns below (two 16-byte
// stores per lane of i = 8 lane + r; eight 4-byte accesses of layout B; two
// 16-byte loads of layout D) then touch every bank once per wavefront.
__device__ __forceinline__ int rot_word(int i) { return i ^ (((i >> 5) & 1) * 28); }

// Rotation + q4_0 of a bf16 row: nibbles at q_off (16 B per 32-element block),
// fp16 scales at s_off.  ts: this warp's 16-byte aligned scratch of kRotScratch
// int64 (256 words for the int32 path; the general path needs all of it).
__device__ __forceinline__ void rot_q4_row_bf16(const uint4 raw, int lane, long long* ts64, uint8_t* a, uint8_t* b,
                                                int64_t q_off, int64_t s_off) {
  int* ts = reinterpret_cast<int*>(ts64);
  // the row's smallest magnitude (bf16 bits) and its L1 norm
  const uint32_t w0 = raw.x & 0x7fff7fffu, w1 = raw.y & 0x7fff7fffu, w2 = raw.z & 0x7fff7fffu,
                 w3 = raw.w & 0x7fff7fffu;
  uint32_t mn = vmin_u16x2(vmin_u16x2(w0, w1), vmin_u16x2(w2, w3));
  mn = vmin_u16x2(mn, prmt(mn, 0u, 0x1032u));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mn = vmin_u16x2(mn, __shfl_xor_sync(kQFull, mn, o));
  float x[8];
  bf16x8_to_f32(raw, x);
  float l1 = (fabsf(x[0]) + fabsf(x[1])) + (fabsf(x[2]) + fabsf(x[3])) +
             ((fabsf(x[4]) + fabsf(x[5])) + (fabsf(x[6]) + fabsf(x[7])));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) l1 += __shfl_xor_sync(kQFull, l1, o);   // same sum in every lane
  // lo = emin - 134: the last bit of the smallest element, hence of every element.
  // Every partial sum of the transform is at most the L1 norm: with the float
  // norm (relative error < 2^-16) at most 2^30 units of 2^lo, they all stay
  // below 2^31.  emin >= 12 keeps 2^(lo - 4) normal; inf/NaN fail the test.
  const int emin = static_cast<int>((mn & 0xffffu) >> 7);
  const float to_fixed = __uint_as_float(static_cast<uint32_t>(max(261 - emin, 1)) << 23);   // 2^-lo
  if (!__all_sync(kQFull, emin >= 12 && emin <= 200 && __fmul_rn(l1, to_fixed) <= 0x1p30f)) {
    rot_q4_row_general(raw, lane, ts64, a, b, q_off, s_off);
    return;
  }
  int v[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) v[r] = __float2int_rn(__fmul_rn(x[r], to_fixed));   // exact integers
  auto stages = [&](int first, int last) {    // butterflies over register bits first..last-1
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
      if (h < first || h >= last) continue;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r & h) continue;
        const int p = v[r], q = v[r + h];
        v[r] = p + q;
        v[r + h] = p - q;
      }
    }
  };
  // layout A: i = 8 lane + r -> index bits 0, 1, 2
  stages(1, 8);
  __syncwarp();
  {
    const int i0 = 8 * lane;
    *reinterpret_cast<int4*>(ts + rot_word(i0)) = make_int4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<int4*>(ts + rot_word(i0 + 4)) = make_int4(v[4], v[5], v[6], v[7]);
  }
  __syncwarp();
  // layout B: i = (lane & 7) | (r & 1) << 3 | (lane >> 3) << 4 | (r >> 1) << 6 -> bits 3, 6, 7.
  // The word is rot_word(ib) with bit 3 toggled for odd r, plus 64 (r >> 1).
  const int wb0 = rot_word((lane & 7) | ((lane >> 3) << 4)), wb1 = wb0 ^ 8;
#pragma unroll
  for (int r = 0; r < 8; ++r) v[r] = ts[((r & 1) ? wb1 : wb0) + 64 * (r >> 1)];
  stages(1, 8);
  __syncwarp();
#pragma unroll
  for (int r = 0; r < 8; ++r) ts[((r & 1) ? wb1 : wb0) + 64 * (r >> 1)] = v[r];
  __syncwarp();
  // layout D (the q4_0 layout): i = 32 (lane >> 2) + 4 (lane & 3) + (r & 3) + 16 (r >> 2):
  // lanes 4b..4b+3 hold block b, byte j of its nibble run pairs r = j & 3 with r + 4
  {
    const int id = 32 * (lane >> 2) + 4 * (lane & 3);
    const int4 lo4 = *reinterpret_cast<const int4*>(ts + rot_word(id));
    const int4 hi4 = *reinterpret_cast<const int4*>(ts + rot_word(id + 16));
    v[0] = lo4.x; v[1] = lo4.y; v[2] = lo4.z; v[3] = lo4.w;
    v[4] = hi4.x; v[5] = hi4.y; v[6] = hi4.z; v[7] = hi4.w;
  }
  stages(4, 8);                               // index bit 4
  {
    const int sgn = (lane & 4) ? -1 : 1;      // index bit 5 = lane bit 2
#pragma unroll
    for (int r = 0; r < 8; ++r) v[r] = __shfl_xor_sync(kQFull, v[r], 4) + sgn * v[r];
  }
  // z = RN(s): y = z * 2^(lo - 4) exactly, so the block maximum and the codes can
  // work on z, with the reciprocal of d carrying the 2^(lo - 4)
  float z[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) z[r] = __int2float_rn(v[r]);
  const float from_fixed = __uint_as_float(static_cast<uint32_t>(emin - 11) << 23);  // 2^(lo - 4)
  // block maximum by magnitude, sign kept; an exact +/- tie goes to the lower index
  float pmax = z[0], nmin = z[0];
#pragma unroll
  for (int r = 1; r < 8; ++r) {
    pmax = fmaxf(pmax, z[r]);
    nmin = fminf(nmin, z[r]);
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    pmax = fmaxf(pmax, __shfl_xor_sync(kQFull, pmax, o));
    nmin = fminf(nmin, __shfl_xor_sync(kQFull, nmin, o));
  }
  const float ap = fabsf(pmax), an = fabsf(nmin);
  float mz = ap > an ? pmax : (an > ap ? nmin : pmax);
  const bool tie = ap == an && pmax != nmin;
  if (__any_sync(kQFull, tie)) {
    // first index (within the block) holding the magnitude ap, and its sign
    uint32_t best = 0xffffffffu;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint32_t j = static_cast<uint32_t>(4 * (lane & 3) + (r & 3) + 16 * (r >> 2));
      const uint32_t k = (j << 1) | (__float_as_uint(z[r]) >> 31);
      if (fabsf(z[r]) == ap && k < best) best = k;
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) best = min(best, __shfl_xor_sync(kQFull, best, o));
    if (tie) mz = (best & 1u) ? -ap : ap;
  }
  const __half dh = __float2half_rn(__fmul_rn(__fmul_rn(mz, from_fixed), -0.125f));
  const float d = __half2float(dh);
  // q = RN(y / d) ~ z * (2^(lo - 4) / d); d = +-inf gives 0, codes 8 as for y / d = 0
  const float rcp = d != 0.0f ? __fmul_rn(rcp_approx(d), from_fixed) : 0.0f;
  constexpr float kMagic8 = kRintMagic + 8.0f;
  uint32_t t[8];
  float worst = 0.0f;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const float q = __fmul_rn(z[r], rcp);
    const float tf = __fadd_rn(q, kMagic8);
    worst = fmaxf(worst, fabsf(__fsub_rn(q, __fsub_rn(tf, kMagic8))));
    t[r] = __float_as_uint(fminf(tf, kRintMagic + 15.0f));
  }
  // |y / d| <= 8 (1 + 2^-11) for a normal d: codes >= 0.  A subnormal d (or a
  // quotient near a half-integer) takes the exact quotient and both clamps.
  if (__any_sync(kQFull, worst > kQuotientSlack || fabsf(d) < 0x1p-14f)) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float q = __fmul_rn(z[r], rcp);
      const float tf = __fadd_rn(q, kMagic8);
      float c = tf;
      if (fabsf(__fsub_rn(q, __fsub_rn(tf, kMagic8))) > kQuotientSlack)
        c = __fadd_rn(rintf(__fdiv_rn(__fmul_rn(z[r], from_fixed), d)), kMagic8);
      t[r] = __float_as_uint(fminf(fmaxf(c, kRintMagic), kRintMagic + 15.0f));
    }
  }
  // code = low nibble of the biased word (2^22 + 8 + rint); byte j = code(r) | code(r + 4) << 4
  const uint32_t lo = low_bytes(t[0], t[1], t[2], t[3]), hi = low_bytes(t[4], t[5], t[6], t[7]);
  st2(a, b, q_off + 4 * lane, (lo & 0x0f0f0f0fu) | ((hi << 4) & 0xf0f0f0f0u));
  if ((lane & 3) == 0) st2(a, b, s_off + 2 * (lane >> 2), dh);
}

// One bf16 row of a single-token append (the fused decode step) through the
// fast paths above: K as int8 (its scale table first built by the warp in ts),
// or rotated q4_0 in the Q4 format; V as rotated q4_0, or int8 in the INT8
// format.  src points at the row's first element (16-byte aligned); same bytes
// as append_k_row / append_v_row.
template <int FMT>
__device__ __forceinline__ void append_k_row_bf16(const CacheView& C, uint8_t* base, int64_t r, const uint16_t* src,
                                                  int lane, long long* ts) {
  const uint4 raw = reinterpret_cast<const uint4*>(src)[lane];
  if (FMT == K8V4_FORMAT_Q4) {
    rot_q4_row_bf16(raw, lane, ts, base, nullptr, r * 128, C.ks_off() + r * 16);
    return;
  }
  float* tab = reinterpret_cast<float*>(ts);
  for (int i = lane; i < 128; i += 32) tab[i] = __fdiv_rn(static_cast<float>(128 + i), 127.0f);
  __syncwarp();
  int8_row_bf16(raw, lane, tab, base, nullptr, r * 256, C.ks_off() + r * 8);
}
template <int FMT>
__device__ __forceinline__ void append_v_row_bf16(const CacheView& C, uint8_t* base, int64_t r, const uint16_t* src,
                                                  int lane, long long* ts) {
  const uint4 raw = reinterpret_cast<const uint4*>(src)[lane];
  if (FMT != K8V4_FORMAT_INT8) {
    rot_q4_row_bf16(raw, lane, ts, base, nullptr, C.v_off() + r * 128, C.vs_off() + r * 16);
    return;
  }
  float* tab = reinterpret_cast<float*>(ts);
  for (int i = lane; i < 128; i += 32) tab[i] = __fdiv_rn(static_cast<float>(128 + i), 127.0f);
  __syncwarp();
  int8_row_bf16(raw, lane, tab, base, nullptr, C.v_off() + r * 256, C.vs_off() + r * 8);
}

}  // namespace
}  // namespace k8v4
