// Split-K flash-decode attention over the k8v4 (or INT8, or Q4) paged cache:
// decode (one query per sequence), the fused decode step (append the newest
// token, then decode), and verify over the INT8 and Q4 comparison formats (n_q
// queries per sequence with per-query step arrays; k8v4 verify runs in
// k8v4_prefill.cu or k8v4_verify.cu).  The fused "mode 3" attention of the hybrid-KV pull request
// ("How": the K loader takes the int8 branch, the V loop the q4 branch, q is not
// rotated and the output is rotated back; "Tests": step and batched forms with
// per-query step arrays).
//
// GB300 design.  One warp owns one query (the 8 query heads of a KV head) and a
// stream of 16-cell tiles.  Tiles are staged into shared memory with 16-byte
// cp.async copies (three stages per tile group), dequantised in registers and
// fed to warp-level tensor-core MMAs (mma.sync m16n8k16), because at GQA 8 the
// decode loop needs about 10 FMA per cache byte, more than the fp32 pipes can
// give at HBM speed:
//   QK^T: A = K codes (16 cells x 16 dims, int8 -> fp16 exactly), B = q (fp16,
//         scaled per head by a power of two; an fp32 q is split into two fp16
//         terms), separate fp32 accumulators for the two 128-lane halves so the
//         two K scales apply after the MMA.  Q4 format (K rotated q4_0 like
//         V): A = K nibbles (ldmatrix, nibble -> fp16 exactly), B = (H/16) q
//         rotated once per warp in fp32 and split into two fp16 terms, a fresh
//         accumulator per 32-lane block scaled by that block's d per cell.
//   PV:   A = V codes (16 rotated dims x 16 cells, nibble -> bf16 exactly via
//         ldmatrix.trans), B = p * d per 32-lane block, split into three bf16
//         terms (24 significant bits), accumulated in fp32 in rotated space.
// Online softmax in the log2 domain.  Each CTA merges its warps and writes one
// partial (m, l, o) per query row, o already rotated back (out = (H/16) o is
// linear, so it commutes with the merge); the combine (k8v4_combine.cu) merges
// the splits.  In the fused decode step the CTA whose cells hold the newest one
// first writes that token (k8v4_quant.cuh row routines), then stages its tiles.
#include <algorithm>

#include "k8v4_quant.cuh"

namespace k8v4 {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kStages = 3;      // cp.async stages per tile group
constexpr int kWarps = 8;       // warps per CTA (tile groups x queries)
constexpr int kPStride = 260;   // floats per partial row: o[256], m, l, 2 pad
// bf16 terms of p * d: three give 24 significant bits, the precision the
// element-wise error budget of the decode paths is derived for; fewer terms
// would leave the budget
constexpr int kPlanes = 3;
static_assert(kPlanes == 3, "p * d must be carried in three bf16 terms");

template <int FMT>
struct Stage {
  static constexpr int kKBytes = FMT == K8V4_FORMAT_Q4 ? 16 * 128 : 16 * 256;    // int8 codes or nibbles
  static constexpr int kVBytes = FMT == K8V4_FORMAT_INT8 ? 16 * 256 : 16 * 128;  // nibbles or int8 codes
  static constexpr int kKsBytes = FMT == K8V4_FORMAT_Q4 ? 16 * 16 : 16 * 8;      // [16][8] f16 or [16][2] f32
  static constexpr int kVsBytes = FMT == K8V4_FORMAT_INT8 ? 16 * 8 : 16 * 16;
  static constexpr int kK = 0;                                            // K [16][256 or 128], swizzled
  static constexpr int kV = kKBytes;                                      // V [16][128 or 256], swizzled
  static constexpr int kKs = kV + kVBytes;
  static constexpr int kVs = kKs + kKsBytes;
  static constexpr int kBytes = kVs + kVsBytes;
};
__host__ __device__ constexpr int stage_bytes_of(int fmt) {
  return fmt == K8V4_FORMAT_K8V4 ? Stage<K8V4_FORMAT_K8V4>::kBytes
         : fmt == K8V4_FORMAT_Q4 ? Stage<K8V4_FORMAT_Q4>::kBytes
                                 : Stage<K8V4_FORMAT_INT8>::kBytes;
}

struct AttendParams {
  CacheView C;
  const void* q;
  const int32_t* pt;
  int64_t max_pages;
  const int32_t* steps;
  int n_seqs, n_q, n_groups, max_seq_len, cells_per_split, splits;
  float sm_scale_log2;
  float* ws;
  int* status;
  const void* k_new;       // fused decode step: the new token's K and V [n_seqs][H][256], else null
  const void* v_new;
  int kv_bf16;
};

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ void mma_f16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ void ldmatrix_x4_t(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
// two fp32 -> bf16x2 (round to nearest even); `lo` lands in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// four int8 codes -> two fp16x2 (exact): 0x64XX is 1024 + XX in fp16
__device__ __forceinline__ void codes_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;            // c + 128
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  uint32_t a = prmt(u, 0x64646464u, 0x4140u), b = prmt(u, 0x64646464u, 0x4342u);
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}
// two nibbles at bits k and k+16 -> bf16x2 of (n - 8), exact: 0x43XX is 128 + XX
__device__ __forceinline__ uint32_t nib_to_bf16(uint32_t r, int k) {
  uint32_t t = ((r >> k) & 0x000f000fu) | 0x43004300u;
  const __nv_bfloat162 bias = __halves2bfloat162(__ushort_as_bfloat16(0x4308), __ushort_as_bfloat16(0x4308));
  __nv_bfloat162 v = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&t), bias);
  return *reinterpret_cast<uint32_t*>(&v);
}
// one word of nibble bytes b0..b3 -> four fp16x2 of (n - 8), exact:
//   lo0 = {b0 & 15, b2 & 15}, lo1 = {b1 & 15, b3 & 15}, hi0 = {b0 >> 4, b2 >> 4}, hi1 = {b1 >> 4, b3 >> 4}.
// 0x640n is 1024 + n in fp16 and 0x64n0 is 1024 + 16 n; (1024 + 16 n) / 16 - 72
// = n - 8 is exact, so one fused multiply-add finishes a high nibble
__device__ __forceinline__ void nibs_to_f16(uint32_t r, uint32_t& lo0, uint32_t& lo1, uint32_t& hi0, uint32_t& hi1) {
  const uint32_t r8 = r >> 8;
  const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
  const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2c00), __ushort_as_half(0x2c00));  // 1/16
  const __half2 m72 = __halves2half2(__ushort_as_half(0xd480), __ushort_as_half(0xd480));      // -72
  uint32_t t0 = (r & 0x000f000fu) | 0x64006400u, t1 = (r8 & 0x000f000fu) | 0x64006400u;
  uint32_t t2 = (r & 0x00f000f0u) | 0x64006400u, t3 = (r8 & 0x00f000f0u) | 0x64006400u;
  __half2 v0 = __hsub2(*reinterpret_cast<__half2*>(&t0), bias);
  __half2 v1 = __hsub2(*reinterpret_cast<__half2*>(&t1), bias);
  __half2 v2 = __hfma2(*reinterpret_cast<__half2*>(&t2), sixteenth, m72);
  __half2 v3 = __hfma2(*reinterpret_cast<__half2*>(&t3), sixteenth, m72);
  lo0 = *reinterpret_cast<uint32_t*>(&v0);
  lo1 = *reinterpret_cast<uint32_t*>(&v1);
  hi0 = *reinterpret_cast<uint32_t*>(&v2);
  hi1 = *reinterpret_cast<uint32_t*>(&v3);
}
// bytes k0 and k1 of r (int8 codes) -> bf16x2 {c_k0, c_k1}, exact
__device__ __forceinline__ uint32_t i8_to_bf16(uint32_t r, uint32_t s0, uint32_t s1) {
  const uint32_t u = r ^ 0x80808080u;
  const float f0 = __uint_as_float(prmt(u, 0x4b000000u, s0)) - 8388736.0f;   // 2^23 + 128
  const float f1 = __uint_as_float(prmt(u, 0x4b000000u, s1)) - 8388736.0f;
  return prmt(__float_as_uint(f0), __float_as_uint(f1), 0x7632u);
}

// 2^x on the special-function unit (relative error ~2^-22; results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- tile loader
// Stage one 16-cell tile of KV head g (cells slot0 .. slot0+15 of one page) with
// 16-byte cp.async copies.  NTHR > 0 fixes the group size at compile time (the
// loops then unroll); NTHR == 0 reads it from nthr.
template <int FMT, int NTHR>
__device__ __forceinline__ void load_tile(const CacheView& C, uint32_t s, const uint8_t* base, int slot0, int g,
                                          int tid, int nthr_rt) {
  const int nthr = NTHR > 0 ? NTHR : nthr_rt;
  const int H = C.H;
  constexpr int kRow = FMT == K8V4_FORMAT_Q4 ? 128 : 256;                 // K bytes per (cell, head)
  constexpr int vRow = FMT == K8V4_FORMAT_INT8 ? 256 : 128;
  const int64_t r0 = static_cast<int64_t>(slot0) * H + g;       // (cell, head) index of the tile's first row
  const uint8_t* kb = base + r0 * kRow;
  const uint8_t* vb = base + C.v_off() + r0 * vRow;
  const uint8_t* ksb = base + C.ks_off() + r0 * (FMT == K8V4_FORMAT_Q4 ? 16 : 8);
  const uint8_t* vsb = base + C.vs_off() + r0 * (FMT == K8V4_FORMAT_INT8 ? 8 : 16);
  const int kst = H * kRow, vst = H * vRow;
  if (FMT == K8V4_FORMAT_Q4) {
    // K nibbles: 16 cells x 8 blocks; block b of cell j stored at b ^ (j & 7)
#pragma unroll
    for (int i = tid; i < 128; i += nthr) {
      const int j = i >> 3, bb = i & 7;
      cp_async16(s + Stage<FMT>::kK + j * 128 + 16 * (bb ^ (j & 7)), kb + j * kst + 16 * bb);
    }
  } else {
    // K codes: 16 cells x 16 chunks; chunk kk of cell j stored at kk ^ (4 * (j & 1))
#pragma unroll
    for (int i = tid; i < 256; i += nthr) {
      const int j = i >> 4, kk = i & 15;
      cp_async16(s + Stage<FMT>::kK + j * 256 + 16 * (kk ^ ((j & 1) << 2)), kb + j * kst + 16 * kk);
    }
  }
  if (FMT != K8V4_FORMAT_INT8) {
    // V nibbles: 16 cells x 8 blocks; block b of cell j stored at b ^ (j & 7)
#pragma unroll
    for (int i = tid; i < 128; i += nthr) {
      const int j = i >> 3, bb = i & 7;
      cp_async16(s + Stage<FMT>::kV + j * 128 + 16 * (bb ^ (j & 7)), vb + j * vst + 16 * bb);
    }
  } else {
#pragma unroll
    for (int i = tid; i < 256; i += nthr) {
      const int j = i >> 4, kk = i & 15;
      cp_async16(s + Stage<FMT>::kV + j * 256 + 16 * (kk ^ (j & 7)), vb + j * vst + 16 * kk);
    }
  }
#pragma unroll
  for (int i = tid; i < 32; i += nthr) {
    const int j = i & 15;
    if (i < 16) {
      if (FMT == K8V4_FORMAT_Q4) cp_async16(s + Stage<FMT>::kKs + 16 * j, ksb + j * (H * 16));
      else cp_async8(s + Stage<FMT>::kKs + 8 * j, ksb + j * (H * 8));
    } else if (FMT != K8V4_FORMAT_INT8) {
      cp_async16(s + Stage<FMT>::kVs + 16 * j, vsb + j * (H * 16));
    } else {
      cp_async8(s + Stage<FMT>::kVs + 8 * j, vsb + j * (H * 8));
    }
  }
}

// ---------------------------------------------------------------- main kernel
template <int FMT, bool QF32, bool NQ1>
__global__ void __launch_bounds__(kWarps * 32, 1) attend_splitk_kernel(const AttendParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  // launched as a programmatic dependent of the previous kernel in the stream
  // (typically the append of the new token): nothing is read before it completes
  asm volatile("griddepcontrol.wait;" ::: "memory");
  using S = Stage<FMT>;
  constexpr int kMT = 16;                                 // PV m-tiles (16 dims each)
  constexpr int kBlocks = FMT == K8V4_FORMAT_INT8 ? 2 : 8;  // V scale blocks per head
  constexpr bool kQ4 = FMT == K8V4_FORMAT_Q4;
  constexpr bool kLo = QF32 || kQ4;                         // q carried as two fp16 terms
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int qi = warp % p.n_q, gi = warp / p.n_q;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int r0 = lane >> 2, c = lane & 3;
  const CacheView& C = p.C;
  const int HQ = C.H * kGqa;

  // ---- visible counts (device values, clipped to the host bound)
  int n_max = 0, n_vis = 0;
  for (int i = 0; i < p.n_q; ++i) {
    int v = p.steps[static_cast<int64_t>(b) * p.n_q + i];
    if (v < 0 || v > p.max_seq_len) {
      if (threadIdx.x == 0 && split == 0 && g == 0) record_status(p.status, K8V4_ERANGE);
      v = v < 0 ? 0 : p.max_seq_len;
    }
    n_max = max(n_max, v);
    if (i == qi) n_vis = v;
  }
  const int c_begin = split * p.cells_per_split;
  const int c_stop = c_begin + p.cells_per_split;
  const int c_end = min(c_stop, n_max);
  const int n_tiles = c_end > c_begin ? (c_end - c_begin + 15) >> 4 : 0;
  const int lim = min(n_vis, c_stop);       // this query's cells in this split end here

  // ---- fused decode step: the CTA whose cells include the newest one (n_vis - 1)
  // appends the new token's K and V there before any warp stages a tile
  if (NQ1 && p.k_new != nullptr) {
    const int cell = n_vis - 1;
    const int raw_len = p.steps[b];
    if (cell >= c_begin && cell < c_stop && raw_len == n_vis) {   // skipped for a clipped length
      if (warp < 2) {
        const int64_t pidx = cell / C.P;
        const int64_t page = pidx < p.max_pages ? p.pt[static_cast<int64_t>(b) * p.max_pages + pidx] : -1;
        if (page >= 0 && page < C.n_pages) {
          uint8_t* base = C.pages + page * C.page_bytes;
          const int64_t r = static_cast<int64_t>(cell % C.P) * C.H + g;
          const int64_t elem = (static_cast<int64_t>(b) * C.H + g) * kD + 8 * lane;
          // each warp's rotation scratch (the pipeline has not started)
          long long* ts = reinterpret_cast<long long*>(smem) + warp * kRotScratch;
          if (warp == 0) {
            if (p.kv_bf16) append_k_row<true, FMT>(C, base, r, p.k_new, elem, lane, ts);
            else append_k_row<false, FMT>(C, base, r, p.k_new, elem, lane, ts);
          } else {
            if (p.kv_bf16) append_v_row<true, FMT>(C, base, r, p.v_new, elem, lane, ts);
            else append_v_row<false, FMT>(C, base, r, p.v_new, elem, lane, ts);
          }
        } else if (warp == 0 && lane == 0) {
          record_status(p.status, K8V4_ERANGE);
        }
      }
      __syncthreads();                      // the new cell's bytes are visible to every warp's copies
    }
  }

  // ---- q fragments (B operand of QK^T).  Int8 K: lane holds head r0, dims
  // 64i + 16c + 4j + e (k-step 4i + j).  Q4 K: the rotated query (H/16) q, dims
  // 32 blk + 16 hf + 4c + e (k-step 2 blk + hf) -- the dims of the nibble bytes
  // 4c .. 4c+3 of block blk that ldmatrix hands this lane
  uint32_t qf[16][2];
  uint32_t qf_lo[kLo ? 16 : 1][2];
  float fscale;                                    // per head: sm_scale * log2(e) / 2^qexp
  {
    const int64_t qrow = ((static_cast<int64_t>(b) * p.n_q + qi) * HQ + g * kGqa + r0) * kD;
    float qv[64];
    if (kQ4) {
      // qv[8 blk + 4 hf + e] = q[32 blk + 16 hf + 4c + e]
#pragma unroll
      for (int t4 = 0; t4 < 16; ++t4) {
        const int64_t e0 = qrow + 16 * t4 + 4 * c;
        if (QF32) {
          const float4 v4 = *reinterpret_cast<const float4*>(static_cast<const float*>(p.q) + e0);
          qv[4 * t4] = v4.x; qv[4 * t4 + 1] = v4.y; qv[4 * t4 + 2] = v4.z; qv[4 * t4 + 3] = v4.w;
        } else {
          const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.q) + e0);
          qv[4 * t4] = __uint_as_float(raw.x << 16);
          qv[4 * t4 + 1] = __uint_as_float(raw.x & 0xffff0000u);
          qv[4 * t4 + 2] = __uint_as_float(raw.y << 16);
          qv[4 * t4 + 3] = __uint_as_float(raw.y & 0xffff0000u);
        }
      }
      // (H/16) q: a butterfly per index bit -- the six in-register bits of t
      // (dims bits 0, 1, 4, 5, 6, 7), then lane bits 0 and 1 (dims bits 2, 3)
#pragma unroll
      for (int hb = 1; hb < 64; hb <<= 1) {
#pragma unroll
        for (int t = 0; t < 64; ++t) {
          if (t & hb) continue;
          const float x0 = qv[t], x1 = qv[t + hb];
          qv[t] = x0 + x1;
          qv[t + hb] = x0 - x1;
        }
      }
#pragma unroll
      for (int m = 1; m <= 2; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int t = 0; t < 64; ++t) {
          const float o2 = __shfl_xor_sync(kFull, qv[t], m);
          qv[t] = upper ? o2 - qv[t] : qv[t] + o2;
        }
      }
#pragma unroll
      for (int t = 0; t < 64; ++t) qv[t] *= 0.0625f;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t e0 = qrow + 64 * i + 16 * c;
        if (QF32) {
          const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.q) + e0);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float4 v4 = src[t];
            qv[16 * i + 4 * t] = v4.x; qv[16 * i + 4 * t + 1] = v4.y;
            qv[16 * i + 4 * t + 2] = v4.z; qv[16 * i + 4 * t + 3] = v4.w;
          }
        } else {
          const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + e0);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint4 raw = src[t];
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              qv[16 * i + 8 * t + 2 * u] = __uint_as_float(w[u] << 16);
              qv[16 * i + 8 * t + 2 * u + 1] = __uint_as_float(w[u] & 0xffff0000u);
            }
          }
        }
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int t = 0; t < 64; ++t) amax = fmaxf(amax, fabsf(qv[t]));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    int ex = amax > 0.0f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127 : 0;
    int sh = 14 - ex;                               // amax * 2^sh in [2^14, 2^15)
    sh = max(-100, min(100, sh));
    const float up = ldexpf(1.0f, sh);
    fscale = p.sm_scale_log2 * ldexpf(1.0f, -sh);
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      // b0 = (k 2c, 2c+1), b1 = (k 2c+8, 2c+9): int8 K dims o+0, o+1 | o+2, o+3;
      // Q4 K (bytes 4c, 4c+2 | 4c+1, 4c+3 of the block) dims o+0, o+2 | o+1, o+3
      const int o = kQ4 ? 4 * ks : 16 * (ks >> 2) + 4 * (ks & 3);
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = __fmul_rn(qv[o + (kQ4 ? ((e & 1) << 1) | (e >> 1) : e)], up);
      const __half2 h0 = __floats2half2_rn(v[0], v[1]), h1 = __floats2half2_rn(v[2], v[3]);
      qf[ks][0] = *reinterpret_cast<const uint32_t*>(&h0);
      qf[ks][1] = *reinterpret_cast<const uint32_t*>(&h1);
      if (kLo) {
        const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
        const __half2 l0 = __floats2half2_rn(v[0] - f0.x, v[1] - f0.y);
        const __half2 l1 = __floats2half2_rn(v[2] - f1.x, v[3] - f1.y);
        qf_lo[ks % (kLo ? 16 : 1)][0] = *reinterpret_cast<const uint32_t*>(&l0);
        qf_lo[ks % (kLo ? 16 : 1)][1] = *reinterpret_cast<const uint32_t*>(&l1);
      }
    }
  }
  // score factors for the heads of the C layout (2c, 2c+1): held by lanes 4h
  const float f0 = __shfl_sync(kFull, fscale, 8 * c), f1 = __shfl_sync(kFull, fscale, 8 * c + 4);

  float o[kMT][4];
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;

  // ---- pipeline over this group's tiles: gi, gi + n_groups, ...
  uint8_t* gbuf = smem + static_cast<size_t>(gi) * kStages * S::kBytes;
  const uint32_t gbuf_s = smem_u32(gbuf);
  const int n_my = n_tiles > gi ? (n_tiles - gi + p.n_groups - 1) / p.n_groups : 0;
  const int tid = qi * 32 + lane, nthr = NQ1 ? 32 : p.n_q * 32;
  // load cursor: page index and slot of the next tile to stage (advanced, never divided again)
  const int step = 16 * p.n_groups;
  int64_t lp = 0;
  int ls = 0;
  {
    const int cell = c_begin + 16 * gi;
    lp = cell / C.P;
    ls = cell - static_cast<int>(lp) * C.P;
  }
  const int32_t* pt_row = p.pt + static_cast<int64_t>(b) * p.max_pages;
  uint32_t vmask = 0;                          // bit s: stage s holds a valid tile
  // the page id of the next tile to stage is read one issue ahead, so the
  // global-load latency hides behind a tile of compute
  int64_t nxt_page = (n_my > 0 && lp < p.max_pages) ? pt_row[lp] : -1;
  auto issue = [&](int stage) {
    const int64_t page = nxt_page;
    if (page >= 0 && page < C.n_pages) {
      load_tile<FMT, NQ1 ? 32 : 0>(C, gbuf_s + stage * S::kBytes, C.pages + page * C.page_bytes, ls, g, tid, nthr);
      vmask |= 1u << stage;
    } else {
      vmask &= ~(1u << stage);
      if (tid == 0) record_status(p.status, K8V4_ERANGE);
    }
    ls += step;
    while (ls >= C.P) { ls -= C.P; ++lp; }
    nxt_page = lp < p.max_pages ? pt_row[lp] : -1;
  };
#pragma unroll 1
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < n_my) issue(s);
    cp_async_commit();
  }
#pragma unroll 1
  for (int it = 0; it < n_my; ++it) {
    const int cur = it % kStages;
    cp_async_wait<kStages - 2>();
    if (NQ1 || nthr == 32) __syncwarp();   // a one-warp group needs no CTA barrier
    else named_barrier(1 + gi, nthr);
    {
      const int nx = it + kStages - 1;
      if (nx < n_my) issue(nx % kStages);
      cp_async_commit();
    }
    const int cell0 = c_begin + 16 * (gi + it * p.n_groups);
    if (!((vmask >> cur) & 1u) || cell0 >= lim) continue;      // nothing visible for this query
    const uint8_t* st = gbuf + cur * S::kBytes;
    const uint32_t st_s = smem_u32(st);

    // ---- QK^T: S^T[cell][head]
    const bool vA = cell0 + r0 < lim, vB = cell0 + r0 + 8 < lim;
    float sc[4];
    if (kQ4) {
      // rotated K nibbles: per 32-lane block a fresh accumulator over its two
      // k-steps (low nibbles: block dims 0-15, high: 16-31) and both q terms,
      // then scaled by the cell's d of that block
      const uint4 dA4 = lds128(st_s + S::kKs + 16 * r0), dB4 = lds128(st_s + S::kKs + 16 * (r0 + 8));
      const uint32_t dAw[4] = {dA4.x, dA4.y, dA4.z, dA4.w}, dBw[4] = {dB4.x, dB4.y, dB4.z, dB4.w};
      float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const int mi = lane >> 3, rr = lane & 7;
      const int lcell = rr + 8 * (mi & 1);
#pragma unroll
      for (int bp = 0; bp < 8; bp += 2) {
        uint32_t R[4];
        ldmatrix_x4(R, st_s + S::kK + lcell * 128 + 16 * ((bp + (mi >> 1)) ^ (lcell & 7)));
        uint32_t alo[2][4], ahi[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {   // R[2h], R[2h + 1]: cells r0, r0 + 8, bytes 4c .. 4c+3
          nibs_to_f16(R[2 * h], alo[h][0], alo[h][2], ahi[h][0], ahi[h][2]);
          nibs_to_f16(R[2 * h + 1], alo[h][1], alo[h][3], ahi[h][1], ahi[h][3]);
        }
        float acc[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.0f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int ks = 2 * (bp + h) + hf;
            mma_f16(acc[h], hf ? ahi[h] : alo[h], qf[ks][0], qf[ks][1]);
            mma_f16(acc[h], hf ? ahi[h] : alo[h], qf_lo[ks % (kLo ? 16 : 1)][0], qf_lo[ks % (kLo ? 16 : 1)][1]);
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int blk = bp + h;
          uint32_t wa = dAw[blk >> 1], wb = dBw[blk >> 1];
          const float2 fa = __half22float2(*reinterpret_cast<__half2*>(&wa));
          const float2 fb = __half22float2(*reinterpret_cast<__half2*>(&wb));
          const float da = (blk & 1) ? fa.y : fa.x, db = (blk & 1) ? fb.y : fb.x;
          s4[0] = fmaf(da, acc[h][0], s4[0]);
          s4[1] = fmaf(da, acc[h][1], s4[1]);
          s4[2] = fmaf(db, acc[h][2], s4[2]);
          s4[3] = fmaf(db, acc[h][3], s4[3]);
        }
      }
      sc[0] = vA ? s4[0] * f0 : -INFINITY;
      sc[1] = vA ? s4[1] * f1 : -INFINITY;
      sc[2] = vB ? s4[2] * f0 : -INFINITY;
      sc[3] = vB ? s4[3] * f1 : -INFINITY;
    } else {
      // int8 K: the two 128-lane halves accumulated separately (two
      // accumulators per half keep four independent MMA chains in flight)
      float acc[4][4];
#pragma unroll
      for (int t = 0; t < 4; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 ka = lds128(st_s + S::kK + r0 * 256 + 16 * ((4 * i + c) ^ ((r0 & 1) << 2)));
        const uint4 kb = lds128(st_s + S::kK + (r0 + 8) * 256 + 16 * ((4 * i + c) ^ ((r0 & 1) << 2)));
        const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb.x, kb.y, kb.z, kb.w};
        uint32_t a[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          codes_to_f16(wa[j], a[j][0], a[j][2]);
          codes_to_f16(wb[j], a[j][1], a[j][3]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float* dst = acc[2 * (i >> 1) + (j & 1)];
          mma_f16(dst, a[j], qf[4 * i + j][0], qf[4 * i + j][1]);
          if (QF32) mma_f16(dst, a[j], qf_lo[(4 * i + j) % (kLo ? 16 : 1)][0], qf_lo[(4 * i + j) % (kLo ? 16 : 1)][1]);
        }
      }
      float a0[4], a1[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        a0[t] = acc[0][t] + acc[1][t];
        a1[t] = acc[2][t] + acc[3][t];
      }
      const float2 kA = *reinterpret_cast<const float2*>(st + S::kKs + 8 * r0);
      const float2 kB = *reinterpret_cast<const float2*>(st + S::kKs + 8 * (r0 + 8));
      sc[0] = vA ? (kA.x * a0[0] + kA.y * a1[0]) * f0 : -INFINITY;
      sc[1] = vA ? (kA.x * a0[1] + kA.y * a1[1]) * f1 : -INFINITY;
      sc[2] = vB ? (kB.x * a0[2] + kB.y * a1[2]) * f0 : -INFINITY;
      sc[3] = vB ? (kB.x * a0[3] + kB.y * a1[3]) * f1 : -INFINITY;
    }

    // ---- online softmax (heads 2c, 2c+1)
    float t0 = fmaxf(sc[0], sc[2]), t1 = fmaxf(sc[1], sc[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      t0 = fmaxf(t0, __shfl_xor_sync(kFull, t0, off));
      t1 = fmaxf(t1, __shfl_xor_sync(kFull, t1, off));
    }
    const float mn0 = fmaxf(m0, t0), mn1 = fmaxf(m1, t1);   // finite: cell0 is visible
    const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
    float pr[4];
    pr[0] = ex2(sc[0] - mn0);
    pr[1] = ex2(sc[1] - mn1);
    pr[2] = ex2(sc[2] - mn0);
    pr[3] = ex2(sc[3] - mn1);
    l0 = l0 * al0 + (pr[0] + pr[2]);
    l1 = l1 * al1 + (pr[1] + pr[3]);
    m0 = mn0;
    m1 = mn1;
    if (__any_sync(kFull, al0 != 1.0f || al1 != 1.0f)) {
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        const float2 al = make_float2(al0, al1);
        const float2 x = __fmul2_rn(make_float2(o[mt][0], o[mt][1]), al);
        const float2 y = __fmul2_rn(make_float2(o[mt][2], o[mt][3]), al);
        o[mt][0] = x.x; o[mt][1] = x.y; o[mt][2] = y.x; o[mt][3] = y.y;
      }
    }

    // ---- transpose p to the B layout: lane gets head r0, cells 2c, 2c+1, 2c+8, 2c+9
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
    const int pc[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
    const float2 P01 = make_float2(P[0], P[1]), P23 = make_float2(P[2], P[3]);

    // ---- PV in rotated space
    if (FMT != K8V4_FORMAT_INT8) {
      uint4 dv[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) dv[t] = *reinterpret_cast<const uint4*>(st + S::kVs + 16 * pc[t]);
      const int mi = lane >> 3, rr = lane & 7;
      const int lcell = rr + 8 * (mi & 1);
#pragma unroll
      for (int bp = 0; bp < 8; bp += 2) {
        uint32_t R[4];
        ldmatrix_x4_t(R, st_s + S::kV + lcell * 128 + 16 * ((bp + (mi >> 1)) ^ (lcell & 7)));
        uint32_t B[2][kPlanes][2];
        uint32_t alo[2][4], ahi[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int bl = bp + h;
          // d of block bl for cells (2c, 2c+1) and (2c+8, 2c+9), as fp16 pairs
          const uint32_t sel = (bl & 1) ? 0x7632u : 0x5410u;
          const uint32_t wA = (bl >> 1) == 0 ? dv[0].x : (bl >> 1) == 1 ? dv[0].y : (bl >> 1) == 2 ? dv[0].z : dv[0].w;
          const uint32_t wB = (bl >> 1) == 0 ? dv[1].x : (bl >> 1) == 1 ? dv[1].y : (bl >> 1) == 2 ? dv[1].z : dv[1].w;
          const uint32_t wC = (bl >> 1) == 0 ? dv[2].x : (bl >> 1) == 1 ? dv[2].y : (bl >> 1) == 2 ? dv[2].z : dv[2].w;
          const uint32_t wD = (bl >> 1) == 0 ? dv[3].x : (bl >> 1) == 1 ? dv[3].y : (bl >> 1) == 2 ? dv[3].z : dv[3].w;
          uint32_t d01 = prmt(wA, wB, sel), d23 = prmt(wC, wD, sel);
          float2 x01 = __fmul2_rn(P01, __half22float2(*reinterpret_cast<__half2*>(&d01)));
          float2 x23 = __fmul2_rn(P23, __half22float2(*reinterpret_cast<__half2*>(&d23)));
#pragma unroll
          for (int pl = 0; pl < kPlanes; ++pl) {
            B[h][pl][0] = pack_bf16(x01.x, x01.y);
            B[h][pl][1] = pack_bf16(x23.x, x23.y);
            if (pl + 1 < kPlanes) {   // exact residuals: x - bf16(x)
              x01 = __ffma2_rn(make_float2(bf16_lo(B[h][pl][0]), bf16_hi(B[h][pl][0])), make_float2(-1.0f, -1.0f), x01);
              x23 = __ffma2_rn(make_float2(bf16_lo(B[h][pl][1]), bf16_hi(B[h][pl][1])), make_float2(-1.0f, -1.0f), x23);
            }
          }
          const uint32_t Ra = R[2 * h], Rb = R[2 * h + 1];
          alo[h][0] = nib_to_bf16(Ra, 0); alo[h][1] = nib_to_bf16(Ra, 8);
          alo[h][2] = nib_to_bf16(Rb, 0); alo[h][3] = nib_to_bf16(Rb, 8);
          ahi[h][0] = nib_to_bf16(Ra, 4); ahi[h][1] = nib_to_bf16(Ra, 12);
          ahi[h][2] = nib_to_bf16(Rb, 4); ahi[h][3] = nib_to_bf16(Rb, 12);
        }
#pragma unroll
        for (int pl = 0; pl < kPlanes; ++pl) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            mma_bf16(o[2 * (bp + h)], alo[h], B[h][pl][0], B[h][pl][1]);
            mma_bf16(o[2 * (bp + h) + 1], ahi[h], B[h][pl][0], B[h][pl][1]);
          }
        }
      }
    } else {
      float sv[4][2];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 v2 = *reinterpret_cast<const float2*>(st + S::kVs + 8 * pc[t]);
        sv[t][0] = v2.x;
        sv[t][1] = v2.y;
      }
      const int mi = lane >> 3, rr = lane & 7;
      const int lcell = rr + 8 * (mi & 1);
#pragma unroll
      for (int half = 0; half < kBlocks; ++half) {
        float x[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) x[t] = P[t] * sv[t][half];
        uint32_t B[kPlanes][2];
#pragma unroll
        for (int pl = 0; pl < kPlanes; ++pl) {
          B[pl][0] = pack_bf16(x[0], x[1]);
          B[pl][1] = pack_bf16(x[2], x[3]);
          if (pl + 1 < kPlanes) {
            x[0] -= bf16_lo(B[pl][0]); x[1] -= bf16_hi(B[pl][0]);
            x[2] -= bf16_lo(B[pl][1]); x[3] -= bf16_hi(B[pl][1]);
          }
        }
#pragma unroll
        for (int mp = 0; mp < 8; mp += 2) {
          const int mt0 = 8 * half + mp;
          uint32_t R[4];
          ldmatrix_x4_t(R, st_s + S::kV + lcell * 256 + 16 * ((mt0 + (mi >> 1)) ^ (lcell & 7)));
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t Ra = R[2 * h], Rb = R[2 * h + 1];
            uint32_t a[4] = {i8_to_bf16(Ra, 0x7540u, 0x7542u), i8_to_bf16(Ra, 0x7541u, 0x7543u),
                             i8_to_bf16(Rb, 0x7540u, 0x7542u), i8_to_bf16(Rb, 0x7541u, 0x7543u)};
#pragma unroll
            for (int pl = 0; pl < kPlanes; ++pl) mma_bf16(o[mt0 + h], a, B[pl][0], B[pl][1]);
          }
        }
      }
    }
  }
  cp_async_wait<0>();

  // ---- finish: row sums across the 8 lanes of each head, then the CTA merge
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, off);
    l1 += __shfl_xor_sync(kFull, l1, off);
  }
  __syncthreads();
  float* mo = reinterpret_cast<float*>(smem);                 // [warps][8 * 256 + 16]
  constexpr int kWS = 8 * 256 + 16;
  float* mine = mo + static_cast<size_t>(warp) * kWS;
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt) {
    int d0;
    if (FMT != K8V4_FORMAT_INT8) d0 = 32 * (mt >> 1) + 16 * (mt & 1) + 2 * r0;
    else d0 = 16 * mt + 2 * r0;
    *reinterpret_cast<float2*>(mine + (2 * c) * 256 + d0) = make_float2(o[mt][0], o[mt][2]);
    *reinterpret_cast<float2*>(mine + (2 * c + 1) * 256 + d0) = make_float2(o[mt][1], o[mt][3]);
  }
  if (r0 == 0) {
    mine[2048 + 2 * c] = m0;
    mine[2048 + 2 * c + 1] = m1;
    mine[2056 + 2 * c] = l0;
    mine[2056 + 2 * c + 1] = l1;
  }
  __syncthreads();
  // one warp per output row (query, head): merge the tile groups, bring the
  // partial back from rotated space (out = (H/16) o is linear, so the split
  // combine can work on un-rotated partials) and write (o, m, l)
  const int n_rows = p.n_q * kGqa;
  for (int rr = warp; rr < n_rows; rr += blockDim.x >> 5) {
    const int q2 = rr >> 3, h = rr & 7;
    float M = -INFINITY;
    for (int gg = 0; gg < p.n_groups; ++gg) M = fmaxf(M, mo[static_cast<size_t>(gg * p.n_q + q2) * kWS + 2048 + h]);
    float v[8], L = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.0f;
    if (M != -INFINITY) {
      for (int gg = 0; gg < p.n_groups; ++gg) {
        const float* src = mo + static_cast<size_t>(gg * p.n_q + q2) * kWS;
        const float mg = src[2048 + h];
        if (mg == -INFINITY) continue;
        const float sc2 = exp2f(mg - M);
        const float4 x0 = *reinterpret_cast<const float4*>(src + h * 256 + 8 * lane);
        const float4 x1 = *reinterpret_cast<const float4*>(src + h * 256 + 8 * lane + 4);
        v[0] += x0.x * sc2; v[1] += x0.y * sc2; v[2] += x0.z * sc2; v[3] += x0.w * sc2;
        v[4] += x1.x * sc2; v[5] += x1.y * sc2; v[6] += x1.z * sc2; v[7] += x1.w * sc2;
        L += src[2056 + h] * sc2;
      }
    }
    if (FMT != K8V4_FORMAT_INT8) {
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
          const float t = __shfl_xor_sync(kFull, v[e], m);
          v[e] = upper ? t - v[e] : v[e] + t;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] *= 0.0625f;
    }
    float* dst = p.ws + ((((static_cast<int64_t>(b) * p.splits + split) * p.n_q + q2) * HQ) + g * kGqa + h) * kPStride;
    reinterpret_cast<float4*>(dst + 8 * lane)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst + 8 * lane)[1] = make_float4(v[4], v[5], v[6], v[7]);
    if (lane == 0) {
      dst[256] = M;
      dst[257] = L;
    }
  }
  // the combine kernel may start once every partial of this grid is written
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int FMT, bool QF32, bool NQ1>
int launch_impl(const Launch& L, const AttendParams& p, const AttendPlan& plan, float* out) {
  const size_t stage_bytes = static_cast<size_t>(plan.n_groups) * kStages * Stage<FMT>::kBytes;
  const size_t merge_bytes = static_cast<size_t>(plan.warps) * (8 * 256 + 16) * sizeof(float);
  const size_t smem = stage_bytes > merge_bytes ? stage_bytes : merge_bytes;
  auto kern = attend_splitk_kernel<FMT, QF32, NQ1>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return K8V4_ECUDA;
  // programmatic dependent launch: the CTAs are placed while the previous kernel
  // (the new token's append) finishes; the kernel's first act is griddepcontrol.wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.splits, p.C.H, p.n_seqs);
  cfg.blockDim = dim3(plan.warps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return K8V4_ECUDA;
  if (cudaGetLastError() != cudaSuccess) return K8V4_ECUDA;
  return launch_combine(L, p.ws, plan.splits, p.n_seqs, p.n_q, p.C.H, out);
}

}  // namespace

namespace {
AttendPlan plan_attend_base(const CacheView& C, int n_seqs, int n_q, int max_seq_len, int num_sms) {
  // several queries per sequence over a k8v4 cache: tiles dequantised once and
  // shared by all queries -- on the tcgen05 kernel (bf16 q, pages of 64k cells)
  // or on the warp-MMA verify kernel; the workspace covers either
  if (n_q > 1 && C.fmt == K8V4_FORMAT_K8V4) {
    // bf16 queries run the tcgen05 prefill kernel split over cells (pages of a
    // multiple of 64 cells) or the team-of-warps TMA kernel, fp32 queries the
    // warp-MMA one; the workspace covers each
    AttendPlan mw = plan_verify(C, n_seqs, n_q, max_seq_len, num_sms);
    if (verify_ws_supported(C, n_q, K8V4_BF16))
      mw.ws_bytes = std::max(mw.ws_bytes, plan_verify_ws(C, n_seqs, n_q, max_seq_len, num_sms).ws_bytes);
    if (C.P % 64 == 0)
      mw.ws_bytes = std::max(mw.ws_bytes, plan_verify_tc(C, n_seqs, n_q, max_seq_len, num_sms).ws_bytes);
    return mw;
  }
  if (n_q == 1 && decode_ws_supported(C)) return plan_decode(C, n_seqs, max_seq_len, num_sms);
  AttendPlan pl{};
  pl.n_q = n_q;
  pl.n_groups = n_q >= kWarps ? 1 : kWarps / n_q;
  if (n_q > 1 && pl.n_groups > 15) pl.n_groups = 15;   // named barriers 1..15
  pl.warps = pl.n_groups * n_q;
  const int tiles = max(1, (max_seq_len + 15) / 16);
  const int stage_bytes = pl.n_groups * kStages * stage_bytes_of(C.fmt);
  const int ctas_per_sm = max(1, min(4, (200 * 1024) / max(stage_bytes, 1)));
  const int64_t pairs = static_cast<int64_t>(C.H) * n_seqs;
  const int64_t target = static_cast<int64_t>(num_sms) * ctas_per_sm;
  // at most one wave (one CTA per SM slot): a second, partly filled wave of
  // smaller CTAs measured slower than fewer, longer CTAs (each CTA pays its q
  // setup, pipeline fill and merge epilogue once)
  const int64_t max_splits = std::max(1, tiles / (2 * pl.n_groups));
  int64_t splits = std::max<int64_t>(1, std::min<int64_t>(target / pairs, max_splits));
  const int tps = static_cast<int>((tiles + splits - 1) / splits);
  pl.cells_per_split = 16 * tps;
  pl.splits = (tiles + tps - 1) / tps;
  pl.ws_bytes = static_cast<size_t>(n_seqs) * pl.splits * n_q * C.H * kGqa * kPStride * sizeof(float);
  return pl;
}

}  // namespace

AttendPlan plan_attend(const CacheView& C, int n_seqs, int n_q, int max_seq_len, int num_sms) {
  return plan_attend_base(C, n_seqs, n_q, max_seq_len, num_sms);
}

int launch_attend(const Launch& L, const CacheView& C, const AttendPlan& plan, const void* q, int q_dtype,
                  const int32_t* pt, int64_t max_pages, const int32_t* steps, int n_seqs, int max_seq_len,
                  float sm_scale, float* out, void* ws, const void* k_new, const void* v_new, int kv_dtype) {
  if (n_seqs == 0) return K8V4_OK;
  if (plan.n_q > 1 && C.fmt == K8V4_FORMAT_K8V4) {
    if (q_dtype == K8V4_BF16 && C.P % 64 == 0) {
      const AttendPlan tp = plan_verify_tc(C, n_seqs, plan.n_q, max_seq_len, L.num_sms);
      return launch_verify_tc(L, C, tp, q, pt, max_pages, steps, n_seqs, max_seq_len, sm_scale, out, ws);
    }
    if (verify_ws_supported(C, plan.n_q, q_dtype))
      return launch_verify_ws(L, C, q, pt, max_pages, steps, n_seqs, plan.n_q, max_seq_len, sm_scale, out, ws);
    const AttendPlan mw = plan_verify(C, n_seqs, plan.n_q, max_seq_len, L.num_sms);
    return launch_verify(L, C, mw, q, q_dtype, pt, max_pages, steps, n_seqs, max_seq_len, sm_scale, out, ws);
  }
  if (plan.n_q == 1 && decode_ws_supported(C))
    return launch_decode(L, C, plan, q, q_dtype, pt, max_pages, steps, n_seqs, max_seq_len, sm_scale, out, ws,
                         k_new, v_new, kv_dtype, wait_limit_ns());
  AttendParams p;
  p.C = C;
  p.q = q;
  p.pt = pt;
  p.max_pages = max_pages;
  p.steps = steps;
  p.n_seqs = n_seqs;
  p.n_q = plan.n_q;
  p.n_groups = plan.n_groups;
  p.max_seq_len = max_seq_len;
  p.cells_per_split = plan.cells_per_split;
  p.splits = plan.splits;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.ws = static_cast<float*>(ws);
  p.status = L.status;
  p.k_new = k_new;
  p.v_new = v_new;
  p.kv_bf16 = kv_dtype == K8V4_BF16 ? 1 : 0;
  const bool f32 = q_dtype == K8V4_F32, one = plan.n_q == 1;
  if (C.fmt == K8V4_FORMAT_K8V4) {
    // k8v4 with n_q > 1 left above; here n_q == 1
    return f32 ? launch_impl<K8V4_FORMAT_K8V4, true, true>(L, p, plan, out)
               : launch_impl<K8V4_FORMAT_K8V4, false, true>(L, p, plan, out);
  }
  if (C.fmt == K8V4_FORMAT_Q4) {
    if (f32) return one ? launch_impl<K8V4_FORMAT_Q4, true, true>(L, p, plan, out)
                        : launch_impl<K8V4_FORMAT_Q4, true, false>(L, p, plan, out);
    return one ? launch_impl<K8V4_FORMAT_Q4, false, true>(L, p, plan, out)
               : launch_impl<K8V4_FORMAT_Q4, false, false>(L, p, plan, out);
  }
  if (f32) return one ? launch_impl<K8V4_FORMAT_INT8, true, true>(L, p, plan, out)
                      : launch_impl<K8V4_FORMAT_INT8, true, false>(L, p, plan, out);
  return one ? launch_impl<K8V4_FORMAT_INT8, false, true>(L, p, plan, out)
             : launch_impl<K8V4_FORMAT_INT8, false, false>(L, p, plan, out);
}

}  // namespace k8v4
