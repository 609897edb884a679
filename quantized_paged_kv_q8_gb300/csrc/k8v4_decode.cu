// Split-K decode attention over the k8v4 cache (and the INT8 comparison cache):
// one query (the 8 query heads of a KV head) per sequence, optionally fused with
// the append of the sequence's newest token.  This is the decode "mode 3"
// attention of the hybrid-KV pull request ("How": the K loader takes the int8
// branch, the V loop the q4 branch, q is not rotated and the output is rotated
// back; "Tests": the step form against a host attention over the same
// dequantised K/V).
//
// GB300 design.  A CTA owns one (sequence, KV head, cell range); its W worker
// warps take the range's 16-cell tiles round robin (worker w: tiles w, w + W,
// ...), and each worker runs its tiles start to finish with no hand-off:
//   - one elected lane issues the TMA copies of the worker's next tile -- K codes
//     (two 128-byte-swizzled boxes), V nibbles (one box), and the K and V scale
//     runs (plain bulk copies) -- into the worker's own two-stage ring, so a
//     tile's loads fly while the previous tile is computed;
//   - QK: K codes -> fp16 in registers, S^T = K q^T on mma.sync m16n8k16
//     (cells x 8 heads), the two per-half K scales;
//   - softmax against a per-head reference ref = 8 B, B = the running maximum
//     over the worker's tiles of the integer bucket ceil(max / 8): p' = 2^(s -
//     ref + 14) <= 2^14, and the accumulators are rescaled by an exact power of
//     two only when B rises (rare after the first tiles); the sums stay per lane
//     until the end;
//   - PV: p' in two fp16 terms transposed to the MMA B layout in registers; V
//     nibbles -> (n - 8)/8 in fp16 (exact), times the block's fp16 scale d as two
//     exact fp16 terms (the product has at most 15 significant bits); O += V^hat
//     p' as three MMAs (hi.hi + hi.lo + lo.hi) per 16-dim m-tile, in rotated
//     space.  The INT8 format's V (per-half fp32 scale) instead multiplies p' by
//     the scale in fp32 and carries the product in three bf16 terms.
// Every warp runs the same code, so the instruction cache holds one loop.  The
// epilogue merges the workers' partials (exact power-of-two rescaling to the
// largest bucket), brings each row back from rotated space (out = (H/16) o is
// linear) and writes (o, m, l) for the split combine.  The result depends on the
// data alone, not on the order in which warps run.
//
// Every mbarrier wait is bounded in time (1 s by default; the launch can pass
// another bound): on timeout the warp records K8V4_ECUDA and raises the CTA's
// abort flag so that the other warps stop too, and each warp waits (bounded)
// for the copies it issued before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "k8v4_quant.cuh"

namespace k8v4 {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxWorkers = 12;                        // worker warps per CTA (bf16 queries)
constexpr int kMaxWorkersF32 = 8;                      // fp32 queries carry twice the q registers
constexpr int kPStride = 260;                          // floats per partial row: o[256], m, l, 2 pad
constexpr uint32_t kWaitDefaultNs = 1000000000u;       // 1 s
constexpr int kBucketClamp = 1 << 24;
constexpr int kSmemCap = 227 * 1024;
// A worker's partial in the epilogue: [8 heads][kHeadStride] floats of o, then 8
// buckets and 8 sums.  A head stride of 4 mod 16 floats puts the four lane
// groups of one fragment store in four different bank octets.
constexpr int kHeadStride = 260;
constexpr int kPartBucket = 8 * kHeadStride;
constexpr int kPartSum = kPartBucket + 8;
constexpr int kPartFloats = kPartSum + 8;

// Shared-memory layout of one CTA (offsets from the 1024-aligned base): per
// worker two stages of [K 4096][V][K scales][V scales], then the mbarriers.
struct Layout {
  int workers;
  int v_bytes, ksc_bytes, vsc_bytes;
  int v_off, ksc_off, vsc_off;      // within a stage
  int stage_bytes;                  // a multiple of 1024 (the swizzled boxes)
  int tx_bytes;                     // bytes the copies of one stage deliver
  int bar_off;
  int total;                        // dynamic shared memory to request (with alignment slack)
};

inline Layout layout_of(int fmt, int H, int max_workers) {
  Layout L;
  const bool i8 = fmt == K8V4_FORMAT_INT8;
  L.v_bytes = i8 ? 4096 : 2048;
  L.ksc_bytes = 128 * H;                          // [16 cells][H][2] f32
  L.vsc_bytes = i8 ? 128 * H : 256 * H;           // [16][H][2] f32 or [16][H][8] f16
  L.v_off = 4096;
  L.ksc_off = L.v_off + L.v_bytes;
  L.vsc_off = L.ksc_off + L.ksc_bytes;
  L.stage_bytes = (L.vsc_off + L.vsc_bytes + 1023) & ~1023;
  // a worker's partial (kPartFloats floats) goes into its own two stages
  L.stage_bytes = std::max(L.stage_bytes, (kPartFloats * 2 + 1023) & ~1023);
  L.tx_bytes = 4096 + L.v_bytes + L.ksc_bytes + L.vsc_bytes;
  for (L.workers = max_workers; L.workers > 1; --L.workers) {
    L.bar_off = L.workers * 2 * L.stage_bytes;
    L.total = L.bar_off + 16 * L.workers + 16 + 1024;
    if (L.total <= kSmemCap) break;
  }
  L.bar_off = L.workers * 2 * L.stage_bytes;
  L.total = L.bar_off + 16 * L.workers + 16 + 1024;
  return L;
}

struct DecodeParams {
  CacheView C;
  const void* q;
  const int32_t* pt;
  int64_t max_pages;
  const int32_t* steps;
  int max_seq_len, cells_per_split, splits;
  int cell_base, cell_limit;  // the cell range the splits cover: [cell_base, cell_limit)
  float sm_scale_log2;
  float* ws;
  int* status;
  const void* k_new;      // fused decode step: the new token's K and V [n_seqs][H][256], else null
  const void* v_new;
  int kv_bf16;
  uint32_t wait_ns;       // bound of every mbarrier wait, nanoseconds
  int withhold;           // diagnostics: worker 0 of CTA (0, 0, 0) never issues its tile 0
  FastDiv page_div;       // division by the page size P
  Layout L;
};
// ---------------------------------------------------------------- PTX wrappers
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
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float2 lds64f(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}
// two fp32 -> bf16x2 (round to nearest even); `lo` lands in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 2^e exactly for e >= -126, 0 below
__device__ __forceinline__ float pow2i(int e) { return e < -126 ? 0.0f : __int_as_float((e + 127) << 23); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// one non-blocking test of the phase
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// One poll that may suspend the thread for up to `ns` nanoseconds (it resumes as
// soon as the phase completes).
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of parity `parity`: false once `limit_ns` nanoseconds have
// passed without it, or once the CTA's abort flag is up.  A waiting warp sleeps
// in the barrier instead of spinning, so it takes no issue slots from the warps
// that do the work.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit_ns, const volatile int* abort) {
  if (mbar_try(bar, parity)) return true;
  if (limit_ns < 1000u) return false;        // a bound under 1 us: one poll, no waiting
  const uint64_t t0 = global_ns();
  for (;;) {
    if (global_ns() - t0 >= limit_ns) return false;
    if (mbar_try_sleep(bar, parity, 20000u)) return true;
    if (*abort) return false;
  }
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

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
// one word of nibble bytes b0..b3 -> four fp16x2 of (n - 8) / 8, exact:
//   lo0 = {b0 & 15, b2 & 15}, lo1 = {b1 & 15, b3 & 15}, hi0 = {b0 >> 4, b2 >> 4}, hi1 = {b1 >> 4, b3 >> 4}.
// 0x640n is 1024 + n and 0x64n0 is 1024 + 16 n in fp16; (1024 + n) / 8 - 129 and
// (1024 + 16 n) / 128 - 9 are both (n - 8) / 8, each one exact fused multiply-add
__device__ __forceinline__ void nibs_to_f16_8th(uint32_t r, uint32_t& lo0, uint32_t& lo1, uint32_t& hi0,
                                                uint32_t& hi1) {
  const uint32_t r8 = r >> 8;
  const __half2 eighth = __halves2half2(__ushort_as_half(0x3000), __ushort_as_half(0x3000));    // 1/8
  const __half2 m129 = __halves2half2(__ushort_as_half(0xd808), __ushort_as_half(0xd808));      // -129
  const __half2 c128th = __halves2half2(__ushort_as_half(0x2000), __ushort_as_half(0x2000));    // 1/128
  const __half2 m9 = __halves2half2(__ushort_as_half(0xc880), __ushort_as_half(0xc880));        // -9
  uint32_t t0 = (r & 0x000f000fu) | 0x64006400u, t1 = (r8 & 0x000f000fu) | 0x64006400u;
  uint32_t t2 = (r & 0x00f000f0u) | 0x64006400u, t3 = (r8 & 0x00f000f0u) | 0x64006400u;
  __half2 v0 = __hfma2(*reinterpret_cast<__half2*>(&t0), eighth, m129);
  __half2 v1 = __hfma2(*reinterpret_cast<__half2*>(&t1), eighth, m129);
  __half2 v2 = __hfma2(*reinterpret_cast<__half2*>(&t2), c128th, m9);
  __half2 v3 = __hfma2(*reinterpret_cast<__half2*>(&t3), c128th, m9);
  lo0 = *reinterpret_cast<uint32_t*>(&v0);
  lo1 = *reinterpret_cast<uint32_t*>(&v1);
  hi0 = *reinterpret_cast<uint32_t*>(&v2);
  hi1 = *reinterpret_cast<uint32_t*>(&v3);
}
// x * d as two fp16 terms: hi = RN(x d), lo = x d - hi (exact: x = (n - 8)/8 has
// 4 significant bits, so x d has at most 15, and the fused multiply-add's
// exact residual is representable)
__device__ __forceinline__ void mul_split(uint32_t x, uint32_t d, uint32_t& hi, uint32_t& lo) {
  const __half2 xh = *reinterpret_cast<const __half2*>(&x), dh = *reinterpret_cast<const __half2*>(&d);
  const __half2 a = __hmul2(xh, dh);
  const __half2 b = __hfma2(xh, dh, __hneg2(a));
  hi = *reinterpret_cast<const uint32_t*>(&a);
  lo = *reinterpret_cast<const uint32_t*>(&b);
}
// bytes k0 and k1 of r (int8 codes) -> bf16x2 {c_k0, c_k1}, exact
__device__ __forceinline__ uint32_t i8_to_bf16(uint32_t r, uint32_t s0, uint32_t s1) {
  const uint32_t u = r ^ 0x80808080u;
  const float f0 = __uint_as_float(prmt(u, 0x4b000000u, s0)) - 8388736.0f;   // 2^23 + 128
  const float f1 = __uint_as_float(prmt(u, 0x4b000000u, s1)) - 8388736.0f;
  return prmt(__float_as_uint(f0), __float_as_uint(f1), 0x7632u);
}

// MMA row r (0..7) of a tile holds cell sigma(r) = (r >> 1) | ((r & 1) << 2), and
// row r + 8 holds cell 8 + sigma(r): the two cells a quarter-warp reads in one
// 128-bit shared load then differ in bit 2, which the 128-byte swizzle turns
// into disjoint bank groups
__device__ __forceinline__ int sigma(int r) { return (r >> 1) | ((r & 1) << 2); }

// ---------------------------------------------------------------- the kernel
template <int FMT, bool QF32>
__global__ void __launch_bounds__(32 * (QF32 ? kMaxWorkersF32 : kMaxWorkers), 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  constexpr bool kI8 = FMT == K8V4_FORMAT_INT8;
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t sb = (raw_s + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (sb - raw_s);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int W = blockDim.x >> 5;
  const Layout& LY = p.L;
  const uint32_t full = sb + LY.bar_off + 16 * w;                       // this worker's two stage barriers
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + LY.bar_off + 16 * W);
  // what needs no input of the previous kernel comes before the dependency
  // wait: the tensor maps (kernel parameters) into the descriptor cache, and
  // each worker's own stage barriers (its lane 0 issues that worker's copies)
  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
    *abort_flag = 0;
  }
  if (lane == 0) {
    mbar_init(full, 1);
    mbar_init(full + 8, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // launched as a programmatic dependent of the previous kernel in the stream:
  // nothing is read before it completes
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const CacheView& C = p.C;
  const int H = C.H, HQ = H * kGqa;
  const int r0 = lane >> 2, c = lane & 3;

  int n_vis = p.steps[b];
  if (n_vis < 0 || n_vis > p.max_seq_len) {
    if (threadIdx.x == 0 && split == 0 && g == 0) record_status(p.status, K8V4_ERANGE);
    n_vis = n_vis < 0 ? 0 : p.max_seq_len;
  }
  const int c_begin = p.cell_base + split * p.cells_per_split;
  const int c_stop = min(c_begin + p.cells_per_split, p.cell_limit);
  const int c_end = min(c_stop, n_vis);
  const int n_tiles = c_end > c_begin ? (c_end - c_begin + 15) >> 4 : 0;
  const int n_my = n_tiles > w ? (n_tiles - w + W - 1) / W : 0;      // tiles w + W u
  const uint32_t ring = sb + w * 2 * LY.stage_bytes;
  // a cell range past the sequence's visible cells (a short sequence of a
  // ragged batch; never the range holding a new token) only marks its partial
  // rows empty (m = -inf: the combine skips them) and leaves
  if (n_tiles == 0) {
    if (threadIdx.x < kGqa) {
      float* dst = p.ws + ((static_cast<int64_t>(b) * p.splits + split) * HQ + g * kGqa + threadIdx.x) * kPStride;
      dst[256] = -INFINITY;
      dst[257] = 0.0f;
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    return;
  }

  // ---- fused decode step: the CTA whose cells include the newest one (n_vis - 1)
  // writes the new token's K and V there before any copy of the pipeline starts
  // (the condition is the same for the whole CTA)
  const int new_cell = n_vis - 1;
  if (p.k_new != nullptr && new_cell >= c_begin && new_cell < c_stop && p.steps[b] == n_vis) {   // skipped for a clipped length
    if (w < 2) {
      const int64_t pidx = new_cell / C.P;
      const int64_t page = pidx < p.max_pages ? p.pt[static_cast<int64_t>(b) * p.max_pages + pidx] : -1;
      if (page >= 0 && page < C.n_pages) {
        uint8_t* base = C.pages + page * C.page_bytes;
        const int64_t r = static_cast<int64_t>(new_cell % C.P) * H + g;
        const int64_t elem = (static_cast<int64_t>(b) * H + g) * kD + 8 * lane;
        long long* ts = reinterpret_cast<long long*>(sm) + w * kRotScratch;   // stage memory, not yet in use
        // bf16 rows take the bulk append's fast paths (same bytes, fewer
        // instructions: this CTA's copies wait for them)
        if (w == 0) {
          if (p.kv_bf16) append_k_row_bf16<FMT>(C, base, r, static_cast<const uint16_t*>(p.k_new) + elem - 8 * lane, lane, ts);
          else append_k_row<false, FMT>(C, base, r, p.k_new, elem, lane, ts);
        } else {
          if (p.kv_bf16) append_v_row_bf16<FMT>(C, base, r, static_cast<const uint16_t*>(p.v_new) + elem - 8 * lane, lane, ts);
          else append_v_row<false, FMT>(C, base, r, p.v_new, elem, lane, ts);
        }
      } else if (w == 0 && lane == 0) {
        record_status(p.status, K8V4_ERANGE);
      }
      // the TMA copies (async proxy) that read this cell, and that later
      // overwrite the scratch, come after the block barrier below
      asm volatile("fence.proxy.async;" ::: "memory");
    }
    __syncthreads();
  }

  // ---- q loads (lane: head r0, dims 64 i + 16 c + [0, 16)), issued ahead of the
  // first copies so that they do not queue behind them; converted further down
  constexpr int kQraw = QF32 ? 16 : 8;
  uint4 qraw[kQraw];
  {
    const int64_t qrow = (static_cast<int64_t>(b) * HQ + g * kGqa + r0) * kD;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t e0 = qrow + 64 * i + 16 * c;
      const uint4* src = QF32 ? reinterpret_cast<const uint4*>(static_cast<const float*>(p.q) + e0)
                              : reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + e0);
#pragma unroll
      for (int t = 0; t < kQraw / 4; ++t) qraw[(kQraw / 4) * i + t] = src[t];
    }
  }

  // ---- this worker's copies: local tile u -> stage u & 1.  Page ids of 32
  // consecutive local tiles are held one per lane.
  const int32_t* pt_row = p.pt + static_cast<int64_t>(b) * p.max_pages;
  int win0 = -1000000, win_page = -1;
  auto page_of = [&](int u) -> int {         // warp-uniform u; all lanes call
    if (u < win0 || u >= win0 + 32) {
      win0 = u;
      const int cell = c_begin + 16 * (w + W * (u + lane));
      const int64_t pidx = cell >= 0 ? static_cast<int64_t>(p.page_div.div(static_cast<uint32_t>(cell))) : 0;
      win_page = (u + lane < n_my && pidx < p.max_pages) ? pt_row[pidx] : -1;
    }
    const int page = __shfl_sync(kFull, win_page, u - win0);
    return (page >= 0 && page < C.n_pages) ? page : -1;
  };
  // an out-of-range page id issues no copy (the stage barrier is completed by a
  // plain arrive) and is recorded; the tile is then skipped.  Diagnostics: with
  // p.withhold, worker 0 of CTA (0, 0, 0) issues nothing for its tile 0, so its
  // first wait runs out after the wait bound (a phase that nothing completes)
  const bool withheld = p.withhold && w == 0 && split == 0 && g == 0 && b == 0;
  auto issue = [&](int u, int page) {
    if (lane == 0) {
      const uint32_t st = ring + (u & 1) * LY.stage_bytes;
      const uint32_t bar = full + 8 * (u & 1);
      if (page >= 0) {
        const int cell0 = c_begin + 16 * (w + W * u);
        const int slot0 = cell0 - static_cast<int>(p.page_div.div(static_cast<uint32_t>(cell0))) * C.P;
        mbar_expect_tx(bar, LY.tx_bytes);
        tma_load_4d(st, &tm_k, 0, g, slot0, page, bar);
        tma_load_4d(st + 2048, &tm_k, 128, g, slot0, page, bar);
        tma_load_4d(st + LY.v_off, &tm_v, 0, g, slot0, page, bar);
        if (kI8) tma_load_4d(st + LY.v_off + 2048, &tm_v, 128, g, slot0, page, bar);
        const uint8_t* pg = C.pages + static_cast<int64_t>(page) * C.page_bytes;
        bulk_load(st + LY.ksc_off, pg + C.ks_off() + static_cast<int64_t>(slot0) * 8 * H, LY.ksc_bytes, bar);
        bulk_load(st + LY.vsc_off, pg + C.vs_off() + static_cast<int64_t>(slot0) * (kI8 ? 8 : 16) * H,
                  LY.vsc_bytes, bar);
      } else {
        record_status(p.status, K8V4_ERANGE);
        mbar_arrive(bar);
      }
    }
  };
  // the first two copies go out before the q set-up, whose loads overlap them
  int issued = 0;
  for (; issued < min(2, n_my); ++issued) {
    const int page = page_of(issued);
    if (!(withheld && issued == 0)) issue(issued, page);
  }

  // ---- q fragments (B operand of S^T = K q^T): lane holds head r0, dims
  // 64 i + 16 c + 4 j + e of k-step 4 i + j
  uint32_t qf[16][2];
  uint32_t qf_lo[QF32 ? 16 : 1][2];
  float f0, f1;                        // score factors of heads 2c, 2c+1
  {
    float qv[64];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (QF32) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint4 raw = qraw[4 * i + t];
          qv[16 * i + 4 * t] = __uint_as_float(raw.x); qv[16 * i + 4 * t + 1] = __uint_as_float(raw.y);
          qv[16 * i + 4 * t + 2] = __uint_as_float(raw.z); qv[16 * i + 4 * t + 3] = __uint_as_float(raw.w);
        }
      } else {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint4 raw = qraw[2 * i + t];
          const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            qv[16 * i + 8 * t + 2 * u] = __uint_as_float(wv[u] << 16);
            qv[16 * i + 8 * t + 2 * u + 1] = __uint_as_float(wv[u] & 0xffff0000u);
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
    const float fscale = p.sm_scale_log2 * ldexpf(1.0f, -sh);
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      // b0 = (k 2c, 2c+1), b1 = (k 2c+8, 2c+9): K dims o+0, o+1 | o+2, o+3
      const int o = 16 * (ks >> 2) + 4 * (ks & 3);
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = __fmul_rn(qv[o + e], up);
      const __half2 h0 = __floats2half2_rn(v[0], v[1]), h1 = __floats2half2_rn(v[2], v[3]);
      qf[ks][0] = *reinterpret_cast<const uint32_t*>(&h0);
      qf[ks][1] = *reinterpret_cast<const uint32_t*>(&h1);
      if (QF32) {
        const float2 a0 = __half22float2(h0), a1 = __half22float2(h1);
        const __half2 l0 = __floats2half2_rn(v[0] - a0.x, v[1] - a0.y);
        const __half2 l1 = __floats2half2_rn(v[2] - a1.x, v[3] - a1.y);
        qf_lo[ks % (QF32 ? 16 : 1)][0] = *reinterpret_cast<const uint32_t*>(&l0);
        qf_lo[ks % (QF32 ? 16 : 1)][1] = *reinterpret_cast<const uint32_t*>(&l1);
      }
    }
    // score factors for the heads of the C layout (2c, 2c+1): held by lanes 4h
    f0 = __shfl_sync(kFull, fscale, 8 * c);
    f1 = __shfl_sync(kFull, fscale, 8 * c + 4);
  }
  __syncthreads();

  // K fragment addresses within a stage (two 128-byte-swizzled [16][128] halves)
  const int rowA = sigma(r0), rowB = 8 + sigma(r0);
  uint32_t offA[4], offB[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int ch = 4 * (i & 1) + c;
    offA[i] = 2048 * (i >> 1) + rowA * 128 + 16 * (ch ^ (rowA & 7));
    offB[i] = 2048 * (i >> 1) + rowB * 128 + 16 * (ch ^ (rowB & 7));
  }
  const uint32_t ksA = LY.ksc_off + (rowA * H + g) * 8, ksB = LY.ksc_off + (rowB * H + g) * 8;
  // V fragment rows: matrix mi = lane >> 3 holds cells 8 (mi & 1) + sigma(0..7);
  // the B fragment's four cells are k = 2c, 2c+1, 2c+8, 2c+9
  const int mi = lane >> 3;
  const int vcell = 8 * (mi & 1) + sigma(lane & 7);
  const uint32_t vrow = LY.v_off + vcell * 128;
  const int vsw = vcell & 7;
  const int kc[4] = {sigma(2 * c), sigma(2 * c + 1), 8 + sigma(2 * c), 8 + sigma(2 * c + 1)};
  uint32_t soff[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) soff[i] = LY.vsc_off + (kc[i] * H + g) * (kI8 ? 8 : 16);

  constexpr int kMT = 16;              // 16-dim m-tiles of the 256 output dims (rotated space)
  float o[kMT][4];
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
  int M0 = INT_MIN, M1 = INT_MIN;      // running buckets of heads 2c, 2c+1
  float l0 = 0.0f, l1 = 0.0f;          // this lane's share of the sums of p' (heads 2c, 2c+1)
  const uint32_t wait_ns = p.wait_ns;
  bool aborted = false;                // this warp left the loop with copies in flight

  for (int u = 0; u < n_my; ++u) {
    const int s = u & 1;
    if (!__all_sync(kFull, mbar_wait(full + 8 * s, (u >> 1) & 1, wait_ns, abort_flag))) {
      if (lane == 0) {
        *abort_flag = 1;
        record_status(p.status, K8V4_ECUDA);
      }
      aborted = true;
      break;
    }
    const uint32_t st = ring + s * LY.stage_bytes;
    if (page_of(u) >= 0) {
      // ---- S^T[cell][head]: the two 128-lane halves accumulated separately
      // (two accumulators per half keep four MMA chains in flight)
      float acc[4][4];
#pragma unroll
      for (int a4 = 0; a4 < 4; ++a4) acc[a4][0] = acc[a4][1] = acc[a4][2] = acc[a4][3] = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 ka = lds128(st + offA[i]);
        const uint4 kb = lds128(st + offB[i]);
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
          if (QF32) mma_f16(dst, a[j], qf_lo[(4 * i + j) % (QF32 ? 16 : 1)][0], qf_lo[(4 * i + j) % (QF32 ? 16 : 1)][1]);
        }
      }
      const float2 kA = lds64f(st + ksA), kB = lds64f(st + ksB);
      const int cell0 = c_begin + 16 * (w + W * u);
      const bool vA = cell0 + rowA < n_vis, vB = cell0 + rowB < n_vis;
      float sc[4];
      sc[0] = vA ? (kA.x * (acc[0][0] + acc[1][0]) + kA.y * (acc[2][0] + acc[3][0])) * f0 : -INFINITY;
      sc[1] = vA ? (kA.x * (acc[0][1] + acc[1][1]) + kA.y * (acc[2][1] + acc[3][1])) * f1 : -INFINITY;
      sc[2] = vB ? (kB.x * (acc[0][2] + acc[1][2]) + kB.y * (acc[2][2] + acc[3][2])) * f0 : -INFINITY;
      sc[3] = vB ? (kB.x * (acc[0][3] + acc[1][3]) + kB.y * (acc[2][3] + acc[3][3])) * f1 : -INFINITY;

      // ---- softmax: the running bucket per head, raised by this tile's
      // ceil(max / 8); the accumulators follow by an exact power of two.  No
      // score above the running reference 8 M needs no maximum at all.
      int nb0 = M0, nb1 = M1;
      const bool up0 = sc[0] > 8.0f * M0 || sc[2] > 8.0f * M0, up1 = sc[1] > 8.0f * M1 || sc[3] > 8.0f * M1;
      if (__any_sync(kFull, up0 || up1)) {
        float t0 = fmaxf(sc[0], sc[2]), t1 = fmaxf(sc[1], sc[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          t0 = fmaxf(t0, __shfl_xor_sync(kFull, t0, off));
          t1 = fmaxf(t1, __shfl_xor_sync(kFull, t1, off));
        }
        nb0 = max(M0, static_cast<int>(fminf(fmaxf(ceilf(t0 * 0.125f), -kBucketClamp), kBucketClamp)));
        nb1 = max(M1, static_cast<int>(fminf(fmaxf(ceilf(t1 * 0.125f), -kBucketClamp), kBucketClamp)));
        const float g0 = M0 == INT_MIN ? 0.0f : pow2i(8 * (M0 - nb0));
        const float g1 = M1 == INT_MIN ? 0.0f : pow2i(8 * (M1 - nb1));
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          o[mt][0] *= g0; o[mt][2] *= g0;
          o[mt][1] *= g1; o[mt][3] *= g1;
        }
        l0 *= g0;
        l1 *= g1;
        M0 = nb0;
        M1 = nb1;
      }
      const float rf0 = static_cast<float>(8 * nb0 - 14), rf1 = static_cast<float>(8 * nb1 - 14);
      float pr[4];
      pr[0] = ex2(sc[0] - rf0);        // p' = 2^(s - ref + 14) <= 2^14
      pr[1] = ex2(sc[1] - rf1);
      pr[2] = ex2(sc[2] - rf0);
      pr[3] = ex2(sc[3] - rf1);
      l0 += pr[0] + pr[2];
      l1 += pr[1] + pr[3];

      // ---- PV in rotated space; p' goes to the MMA B layout (head r0; cells
      // 2c, 2c+1 | 2c+8, 2c+9) by warp transposes
      if (!kI8) {
        const uint32_t h01 = pack_f16(pr[0], pr[1]), h23 = pack_f16(pr[2], pr[3]);
        const float2 e01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 e23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        const uint32_t q01 = pack_f16(pr[0] - e01.x, pr[1] - e01.y), q23 = pack_f16(pr[2] - e23.x, pr[3] - e23.y);
        const uint32_t ph0 = movmatrix_t(h01), ph1 = movmatrix_t(h23);   // hi = RN(p')
        const uint32_t pl0 = movmatrix_t(q01), pl1 = movmatrix_t(q23);   // lo = RN(p' - hi)
#pragma unroll
        for (int bp = 0; bp < 4; ++bp) {
          // V^hat = (n - 8) d in two exact fp16 terms; m-tile 2 blk + hf = block
          // blk, dims 16 hf .. 16 hf + 15
          uint32_t R[4];
          ldmatrix_x4_t(R, st + vrow + 16 * ((2 * bp + (mi >> 1)) ^ vsw));
          // the fp16 d of blocks 2bp, 2bp+1 for the fragment's four cells
          const uint32_t w0 = lds32(st + soff[0] + 4 * bp), w1 = lds32(st + soff[1] + 4 * bp);
          const uint32_t w2 = lds32(st + soff[2] + 4 * bp), w3 = lds32(st + soff[3] + 4 * bp);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t sel = h ? 0x7632u : 0x5410u;
            const uint32_t d01 = prmt(w0, w1, sel), d89 = prmt(w2, w3, sel);   // d of block 2bp+h, cell pairs
            uint32_t xa[4], xb[4];          // (n-8)/8: [lo0, lo1, hi0, hi1] of cells 0-7 and 8-15
            nibs_to_f16_8th(R[2 * h], xa[0], xa[1], xa[2], xa[3]);
            nibs_to_f16_8th(R[2 * h + 1], xb[0], xb[1], xb[2], xb[3]);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              uint32_t ah[4], al[4];
              mul_split(xa[2 * hf], d01, ah[0], al[0]);
              mul_split(xa[2 * hf + 1], d01, ah[1], al[1]);
              mul_split(xb[2 * hf], d89, ah[2], al[2]);
              mul_split(xb[2 * hf + 1], d89, ah[3], al[3]);
              float* acc2 = o[2 * (2 * bp + h) + hf];
              mma_f16(acc2, ah, ph0, ph1);
              mma_f16(acc2, ah, pl0, pl1);
              mma_f16(acc2, al, ph0, ph1);
            }
          }
        }
      } else {
        // INT8 V: B = p' * s_v per 128-lane half in three bf16 terms; A = codes (exact in bf16)
        const uint32_t u0 = __float_as_uint(pr[0]), u1 = __float_as_uint(pr[1]);
        const uint32_t u2 = __float_as_uint(pr[2]), u3 = __float_as_uint(pr[3]);
        const uint32_t th0 = movmatrix_t(prmt(u0, u1, 0x7632u)), tl0 = movmatrix_t(prmt(u0, u1, 0x5410u));
        const uint32_t th1 = movmatrix_t(prmt(u2, u3, 0x7632u)), tl1 = movmatrix_t(prmt(u2, u3, 0x5410u));
        const float P4[4] = {__uint_as_float(prmt(tl0, th0, 0x5410u)), __uint_as_float(prmt(tl0, th0, 0x7632u)),
                             __uint_as_float(prmt(tl1, th1, 0x5410u)), __uint_as_float(prmt(tl1, th1, 0x7632u))};
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
          float x[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) x[i] = P4[i] * __uint_as_float(lds32(st + soff[i] + 4 * hv));
          uint32_t B[3][2];
#pragma unroll
          for (int pl = 0; pl < 3; ++pl) {
            B[pl][0] = pack_bf16(x[0], x[1]);
            B[pl][1] = pack_bf16(x[2], x[3]);
            if (pl < 2) {
              x[0] -= bf16_lo(B[pl][0]); x[1] -= bf16_hi(B[pl][0]);
              x[2] -= bf16_lo(B[pl][1]); x[3] -= bf16_hi(B[pl][1]);
            }
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            // 16-dim chunks 8 hv + 2 jj, + 1
            const int ch = 2 * jj + (mi >> 1);
            uint32_t R[4];
            ldmatrix_x4_t(R, st + 2048 * hv + vrow + 16 * (ch ^ vsw));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t Ra = R[2 * h], Rb = R[2 * h + 1];
              const uint32_t a[4] = {i8_to_bf16(Ra, 0x7540u, 0x7542u), i8_to_bf16(Ra, 0x7541u, 0x7543u),
                                     i8_to_bf16(Rb, 0x7540u, 0x7542u), i8_to_bf16(Rb, 0x7541u, 0x7543u)};
#pragma unroll
              for (int pl = 0; pl < 3; ++pl) mma_bf16(o[8 * hv + 2 * jj + h], a, B[pl][0], B[pl][1]);
            }
          }
        }
      }
    }
    // the stage is consumed: refill it with tile u + 2
    __syncwarp();
    if (issued < n_my) {
      issue(issued, page_of(issued));
      ++issued;
    }
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, off);
    l1 += __shfl_xor_sync(kFull, l1, off);
  }

  // ---------------------------------------------------------------- epilogue
  // Each worker writes its partial (kPartFloats: o by rotated dim, buckets,
  // sums) into its own two stages as soon as its loop ends, while the others
  // may still stream.  A worker that left the loop early first waits (bounded)
  // for its copies still in flight.  A head with nothing visible writes zeros,
  // so the merge below needs no test.
  if (aborted && lane == 0) {
    if (withheld) mbar_arrive(full);   // the withheld tile 0: nothing in flight, close its phase
    for (int u = max(0, issued - 2); u < issued; ++u) {
      const uint64_t t0 = global_ns();
      while (!mbar_try_sleep(full + 8 * (u & 1), (u >> 1) & 1, 20000u) && global_ns() - t0 < kWaitDefaultNs) {
      }
    }
  }
  __syncwarp();
  float* mine = reinterpret_cast<float*>(sm + w * 2 * LY.stage_bytes);
  const bool live0 = M0 != INT_MIN, live1 = M1 != INT_MIN;
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt) {
    const int d0 = kI8 ? 16 * mt + 2 * r0 : 32 * (mt >> 1) + 16 * (mt & 1) + 2 * r0;
    *reinterpret_cast<float2*>(mine + (2 * c) * kHeadStride + d0) =
        live0 ? make_float2(o[mt][0], o[mt][2]) : make_float2(0.0f, 0.0f);
    *reinterpret_cast<float2*>(mine + (2 * c + 1) * kHeadStride + d0) =
        live1 ? make_float2(o[mt][1], o[mt][3]) : make_float2(0.0f, 0.0f);
  }
  if (r0 == 0) {
    reinterpret_cast<int*>(mine + kPartBucket)[2 * c] = M0;
    reinterpret_cast<int*>(mine + kPartBucket)[2 * c + 1] = M1;
    mine[kPartSum + 2 * c] = l0;
    mine[kPartSum + 2 * c + 1] = l1;
  }
  __syncthreads();
  // one warp per head: merge the workers' partials at the largest bucket (lane
  // j reads worker j's bucket and sum), bring the row back from rotated space
  // and write (o, m, l).  The lane holds dims 4 lane + e and 128 + 4 lane + e
  // (e < 4) as v[e] and v[4 + e], so every shared-memory read is conflict free.
  for (int h = w; h < kGqa; h += W) {
    const float* mj_part = reinterpret_cast<const float*>(sm + min(lane, W - 1) * 2 * LY.stage_bytes);
    const int mj = lane < W ? reinterpret_cast<const int*>(mj_part + kPartBucket)[h] : INT_MIN;
    const float lj = lane < W ? mj_part[kPartSum + h] : 0.0f;
    int Mx = mj;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) Mx = max(Mx, __shfl_xor_sync(kFull, Mx, off));
    const float fj = mj == INT_MIN ? 0.0f : pow2i(8 * (mj - Mx));
    float v[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    float L = 0.0f;
#pragma unroll
    for (int j = 0; j < (QF32 ? kMaxWorkersF32 : kMaxWorkers); ++j) {
      const float f = __shfl_sync(kFull, fj, j), lw = __shfl_sync(kFull, lj, j);   // 0 for j >= W
      if (j < W) {
        const float* src = reinterpret_cast<const float*>(sm + j * 2 * LY.stage_bytes) + h * kHeadStride;
        const float4 x0 = *reinterpret_cast<const float4*>(src + 4 * lane);
        const float4 x1 = *reinterpret_cast<const float4*>(src + 128 + 4 * lane);
        v[0] += x0.x * f; v[1] += x0.y * f; v[2] += x0.z * f; v[3] += x0.w * f;
        v[4] += x1.x * f; v[5] += x1.y * f; v[6] += x1.z * f; v[7] += x1.w * f;
        L += lw * f;
      }
    }
    float scale;
    if (!kI8) {
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
      scale = 1.0f / 32768.0f;          // 1/16 of the transform, 2^-11 of p' (2^14) and (n-8)/8 (2^-3)
    } else {
      scale = 1.0f / 16384.0f;          // 2^-14 of p'
    }
    float* dst = p.ws + ((static_cast<int64_t>(b) * p.splits + split) * HQ + g * kGqa + h) * kPStride;
    reinterpret_cast<float4*>(dst)[lane] = make_float4(v[0] * scale, v[1] * scale, v[2] * scale, v[3] * scale);
    reinterpret_cast<float4*>(dst)[32 + lane] = make_float4(v[4] * scale, v[5] * scale, v[6] * scale, v[7] * scale);
    if (lane == 0) {
      dst[256] = Mx == INT_MIN ? -INFINITY : static_cast<float>(8 * Mx);
      dst[257] = L * (1.0f / 16384.0f);
    }
  }
  // the combine kernel may start once every partial of this grid is written
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- verify: several queries per sequence
// The speculative-decoding window of the pull request's "Tests" (a batch of
// queries per sequence, each with its own step, i.e. visible length), over the
// k8v4 format with bf16 queries.  The queries read the same cells, so each
// 16-cell tile is copied once and converted once for all of them:
//   - a CTA runs kVTeams teams of four warps; a team takes the range's tiles
//     round robin (team t: tiles t, t + kVTeams, ...), and one lane of the team
//     keeps kVStages of them in flight with the same TMA copies as decode;
//   - warp j of a team owns dims [64 j, 64 j + 64): it converts that quarter of
//     the tile's K codes and computes the partial scores of every query over
//     those dims (K scale of its half applied), and it converts that quarter of
//     the V nibbles and accumulates O^T for every query over those dims -- so
//     the accumulators (4 m-tiles x NQ queries) fit in registers;
//   - the four partial scores of a (cell, query, head) meet in shared memory;
//     warp q % 4 owns query q: it sums them (fixed order), masks the cells past
//     the query's step, runs decode's bucketed softmax and publishes p' (two
//     fp16 terms in the MMA B layout) with the accumulator rescale factors;
//   - one named barrier per tile orders the team: after it, the owners run the
//     softmax of tile u while every warp accumulates PV of tile u - 1 (scores
//     and p' double-buffered), so the owners' work overlaps the others'.  A
//     timeout or a bad page never leaves a warp waiting: every warp reaches
//     the barrier each iteration, and the team leaves the loop together on a
//     flag its first warp published before the barrier.
// The partial rows (o, m, l) per (query, head) go to the split combine.
constexpr int kVTeams = 2;
constexpr int kVStages = 6;
constexpr int kVMaxQ = 8;

struct VLayout {
  int stage_bytes, v_off, ksc_off, vsc_off, tx_bytes;   // the decode stage (K8V4 format)
  int q_off, x_off, pb_off, flag_off, bar_off, total;
};

inline VLayout vlayout_of(int H, int nq) {
  const Layout D = layout_of(K8V4_FORMAT_K8V4, H, 1);
  VLayout L;
  L.stage_bytes = D.stage_bytes;
  L.v_off = D.v_off;
  L.ksc_off = D.ksc_off;
  L.vsc_off = D.vsc_off;
  L.tx_bytes = D.tx_bytes;
  const int ring = kVTeams * kVStages * L.stage_bytes;
  L.q_off = ring;                                   // [4 warps][nq][32 lanes][4 k-steps][2 words]
  L.x_off = L.q_off + 4 * nq * 32 * 8 * 4;          // [2 tiles][team][4 warps][nq][32 lanes][4] f32
  L.pb_off = L.x_off + 2 * kVTeams * 4 * nq * 32 * 16;   // [2 tiles][team][nq][32 lanes][8 words]
  const int work_end = L.pb_off + 2 * kVTeams * nq * 32 * 32;
  const int merge = kVTeams * nq * kGqa * 258 * 4;  // epilogue: [team][nq x 8 rows][258] f32
  L.flag_off = (std::max(work_end, merge) + 15) & ~15;   // abort word, then two stop words per team
  L.bar_off = L.flag_off + 32;                      // full barriers [team][stage]
  L.total = L.bar_off + 8 * kVTeams * kVStages + 1024;
  return L;
}

struct VerifyWsParams {
  CacheView C;
  const uint16_t* q;       // bf16 [n_seqs][nq][8 H][256]
  const int32_t* pt;
  int64_t max_pages;
  const int32_t* steps;    // [n_seqs][nq]
  int max_seq_len, cells_per_split, splits;
  float sm_scale_log2;
  float* ws;               // partial rows [n_seqs][splits][nq][8 H][260]
  int* status;
  uint32_t wait_ns;
  FastDiv page_div;
  VLayout L;
};

template <int NQ>
__global__ void __launch_bounds__(32 * 4 * kVTeams, 1)
    verify_ws_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const VerifyWsParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  constexpr int kOwn = (NQ + 3) / 4;                // queries a warp owns at most
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t sb = (raw_s + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (sb - raw_s);
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int team = wid >> 2, j = wid & 3;           // warp j of the team: dims [64 j, 64 j + 64)
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const CacheView& C = p.C;
  const VLayout& LY = p.L;
  const int H = C.H, HQ = H * kGqa;
  const int r0 = lane >> 2, c = lane & 3;

  // visible lengths: every query's (for the tile range), the owned ones kept
  int n_max = 0;
  int vis_o[kOwn];
#pragma unroll
  for (int k = 0; k < kOwn; ++k) vis_o[k] = 0;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    int v = p.steps[static_cast<int64_t>(b) * NQ + q];
    if (v < 0 || v > p.max_seq_len) {
      if (threadIdx.x == 0 && split == 0 && g == 0) record_status(p.status, K8V4_ERANGE);
      v = v < 0 ? 0 : p.max_seq_len;
    }
    n_max = max(n_max, v);
    if (q % 4 == j) vis_o[q / 4] = v;
  }
  const int c_begin = split * p.cells_per_split;
  const int c_end = min(c_begin + p.cells_per_split, n_max);
  const int n_tiles = c_end > c_begin ? (c_end - c_begin + 15) >> 4 : 0;
  const int n_my = n_tiles > team ? (n_tiles - team + kVTeams - 1) / kVTeams : 0;   // tiles team + kVTeams u

  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + LY.flag_off);
  volatile int* stop_words = reinterpret_cast<volatile int*>(sm + LY.flag_off + 8 + 8 * team);   // [2]
  const uint32_t full = sb + LY.bar_off + 8 * kVStages * team;   // this team's stage barriers
  const uint32_t ring = sb + team * kVStages * LY.stage_bytes;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kVTeams * kVStages; ++i) mbar_init(sb + LY.bar_off + 8 * i, 1);
    *abort_flag = 0;
    for (int t = 0; t < 2 * kVTeams; ++t) reinterpret_cast<volatile int*>(sm + LY.flag_off + 8)[t] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---- q fragments of every query into shared memory (team 0's warp j writes
  // the k-steps of dims [64 j, 64 j + 64), read back by warp j of each team),
  // and the score factors: lane (r0, c) holds head r0's 64 dims 64 i + 16 c + ...
  float* fq = reinterpret_cast<float*>(sm + LY.pb_off);      // [nq][8] factors, before the P buffer is used
  if (team == 0) {
    for (int q = 0; q < NQ; ++q) {
      const int64_t qrow = ((static_cast<int64_t>(b) * NQ + q) * HQ + g * kGqa + r0) * kD;
      // the row's largest magnitude (this lane: dims 64 i + 16 c + 0..15; the four lanes of the row)
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow + 64 * i + 16 * c);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint4 raw = src[t];
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(raw.x)), fabsf(bf16_hi(raw.x))),
                                   fmaxf(fabsf(bf16_lo(raw.y)), fabsf(bf16_hi(raw.y)))));
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(raw.z)), fabsf(bf16_hi(raw.z))),
                                   fmaxf(fabsf(bf16_lo(raw.w)), fabsf(bf16_hi(raw.w)))));
        }
      }
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
      const int ex = amax > 0.0f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127 : 0;
      const int sh = max(-100, min(100, 14 - ex));
      const float up = ldexpf(1.0f, sh);
      // k-steps 4 j + jj: dims 64 j + 16 c + 4 jj + (0..3)
      float qv[16];
      {
        const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow + 64 * j + 16 * c);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint4 raw = src[t];
          const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            qv[8 * t + 2 * u] = bf16_lo(wv[u]);
            qv[8 * t + 2 * u + 1] = bf16_hi(wv[u]);
          }
        }
      }
      uint32_t wq[8];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = __fmul_rn(qv[4 * jj + e], up);
        const __half2 h0 = __floats2half2_rn(v[0], v[1]), h1 = __floats2half2_rn(v[2], v[3]);
        wq[2 * jj] = *reinterpret_cast<const uint32_t*>(&h0);
        wq[2 * jj + 1] = *reinterpret_cast<const uint32_t*>(&h1);
      }
      uint4* dq = reinterpret_cast<uint4*>(sm + LY.q_off + ((j * NQ + q) * 32 + lane) * 32);
      dq[0] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
      dq[1] = make_uint4(wq[4], wq[5], wq[6], wq[7]);
      if (j == 0 && c == 0) fq[q * kGqa + r0] = p.sm_scale_log2 * ldexpf(1.0f, -sh);
    }
  }
  __syncthreads();
  // the owned queries' score factors for heads 2c, 2c + 1
  float f0o[kOwn], f1o[kOwn];
#pragma unroll
  for (int k = 0; k < kOwn; ++k) {
    const int q = j + 4 * k;
    f0o[k] = q < NQ ? fq[q * kGqa + 2 * c] : 0.0f;
    f1o[k] = q < NQ ? fq[q * kGqa + 2 * c + 1] : 0.0f;
  }
  __syncthreads();                                   // fq is overwritten by the P buffer below

  // ---- this team's copies: local tile u -> stage u % kVStages (the decode copies)
  const int32_t* pt_row = p.pt + static_cast<int64_t>(b) * p.max_pages;
  int win0 = -1000000, win_page = -1;
  auto page_of = [&](int u) -> int {         // warp-uniform u; all lanes call
    if (u < win0 || u >= win0 + 32) {
      win0 = u;
      const int cell = c_begin + 16 * (team + kVTeams * (u + lane));
      const int64_t pidx = static_cast<int64_t>(p.page_div.div(static_cast<uint32_t>(cell)));
      win_page = (u + lane < n_my && pidx < p.max_pages) ? pt_row[pidx] : -1;
    }
    const int page = __shfl_sync(kFull, win_page, u - win0);
    return (page >= 0 && page < C.n_pages) ? page : -1;
  };
  auto issue = [&](int u, int page) {        // team warp 0 only, all lanes call
    if (lane == 0) {
      const uint32_t st = ring + (u % kVStages) * LY.stage_bytes;
      const uint32_t bar = full + 8 * (u % kVStages);
      if (page >= 0) {
        const int cell0 = c_begin + 16 * (team + kVTeams * u);
        const int slot0 = cell0 - static_cast<int>(p.page_div.div(static_cast<uint32_t>(cell0))) * C.P;
        mbar_expect_tx(bar, LY.tx_bytes);
        tma_load_4d(st, &tm_k, 0, g, slot0, page, bar);
        tma_load_4d(st + 2048, &tm_k, 128, g, slot0, page, bar);
        tma_load_4d(st + LY.v_off, &tm_v, 0, g, slot0, page, bar);
        const uint8_t* pg = C.pages + static_cast<int64_t>(page) * C.page_bytes;
        bulk_load(st + LY.ksc_off, pg + C.ks_off() + static_cast<int64_t>(slot0) * 8 * H, 128 * H, bar);
        bulk_load(st + LY.vsc_off, pg + C.vs_off() + static_cast<int64_t>(slot0) * 16 * H, 256 * H, bar);
      } else {
        record_status(p.status, K8V4_ERANGE);
        mbar_arrive(bar);
      }
    }
  };
  if (j == 0) {
    if (lane == 0 && n_my > 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
    }
    for (int u = 0; u < min(kVStages, n_my); ++u) issue(u, page_of(u));
  }
  int issued = min(kVStages, n_my);

  // K fragment addresses of this warp's quarter (decode's i = j), V fragment rows
  const int rowA = sigma(r0), rowB = 8 + sigma(r0);
  uint32_t offA, offB;
  {
    const int ch = 4 * (j & 1) + c;
    offA = 2048 * (j >> 1) + rowA * 128 + 16 * (ch ^ (rowA & 7));
    offB = 2048 * (j >> 1) + rowB * 128 + 16 * (ch ^ (rowB & 7));
  }
  const uint32_t ksA = LY.ksc_off + (rowA * H + g) * 8 + 4 * (j >> 1);   // this half's K scale
  const uint32_t ksB = LY.ksc_off + (rowB * H + g) * 8 + 4 * (j >> 1);
  const int mi = lane >> 3;
  const int vcell = 8 * (mi & 1) + sigma(lane & 7);
  const uint32_t vrow = LY.v_off + vcell * 128;
  const int vsw = vcell & 7;
  const int kc4[4] = {sigma(2 * c), sigma(2 * c + 1), 8 + sigma(2 * c), 8 + sigma(2 * c + 1)};
  uint32_t soff[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) soff[i] = LY.vsc_off + (kc4[i] * H + g) * 16 + 4 * j;   // blocks 2j, 2j + 1
  const uint32_t qsm = sb + LY.q_off + ((j * NQ) * 32 + lane) * 32;         // + q * 1024
  // tile u's buffers: (u & 1) * kVTeams + team
  float* xs0 = reinterpret_cast<float*>(sm + LY.x_off) + static_cast<int64_t>(team) * 4 * NQ * 32 * 4;
  uint32_t* pb0 = reinterpret_cast<uint32_t*>(sm + LY.pb_off) + static_cast<int64_t>(team) * NQ * 32 * 8;
  constexpr int kXBuf = kVTeams * 4 * NQ * 32 * 4, kPBuf = kVTeams * NQ * 32 * 8;

  float o[4][NQ][4];                 // m-tiles 4 j .. 4 j + 3 (rotated space) x queries
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int q = 0; q < NQ; ++q) o[mt][q][0] = o[mt][q][1] = o[mt][q][2] = o[mt][q][3] = 0.0f;
  int M0[kOwn], M1[kOwn];
  float l0[kOwn], l1[kOwn];
#pragma unroll
  for (int k = 0; k < kOwn; ++k) {
    M0[k] = M1[k] = INT_MIN;
    l0[k] = l1[k] = 0.0f;
  }
  const uint32_t wait_ns = p.wait_ns;
  const int bar_id = 1 + team;

  bool work_prev = false;
  for (int u = 0; u <= n_my; ++u) {
    // iteration u: scores of tile u (u < n_my), then after the barrier the
    // owners' softmax of tile u beside every warp's PV of tile u - 1
    const bool have = u < n_my;
    const int s = u % kVStages;
    const uint32_t st = ring + s * LY.stage_bytes;
    float* xs = xs0 + (u & 1) * kXBuf;
    uint32_t* pb = pb0 + (u & 1) * kPBuf;
    bool work = false;
    if (have) {
      const bool ok = __all_sync(kFull, mbar_wait(full + 8 * s, (u / kVStages) & 1, wait_ns, abort_flag));
      if (!ok && lane == 0) {
        *abort_flag = 1;
        record_status(p.status, K8V4_ECUDA);
      }
      work = ok && page_of(u) >= 0;
    }
    // ---- partial scores over this warp's 64 dims, every query
    if (work) {
      const uint4 ka = lds128(st + offA), kb = lds128(st + offB);
      const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb.x, kb.y, kb.z, kb.w};
      uint32_t a[4][4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        codes_to_f16(wa[jj], a[jj][0], a[jj][2]);
        codes_to_f16(wb[jj], a[jj][1], a[jj][3]);
      }
      const float sA = __uint_as_float(lds32(st + ksA)), sB = __uint_as_float(lds32(st + ksB));
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const uint4 q0 = lds128(qsm + q * 1024), q1 = lds128(qsm + q * 1024 + 16);
        float e[4] = {0.0f, 0.0f, 0.0f, 0.0f}, f[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_f16(e, a[0], q0.x, q0.y);
        mma_f16(f, a[1], q0.z, q0.w);
        mma_f16(e, a[2], q1.x, q1.y);
        mma_f16(f, a[3], q1.z, q1.w);
        *reinterpret_cast<float4*>(xs + ((j * NQ + q) * 32 + lane) * 4) =
            make_float4(sA * (e[0] + f[0]), sA * (e[1] + f[1]), sB * (e[2] + f[2]), sB * (e[3] + f[3]));
      }
    }
    named_barrier(bar_id, 128);
    // the stop word of the previous iteration (published before this barrier)
    if (u >= 1 && stop_words[(u - 1) & 1]) break;
    if (j == 0) {
      // every warp is past PV(u - 2): refill that tile's stage with tile u - 2 + kVStages
      if (u >= 2 && issued < n_my && !*abort_flag) {
        issue(issued, page_of(issued));
        ++issued;
      }
      if (lane == 0) stop_words[u & 1] = *abort_flag;
    }
    // ---- softmax of the owned queries over tile u
    if (have) {
      const int cell0 = c_begin + 16 * (team + kVTeams * u);
#pragma unroll
      for (int k = 0; k < kOwn; ++k) {
        const int q = j + 4 * k;
        if (q >= NQ) continue;
        float sc[4];
        {
          float4 x[4];
#pragma unroll
          for (int jw = 0; jw < 4; ++jw) x[jw] = *reinterpret_cast<const float4*>(xs + ((jw * NQ + q) * 32 + lane) * 4);
          const bool vA = work && cell0 + rowA < vis_o[k], vB = work && cell0 + rowB < vis_o[k];
          sc[0] = vA ? ((x[0].x + x[1].x) + (x[2].x + x[3].x)) * f0o[k] : -INFINITY;
          sc[1] = vA ? ((x[0].y + x[1].y) + (x[2].y + x[3].y)) * f1o[k] : -INFINITY;
          sc[2] = vB ? ((x[0].z + x[1].z) + (x[2].z + x[3].z)) * f0o[k] : -INFINITY;
          sc[3] = vB ? ((x[0].w + x[1].w) + (x[2].w + x[3].w)) * f1o[k] : -INFINITY;
        }
        int nb0 = M0[k], nb1 = M1[k];
        float g0 = 1.0f, g1 = 1.0f;
        const bool up0 = sc[0] > 8.0f * M0[k] || sc[2] > 8.0f * M0[k], up1 = sc[1] > 8.0f * M1[k] || sc[3] > 8.0f * M1[k];
        if (__any_sync(kFull, up0 || up1)) {
          float t0 = fmaxf(sc[0], sc[2]), t1 = fmaxf(sc[1], sc[3]);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            t0 = fmaxf(t0, __shfl_xor_sync(kFull, t0, off));
            t1 = fmaxf(t1, __shfl_xor_sync(kFull, t1, off));
          }
          nb0 = max(M0[k], static_cast<int>(fminf(fmaxf(ceilf(t0 * 0.125f), -kBucketClamp), kBucketClamp)));
          nb1 = max(M1[k], static_cast<int>(fminf(fmaxf(ceilf(t1 * 0.125f), -kBucketClamp), kBucketClamp)));
          g0 = M0[k] == INT_MIN ? 0.0f : pow2i(8 * (M0[k] - nb0));
          g1 = M1[k] == INT_MIN ? 0.0f : pow2i(8 * (M1[k] - nb1));
          l0[k] *= g0;
          l1[k] *= g1;
          M0[k] = nb0;
          M1[k] = nb1;
        }
        const float rf0 = static_cast<float>(8 * nb0 - 14), rf1 = static_cast<float>(8 * nb1 - 14);
        float pr[4];
        pr[0] = ex2(sc[0] - rf0);
        pr[1] = ex2(sc[1] - rf1);
        pr[2] = ex2(sc[2] - rf0);
        pr[3] = ex2(sc[3] - rf1);
        l0[k] += pr[0] + pr[2];
        l1[k] += pr[1] + pr[3];
        const uint32_t h01 = pack_f16(pr[0], pr[1]), h23 = pack_f16(pr[2], pr[3]);
        const float2 e01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 e23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        const uint32_t q01 = pack_f16(pr[0] - e01.x, pr[1] - e01.y), q23 = pack_f16(pr[2] - e23.x, pr[3] - e23.y);
        uint4* dst = reinterpret_cast<uint4*>(pb + (q * 32 + lane) * 8);
        dst[0] = make_uint4(movmatrix_t(h01), movmatrix_t(h23), movmatrix_t(q01), movmatrix_t(q23));
        dst[1] = make_uint4(__float_as_uint(g0), __float_as_uint(g1), 0u, 0u);
      }
    }
    // ---- PV of tile u - 1 over this warp's dims: rescale, then O^T += V^hat p' per query
    if (u >= 1 && work_prev) {
      const uint32_t stp = ring + ((u - 1) % kVStages) * LY.stage_bytes;
      const uint32_t* pbp = pb0 + ((u - 1) & 1) * kPBuf;
      uint32_t ph[NQ][4];
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const uint4 pp = *reinterpret_cast<const uint4*>(pbp + (q * 32 + lane) * 8);
        const uint4 gg = *reinterpret_cast<const uint4*>(pbp + (q * 32 + lane) * 8 + 4);
        ph[q][0] = pp.x; ph[q][1] = pp.y; ph[q][2] = pp.z; ph[q][3] = pp.w;
        const float g0 = __uint_as_float(gg.x), g1 = __uint_as_float(gg.y);
        if (__any_sync(kFull, g0 != 1.0f || g1 != 1.0f)) {
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            o[mt][q][0] *= g0; o[mt][q][2] *= g0;
            o[mt][q][1] *= g1; o[mt][q][3] *= g1;
          }
        }
      }
      uint32_t R[4];
      ldmatrix_x4_t(R, stp + vrow + 16 * ((2 * j + (mi >> 1)) ^ vsw));
      const uint32_t w0 = lds32(stp + soff[0]), w1 = lds32(stp + soff[1]);
      const uint32_t w2 = lds32(stp + soff[2]), w3 = lds32(stp + soff[3]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t sel = h ? 0x7632u : 0x5410u;
        const uint32_t d01 = prmt(w0, w1, sel), d89 = prmt(w2, w3, sel);
        uint32_t xa[4], xb[4];
        nibs_to_f16_8th(R[2 * h], xa[0], xa[1], xa[2], xa[3]);
        nibs_to_f16_8th(R[2 * h + 1], xb[0], xb[1], xb[2], xb[3]);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t ah[4], al[4];
          mul_split(xa[2 * hf], d01, ah[0], al[0]);
          mul_split(xa[2 * hf + 1], d01, ah[1], al[1]);
          mul_split(xb[2 * hf], d89, ah[2], al[2]);
          mul_split(xb[2 * hf + 1], d89, ah[3], al[3]);
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            float* acc2 = o[2 * h + hf][q];
            mma_f16(acc2, ah, ph[q][0], ph[q][1]);
            mma_f16(acc2, ah, ph[q][2], ph[q][3]);
            mma_f16(acc2, al, ph[q][0], ph[q][1]);
          }
        }
      }
    }
    work_prev = work;
  }
#pragma unroll
  for (int k = 0; k < kOwn; ++k) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0[k] += __shfl_xor_sync(kFull, l0[k], off);
      l1[k] += __shfl_xor_sync(kFull, l1[k], off);
    }
  }

  // ---------------------------------------------------------------- epilogue
  __syncthreads();
  if (*abort_flag) {
    // copies still in flight land before the stage memory is reused
    if (j == 0 && lane == 0) {
      for (int u = max(0, issued - kVStages); u < issued; ++u) {
        const uint64_t t0 = global_ns();
        while (!mbar_try_sleep(full + 8 * (u % kVStages), (u / kVStages) & 1, 20000u) &&
               global_ns() - t0 < kWaitDefaultNs) {
        }
      }
    }
    __syncthreads();
  }
  // each team's partial: [nq x 8 rows][258] = o[256], bucket, l
  float* mine = reinterpret_cast<float*>(sm) + static_cast<int64_t>(team) * NQ * kGqa * 258;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int gm = 4 * j + mt;
      const int d0 = 32 * (gm >> 1) + 16 * (gm & 1) + 2 * r0;
      *reinterpret_cast<float2*>(mine + (q * kGqa + 2 * c) * 258 + d0) = make_float2(o[mt][q][0], o[mt][q][2]);
      *reinterpret_cast<float2*>(mine + (q * kGqa + 2 * c + 1) * 258 + d0) = make_float2(o[mt][q][1], o[mt][q][3]);
    }
  }
  if (r0 == 0) {
#pragma unroll
    for (int k = 0; k < kOwn; ++k) {
      const int q = j + 4 * k;
      if (q >= NQ) continue;
      reinterpret_cast<int*>(mine + (q * kGqa + 2 * c) * 258)[256] = M0[k];
      reinterpret_cast<int*>(mine + (q * kGqa + 2 * c + 1) * 258)[256] = M1[k];
      mine[(q * kGqa + 2 * c) * 258 + 257] = l0[k];
      mine[(q * kGqa + 2 * c + 1) * 258 + 257] = l1[k];
    }
  }
  __syncthreads();
  // one warp per row: merge the teams at the largest bucket, rotate back, write (o, m, l)
  const float* part = reinterpret_cast<const float*>(sm);
  for (int row = wid; row < NQ * kGqa; row += 4 * kVTeams) {
    int Mx = INT_MIN;
#pragma unroll
    for (int t = 0; t < kVTeams; ++t) Mx = max(Mx, reinterpret_cast<const int*>(part + (t * NQ * kGqa + row) * 258)[256]);
    float v[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    float L = 0.0f;
    if (Mx != INT_MIN) {
#pragma unroll
      for (int t = 0; t < kVTeams; ++t) {
        const float* src = part + (t * NQ * kGqa + row) * 258;
        const int mt = reinterpret_cast<const int*>(src)[256];
        if (mt == INT_MIN) continue;
        const float sc2 = pow2i(8 * (mt - Mx));
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float2 x = *reinterpret_cast<const float2*>(src + 8 * lane + e);
          v[e] += x.x * sc2;
          v[e + 1] += x.y * sc2;
        }
        L += src[257] * sc2;
      }
    }
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
    constexpr float scale = 1.0f / 32768.0f;   // 1/16 of the transform, 2^-11 of p' (2^14) and (n-8)/8 (2^-3)
    const int q = row / kGqa, h = row % kGqa;
    float* dst = p.ws + ((((static_cast<int64_t>(b) * p.splits + split) * NQ + q) * HQ) + g * kGqa + h) * kPStride;
    reinterpret_cast<float4*>(dst + 8 * lane)[0] = make_float4(v[0] * scale, v[1] * scale, v[2] * scale, v[3] * scale);
    reinterpret_cast<float4*>(dst + 8 * lane)[1] = make_float4(v[4] * scale, v[5] * scale, v[6] * scale, v[7] * scale);
    if (lane == 0) {
      dst[256] = Mx == INT_MIN ? -INFINITY : static_cast<float>(8 * Mx);
      dst[257] = L * (1.0f / 16384.0f);
    }
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- tensor maps
// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A run of rows [P][H][row_bytes] per page, as a 4-D byte tensor (byte, head,
// cell, page) with box_rows-cell x 128-byte boxes, 128-byte swizzled.
bool encode_rows(CUtensorMap* m, const CacheView& C, int64_t run_off, int row_bytes, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(C.H),
                              static_cast<cuuint64_t>(C.P), static_cast<cuuint64_t>(C.n_pages)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(row_bytes) * C.H,
                                 static_cast<cuuint64_t>(C.page_bytes)};
  const cuuint32_t box[4] = {128, 1, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, C.pages + run_off, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The maps of the last kMapCache caches (encoding is host work, done once per
// cache; a server cycling through more caches than that re-encodes)
constexpr int kMapCache = 64;
struct MapEntry {
  const uint8_t* pages = nullptr;
  int64_t n_pages = 0;
  int P = 0, H = 0, fmt = 0, box = 0;
  CUtensorMap k, v;
};
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

bool maps_of(const CacheView& C, CUtensorMap* k, CUtensorMap* v, int box_rows = 16) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (const MapEntry& e : g_maps) {
    if (e.pages == C.pages && e.n_pages == C.n_pages && e.P == C.P && e.H == C.H && e.fmt == C.fmt &&
        e.box == box_rows) {
      *k = e.k;
      *v = e.v;
      return true;
    }
  }
  MapEntry& e = g_maps[g_map_next];
  if (!encode_rows(&e.k, C, 0, 256, box_rows) ||
      !encode_rows(&e.v, C, C.v_off(), C.fmt == K8V4_FORMAT_INT8 ? 256 : 128, box_rows)) {
    e.pages = nullptr;
    return false;
  }
  e.pages = C.pages;
  e.n_pages = C.n_pages;
  e.P = C.P;
  e.H = C.H;
  e.fmt = C.fmt;
  e.box = box_rows;
  g_map_next = (g_map_next + 1) % kMapCache;
  *k = e.k;
  *v = e.v;
  return true;
}

template <int FMT, bool QF32>
int launch_impl(const Launch& L, DecodeParams p, int n_seqs, float* out, bool partial) {
  p.L = layout_of(FMT, p.C.H, QF32 ? kMaxWorkersF32 : kMaxWorkers);
  CUtensorMap mk, mv;
  if (!maps_of(p.C, &mk, &mv)) return K8V4_ECUDA;
  auto kern = decode_kernel<FMT, QF32>;
  // up to 227 KB per CTA: ask for the largest shared-memory carveout
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.L.total) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return K8V4_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.C.H, n_seqs);
  cfg.blockDim = dim3(32 * p.L.workers);
  cfg.dynamicSmemBytes = p.L.total;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, mk, mv, p) != cudaSuccess) return K8V4_ECUDA;
  if (cudaGetLastError() != cudaSuccess) return K8V4_ECUDA;
  return partial ? launch_combine_partial(L, p.ws, p.splits, n_seqs, p.C.H, out)
                 : launch_combine(L, p.ws, p.splits, n_seqs, 1, p.C.H, out);
}

}  // namespace

bool decode_ws_supported(const CacheView& C) {
  return (C.fmt == K8V4_FORMAT_K8V4 || C.fmt == K8V4_FORMAT_INT8) && C.n_pages < (int64_t(1) << 31) &&
         C.page_bytes < (int64_t(1) << 39);
}

AttendPlan plan_decode(const CacheView& C, int n_seqs, int max_seq_len, int num_sms) {
  AttendPlan pl{};
  pl.n_q = 1;
  pl.n_groups = 1;
  pl.warps = kMaxWorkers;
  const int tiles = std::max(1, (max_seq_len + 15) / 16);
  const int64_t pairs = static_cast<int64_t>(C.H) * n_seqs;
  // one CTA per SM: split each (sequence, KV head) into the number of cell
  // ranges that minimises waves x (tiles per range + a CTA's fixed cost), each
  // range keeping at least 2 tiles per worker warp.  The fixed cost (q set-up,
  // pipeline fill, the workers' merge) is worth about kCtaFixedTiles tiles of
  // a CTA's streaming: without it, 32 sequences of 8,192 cells chose 8 waves of
  // 27-tile CTAs (120 us) over one wave of 256-tile CTAs (75 us).
  constexpr int kCtaFixedTiles = 32;
  const int max_splits = std::max(1, std::min(1024, tiles / (2 * kMaxWorkers)));
  int64_t best_cost = INT64_MAX;
  int best = 1;
  for (int sp = 1; sp <= max_splits; ++sp) {
    const int64_t waves = (pairs * sp + num_sms - 1) / num_sms;
    const int64_t cost = waves * ((tiles + sp - 1) / sp + kCtaFixedTiles);
    if (cost < best_cost) {
      best_cost = cost;
      best = sp;
    }
  }
  const int tps = (tiles + best - 1) / best;
  pl.cells_per_split = 16 * tps;
  pl.splits = (tiles + tps - 1) / tps;
  pl.ws_bytes = static_cast<size_t>(n_seqs) * pl.splits * C.H * kGqa * kPStride * sizeof(float);
  return pl;
}

namespace {
DecodeParams params_of(const Launch& L, const CacheView& C, const AttendPlan& plan, const void* q, const int32_t* pt,
                       int64_t max_pages, const int32_t* steps, int max_seq_len, float sm_scale, void* ws,
                       uint32_t wait_ns) {
  DecodeParams p;
  p.C = C;
  p.q = q;
  p.pt = pt;
  p.max_pages = max_pages;
  p.steps = steps;
  p.max_seq_len = max_seq_len;
  p.cells_per_split = plan.cells_per_split;
  p.splits = plan.splits;
  p.cell_base = 0;
  p.cell_limit = max_seq_len;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.ws = static_cast<float*>(ws);
  p.status = L.status;
  p.k_new = nullptr;
  p.v_new = nullptr;
  p.kv_bf16 = 1;
  p.wait_ns = wait_ns ? wait_ns : kWaitDefaultNs;
  p.withhold = withheld_copy();
  p.page_div = FastDiv(static_cast<uint32_t>(C.P));
  return p;
}
int dispatch(const Launch& L, const DecodeParams& p, int fmt, bool f32, int n_seqs, float* out, bool partial) {
  if (fmt == K8V4_FORMAT_K8V4)
    return f32 ? launch_impl<K8V4_FORMAT_K8V4, true>(L, p, n_seqs, out, partial)
               : launch_impl<K8V4_FORMAT_K8V4, false>(L, p, n_seqs, out, partial);
  return f32 ? launch_impl<K8V4_FORMAT_INT8, true>(L, p, n_seqs, out, partial)
             : launch_impl<K8V4_FORMAT_INT8, false>(L, p, n_seqs, out, partial);
}

template <int NQ>
int launch_verify_ws_n(const Launch& L, const VerifyWsParams& p, int n_seqs, float* out) {
  CUtensorMap mk, mv;
  if (!maps_of(p.C, &mk, &mv)) return K8V4_ECUDA;
  auto kern = verify_ws_kernel<NQ>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.L.total) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return K8V4_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.C.H, n_seqs);
  cfg.blockDim = dim3(32 * 4 * kVTeams);
  cfg.dynamicSmemBytes = p.L.total;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, mk, mv, p) != cudaSuccess) return K8V4_ECUDA;
  if (cudaGetLastError() != cudaSuccess) return K8V4_ECUDA;
  return launch_combine(L, p.ws, p.splits, n_seqs, NQ, p.C.H, out);
}
}  // namespace

int launch_decode(const Launch& L, const CacheView& C, const AttendPlan& plan, const void* q, int q_dtype,
                  const int32_t* pt, int64_t max_pages, const int32_t* steps, int n_seqs, int max_seq_len,
                  float sm_scale, float* out, void* ws, const void* k_new, const void* v_new, int kv_dtype,
                  uint32_t wait_ns) {
  if (n_seqs == 0) return K8V4_OK;
  DecodeParams p = params_of(L, C, plan, q, pt, max_pages, steps, max_seq_len, sm_scale, ws, wait_ns);
  p.k_new = k_new;
  p.v_new = v_new;
  p.kv_bf16 = kv_dtype == K8V4_BF16 ? 1 : 0;
  return dispatch(L, p, C.fmt, q_dtype == K8V4_F32, n_seqs, out, false);
}

int launch_decode_partial(const Launch& L, const CacheView& C, const AttendPlan& plan, const void* q, int q_dtype,
                          const int32_t* pt, int64_t max_pages, const int32_t* steps, int n_seqs,
                          int max_seq_len, int cell_begin, int cell_end, float sm_scale, float* partial, void* ws,
                          uint32_t wait_ns) {
  if (n_seqs == 0) return K8V4_OK;
  DecodeParams p = params_of(L, C, plan, q, pt, max_pages, steps, max_seq_len, sm_scale, ws, wait_ns);
  p.cell_base = cell_begin;
  p.cell_limit = cell_end;
  return dispatch(L, p, C.fmt, q_dtype == K8V4_F32, n_seqs, partial, true);
}


bool verify_ws_supported(const CacheView& C, int n_q, int q_dtype) {
  return C.fmt == K8V4_FORMAT_K8V4 && q_dtype == K8V4_BF16 && n_q >= 2 && n_q <= kVMaxQ &&
         C.n_pages < (int64_t(1) << 31) && C.page_bytes < (int64_t(1) << 39);
}

AttendPlan plan_verify_ws(const CacheView& C, int n_seqs, int n_q, int max_seq_len, int num_sms) {
  AttendPlan pl{};
  pl.n_q = n_q;
  pl.n_groups = 1;
  pl.warps = 4 * kVTeams;
  const int tiles = std::max(1, (max_seq_len + 15) / 16);
  // one CTA per SM at a time; about four CTAs per SM over the grid, so that the
  // splits past a short sequence's end (which return at once) leave no SM idle,
  // and at least four tiles per team
  const int64_t pairs = static_cast<int64_t>(C.H) * n_seqs;
  int64_t splits = (4ll * num_sms + pairs - 1) / std::max<int64_t>(pairs, 1);
  splits = std::max<int64_t>(1, std::min<int64_t>(splits, std::max(1, tiles / (4 * kVTeams))));
  const int tps = static_cast<int>((tiles + splits - 1) / splits);
  pl.cells_per_split = 16 * tps;
  pl.splits = (tiles + tps - 1) / tps;
  pl.ws_bytes = static_cast<size_t>(n_seqs) * pl.splits * n_q * C.H * kGqa * kPStride * sizeof(float);
  return pl;
}

int launch_verify_ws(const Launch& L, const CacheView& C, const void* q, const int32_t* pt, int64_t max_pages,
                     const int32_t* steps, int n_seqs, int n_q, int max_seq_len, float sm_scale, float* out, void* ws) {
  if (n_seqs == 0) return K8V4_OK;
  const AttendPlan plan = plan_verify_ws(C, n_seqs, n_q, max_seq_len, L.num_sms);
  VerifyWsParams p;
  p.C = C;
  p.q = static_cast<const uint16_t*>(q);
  p.pt = pt;
  p.max_pages = max_pages;
  p.steps = steps;
  p.max_seq_len = max_seq_len;
  p.cells_per_split = plan.cells_per_split;
  p.splits = plan.splits;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.ws = static_cast<float*>(ws);
  p.status = L.status;
  p.wait_ns = wait_limit_ns() ? wait_limit_ns() : kWaitDefaultNs;
  p.page_div = FastDiv(static_cast<uint32_t>(C.P));
  p.L = vlayout_of(C.H, n_q);
  if (p.L.total > kSmemCap + 1024) return K8V4_EINVAL;
  switch (n_q) {
    case 2: return launch_verify_ws_n<2>(L, p, n_seqs, out);
    case 3: return launch_verify_ws_n<3>(L, p, n_seqs, out);
    case 4: return launch_verify_ws_n<4>(L, p, n_seqs, out);
    case 5: return launch_verify_ws_n<5>(L, p, n_seqs, out);
    case 6: return launch_verify_ws_n<6>(L, p, n_seqs, out);
    case 7: return launch_verify_ws_n<7>(L, p, n_seqs, out);
    case 8: return launch_verify_ws_n<8>(L, p, n_seqs, out);
    default: return K8V4_EINVAL;
  }
}

}  // namespace k8v4
