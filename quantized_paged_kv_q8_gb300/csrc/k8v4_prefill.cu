// Chunked-prefill attention over the k8v4 paged cache on the 5th-generation
// tensor cores (tcgen05 + TMEM): the prompt form of the hybrid-KV pull request's
// fused attention ("How": mode 3 runs for decode, prefill and verify; q is not
// rotated, the output is computed in rotated space and rotated back).
//
// One CTA owns 128 query rows = 16 tokens x the 8 query heads of one KV head
// (GQA packing: all 128 rows read the same K/V), and sweeps the cells visible to
// them in tiles of 64:
//   1. 16-byte cp.async copies bring the tile's raw runs (int8 K, K scales, V
//      nibbles, fp16 V scales) into shared memory (double-buffered);
//   2. all 256 threads dequantise it into fp16 operand tiles in the 128-byte
//      swizzled layouts tcgen05 reads: K codes (exact in fp16) K-major, and
//      Vhat_rot = (q - 8) * d as two fp16 planes V1 = RN(Vhat), V2 = Vhat - V1
//      (both exact), MN-major;
//   3. one thread issues S_h = Q_h K_h^T for the two 128-lane halves (separate
//      TMEM accumulators, because each half has its own K scale), M=128, N=64,
//      K=16 per instruction, and commits to an mbarrier;
//   4. all 16 warps (TMEM lane = row; four threads per row, 16 cells each) read
//      S, apply the K scales and the online softmax (log2 domain), and write
//      P * 2^7 back into TMEM (over S) as two fp16 planes P1 = RN(P),
//      P2 = RN(P - P1) (22 significant bits);
//   5. one thread issues O_tile += P1 V1 + P1 V2 + P2 V1 (A from TMEM, M=128,
//      N=256, K=16; the dropped P2 V2 term is below 2^-22 of the product).
//      P is taken against a per-row reference maximum that moves only when a
//      tile's maximum exceeds it by more than 2^8 (so P * 2^7 <= 2^15 stays in
//      fp16); while no row moves its reference, consecutive tiles accumulate in
//      the same TMEM tile.  When some row moves it, or after kChain tiles, every
//      thread folds its 64 dims of O_tile into an fp32 register accumulator,
//      o = (o + O_tile) * 2^(m_old - m_new), and the next tile starts a fresh
//      TMEM tile: accumulating all tiles inside TMEM would let the tensor
//      core's per-instruction accumulation rounding build up over thousands of
//      steps.
// fp16 operands with one rounding would leave errors near 1e-4 at 2^18 cells,
// above the 2e-5 bar; the split planes bring them to the fp32 level.
// The epilogue divides by l, applies the inverse Walsh-Hadamard transform
// (out = (H/16) o) per row and writes fp32 rows.
//
// Every mbarrier wait is bounded: on timeout the kernel records an error in the
// device status word, stops issuing work, waits (bounded) for its own
// outstanding copies and MMAs, frees its TMEM and returns.
#include <algorithm>

#include "k8v4_tc.cuh"

namespace k8v4 {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRows = 128;            // query rows per CTA (16 tokens x 8 heads)
constexpr int kTokens = kRows / kGqa; // 16
constexpr int kTileN = 64;            // cells per tile
constexpr int kThreads = 512;

// shared memory map (bytes); every operand tile 1024-byte aligned
constexpr int kQOff = 0;                       // Q fp16 [4 chunks][128 rows][128 B]  = 65536
constexpr int kKfOff = kQOff + 65536;          // K fp16 [4 chunks][64 cells][128 B]  = 32768
constexpr int kVfOff = kKfOff + 32768;         // Vhat fp16 2 planes x [4 atoms][64 cells][128 B] = 65536
constexpr int kRawK = 64 * 256;                // raw tile: K codes [64][256]
constexpr int kRawV = 64 * 128;                //           V nibbles [64][128]
constexpr int kRawKs = 64 * 8;                 //           K scales [64][2] f32
constexpr int kRawVs = 64 * 16;                //           V scales [64][8] f16
constexpr int kRawBytes = kRawK + kRawV + kRawKs + kRawVs;   // 26112
constexpr int kRawOff = kVfOff + 65536;        // 2 raw stages
constexpr int kBarOff = kRawOff + 2 * kRawBytes;             // mbarriers + tmem slot
constexpr int kKsBufOff = kBarOff + 64;                      // K scales of the current tile [64][2] f32
constexpr int kRedOff = kKsBufOff + 512;                     // [4][128] f32 exchange + [128] f32 factors
constexpr int kSmemBytes = kRedOff + 2048 + 512;
static_assert(kRawOff % 1024 == 0, "alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
// the epilogue reuses [kKfOff, kKfOff + 128 KB) as a fp32 [128][256] row buffer
static_assert(kBarOff - kKfOff >= 128 * 256 * 4, "epilogue buffer");

constexpr uint32_t kTmemCols = 512;    // S buffers [0,128) and [128,256) (S0 | S1 each; P1/P2 reuse
                                       // the buffer's S0 columns), O_tile [256,512)
constexpr uint32_t kSBuf = 128, kS0Col = 0, kS1Col = 64, kOCol = 256, kP1Col = 0, kP2Col = 32;
constexpr uint32_t kWaitDefaultNs = 1000000000u;   // 1 s: the default bound of an mbarrier wait
constexpr float kSlack = 8.0f;                // log2 headroom of P above its row's reference maximum
constexpr int kChain = 4;                     // tiles accumulated in one TMEM O tile at most

struct PrefillParams {
  CacheView C;
  const uint16_t* q;       // bf16 [n_seqs][n_q_tok][HQ][256]
  const int32_t* pt;       // [n_seqs][max_pages]
  int64_t max_pages;
  const int32_t* steps;    // [n_seqs][n_q_tok] or null (causal)
  int seq_len, n_q_tok;
  int splits, cells_per_split;   // split-K over the cells (1 split: the whole range)
  float sm_scale_log2;
  float* out;              // final rows [n_seqs][n_q_tok][HQ][256], or null
  float* ws;               // else partial rows (o[256], m, l) for the combine
  int* status;
  uint32_t wait_ns;        // bound of the pipeline's mbarrier waits, nanoseconds
};

// ---------------------------------------------------------------- the kernel
// 16 warps.  Row r of the 128 query rows lives in TMEM lane r and is served by
// four threads, one per "part" (tid = part * 128 + r): each part reads 16 of the
// tile's 64 scores and owns 64 of the 256 output dims (its share of O stays in
// registers as fp32 across tiles).
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = tid & (kRows - 1), part = tid >> 7;
  const int g = blockIdx.y;
  const int tok0 = blockIdx.x * kTokens;
  const int b = blockIdx.z / p.splits, split = blockIdx.z % p.splits;
  const CacheView& C = p.C;
  const int HQ = C.H * kGqa;
  const int32_t* pt = p.pt + static_cast<int64_t>(b) * p.max_pages;
  const uint16_t* qs = p.q + static_cast<int64_t>(b) * p.n_q_tok * HQ * kD;

  const uint32_t bar_s = sbase + kBarOff, bar_o = sbase + kBarOff + 8, bar_d = sbase + kBarOff + 32;
  const uint32_t tmem_slot = sbase + kBarOff + 16;
  int* nmax_s = reinterpret_cast<int*>(smem + kBarOff + 28);
  float* red = reinterpret_cast<float*>(smem + kRedOff);           // [4][128] partial maxima / sums
  float* fsc = reinterpret_cast<float*>(smem + kRedOff + 2048);    // [128] score factor per row

  // ---- visibility of this thread's row
  int my_vis = 0;
  {
    const int t = tok0 + row / kGqa;
    if (t < p.n_q_tok) {
      int v = p.steps ? p.steps[static_cast<int64_t>(b) * p.n_q_tok + t] : p.seq_len - p.n_q_tok + t + 1;
      if (v < 0 || v > p.seq_len) {
        if (part == 0) record_status(p.status, K8V4_ERANGE);
        v = v < 0 ? 0 : p.seq_len;
      }
      my_vis = v;
    }
  }
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_d, 1);
    *nmax_s = 0;
    *reinterpret_cast<int*>(smem + kBarOff + 24) = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (part == 0 && my_vis > 0) atomicMax(nmax_s, my_vis);
  __syncthreads();
  // a split past every row's visible cells (a short sequence of a verify batch)
  // only marks its partial rows empty (m = -inf: the combine skips them) and
  // leaves before tensor memory, Q and the pipeline are set up
  if (p.ws && split * p.cells_per_split >= *nmax_s) {
    for (int r = tid; r < kRows; r += kThreads) {
      const int t = tok0 + r / kGqa, h = r % kGqa;
      if (t >= p.n_q_tok) continue;
      float* dst = p.ws + ((((static_cast<int64_t>(b) * p.splits + split) * p.n_q_tok + t) * HQ) + g * kGqa + h) * 260;
      dst[256] = -INFINITY;
      dst[257] = 0.0f;
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    return;
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);

  // ---- Q rows -> fp16 with a per-row power-of-two scale, swizzled K-major;
  // the four parts of a row convert dims [64 part, 64 part + 64)
  {
    const int t = tok0 + row / kGqa, h = row % kGqa;
    uint4 raw[8];
    if (t < p.n_q_tok) {
      const uint4* src = reinterpret_cast<const uint4*>(qs + (static_cast<int64_t>(t) * HQ + g * kGqa + h) * kD + 64 * part);
#pragma unroll
      for (int i = 0; i < 8; ++i) raw[i] = src[i];
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) raw[i] = make_uint4(0, 0, 0, 0);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[u] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[u] & 0xffff0000u)));
      }
    }
    red[part * kRows + row] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(red[row], red[kRows + row]), fmaxf(red[2 * kRows + row], red[3 * kRows + row]));
    const int ex = amax > 0.0f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127 : 0;
    const int sh = max(-100, min(100, 14 - ex));
    const float up = ldexpf(1.0f, sh);
    if (part == 0) fsc[row] = p.sm_scale_log2 * ldexpf(1.0f, -sh);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
      uint32_t hv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float a = __fmul_rn(__uint_as_float(w[u] << 16), up);
        const float b = __fmul_rn(__uint_as_float(w[u] & 0xffff0000u), up);
        const __half2 h2 = __floats2half2_rn(a, b);
        hv[u] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      // dims 64 part + 8i .. +7: chunk = part, unit = i
      sts128(sbase + kQOff + part * 16384 + swz(row, i), hv[0], hv[1], hv[2], hv[3]);
    }
  }
  __syncthreads();
  const float my_f = fsc[row];
  // this CTA's tiles: [tile_lo, tile_lo + n_tiles) of the cells visible to any row
  const int c_begin = split * p.cells_per_split;
  const int c_end = min(*nmax_s, c_begin + p.cells_per_split);
  const int tile_lo = c_begin / kTileN;
  const int n_tiles = c_end > c_begin ? (c_end - c_begin + kTileN - 1) / kTileN : 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kBarOff + 16);
  const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;

  // ---- raw tile loader (all threads, 16-byte cp.async)
  // page ids are read one load ahead (tiles are staged in order 0, 1, 2, ...)
  auto fetch_page = [&](int tile) -> int64_t {
    const int64_t pidx = static_cast<int64_t>(tile_lo + tile) * kTileN / C.P;
    return (tile < n_tiles && pidx < p.max_pages) ? static_cast<int64_t>(pt[pidx]) : -1;
  };
  int64_t pf_page = fetch_page(0);
  auto load_raw = [&](int tile, int stage) {
    const int cell0 = (tile_lo + tile) * kTileN;
    const uint32_t dst = sbase + kRawOff + stage * kRawBytes;
    const int64_t page = pf_page;
    pf_page = fetch_page(tile + 1);
    if (page < 0 || page >= C.n_pages) return false;
    const int slot0 = cell0 % C.P;       // P is a multiple of 64 here
    const uint8_t* base = C.pages + page * C.page_bytes;
    // raw K chunk kk of cell j sits at 16 * (kk ^ (j & 15)), raw V block b of cell
    // j at 16 * (b ^ (j & 7)): eight consecutive cells then hit eight different
    // bank groups when the converters read one chunk of each
    for (int i = tid; i < 64 * 16; i += kThreads) {              // K codes
      const int j = i >> 4, kk = i & 15;
      cp_async16(dst + j * 256 + 16 * (kk ^ (j & 15)), base + (static_cast<int64_t>(slot0 + j) * C.H + g) * 256 + 16 * kk);
    }
    {                                                            // V nibbles: 64 cells x 8 blocks
      const int j = tid >> 3, kk = tid & 7;
      cp_async16(dst + kRawK + j * 128 + 16 * (kk ^ (j & 7)),
                 base + C.v_off() + (static_cast<int64_t>(slot0 + j) * C.H + g) * 128 + 16 * kk);
    }
    if (tid < 64) {
      const int64_t r = static_cast<int64_t>(slot0 + tid) * C.H + g;
      cp_async8(dst + kRawK + kRawV + 8 * tid, base + C.ks_off() + r * 8);
      cp_async16(dst + kRawK + kRawV + kRawKs + 16 * tid, base + C.vs_off() + r * 16);
    }
    return true;
  };

  // ---- dequantisation of one raw stage into the operand tiles
  auto convert_k = [&](int stage) {                 // K codes -> Kf (fp16, exact), K scales -> ks buffer
    const uint32_t raw = sbase + kRawOff + stage * kRawBytes;
    for (int i = tid; i < 64 * 16; i += kThreads) {  // (cell j, 16-byte chunk kk); j fastest so a
      const int j = i & 63, kk = i >> 6;              // quarter-warp covers 8 cells of one chunk
      const uint4 w = lds128(raw + j * 256 + 16 * (kk ^ (j & 15)));
      uint32_t h[8];
      i8x4_to_f16(w.x, h[0], h[1]);
      i8x4_to_f16(w.y, h[2], h[3]);
      i8x4_to_f16(w.z, h[4], h[5]);
      i8x4_to_f16(w.w, h[6], h[7]);
      const int dim = 16 * kk, chunk = dim >> 6, unit = (dim & 63) >> 3;
      const uint32_t dst = sbase + kKfOff + chunk * 8192;
      sts128(dst + swz(j, unit), h[0], h[1], h[2], h[3]);
      sts128(dst + swz(j, unit + 1), h[4], h[5], h[6], h[7]);
    }
    if (tid < 64)
      reinterpret_cast<float2*>(smem + kKsBufOff)[tid] =
          reinterpret_cast<const float2*>(smem + kRawOff + stage * kRawBytes + kRawK + kRawV)[tid];
  };
  auto convert_v = [&](int stage) {                 // V nibbles x d -> Vf planes (fp16, exact split)
    const uint32_t raw = sbase + kRawOff + stage * kRawBytes;
    const int j = tid & 63, b = tid >> 6;           // (cell j, block b): one item per thread, j fastest
    const uint4 w = lds128(raw + kRawK + j * 128 + 16 * (b ^ (j & 7)));
    const __half dh = *reinterpret_cast<const __half*>(smem + kRawOff + stage * kRawBytes + kRawK + kRawV +
                                                          kRawKs + 16 * j + 2 * b);
    const __half2 d2 = __halves2half2(dh, dh);
    const uint32_t ws4[4] = {w.x, w.y, w.z, w.w};
    uint32_t lo[2][8], hi[2][8];   // [plane] dims 32b + (0..15) and 32b + 16 + (0..15), 8 pairs each
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t t01 = prmt(ws4[q], 0u, 0x5140u);   // {b0, 0, b1, 0}
      const uint32_t t23 = prmt(ws4[q], 0u, 0x5342u);   // {b2, 0, b3, 0}
      nib_vhat(t01, 0, d2, lo[0][2 * q], lo[1][2 * q]);
      nib_vhat(t23, 0, d2, lo[0][2 * q + 1], lo[1][2 * q + 1]);
      nib_vhat(t01, 4, d2, hi[0][2 * q], hi[1][2 * q]);
      nib_vhat(t23, 4, d2, hi[0][2 * q + 1], hi[1][2 * q + 1]);
    }
    const int atom = b >> 1, unit0 = 4 * (b & 1);
#pragma unroll
    for (int pl = 0; pl < 2; ++pl) {
      const uint32_t dst = sbase + kVfOff + pl * 32768 + atom * 8192;
      sts128(dst + swz(j, unit0), lo[pl][0], lo[pl][1], lo[pl][2], lo[pl][3]);
      sts128(dst + swz(j, unit0 + 1), lo[pl][4], lo[pl][5], lo[pl][6], lo[pl][7]);
      sts128(dst + swz(j, unit0 + 2), hi[pl][0], hi[pl][1], hi[pl][2], hi[pl][3]);
      sts128(dst + swz(j, unit0 + 3), hi[pl][4], hi[pl][5], hi[pl][6], hi[pl][7]);
    }
  };
  // ---- tensor-core work (one thread issues)
  // The operand tiles sit at fixed addresses, so their descriptors are built
  // once; a descriptor of base + off is the base descriptor plus off / 16 (the
  // 14-bit address field cannot carry: shared addresses stay below 2^18).
  const uint64_t dq0 = smem_desc(sbase + kQOff, 16, 1024);
  const uint64_t dk0 = smem_desc(sbase + kKfOff, 16, 1024);
  const uint64_t dv0 = smem_desc(sbase + kVfOff, 8192, 1024);
  auto issue_qk = [&](int buf) {                  // S[buf]_h = Q_h Kf_h^T, fresh accumulators
    tc_fence_after();
    constexpr uint32_t idS = idesc_f16(128, 64, false, false);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int chunk = 2 * h + (kk >> 2);
        const uint32_t off = (kk & 3) * 32;
        const uint64_t a = dq0 + ((chunk * 16384 + off) >> 4);
        const uint64_t b = dk0 + ((chunk * 8192 + off) >> 4);
        mma_f16(tmem + kSBuf * buf + (h ? kS1Col : kS0Col), a, b, idS, kk > 0 ? 1u : 0u);
      }
    }
    mma_commit(bar_s);
  };
  auto issue_pv = [&](int buf, bool fresh) {      // O_tile (+)= P1 V1 + P1 V2 + P2 V1 (P in S[buf])
    tc_fence_after();
    constexpr uint32_t idO = idesc_f16(128, 256, false, true);
    const uint32_t pb = tmem + kSBuf * buf;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {               // 16 cells = 8 TMEM columns of fp16 pairs
      const uint64_t v1 = dv0 + ((kk * 2048) >> 4);
      const uint64_t v2 = dv0 + ((32768 + kk * 2048) >> 4);
      mma_f16_ta(tmem + kOCol, pb + kP1Col + 8 * kk, v1, idO, (kk > 0 || !fresh) ? 1u : 0u);
      mma_f16_ta(tmem + kOCol, pb + kP1Col + 8 * kk, v2, idO, 1u);
      mma_f16_ta(tmem + kOCol, pb + kP2Col + 8 * kk, v1, idO, 1u);
    }
    mma_commit(bar_o);
  };

  // Pipeline, iteration i (S double-buffered in TMEM; Kf, Vf, O_tile single):
  //   (a) wait QK(i), softmax(i)            -- the tensor core runs PV(i-1)
  //   (b) wait PV(i-1), merge O_tile(i-1)
  //   (c) convert K(i+1), issue QK(i+1)
  //   (d) convert V(i), issue PV(i)         -- QK(i+1) runs meanwhile
  //   then prefetch raw(i+2) into the stage V(i) came from.
  bool ok_tile[2] = {false, false};
  if (n_tiles > 0) ok_tile[0] = load_raw(0, 0);
  cp_async_commit();
  if (n_tiles > 1) ok_tile[1] = load_raw(1, 1);
  cp_async_commit();

  float o_run[64];                 // this part's 64 dims of the row's O (rotated space)
#pragma unroll
  for (int i = 0; i < 64; ++i) o_run[i] = 0.0f;
  float m_run = -INFINITY, l_part = 0.0f, alpha = 1.0f;   // m_run: the row's reference maximum
  bool need = false;               // this row moved its reference on the current tile
  int chain = 0;                   // tiles in the current TMEM O tile
  int* flag_s = reinterpret_cast<int*>(smem + kBarOff + 24);   // a wait timed out (set by warp 0)
  uint32_t phase_s = 0, phase_o = 0;
  bool failed = false;
  uint32_t valid_bits = 0;         // bit (t & 1): tile t's page id was valid

  // wait on `bar` (warp 0 polls) and OR `pred` over the CTA: 1 / 0, or -1 on timeout
  auto wait_bar_or = [&](uint32_t bar, uint32_t& phase, bool pred) -> int {
    if (warp == 0 && !mbar_wait(bar, phase & 1, p.wait_ns) && lane == 0) *reinterpret_cast<volatile int*>(flag_s) = 1;
    ++phase;
    const int any = __syncthreads_or(pred ? 1 : 0);
    if (*reinterpret_cast<volatile int*>(flag_s)) { failed = true; return -1; }
    tc_fence_after();
    return any;
  };
  auto wait_bar = [&](uint32_t bar, uint32_t& phase) -> bool {   // one warp polls, all synchronise
    if (warp == 0 && !mbar_wait(bar, phase & 1, p.wait_ns)) failed = true;
    ++phase;
    if (__syncthreads_or(failed ? 1 : 0)) { failed = true; return false; }
    tc_fence_after();
    return true;
  };
  auto merge = [&](float a) {      // o_run = (o_run + O_tile) * a (IEEE fp32)
    float o[32];
    const float2 a2 = make_float2(a, a);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      tmem_ld32(tmem + lane_base + kOCol + 64 * part + 32 * h, o);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 r = __fmul2_rn(__fadd2_rn(make_float2(o_run[32 * h + i], o_run[32 * h + i + 1]),
                                               make_float2(o[i], o[i + 1])), a2);
        o_run[32 * h + i] = r.x;
        o_run[32 * h + i + 1] = r.y;
      }
    }
    tc_fence_before();
  };
  auto stage_k = [&](int t) {      // (c): convert K(t) and issue QK(t)
    cp_async_wait<0>();            // raw(t) is the most recently committed copy group
    const bool ok = __syncthreads_and(ok_tile[t & 1] ? 1 : 0) != 0;   // also: raw(t) visible to all
    valid_bits = ok ? (valid_bits | (1u << (t & 1))) : (valid_bits & ~(1u << (t & 1)));
    convert_k(t & 1);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) issue_qk(t & 1);
  };

  if (n_tiles > 0) stage_k(0);

  for (int it = 0; it < n_tiles; ++it) {
    const int buf = it & 1;
    const bool valid_cur = (valid_bits >> buf) & 1u;
    if (!valid_cur && tid == 0) record_status(p.status, K8V4_ERANGE);
    // ---- (a) scores of tile it: this part's 16 cells, row max across the parts
    if (!wait_bar(bar_s, phase_s)) break;
    const int cell0 = (tile_lo + it) * kTileN;
    float sc[16];
    {
      const float* ks = reinterpret_cast<const float*>(smem + kKsBufOff);
      float a[16], b[16];
      tmem_ld16(tmem + lane_base + kSBuf * buf + kS0Col + 16 * part, a);
      tmem_ld16(tmem + lane_base + kSBuf * buf + kS1Col + 16 * part, b);
      const int vis = valid_cur ? my_vis - cell0 - 16 * part : 0;   // cells [0, vis) of this part
      // sc holds the unscaled scores; my_f > 0, so the maximum commutes with it
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 16; c += 2) {
        const float4 k2 = *reinterpret_cast<const float4*>(ks + 2 * (16 * part + c));
        sc[c] = k2.x * a[c] + k2.y * b[c];
        sc[c + 1] = k2.z * a[c + 1] + k2.w * b[c + 1];
      }
      if (vis < 16) {
#pragma unroll
        for (int c = 0; c < 16; ++c) sc[c] = c < vis ? sc[c] : -INFINITY;
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) mx = fmaxf(mx, sc[c]);
      red[part * kRows + row] = mx * my_f;
    }
    __syncthreads();
    {
      const float mt = fmaxf(fmaxf(red[row], red[kRows + row]), fmaxf(red[2 * kRows + row], red[3 * kRows + row]));
      // the reference moves only when the tile's maximum exceeds it by more than
      // kSlack (always on the row's first visible tile: m_run = -inf)
      need = mt > m_run + kSlack;
      const float m_new = need ? mt : m_run;
      alpha = need ? exp2f(m_run - m_new) : 1.0f;                  // 0 on the first visible tile
      // p * 2^7 = exp2(s - m + 7) <= 2^15; the 2^7 keeps small probabilities normal in fp16
      const float mu = (m_new == -INFINITY ? 0.0f : m_new) - 7.0f;
      m_run = m_new;
      float p1v[8], p2v[8];
      float2 psum2 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int c = 0; c < 16; c += 2) {
        const float a = ex2_ftz(fmaf(sc[c], my_f, -mu)), b = ex2_ftz(fmaf(sc[c + 1], my_f, -mu));
        // hi plane: fp16(a); lo plane: fp16 of the exact fp32 residual
        const __half2 h1 = __floats2half2_rn(a, b);
        const float2 f1 = __half22float2(h1);
        const float2 r = __ffma2_rn(f1, make_float2(-1.0f, -1.0f), make_float2(a, b));   // exact
        const __half2 h2 = __floats2half2_rn(r.x, r.y);
        psum2 = __fadd2_rn(psum2, make_float2(a, b));
        p1v[c >> 1] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&h1));
        p2v[c >> 1] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&h2));
      }
      l_part = l_part * alpha + (psum2.x + psum2.y);
      // P planes overwrite S[buf]'s S0 columns: every part has read its scores (barrier above)
      tmem_st8(tmem + lane_base + kSBuf * buf + kP1Col + 8 * part, p1v);
      tmem_st8(tmem + lane_base + kSBuf * buf + kP2Col + 8 * part, p2v);
    }
    tc_fence_before();
    // ---- (b) PV(it-1) done (Vf is free again); if some row moved its reference
    // (or the chain is long), fold the TMEM O tile into the registers
    bool fresh = true;
    if (it > 0) {
      const int any = wait_bar_or(bar_o, phase_o, need || chain >= kChain);
      if (any < 0) break;
      fresh = any != 0;
      if (fresh) merge(alpha);
    }
    chain = fresh ? 1 : chain + 1;
    // ---- (c) next tile's K and its scores
    if (it + 1 < n_tiles) stage_k(it + 1);
    // ---- (d) this tile's V and O_tile = P V
    convert_v(buf);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) issue_pv(buf, fresh);
    if (it + 2 < n_tiles) ok_tile[buf] = load_raw(it + 2, buf);   // raw stage `buf` is consumed
    cp_async_commit();
  }
  // ---- the last tile's O_tile
  if (!failed && n_tiles > 0) {
    if (wait_bar(bar_o, phase_o)) merge(1.0f);
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- epilogue: o / l, inverse Walsh-Hadamard transform, write rows
  if (!failed) {
    red[part * kRows + row] = l_part;
    __syncthreads();
    const float l = (red[row] + red[kRows + row]) + (red[2 * kRows + row] + red[3 * kRows + row]);
    // final rows: O / l (both carry the 2^7 factor of P); partial rows keep O, m and l
    const float inv = p.ws ? 1.0f : (l > 0.0f ? 1.0f / l : 0.0f);
    if (p.ws && part == 0) fsc[row] = l;             // the row's l for the partial writer
    float* mrow = reinterpret_cast<float*>(smem + kRedOff);        // red is free again after the read above
    __syncthreads();
    if (p.ws && part == 0) mrow[row] = m_run;
    float* rowbuf = reinterpret_cast<float*>(smem + kKfOff);     // [128][256] fp32, rotated by 4 * row
#pragma unroll
    for (int i = 0; i < 64; i += 4) {
      const int d = 64 * part + i;
      *reinterpret_cast<float4*>(rowbuf + row * 256 + ((d + 4 * row) & 255)) =
          make_float4(o_run[i] * inv, o_run[i + 1] * inv, o_run[i + 2] * inv, o_run[i + 3] * inv);
    }
    __syncthreads();
    for (int r = warp; r < kRows; r += kThreads / 32) {
      const int t = tok0 + r / kGqa, h = r % kGqa;
      if (t >= p.n_q_tok) continue;
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; e += 4) {
        const float4 x = *reinterpret_cast<const float4*>(rowbuf + r * 256 + ((8 * lane + e + 4 * r) & 255));
        v[e] = x.x; v[e + 1] = x.y; v[e + 2] = x.z; v[e + 3] = x.w;
      }
#pragma unroll
      for (int hh = 1; hh < 8; hh <<= 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (e & hh) continue;
          const float a = v[e], b = v[e + hh];
          v[e] = a + b;
          v[e + hh] = a - b;
        }
      }
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = __shfl_xor_sync(kFull, v[e], m);
          v[e] = upper ? x - v[e] : v[e] + x;
        }
      }
      float* dst = p.ws ? p.ws + ((((static_cast<int64_t>(b) * p.splits + split) * p.n_q_tok + t) * HQ) + g * kGqa + h) * 260
                        : p.out + ((static_cast<int64_t>(b) * p.n_q_tok + t) * HQ + g * kGqa + h) * kD;
      reinterpret_cast<float4*>(dst + 8 * lane)[0] = make_float4(v[0] * 0.0625f, v[1] * 0.0625f, v[2] * 0.0625f, v[3] * 0.0625f);
      reinterpret_cast<float4*>(dst + 8 * lane)[1] = make_float4(v[4] * 0.0625f, v[5] * 0.0625f, v[6] * 0.0625f, v[7] * 0.0625f);
      if (p.ws && lane == 0) {
        dst[256] = mrow[r];
        dst[257] = fsc[r];
      }
    }
  } else {
    if (tid == 0) {
      record_status(p.status, K8V4_ECUDA);
      mma_commit(bar_d);                     // let in-flight MMAs drain (bounded by the default)
      (void)mbar_wait(bar_d, 0, kWaitDefaultNs);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // a combine launched as a programmatic dependent may start: every partial is written
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

int launch_prefill(const Launch& L, const CacheView& C, const void* q, const int32_t* pt, int64_t max_pages,
                   int seq_len, int n_q_tok, const int32_t* steps, float sm_scale, float* out) {
  if (C.P % kTileN != 0) return K8V4_EINVAL;          // tiles of 64 cells never straddle a page
  if (n_q_tok == 0) return K8V4_OK;
  PrefillParams p;
  p.C = C;
  p.q = static_cast<const uint16_t*>(q);
  p.pt = pt;
  p.max_pages = max_pages;
  p.steps = steps;
  p.seq_len = seq_len;
  p.n_q_tok = n_q_tok;
  p.splits = 1;
  p.cells_per_split = seq_len + kTileN;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.out = out;
  p.ws = nullptr;
  p.status = L.status;
  p.wait_ns = wait_limit_ns() ? wait_limit_ns() : kWaitDefaultNs;
  if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return K8V4_ECUDA;
  const dim3 grid((n_q_tok + kTokens - 1) / kTokens, C.H, 1);
  prefill_kernel<<<grid, kThreads, kSmemBytes, L.stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? K8V4_OK : K8V4_ECUDA;
}

// Verify on the prefill kernel: the n_q (<= 16) queries of a sequence are the
// CTA's tokens; the cells are split over CTAs, each writing partial rows that
// launch_combine merges.
AttendPlan plan_verify_tc(const CacheView& C, int n_seqs, int n_q, int max_seq_len, int num_sms) {
  AttendPlan pl{};
  pl.n_q = n_q;
  pl.n_groups = 1;
  pl.warps = kThreads / 32;
  const int tiles = max(1, (max_seq_len + kTileN - 1) / kTileN);
  // many short CTAs (one resident per SM at a time): the block scheduler hands
  // the next split to whichever SM frees up, so sequences of unequal length
  // balance out and the tail is one short CTA; at least two CTAs per SM
  constexpr int kTilesPerSplit = 16;
  const int64_t pairs = static_cast<int64_t>(C.H) * n_seqs;
  int64_t splits = std::max<int64_t>((2ll * num_sms + pairs - 1) / pairs,
                                     (tiles + kTilesPerSplit - 1) / kTilesPerSplit);
  splits = std::max<int64_t>(1, std::min<int64_t>(splits, tiles));
  const int tps = static_cast<int>((tiles + splits - 1) / splits);
  pl.cells_per_split = kTileN * tps;
  pl.splits = (tiles + tps - 1) / tps;
  pl.ws_bytes = static_cast<size_t>(n_seqs) * pl.splits * n_q * C.H * kGqa * 260 * sizeof(float);
  return pl;
}

int launch_verify_tc(const Launch& L, const CacheView& C, const AttendPlan& plan, const void* q,
                     const int32_t* pt, int64_t max_pages, const int32_t* steps, int n_seqs, int max_seq_len,
                     float sm_scale, float* out, void* ws) {
  if (n_seqs == 0) return K8V4_OK;
  PrefillParams p;
  p.C = C;
  p.q = static_cast<const uint16_t*>(q);
  p.pt = pt;
  p.max_pages = max_pages;
  p.steps = steps;
  p.seq_len = max_seq_len;
  p.n_q_tok = plan.n_q;
  p.splits = plan.splits;
  p.cells_per_split = plan.cells_per_split;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.out = nullptr;
  p.ws = static_cast<float*>(ws);
  p.status = L.status;
  p.wait_ns = wait_limit_ns() ? wait_limit_ns() : kWaitDefaultNs;
  if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return K8V4_ECUDA;
  const dim3 grid((plan.n_q + kTokens - 1) / kTokens, C.H, n_seqs * plan.splits);
  prefill_kernel<<<grid, kThreads, kSmemBytes, L.stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return K8V4_ECUDA;
  return launch_combine(L, p.ws, plan.splits, n_seqs, plan.n_q, C.H, out);
}

}  // namespace k8v4
