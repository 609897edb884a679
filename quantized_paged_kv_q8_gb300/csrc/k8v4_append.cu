// Append (quantise + paged write) and dequantise kernels of the k8v4 cache.
//
// Follows the hybrid-KV pull request "--kv k8v4: hybrid KV cache -- INT8 K +
// Hadamard-rotated Q4_0 V (816 B/cell)", sections "What" and "How": K stays
// unrotated INT8 (ties to even), V is rotated by the 256-point Walsh-Hadamard
// transform and quantised to Q4_0, and each token is written through the page
// table (in the all-q4_0 comparison format K is rotated and quantised like V).
// Unlike the pages' engine (separate q8 and q4 append launches with
// the unused half folded onto one pool) this is one fused kernel: one warp per
// (token, KV head) loads K and V once, quantises K, rotates V exactly, quantises
// it, and stores all four runs with vector stores (for short appends a warp pair
// per (token, head) does the K and the V halves concurrently).  For a streamed
// cache the same warp stores each row twice, to the host mirror page and to the
// page's resident device slot (the streaming pull request's writers write both
// copies, "How"), so the two copies cannot drift apart.
//
// The rotation is defined as the correctly rounded fp32 value of the exact
// (H x) / 16.  The warp computes it with an int64 fixed-point fast Walsh-Hadamard
// transform whenever the vector's values span at most 2^54 (the common case);
// otherwise it falls back to an exact multi-limb sum per output element.
#include <algorithm>

#include "k8v4_quant.cuh"

namespace k8v4 {
namespace {

constexpr int kWarps = 8;

// ------------------------------------------------------------------ append
// MIRROR: a streamed cache -- the page table holds host-mirror page ids; every
// row goes to the mirror page M and, when slot_of_page says the page is
// resident, to its device slot in C as well (one quantisation, two stores)
template <bool BF16, int FMT, bool MIRROR>
__global__ void __launch_bounds__(kWarps * 32) append_kernel(CacheView C, CacheView M, const int32_t* __restrict__ slot_of_page,
                                                             const int32_t* __restrict__ pt, int64_t max_pages,
                                                             const int64_t* __restrict__ pos, int n_seqs, int n_tok,
                                                             const void* __restrict__ k, const void* __restrict__ v,
                                                             int split_kv, FastDiv div_h, FastDiv div_tok, FastDiv div_p,
                                                             int* status) {
  __shared__ long long stage[kWarps][kRotScratch];
  // a kernel launched after this one as a programmatic dependent (the decode
  // attention) may start its launch now; it waits for this grid's completion
  // (griddepcontrol.wait) before it reads the cache
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  // (seq, token, head) per warp, or, for short appends (a decode step's token),
  // (seq, token, head, half): warp pairs split a (token, head) into its K half
  // (int8 quantisation; rotation + q4_0 in the Q4 format) and its V half
  // (rotation + q4_0, or int8), which run concurrently.  The host keeps every
  // warp index below 2^31, and a cell that passes the range check is below
  // max_pages * P <= 2^31, so the index arithmetic runs in 32 bits.
  const int64_t wi = static_cast<int64_t>(blockIdx.x) * kWarps + w;
  const int64_t total = static_cast<int64_t>(n_seqs) * n_tok * C.H;
  if (wi >= (split_kv ? 2 * total : total)) return;
  const int role = split_kv ? static_cast<int>(wi & 1) : 2;             // 0: K only, 1: V only, 2: both
  const uint32_t item = static_cast<uint32_t>(split_kv ? wi >> 1 : wi);  // (seq, token, head)
  const uint32_t it = div_h.div(item);
  const int g = static_cast<int>(item - it * static_cast<uint32_t>(C.H));
  const uint32_t b = div_tok.div(it);
  const int t = static_cast<int>(it - b * static_cast<uint32_t>(n_tok));
  const int64_t cell = pos[b] + t;
  if (cell < 0 || cell >= max_pages * C.P) { if (lane == 0) record_status(status, K8V4_ERANGE); return; }
  const uint32_t pidx = div_p.div(static_cast<uint32_t>(cell));
  const int cslot = static_cast<int>(static_cast<uint32_t>(cell) - pidx * static_cast<uint32_t>(C.P));
  const int64_t page = pt[static_cast<int64_t>(b) * max_pages + pidx];
  const int64_t r = static_cast<int64_t>(cslot) * C.H + g;
  const int64_t elem = static_cast<int64_t>(item) * kD + 8 * lane;
  uint8_t* base;
  uint8_t* base2 = nullptr;
  if (MIRROR) {
    if (page < 0 || page >= M.n_pages) { if (lane == 0) record_status(status, K8V4_ERANGE); return; }
    base = M.pages + page * M.page_bytes;
    const int dslot = slot_of_page[page];
    if (dslot >= 0 && dslot < C.n_pages) base2 = C.pages + static_cast<int64_t>(dslot) * C.page_bytes;
    else if (dslot != -1 && lane == 0) record_status(status, K8V4_ERANGE);   // mirror written, slot skipped
  } else {
    if (page < 0 || page >= C.n_pages) { if (lane == 0) record_status(status, K8V4_ERANGE); return; }
    base = C.pages + page * C.page_bytes;
  }
  if (role != 1) append_k_row<BF16, FMT>(C, base, r, k, elem, lane, stage[w], base2);
  if (role != 0) append_v_row<BF16, FMT>(C, base, r, v, elem, lane, stage[w], base2);
}

// ------------------------------------------------------------------ bulk bf16 append
// The long appends of bf16 rows (a prompt chunk, a cache build): a persistent
// grid of 8-warp CTAs, each warp stepping through a contiguous run of (seq,
// token, head) items; the warp loads the next item's K and V rows (16 B per
// lane each) before it quantises the current one, so every warp keeps 1 KB of
// loads in flight while it computes.  The rows are quantised by the bf16 fast paths (int8 K, exact
// rotation + q4_0 V, same bytes as append_kernel).
template <int FMT, bool MIRROR>
__global__ void __launch_bounds__(kWarps * 32, 3) append_bf16_kernel(
    CacheView C, CacheView M, const int32_t* __restrict__ slot_of_page, const int32_t* __restrict__ pt,
    int64_t max_pages, const int64_t* __restrict__ pos, int n_seqs, int n_tok, const uint16_t* __restrict__ k,
    const uint16_t* __restrict__ v, FastDiv div_h, FastDiv div_tok, FastDiv div_p, int* status) {
  __shared__ __align__(16) long long stage[kWarps][kRotScratch];
  __shared__ float scale_tab[128];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  long long* ts = stage[w];
  fill_int8_scale_table(scale_tab);
  __syncthreads();
  // Each warp takes a contiguous run of (seq, token, head) items and steps
  // through it: the head, token and sequence indices advance by increments, and
  // the page lookup is redone only when a token crosses into another page or
  // sequence.  The host keeps total below 2^31, and a cell that passes the range
  // check is below max_pages * P <= 2^31, so the index arithmetic runs in 32 bits.
  const uint32_t total = static_cast<uint32_t>(n_seqs) * static_cast<uint32_t>(n_tok) * static_cast<uint32_t>(C.H);
  const uint32_t n_warps = gridDim.x * kWarps;
  const uint32_t per = (total + n_warps - 1) / n_warps;
  uint32_t item = (blockIdx.x * kWarps + w) * per;
  const uint32_t item_end = min(item + per, total);
  if (item >= item_end) return;
  const uint4* kp = reinterpret_cast<const uint4*>(k + static_cast<int64_t>(item) * kD) + lane;
  const uint4* vp = reinterpret_cast<const uint4*>(v + static_cast<int64_t>(item) * kD) + lane;
  uint4 kr = __ldcs(kp), vr = __ldcs(vp);
  const uint32_t it0 = div_h.div(item);
  int g = static_cast<int>(item - it0 * static_cast<uint32_t>(C.H));
  uint32_t b = div_tok.div(it0);
  int t = static_cast<int>(it0 - b * static_cast<uint32_t>(n_tok));
  const int64_t cell_limit = max_pages * C.P;
  int64_t cell = pos[b] + t;
  bool lookup = true;                   // the page of `cell` must be looked up
  int cslot = 0;
  uint8_t* base = nullptr;
  uint8_t* base2 = nullptr;
  for (; item < item_end; ++item) {
    const uint4 kc = kr, vc = vr;
    if (item + 1 < item_end) {
      kp += kD / 8;
      vp += kD / 8;
      kr = __ldcs(kp);
      vr = __ldcs(vp);
    }
    const bool in_range = cell >= 0 && cell < cell_limit;
    if (in_range && lookup) {
      const uint32_t pidx = div_p.div(static_cast<uint32_t>(cell));
      cslot = static_cast<int>(static_cast<uint32_t>(cell) - pidx * static_cast<uint32_t>(C.P));
      const int64_t page = pt[static_cast<int64_t>(b) * max_pages + pidx];
      base = nullptr;
      base2 = nullptr;
      if (MIRROR) {
        if (page >= 0 && page < M.n_pages) {
          base = M.pages + page * M.page_bytes;
          const int dslot = slot_of_page[page];
          if (dslot >= 0 && dslot < C.n_pages) base2 = C.pages + static_cast<int64_t>(dslot) * C.page_bytes;
          else if (dslot != -1 && lane == 0) record_status(status, K8V4_ERANGE);
        }
      } else if (page >= 0 && page < C.n_pages) {
        base = C.pages + page * C.page_bytes;
      }
      lookup = false;
    }
    if (!in_range || base == nullptr) {
      if (lane == 0) record_status(status, K8V4_ERANGE);
    } else {
      const int r = cslot * C.H + g;
      if (FMT == K8V4_FORMAT_Q4) rot_q4_row_bf16(kc, lane, ts, base, base2, r * 128, C.ks_off() + r * 16);
      else int8_row_bf16(kc, lane, scale_tab, base, base2, r * 256, C.ks_off() + r * 8);
      if (FMT == K8V4_FORMAT_INT8) int8_row_bf16(vc, lane, scale_tab, base, base2, C.v_off() + r * 256, C.vs_off() + r * 8);
      else rot_q4_row_bf16(vc, lane, ts, base, base2, C.v_off() + r * 128, C.vs_off() + r * 16);
    }
    // the next item: head, then token (its cell), then sequence
    if (++g == C.H) {
      g = 0;
      if (++t == n_tok) {
        t = 0;
        if (++b < static_cast<uint32_t>(n_seqs)) cell = pos[b];
        lookup = true;
      } else {
        ++cell;
        if (++cslot == C.P) lookup = true;
      }
    }
  }
}

// ------------------------------------------------------------------ dequant
// Rotated-space values (code - 8) * d of one q4_0 row, elements 8 * lane + r:
// block lane / 4; element e of a block is the low nibble of byte e (e < 16) or
// the high nibble of byte e - 16
__device__ __forceinline__ void read_q4_row(const uint8_t* nib, const uint8_t* scales, int lane, float x[8]) {
  const int blk = lane >> 2, e0 = 8 * (lane & 3);
  const float d = __half2float(*reinterpret_cast<const __half*>(scales + 2 * blk));
  const uint2 raw = *reinterpret_cast<const uint2*>(nib + 16 * blk + (e0 & 15));
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t word = q < 4 ? raw.x : raw.y;
    const uint32_t byte = (word >> (8 * (q & 3))) & 0xffu;
    const int code = e0 < 16 ? static_cast<int>(byte & 0xfu) : static_cast<int>(byte >> 4);
    x[q] = __fmul_rn(static_cast<float>(code - 8), d);
  }
}

template <int FMT>
__global__ void __launch_bounds__(kWarps * 32) dequant_kernel(CacheView C, const int32_t* __restrict__ pt,
                                                              int64_t max_pages, int64_t start, int64_t n_cells,
                                                              float* __restrict__ k_out, float* __restrict__ v_rot_out,
                                                              float* __restrict__ v_out, int* status) {
  __shared__ long long stage[kWarps][kRotScratch];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kWarps + w;   // (cell, head)
  if (item >= n_cells * C.H) return;
  const int g = static_cast<int>(item % C.H);
  const int64_t cell = start + item / C.H;
  const int64_t pidx = cell / C.P;
  const int64_t page = (cell >= 0 && pidx < max_pages) ? pt[pidx] : -1;
  float* ko = k_out + item * kD + 8 * lane;
  float* vr = v_rot_out + item * kD + 8 * lane;
  float* vo = v_out ? v_out + item * kD + 8 * lane : nullptr;
  if (page < 0 || page >= C.n_pages) {
    if (lane == 0) record_status(status, K8V4_ERANGE);
    return;
  }
  const int64_t r = (cell % C.P) * C.H + g;
  const uint8_t* base = C.pages + page * C.page_bytes;
  float x[8];
  if (FMT == K8V4_FORMAT_Q4) {
    // rotated-space K, then the exact inverse rotation (H/16 is its own inverse)
    read_q4_row(base + r * 128, base + C.ks_off() + r * 16, lane, x);
    rotate_exact(x, lane, stage[w]);
  } else {
    const float2 ks = *reinterpret_cast<const float2*>(base + C.ks_off() + r * 8);
    const float s = lane < 16 ? ks.x : ks.y;
    const uint2 kc = *reinterpret_cast<const uint2*>(base + r * 256 + 8 * lane);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t word = q < 4 ? kc.x : kc.y;
      const int c = static_cast<int8_t>((word >> (8 * (q & 3))) & 0xffu);
      x[q] = __fmul_rn(static_cast<float>(c), s);
    }
  }
  reinterpret_cast<float4*>(ko)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(ko)[1] = make_float4(x[4], x[5], x[6], x[7]);
  if (FMT != K8V4_FORMAT_INT8) {
    read_q4_row(base + C.v_off() + r * 128, base + C.vs_off() + r * 16, lane, x);
  } else {
    const float2 vsc = *reinterpret_cast<const float2*>(base + C.vs_off() + r * 8);
    const float sv = lane < 16 ? vsc.x : vsc.y;
    const uint2 vc = *reinterpret_cast<const uint2*>(base + C.v_off() + r * 256 + 8 * lane);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t word = q < 4 ? vc.x : vc.y;
      const int c = static_cast<int8_t>((word >> (8 * (q & 3))) & 0xffu);
      x[q] = __fmul_rn(static_cast<float>(c), sv);
    }
  }
  reinterpret_cast<float4*>(vr)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(vr)[1] = make_float4(x[4], x[5], x[6], x[7]);
  if (vo) {
    if (FMT != K8V4_FORMAT_INT8) rotate_exact(x, lane, stage[w]);
    reinterpret_cast<float4*>(vo)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4*>(vo)[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
}

}  // namespace

template <bool BF16, int FMT>
void append_launch(const Launch& L, dim3 grid, dim3 block, const CacheView& C, const CacheView* M, const int32_t* slot,
                   const int32_t* pt, int64_t max_pages, const int64_t* pos, int n_seqs, int n_tok, const void* k,
                   const void* v, int split) {
  const FastDiv dh(static_cast<uint32_t>(C.H)), dt(static_cast<uint32_t>(n_tok)), dp(static_cast<uint32_t>(C.P));
  if (BF16 && !split) {
    // persistent: three 8-warp CTAs per SM (85 registers a thread), or fewer when the items run out
    const int64_t items = static_cast<int64_t>(n_seqs) * n_tok * C.H;
    const int64_t want = (items + kWarps - 1) / kWarps;
    const dim3 pgrid(static_cast<unsigned>(std::min<int64_t>(want, static_cast<int64_t>(L.num_sms) * 3)));
    const auto* kb = static_cast<const uint16_t*>(k);
    const auto* vb = static_cast<const uint16_t*>(v);
    if (M) append_bf16_kernel<FMT, true><<<pgrid, block, 0, L.stream>>>(C, *M, slot, pt, max_pages, pos, n_seqs, n_tok, kb, vb, dh, dt, dp, L.status);
    else append_bf16_kernel<FMT, false><<<pgrid, block, 0, L.stream>>>(C, C, nullptr, pt, max_pages, pos, n_seqs, n_tok, kb, vb, dh, dt, dp, L.status);
    return;
  }
  if (M) append_kernel<BF16, FMT, true><<<grid, block, 0, L.stream>>>(C, *M, slot, pt, max_pages, pos, n_seqs, n_tok, k, v, split, dh, dt, dp, L.status);
  else append_kernel<BF16, FMT, false><<<grid, block, 0, L.stream>>>(C, C, nullptr, pt, max_pages, pos, n_seqs, n_tok, k, v, split, dh, dt, dp, L.status);
}

int launch_append(const Launch& L, const CacheView& C, const int32_t* pt, int64_t max_pages, int n_seqs,
                  const int64_t* pos, int n_tok, const void* k, const void* v, int dtype, const CacheView* mirror,
                  const int32_t* slot_of_page) {
  const int64_t items = static_cast<int64_t>(n_seqs) * n_tok * C.H;
  if (items == 0) return K8V4_OK;
  // short appends (up to a few thousand (token, head) items, e.g. a decode
  // step) take a warp pair per item for latency; long ones a warp per item
  const int split = items * 2 <= static_cast<int64_t>(L.num_sms) * 16 ? 1 : 0;
  if ((split ? 2 : 1) * items >= (int64_t(1) << 31)) return K8V4_EINVAL;   // warp indices stay below 2^31
  const int64_t blocks = ((split ? 2 : 1) * items + kWarps - 1) / kWarps;
  const dim3 grid(static_cast<unsigned>(blocks)), block(kWarps * 32);
  const bool bf = dtype == K8V4_BF16;
  const CacheView* M = mirror;
  const int32_t* so = slot_of_page;
  if (C.fmt == K8V4_FORMAT_K8V4) {
    if (bf) append_launch<true, K8V4_FORMAT_K8V4>(L, grid, block, C, M, so, pt, max_pages, pos, n_seqs, n_tok, k, v, split);
    else append_launch<false, K8V4_FORMAT_K8V4>(L, grid, block, C, M, so, pt, max_pages, pos, n_seqs, n_tok, k, v, split);
  } else if (C.fmt == K8V4_FORMAT_Q4) {
    if (bf) append_launch<true, K8V4_FORMAT_Q4>(L, grid, block, C, M, so, pt, max_pages, pos, n_seqs, n_tok, k, v, split);
    else append_launch<false, K8V4_FORMAT_Q4>(L, grid, block, C, M, so, pt, max_pages, pos, n_seqs, n_tok, k, v, split);
  } else {
    if (bf) append_launch<true, K8V4_FORMAT_INT8>(L, grid, block, C, M, so, pt, max_pages, pos, n_seqs, n_tok, k, v, split);
    else append_launch<false, K8V4_FORMAT_INT8>(L, grid, block, C, M, so, pt, max_pages, pos, n_seqs, n_tok, k, v, split);
  }
  return cudaGetLastError() == cudaSuccess ? K8V4_OK : K8V4_ECUDA;
}

int launch_dequant(const Launch& L, const CacheView& C, const int32_t* pt, int64_t max_pages, int64_t start,
                   int64_t n_cells, float* k_out, float* v_rot_out, float* v_out) {
  const int64_t items = n_cells * C.H;
  if (items == 0) return K8V4_OK;
  const int64_t blocks = (items + kWarps - 1) / kWarps;
  if (blocks > 0x7fffffffll) return K8V4_EINVAL;
  const dim3 grid(static_cast<unsigned>(blocks)), block(kWarps * 32);
  if (C.fmt == K8V4_FORMAT_K8V4)
    dequant_kernel<K8V4_FORMAT_K8V4><<<grid, block, 0, L.stream>>>(C, pt, max_pages, start, n_cells, k_out, v_rot_out, v_out, L.status);
  else if (C.fmt == K8V4_FORMAT_Q4)
    dequant_kernel<K8V4_FORMAT_Q4><<<grid, block, 0, L.stream>>>(C, pt, max_pages, start, n_cells, k_out, v_rot_out, v_out, L.status);
  else
    dequant_kernel<K8V4_FORMAT_INT8><<<grid, block, 0, L.stream>>>(C, pt, max_pages, start, n_cells, k_out, v_rot_out, v_out, L.status);
  return cudaGetLastError() == cudaSuccess ? K8V4_OK : K8V4_ECUDA;
}

}  // namespace k8v4
