// Streamed caches: the page lookups of one attention call and the page mover.
//
// Follows "kv: --kv k8v4 streams with --kv-resident" ("How": a block moves
// between pinned host RAM and VRAM as its byte runs -- for k8v4 the K codes,
// the K scales and the V q4_0 -- and every writer writes both copies; "Tests":
// streamed and resident attention are bitwise equal).
//
// GB300 design.  The host mirror is page-locked memory that the GPU reads
// directly over NVLink-C2C, so moving a page is a kernel, not a copy call per
// page or per run: one CTA per page in flight, 16-byte loads from the mirror
// (four in flight per thread), stores into the page's staging slot.  A page of
// this cache is one contiguous region holding all of its runs, so a whole-page
// copy moves every run at once.  The lookup is a single CTA: a block-wide scan
// over the (sequence, page index) entries gives each miss its rank, hence its
// staging slot, in lookup order -- the same slots on every run, so a streamed
// call is reproducible bit for bit.
#include <algorithm>

#include "k8v4_common.cuh"

namespace k8v4 {
namespace {

constexpr int kResolveThreads = 1024;   // 32 warps: one warp-sum slot per lane of warp 0
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

// dev_pt[e] for every entry e = (b, i) of the page table: the resident slot of
// the page, the staging slot its copy goes to, or -1 (not read, or an error);
// moves[r] = (host page, slot) of the r-th miss; *count = copies to make
__global__ void __launch_bounds__(kResolveThreads) resolve_kernel(CacheView M, CacheView C,
                                                                  const int32_t* __restrict__ slot_of_page,
                                                                  int n_resident, const int32_t* __restrict__ pt,
                                                                  int64_t max_pages, const int32_t* __restrict__ lens,
                                                                  int n_seqs, int max_seq_len,
                                                                  int32_t* __restrict__ dev_pt, int* __restrict__ count,
                                                                  int2* __restrict__ moves, int* status) {
  __shared__ int warp_incl[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  const int64_t total = static_cast<int64_t>(n_seqs) * max_pages;
  const int64_t cap = C.n_pages - n_resident;                 // staging slots
#pragma unroll 1
  for (int64_t e0 = 0; e0 < total; e0 += kResolveThreads) {
    const int64_t e = e0 + tid;
    int out = -1, hp = -1;
    bool miss = false;
    if (e < total) {
      const int b = static_cast<int>(e / max_pages);
      const int64_t i = e - static_cast<int64_t>(b) * max_pages;
      int n = lens[b];
      if (n < 0 || n > max_seq_len) {
        if (i == 0) record_status(status, K8V4_ERANGE);
        n = n < 0 ? 0 : max_seq_len;
      }
      if (i * C.P < n) {
        hp = pt[e];
        if (hp < 0 || hp >= M.n_pages) {
          record_status(status, K8V4_ERANGE);
        } else {
          const int s = slot_of_page[hp];
          if (s >= 0 && s < n_resident) out = s;
          else if (s == -1) miss = true;
          else record_status(status, K8V4_ERANGE);
        }
      }
    }
    // exclusive rank of this entry's miss among the block's, plus the carry
    const unsigned ballot = __ballot_sync(0xffffffffu, miss);
    const int in_warp = __popc(ballot & ((1u << lane) - 1u));
    if (lane == 0) warp_incl[warp] = __popc(ballot);
    __syncthreads();
    if (warp == 0) {
      int x = warp_incl[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      warp_incl[lane] = x;
    }
    __syncthreads();
    const int rank = carry + (warp ? warp_incl[warp - 1] : 0) + in_warp;
    if (miss) {
      if (rank < cap) {
        out = n_resident + rank;
        moves[rank] = make_int2(hp, out);
      } else {
        record_status(status, K8V4_ENOSPACE);
      }
    }
    if (e < total) dev_pt[e] = out;
    __syncthreads();
    if (tid == 0) carry += warp_incl[31];
    __syncthreads();
  }
  if (tid == 0) *count = static_cast<int>(min(static_cast<int64_t>(carry), cap));
}

// Copy whole pages: moves[m] = (host page, device slot), m < *count (or n)
__global__ void __launch_bounds__(kCopyThreads) copy_kernel(CacheView M, CacheView C, const int* __restrict__ count,
                                                            int n, const int2* __restrict__ moves, int* status) {
  const int cnt = count ? *count : n;
  const int64_t nvec = C.page_bytes / 16;
#pragma unroll 1
  for (int m = blockIdx.x; m < cnt; m += gridDim.x) {
    const int2 mv = moves[m];
    if (mv.x < 0 || mv.x >= M.n_pages || mv.y < 0 || mv.y >= C.n_pages) {
      if (threadIdx.x == 0) record_status(status, K8V4_ERANGE);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(M.pages + static_cast<int64_t>(mv.x) * M.page_bytes);
    uint4* dst = reinterpret_cast<uint4*>(C.pages + static_cast<int64_t>(mv.y) * C.page_bytes);
    int64_t i = threadIdx.x;
#pragma unroll 1
    for (; i + (kCopyUnroll - 1) * kCopyThreads < nvec; i += kCopyUnroll * kCopyThreads) {
      uint4 t[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) t[u] = src[i + u * kCopyThreads];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) dst[i + u * kCopyThreads] = t[u];
    }
#pragma unroll 1
    for (; i < nvec; i += kCopyThreads) dst[i] = src[i];
  }
}

int copy_grid(const Launch& L, int64_t max_moves) {
  const int64_t g = std::min<int64_t>(max_moves, static_cast<int64_t>(L.num_sms) * 8);
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

size_t stream_ws_bytes(int n_seqs, int64_t max_pages) {
  return 16 + 8 * static_cast<size_t>(n_seqs) * static_cast<size_t>(max_pages);
}

int launch_stream_resolve(const Launch& L, const CacheView& M, const CacheView& C, const int32_t* slot_of_page,
                          int n_resident, const int32_t* pt, int64_t max_pages, const int32_t* lens, int n_seqs,
                          int max_seq_len, int32_t* dev_pt, void* ws) {
  if (n_seqs == 0) return K8V4_OK;
  int* count = static_cast<int*>(ws);
  int2* moves = reinterpret_cast<int2*>(static_cast<uint8_t*>(ws) + 16);
  resolve_kernel<<<1, kResolveThreads, 0, L.stream>>>(M, C, slot_of_page, n_resident, pt, max_pages, lens, n_seqs,
                                                       max_seq_len, dev_pt, count, moves, L.status);
  if (cudaGetLastError() != cudaSuccess) return K8V4_ECUDA;
  // at most one copy per page a sequence can read, and no more than the staging slots
  const int64_t reach = std::min<int64_t>(max_pages, (static_cast<int64_t>(max_seq_len) + C.P - 1) / C.P);
  const int64_t max_moves = std::min<int64_t>(reach * n_seqs, C.n_pages - n_resident);
  if (max_moves <= 0) return K8V4_OK;
  copy_kernel<<<copy_grid(L, max_moves), kCopyThreads, 0, L.stream>>>(M, C, count, 0, moves, L.status);
  return cudaGetLastError() == cudaSuccess ? K8V4_OK : K8V4_ECUDA;
}

int launch_stream_copy(const Launch& L, const CacheView& M, const CacheView& C, const int32_t* pages, int n) {
  if (n == 0) return K8V4_OK;
  copy_kernel<<<copy_grid(L, n), kCopyThreads, 0, L.stream>>>(M, C, nullptr, n, reinterpret_cast<const int2*>(pages),
                                                              L.status);
  return cudaGetLastError() == cudaSuccess ? K8V4_OK : K8V4_ECUDA;
}

}  // namespace k8v4
