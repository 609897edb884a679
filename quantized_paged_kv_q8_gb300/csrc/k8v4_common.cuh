// Internal definitions shared by the k8v4 CUDA translation units: the device
// view of a cache, the page-layout offsets, the device status word, small PTX
// wrappers, and the host-side launch functions the C ABI calls.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/k8v4.h"

namespace k8v4 {

constexpr int kD = 256;   // head_dim
constexpr int kGqa = 8;   // query heads per KV head

// Bytes per (cell, head) of each format.  K8V4: 256 K codes + 8 (two fp32
// scales) + 128 V nibbles + 16 (eight fp16 scales) = 408; INT8: 256 + 8 + 256 +
// 8 = 528; Q4: 128 + 16 + 128 + 16 = 288.
__host__ __device__ constexpr int cell_head_bytes(int fmt) {
  return fmt == K8V4_FORMAT_K8V4 ? 408 : fmt == K8V4_FORMAT_Q4 ? 288 : 528;
}

// Device view of a cache.  Page p starts at pages + p * page_bytes; inside it
// the runs are K ([P][H][256] int8 codes, or [P][H][8][16] nibbles for Q4),
// K scales ([P][H][2] f32, or [P][H][8] f16 for Q4), V ([P][H][8][16] nibbles,
// or [P][H][256] int8 codes for INT8) and V scales ([P][H][8] f16, or [P][H][2]
// f32 for INT8).  r = slot * H + head indexes a (cell, head) inside a run.
struct CacheView {
  uint8_t* pages;
  int64_t n_pages;
  int64_t page_bytes;
  int P;
  int H;
  int fmt;

  __host__ __device__ int k_row_bytes() const { return fmt == K8V4_FORMAT_Q4 ? 128 : 256; }
  __host__ __device__ int ks_row_bytes() const { return fmt == K8V4_FORMAT_Q4 ? 16 : 8; }
  __host__ __device__ int v_row_bytes() const { return fmt == K8V4_FORMAT_INT8 ? 256 : 128; }
  __host__ __device__ int vs_row_bytes() const { return fmt == K8V4_FORMAT_INT8 ? 8 : 16; }
  __host__ __device__ int64_t ks_off() const { return static_cast<int64_t>(k_row_bytes()) * H * P; }
  __host__ __device__ int64_t v_off() const { return static_cast<int64_t>(k_row_bytes() + ks_row_bytes()) * H * P; }
  __host__ __device__ int64_t vs_off() const {
    return static_cast<int64_t>(k_row_bytes() + ks_row_bytes() + v_row_bytes()) * H * P;
  }
};

// ---------------------------------------------------------------- division
// Division by a kernel-invariant divisor d >= 1 for dividends below 2^31, by the
// round-up multiply-high method: s = ceil(log2 d), m = floor(2^32 (2^s - d) / d)
// + 1, q = (umulhi(n, m) + n) >> s (exact for every n < 2^31; the sum stays
// below 2^32).  Three instructions instead of a 64-bit division routine.
struct FastDiv {
  uint32_t d = 1, m = 1;
  int s = 0;
  FastDiv() = default;
  __host__ explicit FastDiv(uint32_t div) : d(div) {
    while ((1ull << s) < d) ++s;
    m = static_cast<uint32_t>(((1ull << 32) * ((1ull << s) - d)) / d + 1);
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const { return (__umulhi(n, m) + n) >> s; }
};

// ---------------------------------------------------------------- status word
// Kernels record the first device-side error here (compare-and-swap from 0) and
// skip the offending access; the host reads and clears it.
__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- host side
struct Launch {
  cudaStream_t stream;
  int* status;      // device status word of the current device
  int num_sms;
};

// mirror != null: a streamed cache -- pt holds host-mirror page ids, every row is
// written to the mirror and, where slot_of_page[page] >= 0, to that slot of C
int launch_append(const Launch& L, const CacheView& C, const int32_t* pt, int64_t max_pages, int n_seqs,
                  const int64_t* pos, int n_tok, const void* k, const void* v, int dtype,
                  const CacheView* mirror = nullptr, const int32_t* slot_of_page = nullptr);
// streamed caches: look up the pages the sequences read (resident slot, or a copy
// from the host mirror M into a staging slot of C) and copy the misses
int launch_stream_resolve(const Launch& L, const CacheView& M, const CacheView& C, const int32_t* slot_of_page,
                          int n_resident, const int32_t* pt, int64_t max_pages, const int32_t* lens, int n_seqs,
                          int max_seq_len, int32_t* dev_pt, void* ws);
int launch_stream_copy(const Launch& L, const CacheView& M, const CacheView& C, const int32_t* pages, int n);
size_t stream_ws_bytes(int n_seqs, int64_t max_pages);
int launch_dequant(const Launch& L, const CacheView& C, const int32_t* pt, int64_t max_pages, int64_t start,
                   int64_t n_cells, float* k_out, float* v_rot_out, float* v_out);

struct AttendPlan {
  int n_q, n_groups, warps, splits, cells_per_split;
  size_t ws_bytes;
};
AttendPlan plan_attend(const CacheView& C, int n_seqs, int n_q, int max_seq_len, int num_sms);
// k_new / v_new (n_q = 1 only): append each sequence's newest token (cell
// steps[b] - 1) from them before attending -- the fused decode step
int launch_attend(const Launch& L, const CacheView& C, const AttendPlan& plan, const void* q, int q_dtype,
                  const int32_t* pt, int64_t max_pages, const int32_t* steps, int n_seqs, int max_seq_len,
                  float sm_scale, float* out, void* ws, const void* k_new = nullptr, const void* v_new = nullptr,
                  int kv_dtype = K8V4_BF16);
AttendPlan plan_verify(const CacheView& C, int n_seqs, int n_q, int max_seq_len, int num_sms);
int launch_verify(const Launch& L, const CacheView& C, const AttendPlan& plan, const void* q, int q_dtype,
                  const int32_t* pt, int64_t max_pages, const int32_t* steps, int n_seqs, int max_seq_len,
                  float sm_scale, float* out, void* ws);
AttendPlan plan_verify_tc(const CacheView& C, int n_seqs, int n_q, int max_seq_len, int num_sms);
int launch_verify_tc(const Launch& L, const CacheView& C, const AttendPlan& plan, const void* q,
                     const int32_t* pt, int64_t max_pages, const int32_t* steps, int n_seqs, int max_seq_len,
                     float sm_scale, float* out, void* ws);
// the warp-specialised TMA decode kernel (k8v4_decode.cu): one query per
// sequence over the K8V4 or INT8 format; spin = mbarrier poll limit (0: default)
bool decode_ws_supported(const CacheView& C);
AttendPlan plan_decode(const CacheView& C, int n_seqs, int max_seq_len, int num_sms);
int launch_decode(const Launch& L, const CacheView& C, const AttendPlan& plan, const void* q, int q_dtype,
                  const int32_t* pt, int64_t max_pages, const int32_t* steps, int n_seqs, int max_seq_len,
                  float sm_scale, float* out, void* ws, const void* k_new, const void* v_new, int kv_dtype,
                  uint32_t spin);
// cells [cell_begin, cell_end) of every sequence only, merged into unnormalised
// partial rows [n_seqs][8 H][260] (o[256], m as a base-2 exponent, l); the plan
// is plan_decode over cell_end - cell_begin cells
int launch_decode_partial(const Launch& L, const CacheView& C, const AttendPlan& plan, const void* q, int q_dtype,
                          const int32_t* pt, int64_t max_pages, const int32_t* steps, int n_seqs,
                          int max_seq_len, int cell_begin, int cell_end, float sm_scale, float* partial, void* ws,
                          uint32_t wait_ns);
// the team-of-warps TMA verify kernel (k8v4_decode.cu): 2..8 queries per
// sequence over the K8V4 format with bf16 queries
bool verify_ws_supported(const CacheView& C, int n_q, int q_dtype);
AttendPlan plan_verify_ws(const CacheView& C, int n_seqs, int n_q, int max_seq_len, int num_sms);
int launch_verify_ws(const Launch& L, const CacheView& C, const void* q, const int32_t* pt, int64_t max_pages,
                     const int32_t* steps, int n_seqs, int n_q, int max_seq_len, float sm_scale, float* out, void* ws);
// the bound of the mbarrier waits in the tensor-memory and TMA kernels (ns; 0: default)
uint32_t wait_limit_ns();
// diagnostics: nonzero makes the TMA decode kernel withhold its first CTA's first copy
int withheld_copy();
// weighted sum of split partials (o[256], m, l rows of 260 floats) -> out, launched programmatically dependent
int launch_combine(const Launch& L, const float* ws, int splits, int n_seqs, int n_q, int H, float* out);
// the splits of a one-query decode merged into one unnormalised partial row per (sequence, query head)
int launch_combine_partial(const Launch& L, const float* ws, int splits, int n_seqs, int H, float* partial);
// gathered partials [n_parts][n_seqs][rows][260] -> out [n_seqs][rows][256]
int launch_combine_parts(const Launch& L, const float* parts, int n_parts, int n_seqs, int n_rows_per_seq,
                         float* out);
int launch_prefill(const Launch& L, const CacheView& C, const void* q, const int32_t* pt, int64_t max_pages,
                   int seq_len, int n_q_tok, const int32_t* steps, float sm_scale, float* out);

}  // namespace k8v4
