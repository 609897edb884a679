// attn_k8v4_decode_noalloc: decode attention for callers that cannot allocate
// device memory.  Some hosts own no device allocator of their own (a plain C
// program embedding the library with a fixed device budget handed out up
// front, or a framework whose pool already holds all device memory), and some
// loops must not call cudaMalloc/cudaFree at all because cudaFree synchronises
// the whole device.  Such callers still pass their inputs and outputs; the
// split-K partials go to a fixed array that lives in this library's own device
// memory instead of a caller-provided workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kNoallocScratchBytes for it until the process exits.  Host code
// cannot use the variable's name as a device address (it is a host-side
// stand-in), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current and caches it.
#include <mutex>

#include "k8v4_common.cuh"

namespace k8v4 {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(4) << 20;   // 4 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDev] = {};

// Device address of the scratch array on the current device (looked up once).
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return K8V4_EDEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return K8V4_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return K8V4_OK;
}

}  // namespace
}  // namespace k8v4

extern "C" int attn_k8v4_decode_noalloc(const k8v4_cache* cache, const void* q, int32_t q_dtype,
                                        const int32_t* page_table, int64_t max_pages, const int32_t* seq_lens,
                                        int32_t n_seqs, int32_t max_seq_len, float sm_scale, float* out,
                                        void* stream) {
  if (n_seqs < 0 || max_seq_len < 0) return K8V4_EINVAL;
  const size_t need = attn_k8v4_workspace_bytes(cache, n_seqs, 1, max_seq_len);
  if (n_seqs > 0 && need == 0) return K8V4_EINVAL;          // bad descriptor or sizes
  if (need > k8v4::kNoallocScratchBytes) return K8V4_ENOSPACE;
  void* scratch = nullptr;
  const int rc = k8v4::noalloc_scratch(&scratch);
  if (rc != K8V4_OK) return rc;
  // Every partial the combine reads is written earlier in the same call, so the
  // array needs no clearing between calls.
  return attn_k8v4_decode(cache, q, q_dtype, page_table, max_pages, seq_lens, n_seqs, max_seq_len, sm_scale, out,
                          scratch, k8v4::kNoallocScratchBytes, stream);
}
