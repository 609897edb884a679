// The extern "C" entry points declared in include/k8v4.h: host-side argument
// validation, the per-device status word, and the launches.
#include <atomic>
#include <mutex>

#include "k8v4_common.cuh"

namespace k8v4 {
namespace {

// First device-side error since the last k8v4_last_device_status() (0 = none).
__device__ int g_status_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int code = K8V4_EDEVICE;
  int* status = nullptr;
  int num_sms = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<uint32_t> g_wait_ns{0};       // 0: each kernel's default bound
std::atomic<int> g_withhold{0};           // diagnostics: the TMA decode kernel withholds one copy

// Per-device set-up, done once with the device current: check that it is an
// sm_103 part and find the device address of the status word.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return K8V4_EDEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    s.ready = true;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      s.code = K8V4_ECUDA;
    } else if (major != 10 || minor != 3) {
      s.code = K8V4_EDEVICE;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
        s.code = K8V4_ECUDA;
      } else {
        s.status = static_cast<int*>(p);
        s.num_sms = sms;
        s.code = K8V4_OK;
      }
    }
  }
  *out = &s;
  return s.code;
}

int make_launch(void* stream, Launch* L) {
  DeviceState* s = nullptr;
  const int rc = device_state(&s);
  if (rc != K8V4_OK) return rc;
  L->stream = static_cast<cudaStream_t>(stream);
  L->status = s->status;
  L->num_sms = s->num_sms;
  return K8V4_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int view_of(const k8v4_cache* c, CacheView* v) {
  if (!c || !c->pages) return K8V4_EINVAL;
  if (c->format != K8V4_FORMAT_K8V4 && c->format != K8V4_FORMAT_INT8 && c->format != K8V4_FORMAT_Q4)
    return K8V4_EINVAL;
  if (c->head_dim != kD || c->n_kv_heads < 1 || c->n_kv_heads > 8) return K8V4_EINVAL;
  if (c->page_size < 16 || c->page_size > 4096 || c->page_size % 16) return K8V4_EINVAL;
  if (c->n_pages < 1 || c->n_pages > (int64_t(1) << 40)) return K8V4_EINVAL;
  if (!aligned(c->pages, 256)) return K8V4_EALIGN;
  v->pages = static_cast<uint8_t*>(c->pages);
  v->n_pages = c->n_pages;
  v->P = c->page_size;
  v->H = c->n_kv_heads;
  v->fmt = c->format;
  v->page_bytes = static_cast<int64_t>(c->page_size) * c->n_kv_heads * cell_head_bytes(c->format);
  return K8V4_OK;
}

int check_table(const CacheView& v, const int32_t* pt, int64_t max_pages) {
  if (!pt) return K8V4_EINVAL;
  if (max_pages < 1 || max_pages > (int64_t(1) << 31) / v.P) return K8V4_EINVAL;
  if (!aligned(pt, 4)) return K8V4_EALIGN;
  return K8V4_OK;
}

// The host mirror of a streamed cache: the same format, P and H as the device
// cache, pages in page-locked host memory that the device can address.  Called
// after make_launch (needs the device context); `M` gets the device-side address.
int mirror_of(const k8v4_cache* host, const CacheView& C, CacheView* M) {
  int rc = view_of(host, M);
  if (rc) return rc;
  if (M->fmt != C.fmt || M->P != C.P || M->H != C.H) return K8V4_EINVAL;
  return K8V4_OK;
}
int mirror_address(const k8v4_cache* host, CacheView* M) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host->pages) != cudaSuccess) {
    cudaGetLastError();                   // clear the error state the failed query left
    return K8V4_EINVAL;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return K8V4_EINVAL;
  M->pages = static_cast<uint8_t*>(a.devicePointer);
  return K8V4_OK;
}

}  // namespace

uint32_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int withheld_copy() { return g_withhold.load(std::memory_order_relaxed); }

}  // namespace k8v4

using namespace k8v4;

extern "C" {

size_t k8v4_bytes_per_cell(int32_t format, int32_t n_kv_heads) {
  if (n_kv_heads < 1 || n_kv_heads > 8) return 0;
  if (format != K8V4_FORMAT_K8V4 && format != K8V4_FORMAT_INT8 && format != K8V4_FORMAT_Q4) return 0;
  return static_cast<size_t>(n_kv_heads) * cell_head_bytes(format);
}

const char* k8v4_status_string(int status) {
  switch (status) {
    case K8V4_OK: return "ok";
    case K8V4_EINVAL: return "invalid argument";
    case K8V4_ERANGE: return "position, length or page id out of range";
    case K8V4_EALIGN: return "misaligned pointer";
    case K8V4_ECUDA: return "CUDA runtime error";
    case K8V4_EDEVICE: return "no sm_103 device";
    case K8V4_ENOSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int k8v4_device_check(void) {
  DeviceState* s = nullptr;
  return device_state(&s);
}

int kv_append_k8v4(const k8v4_cache* cache, const int32_t* page_table, int64_t max_pages, int32_t n_seqs,
                   const int64_t* pos, int32_t n_tok, const void* k, const void* v, int32_t dtype, void* stream) {
  CacheView C;
  int rc = view_of(cache, &C);
  if (rc) return rc;
  if ((rc = check_table(C, page_table, max_pages))) return rc;
  if (n_seqs < 0 || n_tok < 0 || (dtype != K8V4_F32 && dtype != K8V4_BF16)) return K8V4_EINVAL;
  if (n_seqs == 0 || n_tok == 0) return K8V4_OK;
  if (!pos || !k || !v) return K8V4_EINVAL;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(pos, 8)) return K8V4_EALIGN;
  Launch L;
  if ((rc = make_launch(stream, &L))) return rc;
  return launch_append(L, C, page_table, max_pages, n_seqs, pos, n_tok, k, v, dtype);
}

size_t attn_k8v4_workspace_bytes(const k8v4_cache* cache, int32_t n_seqs, int32_t n_q_per_seq, int32_t max_seq_len) {
  CacheView C;
  if (view_of(cache, &C) != K8V4_OK) return 0;
  if (n_seqs < 0 || n_q_per_seq < 1 || n_q_per_seq > 8 || max_seq_len < 0) return 0;
  DeviceState* s = nullptr;
  const int sms = device_state(&s) == K8V4_OK ? s->num_sms : 152;
  return plan_attend(C, n_seqs, n_q_per_seq, max_seq_len, sms).ws_bytes;
}

static int attend_common(const k8v4_cache* cache, const void* q, int32_t q_dtype, const int32_t* page_table,
                         int64_t max_pages, const int32_t* steps, int32_t n_seqs, int32_t n_q, int32_t max_seq_len,
                         float sm_scale, float* out, void* ws, size_t ws_bytes, void* stream,
                         const void* k_new = nullptr, const void* v_new = nullptr, int32_t kv_dtype = K8V4_BF16) {
  CacheView C;
  int rc = view_of(cache, &C);
  if (rc) return rc;
  if ((rc = check_table(C, page_table, max_pages))) return rc;
  if (n_seqs < 0 || n_seqs > 65535 || n_q < 1 || n_q > 8) return K8V4_EINVAL;
  if (q_dtype != K8V4_F32 && q_dtype != K8V4_BF16) return K8V4_EINVAL;
  if (max_seq_len < 0 || static_cast<int64_t>(max_seq_len) > max_pages * C.P) return K8V4_EINVAL;
  if (!(sm_scale > 0.0f) || sm_scale > 1e30f) return K8V4_EINVAL;
  if (n_seqs == 0) return K8V4_OK;
  if (!q || !steps || !out || !ws) return K8V4_EINVAL;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(ws, 256) || !aligned(steps, 4)) return K8V4_EALIGN;
  Launch L;
  if ((rc = make_launch(stream, &L))) return rc;
  const AttendPlan plan = plan_attend(C, n_seqs, n_q, max_seq_len, L.num_sms);
  if (ws_bytes < plan.ws_bytes) return K8V4_ENOSPACE;
  return launch_attend(L, C, plan, q, q_dtype, page_table, max_pages, steps, n_seqs, max_seq_len, sm_scale, out, ws,
                       k_new, v_new, kv_dtype);
}

int attn_k8v4_decode(const k8v4_cache* cache, const void* q, int32_t q_dtype, const int32_t* page_table,
                     int64_t max_pages, const int32_t* seq_lens, int32_t n_seqs, int32_t max_seq_len, float sm_scale,
                     float* out, void* workspace, size_t workspace_bytes, void* stream) {
  return attend_common(cache, q, q_dtype, page_table, max_pages, seq_lens, n_seqs, 1, max_seq_len, sm_scale, out,
                       workspace, workspace_bytes, stream);
}

int attn_k8v4_decode_step(const k8v4_cache* cache, const void* q, int32_t q_dtype, const void* k_new,
                          const void* v_new, int32_t kv_dtype, const int32_t* page_table, int64_t max_pages,
                          const int32_t* seq_lens, int32_t n_seqs, int32_t max_seq_len, float sm_scale,
                          float* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (n_seqs > 0) {
    if (!k_new || !v_new) return K8V4_EINVAL;
    if (kv_dtype != K8V4_F32 && kv_dtype != K8V4_BF16) return K8V4_EINVAL;
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return K8V4_EALIGN;
  }
  return attend_common(cache, q, q_dtype, page_table, max_pages, seq_lens, n_seqs, 1, max_seq_len, sm_scale, out,
                       workspace, workspace_bytes, stream, k_new, v_new, kv_dtype);
}

int attn_k8v4_verify(const k8v4_cache* cache, const void* q, int32_t q_dtype, const int32_t* page_table,
                     int64_t max_pages, const int32_t* step_arrays, int32_t n_seqs, int32_t n_q, int32_t max_seq_len,
                     float sm_scale, float* out, void* workspace, size_t workspace_bytes, void* stream) {
  return attend_common(cache, q, q_dtype, page_table, max_pages, step_arrays, n_seqs, n_q, max_seq_len, sm_scale, out,
                       workspace, workspace_bytes, stream);
}

size_t attn_k8v4_partial_workspace_bytes(const k8v4_cache* cache, int32_t n_seqs, int32_t cell_begin,
                                         int32_t cell_end) {
  CacheView C;
  if (view_of(cache, &C) != K8V4_OK || !decode_ws_supported(C)) return 0;
  if (n_seqs < 0 || cell_begin < 0 || cell_end < cell_begin) return 0;
  DeviceState* s = nullptr;
  const int sms = device_state(&s) == K8V4_OK ? s->num_sms : 152;
  return plan_decode(C, n_seqs, cell_end - cell_begin, sms).ws_bytes;
}

int attn_k8v4_decode_partial(const k8v4_cache* cache, const void* q, int32_t q_dtype, const int32_t* page_table,
                             int64_t max_pages, const int32_t* seq_lens, int32_t n_seqs, int32_t max_seq_len,
                             int32_t cell_begin, int32_t cell_end, float sm_scale, float* partial, void* workspace,
                             size_t workspace_bytes, void* stream) {
  CacheView C;
  int rc = view_of(cache, &C);
  if (rc) return rc;
  if (!decode_ws_supported(C)) return K8V4_EINVAL;
  if ((rc = check_table(C, page_table, max_pages))) return rc;
  if (n_seqs < 0 || n_seqs > 65535) return K8V4_EINVAL;
  if (q_dtype != K8V4_F32 && q_dtype != K8V4_BF16) return K8V4_EINVAL;
  if (max_seq_len < 0 || static_cast<int64_t>(max_seq_len) > max_pages * C.P) return K8V4_EINVAL;
  if (cell_begin < 0 || cell_begin % 16 != 0 || cell_end < cell_begin) return K8V4_EINVAL;
  if (cell_end % 16 != 0 && cell_end < max_seq_len) return K8V4_EINVAL;
  if (!(sm_scale > 0.0f) || sm_scale > 1e30f) return K8V4_EINVAL;
  if (n_seqs == 0) return K8V4_OK;
  if (!q || !seq_lens || !partial || !workspace) return K8V4_EINVAL;
  if (!aligned(q, 16) || !aligned(partial, 16) || !aligned(workspace, 256) || !aligned(seq_lens, 4))
    return K8V4_EALIGN;
  Launch L;
  if ((rc = make_launch(stream, &L))) return rc;
  const AttendPlan plan = plan_decode(C, n_seqs, cell_end - cell_begin, L.num_sms);
  if (workspace_bytes < plan.ws_bytes) return K8V4_ENOSPACE;
  return launch_decode_partial(L, C, plan, q, q_dtype, page_table, max_pages, seq_lens, n_seqs, max_seq_len,
                               cell_begin, cell_end, sm_scale, partial, workspace, wait_limit_ns());
}

int attn_k8v4_combine_partials(const float* parts, int32_t n_parts, int32_t n_seqs, int32_t n_rows, float* out,
                               void* stream) {
  if (n_parts < 1 || n_parts > (1 << 20) || n_seqs < 0 || n_rows < 1 || n_rows > 4096) return K8V4_EINVAL;
  if (static_cast<int64_t>(n_seqs) * n_rows > (int64_t(1) << 31) - 1) return K8V4_EINVAL;
  if (n_seqs == 0) return K8V4_OK;
  if (!parts || !out) return K8V4_EINVAL;
  if (!aligned(parts, 16) || !aligned(out, 16)) return K8V4_EALIGN;
  Launch L;
  int rc = make_launch(stream, &L);
  if (rc) return rc;
  return launch_combine_parts(L, parts, n_parts, n_seqs, n_rows, out);
}

void k8v4_set_wait_limit_ns(uint32_t ns) { g_wait_ns.store(ns, std::memory_order_relaxed); }

void k8v4_set_withheld_copy(int32_t on) { g_withhold.store(on ? 1 : 0, std::memory_order_relaxed); }

int attn_k8v4_prefill(const k8v4_cache* cache, const void* q, int32_t q_dtype, const int32_t* page_table,
                      int64_t max_pages, int32_t seq_len, int32_t n_q_tok, const int32_t* step_arrays, float sm_scale,
                      float* out, void* stream) {
  CacheView C;
  int rc = view_of(cache, &C);
  if (rc) return rc;
  if (C.fmt != K8V4_FORMAT_K8V4) return K8V4_EINVAL;
  if ((rc = check_table(C, page_table, max_pages))) return rc;
  if (q_dtype != K8V4_BF16) return K8V4_EINVAL;
  if (n_q_tok < 0 || seq_len < 0 || static_cast<int64_t>(seq_len) > max_pages * C.P) return K8V4_EINVAL;
  if (!step_arrays && n_q_tok > seq_len) return K8V4_EINVAL;
  if (!(sm_scale > 0.0f) || sm_scale > 1e30f) return K8V4_EINVAL;
  if (n_q_tok == 0) return K8V4_OK;
  if (!q || !out) return K8V4_EINVAL;
  if (!aligned(q, 16) || !aligned(out, 16)) return K8V4_EALIGN;
  Launch L;
  if ((rc = make_launch(stream, &L))) return rc;
  return launch_prefill(L, C, q, page_table, max_pages, seq_len, n_q_tok, step_arrays, sm_scale, out);
}

int kv_dequant_k8v4(const k8v4_cache* cache, const int32_t* page_table, int64_t max_pages, int64_t start,
                    int64_t n_cells, float* k_out, float* v_rot_out, float* v_out, void* stream) {
  CacheView C;
  int rc = view_of(cache, &C);
  if (rc) return rc;
  if ((rc = check_table(C, page_table, max_pages))) return rc;
  if (start < 0 || n_cells < 0 || start + n_cells > max_pages * C.P) return K8V4_EINVAL;
  if (n_cells == 0) return K8V4_OK;
  if (!k_out || !v_rot_out) return K8V4_EINVAL;
  if (!aligned(k_out, 16) || !aligned(v_rot_out, 16) || (v_out && !aligned(v_out, 16))) return K8V4_EALIGN;
  Launch L;
  if ((rc = make_launch(stream, &L))) return rc;
  return launch_dequant(L, C, page_table, max_pages, start, n_cells, k_out, v_rot_out, v_out);
}

int kv_append_k8v4_mirrored(const k8v4_cache* host, const k8v4_cache* dev, const int32_t* slot_of_page,
                            const int32_t* page_table, int64_t max_pages, int32_t n_seqs, const int64_t* pos,
                            int32_t n_tok, const void* k, const void* v, int32_t dtype, void* stream) {
  CacheView C, M;
  int rc = view_of(dev, &C);
  if (rc) return rc;
  if ((rc = mirror_of(host, C, &M))) return rc;
  if ((rc = check_table(M, page_table, max_pages))) return rc;
  if (n_seqs < 0 || n_tok < 0 || (dtype != K8V4_F32 && dtype != K8V4_BF16)) return K8V4_EINVAL;
  if (n_seqs == 0 || n_tok == 0) return K8V4_OK;
  if (!pos || !k || !v || !slot_of_page) return K8V4_EINVAL;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(pos, 8) || !aligned(slot_of_page, 4)) return K8V4_EALIGN;
  Launch L;
  if ((rc = make_launch(stream, &L))) return rc;
  if ((rc = mirror_address(host, &M))) return rc;
  return launch_append(L, C, page_table, max_pages, n_seqs, pos, n_tok, k, v, dtype, &M, slot_of_page);
}

size_t kv_stream_workspace_bytes(int32_t n_seqs, int64_t max_pages) {
  if (n_seqs < 0 || max_pages < 1 || static_cast<int64_t>(n_seqs) * max_pages > (int64_t(1) << 28)) return 0;
  return stream_ws_bytes(n_seqs, max_pages);
}

int kv_stream_resolve(const k8v4_cache* host, const k8v4_cache* dev, const int32_t* slot_of_page, int32_t n_resident,
                      const int32_t* page_table, int64_t max_pages, const int32_t* seq_lens, int32_t n_seqs,
                      int32_t max_seq_len, int32_t* dev_page_table, void* workspace, size_t workspace_bytes,
                      void* stream) {
  CacheView C, M;
  int rc = view_of(dev, &C);
  if (rc) return rc;
  if ((rc = mirror_of(host, C, &M))) return rc;
  if ((rc = check_table(M, page_table, max_pages))) return rc;
  if (n_seqs < 0 || n_seqs > 65535 || static_cast<int64_t>(n_seqs) * max_pages > (int64_t(1) << 28))
    return K8V4_EINVAL;
  if (n_resident < 0 || n_resident > C.n_pages) return K8V4_EINVAL;
  if (max_seq_len < 0 || static_cast<int64_t>(max_seq_len) > max_pages * C.P) return K8V4_EINVAL;
  if (n_seqs == 0) return K8V4_OK;
  if (!slot_of_page || !seq_lens || !dev_page_table || !workspace) return K8V4_EINVAL;
  if (!aligned(slot_of_page, 4) || !aligned(seq_lens, 4) || !aligned(dev_page_table, 4) || !aligned(workspace, 16))
    return K8V4_EALIGN;
  if (workspace_bytes < stream_ws_bytes(n_seqs, max_pages)) return K8V4_ENOSPACE;
  Launch L;
  if ((rc = make_launch(stream, &L))) return rc;
  if ((rc = mirror_address(host, &M))) return rc;
  return launch_stream_resolve(L, M, C, slot_of_page, n_resident, page_table, max_pages, seq_lens, n_seqs,
                               max_seq_len, dev_page_table, workspace);
}

int kv_stream_copy(const k8v4_cache* host, const k8v4_cache* dev, const int32_t* pages, int32_t n, void* stream) {
  CacheView C, M;
  int rc = view_of(dev, &C);
  if (rc) return rc;
  if ((rc = mirror_of(host, C, &M))) return rc;
  if (n < 0) return K8V4_EINVAL;
  if (n == 0) return K8V4_OK;
  if (!pages) return K8V4_EINVAL;
  if (!aligned(pages, 8)) return K8V4_EALIGN;
  Launch L;
  if ((rc = make_launch(stream, &L))) return rc;
  if ((rc = mirror_address(host, &M))) return rc;
  return launch_stream_copy(L, M, C, pages, n);
}

int k8v4_last_device_status(void* stream) {
  Launch L;
  int rc = make_launch(stream, &L);
  if (rc) return rc;
  if (cudaStreamSynchronize(L.stream) != cudaSuccess) return K8V4_ECUDA;
  int value = 0;
  if (cudaMemcpy(&value, L.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return K8V4_ECUDA;
  const int zero = 0;
  if (cudaMemcpy(L.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return K8V4_ECUDA;
  return value;
}

}  // extern "C"
