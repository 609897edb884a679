// Combine of the split-K partials of decode and verify: each split wrote, per
// output row, its un-rotated o[256] together with its running maximum m (log2
// domain) and sum l; the row's result is sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
//
// One CTA per (row, 32-dim chunk), eight warps.  Warp w folds splits w, w + 8,
// ... into a running (M, L, acc) with the online-softmax update, so every load
// of a split is independent of the others (no separate maximum pass); the eight
// warp states are merged in shared memory.  Launched as a programmatic
// dependent of the split kernel: the launch overlaps the split kernel's tail and
// griddepcontrol.wait holds the loads until the partials are written.
#include "k8v4_common.cuh"

namespace k8v4 {
namespace {

constexpr int kPStride = 260;   // floats per partial row: o[256], m, l, 2 pad

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ ws, int splits, int n_q, int HQ,
                                                      float* __restrict__ out) {
  __shared__ float wm[8], wl[8], wacc[8][32];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int row = blockIdx.x, chunk = blockIdx.y;   // row = (b, qi, head)
  const int head = row % HQ;
  const int bq = row / HQ;
  const int b = bq / n_q, qi = bq % n_q;
  const int64_t stride = static_cast<int64_t>(n_q) * HQ * kPStride;     // between splits
  const float* base = ws + ((static_cast<int64_t>(b) * splits * n_q + qi) * HQ + head) * kPStride;
  const int dim = chunk * 32 + lane;
  float M = -INFINITY, L = 0.0f, acc = 0.0f;
#pragma unroll 4
  for (int s = warp; s < splits; s += 8) {
    const float* src = base + s * stride;
    const float ms = src[256], ls = src[257], x = src[dim];
    if (ms == -INFINITY) continue;                     // nothing visible in this split
    const float mn = fmaxf(M, ms);
    const float a = exp2f(M - mn), w = exp2f(ms - mn);  // a = 0 while M = -inf
    acc = acc * a + x * w;
    L = L * a + ls * w;
    M = mn;
  }
  if (lane == 0) {
    wm[warp] = M;
    wl[warp] = L;
  }
  wacc[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float Mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < 8; ++w) Mt = fmaxf(Mt, wm[w]);
    float v = 0.0f, Lt = 0.0f;
    if (Mt != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        if (wm[w] == -INFINITY) continue;
        const float f = exp2f(wm[w] - Mt);
        v += wacc[w][lane] * f;
        Lt += wl[w] * f;
      }
    }
    out[static_cast<int64_t>(row) * kD + dim] = Lt > 0.0f ? v / Lt : 0.0f;
  }
}

}  // namespace

int launch_combine(const Launch& L, const float* ws, int splits, int n_seqs, int n_q, int H, float* out) {
  const int rows = n_seqs * n_q * H * kGqa;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows, kD / 32);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, combine_kernel, ws, splits, n_q, H * kGqa, out) != cudaSuccess) return K8V4_ECUDA;
  return cudaGetLastError() == cudaSuccess ? K8V4_OK : K8V4_ECUDA;
}

}  // namespace k8v4
