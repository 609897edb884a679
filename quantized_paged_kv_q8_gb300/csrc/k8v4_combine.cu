// Combine of split-K partials: each split (or, for the cell-range split across
// GPUs, each rank) wrote, per output row, its un-rotated o[256] together with
// its running maximum m (base-2 exponent) and sum l; the row's result is
// sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.  The same kernel can instead
// write the merged partial itself (o, M, L unnormalised), which is what one GPU
// of a cell-range split hands to the others.
//
// One CTA per (row, 32-dim chunk), eight warps.  Warp w takes splits w, w + 8,
// ... in rounds of R: every load of a round (each split's m and l, and the
// lane's element of o) is issued before any is used, so a round costs one L2
// round trip; the round is folded at its own maximum into the warp's running
// (M, L, acc), and the eight warp states are merged in shared memory.  Two
// instantiations: R = 12 (64 registers, four CTAs per SM) for many splits, so
// that a long single-sequence decode (76 splits per KV head on 152 SMs) takes
// one round; R = 3 (32 registers, eight CTAs per SM) for up to 24 splits, where
// a batch of sequences brings thousands of rows.  Launched as a programmatic
// dependent of the split kernel: the launch overlaps the split kernel's tail and
// griddepcontrol.wait holds the loads until the partials are written.
#include "k8v4_common.cuh"

namespace k8v4 {
namespace {

constexpr int kPStride = 260;   // floats per partial row: o[256], m, l, 2 pad
constexpr int kRoundMany = 12;  // splits per warp whose loads are in flight together
constexpr int kRoundFew = 3;

// row r = (b, rr) with rr < rows_per_b; split s of row r at
// src + b * b_stride + s * split_stride + rr * kPStride
template <int R>
__global__ void __launch_bounds__(256, R <= kRoundFew ? 8 : 4)
    combine_kernel(const float* __restrict__ src, int splits, int64_t split_stride, int64_t b_stride, int rows_per_b,
                   float* __restrict__ out, int write_partial) {
  __shared__ float wm[8], wl[8], wacc[8][32];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int row = blockIdx.x, chunk = blockIdx.y;
  const int b = row / rows_per_b, rr = row % rows_per_b;
  const float* base = src + b * b_stride + static_cast<int64_t>(rr) * kPStride;
  const int dim = chunk * 32 + lane;
  float M = -INFINITY, L = 0.0f, acc = 0.0f;
  for (int s0 = warp; s0 < splits; s0 += 8 * R) {
    float ms[R], ls[R], xs[R];
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const int s = s0 + 8 * k;
      ms[k] = -INFINITY;
      ls[k] = xs[k] = 0.0f;
      if (s < splits) {
        const float* p = base + s * split_stride;
        ms[k] = p[256];
        ls[k] = p[257];
        xs[k] = p[dim];
      }
    }
    float mr = M;
#pragma unroll
    for (int k = 0; k < R; ++k) mr = fmaxf(mr, ms[k]);
    if (mr == -INFINITY) continue;                      // nothing visible yet (the same for the warp)
    const float a = exp2f(M - mr);                      // 0 while M = -inf
    acc *= a;
    L *= a;
#pragma unroll
    for (int k = 0; k < R; ++k) {
      if (ms[k] == -INFINITY) continue;                 // a split with nothing visible
      const float wk = exp2f(ms[k] - mr);
      acc += xs[k] * wk;
      L += ls[k] * wk;
    }
    M = mr;
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
    if (write_partial) {
      float* dst = out + static_cast<int64_t>(row) * kPStride;
      dst[dim] = v;
      if (chunk == 0 && lane == 0) {
        dst[256] = Mt;
        dst[257] = Lt;
        dst[258] = 0.0f;
        dst[259] = 0.0f;
      }
    } else {
      out[static_cast<int64_t>(row) * kD + dim] = Lt > 0.0f ? v / Lt : 0.0f;
    }
  }
}

int launch(const Launch& L, const float* src, int splits, int64_t split_stride, int64_t b_stride, int n_seqs,
           int rows_per_b, float* out, int write_partial) {
  const int rows = n_seqs * rows_per_b;
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
  const cudaError_t e =
      splits <= 8 * kRoundFew
          ? cudaLaunchKernelEx(&cfg, combine_kernel<kRoundFew>, src, splits, split_stride, b_stride, rows_per_b, out,
                               write_partial)
          : cudaLaunchKernelEx(&cfg, combine_kernel<kRoundMany>, src, splits, split_stride, b_stride, rows_per_b, out,
                               write_partial);
  if (e != cudaSuccess) return K8V4_ECUDA;
  return cudaGetLastError() == cudaSuccess ? K8V4_OK : K8V4_ECUDA;
}

}  // namespace

int launch_combine(const Launch& L, const float* ws, int splits, int n_seqs, int n_q, int H, float* out) {
  const int rows_per_b = n_q * H * kGqa;
  const int64_t split_stride = static_cast<int64_t>(rows_per_b) * kPStride;
  return launch(L, ws, splits, split_stride, split_stride * splits, n_seqs, rows_per_b, out, 0);
}

int launch_combine_partial(const Launch& L, const float* ws, int splits, int n_seqs, int H, float* partial) {
  const int rows_per_b = H * kGqa;
  const int64_t split_stride = static_cast<int64_t>(rows_per_b) * kPStride;
  return launch(L, ws, splits, split_stride, split_stride * splits, n_seqs, rows_per_b, partial, 1);
}

int launch_combine_parts(const Launch& L, const float* parts, int n_parts, int n_seqs, int n_rows_per_seq,
                         float* out) {
  const int64_t b_stride = static_cast<int64_t>(n_rows_per_seq) * kPStride;
  return launch(L, parts, n_parts, b_stride * n_seqs, b_stride, n_seqs, n_rows_per_seq, out, 0);
}

}  // namespace k8v4
