// Conv-window kernel: pending conv fold + tree-aware causal depthwise conv,
// activation and per-head L2 normalisation of q and k.
//
// Luce DFlash README, "How it works" (ggml_ssm_conv_tree: each sibling reads its
// K-1 window along the parent chain, not DFS order); SpecLA article,
// "状态驻留验证" (ggml_ssm_conv_specla) and "延迟融合提交" (the pending path's raw
// rows are folded into the committed window before the verify reads it).
//
// One CTA per (request, layer, channel group); a group is one q head, one k head
// or one v head, one thread per channel.  Every thread owns one channel of the
// committed window, so the fold and the write-back need no synchronisation; the
// only block-wide step is the sum of squares for the q/k normalisation.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kConvThreads = 128;

template <typename InT>
__device__ __forceinline__ float load_in(const InT* p, size_t i);
template <>
__device__ __forceinline__ float load_in<float>(const float* p, size_t i) {
  return __ldg(p + i);
}
template <>
__device__ __forceinline__ float load_in<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red[] may still be read by the previous call
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kConvThreads / 32; ++w) s += red[w];
  return s;
}

template <typename InT>
__global__ void __launch_bounds__(kConvThreads) conv_window_kernel(ConvParams p) {
  __shared__ float red[kConvThreads / 32];
  const int bl = blockIdx.x;                 // request * layers + layer
  const int b = bl / p.layers, l = bl % p.layers;
  const int grp = blockIdx.y;
  const int nq = p.Hk * p.dk;
  int kind, c0, width;                       // kind 0: q head, 1: k head, 2: v head
  if (grp < p.Hk) {
    kind = 0; c0 = grp * p.dk; width = p.dk;
  } else if (grp < 2 * p.Hk) {
    kind = 1; c0 = nq + (grp - p.Hk) * p.dk; width = p.dk;
  } else {
    kind = 2; c0 = 2 * nq + (grp - 2 * p.Hk) * p.dv; width = p.dv;
  }
  const int t = threadIdx.x;
  const bool active = t < width;
  const int c = c0 + (active ? t : 0);
  const int K = p.K, C = p.C;
  const InT* x = static_cast<const InT*>(p.x_raw);

  // Committed window of this channel, oldest row first.
  float win[GDN_MAX_TAPS - 1];
  float w[GDN_MAX_TAPS];
  if (p.conv_mode == 1) {
    float* cs = p.conv_state + static_cast<size_t>(bl) * (K - 1) * C + c;
    for (int j = 0; j < K - 1; ++j) win[j] = active ? cs[static_cast<size_t>(j) * C] : 0.f;
    if (p.fold) {
      const int L = p.pend_len[b];
      if (L > 0) {
        const int32_t* path = p.pend_path + static_cast<size_t>(b) * p.n_max;
        const float* px = p.pend_x + static_cast<size_t>(bl) * p.n_max * C + c;
        for (int i = (L > K - 1 ? L - (K - 1) : 0); i < L; ++i) {
          for (int j = 0; j + 1 < K - 1; ++j) win[j] = win[j + 1];
          if (K > 1) win[K - 2] = active ? px[static_cast<size_t>(path[i]) * C] : 0.f;
        }
        if (active)
          for (int j = 0; j < K - 1; ++j) cs[static_cast<size_t>(j) * C] = win[j];
      }
    }
  }
  if (p.words == nullptr) return;  // fold only
  if (p.conv_mode == 1) {
    const float* cw = p.conv_w + (static_cast<size_t>(l) * C + c) * K;
    for (int j = 0; j < K; ++j) w[j] = active ? cw[j] : 0.f;
  }

  const SchedLayout lay{p.n_max};
  const int32_t* rec = p.words + static_cast<size_t>(b) * lay.words();
  const int n = rec[0];
  const int32_t* parent = rec + lay.parent();
  if (n < 1 || n > p.n_max) {
    if (threadIdx.x == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
    return;
  }
  const size_t xrow0 = static_cast<size_t>(bl) * p.n_max;   // row of node 0 of this (request, layer)

  for (int node = 0; node < n; ++node) {
    const float xs = active ? load_in<InT>(x, (xrow0 + node) * C + c) : 0.f;
    float y = xs;
    if (p.conv_mode == 1) {
      // tap K-1 multiplies the node itself, tap K-1-i its i-th predecessor on the
      // root path; past the root the committed window supplies the rows.
      y = w[K - 1] * xs;
      int m = parent[node];
      int ci = K - 2;
      for (int i = 1; i < K; ++i) {
        float xv;
        if (m >= 0) {
          xv = active ? load_in<InT>(x, (xrow0 + m) * C + c) : 0.f;
          m = parent[m];
          if (m >= node) m = -1;  // parents precede children; a corrupt entry ends the walk
        } else {
          xv = win[ci--];
        }
        y = fmaf(w[K - 1 - i], xv, y);
      }
      if (active) p.x_out[(xrow0 + node) * C + c] = xs;
    }
    if (p.act == 1) y = y / (1.f + expf(-y));
    if (kind < 2) {
      const float ss = block_sum(active ? y * y : 0.f, red);
      y = y * (1.f / sqrtf(ss + p.l2_eps));
      if (kind == 0) {
        y *= p.q_scale;
        if (active) p.q_out[((xrow0 + node) * p.Hk + grp) * p.dk + t] = y;
      } else if (active) {
        p.k_out[((xrow0 + node) * p.Hk + (grp - p.Hk)) * p.dk + t] = y;
      }
    } else if (active) {
      p.v_out[((xrow0 + node) * p.Hv + (grp - 2 * p.Hk)) * p.dv + t] = y;
    }
  }
}

}  // namespace

cudaError_t launch_conv(const ConvParams& p, cudaStream_t s) {
  dim3 grid(p.B * p.layers, 2 * p.Hk + p.Hv);
  if (p.in_dtype == GDN_DTYPE_BF16)
    conv_window_kernel<__nv_bfloat16><<<grid, kConvThreads, 0, s>>>(p);
  else
    conv_window_kernel<float><<<grid, kConvThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
