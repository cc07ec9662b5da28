// Conv-window kernel: pending conv fold + tree-aware causal depthwise conv,
// activation and per-head L2 normalisation of q and k.
//
// Luce DFlash README, "How it works" (ggml_ssm_conv_tree: each sibling reads its
// K-1 window along the parent chain, not DFS order); SpecLA article,
// "状态驻留验证" (ggml_ssm_conv_specla) and "延迟融合提交" (the pending path's raw
// rows are folded into the committed window before the verify reads it).
//
// One CTA per (request, layer, group of whole heads of one kind -- q, k or v --
// spanning at most 256 channels); every thread owns four adjacent channels, so
// loads of the raw rows are 8-byte (bf16) or 16-byte (fp32) per lane, stores
// 16-byte, and a head of up to 128 channels lies within one warp.
//   phase 0: TMA bulk copies bring the block's slice of every node's raw row
//            into shared memory; meanwhile each thread folds the pending raw
//            rows into its channels' committed window (it owns them, so the
//            write-back needs no barrier) and one thread per node records the
//            node's K-1 nearest ancestors;
//   phase 1: for every node convolve the window (tree ancestors, then the
//            committed rows past the root), apply SiLU, copy the raw row into
//            the factor bank, normalise q and k over each head's channels (a
//            shuffle over the head's lanes: no barrier per node) and write
//            q_hat / k_hat / v at once.
// Nothing per node stays in shared memory but the staged raw rows, so a CTA
// needs ~12 KB.  The kernel is bound by its instruction issue as much as by its
// bytes, so the per-node work is kept lean: four channels share every index,
// branch and reduction step, the row pointers advance by a row per node, and
// the norm's reciprocal square root is the hardware approximation (rsqrtf,
// within 2 ulp; the keys' tolerance is 1e-5).
// SiLU uses the fast exp and divide intrinsics (relative error ~1e-7).
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kConvThreads = 64;
constexpr int kConvPer = 4;                                // channels per thread
constexpr int kConvChannels = kConvPer * kConvThreads;     // channels per CTA

// Four consecutive raw values as fp32 (16-byte aligned for fp32, 8-byte for bf16).
template <typename InT>
__device__ __forceinline__ float4 raw4(const InT* p);
template <>
__device__ __forceinline__ float4 raw4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 raw4<__nv_bfloat16>(const __nv_bfloat16* p) {
  // a bf16 value is the upper half of the fp32 value with the same bits; the lower address holds the
  // lower half of each 32-bit word
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xFFFF0000u));
}
__device__ __forceinline__ float4 fma4(float4 a, float4 b, float4 c) {
  return make_float4(fmaf(a.x, b.x, c.x), fmaf(a.y, b.y, c.y), fmaf(a.z, b.z, c.z), fmaf(a.w, b.w, c.w));
}

__device__ __forceinline__ float silu(float y) { return __fdividef(y, 1.f + __expf(-y)); }

// Head group of blockIdx.y: kind (0 q, 1 k, 2 v), first head, head count, head size.
struct HeadGroup {
  int kind, head0, heads, hsz, cbase;
};
__device__ __forceinline__ HeadGroup head_group(const ConvParams& p, int y) {
  const int hq = kConvChannels / p.dk, hv = kConvChannels / p.dv;   // heads per group
  const int gq = (p.Hk + hq - 1) / hq;
  HeadGroup g;
  if (y < 2 * gq) {
    g.kind = y < gq ? 0 : 1;
    const int yy = y - g.kind * gq;
    g.head0 = yy * hq;
    g.heads = min(hq, p.Hk - g.head0);
    g.hsz = p.dk;
    g.cbase = g.kind * p.Hk * p.dk + g.head0 * p.dk;
  } else {
    g.kind = 2;
    g.head0 = (y - 2 * gq) * hv;
    g.heads = min(hv, p.Hv - g.head0);
    g.hsz = p.dv;
    g.cbase = 2 * p.Hk * p.dk + g.head0 * p.dv;
  }
  return g;
}

// KT > 0 fixes the number of taps at compile time (window and taps stay in
// registers); KT = 0 reads it from the parameters.
template <typename InT, int KT>
__global__ void __launch_bounds__(kConvThreads) conv_window_kernel(ConvParams p) {
  // shared: xs [n_max][256] InT | anc [n_max][K-1] int32 | mbarrier
  extern __shared__ float4 smem_conv[];
  InT* xs = reinterpret_cast<InT*>(smem_conv);
  int32_t* anc = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(xs) + p.n_max * kConvChannels * sizeof(InT));
  uint64_t* bar = reinterpret_cast<uint64_t*>(anc + ((p.n_max * (GDN_MAX_TAPS - 1) + 3) & ~3));
  const int bl = blockIdx.x;                   // request * layers + layer
  const int b = bl / p.layers, l = bl % p.layers;
  const int tid = threadIdx.x;
  const HeadGroup hg = head_group(p, blockIdx.y);
  const int width = hg.heads * hg.hsz;         // channels of this block
  const int c = hg.cbase + kConvPer * tid;     // first of this thread's four channels
  const bool active = kConvPer * tid < width;
  const int K = KT > 0 ? KT : p.K, C = p.C;
  const InT* x = static_cast<const InT*>(p.x_raw);
  if (__syncthreads_or(launch_aborted(p.err))) return;   // an earlier CTA gave up on a wait (one verdict)

  const SchedLayout lay{p.n_max};
  const int32_t* rec = p.words ? p.words + static_cast<size_t>(b) * lay.words() : nullptr;
  int n = 0;
  const size_t xrow0 = static_cast<size_t>(bl) * p.n_max;   // row of node 0 of this (request, layer)
  if (rec) {
    n = rec[0];
    if (n < 1 || n > p.n_max) {
      if (tid == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
      return;
    }
    if (tid == 0) mbar_init(bar);
    __syncthreads();
    if (tid < 32) {   // phase 0: raw rows of the block's channels, every node
      if (tid == 0) mbar_expect(bar, static_cast<uint32_t>(n) * width * sizeof(InT));
      __syncwarp();
      for (int node = tid; node < n; node += 32)
        bulk_g2s(xs + node * kConvChannels, x + (xrow0 + node) * C + hg.cbase, width * sizeof(InT), bar);
    }
    const int32_t* parent = rec + lay.parent();
    for (int node = tid; node < n; node += kConvThreads) {
      // ancestors 1..K-1 along the root path; -(j+1) = committed row K-1-j when the path runs out
      int m = parent[node], back = 0;
      for (int i = 1; i < K; ++i) {
        if (m >= 0 && m < node) {
          anc[node * (GDN_MAX_TAPS - 1) + i - 1] = m;
          m = parent[m];
        } else {
          anc[node * (GDN_MAX_TAPS - 1) + i - 1] = -(++back);
          m = -1;
        }
      }
    }
  }

  // Committed window of the four channels, oldest row first (fold the pending rows in first).
  float4 win[GDN_MAX_TAPS - 1];
  if (p.conv_mode == 1 && active) {
    float* cs = p.conv_state + static_cast<size_t>(bl) * (K - 1) * C + c;
#pragma unroll
    for (int j = 0; j < K - 1; ++j) win[j] = *reinterpret_cast<const float4*>(cs + static_cast<size_t>(j) * C);
    if (p.fold) {
      const int L = p.pend_len[b];
      if (L > 0) {
        const int32_t* path = p.pend_path + static_cast<size_t>(b) * p.n_max;
        const float* px = p.pend_x + static_cast<size_t>(bl) * p.n_max * C + c;
        for (int i = (L > K - 1 ? L - (K - 1) : 0); i < L; ++i) {
#pragma unroll
          for (int j = 0; j + 1 < K - 1; ++j) win[j] = win[j + 1];
          if (K > 1)
            win[K - 2] = *reinterpret_cast<const float4*>(px + static_cast<size_t>(path[i] & kPathNodeMask) * C);
        }
#pragma unroll
        for (int j = 0; j < K - 1; ++j) *reinterpret_cast<float4*>(cs + static_cast<size_t>(j) * C) = win[j];
      }
    }
  }
  if (rec == nullptr) return;  // fold only

  float4 w[GDN_MAX_TAPS];
  if (p.conv_mode == 1 && active) {
    const float* cw = p.conv_w + (static_cast<size_t>(l) * C + c) * K;
#pragma unroll
    for (int j = 0; j < K; ++j) w[j] = make_float4(cw[j], cw[K + j], cw[2 * K + j], cw[3 * K + j]);
  }
  if (!__syncthreads_and(mbar_wait(bar, 0))) {   // one verdict for the CTA; also publishes the ancestor table
    if (tid == 0) device_error(p.err, GDN_DEVERR_TIMEOUT, b);
    mbar_wait(bar, 0);   // let the copies land before the CTA exits
    return;
  }

  // per node: conv + activation, then (q and k heads) the L2 normalisation over the head's channels, and the
  // outputs written at once.  A head's channels are hsz / 4 consecutive lanes of one warp (8, 16 or 32 for
  // heads of 32, 64 or 128), so a shuffle over those lanes sums their squares; the lanes past the group's
  // channels form whole segments of their own and add zeros.
  const int hthreads = hg.hsz / kConvPer;                 // lanes per head
  const int hh = (kConvPer * tid) / hg.hsz;               // head within the group
  const int e0 = kConvPer * tid - hh * hg.hsz;            // first channel within the head
  const int kind = hg.kind;
  float* dst = nullptr;
  size_t dst_row = 0;
  if (kind == 0) {
    dst = p.q_out + static_cast<size_t>(hg.head0 + hh) * p.dk + e0;
    dst_row = static_cast<size_t>(p.Hk) * p.dk;
  } else if (kind == 1) {
    dst = p.k_out + static_cast<size_t>(hg.head0 + hh) * p.dk + e0;
    dst_row = static_cast<size_t>(p.Hk) * p.dk;
  } else {
    dst = p.v_out + static_cast<size_t>(hg.head0 + hh) * p.dv + e0;
    dst_row = static_cast<size_t>(p.Hv) * p.dv;
  }
  dst += xrow0 * dst_row;                                 // node 0's row; one row further per node
  float* xo = p.conv_mode == 1 ? p.x_out + xrow0 * C + c : nullptr;
  const InT* xt = xs + kConvPer * tid;                    // this thread's channels in the staged rows
  for (int node = 0; node < n; ++node) {
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active) {
      const float4 x0 = raw4<InT>(xt + node * kConvChannels);
      y = x0;
      if (p.conv_mode == 1) {
        // tap K-1 multiplies the node itself, tap K-1-i its i-th predecessor on the
        // root path; past the root the committed window supplies the rows.
        y = make_float4(w[K - 1].x * x0.x, w[K - 1].y * x0.y, w[K - 1].z * x0.z, w[K - 1].w * x0.w);
#pragma unroll
        for (int i = 1; i < K; ++i) {
          const int a = anc[node * (GDN_MAX_TAPS - 1) + i - 1];
          float4 xv;
          if (a >= 0) {
            xv = raw4<InT>(xt + a * kConvChannels);
          } else {
            // committed row K-1+a (a = -1 is the latest); register-resident select
            const int ci = K - 1 + a;
            xv = win[0];
#pragma unroll
            for (int j = 1; j < GDN_MAX_TAPS - 1; ++j)
              if (j < K - 1 && j == ci) xv = win[j];
          }
          y = fma4(w[K - 1 - i], xv, y);
        }
        *reinterpret_cast<float4*>(xo) = x0;
        xo += C;
      }
      if (p.act == 1) {
        y.x = silu(y.x);
        y.y = silu(y.y);
        y.z = silu(y.z);
        y.w = silu(y.w);
      }
    }
    float scale = 1.f;
    if (kind < 2) {   // CTA-uniform
      float ss = fmaf(y.x, y.x, fmaf(y.y, y.y, fmaf(y.z, y.z, y.w * y.w)));
      for (int o = hthreads / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      scale = rsqrtf(ss + p.l2_eps);
      if (kind == 0) scale *= p.q_scale;
    }
    if (active) *reinterpret_cast<float4*>(dst) = make_float4(y.x * scale, y.y * scale, y.z * scale, y.w * scale);
    dst += dst_row;
  }
}

template <typename InT, int KT>
cudaError_t launch_t(const ConvParams& p, cudaStream_t s) {
  const int hq = kConvChannels / p.dk, hv = kConvChannels / p.dv;
  dim3 grid(p.B * p.layers, 2 * ((p.Hk + hq - 1) / hq) + (p.Hv + hv - 1) / hv);
  const size_t smem =
      p.words ? static_cast<size_t>(p.n_max) * kConvChannels * sizeof(InT) + ((p.n_max * (GDN_MAX_TAPS - 1) + 3) & ~3) * 4 + 16
              : 0;
  auto k = conv_window_kernel<InT, KT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  k<<<grid, kConvThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv(const ConvParams& p, cudaStream_t s) {
  if (p.in_dtype == GDN_DTYPE_BF16)
    return p.K == 4 ? launch_t<__nv_bfloat16, 4>(p, s) : launch_t<__nv_bfloat16, 0>(p, s);
  return p.K == 4 ? launch_t<float, 4>(p, s) : launch_t<float, 0>(p, s);
}

}  // namespace gdn
