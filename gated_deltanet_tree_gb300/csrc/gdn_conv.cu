// Conv-window kernel: pending conv fold + tree-aware causal depthwise conv,
// activation and per-head L2 normalisation of q and k.
//
// Luce DFlash README, "How it works" (ggml_ssm_conv_tree: each sibling reads its
// K-1 window along the parent chain, not DFS order); SpecLA article,
// "状态驻留验证" (ggml_ssm_conv_specla) and "延迟融合提交" (the pending path's raw
// rows are folded into the committed window before the verify reads it).
//
// One CTA per (request, layer, group of whole heads of one kind -- q, k or v --
// spanning at most 256 channels); every thread owns two adjacent channels, so
// loads of the raw rows are 4-byte (bf16) or 8-byte (fp32) per lane and
// coalesced.
//   phase 0: TMA bulk copies bring the block's slice of every node's raw row
//            into shared memory; meanwhile each thread folds the pending raw
//            rows into its channels' committed window (it owns them, so the
//            write-back needs no barrier) and one thread per node records the
//            node's K-1 nearest ancestors;
//   phase 1: for every node convolve the window (tree ancestors, then the
//            committed rows past the root), apply SiLU, copy the raw row into
//            the factor bank, normalise q and k over each head's channels (a
//            segmented shuffle; a 128-channel head's two warps add their halves
//            through shared memory) and write q_hat / k_hat / v at once.
// Nothing per node stays in shared memory but the staged raw rows, so a CTA
// needs ~12 KB and the SM's thread count, not its shared memory, bounds the
// CTAs resident at once.
// SiLU uses the fast exp and divide intrinsics (relative error ~1e-7).
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kConvThreads = 128;
constexpr int kConvChannels = 2 * kConvThreads;   // channels per CTA

template <typename InT>
__device__ __forceinline__ float2 raw2(const InT* p);
template <>
__device__ __forceinline__ float2 raw2<float>(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
template <>
__device__ __forceinline__ float2 raw2<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
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
  // shared: xs [n_max][256] InT | anc [n_max][K-1] int32 | mbarrier | partial sums [2][warps] f32
  extern __shared__ float4 smem_conv[];
  InT* xs = reinterpret_cast<InT*>(smem_conv);
  int32_t* anc = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(xs) + p.n_max * kConvChannels * sizeof(InT));
  uint64_t* bar = reinterpret_cast<uint64_t*>(anc + ((p.n_max * (GDN_MAX_TAPS - 1) + 3) & ~3));
  const int bl = blockIdx.x;                   // request * layers + layer
  const int b = bl / p.layers, l = bl % p.layers;
  const int tid = threadIdx.x;
  const HeadGroup hg = head_group(p, blockIdx.y);
  const int width = hg.heads * hg.hsz;         // channels of this block
  const int c = hg.cbase + 2 * tid;            // first of this thread's two channels
  const bool active = 2 * tid < width;
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

  // Committed window of the two channels, oldest row first (fold the pending rows in first).
  float2 win[GDN_MAX_TAPS - 1];
  if (p.conv_mode == 1 && active) {
    float* cs = p.conv_state + static_cast<size_t>(bl) * (K - 1) * C + c;
#pragma unroll
    for (int j = 0; j < K - 1; ++j) win[j] = *reinterpret_cast<const float2*>(cs + static_cast<size_t>(j) * C);
    if (p.fold) {
      const int L = p.pend_len[b];
      if (L > 0) {
        const int32_t* path = p.pend_path + static_cast<size_t>(b) * p.n_max;
        const float* px = p.pend_x + static_cast<size_t>(bl) * p.n_max * C + c;
        for (int i = (L > K - 1 ? L - (K - 1) : 0); i < L; ++i) {
#pragma unroll
          for (int j = 0; j + 1 < K - 1; ++j) win[j] = win[j + 1];
          if (K > 1)
            win[K - 2] = *reinterpret_cast<const float2*>(px + static_cast<size_t>(path[i] & kPathNodeMask) * C);
        }
#pragma unroll
        for (int j = 0; j < K - 1; ++j) *reinterpret_cast<float2*>(cs + static_cast<size_t>(j) * C) = win[j];
      }
    }
  }
  if (rec == nullptr) return;  // fold only

  float2 w[GDN_MAX_TAPS];
  if (p.conv_mode == 1 && active) {
    const float* cw = p.conv_w + (static_cast<size_t>(l) * C + c) * K;
#pragma unroll
    for (int j = 0; j < K; ++j) w[j] = make_float2(cw[j], cw[K + j]);
  }
  if (!__syncthreads_and(mbar_wait(bar, 0))) {   // one verdict for the CTA; also publishes the ancestor table
    if (tid == 0) device_error(p.err, GDN_DEVERR_TIMEOUT, b);
    mbar_wait(bar, 0);   // let the copies land before the CTA exits
    return;
  }

  // per node: conv + activation, then (q and k heads) the L2 normalisation over the head's channels, and the
  // outputs written at once.  A head's channels are hsz / 2 consecutive threads: a segmented shuffle sums
  // their squares; a 128-channel head spans two warps, which add their halves through a shared slot
  // (double-buffered by node parity, so one barrier per node suffices).
  const int lane = tid & 31, warp = tid >> 5;
  const int hthreads = hg.hsz / 2;                  // threads per head
  const int hh = (2 * tid) / hg.hsz;                // head within the group
  const int e0 = 2 * tid - hh * hg.hsz;             // first channel within the head
  float* part = reinterpret_cast<float*>(bar + 1);  // [2][kConvThreads / 32]
  const int kind = hg.kind;
  float* dst0 = nullptr;
  size_t dst_row = 0;
  if (kind == 0) {
    dst0 = p.q_out + static_cast<size_t>(hg.head0 + hh) * p.dk + e0;
    dst_row = static_cast<size_t>(p.Hk) * p.dk;
  } else if (kind == 1) {
    dst0 = p.k_out + static_cast<size_t>(hg.head0 + hh) * p.dk + e0;
    dst_row = static_cast<size_t>(p.Hk) * p.dk;
  } else {
    dst0 = p.v_out + static_cast<size_t>(hg.head0 + hh) * p.dv + e0;
    dst_row = static_cast<size_t>(p.Hv) * p.dv;
  }
  for (int node = 0; node < n; ++node) {
    float2 y = make_float2(0.f, 0.f);
    if (active) {
      const float2 xs0 = raw2<InT>(xs + node * kConvChannels + 2 * tid);
      y = xs0;
      if (p.conv_mode == 1) {
        // tap K-1 multiplies the node itself, tap K-1-i its i-th predecessor on the
        // root path; past the root the committed window supplies the rows.
        y.x = w[K - 1].x * xs0.x;
        y.y = w[K - 1].y * xs0.y;
#pragma unroll
        for (int i = 1; i < K; ++i) {
          const int a = anc[node * (GDN_MAX_TAPS - 1) + i - 1];
          float2 xv;
          if (a >= 0) {
            xv = raw2<InT>(xs + a * kConvChannels + 2 * tid);
          } else {
            // committed row K-1+a (a = -1 is the latest); register-resident select
            const int ci = K - 1 + a;
            xv = win[0];
#pragma unroll
            for (int j = 1; j < GDN_MAX_TAPS - 1; ++j)
              if (j < K - 1 && j == ci) xv = win[j];
          }
          y.x = fmaf(w[K - 1 - i].x, xv.x, y.x);
          y.y = fmaf(w[K - 1 - i].y, xv.y, y.y);
        }
        *reinterpret_cast<float2*>(p.x_out + (xrow0 + node) * C + c) = xs0;
      }
      if (p.act == 1) {
        y.x = silu(y.x);
        y.y = silu(y.y);
      }
    }
    float scale = 1.f;
    if (kind < 2) {   // CTA-uniform
      float ss = fmaf(y.x, y.x, y.y * y.y);
      for (int o = (hthreads < 32 ? hthreads : 32) / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (hthreads > 32) {   // two warps per head
        if (lane == 0) part[(node & 1) * (kConvThreads / 32) + warp] = ss;
        __syncthreads();
        ss += part[(node & 1) * (kConvThreads / 32) + (warp ^ 1)];
      }
      scale = 1.f / sqrtf(ss + p.l2_eps);
      if (kind == 0) scale *= p.q_scale;
    }
    if (active)
      *reinterpret_cast<float2*>(dst0 + (xrow0 + node) * dst_row) = make_float2(y.x * scale, y.y * scale);
  }
}

template <typename InT, int KT>
cudaError_t launch_t(const ConvParams& p, cudaStream_t s) {
  const int hq = kConvChannels / p.dk, hv = kConvChannels / p.dv;
  dim3 grid(p.B * p.layers, 2 * ((p.Hk + hq - 1) / hq) + (p.Hv + hv - 1) / hv);
  const size_t smem =
      p.words ? static_cast<size_t>(p.n_max) * kConvChannels * sizeof(InT) +
                    ((p.n_max * (GDN_MAX_TAPS - 1) + 3) & ~3) * 4 + 16 + 2 * (kConvThreads / 32) * 4
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
