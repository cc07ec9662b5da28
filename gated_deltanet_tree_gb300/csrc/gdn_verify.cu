// State-resident chain verify with the deferred commit folded into the tile load.
//
// SpecLA article: "状态驻留验证" (the nodes of a chain are processed serially in
// one kernel with the state tile held in registers), "链分解与依赖波 HLD 调度"
// (heavy-light chains, boundary states materialised at branch points, waves),
// "延迟融合提交" (the pending accepted path is folded into the state tile when it
// is loaded, the committed state is written back once, and verification goes
// on with the same live tile).
//
// Work unit: one CTA per (request, layer, v-head, column slice of d_v).  The CTA
// walks every chain of its tree in schedule order (wave, head): the root chain
// continues from the folded committed state; any other chain reloads the state
// that a chain of an earlier wave stored at its boundary slot.  Each thread owns
// one column of the slice and RPT = dk / TPC rows of it, so p = T^T k and
// o = T^T q are in-thread sums plus (TPC = 2) one shuffle.  The per-node q/k of
// the whole tree are staged in shared memory once.
//
// Arithmetic order is fixed so that the fold reproduces the verify bitwise:
// both compute T <- fmaf(k, u, g * T) with the same u.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kVerifyThreads = 128;

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

template <int DK, int TPC, typename InT>
__global__ void __launch_bounds__(kVerifyThreads) chain_verify_kernel(VerifyParams p, int cpb) {
  constexpr int RPT = DK / TPC;             // rows of the tile per thread
  static_assert(RPT % 4 == 0, "rows per thread must be a multiple of 4");
  extern __shared__ float4 smem4[];
  float* kq = reinterpret_cast<float*>(smem4);   // [n][2][DK]: k_hat then q_hat of every node

  const int slices = p.dv / cpb;
  int cta = blockIdx.x;
  const int s = cta % slices;
  cta /= slices;
  const int h = cta % p.Hv;
  cta /= p.Hv;
  const int l = cta % p.layers;
  const int b = cta / p.layers;
  const int bl = b * p.layers + l;
  const int kh = h / p.R;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kColsPerWarp = 32 / TPC;
  const int half = lane / kColsPerWarp;
  const int col = s * cpb + warp * kColsPerWarp + (lane % kColsPerWarp);
  const int row0 = half * RPT;
  const size_t tile = static_cast<size_t>(DK) * p.dv;

  float T[RPT];
  float* st = p.state + (static_cast<size_t>(bl) * p.Hv + h) * tile + static_cast<size_t>(row0) * p.dv + col;
#pragma unroll
  for (int r = 0; r < RPT; ++r) T[r] = st[static_cast<size_t>(r) * p.dv];

  // Deferred commit: T <- exp(a) T + k u^T along the pending path, gathered by node index.
  if (p.fold) {
    const int L = p.pend_len[b];
    const int32_t* path = p.pend_path + static_cast<size_t>(b) * p.n_max;
    for (int i = 0; i < L; ++i) {
      const size_t row = static_cast<size_t>(bl) * p.n_max + path[i];
      const float g = expf(p.pend_a[row * p.Hv + h]);
      const float u = p.pend_u[(row * p.Hv + h) * p.dv + col];
      const float4* k4 = reinterpret_cast<const float4*>(p.pend_k + (row * p.Hk + kh) * DK + row0);
#pragma unroll
      for (int r4 = 0; r4 < RPT / 4; ++r4) {
        const float4 kv = __ldg(k4 + r4);
        T[4 * r4 + 0] = fmaf(kv.x, u, g * T[4 * r4 + 0]);
        T[4 * r4 + 1] = fmaf(kv.y, u, g * T[4 * r4 + 1]);
        T[4 * r4 + 2] = fmaf(kv.z, u, g * T[4 * r4 + 2]);
        T[4 * r4 + 3] = fmaf(kv.w, u, g * T[4 * r4 + 3]);
      }
    }
    if (L > 0) {
#pragma unroll
      for (int r = 0; r < RPT; ++r) st[static_cast<size_t>(r) * p.dv] = T[r];
    }
  }
  if (p.words == nullptr) return;  // fold only

  const SchedLayout lay{p.n_max};
  const int32_t* rec = p.words + static_cast<size_t>(b) * lay.words();
  const int n = rec[0];
  const int n_chains = rec[1];
  if (n < 1 || n > p.n_max || n_chains < 1 || n_chains > n) {
    if (threadIdx.x == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
    return;
  }
  const int32_t* bslot = rec + lay.bslot();
  const int32_t* csrc = rec + lay.chain_src();
  const int32_t* coff = rec + lay.chain_off();
  const int32_t* cnodes = rec + lay.chain_nodes();

  // Stage k_hat and q_hat of every node of the tree.
  {
    const size_t nrow0 = static_cast<size_t>(bl) * p.n_max;
    for (int idx = threadIdx.x; idx < n * (DK / 4); idx += blockDim.x) {
      const int node = idx / (DK / 4), e4 = idx % (DK / 4);
      const size_t src = ((nrow0 + node) * p.Hk + kh) * DK;
      smem4[(node * 2 + 0) * (DK / 4) + e4] = __ldg(reinterpret_cast<const float4*>(p.k_in + src) + e4);
      smem4[(node * 2 + 1) * (DK / 4) + e4] = __ldg(reinterpret_cast<const float4*>(p.q_in + src) + e4);
    }
  }
  __syncthreads();

  const InT* beta = static_cast<const InT*>(p.beta);
  const InT* logg = static_cast<const InT*>(p.log_g);
  float* bnd_base = p.boundary + (static_cast<size_t>(bl) * p.nb_max * p.Hv + h) * tile +
                    static_cast<size_t>(row0) * p.dv + col;
  const size_t slot_stride = static_cast<size_t>(p.Hv) * tile;

  for (int c = 0; c < n_chains; ++c) {
    const int src = csrc[c];
    const int i0 = coff[c], i1 = coff[c + 1];
    if (src >= p.nb_max || i0 < 0 || i1 > n || i0 > i1) {
      if (threadIdx.x == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
      return;
    }
    if (src >= 0) {
      const float* bs = bnd_base + static_cast<size_t>(src) * slot_stride;
#pragma unroll
      for (int r = 0; r < RPT; ++r) T[r] = bs[static_cast<size_t>(r) * p.dv];
    }
    for (int i = i0; i < i1; ++i) {
      const int node = cnodes[i];
      if (node < 0 || node >= n) {
        if (threadIdx.x == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
        return;
      }
      const size_t row = static_cast<size_t>(bl) * p.n_max + node;
      const float a = load_in<InT>(logg, row * p.Hv + h);
      const float bt = load_in<InT>(beta, row * p.Hv + h);
      const float v = p.v_in[(row * p.Hv + h) * p.dv + col];
      const float g = expf(a);
      const float4* k4 = reinterpret_cast<const float4*>(kq + (node * 2 + 0) * DK + row0);
      const float4* q4 = reinterpret_cast<const float4*>(kq + (node * 2 + 1) * DK + row0);

      float pk = 0.f;
#pragma unroll
      for (int r4 = 0; r4 < RPT / 4; ++r4) {
        const float4 kv = k4[r4];
        T[4 * r4 + 0] = g * T[4 * r4 + 0];
        T[4 * r4 + 1] = g * T[4 * r4 + 1];
        T[4 * r4 + 2] = g * T[4 * r4 + 2];
        T[4 * r4 + 3] = g * T[4 * r4 + 3];
        pk = fmaf(T[4 * r4 + 0], kv.x, pk);
        pk = fmaf(T[4 * r4 + 1], kv.y, pk);
        pk = fmaf(T[4 * r4 + 2], kv.z, pk);
        pk = fmaf(T[4 * r4 + 3], kv.w, pk);
      }
      if (TPC == 2) pk += __shfl_xor_sync(0xffffffffu, pk, kColsPerWarp);
      const float u = bt * (v - pk);
      float o = 0.f;
#pragma unroll
      for (int r4 = 0; r4 < RPT / 4; ++r4) {
        const float4 kv = k4[r4];
        const float4 qv = q4[r4];
        T[4 * r4 + 0] = fmaf(kv.x, u, T[4 * r4 + 0]);
        T[4 * r4 + 1] = fmaf(kv.y, u, T[4 * r4 + 1]);
        T[4 * r4 + 2] = fmaf(kv.z, u, T[4 * r4 + 2]);
        T[4 * r4 + 3] = fmaf(kv.w, u, T[4 * r4 + 3]);
        o = fmaf(T[4 * r4 + 0], qv.x, o);
        o = fmaf(T[4 * r4 + 1], qv.y, o);
        o = fmaf(T[4 * r4 + 2], qv.z, o);
        o = fmaf(T[4 * r4 + 3], qv.w, o);
      }
      if (TPC == 2) o += __shfl_xor_sync(0xffffffffu, o, kColsPerWarp);
      if (half == 0) {
        p.out_o[(row * p.Hv + h) * p.dv + col] = o;
        p.u_out[(row * p.Hv + h) * p.dv + col] = u;
      }
      if (threadIdx.x == 0 && s == 0) p.a_out[row * p.Hv + h] = a;
      const int slot = bslot[node];
      if (slot >= p.nb_max) {
        if (threadIdx.x == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
      } else if (slot >= 0) {
        float* bs = bnd_base + static_cast<size_t>(slot) * slot_stride;
#pragma unroll
        for (int r = 0; r < RPT; ++r) bs[static_cast<size_t>(r) * p.dv] = T[r];
      }
    }
  }
}

template <int DK, int TPC, typename InT>
cudaError_t launch_t(const VerifyParams& p, cudaStream_t s) {
  const int cpb = min(p.dv, kVerifyThreads / TPC);    // columns per CTA
  const int threads = cpb * TPC;
  const size_t grid = static_cast<size_t>(p.B) * p.layers * p.Hv * (p.dv / cpb);
  const size_t smem = p.words ? static_cast<size_t>(p.n_max) * 2 * DK * sizeof(float) : 0;
  auto kern = chain_verify_kernel<DK, TPC, InT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<static_cast<unsigned>(grid), threads, smem, s>>>(p, cpb);
  return cudaGetLastError();
}

template <typename InT>
cudaError_t launch_dtype(const VerifyParams& p, cudaStream_t s) {
  switch (p.dk) {
    case 32: return launch_t<32, 1, InT>(p, s);
    case 64: return launch_t<64, 1, InT>(p, s);
    case 128: return launch_t<128, 2, InT>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool verify_supported(int dk, int dv) {
  const bool dk_ok = dk == 32 || dk == 64 || dk == 128;
  const bool dv_ok = dv == 32 || dv == 64 || dv == 128;
  return dk_ok && dv_ok;
}

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t s) {
  if (p.in_dtype == GDN_DTYPE_BF16) return launch_dtype<__nv_bfloat16>(p, s);
  return launch_dtype<float>(p, s);
}

}  // namespace gdn
