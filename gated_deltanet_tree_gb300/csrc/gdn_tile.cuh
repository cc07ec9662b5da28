// A thread's register tile of a [d_k][d_v] state and the operations both verify
// kernels apply to it: the packed f32x2 arithmetic, the lazily decayed update of
// the gated delta rule, and the fold of a committed node.  Both kernels fold with
// these same functions, so a state folded by one equals, bit for bit, the state
// the other stored for the same node.
#pragma once
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {

typedef unsigned long long u64;

constexpr int kCols = 4;                  // columns per thread
constexpr int kFoldChunk = 16;            // pending nodes staged per fold step
constexpr float kGammaFloor = 1.0e-12f;   // below this the decay is applied to the tile at once

__device__ __forceinline__ u64 pack2(float lo, float hi) {
  u64 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(u64 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
  u64 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

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

// RPT consecutive rows x kCols consecutive columns, held as packed (row r, row r + 1) pairs:
// T[c][j] = (T[row0 + 2j][c0 + c], T[row0 + 2j + 1][c0 + c]).  Row pointers below point at the
// thread's first element; `ld` is the row stride in floats.
template <int RPT>
struct RegTile {
  static constexpr int NP = RPT / 2;
  u64 T[kCols][NP];

  __device__ __forceinline__ void load(const float* base, size_t ld) {
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const float4 r0 = *reinterpret_cast<const float4*>(base + static_cast<size_t>(2 * j) * ld);
      const float4 r1 = *reinterpret_cast<const float4*>(base + static_cast<size_t>(2 * j + 1) * ld);
      T[0][j] = pack2(r0.x, r1.x);
      T[1][j] = pack2(r0.y, r1.y);
      T[2][j] = pack2(r0.z, r1.z);
      T[3][j] = pack2(r0.w, r1.w);
    }
  }
  __device__ __forceinline__ void store(float* base, size_t ld) const {
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const float2 a0 = unpack2(T[0][j]), a1 = unpack2(T[1][j]), a2 = unpack2(T[2][j]), a3 = unpack2(T[3][j]);
      *reinterpret_cast<float4*>(base + static_cast<size_t>(2 * j) * ld) = make_float4(a0.x, a1.x, a2.x, a3.x);
      *reinterpret_cast<float4*>(base + static_cast<size_t>(2 * j + 1) * ld) = make_float4(a0.y, a1.y, a2.y, a3.y);
    }
  }
  // store gamma T without touching the registers
  __device__ __forceinline__ void store_scaled(float* base, size_t ld, float gam) const {
    const u64 g2 = pack2(gam, gam);
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const float2 a0 = unpack2(mul2(g2, T[0][j])), a1 = unpack2(mul2(g2, T[1][j]));
      const float2 a2 = unpack2(mul2(g2, T[2][j])), a3 = unpack2(mul2(g2, T[3][j]));
      *reinterpret_cast<float4*>(base + static_cast<size_t>(2 * j) * ld) = make_float4(a0.x, a1.x, a2.x, a3.x);
      *reinterpret_cast<float4*>(base + static_cast<size_t>(2 * j + 1) * ld) = make_float4(a0.y, a1.y, a2.y, a3.y);
    }
  }
  // T <- gamma T
  __device__ __forceinline__ void materialise(float gam) {
    const u64 g2 = pack2(gam, gam);
#pragma unroll
    for (int c = 0; c < kCols; ++c)
#pragma unroll
      for (int j = 0; j < NP; ++j) T[c][j] = mul2(g2, T[c][j]);
  }
  // pass B without the decay: T <- fmaf(k, ut_c, T); krows = k + row0 (16-byte aligned)
  __device__ __forceinline__ void update_lazy(const float* krows, float4 ut) {
    const u64 u2[kCols] = {pack2(ut.x, ut.x), pack2(ut.y, ut.y), pack2(ut.z, ut.z), pack2(ut.w, ut.w)};
    const ulonglong2* k4 = reinterpret_cast<const ulonglong2*>(krows);
#pragma unroll
    for (int j4 = 0; j4 < NP / 2; ++j4) {
      const ulonglong2 kk = k4[j4];
#pragma unroll
      for (int c = 0; c < kCols; ++c) {
        T[c][2 * j4 + 0] = fma2(kk.x, u2[c], T[c][2 * j4 + 0]);
        T[c][2 * j4 + 1] = fma2(kk.y, u2[c], T[c][2 * j4 + 1]);
      }
    }
  }
  // One node of the gated delta rule on the lazily decayed tile (state = gamma T): gam1 is the
  // node's gamma' = gamma g; returns the new gamma.  Below the floor the decay goes into the tile
  // first, then the update is the plain one.
  __device__ __forceinline__ float advance(const float* krows, float gam1, float4 u) {
    if (gam1 < kGammaFloor) {
      materialise(gam1);
      gam1 = 1.f;
    }
    const float r = __fdividef(1.f, gam1);
    update_lazy(krows, make_float4(u.x * r, u.y * r, u.z * r, u.w * r));
    return gam1;
  }
  // Partial dot products of the tile's columns with k and q over the thread's rows, as packed
  // (even rows, odd rows) sums: ak[c] . (1, 1) = sum_r T[r][c] k[r].
  __device__ __forceinline__ void dots(const float* krows, const float* qrows, u64 (&ak)[kCols],
                                       u64 (&aq)[kCols]) const {
    const ulonglong2* k4 = reinterpret_cast<const ulonglong2*>(krows);
    const ulonglong2* q4 = reinterpret_cast<const ulonglong2*>(qrows);
    const u64 zero2 = pack2(0.f, 0.f);
#pragma unroll
    for (int cc = 0; cc < kCols; ++cc) ak[cc] = aq[cc] = zero2;
#pragma unroll
    for (int j4 = 0; j4 < NP / 2; ++j4) {
      const ulonglong2 kk = k4[j4];
      const ulonglong2 qq = q4[j4];
#pragma unroll
      for (int cc = 0; cc < kCols; ++cc) {
        ak[cc] = fma2(T[cc][2 * j4 + 0], kk.x, ak[cc]);
        aq[cc] = fma2(T[cc][2 * j4 + 0], qq.x, aq[cc]);
        ak[cc] = fma2(T[cc][2 * j4 + 1], kk.y, ak[cc]);
        aq[cc] = fma2(T[cc][2 * j4 + 1], qq.y, aq[cc]);
      }
    }
  }
};

// One column of a [d_k][d_v] state, NR consecutive rows of it, as packed (row r, row r + 1) pairs:
// T[j] = (T[row0 + 2j][c], T[row0 + 2j + 1][c]).  The element operations are those of RegTile
// (same operands, same order), so a state folded in one layout equals, bit for bit, the state
// folded or stored in the other.  Pointers point at the thread's first element; `ld` is the row
// stride in floats.
template <int NR>
struct ColTile {
  static constexpr int NP = NR / 2;
  u64 T[NP];

  __device__ __forceinline__ void load(const float* base, size_t ld) {
#pragma unroll
    for (int j = 0; j < NP; ++j)
      T[j] = pack2(base[static_cast<size_t>(2 * j) * ld], base[static_cast<size_t>(2 * j + 1) * ld]);
  }
  __device__ __forceinline__ void store(float* base, size_t ld) const {
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const float2 a = unpack2(T[j]);
      base[static_cast<size_t>(2 * j) * ld] = a.x;
      base[static_cast<size_t>(2 * j + 1) * ld] = a.y;
    }
  }
  __device__ __forceinline__ void materialise(float gam) {
    const u64 g2 = pack2(gam, gam);
#pragma unroll
    for (int j = 0; j < NP; ++j) T[j] = mul2(g2, T[j]);
  }
  // T <- fmaf(k, ut, T); krows = k + row0 (16-byte aligned; shared or global memory)
  __device__ __forceinline__ void update_lazy(const float* krows, float ut) {
    const u64 u2 = pack2(ut, ut);
    const ulonglong2* k4 = reinterpret_cast<const ulonglong2*>(krows);
#pragma unroll
    for (int j4 = 0; j4 < NP / 2; ++j4) {
      const ulonglong2 kk = k4[j4];
      T[2 * j4 + 0] = fma2(kk.x, u2, T[2 * j4 + 0]);
      T[2 * j4 + 1] = fma2(kk.y, u2, T[2 * j4 + 1]);
    }
  }
  // RegTile::advance for one column
  __device__ __forceinline__ float advance(const float* krows, float gam1, float u) {
    if (gam1 < kGammaFloor) {
      materialise(gam1);
      gam1 = 1.f;
    }
    const float r = __fdividef(1.f, gam1);
    update_lazy(krows, u * r);
    return gam1;
  }
};

// The four column sums of packed (even, odd) partials.
__device__ __forceinline__ float4 fold_pairs(const u64 (&a)[kCols]) {
  const float2 a0 = unpack2(a[0]), a1 = unpack2(a[1]), a2 = unpack2(a[2]), a3 = unpack2(a[3]);
  return make_float4(a0.x + a0.y, a1.x + a1.y, a2.x + a2.y, a3.x + a3.y);
}

}  // namespace gdn
