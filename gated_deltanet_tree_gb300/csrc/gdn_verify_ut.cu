// Tree verify in the tree-masked UT form, with the deferred commit folded into
// the state load.
//
// SpecLA article, "状态驻留验证": besides the chain kernels, the method has a
// topology-masked version of the UT decomposition.  Written out: with T0 the
// committed state (after the fold), Gamma_t the product of the gates on the root
// path up to node t, rho_ts = Gamma_t / Gamma_s (the gates strictly below s on
// the path to t), G_ts = k_t . k_s and H_ts = q_t . k_s,
//   u_t = beta_t v_t - beta_t Gamma_t (T0^T k_t) - sum_{s ancestor of t} beta_t rho_ts G_ts u_s
//   o_t = Gamma_t (T0^T q_t) + H_tt u_t + sum_{s ancestor of t} rho_ts H_ts u_s
// which is the gated delta rule replayed along every root path.  The heavy part,
// T0^T k_t and T0^T q_t for all nodes, has no dependency between nodes: every
// node is one sweep over the register tile, and the sweeps of a batch of nodes
// share one cross-warp reduction.  The substitution is taken out of the d_v
// columns: with A_ts = beta_t rho_ts G_ts (s an ancestor of t), the unit lower
// triangular I + A keeps the tree's ancestor pattern, and so does its inverse
// M, one row per node from that node's root path; with C_ts = rho_ts H_ts,
// every (node, column) then needs only independent sums over the ancestors:
//   u_t = B_t + sum_s M_ts B_s,   B_s = beta_s v_s - beta_s Gamma_s (T0^T k_s)
//   o_t = Gamma_t (T0^T q_t) + H_tt u_t + sum_s C_ts u_s.
// Boundary states, when the caller asks for them, are replayed from T0 with the
// fold's own operations, so a later fold reproduces them bit for bit.
//
// Work unit: one CTA per (request, layer, v-head), all of d_v.  A thread owns
// RPT rows x 4 columns of the [d_k][d_v] tile (RegTile); the lanes of a warp run
// along the columns, so a warp-wide 16-byte load of the state covers whole rows.
#include "gdn_tile.cuh"

namespace gdn {
namespace {


// Shared-memory layout (4-byte words): staged rows, the B and Gamma R rows of every node, per-node
// tables, the ancestor-pair tables, a region used in turn by the fold, by the Gram's A table and by the
// partial sums, then int tables, the schedule record and the mbarrier.  The v rows become the u rows once
// every B row is formed.
template <int DK, int DV>
struct UtSmem {
  int n_max, warps;
  __host__ __device__ int pairs() const { return n_max * (n_max - 1) / 2; }
  __host__ __device__ int batch() const { return n_max > 32 ? 2 : 4; }                       // nodes per reduction
  __host__ __device__ int kq(int node) const { return node * 2 * DK; }                       // [n_max][2][DK]
  __host__ __device__ int v(int node) const { return n_max * 2 * DK + node * DV; }           // [n_max][DV] v, then u
  __host__ __device__ int bm(int node) const { return v(n_max) + node * DV; }                // [n_max][DV] B rows
  __host__ __device__ int rr(int node) const { return bm(n_max) + node * DV; }               // [n_max][DV] Gamma R rows
  __host__ __device__ int sc(int node) const { return rr(n_max) + 4 * node; }                // (g, beta, -, a)
  __host__ __device__ int gm(int node) const { return sc(n_max) + 4 * node; }                // (Gamma, beta Gamma, H_tt, -)
  __host__ __device__ int pm(int i) const { return gm(n_max) + 2 * i; }                      // [pairs] (M, row offset)
  __host__ __device__ int pc(int i) const { return pm(pairs()) + 2 * i; }                    // [pairs] (C, row offset)
  __host__ __device__ int region() const { return (pc(pairs()) + 3) & ~3; }
  __host__ __device__ int fk(int i) const { return region() + i * DK; }                      // fold: [kFoldChunk][DK]
  __host__ __device__ int fu(int i) const { return region() + kFoldChunk * DK + i * DV; }    // fold: [kFoldChunk][DV]
  __host__ __device__ int fg() const { return region() + kFoldChunk * (DK + DV); }           // fold: [kFoldChunk]
  __host__ __device__ int ra(int i) const { return region() + i; }                           // Gram: [pairs] A
  __host__ __device__ int ranc(int i) const { return region() + pairs() + i; }               // Gram: [pairs] ancestor
  __host__ __device__ int part(int w, int tb, int k) const {                                 // [warps][batch][2][DV]
    return region() + ((w * batch() + tb) * 2 + k) * DV;
  }
  __host__ __device__ int region_words() const {
    const int fold = kFoldChunk * (DK + DV) + kFoldChunk;
    const int gram = 2 * pairs();
    const int parts = warps * batch() * 2 * DV;
    const int m = fold > gram ? fold : gram;
    return ((m > parts ? m : parts) + 3) & ~3;
  }
  // int tables
  __host__ __device__ int coff(int t) const { return region() + region_words() + t; }        // [n_max + 1] pair offsets
  __host__ __device__ int path(int i) const { return coff(n_max + 1) + i; }                  // [n_max] scratch
  __host__ __device__ int flag() const { return path(n_max); }
  __host__ __device__ int rec0() const { return flag() + 1; }
  __host__ __device__ int bar0() const { return (rec0() + SchedLayout{n_max}.words() + 3) & ~3; }
  __host__ __device__ size_t bytes() const { return static_cast<size_t>(bar0() + 4) * 4; }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

template <int DK, int DV, int RPT>
__host__ __device__ constexpr int ut_threads() {
  return (DK / RPT) * (DV / kCols);
}

template <int DK, int DV, int RPT, typename InT>
__global__ void __launch_bounds__(ut_threads<DK, DV, RPT>(), 65536 / (ut_threads<DK, DV, RPT>() * 128))
    ut_verify_kernel(VerifyParams p) {
  constexpr int CG = DV / kCols;              // column groups
  constexpr int THREADS = ut_threads<DK, DV, RPT>();
  constexpr int W = THREADS / 32;             // warps
  constexpr int EPL = DK / 32;                // k / q elements per lane in the Gram dots
  static_assert(THREADS % 32 == 0 && 32 % CG == 0, "layout");
  static_assert(THREADS >= DV, "one thread per d_v column in the substitution");
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  int* si = reinterpret_cast<int*>(smem4);
  const UtSmem<DK, DV> L{p.n_max, W};

  int cta = blockIdx.x;
  const int h = cta % p.Hv;
  cta /= p.Hv;
  const int l = cta % p.layers;
  const int b = cta / p.layers;
  const int bl = b * p.layers + l;
  const int kh = h / p.R;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int cg = tid % CG, rg = tid / CG;
  const int c0 = cg * kCols, row0 = rg * RPT;

  RegTile<RPT> R;
  float* st = p.state + ((static_cast<size_t>(bl) * p.Hv + h) * DK + row0) * DV + c0;
  R.load(st, DV);

  if (__syncthreads_or(launch_aborted(p.err))) return;   // an earlier CTA gave up on a wait
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bar0());
  if (tid == 0) mbar_init(bar);
  const SchedLayout lay{p.n_max};
  const int32_t* rec = p.words + static_cast<size_t>(b) * lay.words();
  const int n = rec[0];
  if (n < 1 || n > p.n_max) {
    if (tid == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
    return;
  }
  int32_t* srec = si + L.rec0();
  for (int i = tid; i < lay.words(); i += THREADS) srec[i] = rec[i];
  const int Lp = p.fold ? p.pend_len[b] : 0;
  const int32_t* path = p.pend_path + static_cast<size_t>(b) * p.n_max;
  const size_t nrow0 = static_cast<size_t>(bl) * p.n_max;
  __syncthreads();   // barrier initialised, record staged

  // ---- asynchronous staging: k_hat, q_hat (k-head kh) and the v row of every node, the pending path's
  // k / u rows chunk by chunk; gates and betas by plain loads
  const InT* beta = static_cast<const InT*>(p.beta);
  const InT* logg = static_cast<const InT*>(p.log_g);
  uint32_t phase = 0;
  auto stage = [&](bool tree, int f0, int fn) -> bool {
    const uint32_t bytes = (tree ? static_cast<uint32_t>(n) * (2 * DK + DV) * 4 : 0u) +
                           static_cast<uint32_t>(fn) * (DK + DV) * 4;
    if (bytes == 0) return true;
    if (warp == 0) {
      if (lane == 0) mbar_expect(bar, bytes);
      __syncwarp();
      if (tree)
        for (int node = lane; node < n; node += 32) {
          const size_t row = nrow0 + node;
          bulk_g2s(sm + L.kq(node), p.k_in + (row * p.Hk + kh) * DK, DK * 4, bar);
          bulk_g2s(sm + L.kq(node) + DK, p.q_in + (row * p.Hk + kh) * DK, DK * 4, bar);
          bulk_g2s(sm + L.v(node), p.v_in + (row * p.Hv + h) * DV, DV * 4, bar);
        }
      for (int i = lane; i < fn; i += 32) {
        const size_t row = nrow0 + (path[f0 + i] & kPathNodeMask);
        bulk_g2s(sm + L.fk(i), p.pend_k + (row * p.Hk + kh) * DK, DK * 4, bar);
        bulk_g2s(sm + L.fu(i), p.pend_u + (row * p.Hv + h) * DV, DV * 4, bar);
      }
    }
    if (tree)
      for (int node = tid; node < n; node += THREADS) {
        const float a = load_in<InT>(logg, (nrow0 + node) * p.Hv + h);
        sm[L.sc(node) + 0] = expf(a);
        sm[L.sc(node) + 1] = load_in<InT>(beta, (nrow0 + node) * p.Hv + h);
        sm[L.sc(node) + 3] = a;
        p.a_out[(nrow0 + node) * p.Hv + h] = a;   // the bank's log-gate, exact
      }
    for (int i = tid; i < fn; i += THREADS)
      sm[L.fg() + i] = expf(p.pend_a[(nrow0 + (path[f0 + i] & kPathNodeMask)) * p.Hv + h]);
    // one verdict for the whole CTA (this barrier also makes the plain-loaded scalars visible)
    const bool ok = __syncthreads_and(mbar_wait(bar, phase));
    phase ^= 1;
    if (!ok) {
      if (tid == 0) device_error(p.err, GDN_DEVERR_TIMEOUT, b);
      mbar_wait(bar, phase ^ 1);   // let the copies land before the CTA exits
      return false;
    }
    return true;
  };

  // ---- deferred commit: the pending path folded into the tile, as in the chain kernel (same RegTile
  // operations, same materialisation points), then the committed state written once
  float gam = 1.f;
  if (!stage(true, 0, min(Lp, kFoldChunk))) return;
  for (int f0 = 0; f0 < Lp; f0 += kFoldChunk) {
    const int fn = min(kFoldChunk, Lp - f0);
    if (f0 > 0) {
      __syncthreads();   // previous chunk consumed
      if (!stage(false, f0, fn)) return;
    }
    for (int i = 0; i < fn; ++i) {
      if (path[f0 + i] & kPathHeadFlag) {
        R.materialise(gam);
        gam = 1.f;
      }
      gam = R.advance(sm + L.fk(i) + row0, gam * sm[L.fg() + i], *reinterpret_cast<const float4*>(sm + L.fu(i) + c0));
    }
  }
  if (Lp > 0) {
    R.materialise(gam);
    R.store(st, DV);
  }
  const int32_t* parent = srec + lay.parent();
  const int32_t* bslot = srec + lay.bslot();
  const int32_t* nflags = srec + lay.nflags();

  // ---- pair offsets (ancestor counts) and the schedule's validity, then the Gram coefficients
  if (tid == 0) {
    int ok = parent[0] == -1;
    int* coff = si + L.coff(0);
    int* depth = si + L.path(0);   // scratch until the boundary replay
    coff[0] = 0;
    depth[0] = 0;
    for (int t = 1; t < n; ++t) {
      const int pt = parent[t];
      ok &= (pt >= 0 && pt < t);
      depth[t] = (pt >= 0 && pt < t) ? depth[pt] + 1 : 0;
      coff[t] = coff[t - 1] + depth[t - 1];
    }
    coff[n] = coff[n - 1] + depth[n - 1];
    si[L.flag()] = ok;
  }
  __syncthreads();   // the fold's region is free again; offsets visible
  if (!si[L.flag()]) {
    if (tid == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
    return;
  }
  for (int t = warp; t < n; t += W) {   // one warp per node: lanes split d_k
    float kt[EPL], qt[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kt[e] = sm[L.kq(t) + lane * EPL + e];
      qt[e] = sm[L.kq(t) + DK + lane * EPL + e];
    }
    float hq = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) hq = fmaf(qt[e], kt[e], hq);
    hq = warp_sum(hq);
    const float gt = sm[L.sc(t) + 0], bt = sm[L.sc(t) + 1];
    float rho = gt;   // Gamma_t / Gamma_s for the ancestor s being visited
    int i = si[L.coff(t)];
    for (int s = parent[t]; s >= 0; s = parent[s], ++i) {
      float kk = 0.f, qk = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float ks = sm[L.kq(s) + lane * EPL + e];
        kk = fmaf(kt[e], ks, kk);
        qk = fmaf(qt[e], ks, qk);
      }
      kk = warp_sum(kk);
      qk = warp_sum(qk);
      if (lane == 0) {
        si[L.ranc(i)] = s;
        sm[L.ra(i)] = bt * rho * kk;
        *reinterpret_cast<float2*>(sm + L.pc(i)) = make_float2(rho * qk, __int_as_float(s * DV));
      }
      rho *= sm[L.sc(s) + 0];
    }
    if (lane == 0) *reinterpret_cast<float4*>(sm + L.gm(t)) = make_float4(rho, bt * rho, hq, 0.f);
  }
  __syncthreads();

  // ---- M = (I + A)^-1 over the ancestor pairs.  I + A keeps the ancestor pattern, so the rows of a node
  // and its ancestors form a closed lower-triangular block L (the root path a_0 .. a_d = t), and row t of M
  // is row d of L^-1: x_d = 1, x_j = -sum_{i>j} x_i A(a_i, a_j), a_j being the (i-j)-th ancestor of a_i.
  // Rows are independent: one thread per node.
  for (int t = tid; t < n; t += THREADS) {
    const int i0 = si[L.coff(t)], d = si[L.coff(t + 1)] - i0;
    // x_i for i < d sits in pm at position i0 + d - i - 1 (nearest ancestor first); x_d = 1
    for (int j = d - 1; j >= 0; --j) {
      const int aj = si[L.ranc(i0 + d - j - 1)];
      float acc = sm[L.ra(i0 + d - j - 1)];   // i = d: x_d A(t, a_j)
      for (int i = j + 1; i < d; ++i) {
        const int ai = si[L.ranc(i0 + d - i - 1)];
        acc = fmaf(sm[L.pm(i0 + d - i - 1)], sm[L.ra(si[L.coff(ai)] + i - j - 1)], acc);
      }
      *reinterpret_cast<float2*>(sm + L.pm(i0 + d - j - 1)) = make_float2(-acc, __int_as_float(aj * DV));
    }
  }
  __syncthreads();   // the region now takes the partial sums

  // ---- T0^T k_t and T0^T q_t for a batch of nodes, reduced over the warps; then u and o of the
  // batch by forward substitution, thread c owning d_v column c for every node
  const size_t node_stride = static_cast<size_t>(p.Hv) * DV;
  float* o_col = p.out_o + (nrow0 * p.Hv + h) * DV;
  float* u_col = p.u_out + (nrow0 * p.Hv + h) * DV;
  const int nbat = L.batch();
  for (int base = 0; base < n; base += nbat) {
    const int nb = min(nbat, n - base);
    for (int tb = 0; tb < nb; ++tb) {
      const int t = base + tb;
      u64 ak[kCols], aq[kCols];
      R.dots(sm + L.kq(t) + row0, sm + L.kq(t) + DK + row0, ak, aq);
      float4 sk = fold_pairs(ak), sq = fold_pairs(aq);
#pragma unroll
      for (int m = CG; m < 32; m <<= 1) {   // row groups inside the warp (none when CG = 32)
        sk.x += __shfl_xor_sync(0xffffffffu, sk.x, m);
        sk.y += __shfl_xor_sync(0xffffffffu, sk.y, m);
        sk.z += __shfl_xor_sync(0xffffffffu, sk.z, m);
        sk.w += __shfl_xor_sync(0xffffffffu, sk.w, m);
        sq.x += __shfl_xor_sync(0xffffffffu, sq.x, m);
        sq.y += __shfl_xor_sync(0xffffffffu, sq.y, m);
        sq.z += __shfl_xor_sync(0xffffffffu, sq.z, m);
        sq.w += __shfl_xor_sync(0xffffffffu, sq.w, m);
      }
      // lanes of the same column group now hold equal sums: all store (same value, same address)
      *reinterpret_cast<float4*>(sm + L.part(warp, tb, 0) + c0) = sk;
      *reinterpret_cast<float4*>(sm + L.part(warp, tb, 1) + c0) = sq;
    }
    __syncthreads();
    // four adjacent columns per job: (node of the batch, k or q, column group)
    for (int idx = tid; idx < nb * 2 * CG; idx += THREADS) {
      const int tb = idx / (2 * CG), k = (idx / CG) & 1, c = (idx % CG) * kCols;
      const int t = base + tb;
      const float* src = sm + L.part(0, tb, k) + c;
      const int wstride = L.part(1, 0, 0) - L.part(0, 0, 0);
      float4 acc = *reinterpret_cast<const float4*>(src);
#pragma unroll
      for (int w = 1; w < W; ++w) {
        const float4 x = *reinterpret_cast<const float4*>(src + w * wstride);
        acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
      }
      const float4 g4 = *reinterpret_cast<const float4*>(sm + L.gm(t));
      if (k == 0) {   // B_t = beta_t v_t - beta_t Gamma_t (T0^T k_t)
        const float bt = sm[L.sc(t) + 1];
        const float4 vv = *reinterpret_cast<const float4*>(sm + L.v(t) + c);
        *reinterpret_cast<float4*>(sm + L.bm(t) + c) =
            make_float4(fmaf(-g4.y, acc.x, bt * vv.x), fmaf(-g4.y, acc.y, bt * vv.y),
                        fmaf(-g4.y, acc.z, bt * vv.z), fmaf(-g4.y, acc.w, bt * vv.w));
      } else {        // Gamma_t (T0^T q_t)
        *reinterpret_cast<float4*>(sm + L.rr(t) + c) =
            make_float4(g4.x * acc.x, g4.x * acc.y, g4.x * acc.z, g4.x * acc.w);
      }
    }
    __syncthreads();   // partials consumed before the next batch writes them
  }

  // ---- u_t = B_t + sum_pairs M B_anc, then o_t = Gamma_t R_t + H_tt u_t + sum_pairs C u_anc: every
  // (node, group of four columns) on its own, adjacent threads on adjacent column groups
  const float* brow = sm + L.bm(0);
  for (int job = tid; job < n * CG; job += THREADS) {
    const int t = job / CG, c = (job % CG) * kCols;
    const int i0 = si[L.coff(t)], i1 = si[L.coff(t + 1)];
    float4 u = *reinterpret_cast<const float4*>(brow + t * DV + c);
    for (int i = i0; i < i1; ++i) {
      const float2 e = *reinterpret_cast<const float2*>(sm + L.pm(i));
      const float4 x = *reinterpret_cast<const float4*>(brow + __float_as_int(e.y) + c);
      u.x = fmaf(e.x, x.x, u.x); u.y = fmaf(e.x, x.y, u.y); u.z = fmaf(e.x, x.z, u.z); u.w = fmaf(e.x, x.w, u.w);
    }
    *reinterpret_cast<float4*>(sm + L.v(t) + c) = u;   // the v row is consumed: it becomes the u row
    *reinterpret_cast<float4*>(u_col + t * node_stride + c) = u;
  }
  __syncthreads();
  const float* urow = sm + L.v(0);
  for (int job = tid; job < n * CG; job += THREADS) {
    const int t = job / CG, c = (job % CG) * kCols;
    const int i0 = si[L.coff(t)], i1 = si[L.coff(t + 1)];
    const float htt = sm[L.gm(t) + 2];
    const float4 ut = *reinterpret_cast<const float4*>(urow + t * DV + c);
    float4 o = *reinterpret_cast<const float4*>(sm + L.rr(t) + c);
    o.x = fmaf(htt, ut.x, o.x); o.y = fmaf(htt, ut.y, o.y); o.z = fmaf(htt, ut.z, o.z); o.w = fmaf(htt, ut.w, o.w);
    for (int i = i0; i < i1; ++i) {
      const float2 e = *reinterpret_cast<const float2*>(sm + L.pc(i));
      const float4 x = *reinterpret_cast<const float4*>(urow + __float_as_int(e.y) + c);
      o.x = fmaf(e.x, x.x, o.x); o.y = fmaf(e.x, x.y, o.y); o.z = fmaf(e.x, x.z, o.z); o.w = fmaf(e.x, x.w, o.w);
    }
    *reinterpret_cast<float4*>(o_col + t * node_stride + c) = o;
  }

  // ---- boundary states on request: replayed from T0 with the fold's operations and materialisation
  // points, so the next fold of a path through the node reproduces them bit for bit
  if (!p.boundary_out) return;
  for (int node = 0; node < n; ++node) {
    const int slot = bslot[node];
    if (slot < 0 || slot >= p.nb_max) continue;
    if (tid == 0) {   // the root path of `node`, root first
      int m = 0;
      for (int v = node; v >= 0; v = parent[v]) ++m;
      si[L.flag()] = m;
      for (int v = node, i = m - 1; v >= 0; v = parent[v], --i) si[L.path(i)] = v;
    }
    __syncthreads();
    R.load(st, DV);   // T0: the committed state this CTA wrote, or the input state when nothing was folded
    const int m = si[L.flag()];
    float g = 1.f;
    for (int i = 0; i < m; ++i) {
      const int v = si[L.path(i)];
      if (i > 0 && (nflags[si[L.path(i - 1)]] & kNodeMaterialised)) {
        R.materialise(g);
        g = 1.f;
      }
      g = R.advance(sm + L.kq(v) + row0, g * sm[L.sc(v) + 0], *reinterpret_cast<const float4*>(sm + L.v(v) + c0));
    }
    R.materialise(g);
    R.store(p.boundary + ((static_cast<size_t>(bl) * p.nb_max + slot) * p.Hv + h) * DK * DV +
                static_cast<size_t>(row0) * DV + c0,
            DV);
    __syncthreads();   // the path table is rewritten for the next node
  }
}

template <int DK, int DV, int RPT, typename InT>
cudaError_t launch_ut_t(const VerifyParams& p, cudaStream_t s) {
  constexpr int threads = ut_threads<DK, DV, RPT>();
  const UtSmem<DK, DV> L{p.n_max, threads / 32};
  const size_t smem = L.bytes();
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  auto kern = ut_verify_kernel<DK, DV, RPT, InT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const size_t grid = static_cast<size_t>(p.B) * p.layers * p.Hv;
  kern<<<static_cast<unsigned>(grid), threads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int DK, int RPT, typename InT>
cudaError_t launch_ut_dv(const VerifyParams& p, cudaStream_t s) {
  switch (p.dv) {
    case 32: return launch_ut_t<DK, 32, RPT, InT>(p, s);
    case 64: return launch_ut_t<DK, 64, RPT, InT>(p, s);
    case 128: return launch_ut_t<DK, 128, RPT, InT>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename InT>
cudaError_t launch_ut_dtype(const VerifyParams& p, cudaStream_t s) {
  switch (p.dk) {
    case 32: return launch_ut_dv<32, 8, InT>(p, s);
    case 64: return launch_ut_dv<64, 16, InT>(p, s);
    case 128: return launch_ut_dv<128, 16, InT>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_verify_ut(const VerifyParams& p, cudaStream_t s) {
  if (p.in_dtype == GDN_DTYPE_BF16) return launch_ut_dtype<__nv_bfloat16>(p, s);
  return launch_ut_dtype<float>(p, s);
}

}  // namespace gdn
