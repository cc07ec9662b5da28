// Tree verify in the tree-masked UT form with the dense part on the tensor cores.
//
// SpecLA article, "状态驻留验证" (the topology-masked UT decomposition) and
// "延迟融合提交" (the pending path folded into the state tile at load).  With T0
// the committed state after the fold, Gamma_t the product of the gates on the
// root path up to node t, rho_ts = Gamma_t / Gamma_s, G_ts = k_t . k_s and
// H_ts = q_t . k_s,
//   u_t = beta_t v_t - beta_t Gamma_t (T0^T k_t) - sum_{s ancestor of t} beta_t rho_ts G_ts u_s
//   o_t = Gamma_t (T0^T q_t) + H_tt u_t + sum_{s ancestor of t} rho_ts H_ts u_s.
// Two products hold nearly all the arithmetic and have no dependency between
// nodes: T0^T [k_0 .. k_{n-1} q_0 .. q_{n-1}] (d_v x d_k times d_k x 2n per
// head) and the Gram rows [k; q] k^T.  Both run here as tcgen05 MMAs of kind
// tf32, split three ways (hi*hi + hi*lo + lo*hi) so that they carry fp32
// accuracy; what follows them (the ancestor-pattern inverse M = (I + A)^-1, the
// sums over ancestors) is the same as in the CUDA-core UT kernel.
//
// Work unit: one CTA per (request, layer, v-head), 256 threads, d_v = 128.
// Thread (warp w, lane) owns column c = 32 (w % 4) + lane of the [d_k][d_v]
// state and rows d_k/2 (w / 4) .. + d_k/2 (ColTile), which is exactly the
// tensor-memory lane and column range it may write with the 32x32b shape: the
// folded tile goes from registers into tensor memory as the A operand
// (lane = d_v column, column = d_k row) without crossing threads.
//
// Tensor memory, 256 columns per CTA:
//   [0, d_k)          A = T0^T, first its tf32 high part, then (after the MMAs
//                     reading it completed) its low part
//   [128, 128 + 2 NB) D = T0^T [k | q]: column t is T0^T k_t, column NB + t is T0^T q_t
//   [192, 192 + NG)   Gram: lane x < NB is k_x . k_s, lane NB + t is q_t . k_s (column s)
// with NB = n rounded up to 8 and NG = NB rounded up to 16.
//
// Shared-memory operand [k | q] (B of the first product, both operands of the
// Gram): rows 0..NB-1 the k_hat rows, NB..2NB-1 the q_hat rows (rows >= n are
// zero), K-major without swizzle, chunk-major: the 16-byte chunk kc of row r at
// kc * 2NB * 16 + r * 16, so the 8-row core matrices are contiguous (SBO = 128)
// and K-adjacent ones 2NB * 16 bytes apart (LBO).  The Gram's A operand reads
// this buffer as 128 rows; the rows past 2NB land in the following bytes, which
// the layout reserves, and only produce Gram lanes that are never read.
#include "gdn_tile.cuh"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

constexpr int kTcDv = 128;           // d_v: the MMA's M
constexpr int kTcThreads = 256;
constexpr uint32_t kTcCols = 256;    // tensor-memory columns per CTA
constexpr uint32_t kTcColD = 128;    // first column of T0^T [k | q]
constexpr uint32_t kTcColG = 192;    // first column of the Gram rows
constexpr int kTcMaxNodes = 32;      // 2 NB <= 64 and NG <= 32 columns

// Shared-memory layout (4-byte words).
template <int DK>
struct TcSmem {
  int n_max;
  static constexpr int DV = kTcDv;
  __host__ __device__ int nbm() const { return (n_max + 7) & ~7; }
  __host__ __device__ int ngm() const { return (nbm() + 15) & ~15; }
  __host__ __device__ int pairs() const { return n_max * (n_max - 1) / 2; }
  __host__ __device__ int bh() const { return 0; }                                  // [DK/4][2 NB][4] hi
  __host__ __device__ int bl() const { return 2 * nbm() * DK; }                     // [DK/4][2 NB][4] lo
  // + 512 words: the 128-row Gram operand reads up to 2 KB past the lo buffer's last chunk
  __host__ __device__ int v(int node) const { return bl() + 2 * nbm() * DK + 512 + node * DV; }   // v, then u
  __host__ __device__ int bm(int node) const { return v(n_max) + node * DV; }      // B rows
  __host__ __device__ int rr(int node) const { return bm(n_max) + node * DV; }     // Gamma R rows
  __host__ __device__ int sc(int node) const { return rr(n_max) + 4 * node; }      // (g, beta, -, a)
  __host__ __device__ int gm(int node) const { return sc(n_max) + 4 * node; }      // (Gamma, beta Gamma, H_tt, -)
  __host__ __device__ int pm(int i) const { return gm(n_max) + 2 * i; }            // [pairs] (M, row offset)
  __host__ __device__ int pc(int i) const { return pm(pairs()) + 2 * i; }          // [pairs] (C, row offset)
  __host__ __device__ int region() const { return (pc(pairs()) + 3) & ~3; }
  __host__ __device__ int fk(int i) const { return region() + i * DK; }            // fold: [kFoldChunk][DK]
  __host__ __device__ int fu(int i) const { return region() + kFoldChunk * DK + i * DV; }
  __host__ __device__ int fg() const { return region() + kFoldChunk * (DK + DV); }
  __host__ __device__ int gs() const { return ngm() + 4; }                         // Gram row stride
  __host__ __device__ int g2(int x) const { return region() + x * gs(); }          // [2 NB][gs]
  __host__ __device__ int ra(int i) const { return region() + 2 * nbm() * gs() + i; }
  __host__ __device__ int ranc(int i) const { return ra(pairs()) + i; }
  __host__ __device__ int region_words() const {
    const int fold = kFoldChunk * (DK + DV) + kFoldChunk;
    const int gram = 2 * nbm() * gs() + 2 * pairs();
    return ((fold > gram ? fold : gram) + 3) & ~3;
  }
  __host__ __device__ int coff(int t) const { return region() + region_words() + t; }   // [n_max + 1]
  __host__ __device__ int path(int i) const { return coff(n_max + 1) + i; }             // [n_max]
  __host__ __device__ int flag() const { return path(n_max); }
  __host__ __device__ int rec0() const { return flag() + 1; }
  __host__ __device__ int bar0() const { return (rec0() + SchedLayout{n_max}.words() + 3) & ~3; }   // 2 mbarriers
  __host__ __device__ int tslot() const { return bar0() + 4; }
  __host__ __device__ size_t bytes() const { return static_cast<size_t>(tslot() + 4) * 4; }
};

template <int DK, typename InT>
__global__ void __launch_bounds__(kTcThreads, 2) ut_tc_verify_kernel(VerifyParams p) {
  constexpr int DV = kTcDv;
  constexpr int THREADS = kTcThreads;
  constexpr int NR = DK / 2;                  // rows per thread
  constexpr int KC = DK / 4;                  // 16-byte chunks per row
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  int* si = reinterpret_cast<int*>(smem4);
  const TcSmem<DK> L{p.n_max};

  int cta = blockIdx.x;
  const int h = cta % p.Hv;
  cta /= p.Hv;
  const int l = cta % p.layers;
  const int b = cta / p.layers;
  const int bl = b * p.layers + l;
  const int kh = h / p.R;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int quarter = warp & 3, half = warp >> 2;
  const int c = 32 * quarter + lane;          // d_v column = tensor-memory lane
  const int row0 = half * NR;                 // first d_k row = first A column

  // ---- tensor memory first: warp 0 allocates and gives up the allocation permit at once (until a CTA
  // does, the SM holds back further CTAs of this kernel); the same warp frees the columns at the end,
  // after every thread's last access.  The body leaves only by CTA-uniform returns.
  uint32_t* tslot = reinterpret_cast<uint32_t*>(si + L.tslot());
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tslot, kTcCols);
    tmem_relinquish();
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tlane = tbase + (static_cast<uint32_t>(32 * quarter) << 16);

  [&]() {
    ColTile<NR> R;
    float* st = p.state + ((static_cast<size_t>(bl) * p.Hv + h) * DK + row0) * DV + c;
    R.load(st, DV);

    if (__syncthreads_or(launch_aborted(p.err))) return;   // an earlier CTA gave up on a wait
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bar0());   // [0] copies, [1] MMAs
    if (tid == 0) {
      mbar_init(bar);
      mbar_init(bar + 1);
    }
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
    const int NB = (n + 7) & ~7, NG = (NB + 15) & ~15;
    __syncthreads();   // barriers initialised, record staged

    // ---- asynchronous staging: the v row of every node, the pending path's k / u rows chunk by chunk;
    // gates and betas by plain loads
    const InT* beta = static_cast<const InT*>(p.beta);
    const InT* logg = static_cast<const InT*>(p.log_g);
    uint32_t phase = 0;
    auto issue = [&](bool tree, int f0, int fn) {
      const uint32_t bytes = (tree ? static_cast<uint32_t>(n) * DV * 4 : 0u) + static_cast<uint32_t>(fn) * (DK + DV) * 4;
      if (bytes > 0 && warp == 0) {
        if (lane == 0) mbar_expect(bar, bytes);
        __syncwarp();
        if (tree)
          for (int node = lane; node < n; node += 32)
            bulk_g2s(sm + L.v(node), p.v_in + ((nrow0 + node) * p.Hv + h) * DV, DV * 4, bar);
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
      return bytes > 0;
    };
    auto land = [&]() -> bool {   // one verdict for the whole CTA; also publishes the plain-loaded scalars
      const bool ok = __syncthreads_and(mbar_wait(bar, phase));
      phase ^= 1;
      if (!ok) {
        if (tid == 0) device_error(p.err, GDN_DEVERR_TIMEOUT, b);
        mbar_wait(bar, phase ^ 1);   // let the copies land before the CTA exits
      }
      return ok;
    };
    const bool staged = issue(true, 0, min(Lp, kFoldChunk));

    // ---- the [k | q] operand, split into tf32 high and low parts, from the k-head's rows (written by the
    // conv kernel); a warp covers 8 rows x 4 chunks, so its loads read whole 32-byte sectors and its
    // 16-byte shared stores fall on 8 distinct bank groups
    {
      const uint32_t lbo = static_cast<uint32_t>(2 * NB) * 16u;
      const int items = (2 * NB / 8) * (KC / 4);
      for (int it = warp; it < items; it += THREADS / 32) {
        const int r = (it / (KC / 4)) * 8 + (lane & 7);
        const int kc = (it % (KC / 4)) * 4 + (lane >> 3);
        const bool isq = r >= NB;
        const int node = isq ? r - NB : r;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (node < n) {
          const float* src = (isq ? p.q_in : p.k_in) + ((nrow0 + node) * p.Hk + kh) * DK + 4 * kc;
          x = *reinterpret_cast<const float4*>(src);
        }
        float4 hi, lo;
        hi.x = tf32_round(x.x); lo.x = tf32_round(x.x - hi.x);
        hi.y = tf32_round(x.y); lo.y = tf32_round(x.y - hi.y);
        hi.z = tf32_round(x.z); lo.z = tf32_round(x.z - hi.z);
        hi.w = tf32_round(x.w); lo.w = tf32_round(x.w - hi.w);
        const int off = kc * static_cast<int>(lbo / 4) + r * 4;
        *reinterpret_cast<float4*>(sm + L.bh() + off) = hi;
        *reinterpret_cast<float4*>(sm + L.bl() + off) = lo;
      }
      fence_proxy_async();   // visible to the tensor cores after the next barrier
    }

    // ---- deferred commit: the pending path folded into the tile with the chain kernel's operations and
    // materialisation points, then the committed state written once
    float gam = 1.f;
    if (staged && !land()) return;
    for (int f0 = 0; f0 < Lp; f0 += kFoldChunk) {
      const int fn = min(kFoldChunk, Lp - f0);
      if (f0 > 0) {
        __syncthreads();   // previous chunk consumed
        if (issue(false, f0, fn) && !land()) return;
      }
      for (int i = 0; i < fn; ++i) {
        if (path[f0 + i] & kPathHeadFlag) {
          R.materialise(gam);
          gam = 1.f;
        }
        gam = R.advance(sm + L.fk(i) + row0, gam * sm[L.fg() + i], sm[L.fu(i) + c]);
      }
    }
    if (Lp > 0) {
      R.materialise(gam);
      R.store(st, DV);
    }
    const int32_t* parent = srec + lay.parent();
    const int32_t* bslot = srec + lay.bslot();
    const int32_t* nflags = srec + lay.nflags();

    // ---- A = T0^T into tensor memory, tf32 high part
#pragma unroll
    for (int q = 0; q < NR / 16; ++q) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 e = unpack2(R.T[8 * q + j]);
        v[2 * j] = tf32_round(e.x);
        v[2 * j + 1] = tf32_round(e.y);
      }
      tmem_st16(tlane + static_cast<uint32_t>(row0 + 16 * q), v);
    }
    tmem_wait_st();

    // pair offsets (ancestor counts) and the schedule's validity
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
    tmem_fence_before();
    __syncthreads();   // A high part and the [k | q] operand in place; the fold's region is free again
    tmem_fence_after();
    if (!si[L.flag()]) {
      if (tid == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
      return;
    }

    const uint32_t lbo = static_cast<uint32_t>(2 * NB) * 16u;
    const uint32_t sbh = smem_addr(sm + L.bh()), sbl = smem_addr(sm + L.bl());
    const uint32_t id_d = umma_idesc_tf32(128, 2 * NB), id_g = umma_idesc_tf32(128, NG);
    if (tid == 0) {   // products with the high part of A, and the Gram rows
#pragma unroll 1
      for (int s = 0; s < DK / 8; ++s) {
        const uint64_t dh = umma_desc(sbh + 2u * s * lbo, lbo, 128u), dl = umma_desc(sbl + 2u * s * lbo, lbo, 128u);
        umma_tf32_ts(tbase + kTcColD, tbase + 8u * s, dh, id_d, s > 0);
        umma_tf32_ts(tbase + kTcColD, tbase + 8u * s, dl, id_d, 1);
        umma_tf32_ss(tbase + kTcColG, dh, dh, id_g, s > 0);
        umma_tf32_ss(tbase + kTcColG, dh, dl, id_g, 1);
        umma_tf32_ss(tbase + kTcColG, dl, dh, id_g, 1);
      }
      umma_commit(bar + 1);
    }
    uint32_t mphase = 0;
    auto mma_done = [&]() -> bool {
      const bool ok = __syncthreads_and(mbar_wait(bar + 1, mphase));
      mphase ^= 1;
      if (!ok) {
        if (tid == 0) device_error(p.err, GDN_DEVERR_TIMEOUT, b);
        mbar_wait(bar + 1, mphase ^ 1);   // let the MMAs finish before the columns are freed
      }
      tmem_fence_after();
      return ok;
    };
    if (!mma_done()) return;

    // ---- A low part over the high part (its readers completed), then its product with the high [k | q]
#pragma unroll
    for (int q = 0; q < NR / 16; ++q) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 e = unpack2(R.T[8 * q + j]);
        v[2 * j] = tf32_round(e.x - tf32_round(e.x));
        v[2 * j + 1] = tf32_round(e.y - tf32_round(e.y));
      }
      tmem_st16(tlane + static_cast<uint32_t>(row0 + 16 * q), v);
    }
    tmem_wait_st();
    // the Gram rows are complete: lanes < 2 NB to shared memory (warp halves split the columns)
    if (32 * quarter < 2 * NB) {
      for (int cc = half; cc < NG / 16; cc += 2) {
        float v[16];
        tmem_ld16(tlane + kTcColG + 16u * cc, v);
        tmem_wait_ld();
        if (c < 2 * NB) {
          float* dst = sm + L.g2(c) + 16 * cc;
#pragma unroll
          for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      }
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    if (tid == 0) {
#pragma unroll 1
      for (int s = 0; s < DK / 8; ++s)
        umma_tf32_ts(tbase + kTcColD, tbase + 8u * s, umma_desc(sbh + 2u * s * lbo, lbo, 128u), id_d, 1);
      umma_commit(bar + 1);
    }

    // ---- meanwhile: the ancestor-pair coefficients from the Gram rows, one thread per node
    for (int t = tid; t < n; t += THREADS) {
      const float gt = sm[L.sc(t) + 0], bt = sm[L.sc(t) + 1];
      const float* gk = sm + L.g2(t);
      const float* gq = sm + L.g2(NB + t);
      float rho = gt;   // Gamma_t / Gamma_s for the ancestor s being visited
      int i = si[L.coff(t)];
      for (int s = parent[t]; s >= 0; s = parent[s], ++i) {
        si[L.ranc(i)] = s;
        sm[L.ra(i)] = bt * rho * gk[s];
        *reinterpret_cast<float2*>(sm + L.pc(i)) = make_float2(rho * gq[s], __int_as_float(s * DV));
        rho *= sm[L.sc(s) + 0];
      }
      *reinterpret_cast<float4*>(sm + L.gm(t)) = make_float4(rho, bt * rho, gq[t], 0.f);
    }
    __syncthreads();
    // M = (I + A)^-1 over the ancestor pairs: row t of M is the last row of the inverse of the block on
    // t's root path (x_d = 1, x_j = -sum_{i>j} x_i A(a_i, a_j)); rows are independent
    for (int t = tid; t < n; t += THREADS) {
      const int i0 = si[L.coff(t)], d = si[L.coff(t + 1)] - i0;
      for (int j = d - 1; j >= 0; --j) {
        const int aj = si[L.ranc(i0 + d - j - 1)];
        float acc = sm[L.ra(i0 + d - j - 1)];
        for (int i = j + 1; i < d; ++i) {
          const int ai = si[L.ranc(i0 + d - i - 1)];
          acc = fmaf(sm[L.pm(i0 + d - i - 1)], sm[L.ra(si[L.coff(ai)] + i - j - 1)], acc);
        }
        *reinterpret_cast<float2*>(sm + L.pm(i0 + d - j - 1)) = make_float2(-acc, __int_as_float(aj * DV));
      }
    }
    if (!mma_done()) return;   // (its barrier also publishes M)

    // ---- B_t = beta_t v_t - beta_t Gamma_t (T0^T k_t) and Gamma_t (T0^T q_t): thread (column c, half)
    // takes the node columns of its half
    {
      const int nbh = NB / 2, t0 = half * nbh;
      for (int g = 0; g < nbh; g += 4) {
        if (t0 + g >= n) break;   // warp-uniform
        float dk4[4], dq4[4];
        tmem_ld4(tlane + kTcColD + static_cast<uint32_t>(t0 + g), dk4);
        tmem_ld4(tlane + kTcColD + static_cast<uint32_t>(NB + t0 + g), dq4);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = t0 + g + j;
          if (t < n) {
            const float4 g4 = *reinterpret_cast<const float4*>(sm + L.gm(t));
            const float bt = sm[L.sc(t) + 1];
            sm[L.bm(t) + c] = fmaf(-g4.y, dk4[j], bt * sm[L.v(t) + c]);
            sm[L.rr(t) + c] = g4.x * dq4[j];
          }
        }
      }
    }
    tmem_fence_before();
    __syncthreads();

    // ---- u_t = B_t + sum_pairs M B_anc, then o_t = Gamma_t R_t + H_tt u_t + sum_pairs C u_anc: every
    // (node, group of four columns) on its own, adjacent threads on adjacent column groups
    constexpr int CG = DV / kCols;
    const size_t node_stride = static_cast<size_t>(p.Hv) * DV;
    float* o_col = p.out_o + (nrow0 * p.Hv + h) * DV;
    float* u_col = p.u_out + (nrow0 * p.Hv + h) * DV;
    const float* brow = sm + L.bm(0);
    for (int job = tid; job < n * CG; job += THREADS) {
      const int t = job / CG, cc = (job % CG) * kCols;
      const int i0 = si[L.coff(t)], i1 = si[L.coff(t + 1)];
      float4 u = *reinterpret_cast<const float4*>(brow + t * DV + cc);
      for (int i = i0; i < i1; ++i) {
        const float2 e = *reinterpret_cast<const float2*>(sm + L.pm(i));
        const float4 x = *reinterpret_cast<const float4*>(brow + __float_as_int(e.y) + cc);
        u.x = fmaf(e.x, x.x, u.x); u.y = fmaf(e.x, x.y, u.y); u.z = fmaf(e.x, x.z, u.z); u.w = fmaf(e.x, x.w, u.w);
      }
      *reinterpret_cast<float4*>(sm + L.v(t) + cc) = u;   // the v row is consumed: it becomes the u row
      *reinterpret_cast<float4*>(u_col + t * node_stride + cc) = u;
    }
    __syncthreads();
    const float* urow = sm + L.v(0);
    for (int job = tid; job < n * CG; job += THREADS) {
      const int t = job / CG, cc = (job % CG) * kCols;
      const int i0 = si[L.coff(t)], i1 = si[L.coff(t + 1)];
      const float htt = sm[L.gm(t) + 2];
      const float4 ut = *reinterpret_cast<const float4*>(urow + t * DV + cc);
      float4 o = *reinterpret_cast<const float4*>(sm + L.rr(t) + cc);
      o.x = fmaf(htt, ut.x, o.x); o.y = fmaf(htt, ut.y, o.y); o.z = fmaf(htt, ut.z, o.z); o.w = fmaf(htt, ut.w, o.w);
      for (int i = i0; i < i1; ++i) {
        const float2 e = *reinterpret_cast<const float2*>(sm + L.pc(i));
        const float4 x = *reinterpret_cast<const float4*>(urow + __float_as_int(e.y) + cc);
        o.x = fmaf(e.x, x.x, o.x); o.y = fmaf(e.x, x.y, o.y); o.z = fmaf(e.x, x.z, o.z); o.w = fmaf(e.x, x.w, o.w);
      }
      *reinterpret_cast<float4*>(o_col + t * node_stride + cc) = o;
    }

    // ---- boundary states on request: replayed from T0 with the fold's operations and materialisation
    // points (k rows from the bank, exact), so the next fold of a path through the node reproduces them
    // bit for bit
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
        g = R.advance(p.k_in + ((nrow0 + v) * p.Hk + kh) * DK + row0, g * sm[L.sc(v) + 0], sm[L.v(v) + c]);
      }
      R.materialise(g);
      R.store(p.boundary + ((static_cast<size_t>(bl) * p.nb_max + slot) * p.Hv + h) * DK * DV +
                  static_cast<size_t>(row0) * DV + c,
              DV);
      __syncthreads();   // the path table is rewritten for the next node
    }
  }();

  tmem_fence_before();
  __syncthreads();   // every thread's last tensor-memory access is behind this barrier
  if (warp == 0) {
    tmem_fence_after();
    tmem_dealloc(tbase, kTcCols);
  }
}

template <int DK, typename InT>
cudaError_t launch_tc_t(const VerifyParams& p, cudaStream_t s) {
  const TcSmem<DK> L{p.n_max};
  const size_t smem = L.bytes();
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  auto kern = ut_tc_verify_kernel<DK, InT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const size_t grid = static_cast<size_t>(p.B) * p.layers * p.Hv;
  kern<<<static_cast<unsigned>(grid), kTcThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <typename InT>
cudaError_t launch_tc_dtype(const VerifyParams& p, cudaStream_t s) {
  switch (p.dk) {
    case 32: return launch_tc_t<32, InT>(p, s);
    case 64: return launch_tc_t<64, InT>(p, s);
    case 128: return launch_tc_t<128, InT>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool verify_tc_supported(int dk, int dv, int n_max) {
  return dv == kTcDv && (dk == 32 || dk == 64 || dk == 128) && n_max >= 1 && n_max <= kTcMaxNodes;
}

cudaError_t launch_verify_tc(const VerifyParams& p, cudaStream_t s) {
  if (!verify_tc_supported(p.dk, p.dv, p.n_max)) return cudaErrorInvalidValue;
  if (p.in_dtype == GDN_DTYPE_BF16) return launch_tc_dtype<__nv_bfloat16>(p, s);
  return launch_tc_dtype<float>(p, s);
}

}  // namespace gdn
