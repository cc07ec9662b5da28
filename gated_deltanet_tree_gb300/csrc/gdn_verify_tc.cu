// Tree verify in the tree-masked UT form with the dense part on the tensor cores.
//
// SpecLA article, "状态驻留验证" (the topology-masked UT decomposition) and
// "延迟融合提交" (the pending path folded into the state tile at load).  With T0
// the committed state after the fold, Gamma_t the product of the gates on the
// root path up to node t, rho_ts = Gamma_t / Gamma_s, G_ts = k_t . k_s and
// H_ts = q_t . k_s,
//   u_t = beta_t v_t - beta_t Gamma_t (T0^T k_t) - sum_{s ancestor of t} beta_t rho_ts G_ts u_s
//   o_t = Gamma_t (T0^T q_t) + H_tt u_t + sum_{s ancestor of t} rho_ts H_ts u_s.
// Nearly all the arithmetic is one product with no dependency between nodes,
// T0^T [k_0 .. k_{n-1} q_0 .. q_{n-1}] (d_v x d_k times d_k x 2n per head).  It
// runs here as tcgen05 MMAs of kind tf32 split three ways, A_hi B_hi + A_hi B_lo
// + A_lo B_hi, so that it carries fp32 accuracy; so do the Gram rows [k; q] k^T,
// issued before the fold and read out of tensor memory after it.  The tree's
// tables (depths, pair offsets, ancestors, rho and Gamma by a product scan
// across lanes, the pair coefficients, the rows of M = (I + A)^-1) are built by
// warps or threads in parallel while the tensor cores run; u and o are the
// sums over ancestors of the CUDA-core UT kernel.
//
// Work unit: one CTA per (request, layer, v-head), 256 threads, d_v = 128.
// Thread (warp w, lane) owns column c = 32 (w % 4) + lane of the [d_k][d_v]
// state and rows d_k/2 (w / 4) .. + d_k/2 (ColTile), which is exactly the
// tensor-memory lane and column range it may write with the 32x32b shape: the
// folded tile goes from registers into tensor memory as the A operand
// (lane = d_v column, column = d_k row) without crossing threads.
//
// Tensor memory, 256 columns per CTA:
//   [0, d_k)           A = T0^T: first its tf32 high part, then, once the MMAs
//                      reading it completed, its low part
//   [128, 128 + 4 NB)  D: columns t, NB + t, 2 NB + t, 3 NB + t hold T0^T times
//                      the high k_t, high q_t, low k_t and low q_t; before the
//                      first product, the Gram rows
// with NB = n rounded up to 8.  The first product (A high, N = 4 NB) fills all
// four blocks; the second (A low times the high rows, N = 2 NB) accumulates into
// the first two, so T0^T k_t = D[t] + D[2 NB + t] and T0^T q_t = D[NB + t] +
// D[3 NB + t].  The Gram rows are the operand's first 128 rows (k_hi, q_hi,
// k_lo, q_lo, then rows never read out) times the high k rows and times the low
// k rows (N = NB rounded up to 16 each), so G_ts and H_ts are each a sum of
// three lanes.
//
// Shared-memory operand: rows k_hi | q_hi | k_lo | q_lo (NB rows each, rows of
// nodes >= n zero), K-major without swizzle, chunk-major: the 16-byte chunk kc
// of row r at kc * 4 NB * 16 + r * 16, so the 8-row core matrices are contiguous
// (SBO = 128) and K-adjacent ones 4 NB * 16 bytes apart (LBO).
//
// Every CTA also prefetches into L2 the state tile and node rows of the CTA one
// wave of resident CTAs ahead, which starts about when this one ends: its loads
// then wait on L2 rather than on HBM queues.
#include "gdn_tile.cuh"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

constexpr int kTcDv = 128;           // d_v: the MMA's M
constexpr int kTcThreads = 256;
constexpr uint32_t kTcCols = 256;    // tensor-memory columns per CTA
constexpr uint32_t kTcColD = 128;    // first column of T0^T [k_hi | q_hi | k_lo | q_lo]
constexpr int kTcMaxNodes = 32;      // 4 NB <= 128 columns

// Shared-memory layout (4-byte words).
template <int DK>
struct TcSmem {
  int n_max;
  static constexpr int DV = kTcDv;
  __host__ __device__ int nbm() const { return (n_max + 7) & ~7; }
  __host__ __device__ int ngm() const { return (nbm() + 15) & ~15; }
  __host__ __device__ int pairs() const { return n_max * (n_max - 1) / 2; }
  // [DK/4 chunks][4 NB rows][4]: rows k_hi | q_hi | k_lo | q_lo; + 512 words: the 128-row Gram operand
  // reads up to 2 KB past the last chunk's rows
  __host__ __device__ int bq() const { return 0; }
  __host__ __device__ int v(int node) const { return 4 * nbm() * DK + 512 + node * DV; }   // v, then u
  __host__ __device__ int bm(int node) const { return v(n_max) + node * DV; }      // B rows
  __host__ __device__ int rr(int node) const { return bm(n_max) + node * DV; }     // Gamma R rows
  // before the B and Gamma R rows exist, the same area holds first the k and q rows as staged
  // ([n_max][2][DK]), then the Gram rows read out of tensor memory ([4 NB][gs] and [2 NB][gs])
  __host__ __device__ int gs() const { return ngm() + 4; }                         // Gram row stride
  __host__ __device__ int kq(int node) const { return bm(0) + node * 2 * DK; }
  __host__ __device__ int g1(int x) const { return bm(0) + x * gs(); }
  __host__ __device__ int g2(int x) const { return bm(0) + (4 * nbm() + x) * gs(); }
  __host__ __device__ int rows_words() const {
    const int a = 2 * n_max * DV, g = 6 * nbm() * gs();
    return ((a > g ? a : g) + 3) & ~3;
  }
  __host__ __device__ int sc(int node) const { return bm(0) + rows_words() + 4 * node; }   // (g, beta, -, a)
  __host__ __device__ int gm(int node) const { return sc(n_max) + 4 * node; }      // (Gamma, beta Gamma, H_tt, -)
  __host__ __device__ int pm(int i) const { return gm(n_max) + 2 * i; }            // [pairs] (M, row offset)
  // both pair tables start 16-byte aligned, so an even pair index reads two entries at once
  __host__ __device__ int pc(int i) const { return ((pm(pairs()) + 3) & ~3) + 2 * i; }   // [pairs] (C, row offset)
  __host__ __device__ int ra(int i) const { return pc(pairs()) + i; }              // [pairs] rho, then A
  __host__ __device__ int ranc(int i) const { return ra(pairs()) + i; }            // [pairs] ancestor
  __host__ __device__ int ptn(int i) const { return ranc(pairs()) + i; }           // [pairs] node
  __host__ __device__ int region() const { return (ptn(pairs()) + 3) & ~3; }
  __host__ __device__ int fk(int i) const { return region() + i * DK; }            // fold: [kFoldChunk][DK]
  __host__ __device__ int fu(int i) const { return region() + kFoldChunk * DK + i * DV; }
  __host__ __device__ int fg() const { return region() + kFoldChunk * (DK + DV); }
  __host__ __device__ int region_words() const { return (kFoldChunk * (DK + DV) + kFoldChunk + 3) & ~3; }
  __host__ __device__ int coff(int t) const { return region() + region_words() + t; }   // [n_max + 1]
  __host__ __device__ int dep(int t) const { return coff(n_max + 1) + t; }              // [n_max] depth
  __host__ __device__ int ppath(int i) const { return dep(n_max) + i; }                 // [n_max] pending path
  __host__ __device__ int path(int i) const { return ppath(n_max) + i; }                // [n_max] scratch
  __host__ __device__ int flag() const { return path(n_max); }                          // [4] flags and counts
  __host__ __device__ int rec0() const { return flag() + 4; }
  __host__ __device__ int bar0() const { return (rec0() + SchedLayout{n_max}.words() + 3) & ~3; }   // 5 mbarriers
  __host__ __device__ int tslot() const { return bar0() + 10; }
  __host__ __device__ size_t bytes() const { return static_cast<size_t>(tslot() + 2) * 4; }
};

template <int DK, typename InT>
__global__ void __launch_bounds__(kTcThreads, 2) ut_tc_verify_kernel(VerifyParams p) {
  constexpr int DV = kTcDv;
  constexpr int THREADS = kTcThreads;
  constexpr int W = THREADS / 32;
  constexpr int NR = DK / 2;                  // rows per thread
  constexpr int KC = DK / 4;                  // 16-byte chunks per row
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  int* si = reinterpret_cast<int*>(smem4);
  const TcSmem<DK> L{p.n_max};

  auto decode = [&](int cta, int& bb, int& ll, int& hh) {
    hh = cta % p.Hv;
    cta /= p.Hv;
    ll = cta % p.layers;
    bb = cta / p.layers;
  };
  int b, l, h;
  decode(blockIdx.x, b, l, h);
  const int bl = b * p.layers + l;
  const int kh = h / p.R;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int quarter = warp & 3, half = warp >> 2;
  const int c = 32 * quarter + lane;          // d_v column = tensor-memory lane
  const int row0 = half * NR;                 // first d_k row = first A column
  const size_t nrow0 = static_cast<size_t>(bl) * p.n_max;
  const int n_max = p.n_max;
  // mbarriers: [0] node rows, [1] pending rows (one phase per chunk), [2] Gram, [3] high product,
  // [4] low product
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bar0());

  // ---- tensor memory first: warp 0 allocates and gives up the allocation permit at once (until a CTA
  // does, the SM holds back further CTAs of this kernel); the same warp frees the columns at the end,
  // after every thread's last access.  The body leaves only by CTA-uniform returns.
  uint32_t* tslot = reinterpret_cast<uint32_t*>(si + L.tslot());
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tslot, kTcCols);
    tmem_relinquish();
  }

  // ---- every input transfer goes out before the first barrier, so their latencies overlap:
  //   warp 0: the k, q and v rows of all n_max node slots (rows past the tree are read, never used);
  //   warp 1: the pending path and length, then the first chunk of the pending rows;
  //   warp 2: the schedule record and the launch's error word; warp 3: gates and betas;
  //   every thread: its column of the state tile.
  const InT* beta = static_cast<const InT*>(p.beta);
  const InT* logg = static_cast<const InT*>(p.log_g);
  const SchedLayout lay{n_max};
  int32_t* srec = si + L.rec0();
  int32_t* spath = si + L.ppath(0);
  if (warp == 0) {
    if (lane == 0) {
      mbar_init(bar);
      mbar_expect(bar, static_cast<uint32_t>(n_max) * (2 * DK + DV) * 4);
    }
    __syncwarp();
    for (int node = lane; node < n_max; node += 32) {
      const size_t row = nrow0 + node;
      bulk_g2s(sm + L.kq(node), p.k_in + (row * p.Hk + kh) * DK, DK * 4, bar);
      bulk_g2s(sm + L.kq(node) + DK, p.q_in + (row * p.Hk + kh) * DK, DK * 4, bar);
      bulk_g2s(sm + L.v(node), p.v_in + (row * p.Hv + h) * DV, DV * 4, bar);
    }
  } else if (warp == 1) {
    const int lp = p.fold ? p.pend_len[b] : 0;
    const bool lp_ok = lp >= 0 && lp <= n_max;
    const int fn = lp_ok ? min(lp, kFoldChunk) : 0;
    for (int i = lane; i < n_max; i += 32) spath[i] = p.fold ? p.pend_path[static_cast<size_t>(b) * n_max + i] : 0;
    if (lane == 0) {
      si[L.flag() + 1] = lp_ok ? lp : -1;
      mbar_init(bar + 1);
      if (fn > 0) mbar_expect(bar + 1, static_cast<uint32_t>(fn) * (DK + DV) * 4);
    }
    __syncwarp();   // path entries and the barrier visible to the warp
    for (int i = lane; i < fn; i += 32) {
      const size_t row = nrow0 + (spath[i] & kPathNodeMask);
      bulk_g2s(sm + L.fk(i), p.pend_k + (row * p.Hk + kh) * DK, DK * 4, bar + 1);
      bulk_g2s(sm + L.fu(i), p.pend_u + (row * p.Hv + h) * DV, DV * 4, bar + 1);
      sm[L.fg() + i] = expf(p.pend_a[row * p.Hv + h]);
    }
  } else if (warp == 2) {
    const int32_t* rec = p.words + static_cast<size_t>(b) * lay.words();
    for (int i = lane; i < lay.words(); i += 32) srec[i] = rec[i];
    if (lane == 0) {
      si[L.flag() + 2] = launch_aborted(p.err);   // an earlier CTA gave up on a wait
      mbar_init(bar + 2);
      mbar_init(bar + 3);
      mbar_init(bar + 4);
    }
  } else if (warp == 3) {
    for (int node = lane; node < n_max; node += 32) {
      const float a = load_in<InT>(logg, (nrow0 + node) * p.Hv + h);
      sm[L.sc(node) + 0] = expf(a);
      sm[L.sc(node) + 1] = load_in<InT>(beta, (nrow0 + node) * p.Hv + h);
      sm[L.sc(node) + 3] = a;
    }
  }
  ColTile<NR> R;
  float* st = p.state + ((static_cast<size_t>(bl) * p.Hv + h) * DK + row0) * DV + c;
  R.load(st, DV);
  // ---- the CTA one wave ahead (it starts about when this one ends): its state tile and node rows go
  // into L2 now, so its loads find them there
  if (warp == W - 1 && p.prefetch_ahead > 0 && blockIdx.x + p.prefetch_ahead < gridDim.x) {
    int b2, l2, h2;
    decode(blockIdx.x + p.prefetch_ahead, b2, l2, h2);
    const size_t bl2 = static_cast<size_t>(b2) * p.layers + l2;
    const int kh2 = h2 / p.R;
    if (lane < 4) prefetch_l2(p.state + (bl2 * p.Hv + h2) * DK * DV + lane * (DK * DV / 4), DK * DV);
    for (int node = lane; node < n_max; node += 32) {
      const size_t row = bl2 * n_max + node;
      prefetch_l2(p.v_in + (row * p.Hv + h2) * DV, DV * 4);
      if (h2 % p.R == 0) {   // the k-head's rows, once per group of v-heads
        prefetch_l2(p.k_in + (row * p.Hk + kh2) * DK, DK * 4);
        prefetch_l2(p.q_in + (row * p.Hk + kh2) * DK, DK * 4);
      }
    }
  }
  tmem_fence_before();
  __syncthreads();   // barriers initialised, small inputs staged, tensor memory allocated
  tmem_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tlane = tbase + (static_cast<uint32_t>(32 * quarter) << 16);

  [&]() {
    // the copies of warps 0 and 1 are in flight: every exit below waits for them first
    const int n = srec[0];
    const int Lp = si[L.flag() + 1];
    const bool fold_rows = Lp > 0;
    auto drain = [&]() {
      mbar_wait(bar, 0);
      if (fold_rows) mbar_wait(bar + 1, 0);
    };
    if (si[L.flag() + 2]) {
      drain();
      return;
    }
    if (n < 1 || n > n_max || Lp < 0) {
      if (tid == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
      drain();
      return;
    }
    const int NB = (n + 7) & ~7, NG = (NB + 15) & ~15;
    for (int node = tid; node < n; node += THREADS)
      p.a_out[(nrow0 + node) * p.Hv + h] = sm[L.sc(node) + 3];   // the bank's log-gate, exact
    if (!__syncthreads_and(mbar_wait(bar, 0))) {
      if (tid == 0) device_error(p.err, GDN_DEVERR_TIMEOUT, b);
      drain();
      return;
    }

    // ---- the [k | q] operand from the staged rows, split into tf32 high (rows r) and low (rows 2 NB + r)
    // parts; a warp item is 8 rows x 4 chunks whose reads (8 chunk slots) and writes (8 row slots) each
    // fall on distinct banks
    {
      constexpr int kblocks = KC / 8 > 0 ? KC / 8 : 1;
      const int items = (2 * NB / 8) * kblocks * 2;
      const int lbo4 = 4 * NB * 4;   // chunk stride in words
      const int e = lane & 7, q = lane >> 3;
      for (int it = warp; it < items; it += W) {
        const int rb = it / (2 * kblocks), kb = (it / 2) % kblocks, qq = it & 1;
        const int r = 8 * rb + e;
        const int kc = 8 * kb + ((e + q + 4 * qq) & 7);
        if (kc < KC) {
          const bool isq = r >= NB;
          const int node = isq ? r - NB : r;
          float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
          if (node < n) x = *reinterpret_cast<const float4*>(sm + L.kq(node) + (isq ? DK : 0) + 4 * kc);
          float4 hi, lo;
          hi.x = tf32_hi(x.x); lo.x = tf32_lo(x.x);
          hi.y = tf32_hi(x.y); lo.y = tf32_lo(x.y);
          hi.z = tf32_hi(x.z); lo.z = tf32_lo(x.z);
          hi.w = tf32_hi(x.w); lo.w = tf32_lo(x.w);
          *reinterpret_cast<float4*>(sm + L.bq() + kc * lbo4 + 4 * r) = hi;
          *reinterpret_cast<float4*>(sm + L.bq() + kc * lbo4 + 4 * (2 * NB + r)) = lo;
        }
      }
      fence_proxy_async();   // visible to the tensor cores after the next barrier
    }
    const int32_t* parent = srec + lay.parent();
    const int32_t* bslot = srec + lay.bslot();
    const int32_t* nflags = srec + lay.nflags();
    // depths, pair offsets (ancestor counts) and the schedule's validity: one lane per node (n <= 32)
    if (warp == W - 1) {
      const int t = lane;
      bool ok = true;
      if (t < n) ok = t == 0 ? parent[0] == -1 : (parent[t] >= 0 && parent[t] < t);
      ok = __all_sync(FULL, ok);
      int d = 0;
      if (ok && t < n)
        for (int v = t; v > 0; v = parent[v]) ++d;
      int incl = d;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const int y = __shfl_up_sync(FULL, incl, m);
        if (lane >= m) incl += y;
      }
      if (t < n) {
        si[L.dep(t)] = d;
        si[L.coff(t)] = incl - d;
      }
      if (t == n - 1) si[L.coff(n)] = incl;
      if (lane == 0) si[L.flag()] = ok;
    }
    __syncthreads();   // [k | q] operand in place, offsets visible
    if (!si[L.flag()]) {
      if (tid == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
      if (fold_rows) mbar_wait(bar + 1, 0);
      return;
    }
    const uint32_t lbo = static_cast<uint32_t>(4 * NB) * 16u;
    const uint32_t sbq = smem_addr(sm + L.bq());
    if (tid == 0) {   // the Gram rows, while the fold runs: the operand's 128 rows (k_hi, q_hi, k_lo, q_lo,
                      // then unused) times the high k rows and times the low k rows
      const uint32_t id = umma_idesc_tf32(128, NG);
      // descriptors of K step 0; a step advances the start address (in 16-byte units) by 2 lbo
      const uint64_t da0 = umma_desc(sbq, lbo, 128u), db0 = umma_desc(sbq + 2u * NB * 16u, lbo, 128u);
      const uint64_t step = static_cast<uint64_t>((2u * lbo) >> 4);
#pragma unroll
      for (int s = 0; s < DK / 8; ++s) {
        const uint64_t da = da0 + s * step;
        umma_tf32_ss(tbase + kTcColD, da, da, id, s > 0);
        umma_tf32_ss(tbase + kTcColD + NG, da, db0 + s * step, id, s > 0);
      }
      umma_commit(bar + 2);
    }

    // ---- ancestors, one warp per node (warp 0, which issued the MMAs, takes the last): lane j takes v_j,
    // the node at distance j above t (v_0 = t); the product of the gates of v_0 .. v_j is rho_{t, v_{j+1}}
    // and, over the whole path, Gamma_t
    for (int t = W - 1 - warp; t < n; t += W) {
      const int d = si[L.dep(t)];
      int v = t;
      for (int k = 0; k < lane && k < d; ++k) v = parent[v];
      float prod = lane <= d ? sm[L.sc(v) + 0] : 1.f;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const float y = __shfl_up_sync(FULL, prod, m);
        if (lane >= m) prod *= y;
      }
      const float rho = __shfl_up_sync(FULL, prod, 1);   // lane j >= 1: rho_{t, v_j}
      const float gam_t = __shfl_sync(FULL, prod, d);
      if (lane >= 1 && lane <= d) {
        const int i = si[L.coff(t)] + lane - 1;
        si[L.ranc(i)] = v;
        si[L.ptn(i)] = t;
        sm[L.ra(i)] = rho;
      }
      if (lane == 0) {
        const float bt = sm[L.sc(t) + 1];
        *reinterpret_cast<float4*>(sm + L.gm(t)) = make_float4(gam_t, bt * gam_t, 0.f, 0.f);
      }
    }

    // ---- deferred commit: the pending path folded into the tile with the chain kernel's operations and
    // materialisation points, then the committed state written once
    float gam = 1.f;
    uint32_t fphase = 0;
    for (int f0 = 0; f0 < Lp; f0 += kFoldChunk) {
      const int fn = min(kFoldChunk, Lp - f0);
      if (f0 > 0) {   // a later chunk: the previous one consumed, its rows staged like the first
        __syncthreads();
        if (warp == 1) {
          if (lane == 0) mbar_expect(bar + 1, static_cast<uint32_t>(fn) * (DK + DV) * 4);
          __syncwarp();
          for (int i = lane; i < fn; i += 32) {
            const size_t row = nrow0 + (spath[f0 + i] & kPathNodeMask);
            bulk_g2s(sm + L.fk(i), p.pend_k + (row * p.Hk + kh) * DK, DK * 4, bar + 1);
            bulk_g2s(sm + L.fu(i), p.pend_u + (row * p.Hv + h) * DV, DV * 4, bar + 1);
            sm[L.fg() + i] = expf(p.pend_a[row * p.Hv + h]);
          }
        }
      }
      const bool ok = __syncthreads_and(mbar_wait(bar + 1, fphase));   // also publishes the gates
      fphase ^= 1;
      if (!ok) {
        if (tid == 0) device_error(p.err, GDN_DEVERR_TIMEOUT, b);
        mbar_wait(bar + 1, fphase ^ 1);
        mbar_wait(bar + 2, 0);
        return;
      }
      for (int i = 0; i < fn; ++i) {
        if (spath[f0 + i] & kPathHeadFlag) {
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

    // ---- the Gram rows to shared memory (lanes < 4 NB of the first product, < 2 NB of the second; warp
    // halves split the columns), before the products below overwrite their columns
    {
      const bool ok = __syncthreads_and(mbar_wait(bar + 2, 0));   // (the barrier also ends the fold's reads)
      if (!ok) {
        if (tid == 0) device_error(p.err, GDN_DEVERR_TIMEOUT, b);
        mbar_wait(bar + 2, 0);
        return;
      }
      tmem_fence_after();
      if (32 * quarter < 4 * NB) {
        for (int cc = half; cc < 2 * (NG / 16); cc += 2) {
          const bool second = cc >= NG / 16;
          float v[16];
          tmem_ld16(tlane + kTcColD + 16u * cc, v);
          tmem_wait_ld();
          if (c < (second ? 2 * NB : 4 * NB)) {
            float* dst = (second ? sm + L.g2(c) : sm + L.g1(c)) + 16 * (second ? cc - NG / 16 : cc);
#pragma unroll
            for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          }
        }
      }
    }

    // ---- A = T0^T into tensor memory, tf32 high part; its product with all 4 NB rows (high and low k, q)
#pragma unroll
    for (int q = 0; q < NR / 16; ++q) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 e = unpack2(R.T[8 * q + j]);
        v[2 * j] = tf32_hi(e.x);
        v[2 * j + 1] = tf32_hi(e.y);
      }
      tmem_st16(tlane + static_cast<uint32_t>(row0 + 16 * q), v);
    }
    tmem_wait_st();
    tmem_fence_before();
    __syncthreads();   // A high part in place, Gram columns read out; Gram rows and ancestor tables visible
    tmem_fence_after();
    if (tid == 0) {
      const uint32_t id = umma_idesc_tf32(128, 4 * NB);
      const uint64_t d0 = umma_desc(sbq, lbo, 128u), step = static_cast<uint64_t>((2u * lbo) >> 4);
#pragma unroll
      for (int s = 0; s < DK / 8; ++s) umma_tf32_ts(tbase + kTcColD, tbase + 8u * s, d0 + s * step, id, s > 0);
      umma_commit(bar + 3);
    }

    // ---- meanwhile the pair coefficients, a thread per ancestor pair (and per node for H_tt): G and H
    // are the sums of the three split products, A_ts = beta_t rho_ts G_ts and C_ts = rho_ts H_ts
    {
      const int np = si[L.coff(n)];
      for (int job = tid; job < np + n; job += THREADS) {
        const bool diag = job >= np;
        const int t = diag ? job - np : si[L.ptn(job)];
        const int s = diag ? t : si[L.ranc(job)];
        const float hq = sm[L.g1(NB + t) + s] + sm[L.g1(3 * NB + t) + s] + sm[L.g2(NB + t) + s];
        if (diag) {
          sm[L.gm(t) + 2] = hq;
        } else {
          const float gk = sm[L.g1(t) + s] + sm[L.g1(2 * NB + t) + s] + sm[L.g2(t) + s];
          const float rho = sm[L.ra(job)];
          sm[L.ra(job)] = sm[L.sc(t) + 1] * rho * gk;
          *reinterpret_cast<float2*>(sm + L.pc(job)) = make_float2(rho * hq, __int_as_float(s * DV));
        }
      }
    }
    // A low part over the high part once the product reading it completed
    if (!__syncthreads_and(mbar_wait(bar + 3, 0))) {   // (its barrier also publishes the coefficients)
      if (tid == 0) device_error(p.err, GDN_DEVERR_TIMEOUT, b);
      mbar_wait(bar + 3, 0);   // let the MMAs finish before the columns are freed
      return;
    }
    tmem_fence_after();
#pragma unroll
    for (int q = 0; q < NR / 16; ++q) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 e = unpack2(R.T[8 * q + j]);
        v[2 * j] = tf32_lo(e.x);
        v[2 * j + 1] = tf32_lo(e.y);
      }
      tmem_st16(tlane + static_cast<uint32_t>(row0 + 16 * q), v);
    }
    tmem_wait_st();
    tmem_fence_before();
    __syncthreads();   // A low part in place
    tmem_fence_after();
    if (tid == 0) {   // low A times the high rows, into the same columns
      const uint32_t id = umma_idesc_tf32(128, 2 * NB);
      const uint64_t d0 = umma_desc(sbq, lbo, 128u), step = static_cast<uint64_t>((2u * lbo) >> 4);
#pragma unroll
      for (int s = 0; s < DK / 8; ++s) umma_tf32_ts(tbase + kTcColD, tbase + 8u * s, d0 + s * step, id, 1);
      umma_commit(bar + 4);
    }

    // ---- meanwhile M = (I + A)^-1 over the ancestor pairs, one warp per node (warp 0 takes the last).
    // With a_0 .. a_d = t the root path, row t of M is x with x_d = 1 and x_j = -sum_{i>j} x_i A(a_i, a_j):
    // lane j holds x_j and, for i = d .. 1, takes x_i once it is final
    for (int t = W - 1 - warp; t < n; t += W) {
      const int d = si[L.dep(t)], i0 = si[L.coff(t)];
      if (d == 0) continue;
      int aj = 0, cj = 0;
      float x = 0.f;
      if (lane < d) {
        aj = si[L.ranc(i0 + d - lane - 1)];
        cj = si[L.coff(aj)];
        x = -sm[L.ra(i0 + d - lane - 1)];
      }
      for (int i = d - 1; i >= 1; --i) {
        const float xi = __shfl_sync(FULL, x, i);
        const int ci = __shfl_sync(FULL, cj, i);
        if (lane < i) x = fmaf(-sm[L.ra(ci + i - lane - 1)], xi, x);
      }
      if (lane < d) *reinterpret_cast<float2*>(sm + L.pm(i0 + d - lane - 1)) = make_float2(x, __int_as_float(aj * DV));
    }
    if (!__syncthreads_and(mbar_wait(bar + 4, 0))) {   // (its barrier also publishes M)
      if (tid == 0) device_error(p.err, GDN_DEVERR_TIMEOUT, b);
      mbar_wait(bar + 4, 0);
      return;
    }
    tmem_fence_after();

    // ---- B_t = beta_t v_t - beta_t Gamma_t (T0^T k_t) and Gamma_t (T0^T q_t), with T0^T k_t the sum of
    // columns t and 2 NB + t (high and low k) and T0^T q_t that of NB + t and 3 NB + t: thread (column c,
    // half) takes the nodes of its half
    {
      const int nbh = NB / 2, t0 = half * nbh;
      for (int g = 0; g < nbh; g += 4) {
        if (t0 + g >= n) break;   // warp-uniform
        float k1[4], k2[4], q1[4], q2[4];
        const uint32_t col = tlane + kTcColD + static_cast<uint32_t>(t0 + g);
        tmem_ld4(col, k1);
        tmem_ld4(col + 2 * NB, k2);
        tmem_ld4(col + NB, q1);
        tmem_ld4(col + 3 * NB, q2);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = t0 + g + j;
          if (t < n) {
            const float4 g4 = *reinterpret_cast<const float4*>(sm + L.gm(t));
            const float bt = sm[L.sc(t) + 1];
            sm[L.bm(t) + c] = fmaf(-g4.y, k1[j] + k2[j], bt * sm[L.v(t) + c]);
            sm[L.rr(t) + c] = g4.x * (q1[j] + q2[j]);
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
      int i = i0;
      if ((i & 1) && i < i1) {   // to an even pair index: the table is 16-byte aligned there
        const float2 e = *reinterpret_cast<const float2*>(sm + L.pm(i));
        const float4 x = *reinterpret_cast<const float4*>(brow + __float_as_int(e.y) + cc);
        u.x = fmaf(e.x, x.x, u.x); u.y = fmaf(e.x, x.y, u.y); u.z = fmaf(e.x, x.z, u.z); u.w = fmaf(e.x, x.w, u.w);
        ++i;
      }
      for (; i + 1 < i1; i += 2) {   // two ancestors at a time: their loads overlap
        const float4 e2 = *reinterpret_cast<const float4*>(sm + L.pm(i));
        const float4 x = *reinterpret_cast<const float4*>(brow + __float_as_int(e2.y) + cc);
        const float4 y = *reinterpret_cast<const float4*>(brow + __float_as_int(e2.w) + cc);
        u.x = fmaf(e2.x, x.x, u.x); u.y = fmaf(e2.x, x.y, u.y); u.z = fmaf(e2.x, x.z, u.z); u.w = fmaf(e2.x, x.w, u.w);
        u.x = fmaf(e2.z, y.x, u.x); u.y = fmaf(e2.z, y.y, u.y); u.z = fmaf(e2.z, y.z, u.z); u.w = fmaf(e2.z, y.w, u.w);
      }
      if (i < i1) {
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
      int i = i0;
      if ((i & 1) && i < i1) {   // to an even pair index: the table is 16-byte aligned there
        const float2 e = *reinterpret_cast<const float2*>(sm + L.pc(i));
        const float4 x = *reinterpret_cast<const float4*>(urow + __float_as_int(e.y) + cc);
        o.x = fmaf(e.x, x.x, o.x); o.y = fmaf(e.x, x.y, o.y); o.z = fmaf(e.x, x.z, o.z); o.w = fmaf(e.x, x.w, o.w);
        ++i;
      }
      for (; i + 1 < i1; i += 2) {   // two ancestors at a time: their loads overlap
        const float4 e2 = *reinterpret_cast<const float4*>(sm + L.pc(i));
        const float4 x = *reinterpret_cast<const float4*>(urow + __float_as_int(e2.y) + cc);
        const float4 y = *reinterpret_cast<const float4*>(urow + __float_as_int(e2.w) + cc);
        o.x = fmaf(e2.x, x.x, o.x); o.y = fmaf(e2.x, x.y, o.y); o.z = fmaf(e2.x, x.z, o.z); o.w = fmaf(e2.x, x.w, o.w);
        o.x = fmaf(e2.z, y.x, o.x); o.y = fmaf(e2.z, y.y, o.y); o.z = fmaf(e2.z, y.z, o.z); o.w = fmaf(e2.z, y.w, o.w);
      }
      if (i < i1) {
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
        si[L.flag() + 3] = m;
        for (int v = node, i = m - 1; v >= 0; v = parent[v], --i) si[L.path(i)] = v;
      }
      __syncthreads();
      R.load(st, DV);   // T0: the committed state this CTA wrote, or the input state when nothing was folded
      const int m = si[L.flag() + 3];
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
  // Each CTA holds kTcCols of the SM's 512 tensor-memory columns, so at most two may be resident: a third
  // would wait inside tcgen05.alloc until one of them exits.  Asking for more than a third of the SM's
  // 228 KB of shared memory keeps a third CTA off the SM (small d_k and n_max would otherwise fit three).
  constexpr size_t kTwoPerSm = 80 * 1024;
  const size_t smem = L.bytes() > kTwoPerSm ? L.bytes() : kTwoPerSm;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  auto kern = ut_tc_verify_kernel<DK, InT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const size_t grid = static_cast<size_t>(p.B) * p.layers * p.Hv;
  VerifyParams q = p;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTcThreads, smem) == cudaSuccess)
    q.prefetch_ahead = sms * per_sm;   // one wave of resident CTAs
  else
    q.prefetch_ahead = 0;
  cudaGetLastError();   // a failed query only disables the prefetch
  kern<<<static_cast<unsigned>(grid), kTcThreads, smem, s>>>(q);
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
