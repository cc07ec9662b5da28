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
// walks its whole tree depth first, light children before the heavy one, as the
// packed schedule's ops list it: a heavy-light chain continues in registers from
// head to tail; a branching node's state is materialised once and stashed, the
// first child continues from the registers and each later child reloads the
// stash.  Stashes live in tensor memory (tcgen05): the 32x32b access shape gives
// every thread its own TMEM lane, so a register tile moves in and out without
// crossing lanes, and the 256 KB per SM holds two levels of stash for each of
// the four resident CTAs -- enough for every tree whose root paths cross at most
// two light edges (all 22-node top-4 DDTrees here).  Deeper stashes spill to the
// node's boundary slot in HBM, which is also where boundary states are written
// when the caller asks for them.
//
// Thread layout: a thread owns RPT consecutive rows x 4 consecutive columns of
// the [d_k][d_v] tile, held as packed (row r, row r+1) fp32 pairs so the tile
// arithmetic issues as f32x2 instructions.  Lanes run along the columns first
// (CG column groups), so each warp-wide 16-byte load or store of the tile reads
// or writes whole 128-byte lines -- the layout that keeps the state and
// boundary transfers cheap for the load/store pipe.  The reductions over d_k
// (sk = T^T k, sq = T^T q) are in-thread sums, an xor-shuffle across the row
// groups of one warp, and a sum over the warps through a small double-buffered
// shared array (one barrier per node).  Per node:
//   pass A (state before the node):  sk = T^T k,  sq = T^T q
//   p = g sk,  u = beta (v - p),  o = g sq + u (k . q)          (= T'^T q exactly)
//   pass B:  T <- fmaf(k, u, g * T)
// Everything a node needs (k_hat, q_hat, v slice, gate, beta, k.q) is staged in
// shared memory once per tree, and the pending path's factors once per chunk of
// the fold, so the node loop issues no global loads.
//
// Lazy decay: a chain keeps its tile as T~ with a scalar gamma, the state being
// gamma * T~.  A node multiplies only the scalar (gamma' = gamma g), so pass B
// is one FMA per element, T~ += k (u / gamma')^T, and pass A reads
// p = gamma' T~^T k, o = gamma' T~^T q + u (k . q).  The tile is materialised
// (T~ <- gamma T~, gamma = 1) only where the state leaves the registers -- at
// boundary slots and the committed write -- and when gamma' falls below
// kGammaFloor (which also covers g = 0), where that node applies its decay to
// the tile before the update.
//
// The fold repeats exactly these operations with the same u -- including the
// materialisation wherever the accepted path enters a light child, where the
// verify reloaded the stored state -- so the committed state reproduces, bit
// for bit, the state the earlier verify stored for that node.
#include <type_traits>

#include "gdn_tile.cuh"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

constexpr int kVerifyThreads = 128;

// Shared-memory layout (floats): tree region, fold region, then the schedule record (int32).
template <int DK>
struct Smem {
  int n_max, cpb;
  __device__ int kq(int node) const { return node * 2 * DK; }                  // [n_max][2][DK]
  __device__ int v(int node) const { return n_max * 2 * DK + node * cpb; }     // [n_max][cpb]
  // per node one float4: (g = exp(a), beta, k . q, a)
  __device__ int sc(int node) const { return n_max * (2 * DK + cpb) + 4 * node; }
  __device__ int fold0() const { return sc(n_max); }
  __device__ int fk(int i) const { return fold0() + i * DK; }                   // [kFoldChunk][DK]
  __device__ int fu(int i) const { return fold0() + kFoldChunk * DK + i * cpb; } // [kFoldChunk][cpb]
  __device__ int fg() const { return fold0() + kFoldChunk * (DK + cpb); }      // [kFoldChunk]
  __device__ int part0() const { return (fg() + kFoldChunk + 3) & ~3; }        // [2][warps][2][cpb]
  __device__ int rec0(int warps) const { return part0() + 2 * warps * 2 * cpb; } // packed schedule record
  __device__ int bar0(int warps) const { return (rec0(warps) + SchedLayout{n_max}.words() + 3) & ~3; }  // mbarrier
};

template <int DK>
size_t smem_bytes(int n_max, int cpb, int warps) {
  const int fold0 = n_max * (2 * DK + cpb) + 4 * n_max;
  const int part0 = (fold0 + kFoldChunk * (DK + cpb) + kFoldChunk + 3) & ~3;
  const int words = SchedLayout{n_max}.words();
  const int bar0 = (part0 + 2 * warps * 2 * cpb + words + 3) & ~3;
  return static_cast<size_t>(bar0 + 4) * sizeof(float);
}

template <int DK, int RPT, int CPB, typename InT>
__global__ void __launch_bounds__(kVerifyThreads, 4) chain_verify_kernel(VerifyParams p) {
  constexpr int NP = RPT / 2;              // row pairs per column
  constexpr int CG = CPB / kCols;          // column groups per CTA
  constexpr int NW = (DK / RPT) * CG / 32; // warps per CTA
  constexpr int cpb = CPB;
  constexpr int kWords = 2 * kCols * NP;   // 32-bit words of a thread's tile = its tensor-memory columns per level
  static_assert(RPT % 4 == 0 && CG <= 32 && (DK / RPT) * CG % 32 == 0, "layout");
  static_assert(kWords % 32 == 0 && tmem_columns(kTmemLevels * kWords) <= 512, "stash");
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  const Smem<DK> L{p.n_max, cpb};

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
  const int tid = threadIdx.x;

  const int lane = tid & 31, warp = tid >> 5;
  constexpr int nwarps = NW;
  const int cg = tid % CG;                                         // column group
  const int rg = tid / CG;                                         // row group
  const int c0 = cg * kCols;                                       // first column within the slice
  const int col = s * cpb + c0;                                    // first column within d_v
  const int row0 = rg * RPT;
  const size_t tile = static_cast<size_t>(DK) * p.dv;

  // the thread's register tile (RegTile: RPT rows x 4 columns as packed row pairs)
  RegTile<RPT> R;
  auto& T = R.T;
  auto load_tile = [&](const float* base) { R.load(base, p.dv); };
  auto store_tile = [&](float* base) { R.store(base, p.dv); };
  auto materialise = [&](float gam) { R.materialise(gam); };
  auto update_lazy = [&](const float* kvec, float4 ut) { R.update_lazy(kvec + row0, ut); };
  auto advance = [&](const float* kvec, float gam1, float4 u) -> float { return R.advance(kvec + row0, gam1, u); };
  auto store_scaled = [&](float* base, float gam) { R.store_scaled(base, p.dv, gam); };

  float* st = p.state + (static_cast<size_t>(bl) * p.Hv + h) * tile + static_cast<size_t>(row0) * p.dv + col;

  // ---- tensor memory first.  Until a CTA of a kernel that allocates tensor memory gives up its
  // allocation permit, the SM holds back further CTAs of it; so warp 0 allocates the stash this tree's
  // schedule asks for (`levels` copies of every thread's register tile: thread t of warp w owns lane
  // 32 (w % 4) + t, a level is kWords consecutive columns) and relinquishes the permit at once.  The
  // same warp releases the columns at the very end, after every warp's last access; the body below
  // leaves only by uniform returns, so every thread reaches that point.
  const SchedLayout lay{p.n_max};
  const int32_t* rec = p.words ? p.words + static_cast<size_t>(b) * lay.words() : nullptr;
  const int levels_rec = rec ? rec[4] : 0;
  const int levels = (levels_rec >= 0 && levels_rec <= kTmemLevels) ? levels_rec : 0;
  const uint32_t tcols = tmem_columns(levels * kWords);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L.bar0(nwarps) + 2);
  if (warp == 0) {
    __syncwarp();
    if (tcols) tmem_alloc(tslot, tcols);
    tmem_relinquish();
  }
  uint32_t tbase = 0;
  if (tcols) {
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    tbase = *tslot;
  }
  const uint32_t tthread = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16);

  [&]() {
  load_tile(st);

  // ---- schedule header, pending length, staging barrier
  if (__syncthreads_or(launch_aborted(p.err))) return;   // an earlier CTA gave up on a wait
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bar0(nwarps));
  if (tid == 0) mbar_init(bar);
  int n = 0;
  int32_t* srec = reinterpret_cast<int32_t*>(sm + L.rec0(nwarps));
  if (rec) {
    n = rec[0];
    if (n < 1 || n > p.n_max || levels_rec < 0 || levels_rec > kTmemLevels) {
      if (tid == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
      return;
    }
    for (int i = tid; i < lay.words(); i += blockDim.x) srec[i] = rec[i];
  }
  const int Lp = p.fold ? p.pend_len[b] : 0;
  const int32_t* path = p.pend_path + static_cast<size_t>(b) * p.n_max;
  const size_t nrow0 = static_cast<size_t>(bl) * p.n_max;
  __syncthreads();   // barrier initialised

  // ---- asynchronous staging (TMA bulk copies): the tree's k_hat, q_hat (k-head kh) and v slice
  // rows, and the pending path's k / u rows, chunk by chunk; gates and betas by plain loads.
  const InT* beta = static_cast<const InT*>(p.beta);
  const InT* logg = static_cast<const InT*>(p.log_g);
  uint32_t phase = 0;
  auto stage = [&](bool tree, int f0, int fn) -> bool {
    const uint32_t bytes = (tree ? static_cast<uint32_t>(n) * (2 * DK + cpb) * 4 : 0u) +
                           static_cast<uint32_t>(fn) * (DK + cpb) * 4;
    if (bytes == 0) return true;
    if (warp == 0) {
      if (lane == 0) mbar_expect(bar, bytes);
      __syncwarp();
      if (tree)
        for (int node = lane; node < n; node += 32) {
          const size_t row = nrow0 + node;
          bulk_g2s(sm + L.kq(node), p.k_in + (row * p.Hk + kh) * DK, DK * 4, bar);
          bulk_g2s(sm + L.kq(node) + DK, p.q_in + (row * p.Hk + kh) * DK, DK * 4, bar);
          bulk_g2s(sm + L.v(node), p.v_in + (row * p.Hv + h) * p.dv + s * cpb, cpb * 4, bar);
        }
      for (int i = lane; i < fn; i += 32) {
        const size_t row = nrow0 + (path[f0 + i] & kPathNodeMask);
        bulk_g2s(sm + L.fk(i), p.pend_k + (row * p.Hk + kh) * DK, DK * 4, bar);
        bulk_g2s(sm + L.fu(i), p.pend_u + (row * p.Hv + h) * p.dv + s * cpb, cpb * 4, bar);
      }
    }
    if (tree)
      for (int node = tid; node < n; node += blockDim.x) {
        const float a = load_in<InT>(logg, (nrow0 + node) * p.Hv + h);
        sm[L.sc(node) + 0] = expf(a);
        sm[L.sc(node) + 1] = load_in<InT>(beta, (nrow0 + node) * p.Hv + h);
        sm[L.sc(node) + 3] = a;
        if (s == 0) p.a_out[(nrow0 + node) * p.Hv + h] = a;   // the bank's log-gate, exact
      }
    for (int i = tid; i < fn; i += blockDim.x)
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

  // ---- deferred commit: T <- exp(a) T + k u^T along the pending path, gathered by node index
  float gam = 1.f;               // the state is gam * T
  if (!stage(rec != nullptr, 0, min(Lp, kFoldChunk))) return;
  for (int f0 = 0; f0 < Lp; f0 += kFoldChunk) {
    const int fn = min(kFoldChunk, Lp - f0);
    if (f0 > 0) {
      __syncthreads();   // previous chunk consumed
      if (!stage(false, f0, fn)) return;
    }
    for (int i = 0; i < fn; ++i) {
      if (path[f0 + i] & kPathHeadFlag) {   // the verify stored and reloaded the state here
        materialise(gam);
        gam = 1.f;
      }
      gam = advance(sm + L.fk(i), gam * sm[L.fg() + i], *reinterpret_cast<const float4*>(sm + L.fu(i) + c0));
    }
  }
  if (Lp > 0) {
    materialise(gam);            // the committed state; verification continues from exactly these values
    gam = 1.f;
    store_tile(st);
  }
  if (!rec) return;  // fold only

  // ---- k . q of every node (one warp per node)
  for (int node = warp; node < n; node += blockDim.x / 32) {
    const float* kk = sm + L.kq(node);
    float acc = 0.f;
    for (int e = lane; e < DK; e += 32) acc = fmaf(kk[e], kk[DK + e], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) sm[L.sc(node) + 2] = acc;
  }
  __syncthreads();

  const int32_t* parent = srec + lay.parent();
  const int32_t* bslot = srec + lay.bslot();
  const int32_t* ops = srec + lay.ops();
  float* bnd_base = p.boundary + (static_cast<size_t>(bl) * p.nb_max * p.Hv + h) * tile +
                    static_cast<size_t>(row0) * p.dv + col;
  int parity = 0;
  const size_t slot_stride = static_cast<size_t>(p.Hv) * tile;

  // ---- stash moves between the register tile and tensor memory
  auto tmem_put = [&](int level) {
    const uint32_t ta = tthread + static_cast<uint32_t>(level * kWords);
    __syncwarp();   // the warp-collective tcgen05 accesses run converged
#pragma unroll
    for (int half = 0; half < kWords / 32; ++half) {   // 32 words per statement
      u64 v[16];
#pragma unroll
      for (int f = 0; f < 16; ++f) v[f] = T[(16 * half + f) / NP][(16 * half + f) % NP];
      tmem_put32(ta + 32u * half, v);
    }
  };
  auto tmem_get = [&](int level) {
    const uint32_t ta = tthread + static_cast<uint32_t>(level * kWords);
    __syncwarp();
#pragma unroll
    for (int half = 0; half < kWords / 32; ++half) {
      u64 v[16];
      tmem_get32(ta + 32u * half, v);
#pragma unroll
      for (int f = 0; f < 16; ++f) T[(16 * half + f) / NP][(16 * half + f) % NP] = v[f];
    }
  };

  bool preloaded = false;        // the tile already holds the next node's source (loaded during a leaf)
  const size_t node_stride = static_cast<size_t>(p.Hv) * p.dv;          // o and u rows of consecutive nodes
  float* o_base = p.out_o + (nrow0 * p.Hv + h) * p.dv + col;
  float* u_base = p.u_out + (nrow0 * p.Hv + h) * p.dv + col;
  // One node; the leaf flag and the "decay into the tile" flag are compile-time so each
  // combination is its own straight-line body (no predicated rare paths on common nodes).
  auto step = [&](int node, int pre, float g, float4 nsc, auto leaf_t, auto low_t) {
    constexpr bool kLeaf = decltype(leaf_t)::value;
    constexpr bool kLow = decltype(low_t)::value;
    const float* kvec = sm + L.kq(node);

    // pass A on the state before this node
    u64 ak[kCols], aq[kCols];
    R.dots(kvec + row0, kvec + DK + row0, ak, aq);
    // A leaf's updated state is never read (the fold rebuilds it from the factor bank), so the tile
    // is free after pass A: when the next node reloads a stash from HBM, start that load now, under
    // this node's reduction.
    if constexpr (kLeaf) {
      if (pre >= 0) {
        load_tile(bnd_base + static_cast<size_t>(pre) * slot_stride);
        preloaded = true;
      }
    }
    float4 sk = fold_pairs(ak), sq = fold_pairs(aq);
    // row groups of this warp
#pragma unroll
    for (int m = CG; m < 32; m <<= 1) {
      sk.x += __shfl_xor_sync(0xffffffffu, sk.x, m);
      sk.y += __shfl_xor_sync(0xffffffffu, sk.y, m);
      sk.z += __shfl_xor_sync(0xffffffffu, sk.z, m);
      sk.w += __shfl_xor_sync(0xffffffffu, sk.w, m);
      sq.x += __shfl_xor_sync(0xffffffffu, sq.x, m);
      sq.y += __shfl_xor_sync(0xffffffffu, sq.y, m);
      sq.z += __shfl_xor_sync(0xffffffffu, sq.z, m);
      sq.w += __shfl_xor_sync(0xffffffffu, sq.w, m);
    }
    // warps: partials [parity][warp][k|q][cpb]; the row groups of a warp hold equal sums after the
    // butterfly, so every lane stores (same value, same address) and the warp does not diverge
    float* part = sm + L.part0() + parity * (nwarps * 2 * cpb);
    *reinterpret_cast<float4*>(part + (warp * 2 + 0) * cpb + c0) = sk;
    *reinterpret_cast<float4*>(part + (warp * 2 + 1) * cpb + c0) = sq;
    __syncthreads();
    sk = *reinterpret_cast<const float4*>(part + c0);
#pragma unroll
    for (int w = 1; w < nwarps; ++w) {
      const float4 t = *reinterpret_cast<const float4*>(part + (w * 2) * cpb + c0);
      sk.x += t.x; sk.y += t.y; sk.z += t.z; sk.w += t.w;
    }
    parity ^= 1;
    const float bt = nsc.y;
    const float4 v = *reinterpret_cast<const float4*>(sm + L.v(node) + c0);
    float4 u;
    u.x = bt * (v.x - g * sk.x);
    u.y = bt * (v.y - g * sk.y);
    u.z = bt * (v.z - g * sk.z);
    u.w = bt * (v.w - g * sk.w);
    if (rg == 0) {
      sq = *reinterpret_cast<const float4*>(part + cpb + c0);
#pragma unroll
      for (int w = 1; w < nwarps; ++w) {
        const float4 t = *reinterpret_cast<const float4*>(part + (w * 2 + 1) * cpb + c0);
        sq.x += t.x; sq.y += t.y; sq.z += t.z; sq.w += t.w;
      }
      const float kq = nsc.z;
      float4 o;
      o.x = fmaf(u.x, kq, g * sq.x);
      o.y = fmaf(u.y, kq, g * sq.y);
      o.z = fmaf(u.z, kq, g * sq.z);
      o.w = fmaf(u.w, kq, g * sq.w);
      *reinterpret_cast<float4*>(o_base + node * node_stride) = o;
      *reinterpret_cast<float4*>(u_base + node * node_stride) = u;
    }

    if constexpr (!kLeaf) {   // pass B (a leaf's new state is never used)
      float r = 1.f;
      if constexpr (kLow) {
        materialise(g);        // the decay goes into the tile, as in advance()
        gam = 1.f;
      } else {
        r = __fdividef(1.f, g);
        gam = g;
      }
      update_lazy(kvec, make_float4(u.x * r, u.y * r, u.z * r, u.w * r));
    }
  };
  using kT = std::true_type;
  using kF = std::false_type;

  // ---- the nodes in the schedule's depth-first order.  A node continues from the registers or
  // reloads its parent's stash (tensor memory, or the parent's boundary slot in HBM); a node whose
  // state is stashed is materialised first.  Every check below depends only on the schedule record,
  // so the whole CTA takes the same branch.
  bool bad = false;
  for (int i = 0; i < n; ++i) {
    const int op = ops[i];
    const int node = op & kOpNode;
    const int slot = node < n ? bslot[node] : -1;
    if (node >= n || slot >= p.nb_max || ((op & kOpLeaf) && (op & kOpPush)) || ((op & kOpReload) && node == 0)) {
      bad = true;
      break;
    }
    if (op & kOpReload) {
      if (!preloaded) {
        if (op & kOpReloadGlobal) {
          const int src = bslot[parent[node]];
          if (src < 0 || src >= p.nb_max) {
            bad = true;
            break;
          }
          load_tile(bnd_base + static_cast<size_t>(src) * slot_stride);
        } else {
          const int lvl = (op >> kOpReloadLevelShift) & 3;
          if (lvl >= levels) {
            bad = true;
            break;
          }
          tmem_get(lvl);
        }
      }
      gam = 1.f;
    }
    preloaded = false;
    const float4 nsc = *reinterpret_cast<const float4*>(sm + L.sc(node));
    const float g = gam * nsc.x;   // gamma' of this node
    const bool low = g < kGammaFloor;
    if (op & kOpLeaf) {
      // the boundary slot the next node reloads from, if it does so from HBM: loaded during this leaf
      int pre = -1;
      if (i + 1 < n) {
        const int nop = ops[i + 1];
        const int nn = nop & kOpNode;
        if ((nop & kOpReload) && (nop & kOpReloadGlobal) && nn > 0 && nn < n) {
          const int nsrc = bslot[parent[nn]];
          pre = nsrc < p.nb_max ? nsrc : -1;
        }
      }
      if (low) step(node, pre, g, nsc, kT{}, kT{});
      else step(node, pre, g, nsc, kT{}, kF{});
    } else {
      if (low) step(node, -1, g, nsc, kF{}, kT{});
      else step(node, -1, g, nsc, kF{}, kF{});
    }
    if (op & kOpPush) {
      materialise(gam);
      gam = 1.f;
      if (op & kOpPushGlobal) {
        if (slot < 0) {
          bad = true;
          break;
        }
        store_tile(bnd_base + static_cast<size_t>(slot) * slot_stride);
      } else {
        const int lvl = (op >> kOpPushLevelShift) & 3;
        if (lvl >= levels) {
          bad = true;
          break;
        }
        tmem_put(lvl);
        if (p.boundary_out && slot >= 0) store_tile(bnd_base + static_cast<size_t>(slot) * slot_stride);
      }
    } else if (p.boundary_out && slot >= 0) {
      store_scaled(bnd_base + static_cast<size_t>(slot) * slot_stride, gam);
    }
  }
  if (bad && tid == 0) device_error(p.err, GDN_DEVERR_SCHEDULE, b);
  }();

  if (tcols) {
    tmem_fence_before();
    __syncthreads();   // every warp's tensor-memory accesses are complete (each waited on its own)
    tmem_fence_after();
    if (warp == 0) {
      __syncwarp();
      tmem_dealloc(tbase, tcols);
    }
  }
}

template <int DK, int RPT, int CPB, typename InT>
cudaError_t launch_t(const VerifyParams& p, cudaStream_t s) {
  constexpr int threads = (DK / RPT) * CPB / kCols;
  static_assert(threads % 32 == 0 && threads <= kVerifyThreads, "CTA shape");
  const size_t grid = static_cast<size_t>(p.B) * p.layers * p.Hv * (p.dv / CPB);
  const size_t smem = smem_bytes<DK>(p.n_max, CPB, threads / 32);
  auto kern = chain_verify_kernel<DK, RPT, CPB, InT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<static_cast<unsigned>(grid), threads, smem, s>>>(p);
  return cudaGetLastError();
}

// Columns per CTA: as many as 128 threads cover, at most d_v.
template <int DK, int RPT, typename InT>
cudaError_t launch_dv(const VerifyParams& p, cudaStream_t s) {
  constexpr int kMaxCols = kCols * kVerifyThreads / (DK / RPT);
  switch (p.dv) {
    case 32: return launch_t<DK, RPT, 32, InT>(p, s);
    case 64: return launch_t<DK, RPT, (64 < kMaxCols ? 64 : kMaxCols), InT>(p, s);
    case 128: return launch_t<DK, RPT, (128 < kMaxCols ? 128 : kMaxCols), InT>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename InT>
cudaError_t launch_dtype(const VerifyParams& p, cudaStream_t s) {
  switch (p.dk) {
    case 32: return launch_dv<32, 8, InT>(p, s);
    case 64: return launch_dv<64, 16, InT>(p, s);
    case 128: return launch_dv<128, 16, InT>(p, s);
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
