/*
 * gdn_tree.h -- C ABI for state-resident verification of speculative draft
 * trees through Gated DeltaNet (gated delta-rule linear attention) layers.
 *
 * Method: "Lucebox SpecLA 与 Gated DeltaNet 状态驻留验证原理指南" (the SpecLA
 * article), sections "状态驻留验证" (state-resident verify), "链分解与依赖波
 * HLD 调度" (heavy-light chains and dependency waves), "接受因子缓存" (factor
 * banks), "延迟融合提交" (deferred fused commit); and the Luce DFlash README,
 * "How it works" (DDTree tree verify, tree-aware conv window).
 *
 * Per v-head the recurrent state is stored transposed, T = S^T, as a row-major
 * [d_k][d_v] fp32 tile.  One token (x, beta, a) advances (T, W) by
 *   y   = depthwise causal conv of the K-row window [W; x] (or y = x), then SiLU (optional)
 *   q,k = L2-normalised q and k heads of y (q scaled by q_scale), v = v heads of y
 *   T  <- exp(a) * T;  p = T^T k;  u = beta (v - p);  T <- T + k u^T;  o = T^T q
 * which is S' = g S (I - beta k k^T) + beta v k^T, o = S' q.  A draft tree is
 * verified by giving every node the state reached along its own root path.
 *
 * Conventions for every call:
 *  - The caller owns every buffer.  No call allocates device memory.
 *  - Device calls are asynchronous on the given stream, never synchronise the
 *    host, and never trap on the device.  Host-detectable errors (bad sizes,
 *    NULL or misaligned pointers, invalid trees) return a negative status
 *    before anything is launched; gdn_last_error() then describes it.
 *  - Device-detectable errors set bits in the caller's device error words
 *    (gdn_banks.err): an accepted path that is not a root path of the verified
 *    tree (GDN_DEVERR_INVALID_PATH), packed schedule words out of range
 *    (GDN_DEVERR_SCHEDULE), an asynchronous copy or MMA that a bounded wait gave
 *    up on (GDN_DEVERR_TIMEOUT).  gdn_check_error() reads and clears them.
 *    GDN_DEVERR_TIMEOUT is sticky: while it is set, every conv-window, verify and
 *    finish kernel of every later call (not only the rest of the launch that set
 *    it) exits at once without doing work, so outputs stay unwritten and pending
 *    factors stay unfolded.  The host-side bank lifecycle still advances
 *    (pend_bank, verified_bank), and gdn_commit_fold still records paths.  A
 *    caller that reads GDN_ERR_TIMEOUT from gdn_check_error() must therefore treat
 *    the state of the calls made since the last clean check as lost (restore it
 *    from a checkpoint: state, conv_state and the bank fields).
 *  - Device pointers must be 16-byte aligned.
 *  - Per-node arrays are indexed [request][layer][node][...] with a node stride
 *    of n_max; nodes are numbered so that parent[i] < i (node 0 is the root).
 *  - Channel order of a raw input row: [q (Hk*dk) | k (Hk*dk) | v (Hv*dv)],
 *    head-major.  v-head h uses q/k head h / (Hv/Hk).
 */
#ifndef GDN_TREE_H
#define GDN_TREE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 2
#define GDN_MAX_NODES 64   /* largest tree (n_max) the kernels accept */
#define GDN_MAX_TAPS 8     /* largest conv kernel K */

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = -1,   /* a size, pointer or alignment is wrong */
  GDN_ERR_INVALID_TREE = -2,  /* parent[] is not a tree in topological order */
  GDN_ERR_INVALID_PATH = -3,  /* (device) an accepted path is not a root path */
  GDN_ERR_UNSUPPORTED = -4,   /* a head size or mode this build has no kernel for */
  GDN_ERR_CUDA = -5,          /* a CUDA launch or copy failed */
  GDN_ERR_TIMEOUT = -6,       /* (device) a bounded wait on an asynchronous copy or MMA gave up */
  GDN_ERR_CAPACITY = -7,      /* a buffer is smaller than the call needs */
  GDN_ERR_STATE = -8,         /* calls out of order (commit without a verify) */
  GDN_ERR_SCHEDULE = -9       /* (device) packed schedule words out of range */
} gdn_status;

typedef enum { GDN_DTYPE_F32 = 0, GDN_DTYPE_BF16 = 1 } gdn_dtype;

/* Bits of gdn_banks.err[0]. err[1] holds 1 + the first request that set a bit. */
#define GDN_DEVERR_INVALID_PATH 1  /* an accepted path is not a root path; nothing committed */
#define GDN_DEVERR_SCHEDULE 2      /* packed schedule words out of range; the access was skipped */
#define GDN_DEVERR_TIMEOUT 4       /* an asynchronous copy or MMA did not complete in time; the CTA stopped */

/* Shapes and modes of one GDN layer stack. */
typedef struct {
  int32_t Hk, Hv;      /* q/k heads and v-heads; Hv % Hk == 0 */
  int32_t dk, dv;      /* head sizes: dk in {32, 64, 128}; dv in {32, 64, 128} */
  int32_t K;           /* conv taps, 1..GDN_MAX_TAPS (ignored in bypass mode) */
  int32_t conv_mode;   /* 0: y = x (inputs are q|k|v already); 1: causal depthwise conv */
  int32_t act;         /* 0: none; 1: SiLU after the conv */
  int32_t in_dtype;    /* gdn_dtype of x_raw, beta and log_g */
  float q_scale;       /* multiplies the normalised q (1.0 gives o = S' q) */
  float l2_eps;        /* q_hat = q / sqrt(sum q^2 + l2_eps); same for k */
} gdn_dims;

/* ---------------------------------------------------------------------------
 * Heavy-light schedule of one tree (host, pure, O(n)).
 * SpecLA article, "链分解与依赖波 HLD 调度": the heavy child of a node is its
 * child with the largest subtree (ties: smaller index); heavy edges continue a
 * chain and light edges start one; only the states at chain boundaries are
 * materialised; chains are grouped into dependency waves.  Here the wave of a
 * chain is the number of light edges from the root to its head, chains are
 * ordered by (wave, head), boundary nodes are the parents of non-root chain
 * heads (exactly the nodes with two or more children) and get slots in
 * ascending node order.
 *
 * Every array is caller-owned with room for n entries (chain_off and wave_off:
 * n + 1).  On GDN_ERR_INVALID_TREE nothing is written.
 * ------------------------------------------------------------------------- */
typedef struct {
  int32_t n, n_chains, n_waves, n_boundary;
  int32_t* subtree;        /* [n] subtree size of each node */
  int32_t* heavy;          /* [n] heavy child, -1 for a leaf */
  int32_t* chain_of;       /* [n] chain id of each node */
  int32_t* pos_in_chain;   /* [n] position of each node in its chain */
  int32_t* chain_head;     /* [n_chains] first node of each chain */
  int32_t* chain_len;      /* [n_chains] */
  int32_t* chain_off;      /* [n_chains + 1] offsets into chain_nodes */
  int32_t* chain_nodes;    /* [n] chains concatenated, head to tail */
  int32_t* chain_wave;     /* [n_chains] */
  int32_t* chain_src_slot; /* [n_chains] boundary slot the chain starts from, -1 = persistent state */
  int32_t* wave_off;       /* [n_waves + 1] chain-id ranges of each wave */
  int32_t* boundary_slot;  /* [n] slot of a boundary node, -1 otherwise */
  int32_t* boundary_node;  /* [n_boundary] node of each slot */
} gdn_schedule;

gdn_status gdn_hld_schedule(const int32_t* parent, int32_t n, gdn_schedule* out);

/* ---------------------------------------------------------------------------
 * Packed batch schedule: the compact form the kernels read.
 * One record of gdn_schedule_words(n_max) = 5 + 4 n_max int32 per request:
 *   [0] n  [1] n_chains  [2] n_boundary  [3] n_waves
 *   [4] stash levels the verify keeps in tensor memory (0..2)
 *   [5 .. 5+n_max)              parent (unused entries -1)
 *   [5+n_max .. 5+2n_max)       boundary slot of each node (-1: none)
 *   [5+2n_max .. 5+3n_max)      node flags: bit 0 = the state after the node is
 *                               materialised and stashed (its children start from it)
 *   [5+3n_max .. 5+4n_max)      verify ops, one per node in walk order:
 *       bits 0-7   node
 *       bit 8      reload: start from the parent's stash (else continue from the
 *                  previous node's registers -- the previous node is the parent)
 *       bit 9      the stash is the parent's boundary slot in boundary_states
 *                  (else tensor memory, level in bits 10-11)
 *       bit 12     push: after the node, materialise the state and stash it
 *       bit 13     in the node's boundary slot (else tensor memory, level in bits 14-15)
 *       bit 16     leaf: the node has no children
 * Heavy-light walk (SpecLA article, "链分解与依赖波 HLD 调度"): depth first, light
 * children before the heavy child, so every chain runs in registers from head to
 * tail.  A branching node (two or more children = a boundary node) is stashed
 * once; its first child continues from the registers, the others reload the
 * stash, the last (heavy) one releases it.  At most (light edges on a root path)
 * stashes are live; the first two levels sit in tensor memory on the SM, deeper
 * ones spill to the node's boundary slot.
 * gdn_pack_schedules runs gdn_hld_schedule on every request's tree and writes
 * the records into words_host (B * gdn_schedule_words(n_max) int32, caller-
 * owned host memory); *nb_max_out receives the largest boundary count and
 * *depth_max_out the depth of the deepest node (either may be NULL).  The
 * caller copies the words to the device and fills a gdn_batch_schedule.
 * parents: B rows of n_max entries; n[b] nodes of request b are used.
 * ------------------------------------------------------------------------- */
int32_t gdn_schedule_words(int32_t n_max);
gdn_status gdn_pack_schedules(const int32_t* parents, const int32_t* n, int32_t B, int32_t n_max,
                              int32_t* words_host, int32_t* nb_max_out, int32_t* depth_max_out);

/* Per-node-state schedule in the same packed layout, for comparison with the heavy-light one: every node
 * with children stashes its state in its boundary slot (in HBM) and every child reloads it from there -- the
 * rollback-by-snapshot scheme the SpecLA article replaces ("状态驻留验证": state traffic twice per token
 * instead of twice per chain).  The walk is depth first, children by index.  Same arguments and results as
 * gdn_pack_schedules; nb_max is the number of nodes with children. */
gdn_status gdn_pack_schedules_per_node(const int32_t* parents, const int32_t* n, int32_t B, int32_t n_max,
                                       int32_t* words_host, int32_t* nb_max_out, int32_t* depth_max_out);

/* ---------------------------------------------------------------------------
 * DDTree construction with confidence pruning (host, pure).
 * Luce DFlash README, "How it works": a best-first tree of up to `budget`
 * nodes spans the draft's top-K branches at each position (flags
 * --ddtree-budget, default 22, and --ddtree-tau, a confidence margin that
 * SpecLA sets to 6); SpecLA article, section "一键开启": nodes scoring below
 * q* - tau are pruned; section "正确性如何保证": cumulative-score pruning,
 * ancestor closure, budget cap.
 *
 * logp: host, [depth_max][top_k] fp32, row d-1 = the draft's log-probabilities
 *   of its top_k tokens at depth d (every entry <= 0 and not NaN, else
 *   GDN_ERR_INVALID_ARG).  A node is a sequence of ranks; score = cumulative
 *   log-probability from the root (double); the root scores 0.
 * budget: 1..GDN_MAX_NODES nodes, root included.
 * tau: >= 0 prunes every node with score < q* - tau, q* = the best candidate
 *   score (= max_r logp[0][r]); tau < 0 disables pruning; NaN is an error.
 * flags: GDN_DDTREE_CHAIN_SEED inserts the greedy chain (best rank at every
 *   depth, ties to the lower rank) first, as far as it is eligible and fits.
 * The remaining nodes are the best eligible candidates in the order (higher
 * score, lower depth, lexicographically smaller rank sequence), added while
 * the budget allows.  Output (caller-owned, >= budget entries each; depth,
 * rank and score may be NULL), numbered in DFS preorder with children by
 * rank, so parent[0] = -1 and parent[i] < i: parent, depth, rank (root -1),
 * score; *n_out = the node count.  The tree feeds gdn_hld_schedule /
 * gdn_pack_schedules as it is.
 * gdn_ddtree_build_batch builds B trees from logp [B][depth_max][top_k] into
 * parents [B][n_max] (n_max >= budget, unused entries -1) and n [B].
 * ------------------------------------------------------------------------- */
#define GDN_DDTREE_CHAIN_SEED 1
gdn_status gdn_ddtree_build(const float* logp, int32_t depth_max, int32_t top_k, int32_t budget, double tau,
                            int32_t flags, int32_t* parent, int32_t* depth, int32_t* rank, double* score,
                            int32_t* n_out);
gdn_status gdn_ddtree_build_batch(const float* logp, int32_t B, int32_t depth_max, int32_t top_k, int32_t budget,
                                  double tau, int32_t flags, int32_t n_max, int32_t* parents, int32_t* n);

typedef struct {
  int32_t B;               /* requests */
  int32_t n_max;           /* node stride of every per-node array */
  int32_t nb_max;          /* slot stride of boundary_states (>= every request's n_boundary) */
  int32_t depth_max;       /* deepest node of any tree, as the packers return it (0: unknown); trees
                              deeper than GDN_UT_MAX_DEPTH verify by walking chains (gdn_tree_verify) */
  const int32_t* words;    /* device, B * gdn_schedule_words(n_max) int32 */
} gdn_batch_schedule;
#define GDN_UT_MAX_DEPTH 24

/* ---------------------------------------------------------------------------
 * Double-buffered FP32 factor banks (SpecLA article, "接受因子缓存": per node
 * the normalised key, the delta-rule update vector u -- the "residual" that
 * gives T <- g T + k u^T exactly --, the log-gate and the raw conv input; two
 * banks alternate between "pending, consumed by the next verify" and "being
 * written by this verify").
 *
 * Device buffers (caller-allocated, fp32):
 *   k[i] [B][layers][n_max][Hk][dk]    u[i] [B][layers][n_max][Hv][dv]
 *   a[i] [B][layers][n_max][Hv]        x[i] [B][layers][n_max][C]  (C = 2 Hk dk + Hv dv;
 *                                           only read/written in conv_mode 1, may be NULL otherwise)
 *   pend_path [B][n_max] int32, pend_len [B] int32: the accepted path recorded by
 *   gdn_commit_fold -- node index in the low 16 bits, bit 30 set where the path
 *   enters a node whose parent's state the verify materialised (node flags bit 0
 *   of the parent); err [4] int32, zeroed by the caller
 *   before first use.
 * Host fields (set by gdn_banks_init, then advanced by the calls):
 *   write_bank: bank the next verify writes; pend_bank: bank holding the
 *   committed-but-not-folded path (-1: none); verified_bank: bank written by
 *   the last verify not yet committed (-1: none).
 * ------------------------------------------------------------------------- */
typedef struct {
  float* k[2];
  float* u[2];
  float* a[2];
  float* x[2];
  int32_t* pend_path;
  int32_t* pend_len;
  int32_t* err;
  int32_t B, layers, n_max;           /* capacity the buffers were sized for */
  int32_t write_bank, pend_bank, verified_bank;
} gdn_banks;

gdn_status gdn_banks_init(gdn_banks* banks, int32_t B, int32_t layers, int32_t n_max);

/* Workspace gdn_tree_verify needs (bytes): the normalised q and the v rows of
 * every node, fp32.  Pass a device buffer of at least this size. */
size_t gdn_workspace_bytes(const gdn_dims* d, int32_t B, int32_t layers, int32_t n_max);

#define GDN_VERIFY_BOUNDARY_SCRATCH 1   /* boundary_states is scratch, not output */
#define GDN_VERIFY_CHAIN_WALK 2         /* walk the heavy-light chains instead of the tree-masked UT form */
#define GDN_VERIFY_UT_SIMT 4            /* UT form on the CUDA cores even where the tensor-core kernel applies */
#define GDN_VERIFY_TC_PER_HEAD 8        /* tensor-core UT form with one CTA per v-head instead of the persistent kernel */
#define GDN_VERIFY_CHAINS 16            /* every tree is a pure chain (parent[i] = i - 1): chains of up to 64 nodes are
                                           solved on the tensor cores in 16-node segments (d_v = 128); a tree that is
                                           not a chain sets GDN_DEVERR_SCHEDULE and is skipped */

/* ---------------------------------------------------------------------------
 * gdn_tree_verify -- fold the pending path, then verify a batch of trees.
 * SpecLA article, "延迟融合提交" and "状态驻留验证".
 *
 * If a committed path is pending (banks->pend_bank >= 0) its factors are first
 * folded into each head's state tile as it is loaded -- T <- exp(a_t) T + k_t u_t^T
 * along the path, and the conv window takes the path's last K-1 raw rows -- and
 * the committed state and conv window are written back once.  Every node of
 * every tree is then advanced from its parent's state, in the walk order of the
 * packed ops: each chain of the heavy-light schedule keeps its tile in
 * registers from head to tail, and branch states wait in tensor memory.
 *
 *   x_raw      [B][layers][n_max][C]       in_dtype (bf16 or fp32)
 *   conv_w     [layers][C][K]              fp32 (conv_mode 1; else may be NULL)
 *   beta       [B][layers][n_max][Hv]      in_dtype
 *   log_g      [B][layers][n_max][Hv]      in_dtype, a = log of the decay gate
 *   state      [B][layers][Hv][dk][dv]     fp32 in/out: committed state (T = S^T)
 *   conv_state [B][layers][K-1][C]         fp32 in/out: committed raw rows, oldest first (conv_mode 1)
 *   out_o      [B][layers][n_max][Hv][dv]  fp32 out: o of every node
 *   boundary_states [B][layers][nb_max][Hv][dk][dv] fp32 out: the state after each
 *              boundary node, by slot.  May be NULL only if no tree has a boundary.
 *              With GDN_VERIFY_BOUNDARY_SCRATCH in flags it is scratch instead: only
 *              stashes that spill out of tensor memory are written there, and its
 *              contents are unspecified on return.
 *   flags      GDN_VERIFY_BOUNDARY_SCRATCH, GDN_VERIFY_CHAIN_WALK, GDN_VERIFY_UT_SIMT,
 *              GDN_VERIFY_TC_PER_HEAD, GDN_VERIFY_CHAINS (other
 *              bits: GDN_ERR_INVALID_ARG).  By default the nodes are solved in the tree-masked
 *              UT form (article "状态驻留验证": the topology-masked UT decomposition): the
 *              committed state times every node's k and q, with no dependency between nodes,
 *              then a substitution over ancestor pairs.  Where dv = 128 and n_max <= 32, or
 *              dk is 64 or 128, n_max <= 64 and sched->depth_max <= 16, those products (and
 *              for the larger trees the nodes' Gram rows) run on the tensor cores (tcgen05, tf32
 *              split in three for fp32 accuracy); elsewhere, or with GDN_VERIFY_UT_SIMT, on the
 *              CUDA cores.  GDN_VERIFY_CHAIN_WALK walks the packed ops instead: heavy-light chains
 *              in registers, branch states stashed in tensor memory.  All give the same results
 *              up to rounding.  Batches whose sched->depth_max exceeds GDN_UT_MAX_DEPTH walk
 *              chains without the flag: the UT form's per-node work grows with the square of
 *              the depth.  GDN_VERIFY_CHAINS (the caller guarantees that every tree is a chain)
 *              solves chains of up to 64 nodes (dk 64 or 128) in the chunked UT form instead (SpecLA article,
 *              "想深入源码": the chunked Gated DeltaNet form): each 16-node segment is solved
 *              from the running state on the tensor cores, which then absorbs the segment with
 *              the fold's operations.
 *   banks      factors of every node are written into bank write_bank
 *   workspace  >= gdn_workspace_bytes(d, B, layers, n_max) bytes of device memory
 * Rows of nodes >= n[b] are neither read nor written.
 * ------------------------------------------------------------------------- */
gdn_status gdn_tree_verify(const gdn_dims* d, int32_t layers, const gdn_batch_schedule* sched,
                           const void* x_raw, const float* conv_w, const void* beta, const void* log_g,
                           float* state, float* conv_state, float* out_o, float* boundary_states,
                           gdn_banks* banks, void* workspace, size_t workspace_bytes, int32_t flags,
                           cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gdn_tree_verify_noalloc -- gdn_tree_verify without a workspace argument, for
 * callers that cannot allocate device memory where they verify: code running
 * during stream capture (cudaMalloc is not allowed there), engines whose whole
 * device pool belongs to their own allocator, plugins given only buffers and a
 * stream.  The SpecLA article has no counterpart; this is a convenience of this
 * library.
 *
 * Same arguments, semantics and errors as gdn_tree_verify, except that the
 * q/v scratch lives in a fixed array inside the library: GDN_NOALLOC_SCRATCH_BYTES
 * on every GPU that loads the library, kept until the process exits.  A batch
 * whose gdn_workspace_bytes exceeds it is rejected with GDN_ERR_CAPACITY before
 * anything runs (Qwen-like heads: B * layers * n_max <= 2047).  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current, so make it outside any stream capture and with the stream's
 * device current.  Every call shares the array: calls whose kernels may overlap
 * on the GPU race and must be serialised by the caller.  Nothing in the array
 * needs clearing: every scratch row read is written earlier in the same call.
 * ------------------------------------------------------------------------- */
#define GDN_NOALLOC_SCRATCH_BYTES (64u << 20)
gdn_status gdn_tree_verify_noalloc(const gdn_dims* d, int32_t layers, const gdn_batch_schedule* sched,
                                   const void* x_raw, const float* conv_w, const void* beta, const void* log_g,
                                   float* state, float* conv_state, float* out_o, float* boundary_states,
                                   gdn_banks* banks, int32_t flags, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gdn_commit_fold -- record the accepted path of the last verify as pending.
 * SpecLA article, "延迟融合提交" and "接受因子缓存".
 *
 * path [B][sched->n_max] and len [B] are device int32 (so acceptance computed on
 * the GPU needs no host round trip).  A valid path has path[0] = 0 and
 * parent[path[i]] = path[i-1], 0 <= len <= n; len = 0 commits nothing.  The
 * path is checked on the device: an invalid one commits nothing for that
 * request and sets GDN_DEVERR_INVALID_PATH.  No state is touched: the fold
 * happens in the next gdn_tree_verify (or gdn_finish), which reads the factors
 * at the path's node indices, so no factor is copied whatever the path's shape.
 * With flags & GDN_COMMIT_COMPACT the bank is also compacted in place into path
 * order (slot i <- slot path[i]) and the recorded path becomes 0..len-1.
 * Returns GDN_ERR_STATE if no verify happened since the last commit.
 * ------------------------------------------------------------------------- */
#define GDN_COMMIT_COMPACT 1
gdn_status gdn_commit_fold(const gdn_dims* d, int32_t layers, const gdn_batch_schedule* sched,
                           const int32_t* path, const int32_t* len, int32_t flags,
                           gdn_banks* banks, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gdn_finish -- materialise the pending path once (end of generation, switch to
 * plain decoding, cancellation).  SpecLA article, "延迟融合提交"
 * (finish_speculative_state).  Folds the pending factors into state and the
 * pending raw rows into conv_state, exactly as the next verify would; a no-op
 * when nothing is pending.
 * ------------------------------------------------------------------------- */
gdn_status gdn_finish(const gdn_dims* d, int32_t B, int32_t layers, float* state, float* conv_state,
                      gdn_banks* banks, cudaStream_t stream);

/* Synchronise the stream, read and clear banks->err.  Returns GDN_OK or the
 * status of a device error: GDN_ERR_INVALID_PATH, GDN_ERR_TIMEOUT or
 * GDN_ERR_SCHEDULE, checked in that order. */
gdn_status gdn_check_error(gdn_banks* banks, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * gdn_selftest_wait_timeout -- exercises the give-up path of the library's
 * bounded waits.  The source pages have no counterpart: this is a test hook.
 *
 * Launches one CTA on `stream` that arms an mbarrier for 16 bytes no copy
 * will deliver and waits on it with the same bound as every wait in the
 * verify kernels (2^28 clock cycles, ~0.13 s).  The wait gives up, the CTA
 * sets GDN_DEVERR_TIMEOUT in banks->err (request 0) and returns; nothing
 * faults or traps, and the context stays usable.  gdn_check_error() then
 * reports GDN_ERR_TIMEOUT and clears the word.  The bit is sticky (see the
 * conventions above): until gdn_check_error() clears it, verify and finish
 * calls on the same banks do no work, so only call this on banks whose state
 * may be discarded, and check the error before verifying with them again.
 *   banks  only banks->err is used (device, >= 2 int32, 16-byte aligned)
 * Returns GDN_OK once launched; GDN_ERR_INVALID_ARG for a NULL or misaligned
 * error word, GDN_ERR_CUDA if the launch fails.
 * ------------------------------------------------------------------------- */
gdn_status gdn_selftest_wait_timeout(gdn_banks* banks, cudaStream_t stream);

/* Thread-local description of the last failed call on this thread. */
const char* gdn_last_error(void);

int32_t gdn_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GDN_TREE_H */
