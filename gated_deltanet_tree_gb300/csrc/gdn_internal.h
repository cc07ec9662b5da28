// Internal declarations shared by the translation units of the library.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "gdn_tree.h"

namespace gdn {

// Thread-local error message; returns `st` so callers can `return fail(...)`.
gdn_status fail(gdn_status st, const char* fmt, ...);
void clear_error();

#ifdef __CUDACC__
// Flags a device-side error without trapping: bit into err[0], 1 + request into err[1].
__device__ __forceinline__ void device_error(int32_t* err, int bit, int b) {
  atomicOr(&err[0], bit);
  atomicCAS(&err[1], 0, b + 1);
}

// ---- TMA bulk copies completing on an mbarrier (shared by the kernels) ----
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// Global -> shared bulk copy completing on `bar` (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}
constexpr long long kWaitCycles = 1ll << 28;   // ~0.13 s; a healthy copy completes in microseconds
// Bounded wait for phase `parity` of `bar`; false on timeout (the caller flags GDN_DEVERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if (clock64() - t0 > kWaitCycles) return false;
  }
}
// True once some CTA of this launch gave up on a wait: later CTAs exit at once.
__device__ __forceinline__ bool launch_aborted(const int32_t* err) {
  return (*reinterpret_cast<const volatile int32_t*>(err) & GDN_DEVERR_TIMEOUT) != 0;
}
#endif

// Offsets inside one packed schedule record (see gdn_tree.h).
struct SchedLayout {
  int n_max;
  __host__ __device__ int words() const { return 5 + 4 * n_max; }
  __host__ __device__ int parent() const { return 5; }
  __host__ __device__ int bslot() const { return 5 + n_max; }
  __host__ __device__ int nflags() const { return 5 + 2 * n_max; }
  __host__ __device__ int ops() const { return 5 + 3 * n_max; }
};

// One verify op per node, in the order the verify walks the tree (see gdn_tree.h).
constexpr int32_t kOpNode = 0xFF;             // node index
constexpr int32_t kOpReload = 1 << 8;         // start from the parent's stashed state (else: the registers)
constexpr int32_t kOpReloadGlobal = 1 << 9;   // ... stashed in the parent's boundary slot (else: tensor memory)
constexpr int kOpReloadLevelShift = 10;       // 2 bits: tensor-memory level of the reload
constexpr int32_t kOpPush = 1 << 12;          // after the node: materialise and stash its state
constexpr int32_t kOpPushGlobal = 1 << 13;    // ... in the node's boundary slot (else: tensor memory)
constexpr int kOpPushLevelShift = 14;         // 2 bits: tensor-memory level of the push
constexpr int32_t kOpLeaf = 1 << 16;          // no children: the node's update is never read
constexpr int kTmemLevels = 2;                // stash levels kept in tensor memory; deeper ones spill to HBM
// nflags bit: the state after this node is materialised (the verify stashed it)
constexpr int32_t kNodeMaterialised = 1;

// Encoding of a recorded pending-path entry: node index in the low bits; the
// head flag marks a node entered from a materialised state (its parent's state
// was stashed by the verify), where the fold materialises as well.
constexpr int32_t kPathNodeMask = 0xFFFF;
constexpr int32_t kPathHeadFlag = 1 << 30;

struct ConvParams {
  int B, layers, n_max;
  const int32_t* words;        // packed schedules; nullptr: fold only
  int Hk, Hv, dk, dv, K, C, conv_mode, act, in_dtype;
  float q_scale, l2_eps;
  const void* x_raw;           // [B][L][n_max][C]
  const float* conv_w;         // [L][C][K]
  float* conv_state;           // [B][L][K-1][C]
  int fold;                    // fold the pending path's raw rows into conv_state first
  const float* pend_x;         // pending bank x
  const int32_t* pend_path;    // [B][n_max]
  const int32_t* pend_len;     // [B]
  float* q_out;                // workspace q  [B][L][n_max][Hk][dk]
  float* v_out;                // workspace v  [B][L][n_max][Hv][dv]
  float* k_out;                // write bank k [B][L][n_max][Hk][dk]
  float* x_out;                // write bank x [B][L][n_max][C]
  int32_t* err;                // device error words
};

struct VerifyParams {
  int B, layers, n_max, nb_max;
  const int32_t* words;        // packed schedules; nullptr: fold only
  int Hk, Hv, dk, dv, R, in_dtype;
  const void* beta;            // [B][L][n_max][Hv]
  const void* log_g;           // [B][L][n_max][Hv]
  const float* q_in;           // workspace q
  const float* v_in;           // workspace v
  const float* k_in;           // write bank k (normalised keys of this tree)
  float* u_out;                // write bank u [B][L][n_max][Hv][dv]
  float* a_out;                // write bank a [B][L][n_max][Hv]
  float* state;                // [B][L][Hv][dk][dv]
  float* out_o;                // [B][L][n_max][Hv][dv]
  float* boundary;             // [B][L][nb_max][Hv][dk][dv]
  int boundary_out;            // store every boundary state (else the slots only take spills)
  int chain_walk;              // the heavy-light chain walk (else the tree-masked UT form)
  int fold;
  const float* pend_k;
  const float* pend_u;
  const float* pend_a;
  const int32_t* pend_path;
  const int32_t* pend_len;
  int32_t* err;                // device error words
  int prefetch_ahead;          // CTAs ahead whose inputs a CTA prefetches into L2 (0: none)
};

struct CommitParams {
  int B, layers, n_max;
  const int32_t* words;
  const int32_t* path;         // [B][n_max]
  const int32_t* len;          // [B]
  int32_t* pend_path;
  int32_t* pend_len;
  int32_t* err;
  // compaction (in place in one bank)
  float* k; float* u; float* a; float* x;
  int k_words, u_words, a_words, x_words;   // floats per node of each field
};

cudaError_t launch_conv(const ConvParams& p, cudaStream_t s);
cudaError_t launch_verify(const VerifyParams& p, cudaStream_t s);      // chain walk; also the fold-only launches
cudaError_t launch_verify_ut(const VerifyParams& p, cudaStream_t s);   // tree-masked UT form, CUDA cores
cudaError_t launch_verify_tc(const VerifyParams& p, cudaStream_t s);   // tree-masked UT form, tensor cores, a CTA per head
bool verify_tc_supported(int dk, int dv, int n_max);
// the same, persistent and warp-specialised.  mode 0: trees of up to 32 nodes; 1: every tree a pure chain of
// up to 64 nodes, solved in 16-node segments; 2: trees of up to 64 nodes and depth at most 16
cudaError_t launch_verify_tcp(const VerifyParams& p, int mode, cudaStream_t s);
bool verify_tcp_supported(int dk, int dv, int n_max, int mode);
constexpr int kWideMaxDepth = 16;   // deepest node mode 2 takes

cudaError_t launch_commit(const CommitParams& p, int compact, cudaStream_t s);
bool verify_supported(int dk, int dv);

}  // namespace gdn
