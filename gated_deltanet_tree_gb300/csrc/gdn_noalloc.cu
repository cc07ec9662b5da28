// gdn_tree_verify_noalloc: the verify call for callers that cannot allocate
// device memory.
//
// gdn_tree_verify needs a caller-provided workspace for the normalised q and the
// v rows of every node.  Some callers have no way to provide one at the point
// where they verify:
//   - code that runs while a stream is being captured into a CUDA graph, where
//     cudaMalloc is not a permitted call;
//   - engines that reserve the whole device pool up front for their own
//     allocator and forbid any other allocation;
//   - plugins hosted by a framework that hands them only input/output buffers
//     and a stream, with no allocator to call.
// This entry point takes no workspace.  It uses a fixed scratch array that is
// part of the library image: GDN_NOALLOC_SCRATCH_BYTES (64 MiB) on every GPU
// that loads the library, held until the process exits.
//
// The array is shared by every call.  The conv-window kernel writes every
// scratch row the verify kernel of the same call later uses (rows of nodes
// beyond a tree's size may be copied along but are never used), so nothing
// needs clearing between calls; but
// two calls whose kernels overlap on the GPU (different streams, or different
// host threads on one device) race on the same array and must be serialised
// by the caller.
#include <mutex>

#include "gdn_internal.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_on_device[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached.
gdn_status scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gdn::fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return gdn::fail(GDN_ERR_UNSUPPORTED, "device ordinal %d outside 0..%d", dev, kMaxDevices - 1);
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_on_device[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return gdn::fail(GDN_ERR_CUDA, "cudaGetSymbolAddress of the fixed scratch array: %s", cudaGetErrorString(e));
    g_scratch_on_device[dev] = p;
  }
  *out = g_scratch_on_device[dev];
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_tree_verify_noalloc(const gdn_dims* d, int32_t layers, const gdn_batch_schedule* sched,
                                              const void* x_raw, const float* conv_w, const void* beta,
                                              const void* log_g, float* state, float* conv_state, float* out_o,
                                              float* boundary_states, gdn_banks* banks, int32_t flags,
                                              cudaStream_t stream) {
  gdn::clear_error();
  if (!d || !sched) return gdn::fail(GDN_ERR_INVALID_ARG, "dims or schedule is NULL");
  if (layers < 1 || sched->B < 1 || sched->n_max < 1)
    return gdn::fail(GDN_ERR_INVALID_ARG, "B = %d, layers = %d, n_max = %d", sched->B, layers, sched->n_max);
  const size_t need = gdn_workspace_bytes(d, sched->B, layers, sched->n_max);
  if (need == 0) return gdn::fail(GDN_ERR_INVALID_ARG, "invalid dims");
  if (need > GDN_NOALLOC_SCRATCH_BYTES)
    return gdn::fail(GDN_ERR_CAPACITY,
                     "gdn_tree_verify_noalloc: this batch (B=%d, layers=%d, n_max=%d) needs %zu bytes of scratch, "
                     "the fixed scratch holds %zu; split the batch or call gdn_tree_verify with a workspace",
                     sched->B, layers, sched->n_max, need, static_cast<size_t>(GDN_NOALLOC_SCRATCH_BYTES));
  void* ws = nullptr;
  gdn_status st = scratch_on_current_device(&ws);
  if (st != GDN_OK) return st;
  return gdn_tree_verify(d, layers, sched, x_raw, conv_w, beta, log_g, state, conv_state, out_o, boundary_states,
                         banks, ws, GDN_NOALLOC_SCRATCH_BYTES, flags, stream);
}
