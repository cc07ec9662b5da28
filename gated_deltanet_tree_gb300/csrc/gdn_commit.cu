// Commit of an accepted path: device-side check and pending record, and the
// optional DFS-to-path compaction of a factor bank.
//
// SpecLA article, "接受因子缓存": when acceptance follows a chain the banks just
// swap roles with no device copy; on a fork a compaction kernel gathers the
// factors at arbitrary DFS indices back into path order.  Here the next fold
// gathers by node index itself, so recording the path is enough for every
// accepted shape; the compaction remains available for callers that want the
// bank in path order.
#include "gdn_internal.h"

namespace gdn {
namespace {

// One thread per request: check that path[b] is a root path of tree b and
// record it as pending.  An invalid path records nothing (len 0) and flags err.
__global__ void commit_record_kernel(CommitParams p) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  const SchedLayout lay{p.n_max};
  const int32_t* rec = p.words + static_cast<size_t>(b) * lay.words();
  const int n = rec[0];
  const int32_t* parent = rec + lay.parent();
  const int32_t* path = p.path + static_cast<size_t>(b) * p.n_max;
  const int L = p.len[b];
  bool ok = L >= 0 && L <= n;
  int prev = -1;
  for (int i = 0; ok && i < L; ++i) {
    const int v = path[i];
    ok = (i == 0) ? (v == 0) : (v > 0 && v < n && parent[v] == prev);
    prev = v;
  }
  int32_t* pp = p.pend_path + static_cast<size_t>(b) * p.n_max;
  if (ok) {
    const int32_t* nflags = rec + lay.nflags();
    for (int i = 0; i < L; ++i)
      pp[i] = path[i] | ((i > 0 && (nflags[path[i - 1]] & kNodeMaterialised)) ? kPathHeadFlag : 0);
    p.pend_len[b] = L;
  } else {
    p.pend_len[b] = 0;
    device_error(p.err, GDN_DEVERR_INVALID_PATH, b);
  }
}

// In-place compaction of one (request, layer) bank: slot i <- slot path[i].
// path[i] >= i for a root path in topological numbering, so a forward pass
// never reads a slot it has already overwritten; each thread owns a fixed
// element offset of the slot and walks i in order.
__device__ __forceinline__ void compact_field(float* base, int words, const int32_t* path, int L) {
  for (int e = threadIdx.x; e < words; e += blockDim.x)
    for (int i = 0; i < L; ++i) {
      const int src = path[i] & kPathNodeMask;
      if (src != i) base[static_cast<size_t>(i) * words + e] = base[static_cast<size_t>(src) * words + e];
    }
}

__global__ void commit_compact_kernel(CommitParams p) {
  const int bl = blockIdx.x;
  const int b = bl / p.layers;
  const int L = p.pend_len[b];
  const int32_t* path = p.pend_path + static_cast<size_t>(b) * p.n_max;
  bool ident = true;
  for (int i = 0; i < L; ++i) ident = ident && (path[i] & kPathNodeMask) == i;
  if (ident) return;
  const size_t node0 = static_cast<size_t>(bl) * p.n_max;
  switch (blockIdx.y) {
    case 0: compact_field(p.k + node0 * p.k_words, p.k_words, path, L); break;
    case 1: compact_field(p.u + node0 * p.u_words, p.u_words, path, L); break;
    case 2: compact_field(p.a + node0 * p.a_words, p.a_words, path, L); break;
    default:
      if (p.x) compact_field(p.x + node0 * p.x_words, p.x_words, path, L);
      break;
  }
}

// After compaction the recorded path is the identity (chain-head flags kept).
__global__ void commit_identity_kernel(CommitParams p) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  int32_t* pp = p.pend_path + static_cast<size_t>(b) * p.n_max;
  const int L = p.pend_len[b];
  for (int i = 0; i < L; ++i) pp[i] = i | (pp[i] & kPathHeadFlag);
}

}  // namespace

cudaError_t launch_commit(const CommitParams& p, int compact, cudaStream_t s) {
  const int threads = 128;
  const int blocks = (p.B + threads - 1) / threads;
  commit_record_kernel<<<blocks, threads, 0, s>>>(p);
  if (compact) {
    commit_compact_kernel<<<dim3(p.B * p.layers, 4), 256, 0, s>>>(p);
    commit_identity_kernel<<<blocks, threads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace gdn
