// extern "C" entry points: argument checks, the factor-bank lifecycle and the
// kernel launches.  No entry point allocates memory or synchronises the host
// except gdn_check_error.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "gdn_internal.h"

namespace gdn {
namespace {
thread_local char g_msg[512] = "";
}

gdn_status fail(gdn_status st, const char* fmt, ...) {
  char tmp[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(tmp, sizeof(tmp), fmt, ap);
  va_end(ap);
  std::memcpy(g_msg, tmp, sizeof(tmp));
  return st;
}

void clear_error() { g_msg[0] = '\0'; }

}  // namespace gdn

using gdn::fail;

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define GDN_CHECK_PTR(ptr, name)                                                         \
  do {                                                                                   \
    if ((ptr) == nullptr) return fail(GDN_ERR_INVALID_ARG, "%s is NULL", name);          \
    if (!aligned16(ptr)) return fail(GDN_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
  } while (0)

int channels(const gdn_dims* d) { return 2 * d->Hk * d->dk + d->Hv * d->dv; }

gdn_status check_dims(const gdn_dims* d) {
  if (!d) return fail(GDN_ERR_INVALID_ARG, "dims is NULL");
  if (d->Hk < 1 || d->Hv < 1 || d->Hv % d->Hk != 0)
    return fail(GDN_ERR_INVALID_ARG, "heads Hk = %d, Hv = %d: need Hk >= 1 and Hv a multiple of Hk", d->Hk, d->Hv);
  if (!gdn::verify_supported(d->dk, d->dv))
    return fail(GDN_ERR_UNSUPPORTED, "head sizes dk = %d, dv = %d: supported are 32, 64 and 128", d->dk, d->dv);
  if (d->conv_mode != 0 && d->conv_mode != 1) return fail(GDN_ERR_INVALID_ARG, "conv_mode = %d", d->conv_mode);
  if (d->act != 0 && d->act != 1) return fail(GDN_ERR_INVALID_ARG, "act = %d", d->act);
  if (d->in_dtype != GDN_DTYPE_F32 && d->in_dtype != GDN_DTYPE_BF16)
    return fail(GDN_ERR_INVALID_ARG, "in_dtype = %d", d->in_dtype);
  if (d->conv_mode == 1 && (d->K < 1 || d->K > GDN_MAX_TAPS))
    return fail(GDN_ERR_UNSUPPORTED, "conv taps K = %d outside 1..%d", d->K, GDN_MAX_TAPS);
  if (!std::isfinite(d->q_scale) || !std::isfinite(d->l2_eps) || d->l2_eps < 0.f)
    return fail(GDN_ERR_INVALID_ARG, "q_scale / l2_eps not finite or eps negative");
  return GDN_OK;
}

gdn_status check_sched(const gdn_batch_schedule* s) {
  if (!s) return fail(GDN_ERR_INVALID_ARG, "schedule is NULL");
  if (s->B < 1) return fail(GDN_ERR_INVALID_ARG, "schedule B = %d", s->B);
  if (s->n_max < 1 || s->n_max > GDN_MAX_NODES)
    return fail(GDN_ERR_UNSUPPORTED, "n_max = %d outside 1..%d", s->n_max, GDN_MAX_NODES);
  if (s->nb_max < 0 || s->nb_max > s->n_max) return fail(GDN_ERR_INVALID_ARG, "nb_max = %d", s->nb_max);
  GDN_CHECK_PTR(s->words, "schedule words");
  return GDN_OK;
}

gdn_status check_banks(const gdn_banks* bk, int B, int layers, int n_max) {
  if (!bk) return fail(GDN_ERR_INVALID_ARG, "banks is NULL");
  if (bk->B != B || bk->layers != layers || bk->n_max != n_max)
    return fail(GDN_ERR_CAPACITY, "banks sized for B=%d layers=%d n_max=%d, call has B=%d layers=%d n_max=%d", bk->B,
                bk->layers, bk->n_max, B, layers, n_max);
  if (bk->write_bank != 0 && bk->write_bank != 1) return fail(GDN_ERR_STATE, "banks not initialised (write_bank)");
  if (bk->pend_bank != -1 && bk->pend_bank != 1 - bk->write_bank)
    return fail(GDN_ERR_STATE, "banks lifecycle corrupted (pend_bank = %d, write_bank = %d)", bk->pend_bank,
                bk->write_bank);
  GDN_CHECK_PTR(bk->pend_path, "banks.pend_path");
  GDN_CHECK_PTR(bk->pend_len, "banks.pend_len");
  GDN_CHECK_PTR(bk->err, "banks.err");
  return GDN_OK;
}

gdn_status check_bank_fields(const gdn_banks* bk, const gdn_dims* d, int i, const char* which) {
  char name[64];
  std::snprintf(name, sizeof(name), "banks.k[%d] (%s)", i, which);
  GDN_CHECK_PTR(bk->k[i], name);
  std::snprintf(name, sizeof(name), "banks.u[%d] (%s)", i, which);
  GDN_CHECK_PTR(bk->u[i], name);
  std::snprintf(name, sizeof(name), "banks.a[%d] (%s)", i, which);
  GDN_CHECK_PTR(bk->a[i], name);
  if (d->conv_mode == 1) {
    std::snprintf(name, sizeof(name), "banks.x[%d] (%s)", i, which);
    GDN_CHECK_PTR(bk->x[i], name);
  }
  return GDN_OK;
}

gdn_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t ws_q_bytes(const gdn_dims* d, int B, int layers, int n_max) {
  return round_up(static_cast<size_t>(B) * layers * n_max * d->Hk * d->dk * sizeof(float), kAlign);
}

}  // namespace

#define GDN_TRY(expr)                 \
  do {                                \
    gdn_status st_ = (expr);          \
    if (st_ != GDN_OK) return st_;    \
  } while (0)

extern "C" {

int32_t gdn_abi_version(void) { return GDN_ABI_VERSION; }

const char* gdn_last_error(void) { return gdn::g_msg; }

gdn_status gdn_banks_init(gdn_banks* banks, int32_t B, int32_t layers, int32_t n_max) {
  gdn::clear_error();
  if (!banks) return fail(GDN_ERR_INVALID_ARG, "banks is NULL");
  if (B < 1 || layers < 1 || n_max < 1 || n_max > GDN_MAX_NODES)
    return fail(GDN_ERR_INVALID_ARG, "B = %d, layers = %d, n_max = %d", B, layers, n_max);
  banks->B = B;
  banks->layers = layers;
  banks->n_max = n_max;
  banks->write_bank = 0;
  banks->pend_bank = -1;
  banks->verified_bank = -1;
  return GDN_OK;
}

size_t gdn_workspace_bytes(const gdn_dims* d, int32_t B, int32_t layers, int32_t n_max) {
  if (!d || B < 1 || layers < 1 || n_max < 1) return 0;
  return ws_q_bytes(d, B, layers, n_max) +
         round_up(static_cast<size_t>(B) * layers * n_max * d->Hv * d->dv * sizeof(float), kAlign);
}

gdn_status gdn_tree_verify(const gdn_dims* d, int32_t layers, const gdn_batch_schedule* sched, const void* x_raw,
                           const float* conv_w, const void* beta, const void* log_g, float* state,
                           float* conv_state, float* out_o, float* boundary_states, gdn_banks* banks,
                           void* workspace, size_t workspace_bytes, int32_t flags, cudaStream_t stream) {
  gdn::clear_error();
  if (flags & ~(GDN_VERIFY_BOUNDARY_SCRATCH | GDN_VERIFY_CHAIN_WALK | GDN_VERIFY_UT_SIMT | GDN_VERIFY_TC_PER_HEAD |
                GDN_VERIFY_CHAINS))
    return fail(GDN_ERR_INVALID_ARG, "unknown verify flags 0x%x", flags);
  GDN_TRY(check_dims(d));
  GDN_TRY(check_sched(sched));
  if (layers < 1) return fail(GDN_ERR_INVALID_ARG, "layers = %d", layers);
  const int B = sched->B, n_max = sched->n_max;
  GDN_TRY(check_banks(banks, B, layers, n_max));
  GDN_CHECK_PTR(x_raw, "x_raw");
  GDN_CHECK_PTR(beta, "beta");
  GDN_CHECK_PTR(log_g, "log_g");
  GDN_CHECK_PTR(state, "state");
  GDN_CHECK_PTR(out_o, "out_o");
  GDN_CHECK_PTR(workspace, "workspace");
  if (d->conv_mode == 1) {
    GDN_CHECK_PTR(conv_w, "conv_w");
    if (d->K > 1) GDN_CHECK_PTR(conv_state, "conv_state");
  }
  if (sched->nb_max > 0) GDN_CHECK_PTR(boundary_states, "boundary_states");
  const size_t need = gdn_workspace_bytes(d, B, layers, n_max);
  if (workspace_bytes < need)
    return fail(GDN_ERR_CAPACITY, "workspace holds %zu bytes, the call needs %zu", workspace_bytes, need);
  const int cur = banks->write_bank;
  const int pend = banks->pend_bank;
  GDN_TRY(check_bank_fields(banks, d, cur, "write bank"));
  if (pend >= 0) GDN_TRY(check_bank_fields(banks, d, pend, "pending bank"));

  float* ws_q = static_cast<float*>(workspace);
  float* ws_v = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws_q_bytes(d, B, layers, n_max));

  gdn::ConvParams cp{};
  cp.B = B; cp.layers = layers; cp.n_max = n_max; cp.words = sched->words;
  cp.Hk = d->Hk; cp.Hv = d->Hv; cp.dk = d->dk; cp.dv = d->dv; cp.K = d->conv_mode ? d->K : 1;
  cp.C = channels(d); cp.conv_mode = d->conv_mode; cp.act = d->act; cp.in_dtype = d->in_dtype;
  cp.q_scale = d->q_scale; cp.l2_eps = d->l2_eps;
  cp.x_raw = x_raw; cp.conv_w = conv_w; cp.conv_state = conv_state;
  cp.fold = pend >= 0;
  cp.pend_x = pend >= 0 ? banks->x[pend] : nullptr;
  cp.pend_path = banks->pend_path; cp.pend_len = banks->pend_len;
  cp.q_out = ws_q; cp.v_out = ws_v; cp.k_out = banks->k[cur]; cp.x_out = banks->x[cur]; cp.err = banks->err;
  cudaError_t e = gdn::launch_conv(cp, stream);
  if (e != cudaSuccess) return cuda_fail(e, "conv-window launch");

  gdn::VerifyParams vp{};
  vp.B = B; vp.layers = layers; vp.n_max = n_max; vp.nb_max = sched->nb_max; vp.words = sched->words;
  vp.Hk = d->Hk; vp.Hv = d->Hv; vp.dk = d->dk; vp.dv = d->dv; vp.R = d->Hv / d->Hk; vp.in_dtype = d->in_dtype;
  vp.beta = beta; vp.log_g = log_g; vp.q_in = ws_q; vp.v_in = ws_v; vp.k_in = banks->k[cur];
  vp.u_out = banks->u[cur]; vp.a_out = banks->a[cur];
  vp.state = state; vp.out_o = out_o; vp.boundary = boundary_states;
  vp.boundary_out = (flags & GDN_VERIFY_BOUNDARY_SCRATCH) ? 0 : 1;
  // the UT form costs depth^2 per node and depth per (node, column): deep trees walk their chains, unless
  // the caller says every tree is a chain, which the tensor cores then solve in 16-node segments
  const bool chains_tc = (flags & GDN_VERIFY_CHAINS) && !(flags & (GDN_VERIFY_CHAIN_WALK | GDN_VERIFY_UT_SIMT)) &&
                         gdn::verify_tcp_supported(d->dk, d->dv, n_max, 1);
  vp.chain_walk = !chains_tc && ((flags & GDN_VERIFY_CHAIN_WALK) || sched->depth_max > GDN_UT_MAX_DEPTH) ? 1 : 0;
  vp.fold = pend >= 0;
  if (pend >= 0) {
    vp.pend_k = banks->k[pend]; vp.pend_u = banks->u[pend]; vp.pend_a = banks->a[pend];
  }
  vp.pend_path = banks->pend_path; vp.pend_len = banks->pend_len; vp.err = banks->err;
  // trees of 33 to 64 nodes, none deeper than 16 (as the packers report it): one segment on the tensor cores
  const bool wide_tc = !chains_tc && !vp.chain_walk && n_max > 32 && sched->depth_max >= 1 &&
                       sched->depth_max <= gdn::kWideMaxDepth &&
                       !(flags & (GDN_VERIFY_UT_SIMT | GDN_VERIFY_TC_PER_HEAD)) &&
                       gdn::verify_tcp_supported(d->dk, d->dv, n_max, 2);
  if (chains_tc) {
    e = gdn::launch_verify_tcp(vp, 1, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tree-verify launch (tensor cores, chain segments)");
  } else if (wide_tc) {
    e = gdn::launch_verify_tcp(vp, 2, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tree-verify launch (tensor cores, up to 64 nodes)");
  } else if (vp.chain_walk) {
    e = gdn::launch_verify(vp, stream);
    if (e != cudaSuccess) return cuda_fail(e, "chain-verify launch");
  } else if (!(flags & (GDN_VERIFY_UT_SIMT | GDN_VERIFY_TC_PER_HEAD)) &&
             gdn::verify_tcp_supported(d->dk, d->dv, n_max, 0)) {
    e = gdn::launch_verify_tcp(vp, 0, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tree-verify launch (tensor cores, persistent)");
  } else if (!(flags & GDN_VERIFY_UT_SIMT) && gdn::verify_tc_supported(d->dk, d->dv, n_max)) {
    e = gdn::launch_verify_tc(vp, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tree-verify launch (tensor cores)");
  } else {
    e = gdn::launch_verify_ut(vp, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tree-verify launch");
  }

  banks->pend_bank = -1;
  banks->verified_bank = cur;
  return GDN_OK;
}

gdn_status gdn_commit_fold(const gdn_dims* d, int32_t layers, const gdn_batch_schedule* sched, const int32_t* path,
                           const int32_t* len, int32_t flags, gdn_banks* banks, cudaStream_t stream) {
  gdn::clear_error();
  GDN_TRY(check_dims(d));
  GDN_TRY(check_sched(sched));
  if (layers < 1) return fail(GDN_ERR_INVALID_ARG, "layers = %d", layers);
  GDN_TRY(check_banks(banks, sched->B, layers, sched->n_max));
  GDN_CHECK_PTR(path, "path");
  GDN_CHECK_PTR(len, "len");
  if (flags & ~GDN_COMMIT_COMPACT) return fail(GDN_ERR_INVALID_ARG, "unknown commit flags 0x%x", flags);
  const int vb = banks->verified_bank;
  if (vb < 0) return fail(GDN_ERR_STATE, "commit without a verify since the last commit");
  GDN_TRY(check_bank_fields(banks, d, vb, "verified bank"));

  gdn::CommitParams p{};
  p.B = sched->B; p.layers = layers; p.n_max = sched->n_max; p.words = sched->words;
  p.path = path; p.len = len; p.pend_path = banks->pend_path; p.pend_len = banks->pend_len; p.err = banks->err;
  p.k = banks->k[vb]; p.u = banks->u[vb]; p.a = banks->a[vb]; p.x = d->conv_mode == 1 ? banks->x[vb] : nullptr;
  p.k_words = d->Hk * d->dk; p.u_words = d->Hv * d->dv; p.a_words = d->Hv; p.x_words = channels(d);
  cudaError_t e = gdn::launch_commit(p, flags & GDN_COMMIT_COMPACT, stream);
  if (e != cudaSuccess) return cuda_fail(e, "commit launch");
  banks->pend_bank = vb;
  banks->write_bank = 1 - vb;
  banks->verified_bank = -1;
  return GDN_OK;
}

gdn_status gdn_finish(const gdn_dims* d, int32_t B, int32_t layers, float* state, float* conv_state,
                      gdn_banks* banks, cudaStream_t stream) {
  gdn::clear_error();
  GDN_TRY(check_dims(d));
  if (B < 1 || layers < 1) return fail(GDN_ERR_INVALID_ARG, "B = %d, layers = %d", B, layers);
  GDN_TRY(check_banks(banks, B, layers, banks ? banks->n_max : 0));
  const int pend = banks->pend_bank;
  if (pend < 0) return GDN_OK;
  GDN_CHECK_PTR(state, "state");
  if (d->conv_mode == 1 && d->K > 1) GDN_CHECK_PTR(conv_state, "conv_state");
  GDN_TRY(check_bank_fields(banks, d, pend, "pending bank"));

  cudaError_t e;
  if (d->conv_mode == 1 && d->K > 1) {
    gdn::ConvParams cp{};
    cp.B = B; cp.layers = layers; cp.n_max = banks->n_max; cp.words = nullptr;
    cp.Hk = d->Hk; cp.Hv = d->Hv; cp.dk = d->dk; cp.dv = d->dv; cp.K = d->K; cp.C = channels(d);
    cp.conv_mode = 1; cp.act = d->act; cp.in_dtype = d->in_dtype;
    cp.conv_state = conv_state; cp.fold = 1; cp.pend_x = banks->x[pend];
    cp.pend_path = banks->pend_path; cp.pend_len = banks->pend_len; cp.err = banks->err;
    cp.conv_w = nullptr;  // not read in fold-only mode
    e = gdn::launch_conv(cp, stream);
    if (e != cudaSuccess) return cuda_fail(e, "conv fold launch");
  }
  gdn::VerifyParams vp{};
  vp.B = B; vp.layers = layers; vp.n_max = banks->n_max; vp.words = nullptr;
  vp.Hk = d->Hk; vp.Hv = d->Hv; vp.dk = d->dk; vp.dv = d->dv; vp.R = d->Hv / d->Hk; vp.in_dtype = d->in_dtype;
  vp.state = state; vp.fold = 1;
  vp.pend_k = banks->k[pend]; vp.pend_u = banks->u[pend]; vp.pend_a = banks->a[pend];
  vp.pend_path = banks->pend_path; vp.pend_len = banks->pend_len; vp.err = banks->err;
  e = gdn::launch_verify(vp, stream);
  if (e != cudaSuccess) return cuda_fail(e, "state fold launch");
  banks->pend_bank = -1;
  return GDN_OK;
}

namespace {
// One CTA waits on an mbarrier armed for 16 bytes that no copy delivers: the bounded wait gives up and the
// CTA reports the timeout like the verify kernels do.
__global__ void selftest_wait_timeout_kernel(int32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    gdn::mbar_init(&bar);
    gdn::mbar_expect(&bar, 16);
  }
  __syncthreads();
  if (!__syncthreads_and(gdn::mbar_wait(&bar, 0)) && threadIdx.x == 0) gdn::device_error(err, GDN_DEVERR_TIMEOUT, 0);
}
}  // namespace

gdn_status gdn_selftest_wait_timeout(gdn_banks* banks, cudaStream_t stream) {
  gdn::clear_error();
  if (!banks || !banks->err) return fail(GDN_ERR_INVALID_ARG, "banks / banks.err is NULL");
  if (!aligned16(banks->err)) return fail(GDN_ERR_INVALID_ARG, "banks.err is not 16-byte aligned");
  selftest_wait_timeout_kernel<<<1, 32, 0, stream>>>(banks->err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return GDN_OK;
}

gdn_status gdn_check_error(gdn_banks* banks, cudaStream_t stream) {
  gdn::clear_error();
  if (!banks || !banks->err) return fail(GDN_ERR_INVALID_ARG, "banks / banks.err is NULL");
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
  int32_t w[2] = {0, 0};
  e = cudaMemcpyAsync(w, banks->err, sizeof(w), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the error words");
  if (w[0] == 0) return GDN_OK;
  e = cudaMemsetAsync(banks->err, 0, sizeof(w), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the error words");
  if (w[0] & GDN_DEVERR_INVALID_PATH)
    return fail(GDN_ERR_INVALID_PATH, "accepted path of request %d is not a root path of its tree; nothing was "
                "committed for it", w[1] - 1);
  if (w[0] & GDN_DEVERR_TIMEOUT)
    return fail(GDN_ERR_TIMEOUT, "an asynchronous copy of request %d did not complete within the bounded wait; "
                "its outputs are incomplete", w[1] - 1);
  if (w[0] & GDN_DEVERR_SCHEDULE)
    return fail(GDN_ERR_SCHEDULE, "packed schedule of request %d is out of range (n, chains, boundary slots); "
                "the offending accesses were skipped", w[1] - 1);
  return fail(GDN_ERR_CUDA, "unknown device error word 0x%x", w[0]);
}

}  // extern "C"
