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
#endif

// Offsets inside one packed schedule record (see gdn_tree.h).
struct SchedLayout {
  int n_max;
  __host__ __device__ int words() const { return 5 + 5 * n_max; }
  __host__ __device__ int parent() const { return 4; }
  __host__ __device__ int bslot() const { return 4 + n_max; }
  __host__ __device__ int chain_src() const { return 4 + 2 * n_max; }
  __host__ __device__ int chain_off() const { return 4 + 3 * n_max; }
  __host__ __device__ int chain_nodes() const { return 5 + 4 * n_max; }
};

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
  int fold;
  const float* pend_k;
  const float* pend_u;
  const float* pend_a;
  const int32_t* pend_path;
  const int32_t* pend_len;
  int32_t* err;                // device error words
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
cudaError_t launch_verify(const VerifyParams& p, cudaStream_t s);

cudaError_t launch_commit(const CommitParams& p, int compact, cudaStream_t s);
bool verify_supported(int dk, int dv);

}  // namespace gdn
