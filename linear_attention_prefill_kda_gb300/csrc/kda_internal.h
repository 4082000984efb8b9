// Internal launch parameters shared by the host entry points and the kernel
// launchers.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

struct DecodeParams {
  const void *q, *k, *v, *g, *beta;
  const int32_t* state_indices;
  void* state_pool;
  void* out;
  const void *gate, *norm_w;
  int32_t* dev_status;
  int64_t num_slots;
  int N, H, dk, dv;
  float scale, eps;
  kda_dtype in_dtype, state_dtype;
  int gate_act;  // kda_gate_act
};

struct DecodeMultiParams {
  const void *q, *k, *v, *g, *beta;  // [N*K, H, *] token-major
  const int32_t* state_indices;
  void* state_pool;
  void* out;            // [N*K, H, dv]
  void* token_states;   // [N*K, H, dk, dv] state dtype
  const void *gate, *norm_w;
  int32_t* dev_status;
  int64_t num_slots;
  int N, K, H, dk, dv;
  int write_back;
  float scale, eps;
  kda_dtype in_dtype, state_dtype;
  int gate_act;
};

struct CommitParams {
  const void* token_states;
  const int32_t* num_accepted;
  const int32_t* state_indices;
  void* state_pool;
  int32_t* dev_status;
  int64_t num_slots;
  int N, K, H, dk, dv;
  kda_dtype state_dtype;
};

struct NormGateParams {
  const void *o, *gate, *w;
  void* y;
  int64_t rows;  // token rows; each holds H heads of dv
  int H, dv;
  float eps;
  kda_dtype dtype;  // of gate, w and y (and of o unless o_f32)
  bool o_f32;       // o is fp32 scratch regardless of dtype
  int gate_act;     // kda_gate_act
};

struct ConvParams {
  const void *x, *w, *bias;   // x [T or N, C]; w [C, W]; bias [C] or NULL
  void* y;                    // same layout as x
  const int32_t *cu_seqlens, *state_indices, *has_initial_state;  // cu_seqlens: prefill only
  void* pool;                 // [num_slots, W-1, C]
  int32_t* dev_status;
  int64_t T, num_slots;
  int N, C, W;
  int act;                    // 0 identity, 1 SiLU
  kda_dtype dtype;
};

struct NormGateExParams {
  const void *o, *residual, *gate, *w, *b;  // residual, w, b may be NULL
  void *y, *residual_out;                   // residual_out may be NULL
  int64_t rows, gate_row_stride;            // gate row stride in elements
  int H, dv;
  float eps;
  kda_dtype dtype;
  int gate_act;
};

struct PrefillParams {
  const void *q, *k, *v, *g, *beta;
  const int32_t* cu_seqlens;
  const int32_t* state_indices;
  const int32_t* has_initial_state;  // NULL: every sequence starts from its slot
  void* state_pool;
  void* out;
  void* checkpoints;
  int32_t* ckpt_offsets;
  const void *gate, *norm_w;
  void* workspace;
  size_t workspace_bytes;
  float* o_scratch;  // when set, the prefill kernel writes raw o here in fp32
  int32_t* dev_status;
  int64_t T, num_slots, checkpoint_capacity;
  int N, H, dk, dv, chunk, checkpoint_every;
  float scale, eps;
  kda_dtype in_dtype, state_dtype;
  int gate_act;  // kda_gate_act
  // polls of the first bounded wait of the intra-chunk and of the state kernel
  uint32_t intra_first_wait_tries, state_first_wait_tries;
  // The short convolution folded into the prefill (kda_prefill_chunked_conv):
  // q, k, v then point at the projections before the convolution, rows
  // x_row_stride elements apart; the convolution's taps, bias and cache pool
  // cover the channels [q | k | v] (3 H d of them).
  bool conv;
  int64_t x_row_stride;
  const void *conv_w, *conv_b;
  void* conv_pool;
  int64_t conv_num_slots;
  int conv_width, conv_act;
};

// Polls of a bounded on-chip wait before it gives up (mbarrier try_wait polls).
constexpr uint32_t kDefaultWaitTries = 1u << 22;

// Polls of the first bounded wait of the intra-chunk kernel (which = 0) or
// of the state kernel (which = 1): the testing hook
// kda_testing_set_first_wait_tries, the default otherwise.
uint32_t prefill_first_wait_tries(int which);

// Raise a kernel's dynamic shared-memory limit once per (kernel, device), so
// later calls (including those made during stream capture) skip the
// attribute call.
cudaError_t set_smem_once(const void* kernel, int bytes);

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_multi(const DecodeMultiParams& p, cudaStream_t stream);
cudaError_t launch_commit(const CommitParams& p, cudaStream_t stream);
cudaError_t launch_norm_gate(const NormGateParams& p, cudaStream_t stream);
cudaError_t launch_norm_gate_ex(const NormGateExParams& p, cudaStream_t stream);
cudaError_t launch_conv_prefill(const ConvParams& p, cudaStream_t stream);
cudaError_t launch_conv_decode(const ConvParams& p, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream);
// Whether launch_prefill takes the tensor-core kernels for this shape.
bool prefill_uses_tensor_cores(const PrefillParams& p);
// Upper bound over every option (what kda_prefill_workspace_bytes reports).
size_t prefill_workspace_bytes(int N, int64_t T, int H, int dk, int dv, int chunk);
// What one call with these options actually uses (<= the bound).
size_t prefill_workspace_needed(int N, int64_t T, int H, int dk, int dv, int chunk, kda_dtype in_dtype,
                                bool gate);

}  // namespace kda
