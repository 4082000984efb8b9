// extern "C" entry points of libkda: argument validation on the host, then
// asynchronous launches on the caller's stream.  No allocation, no
// synchronisation, no host read of device memory.
#include <math.h>

#include <atomic>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dtype_ok(kda_dtype d) { return d == KDA_F32 || d == KDA_BF16; }
bool dim_ok(int d) { return d == 16 || d == 64 || d == 128; }
bool act_ok(kda_gate_act a) { return a == KDA_GATE_SIGMOID || a == KDA_GATE_SILU; }

// Every non-NULL pointer must be 16-byte aligned; required ones must be non-NULL.
bool ptr_ok(const void* p, bool required) {
  if (!p) return !required;
  return aligned16(p);
}

kda_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

}  // namespace

namespace kda {
namespace {
std::atomic<int32_t> g_first_wait_tries[2] = {{-1}, {-1}};
}
uint32_t prefill_first_wait_tries(int which) {
  const int32_t t = g_first_wait_tries[which & 1].load(std::memory_order_relaxed);
  return t < 0 ? kDefaultWaitTries : (uint32_t)t;
}
}  // namespace kda

extern "C" {

int kda_version(void) { return 105; }

int kda_prefill_path(int dk, int dv, int chunk, kda_dtype in_dtype) {
  if (!dim_ok(dk) || dv != dk || (chunk != 16 && chunk != 64) || !dtype_ok(in_dtype)) return KDA_PATH_UNSUPPORTED;
  kda::PrefillParams q{};
  q.dk = dk; q.dv = dv; q.chunk = chunk; q.in_dtype = in_dtype;
  return kda::prefill_uses_tensor_cores(q) ? KDA_PATH_TENSOR_CORES : KDA_PATH_CUDA_CORES;
}

void kda_testing_set_first_wait_tries(int32_t tries, int32_t kernels) {
  for (int which = 0; which < 2; ++which)
    if (tries < 0 || (kernels >> which) & 1)
      kda::g_first_wait_tries[which].store(tries < 0 ? -1 : tries, std::memory_order_relaxed);
}

const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case KDA_ERR_WORKSPACE: return "workspace too small";
    case KDA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

size_t kda_prefill_workspace_bytes(int N, int64_t T, int H, int dk, int dv, int chunk) {
  if (N < 0 || T < 0 || H <= 0) return 0;
  return kda::prefill_workspace_bytes(N, T, H, dk, dv, chunk);
}

}  // extern "C"

namespace {

// Host-side checks shared by the prefill entry points; on success fills *pp.
// q, k, v may be NULL here when the caller supplies them another way.
kda_status prefill_params(const void* q, const void* k, const void* v, const void* g, const void* beta,
                          kda_dtype in_dtype, const int32_t* cu_seqlens, int N, int64_t T,
                          const int32_t* state_indices, const int32_t* has_initial_state, void* state_pool,
                          int64_t num_slots, kda_dtype state_dtype, void* out, void* checkpoints,
                          int32_t checkpoint_every, int64_t checkpoint_capacity, int32_t* ckpt_offsets,
                          const void* gate, const void* norm_w, float eps, kda_gate_act gate_act, int H, int dk,
                          int dv, int chunk, float scale, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, kda::PrefillParams* pp) {
  if (N < 0 || T < 0 || T > INT32_MAX || H <= 0 || H > 65535 || num_slots <= 0) return KDA_ERR_INVALID_ARG;
  if ((int64_t)N * H > INT32_MAX || (T / 16 + N) * (int64_t)H > INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(in_dtype) || !dtype_ok(state_dtype)) return KDA_ERR_UNSUPPORTED;
  if (!dim_ok(dk) || dv != dk || (chunk != 16 && chunk != 64)) return KDA_ERR_UNSUPPORTED;
  if (checkpoint_every < 0 || (checkpoint_every > 0 && checkpoint_every % chunk != 0))
    return KDA_ERR_INVALID_ARG;
  const bool tokens = T > 0;
  if (!ptr_ok(q, tokens) || !ptr_ok(k, tokens) || !ptr_ok(v, tokens) || !ptr_ok(g, tokens) ||
      !ptr_ok(beta, tokens) || !ptr_ok(out, tokens))
    return KDA_ERR_INVALID_ARG;
  if (!ptr_ok(cu_seqlens, true) || !ptr_ok(state_indices, N > 0) || !ptr_ok(state_pool, true))
    return KDA_ERR_INVALID_ARG;
  if (!ptr_ok(ckpt_offsets, false) || !ptr_ok(dev_status, false) || !ptr_ok(has_initial_state, false))
    return KDA_ERR_INVALID_ARG;
  if (!act_ok(gate_act)) return KDA_ERR_INVALID_ARG;
  if ((gate == nullptr) != (norm_w == nullptr)) return KDA_ERR_INVALID_ARG;
  if (!ptr_ok(gate, false) || !ptr_ok(norm_w, false)) return KDA_ERR_INVALID_ARG;
  if (gate && !(eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if (checkpoint_every > 0) {
    if (!ptr_ok(checkpoints, true)) return KDA_ERR_INVALID_ARG;
    if (checkpoint_capacity < T / checkpoint_every) return KDA_ERR_INVALID_ARG;
  }
  const size_t need = kda::prefill_workspace_needed(N, T, H, dk, dv, chunk, in_dtype, gate != nullptr);
  if (need > 0 && (workspace_bytes < need || !ptr_ok(workspace, true))) return KDA_ERR_WORKSPACE;
  kda::PrefillParams& p = *pp;
  p = kda::PrefillParams{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.cu_seqlens = cu_seqlens;
  p.state_indices = state_indices;
  p.has_initial_state = has_initial_state;
  p.state_pool = state_pool;
  p.out = out;
  p.checkpoints = checkpoints;
  p.ckpt_offsets = ckpt_offsets;
  p.gate = gate; p.norm_w = norm_w;
  p.workspace = workspace;
  p.workspace_bytes = workspace_bytes;
  p.dev_status = dev_status;
  p.T = T; p.num_slots = num_slots; p.checkpoint_capacity = checkpoint_capacity;
  p.N = N; p.H = H; p.dk = dk; p.dv = dv; p.chunk = chunk; p.checkpoint_every = checkpoint_every;
  p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)dk);
  p.eps = eps;
  p.in_dtype = in_dtype; p.state_dtype = state_dtype;
  p.gate_act = gate_act;
  p.intra_first_wait_tries = kda::prefill_first_wait_tries(0);
  p.state_first_wait_tries = kda::prefill_first_wait_tries(1);
  return KDA_OK;
}

// An empty batch only writes the checkpoint offsets' single entry.
kda_status launch_or_empty(const kda::PrefillParams& p, int32_t* ckpt_offsets, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.N == 0) {
    if (ckpt_offsets) return from_cuda(cudaMemsetAsync(ckpt_offsets, 0, sizeof(int32_t), st));
    return KDA_OK;
  }
  return from_cuda(kda::launch_prefill(p, st));
}

}  // namespace

extern "C" {

kda_status kda_prefill_chunked(const void* q, const void* k, const void* v, const void* g,
                               const void* beta, kda_dtype in_dtype, const int32_t* cu_seqlens,
                               int N, int64_t T, const int32_t* state_indices,
                               const int32_t* has_initial_state, void* state_pool,
                               int64_t num_slots, kda_dtype state_dtype, void* out,
                               void* checkpoints, int32_t checkpoint_every,
                               int64_t checkpoint_capacity, int32_t* ckpt_offsets,
                               const void* gate, const void* norm_w, float eps,
                               kda_gate_act gate_act, int H, int dk, int dv, int chunk,
                               float scale, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream) {
  kda::PrefillParams p;
  const kda_status s = prefill_params(q, k, v, g, beta, in_dtype, cu_seqlens, N, T, state_indices,
                                      has_initial_state, state_pool, num_slots, state_dtype, out, checkpoints,
                                      checkpoint_every, checkpoint_capacity, ckpt_offsets, gate, norm_w, eps,
                                      gate_act, H, dk, dv, chunk, scale, workspace, workspace_bytes, dev_status,
                                      &p);
  if (s != KDA_OK) return s;
  return launch_or_empty(p, ckpt_offsets, stream);
}

kda_status kda_prefill_chunked_conv(const void* x_q, const void* x_k, const void* x_v, int64_t x_row_stride,
                                    const void* conv_w, const void* conv_b, int conv_width,
                                    kda_conv_act conv_act, void* conv_state_pool, int64_t conv_num_slots,
                                    const void* g, const void* beta, kda_dtype in_dtype,
                                    const int32_t* cu_seqlens, int N, int64_t T,
                                    const int32_t* state_indices, const int32_t* has_initial_state,
                                    void* state_pool, int64_t num_slots, kda_dtype state_dtype, void* out,
                                    void* checkpoints, int32_t checkpoint_every, int64_t checkpoint_capacity,
                                    int32_t* ckpt_offsets, const void* gate, const void* norm_w, float eps,
                                    kda_gate_act gate_act, int H, int dk, int dv, int chunk, float scale,
                                    void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                    void* stream) {
  kda::PrefillParams p;
  const kda_status s = prefill_params(x_q, x_k, x_v, g, beta, in_dtype, cu_seqlens, N, T, state_indices,
                                      has_initial_state, state_pool, num_slots, state_dtype, out, checkpoints,
                                      checkpoint_every, checkpoint_capacity, ckpt_offsets, gate, norm_w, eps,
                                      gate_act, H, dk, dv, chunk, scale, workspace, workspace_bytes, dev_status,
                                      &p);
  if (s != KDA_OK) return s;
  if (kda_prefill_path(dk, dv, chunk, in_dtype) != KDA_PATH_TENSOR_CORES) return KDA_ERR_UNSUPPORTED;
  if (conv_width < 2 || conv_width > 4) return KDA_ERR_UNSUPPORTED;
  if (conv_act != KDA_CONV_IDENTITY && conv_act != KDA_CONV_SILU) return KDA_ERR_INVALID_ARG;
  // rows of the projections start on 16-byte boundaries
  if (x_row_stride < (int64_t)H * dk || x_row_stride % 8 != 0) return KDA_ERR_INVALID_ARG;
  if (!ptr_ok(conv_w, true) || !ptr_ok(conv_b, false) || !ptr_ok(conv_state_pool, true) || conv_num_slots <= 0)
    return KDA_ERR_INVALID_ARG;
  p.conv = true;
  p.x_row_stride = x_row_stride;
  p.conv_w = conv_w;
  p.conv_b = conv_b;
  p.conv_pool = conv_state_pool;
  p.conv_num_slots = conv_num_slots;
  p.conv_width = conv_width;
  p.conv_act = conv_act;
  return launch_or_empty(p, ckpt_offsets, stream);
}

kda_status kda_decode_step(const void* q, const void* k, const void* v, const void* g,
                           const void* beta, kda_dtype in_dtype, const int32_t* state_indices,
                           int N, void* state_pool, int64_t num_slots, kda_dtype state_dtype,
                           void* out, const void* gate, const void* norm_w, float eps,
                           kda_gate_act gate_act, int H, int dk, int dv, float scale,
                           int32_t* dev_status, void* stream) {
  if (N < 0 || H <= 0 || num_slots <= 0) return KDA_ERR_INVALID_ARG;
  if ((int64_t)N * H > INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(in_dtype) || !dtype_ok(state_dtype)) return KDA_ERR_UNSUPPORTED;
  if (!dim_ok(dk) || dv != dk) return KDA_ERR_UNSUPPORTED;
  if (N == 0) return KDA_OK;
  if (!ptr_ok(q, true) || !ptr_ok(k, true) || !ptr_ok(v, true) || !ptr_ok(g, true) ||
      !ptr_ok(beta, true) || !ptr_ok(out, true) || !ptr_ok(state_indices, true) ||
      !ptr_ok(state_pool, true) || !ptr_ok(dev_status, false))
    return KDA_ERR_INVALID_ARG;
  if ((gate == nullptr) != (norm_w == nullptr)) return KDA_ERR_INVALID_ARG;
  if (!ptr_ok(gate, false) || !ptr_ok(norm_w, false)) return KDA_ERR_INVALID_ARG;
  if (gate && !(eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if (!act_ok(gate_act)) return KDA_ERR_INVALID_ARG;
  kda::DecodeParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.state_indices = state_indices;
  p.state_pool = state_pool;
  p.out = out;
  p.gate = gate; p.norm_w = norm_w;
  p.dev_status = dev_status;
  p.num_slots = num_slots;
  p.N = N; p.H = H; p.dk = dk; p.dv = dv;
  p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)dk);
  p.eps = eps;
  p.in_dtype = in_dtype; p.state_dtype = state_dtype;
  p.gate_act = gate_act;
  return from_cuda(kda::launch_decode(p, static_cast<cudaStream_t>(stream)));
}

kda_status kda_decode_multi(const void* q, const void* k, const void* v, const void* g,
                            const void* beta, kda_dtype in_dtype, const int32_t* state_indices,
                            int N, int K, void* state_pool, int64_t num_slots,
                            kda_dtype state_dtype, void* out, void* token_states, int write_back,
                            const void* gate, const void* norm_w, float eps,
                            kda_gate_act gate_act, int H, int dk, int dv, float scale,
                            int32_t* dev_status, void* stream) {
  if (N < 0 || K < 0 || H <= 0 || num_slots <= 0) return KDA_ERR_INVALID_ARG;
  if ((int64_t)N * H > INT32_MAX || (int64_t)N * K > INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(in_dtype) || !dtype_ok(state_dtype)) return KDA_ERR_UNSUPPORTED;
  if (!dim_ok(dk) || dv != dk) return KDA_ERR_UNSUPPORTED;
  if (N == 0 || K == 0) return KDA_OK;
  if (!ptr_ok(q, true) || !ptr_ok(k, true) || !ptr_ok(v, true) || !ptr_ok(g, true) ||
      !ptr_ok(beta, true) || !ptr_ok(out, true) || !ptr_ok(state_indices, true) ||
      !ptr_ok(state_pool, true) || !ptr_ok(token_states, false) || !ptr_ok(dev_status, false))
    return KDA_ERR_INVALID_ARG;
  if ((gate == nullptr) != (norm_w == nullptr)) return KDA_ERR_INVALID_ARG;
  if (!ptr_ok(gate, false) || !ptr_ok(norm_w, false)) return KDA_ERR_INVALID_ARG;
  if (gate && !(eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if (!act_ok(gate_act)) return KDA_ERR_INVALID_ARG;
  kda::DecodeMultiParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.state_indices = state_indices;
  p.state_pool = state_pool;
  p.out = out;
  p.token_states = token_states;
  p.gate = gate; p.norm_w = norm_w;
  p.dev_status = dev_status;
  p.num_slots = num_slots;
  p.N = N; p.K = K; p.H = H; p.dk = dk; p.dv = dv;
  p.write_back = write_back != 0;
  p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)dk);
  p.eps = eps;
  p.in_dtype = in_dtype; p.state_dtype = state_dtype;
  p.gate_act = gate_act;
  return from_cuda(kda::launch_decode_multi(p, static_cast<cudaStream_t>(stream)));
}

kda_status kda_commit_accepted(const void* token_states, const int32_t* num_accepted,
                               const int32_t* state_indices, int N, int K, void* state_pool,
                               int64_t num_slots, kda_dtype state_dtype, int H, int dk, int dv,
                               int32_t* dev_status, void* stream) {
  if (N < 0 || K < 0 || H <= 0 || num_slots <= 0) return KDA_ERR_INVALID_ARG;
  if ((int64_t)N * H > INT32_MAX || (int64_t)N * K > INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(state_dtype)) return KDA_ERR_UNSUPPORTED;
  if (!dim_ok(dk) || dv != dk) return KDA_ERR_UNSUPPORTED;
  if (N == 0 || K == 0) return KDA_OK;
  if (!ptr_ok(token_states, true) || !ptr_ok(num_accepted, true) || !ptr_ok(state_indices, true) ||
      !ptr_ok(state_pool, true) || !ptr_ok(dev_status, false))
    return KDA_ERR_INVALID_ARG;
  kda::CommitParams p{};
  p.token_states = token_states;
  p.num_accepted = num_accepted;
  p.state_indices = state_indices;
  p.state_pool = state_pool;
  p.dev_status = dev_status;
  p.num_slots = num_slots;
  p.N = N; p.K = K; p.H = H; p.dk = dk; p.dv = dv;
  p.state_dtype = state_dtype;
  return from_cuda(kda::launch_commit(p, static_cast<cudaStream_t>(stream)));
}

kda_status kda_norm_gate_ex(const void* o, const void* residual, void* residual_out,
                            const void* gate, int64_t gate_row_stride, const void* w,
                            const void* b, float eps, kda_gate_act gate_act, void* y, int64_t rows,
                            int H, int dv, kda_dtype dtype, void* stream) {
  if (rows < 0 || H <= 0 || !act_ok(gate_act) || !(eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_F32 && dtype != KDA_BF16 && dtype != KDA_F16) return KDA_ERR_UNSUPPORTED;
  if (!dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
  const int64_t row_elems = (int64_t)H * dv;
  if (gate_row_stride == 0) gate_row_stride = row_elems;
  if (gate_row_stride < row_elems || gate_row_stride % 4 != 0) return KDA_ERR_INVALID_ARG;
  if (rows == 0) return KDA_OK;
  if ((rows * H + 7) / 8 > INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (!ptr_ok(o, true) || !ptr_ok(gate, true) || !ptr_ok(y, true) || !ptr_ok(residual, false) ||
      !ptr_ok(residual_out, false) || !ptr_ok(w, false) || !ptr_ok(b, false))
    return KDA_ERR_INVALID_ARG;
  if (residual_out && residual_out == y) return KDA_ERR_INVALID_ARG;
  kda::NormGateExParams p{};
  p.o = o; p.residual = residual; p.gate = gate; p.w = w; p.b = b;
  p.y = y; p.residual_out = residual_out;
  p.rows = rows; p.gate_row_stride = gate_row_stride;
  p.H = H; p.dv = dv; p.eps = eps; p.dtype = dtype; p.gate_act = gate_act;
  return from_cuda(kda::launch_norm_gate_ex(p, static_cast<cudaStream_t>(stream)));
}

namespace {
kda_status conv_common(const void* weight, const void* bias, kda_dtype dtype, int N, int channels,
                       int width, const int32_t* state_indices, void* pool, int64_t num_slots,
                       kda_conv_act act, int32_t* dev_status) {
  if (N < 0 || channels <= 0 || num_slots <= 0) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(dtype)) return KDA_ERR_UNSUPPORTED;
  if (width < 2 || width > 4 || channels % 8 != 0) return KDA_ERR_UNSUPPORTED;
  if (act != KDA_CONV_IDENTITY && act != KDA_CONV_SILU) return KDA_ERR_INVALID_ARG;
  if (!ptr_ok(weight, true) || !ptr_ok(bias, false) || !ptr_ok(state_indices, N > 0) ||
      !ptr_ok(pool, true) || !ptr_ok(dev_status, false))
    return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}
}  // namespace

kda_status kda_causal_conv1d_prefill(const void* x, const void* weight, const void* bias,
                                     kda_dtype dtype, const int32_t* cu_seqlens, int N, int64_t T,
                                     int channels, int width, const int32_t* state_indices,
                                     const int32_t* has_initial_state, void* conv_state_pool,
                                     int64_t num_slots, kda_conv_act act, void* y,
                                     int32_t* dev_status, void* stream) {
  if (T < 0 || T > INT32_MAX) return KDA_ERR_INVALID_ARG;
  const kda_status st = conv_common(weight, bias, dtype, N, channels, width, state_indices,
                                    conv_state_pool, num_slots, act, dev_status);
  if (st != KDA_OK) return st;
  if (T / 64 + N > 65535) return KDA_ERR_INVALID_ARG;  // tile slots form the grid's y extent
  if (!ptr_ok(cu_seqlens, true) || !ptr_ok(x, T > 0) || !ptr_ok(y, T > 0) ||
      !ptr_ok(has_initial_state, false))
    return KDA_ERR_INVALID_ARG;
  if (N == 0 || T == 0) return KDA_OK;
  kda::ConvParams p{};
  p.x = x; p.w = weight; p.bias = bias; p.y = y;
  p.cu_seqlens = cu_seqlens; p.state_indices = state_indices; p.has_initial_state = has_initial_state;
  p.pool = conv_state_pool; p.dev_status = dev_status;
  p.T = T; p.num_slots = num_slots; p.N = N; p.C = channels; p.W = width; p.act = act;
  p.dtype = dtype;
  return from_cuda(kda::launch_conv_prefill(p, static_cast<cudaStream_t>(stream)));
}

kda_status kda_causal_conv1d_decode(const void* x, const void* weight, const void* bias,
                                    kda_dtype dtype, int N, int channels, int width,
                                    const int32_t* state_indices, void* conv_state_pool,
                                    int64_t num_slots, kda_conv_act act, void* y,
                                    int32_t* dev_status, void* stream) {
  const kda_status st = conv_common(weight, bias, dtype, N, channels, width, state_indices,
                                    conv_state_pool, num_slots, act, dev_status);
  if (st != KDA_OK) return st;
  if (N > 65535) return KDA_ERR_INVALID_ARG;  // sequences form the grid's y extent
  if (!ptr_ok(x, N > 0) || !ptr_ok(y, N > 0)) return KDA_ERR_INVALID_ARG;
  if (N == 0) return KDA_OK;
  kda::ConvParams p{};
  p.x = x; p.w = weight; p.bias = bias; p.y = y;
  p.state_indices = state_indices;
  p.pool = conv_state_pool; p.dev_status = dev_status;
  p.num_slots = num_slots; p.N = N; p.C = channels; p.W = width; p.act = act; p.dtype = dtype;
  return from_cuda(kda::launch_conv_decode(p, static_cast<cudaStream_t>(stream)));
}

kda_status kda_norm_gate(const void* o, const void* gate, const void* w, float eps,
                         kda_gate_act gate_act, void* y, int64_t rows, int H, int dv,
                         kda_dtype dtype, void* stream) {
  if (rows < 0 || H <= 0 || !act_ok(gate_act)) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(dtype)) return KDA_ERR_UNSUPPORTED;
  if (!dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
  if (!(eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if (rows == 0) return KDA_OK;
  if ((rows * H + 7) / 8 > INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (!ptr_ok(o, true) || !ptr_ok(gate, true) || !ptr_ok(w, true) || !ptr_ok(y, true))
    return KDA_ERR_INVALID_ARG;
  kda::NormGateParams p{};
  p.o = o; p.gate = gate; p.w = w; p.y = y;
  p.rows = rows; p.H = H; p.dv = dv; p.eps = eps; p.dtype = dtype; p.gate_act = gate_act;
  return from_cuda(kda::launch_norm_gate(p, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
