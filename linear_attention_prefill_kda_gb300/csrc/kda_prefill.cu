// Prefill dispatch: picks the kernel for the shape and applies the output
// norm-gate ("[Feature][KDA] Add Kimi K3 KDA execution", first section) when
// the kernel did not fuse it.
#include <mutex>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

cudaError_t launch_prefill_simt(const PrefillParams& p, cudaStream_t stream);
bool prefill_tc_supported(const PrefillParams& p);
size_t prefill_tc_workspace_bytes(int N, int64_t T, int H);
cudaError_t launch_prefill_tc(const PrefillParams& p, cudaStream_t stream);

static bool tc_shape(int dk, int dv, int chunk, kda_dtype in_dtype) {
  PrefillParams q{};
  q.dk = dk; q.dv = dv; q.chunk = chunk; q.in_dtype = in_dtype;
  return prefill_tc_supported(q);
}

cudaError_t set_smem_once(const void* kernel, int bytes) {
  constexpr int kMaxEntries = 256;
  static std::mutex mu;
  static const void* keys[kMaxEntries];
  static unsigned long long dev_mask[kMaxEntries];
  static int n = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  std::lock_guard<std::mutex> lock(mu);
  int slot = -1;
  for (int i = 0; i < n; ++i)
    if (keys[i] == kernel) slot = i;
  if (slot >= 0 && (dev_mask[slot] & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (slot < 0 && n < kMaxEntries) { slot = n++; keys[slot] = kernel; dev_mask[slot] = 0; }
  if (slot >= 0) dev_mask[slot] |= bit;
  return cudaSuccess;
}

// The CUDA-core kernel splits dv into slabs of 64 columns.  With dv <= 64 one
// slab holds the whole row and the kernel fuses the norm-gate; with dv = 128
// it runs as a second pass, and with bf16 inputs the raw output is kept in
// fp32 scratch (T x H x dv floats) for that pass, so that it is not rounded
// to bf16 before normalisation.
static bool gate_fused_simt(int dv) { return dv <= 64; }
static bool needs_o_scratch(int dv, kda_dtype in_dtype) { return !gate_fused_simt(dv) && in_dtype != KDA_F32; }

size_t prefill_workspace_bytes(int N, int64_t T, int H, int dk, int dv, int chunk) {
  size_t bytes = (size_t)T * (size_t)H * (size_t)dv * sizeof(float);  // raw-output scratch
  if (tc_shape(dk, dv, chunk, KDA_BF16)) {
    const size_t tc = prefill_tc_workspace_bytes(N, T, H);
    if (tc > bytes) bytes = tc;
  }
  return (bytes + 255) & ~(size_t)255;
}

size_t prefill_workspace_needed(int N, int64_t T, int H, int dk, int dv, int chunk, kda_dtype in_dtype,
                                bool gate) {
  if (tc_shape(dk, dv, chunk, in_dtype)) return prefill_tc_workspace_bytes(N, T, H);
  if (!gate || !needs_o_scratch(dv, in_dtype)) return 0;
  return ((size_t)T * (size_t)H * (size_t)dv * sizeof(float) + 255) & ~(size_t)255;
}

bool prefill_uses_tensor_cores(const PrefillParams& p) { return prefill_tc_supported(p); }

cudaError_t launch_prefill(const PrefillParams& p_in, cudaStream_t stream) {
  if (prefill_tc_supported(p_in)) return launch_prefill_tc(p_in, stream);
  PrefillParams p = p_in;
  const bool scratch = p.gate && p.T > 0 && needs_o_scratch(p.dv, p.in_dtype);
  p.o_scratch = scratch ? reinterpret_cast<float*>(p.workspace) : nullptr;
  cudaError_t e = launch_prefill_simt(p, stream);
  if (e != cudaSuccess) return e;
  if (p.gate && p.T > 0 && !gate_fused_simt(p.dv)) {
    NormGateParams ng{};
    ng.o = scratch ? static_cast<const void*>(p.o_scratch) : p.out;
    ng.o_f32 = scratch;
    ng.gate = p.gate; ng.w = p.norm_w; ng.y = p.out;
    ng.rows = p.T; ng.H = p.H; ng.dv = p.dv; ng.eps = p.eps; ng.dtype = p.in_dtype;
    ng.gate_act = p.gate_act;
    e = launch_norm_gate(ng, stream);
  }
  return e;
}

}  // namespace kda
