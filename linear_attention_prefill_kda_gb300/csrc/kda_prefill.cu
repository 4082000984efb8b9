// Prefill dispatch: picks the kernel for the shape and applies the output
// norm-gate ("[Feature][KDA] Add Kimi K3 KDA execution", first section) when
// the kernel did not fuse it.
#include <mutex>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

cudaError_t launch_prefill_simt(const PrefillParams& p, cudaStream_t stream);

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

size_t prefill_workspace_bytes(int N, int64_t T, int H, int dk, int dv, int chunk) {
  (void)N; (void)T; (void)H; (void)dk; (void)dv; (void)chunk;
  return 0;
}

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream) {
  cudaError_t e = launch_prefill_simt(p, stream);
  if (e != cudaSuccess) return e;
  if (p.gate && p.T > 0) {
    NormGateParams ng{};
    ng.o = p.out; ng.gate = p.gate; ng.w = p.norm_w; ng.y = p.out;
    ng.rows = p.T; ng.H = p.H; ng.dv = p.dv; ng.eps = p.eps; ng.dtype = p.in_dtype;
    e = launch_norm_gate(ng, stream);
  }
  return e;
}

}  // namespace kda
