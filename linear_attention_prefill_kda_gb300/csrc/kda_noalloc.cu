// kda_prefill_chunked_static_scratch: the chunked prefill for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they run the prefill.  Examples are code that runs while a
// stream is being captured into a CUDA graph in the strict capture mode,
// where allocation is an error, and runtimes whose memory is owned by a
// fixed arena they may not grow.  Such callers still own their inputs and
// outputs, but have no way to supply the tensor-core path's scratch.  This
// entry point uses a scratch array that lives in the library itself instead:
// a file-scope __device__ array of KDA_STATIC_SCRATCH_BYTES bytes, created on
// each GPU when the library's device code is loaded there and held until the
// process exits.
//
// Host code cannot use the array's name as a device address (on the host it
// names a stand-in object), so the address is looked up with
// cudaGetSymbolAddress on the first call made with a device current, and
// cached for that device's current CUDA context.  That first call per device
// should therefore happen before any stream capture begins.  The cache is keyed
// by the context's id, which the driver never reuses within a process: after
// cudaDeviceReset (or in another context on the same device) the library's
// module is loaded again at another address, and the next call looks the
// address up again -- that call, too, belongs before any capture.
//
// All calls share the one array; each call overwrites what it needs before
// reading it (nothing in it has to start at zero), and two calls whose
// kernels overlap on the GPU race on it.
#include "../../include/kda.h"
#include "kda_internal.h"

#include <cuda.h>

#include <mutex>

namespace {

__device__ __align__(256) unsigned char g_static_scratch[KDA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
  unsigned long long ctx_id;
  void* ptr;
};
Cached g_scratch[kMaxDevices] = {};

// Id of the calling thread's current context, through the driver entry points
// the runtime hands out (the library does not link the driver library).
cudaError_t current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static cudaError_t resolved = cudaErrorUnknown;
  static std::once_flag once;
  std::call_once(once, [] {
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
        qa == cudaDriverEntryPointSuccess && qb == cudaDriverEntryPointSuccess && a && b) {
      get_current = reinterpret_cast<GetCurrent>(a);
      get_id = reinterpret_cast<GetId>(b);
      resolved = cudaSuccess;
    }
  });
  if (resolved != cudaSuccess) return resolved;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of g_static_scratch in the current device's current context
// (looked up once per context).  With no context current yet, the lookup
// itself makes the device's primary context current, and its id is taken
// afterwards.
cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long id = 0;
  const bool known = current_context_id(&id) == cudaSuccess;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!known || !g_scratch[dev].ptr || g_scratch[dev].ctx_id != id) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return e;
    e = current_context_id(&id);
    if (e != cudaSuccess) return e;
    g_scratch[dev].ptr = ptr;
    g_scratch[dev].ctx_id = id;
  }
  *out = g_scratch[dev].ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" KDA_API kda_status kda_prefill_chunked_static_scratch(
    const void* q, const void* k, const void* v, const void* g, const void* beta, kda_dtype in_dtype,
    const int32_t* cu_seqlens, int N, int64_t T, const int32_t* state_indices,
    const int32_t* has_initial_state, void* state_pool, int64_t num_slots, kda_dtype state_dtype,
    void* out, void* checkpoints, int32_t checkpoint_every, int64_t checkpoint_capacity,
    int32_t* ckpt_offsets, const void* gate, const void* norm_w, float eps, kda_gate_act gate_act,
    int H, int dk, int dv, int chunk, float scale, int32_t* dev_status, void* stream) {
  // Sizes beyond the array are rejected before any device work.
  if (N < 0 || T < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  if (dk != dv || (dk != 16 && dk != 64 && dk != 128) || (chunk != 16 && chunk != 64))
    return KDA_ERR_UNSUPPORTED;
  if (in_dtype != KDA_F32 && in_dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
  const size_t need = kda::prefill_workspace_needed(N, T, H, dk, dv, chunk, in_dtype, gate != nullptr);
  if (need > (size_t)KDA_STATIC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0 && static_scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
  return kda_prefill_chunked(q, k, v, g, beta, in_dtype, cu_seqlens, N, T, state_indices, has_initial_state,
                             state_pool, num_slots, state_dtype, out, checkpoints, checkpoint_every,
                             checkpoint_capacity, ckpt_offsets, gate, norm_w, eps, gate_act, H, dk, dv, chunk,
                             scale, scratch, need > 0 ? (size_t)KDA_STATIC_SCRATCH_BYTES : 0, dev_status,
                             stream);
}
