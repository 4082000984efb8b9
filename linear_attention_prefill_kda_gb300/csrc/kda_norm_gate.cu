// Standalone output RMSNorm-gate ("[Feature][KDA] Add Kimi K3 KDA execution",
// first section: FusedRMSNormGated output normalisation and gating):
//     y = o / sqrt(mean_dv(o^2) + eps) * w * act(gate),  act = sigmoid or SiLU
// One warp per (token, head) row; each lane holds dv/32 elements (dv/4 lanes
// with 4 elements each when dv < 128), loaded as one vector.  Memory bound:
// reads o and gate, writes y once.  y may alias o.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

// o is read as TO (the ABI dtype, or fp32 when the prefill kept its raw
// output in fp32 scratch); gate, w and y are T.
template <int DV, typename T, typename TO>
__global__ void __launch_bounds__(256) norm_gate_kernel(NormGateParams p) {
  constexpr int LANES = DV / 4;  // active lanes, 4 elements each
  static_assert(DV % 4 == 0 && LANES <= 32, "dv must be a multiple of 4 and <= 128");
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int64_t nrows = p.rows * p.H;
  if (row >= nrows) return;
  const TO* o = reinterpret_cast<const TO*>(p.o) + row * DV;
  const T* gt = reinterpret_cast<const T*>(p.gate) + row * DV;
  T* y = reinterpret_cast<T*>(p.y) + row * DV;
  float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane < LANES) x = load4(o + lane * 4);
  float ss = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if (lane >= LANES) return;
  const float inv = rsqrtf(ss / (float)DV + p.eps);
  const float4 g = load4(gt + lane * 4);
  const float4 w = load4(reinterpret_cast<const T*>(p.w) + lane * 4);
  x.x *= inv * w.x * gate_actf(g.x, p.gate_act);
  x.y *= inv * w.y * gate_actf(g.y, p.gate_act);
  x.z *= inv * w.z * gate_actf(g.z, p.gate_act);
  x.w *= inv * w.w * gate_actf(g.w, p.gate_act);
  store4(y + lane * 4, x);
}

template <int DV>
cudaError_t launch_ng_d(const NormGateParams& p, cudaStream_t stream) {
  const int64_t nrows = p.rows * p.H;
  const int64_t blocks = (nrows + 7) / 8;
  if (blocks == 0) return cudaSuccess;
  if (p.dtype == KDA_F32)
    norm_gate_kernel<DV, float, float><<<(unsigned)blocks, 256, 0, stream>>>(p);
  else if (p.o_f32)
    norm_gate_kernel<DV, bf16, float><<<(unsigned)blocks, 256, 0, stream>>>(p);
  else
    norm_gate_kernel<DV, bf16, bf16><<<(unsigned)blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_norm_gate(const NormGateParams& p, cudaStream_t stream) {
  switch (p.dv) {
    case 16: return launch_ng_d<16>(p, stream);
    case 64: return launch_ng_d<64>(p, stream);
    case 128: return launch_ng_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kda
