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

// Norm-gate variants (the coverage list of "[Feature][KDA] ...", testing
// section): x = o + residual (residual optional, the sum optionally stored as
// the prenorm output), z = x rsqrt(mean x^2 + eps) w + b (w, b optional),
// y = z act(gate), the gate row of each token at gate_row_stride elements.
// Same one-warp-per-row shape as above; the sum is formed in fp32.
template <int DV, typename T>
__global__ void __launch_bounds__(256) norm_gate_ex_kernel(NormGateExParams p) {
  constexpr int LANES = DV / 4;
  static_assert(DV % 4 == 0 && LANES <= 32, "dv must be a multiple of 4 and <= 128");
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;  // token * H + head
  if (row >= p.rows * p.H) return;
  const int64_t tok = row / p.H;
  const int head = (int)(row - tok * p.H);
  float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane < LANES) {
    x = load4(reinterpret_cast<const T*>(p.o) + row * DV + lane * 4);
    if (p.residual) {
      const float4 r = load4(reinterpret_cast<const T*>(p.residual) + row * DV + lane * 4);
      x.x += r.x; x.y += r.y; x.z += r.z; x.w += r.w;
    }
  }
  float ss = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if (lane >= LANES) return;
  if (p.residual_out) store4(reinterpret_cast<T*>(p.residual_out) + row * DV + lane * 4, x);
  const float inv = rsqrtf(ss / (float)DV + p.eps);
  float4 w = make_float4(1.f, 1.f, 1.f, 1.f), b = make_float4(0.f, 0.f, 0.f, 0.f);
  if (p.w) w = load4(reinterpret_cast<const T*>(p.w) + lane * 4);
  if (p.b) b = load4(reinterpret_cast<const T*>(p.b) + lane * 4);
  const float4 g = load4(reinterpret_cast<const T*>(p.gate) + tok * p.gate_row_stride + (int64_t)head * DV + lane * 4);
  float4 y;
  y.x = (x.x * inv * w.x + b.x) * gate_actf(g.x, p.gate_act);
  y.y = (x.y * inv * w.y + b.y) * gate_actf(g.y, p.gate_act);
  y.z = (x.z * inv * w.z + b.z) * gate_actf(g.z, p.gate_act);
  y.w = (x.w * inv * w.w + b.w) * gate_actf(g.w, p.gate_act);
  store4(reinterpret_cast<T*>(p.y) + row * DV + lane * 4, y);
}

template <int DV>
cudaError_t launch_ngx_d(const NormGateExParams& p, cudaStream_t stream) {
  const int64_t blocks = (p.rows * p.H + 7) / 8;
  if (blocks == 0) return cudaSuccess;
  if (p.dtype == KDA_F32)
    norm_gate_ex_kernel<DV, float><<<(unsigned)blocks, 256, 0, stream>>>(p);
  else if (p.dtype == KDA_BF16)
    norm_gate_ex_kernel<DV, bf16><<<(unsigned)blocks, 256, 0, stream>>>(p);
  else
    norm_gate_ex_kernel<DV, f16><<<(unsigned)blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_norm_gate_ex(const NormGateExParams& p, cudaStream_t stream) {
  switch (p.dv) {
    case 16: return launch_ngx_d<16>(p, stream);
    case 64: return launch_ngx_d<64>(p, stream);
    case 128: return launch_ngx_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_norm_gate(const NormGateParams& p, cudaStream_t stream) {
  switch (p.dv) {
    case 16: return launch_ng_d<16>(p, stream);
    case 64: return launch_ng_d<64>(p, stream);
    case 128: return launch_ng_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kda
