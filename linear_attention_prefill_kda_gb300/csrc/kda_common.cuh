// Shared device helpers for libkda kernels: dtype conversion and the device
// status latch.  No method arithmetic lives here.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

using bf16 = __nv_bfloat16;
using f16 = __half;

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<bf16>(bf16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_f32<f16>(f16 x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// Four consecutive elements <-> float4.  p must be aligned to 4 elements.
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const bf16* p) {
  uint2 raw = *reinterpret_cast<const uint2*>(p);
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
  float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ float4 load4(const f16* p) {
  uint2 raw = *reinterpret_cast<const uint2*>(p);
  const float2 fa = __half22float2(*reinterpret_cast<__half2*>(&raw.x));
  const float2 fb = __half22float2(*reinterpret_cast<__half2*>(&raw.y));
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store4(f16* p, float4 v) {
  __half2 a = __floats2half2_rn(v.x, v.y);
  __half2 b = __floats2half2_rn(v.z, v.w);
  uint2 raw;
  raw.x = *reinterpret_cast<uint32_t*>(&a);
  raw.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = raw;
}
__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 raw;
  raw.x = *reinterpret_cast<uint32_t*>(&a);
  raw.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = raw;
}

// Streaming variants for data touched once per call (evict-first in L2).
__device__ __forceinline__ float4 load4_stream(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4_stream(const bf16* p) {
  uint2 raw = __ldcs(reinterpret_cast<const uint2*>(p));
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
  float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store4_stream(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }
__device__ __forceinline__ void store4_stream(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 raw;
  raw.x = *reinterpret_cast<uint32_t*>(&a);
  raw.y = *reinterpret_cast<uint32_t*>(&b);
  __stcs(reinterpret_cast<uint2*>(p), raw);
}

// First error wins; a NULL status pointer discards the code.
__device__ __forceinline__ void latch_status(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// A state slot that an earlier sequence of the same call also names: the two
// sequences would read and write one state concurrently.  Run by the threads
// of one CTA per sequence (no barrier); `live(j)` says whether sequence j
// uses its slot at all.
template <typename Live>
__device__ __forceinline__ void check_duplicate_slot(const int32_t* idx, int seq, int32_t slot, int32_t* status,
                                                     Live live) {
  if (slot < 0) return;
  for (int j = threadIdx.x; j < seq; j += blockDim.x)
    if (idx[j] == slot && live(j)) {
      latch_status(status, KDA_DEV_DUP_INDEX);
      break;
    }
}
__device__ __forceinline__ void check_duplicate_slot(const int32_t* idx, int seq, int32_t slot, int32_t* status) {
  check_duplicate_slot(idx, seq, slot, status, [](int) { return true; });
}

__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// Gate activation of the RMSNorm-gate: sigmoid (act 0) or SiLU x*sigmoid(x) (act 1).
__device__ __forceinline__ float gate_actf(float x, int act) {
  const float s = sigmoidf_(x);
  return act == KDA_GATE_SILU ? x * s : s;
}

// Floor applied to the per-token log-decay g by the chunked prefill kernels.
// exp(-30) = 9.4e-14, so a token below the floor still erases the history to
// within 1e-13 of the state; the floor keeps the in-chunk prefix sums of g
// bounded (|G| <= 30 * chunk) so that their fp32 rounding stays ~1e-4 in the
// exponent instead of swallowing the small decays that follow a huge one.
constexpr float kLogDecayFloor = -30.0f;

// SiLU a * sigmoid(a) = a / (1 + 2^(-a log2 e)), from the approximate base-2
// exponential and reciprocal instructions (each within a few fp32 ulps; the
// limits come out exactly: 0 for a -> -inf through 1/inf, a for a -> +inf)
__device__ __forceinline__ float silu_approx(float a) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(a * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return a * r;
}

// Packed fp32 pair arithmetic (two IEEE round-to-nearest operations in one
// instruction, sm_100 family): the same results as the scalar forms, half
// the instructions.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// silu_approx on a pair, with the multiplications and the addition packed.
__device__ __forceinline__ float2 silu_approx2(float2 a) {
  const float2 m = fmul2(a, make_float2(-1.4426950408889634f, -1.4426950408889634f));
  float2 e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.x) : "f"(m.x));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.y) : "f"(m.y));
  const float2 den = fadd2(e, make_float2(1.f, 1.f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(den.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(den.y));
  return fmul2(a, r);
}

// eps of the L2 normalisation of q and k in the prefill with the convolution
// fused in: q <- q / sqrt(|q|^2 + eps).
constexpr float kConvL2Eps = KDA_CONV_L2_EPS;

}  // namespace kda
