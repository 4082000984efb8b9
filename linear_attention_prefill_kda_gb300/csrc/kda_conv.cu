// Short causal convolution ahead of the recurrence ("[Feature][KDA] Add Kimi
// K3 KDA execution", section "KDA execution", step 2: run the causal
// convolution and update its cache).  Depthwise over C channels with width W:
//   y[t, c] = act(bias[c] + sum_{i<W} w[c, i] * xe[t - (W-1) + i, c])
// where xe is the sequence extended on the left by its W-1 cached inputs
// (zero without initial state); the cache then holds the sequence's last W-1
// extended inputs, oldest first.  act = identity or SiLU.
//
// Prefill: a CTA covers 256 channels of one 64-token tile (tile k of sequence
// i has slot cu[i]/64 + i + k, the chunk slots of the prefill); each warp
// takes 8 of the tokens, each lane 8 channels, and loads all its inputs
// before computing.  The W-1 inputs before a warp's tokens come from x or,
// at the start of the sequence, from the cache; a sliding window of them
// stays in registers.  Only the first warp of the first tile reads the old
// cache, and the same threads write the new one after their last read of it,
// so the in-place update needs no ordering across CTAs.
// Memory bound: x is read once (plus W-1 halo rows per tile) and y written once.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kTile = 64;     // tokens per CTA row
constexpr int kThreads = 128; // 8 channels each
constexpr int kVec = 8;

template <typename T>
__device__ __forceinline__ void load8(const T* p, float* v) {
  const float4 a = load4(p), b = load4(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <typename T>
__device__ __forceinline__ void store8(T* p, const float* v) {
  store4(p, make_float4(v[0], v[1], v[2], v[3]));
  store4(p + 4, make_float4(v[4], v[5], v[6], v[7]));
}

// 8 consecutive elements kept as loaded (bf16: one 16-byte vector) until use
template <typename T>
struct Raw8;
template <>
struct Raw8<bf16> {
  uint4 v;
  __device__ __forceinline__ void load(const bf16* p) { v = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void unpack(float* o) const {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      o[2 * i] = f.x;
      o[2 * i + 1] = f.y;
    }
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) { a = load4(p); b = load4(p + 4); }
  __device__ __forceinline__ void unpack(float* o) const {
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
  }
};

// taps of 8 consecutive channels: w[c0 .. c0+8, 0 .. W) is 8W contiguous
// elements (16-byte aligned because c0 is a multiple of 8), read as vectors
template <int W, typename T>
__device__ __forceinline__ void load_taps(const T* wp, float (&wt)[W][kVec]) {
#pragma unroll
  for (int q = 0; q < 2 * W; ++q) {
    const float4 f = load4(wp + 4 * q);
    const float e[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) wt[(4 * q + u) % W][(4 * q + u) / W] = e[u];
  }
}

constexpr int kPrefillThreads = 256;  // 8 warps x 8 tokens = one 64-token tile

template <int W, typename T>
__global__ void __launch_bounds__(kPrefillThreads) conv_prefill_kernel(ConvParams p) {
  constexpr int WM = W - 1;
  constexpr int kSub = kTile / (kPrefillThreads / 32);  // tokens per warp (8)
  __shared__ int s_seq, s_k, s_slot, s_init;
  __shared__ int64_t s_t0, s_t1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t slot = blockIdx.y;
  const int c0 = (blockIdx.x * 32 + lane) * kVec;
  const bool chan = c0 < p.C;
  // taps and bias depend only on the channels: fetched while warp 0 finds the
  // sequence
  float wt[W][kVec], bs[kVec];
  if (chan) {
    load_taps<W>(reinterpret_cast<const T*>(p.w) + (int64_t)c0 * W, wt);
    if (p.bias) {
      load8(reinterpret_cast<const T*>(p.bias) + c0, bs);
    } else {
#pragma unroll
      for (int v = 0; v < kVec; ++v) bs[v] = 0.f;
    }
  }
  // (sequence, tile) of this slot: sequence i owns slots [first(i), first(i+1))
  // with first(i) = cu[i]/64 + i; warp 0 scans 32 sequences per step and also
  // fetches the sequence's bounds, cache slot and initial-state flag
  if (tid < 32) {
    if (lane == 0) s_seq = -1;
    __syncwarp();
    for (int base = 0; base < p.N; base += 32) {
      const int i = base + lane;
      bool mine = false;
      int64_t a = 0, b = 0;
      int32_t sl = 0, hi = 1;
      if (i < p.N) {
        a = p.cu_seqlens[i];
        b = p.cu_seqlens[i + 1];
        sl = p.state_indices[i];
        if (p.has_initial_state) hi = p.has_initial_state[i];
        const int64_t first = a / kTile + i;
        const int64_t nx = i + 1 < p.N ? b / kTile + i + 1 : INT64_MAX;
        mine = first <= slot && slot < nx;
      }
      const unsigned who = __ballot_sync(0xffffffffu, mine);
      if (mine && lane == __ffs(who) - 1) {
        s_seq = i;
        s_k = (int)(slot - (a / kTile + i));
        s_t0 = a;
        s_t1 = b;
        s_slot = sl;
        s_init = hi != 0;
      }
      if (who) break;
    }
  }
  __syncthreads();
  const int seq = s_seq;
  if (seq < 0) return;
  const int64_t t0 = s_t0, t1 = s_t1;
  const int k = s_k;
  if (t0 < 0 || t1 > p.T || t1 < t0) {
    if (k == 0 && tid == 0 && blockIdx.x == 0) latch_status(p.dev_status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  // this warp: tokens [ws, we) of tile k; the first warp of the first tile
  // alone reads the old cache and writes the new one
  const int64_t ws = t0 + (int64_t)k * kTile + warp * kSub;
  const int64_t we = min(ws + kSub, t1);
  const bool owner = k == 0 && warp == 0;
  if (ws >= t1 && !(owner && t1 > t0)) return;
  if (!chan) return;
  const int C = p.C;
  const T* x = reinterpret_cast<const T*>(p.x);
  T* y = reinterpret_cast<T*>(p.y);
  const int32_t sidx = s_slot;
  if (sidx < 0 || sidx >= p.num_slots) {
    if (sidx != -1 && owner && c0 == 0) latch_status(p.dev_status, KDA_DEV_BAD_INDEX);
    const float z[kVec] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int64_t t = ws; t < we; ++t) store8(y + t * C + c0, z);
    return;
  }
  T* cache = reinterpret_cast<T*>(p.pool) + (int64_t)sidx * WM * C + c0;
  const bool init = s_init != 0;
  // the W-1 inputs before ws (oldest first): from x, or from the cache for the
  // first tokens of the sequence (the owner's window is the old cache itself)
  float win[WM][kVec];
#pragma unroll
  for (int j = 0; j < WM; ++j) {
    const int64_t tt = ws - WM + j;
    if (tt >= t0) {
      load8(x + tt * C + c0, win[j]);
    } else if (init) {
      load8(cache + (tt - t0 + WM) * (int64_t)C, win[j]);
    } else {
#pragma unroll
      for (int v = 0; v < kVec; ++v) win[j][v] = 0.f;
    }
  }
  // all of this warp's inputs are loaded before the arithmetic starts
  Raw8<T> raw[kSub];
#pragma unroll
  for (int u = 0; u < kSub; ++u)
    if (ws + u < we) raw[u].load(x + (ws + u) * C + c0);
#pragma unroll
  for (int u = 0; u < kSub; ++u) {
    if (ws + u >= we) break;
    float acc[kVec], xu[kVec];
    raw[u].unpack(xu);
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      float a = bs[v];
#pragma unroll
      for (int j = 0; j < WM; ++j) a += wt[j][v] * win[j][v];
      a += wt[WM][v] * xu[v];
      acc[v] = p.act == 1 ? a * sigmoidf_(a) : a;
    }
    store8(y + (ws + u) * C + c0, acc);
#pragma unroll
    for (int j = 0; j + 1 < WM; ++j)
#pragma unroll
      for (int v = 0; v < kVec; ++v) win[j][v] = win[j + 1][v];
#pragma unroll
    for (int v = 0; v < kVec; ++v) win[WM - 1][v] = xu[v];
  }
  if (owner) {
    // new cache: the last W-1 extended inputs of the sequence, oldest first
    float nw[WM][kVec];
#pragma unroll
    for (int j = 0; j < WM; ++j) {
      const int64_t tt = t1 - WM + j;
      if (tt >= t0) {
        load8(x + tt * C + c0, nw[j]);
      } else if (init) {
        // an input still in the old cache (sequences shorter than W-1): only
        // these threads write the cache, and they have not yet
        load8(cache + (tt - t0 + WM) * (int64_t)C, nw[j]);
      } else {
#pragma unroll
        for (int v = 0; v < kVec; ++v) nw[j][v] = 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < WM; ++j) store8(cache + (int64_t)j * C, nw[j]);
  }
}

template <int W, typename T>
__global__ void __launch_bounds__(kThreads) conv_decode_kernel(ConvParams p) {
  constexpr int WM = W - 1;
  const int seq = blockIdx.y;
  const int c0 = (blockIdx.x * kThreads + threadIdx.x) * kVec;
  if (c0 >= p.C) return;
  const int C = p.C;
  T* y = reinterpret_cast<T*>(p.y) + (int64_t)seq * C + c0;
  const int32_t sidx = p.state_indices[seq];
  if (sidx < 0 || sidx >= p.num_slots) {
    if (sidx != -1 && c0 == 0) latch_status(p.dev_status, KDA_DEV_BAD_INDEX);
    const float z[kVec] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    store8(y, z);
    return;
  }
  T* cache = reinterpret_cast<T*>(p.pool) + (int64_t)sidx * WM * C + c0;
  float win[WM][kVec], xv[kVec], bs[kVec], acc[kVec];
#pragma unroll
  for (int j = 0; j < WM; ++j) load8(cache + (int64_t)j * C, win[j]);
  load8(reinterpret_cast<const T*>(p.x) + (int64_t)seq * C + c0, xv);
  if (p.bias) load8(reinterpret_cast<const T*>(p.bias) + c0, bs);
  else
#pragma unroll
    for (int v = 0; v < kVec; ++v) bs[v] = 0.f;
  float wt[W][kVec];
  load_taps<W>(reinterpret_cast<const T*>(p.w) + (int64_t)c0 * W, wt);
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    float a = bs[v];
#pragma unroll
    for (int j = 0; j < WM; ++j) a += wt[j][v] * win[j][v];
    a += wt[WM][v] * xv[v];
    acc[v] = p.act == 1 ? a * sigmoidf_(a) : a;
  }
  store8(y, acc);
#pragma unroll
  for (int j = 0; j < WM; ++j) store8(cache + (int64_t)j * C, j + 1 < WM ? win[j + 1] : xv);
}

template <typename T>
cudaError_t launch_prefill_t(const ConvParams& p, cudaStream_t stream) {
  const int64_t slots = p.T / kTile + p.N;
  dim3 grid((unsigned)((p.C + 32 * kVec - 1) / (32 * kVec)), (unsigned)slots);  // 256 channels x 64 tokens
  switch (p.W) {
    case 2: conv_prefill_kernel<2, T><<<grid, kPrefillThreads, 0, stream>>>(p); break;
    case 3: conv_prefill_kernel<3, T><<<grid, kPrefillThreads, 0, stream>>>(p); break;
    case 4: conv_prefill_kernel<4, T><<<grid, kPrefillThreads, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_decode_t(const ConvParams& p, cudaStream_t stream) {
  dim3 grid((unsigned)((p.C + kThreads * kVec - 1) / (kThreads * kVec)), (unsigned)p.N);
  switch (p.W) {
    case 2: conv_decode_kernel<2, T><<<grid, kThreads, 0, stream>>>(p); break;
    case 3: conv_decode_kernel<3, T><<<grid, kThreads, 0, stream>>>(p); break;
    case 4: conv_decode_kernel<4, T><<<grid, kThreads, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv_prefill(const ConvParams& p, cudaStream_t stream) {
  return p.dtype == KDA_F32 ? launch_prefill_t<float>(p, stream) : launch_prefill_t<bf16>(p, stream);
}

cudaError_t launch_conv_decode(const ConvParams& p, cudaStream_t stream) {
  return p.dtype == KDA_F32 ? launch_decode_t<float>(p, stream) : launch_decode_t<bf16>(p, stream);
}

}  // namespace kda
