// Short causal convolution ahead of the recurrence ("[Feature][KDA] Add Kimi
// K3 KDA execution", section "KDA execution", step 2: run the causal
// convolution and update its cache).  Depthwise over C channels with width W:
//   y[t, c] = act(bias[c] + sum_{i<W} w[c, i] * xe[t - (W-1) + i, c])
// where xe is the sequence extended on the left by its W-1 cached inputs
// (zero without initial state); the cache then holds the sequence's last W-1
// extended inputs, oldest first.  act = identity or SiLU.
//
// Prefill: a CTA covers one 64-token tile (tile k of sequence i has slot
// cu[i]/64 + i + k, the chunk slots of the prefill) and 256 channels (128 for
// fp32) in sub-blocks of 128.  Each sub-block -- the tile, the W-1 inputs
// before it (from x, or at the start of the sequence from the cache), taps
// and bias -- is staged in shared memory by its own group of 16-byte
// asynchronous copies, so a CTA keeps 36 KB of loads in flight with few
// registers, and the second group is still landing while the first is
// computed.  Each warp then takes 8 of the tokens and each lane 4 channels
// (as 2 pairs for the packed fp32 instructions), with a sliding window of the
// W-1 previous inputs in registers.  Only the
// first tile reads the old cache (in its staging) and it writes the new one
// after the staging barrier, so the in-place update needs no ordering across
// CTAs.
// Memory bound: x is read once (plus W-1 halo rows per tile) and y written once.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_tc.cuh"

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
constexpr int kCh = 128;              // channels of a prefill CTA
constexpr int kPV = 4;                // channels per lane (32 lanes x 4)

// The activation on a pair of channels (identity, or SiLU as silu_approx2).
template <int ACT>
__device__ __forceinline__ float2 conv_act2(float2 a) {
  return ACT == 1 ? silu_approx2(a) : a;
}

template <typename T>
__device__ __forceinline__ void unpack4(float4 f, float* o) {
  o[0] = f.x; o[1] = f.y; o[2] = f.z; o[3] = f.w;
}

// Sub-blocks of 128 channels per prefill CTA: two for 16-bit inputs (one
// lookup of the sequence per 256 channels, and the second sub-block's copies
// still in flight while the first is computed), one for fp32 (static shared
// memory is limited to 48 KB).
template <typename T>
struct ConvSplit {
  static constexpr int value = sizeof(T) == 2 ? 2 : 1;
};

template <int W, typename T, int ACT>
__global__ void __launch_bounds__(kPrefillThreads, 4) conv_prefill_kernel(ConvParams p) {
  constexpr int WM = W - 1;
  constexpr int kSub = kTile / (kPrefillThreads / 32);  // tokens per warp (8)
  constexpr int kSplit = ConvSplit<T>::value;
  constexpr int kRows = kTile + WM;                     // WM halo rows + the tile
  constexpr int kPerPiece = 16 / (int)sizeof(T);        // elements per 16-byte piece
  constexpr int kPieces = kCh / kPerPiece;              // pieces per staged row
  constexpr int kTapOff = kRows * kCh;                  // taps [128 channels][W]
  constexpr int kBiasOff = kTapOff + kCh * W;           // bias [128 channels]
  constexpr int kBlk = kBiasOff + kCh;                  // elements per sub-block
  static_assert((kTapOff * sizeof(T)) % 16 == 0 && (kBiasOff * sizeof(T)) % 16 == 0 &&
                    (kBlk * sizeof(T)) % 16 == 0,
                "staged arrays must start on 16-byte boundaries");
  __shared__ __align__(16) T s_buf[kSplit * kBlk];
  __shared__ int s_seq, s_k, s_slot, s_init;
  __shared__ int64_t s_t0, s_t1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t slot = blockIdx.y;
  const int C = p.C;
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
  const int64_t base = t0 + (int64_t)k * kTile;  // first token of this tile
  if (base >= t1) return;                        // a slot past the sequence's last tile
  const int nt = (int)min((int64_t)kTile, t1 - base);
  const T* x = reinterpret_cast<const T*>(p.x);
  T* y = reinterpret_cast<T*>(p.y);
  const int tb = warp * kSub;  // this warp's first token in the tile
  const int n = min(kSub, nt - tb);
  const int cbase = blockIdx.x * kSplit * kCh;
  const int32_t sidx = s_slot;
  if (sidx < 0 || sidx >= p.num_slots) {
    if (sidx != -1 && k == 0 && tid == 0 && blockIdx.x == 0) latch_status(p.dev_status, KDA_DEV_BAD_INDEX);
#pragma unroll
    for (int sb = 0; sb < kSplit; ++sb) {
      const int c0 = cbase + sb * kCh + lane * kPV;
      if (c0 < C)
        for (int u = 0; u < n; ++u) store4(y + (base + tb + u) * C + c0, make_float4(0.f, 0.f, 0.f, 0.f));
    }
    return;
  }
  if (k == 0 && blockIdx.x == 0) check_duplicate_slot(p.state_indices, seq, sidx, p.dev_status);
  T* cache = reinterpret_cast<T*>(p.pool) + (int64_t)sidx * WM * C;
  const bool init = s_init != 0;
  // Stage each sub-block as its own group of 16-byte asynchronous copies: row
  // r is the extended input at token base - WM + r, from x, or (first tile,
  // r < WM) from cache row r, zero without initial state; then the taps and
  // the bias of its channels (zero without bias).
#pragma unroll
  for (int sb = 0; sb < kSplit; ++sb) {
    T* buf = s_buf + sb * kBlk;
    const int cb = cbase + sb * kCh;
    const int nc = min(kCh, C - cb);  // channels of this sub-block (a multiple of 8)
    if (nc > 0) {
      // each thread keeps one 16-byte column of the rows and steps down them
      constexpr int kRowStep = kPrefillThreads / kPieces;
      const int pc = tid % kPieces, r0 = tid / kPieces;
      const bool cvalid = pc * kPerPiece < nc;
      const int c = cb + pc * kPerPiece;
      const T* src = x + (base - WM + r0) * C + c;  // dereferenced only at tokens >= t0
      T* dst = buf + r0 * kCh + pc * kPerPiece;
      for (int r = r0; r < WM + nt; r += kRowStep, src += (int64_t)kRowStep * C, dst += kRowStep * kCh) {
        if (r < WM && k == 0) {  // before the sequence: the cached input, zero without one
          const bool v = cvalid && init;
          tc::cp_async16(dst, v ? cache + (int64_t)r * C + c : x, v);
        } else {
          tc::cp_async16(dst, cvalid ? src : x, cvalid);
        }
      }
      // taps and bias: one piece per thread
      constexpr int kTapPieces = (kCh * W + kCh) / kPerPiece;
      static_assert(kTapPieces <= kPrefillThreads, "one tap piece per thread");
      if (tid < kTapPieces) {
        const int e = tid * kPerPiece;  // element offset in [taps | bias]
        const bool tap = e < kCh * W;
        const bool valid = tap ? e < nc * W : (p.bias != nullptr && e - kCh * W < nc);
        const T* tsrc = tap ? reinterpret_cast<const T*>(p.w) + (int64_t)cb * W + e
                            : (p.bias ? reinterpret_cast<const T*>(p.bias) + cb + (e - kCh * W) : x);
        tc::cp_async16(buf + kTapOff + e, valid ? tsrc : x, valid);
      }
    }
    tc::cp_async_commit();
  }
#pragma unroll
  for (int sb = 0; sb < kSplit; ++sb) {
    if (sb == 0)
      tc::cp_async_wait_group<kSplit - 1>();
    else
      tc::cp_async_wait_group<0>();
    __syncthreads();
    const T* buf = s_buf + sb * kBlk;
    const int c0 = cbase + sb * kCh + lane * kPV;
    if (c0 >= C) continue;
    const T* sx = buf + lane * kPV;
    if (n > 0) {
      // taps of this lane's 4 channels: 4W contiguous staged elements
      float wt[W][kPV], bs[kPV];
#pragma unroll
      for (int q = 0; q < W; ++q) {
        float e[4];
        unpack4<T>(load4(buf + kTapOff + lane * kPV * W + 4 * q), e);
#pragma unroll
        for (int u = 0; u < 4; ++u) wt[(4 * q + u) % W][(4 * q + u) / W] = e[u];
      }
      unpack4<T>(load4(buf + kBiasOff + lane * kPV), bs);
      float win[WM][kPV];
#pragma unroll
      for (int j = 0; j < WM; ++j) unpack4<T>(load4(sx + (tb + j) * kCh), win[j]);
      T* yw = y + (base + tb) * C + c0;
#pragma unroll
      for (int u = 0; u < kSub; ++u) {
        if (u >= n) break;
        float xu[kPV], acc[kPV];
        unpack4<T>(load4(sx + (tb + WM + u) * kCh), xu);
#pragma unroll
        for (int v = 0; v < kPV; v += 2) {  // channel pairs
          float2 a = make_float2(bs[v], bs[v + 1]);
#pragma unroll
          for (int j = 0; j < WM; ++j)
            a = ffma2(make_float2(wt[j][v], wt[j][v + 1]), make_float2(win[j][v], win[j][v + 1]), a);
          a = ffma2(make_float2(wt[WM][v], wt[WM][v + 1]), make_float2(xu[v], xu[v + 1]), a);
          const float2 r = conv_act2<ACT>(a);
          acc[v] = r.x;
          acc[v + 1] = r.y;
        }
        store4(yw + (int64_t)u * C, make_float4(acc[0], acc[1], acc[2], acc[3]));
#pragma unroll
        for (int j = 0; j + 1 < WM; ++j)
#pragma unroll
          for (int v = 0; v < kPV; ++v) win[j][v] = win[j + 1][v];
#pragma unroll
        for (int v = 0; v < kPV; ++v) win[WM - 1][v] = xu[v];
      }
    }
    // New cache, written by the last warp of the first tile once every read
    // of the old one (the staging above) is done: the sequence's last W-1
    // extended inputs, oldest first.  A sequence inside one tile has them all
    // staged.
    if (k == 0 && warp == kPrefillThreads / 32 - 1) {
      const int64_t len = t1 - t0;
#pragma unroll
      for (int j = 0; j < WM; ++j) {
        const int64_t t = t1 - WM + j;
        const float4 v = len <= kTile ? load4(sx + (len + j) * kCh) : load4(x + t * C + c0);
        store4(cache + (int64_t)j * C + c0, v);
      }
    }
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
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // one thread per sequence scans the earlier sequences' cache slots
    for (int j = 0; j < seq; ++j)
      if (p.state_indices[j] == sidx) {
        latch_status(p.dev_status, KDA_DEV_DUP_INDEX);
        break;
      }
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
    acc[v] = p.act == 1 ? silu_approx(a) : a;
  }
  store8(y, acc);
#pragma unroll
  for (int j = 0; j < WM; ++j) store8(cache + (int64_t)j * C, j + 1 < WM ? win[j + 1] : xv);
}

template <int W, typename T>
cudaError_t launch_prefill_w(const ConvParams& p, dim3 grid, cudaStream_t stream) {
  if (p.act == 1)
    conv_prefill_kernel<W, T, 1><<<grid, kPrefillThreads, 0, stream>>>(p);
  else
    conv_prefill_kernel<W, T, 0><<<grid, kPrefillThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefill_t(const ConvParams& p, cudaStream_t stream) {
  const int64_t slots = p.T / kTile + p.N;
  constexpr int ch = ConvSplit<T>::value * kCh;  // channels per CTA
  dim3 grid((unsigned)((p.C + ch - 1) / ch), (unsigned)slots);
  switch (p.W) {
    case 2: return launch_prefill_w<2, T>(p, grid, stream);
    case 3: return launch_prefill_w<3, T>(p, grid, stream);
    case 4: return launch_prefill_w<4, T>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
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
