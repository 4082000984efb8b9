// Chunked KDA prefill on the Blackwell tensor cores (tcgen05 + TMEM), for
// dk = dv = 128, chunk 64, bf16 inputs (fp32 or bf16 state).
//
// Method ("[Feature][KDA] Add Kimi K3 KDA execution", section "KDA
// execution", step 3).  For a chunk of rows r = 0..63 of one sequence and
// head, chunk-start state S (dk x dv), inclusive in-chunk cumulative
// log-decay G_r = g_0 + ... + g_r:
//   A[r,j]   = beta_r sum_c k_r[c] k_j[c] exp(G_r[c] - G_j[c])          (j < r)
//   Aqk[r,j] = sum_c q_r[c] k_j[c] exp(G_r[c] - G_j[c])                 (j <= r)
//   T' = (I + A)^-1 Diag(beta),  W = T' (K * e^G),  U0 = T' V
//   U  = U0 - W S,   O = scale ((Q * e^G) S + Aqk U)
//   S <- Diag(e^G_last) S + (K * e^(G_last - G))^T U
//
// Two kernels:
//  * kda_intra_kernel -- one CTA per (chunk, head), all chunks in parallel.
//    Computes everything that does not depend on S and stores it in the
//    caller's workspace, already in the shared-memory operand layouts the
//    second kernel's MMAs consume:  [W; Q e^G] (fp16 K-major 128x128),
//    (K e^(G_last-G))^T (fp16 MN-major 128x64), U0 (fp16 64x128), Aqk
//    (fp16 K-major 64x64), e^G_last (fp32 128).  The decay-weighted K K^T and
//    Q K^T use the factorisation exp(G_r - G_m) exp(G_m - G_j) around the
//    chunk's middle row m and a 3-term bf16 split (hi*hi + hi*lo + lo*hi),
//    which keeps them at ~fp32 accuracy; a chunk whose |G - G_m| exceeds 60
//    (extreme decay) takes an exact element-wise path instead.
//  * kda_state_kernel -- one CTA per (sequence, head).  Carries S through the
//    chunks: three fp16 MMAs per chunk (P = [W; Qe^G] S, then Aqk U and
//    (K e^(G_last-G))^T U), the RMSNorm-gate epilogue, checkpoints and the
//    in-place pool write.  The next chunk's operands stream in with bulk
//    async copies while the current chunk computes.
// Precision: the fp16 products (10-bit mantissa) and the fp32 state keep the
// output within the 0.01 bound; see the design notes for the measured budget.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_prefill_shared.cuh"
#include "kda_tc.cuh"

#include <cuda_fp16.h>

namespace kda {
namespace tcp {

constexpr int C = 64;
constexpr int D = 128;
constexpr int kThreads = 256;

// ---- per (chunk slot, head) workspace block --------------------------------
constexpr uint32_t WS_PA = 0;         // fp16 K-major [128 x 128] (SBO 2048): W rows 0-63, Q e^G rows 64-127
constexpr uint32_t WS_KLT = 32768;    // fp16 MN-major [M=c 128 x K=j 64] (K stride 2048)
constexpr uint32_t WS_U0 = 49152;     // fp16 row-major [64][128]
constexpr uint32_t WS_AQK = 65536;    // fp16 K-major [64 x 64] (SBO 1024)
constexpr uint32_t WS_DECAY = 73728;  // fp32 [128]
constexpr uint32_t WS_BYTES = 74240;
constexpr uint32_t WS_COPY0 = 65536;  // PA | KLT | U0
constexpr uint32_t WS_COPY1 = 8704;   // AQK | DECAY

__host__ __device__ inline int64_t num_slots_bound(int64_t T, int N) { return T / C + N; }

// Byte offsets of the operand layouts (16-bit elements).
__device__ __forceinline__ uint32_t kmaj(int r, int k, uint32_t sbo) {
  return (uint32_t)((r >> 3) * sbo + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}
__device__ __forceinline__ uint32_t mnmaj(int m, int k, uint32_t kstr) {
  return (uint32_t)((m >> 3) * 128 + (k >> 3) * kstr + (k & 7) * 16 + (m & 7) * 2);
}

__device__ __forceinline__ uint4 pack_half8(const float* x) {
  uint4 u;
  __half2 h0 = __floats2half2_rn(x[0], x[1]), h1 = __floats2half2_rn(x[2], x[3]);
  __half2 h2 = __floats2half2_rn(x[4], x[5]), h3 = __floats2half2_rn(x[6], x[7]);
  u.x = *reinterpret_cast<uint32_t*>(&h0);
  u.y = *reinterpret_cast<uint32_t*>(&h1);
  u.z = *reinterpret_cast<uint32_t*>(&h2);
  u.w = *reinterpret_cast<uint32_t*>(&h3);
  return u;
}
__device__ __forceinline__ uint4 pack_bf8(const float* x) {
  uint4 u;
  __nv_bfloat162 h0 = __floats2bfloat162_rn(x[0], x[1]), h1 = __floats2bfloat162_rn(x[2], x[3]);
  __nv_bfloat162 h2 = __floats2bfloat162_rn(x[4], x[5]), h3 = __floats2bfloat162_rn(x[6], x[7]);
  u.x = *reinterpret_cast<uint32_t*>(&h0);
  u.y = *reinterpret_cast<uint32_t*>(&h1);
  u.z = *reinterpret_cast<uint32_t*>(&h2);
  u.w = *reinterpret_cast<uint32_t*>(&h3);
  return u;
}
// hi = bf16(x), lo = bf16(x - hi): x ~= hi + lo to ~16 bits.
__device__ __forceinline__ void split_bf8(const float* x, uint4& hi, uint4& lo) {
  float h[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = __bfloat162float(__float2bfloat16_rn(x[i]));
    l[i] = x[i] - h[i];
  }
  hi = pack_bf8(h);
  lo = pack_bf8(l);
}
__device__ __forceinline__ void unpack_bf8(uint4 u, float* x) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(p[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void unpack_half8(uint4 u, float* x) {
  const __half2* p = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(p[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// Bounded wait on an mbarrier phase by every thread; returns false (for all
// threads) when any thread gave up.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity) {
  const bool ok = tc::mbar_wait(bar, parity);
  return __syncthreads_and(ok) != 0;
}

// =====================================================================
// Kernel 1: intra-chunk terms, one CTA per (chunk slot, head)
// =====================================================================
namespace intra {
constexpr uint32_t S_AROW_HI = 0;       // bf16 K-major [128 x 128] (SBO 2048)
constexpr uint32_t S_AROW_LO = 32768;
constexpr uint32_t S_BCOL_HI = 65536;   // bf16 K-major [64 x 128] (SBO 2048)
constexpr uint32_t S_BCOL_LO = 81920;
constexpr uint32_t S_KW = 98304;        // bf16 MN-major [K=j 64 x N=c 128] (K stride 2048)
constexpr uint32_t S_VB = 114688;       // bf16 MN-major [K=j 64 x N=v 128]
constexpr uint32_t S_TP = 131072;       // bf16 K-major [128 x 64] (SBO 1024), rows 64-127 zero
constexpr uint32_t S_END = 147456;
// After the A product completes, the operand area [0, 98304) is reused:
constexpr uint32_t S_AKK = 0;           // fp32 [64][65]   beta-scaled strictly-lower A
constexpr uint32_t S_TF = 16640;        // fp32 [64][65]   (I + A)^-1
constexpr uint32_t S_MB = 33280;        // fp32 [3][16][17] block products of the solve
// exact path scratch inside [0, S_KW): bf16 k, q [64][128], fp32 G [64][128],
// fp32 A_kk, A_qk [64][64]
constexpr uint32_t S_FK = 0, S_FQ = 16384, S_FG = 32768, S_FAKK = 65536, S_FAQK = 65536 + 16384;
static_assert(S_FAQK + 16384 <= S_KW, "exact-path scratch must not reach the live operands");
constexpr uint32_t SMEM_BYTES = S_END + 64 * 4 /*beta*/ + 4 * 64 * 4 /*carry*/ + 4 * 64 * 4 /*Gm*/ +
                                4 * 64 * 4 /*Gl*/ + 64 /*misc*/;
}  // namespace intra

// Element-wise exact A for chunks with extreme decay (rare): no factorisation.
// fk, fq: k and q rows (bf16, exact copies); fg: cumulative gate (fp32).
// Outputs: akk[r][j] = sum_c k_r k_j e^(G_r-G_j) (j < r), aqk[r][j] (j <= r).
__device__ void intra_exact_A(const bf16* fk, const bf16* fq, const float* fg, int n, float* akk, float* aqk) {
  for (int p = threadIdx.x; p < C * C; p += blockDim.x) {
    const int r = p / C, j = p % C;
    float a = 0.f, aq = 0.f;
    if (j <= r && r < n) {
      for (int c = 0; c < D; ++c) {
        const float w = __bfloat162float(fk[j * D + c]) * expf(fg[r * D + c] - fg[j * D + c]);
        a += __bfloat162float(fk[r * D + c]) * w;
        aq += __bfloat162float(fq[r * D + c]) * w;
      }
    }
    akk[r * C + j] = j < r ? a : 0.f;
    aqk[r * C + j] = aq;
  }
}

__global__ void __launch_bounds__(kThreads, 1) kda_intra_kernel(PrefillParams p) {
  using namespace intra;
  extern __shared__ __align__(1024) uint8_t sm[];
  float* s_beta = reinterpret_cast<float*>(sm + S_END);
  float* s_carry = s_beta + 64;       // [side*2+hh][64]
  float* s_gm = s_carry + 4 * 64;     // [side*2+hh][64]
  float* s_gl = s_gm + 4 * 64;        // [side*2+hh][64]
  int* s_misc = reinterpret_cast<int*>(s_gl + 4 * 64);
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t s_tmem;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int side = (warp >> 1) & 1;  // 0: key rows (TMEM lanes 0-63), 1: query rows (64-127)
  const int hh = warp >> 2;          // channel half
  const int r = 32 * (warp & 1) + lane;
  const int head = blockIdx.y;
  const int64_t slot = blockIdx.x;
  const int H = p.H;

  // ---- locate (sequence, chunk) of this slot: slot_first(i) = cu[i]/C + i ----
  if (tid == 0) {
    int lo = 0, hi = p.N - 1, found = -1;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      const int64_t first = (int64_t)p.cu_seqlens[mid] / C + mid;
      if (first <= slot) { found = mid; lo = mid + 1; } else { hi = mid - 1; }
    }
    int seq = -1, kchunk = 0, n = 0;
    if (found >= 0) {
      // skip over zero-length sequences sharing the same first slot
      const int64_t t0 = p.cu_seqlens[found], t1 = p.cu_seqlens[found + 1];
      const int64_t kk = slot - (t0 / C + found);
      const int64_t len = t1 - t0;
      if (t0 >= 0 && len > 0 && t1 <= p.T && kk >= 0 && kk * C < len && p.state_indices[found] >= 0 &&
          p.state_indices[found] < p.num_slots) {
        seq = found;
        kchunk = (int)kk;
        n = (int)(len - kk * C < C ? len - kk * C : C);
      }
    }
    s_misc[0] = seq;
    s_misc[1] = kchunk;
    s_misc[2] = n;
    s_misc[3] = 0;  // range flag
  }
  __syncthreads();
  const int seq = s_misc[0];
  if (seq < 0) return;
  const int n = s_misc[2];
  const int64_t tb = (int64_t)p.cu_seqlens[seq] + (int64_t)s_misc[1] * C;
  uint8_t* ws = reinterpret_cast<uint8_t*>(p.workspace) + (slot * H + head) * (int64_t)WS_BYTES;

  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, 256);
    tc::fence_before_sync();
  }
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
  }
  // zero the lower half of T' (rows 64-127) once
  for (int i = tid; i < 8192 / 16; i += kThreads)
    reinterpret_cast<uint4*>(sm + S_TP + 8192)[i] = make_uint4(0, 0, 0, 0);

  // ---- raw loads for this thread's row and 64 channels ----
  const bf16* gq = reinterpret_cast<const bf16*>(p.q);
  const bf16* gk = reinterpret_cast<const bf16*>(p.k);
  const bf16* gg = reinterpret_cast<const bf16*>(p.g);
  const bf16* gv = reinterpret_cast<const bf16*>(p.v);
  const bool valid = r < n;
  const int64_t rowoff = ((tb + r) * H + head) * (int64_t)D + hh * 64;
  uint4 xr[8];  // k (side 0) or q (side 1), 8 channels per uint4
  float G[64];
  {
    const bf16* src = side == 0 ? gk : gq;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      xr[i] = valid ? __ldg(reinterpret_cast<const uint4*>(src + rowoff) + i) : make_uint4(0, 0, 0, 0);
      const uint4 gr = valid ? __ldg(reinterpret_cast<const uint4*>(gg + rowoff) + i) : make_uint4(0, 0, 0, 0);
      unpack_bf8(gr, G + 8 * i);
#pragma unroll
      for (int u = 0; u < 8; ++u) G[8 * i + u] = fmaxf(G[8 * i + u], kLogDecayFloor);
    }
    if (side == 1) {  // stage V (bf16, exact) in the MN-major B layout of U0 = T' V
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 vr = valid ? __ldg(reinterpret_cast<const uint4*>(gv + rowoff) + i) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sm + S_VB + mnmaj(hh * 64 + 8 * i, r, 2048)) = vr;
      }
    }
    if (side == 0 && hh == 0)
      s_beta[r] = valid ? __bfloat162float(reinterpret_cast<const bf16*>(p.beta)[(tb + r) * H + head]) : 0.f;
  }
  // ---- in-chunk cumulative sum over rows (warp scan over 32 rows + carry) ----
#pragma unroll
  for (int c = 0; c < 64; ++c) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, G[c], d);
      if (lane >= d) G[c] += y;
    }
  }
  const int grp = side * 2 + hh;
  if ((warp & 1) == 0 && lane == 31) {
#pragma unroll
    for (int c = 0; c < 64; ++c) s_carry[grp * 64 + c] = G[c];
  }
  __syncthreads();
  if ((warp & 1) == 1) {
#pragma unroll
    for (int c = 0; c < 64; ++c) G[c] += s_carry[grp * 64 + c];
  }
  const int m = min(C / 2 - 1, n - 1);
  if (r == m) {
#pragma unroll
    for (int c = 0; c < 64; ++c) s_gm[grp * 64 + c] = G[c];
  }
  if (r == n - 1) {
#pragma unroll
    for (int c = 0; c < 64; ++c) s_gl[grp * 64 + c] = G[c];
  }
  __syncthreads();
  // range check for the factorised path
  {
    bool big = false;
#pragma unroll
    for (int c = 0; c < 64; ++c) big |= fabsf(G[c] - s_gm[grp * 64 + c]) > 60.f;
    if (big) atomicOr(&s_misc[3], 1);
  }
  __syncthreads();
  tc::fence_after_sync();
  const bool exact = s_misc[3] != 0;
  const uint32_t tmem = s_tmem;

  // ---- operands ----
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float x[8];
    unpack_bf8(xr[i], x);
    const int c0 = hh * 64 + 8 * i;
    float e_m[8], v1[8], v2[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = 8 * i + u;
      e_m[u] = expf(G[c] - s_gm[grp * 64 + c]);  // e^(G - G_m)
    }
    if (side == 0) {
      // K e^(G-Gm) -> A rows 0-63 ; K e^(Gm-G) -> B rows ; K e^G -> KW ; K e^(Gl-G) -> KLT
#pragma unroll
      for (int u = 0; u < 8; ++u) v1[u] = x[u] * e_m[u];
      uint4 hi, lo;
      if (!exact) {
        split_bf8(v1, hi, lo);
        *reinterpret_cast<uint4*>(sm + S_AROW_HI + kmaj(r, c0, 2048)) = hi;
        *reinterpret_cast<uint4*>(sm + S_AROW_LO + kmaj(r, c0, 2048)) = lo;
#pragma unroll
        for (int u = 0; u < 8; ++u) v2[u] = x[u] / e_m[u];
        split_bf8(v2, hi, lo);
        *reinterpret_cast<uint4*>(sm + S_BCOL_HI + kmaj(r, c0, 2048)) = hi;
        *reinterpret_cast<uint4*>(sm + S_BCOL_LO + kmaj(r, c0, 2048)) = lo;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = 8 * i + u;
        v1[u] = x[u] * expf(G[c]);
        v2[u] = x[u] * expf(s_gl[grp * 64 + c] - G[c]);
      }
      *reinterpret_cast<uint4*>(sm + S_KW + mnmaj(c0, r, 2048)) = pack_bf8(v1);
      *reinterpret_cast<uint4*>(ws + WS_KLT + mnmaj(c0, r, 2048)) = pack_half8(v2);
    } else {
      // Q e^(G-Gm) -> A rows 64-127 ; Q e^G -> [W; Q e^G] rows 64-127 (workspace)
      if (!exact) {
#pragma unroll
        for (int u = 0; u < 8; ++u) v1[u] = x[u] * e_m[u];
        uint4 hi, lo;
        split_bf8(v1, hi, lo);
        *reinterpret_cast<uint4*>(sm + S_AROW_HI + kmaj(64 + r, c0, 2048)) = hi;
        *reinterpret_cast<uint4*>(sm + S_AROW_LO + kmaj(64 + r, c0, 2048)) = lo;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) v1[u] = x[u] * expf(G[8 * i + u]);
      *reinterpret_cast<uint4*>(ws + WS_PA + kmaj(64 + r, c0, 2048)) = pack_half8(v1);
    }
  }
  if (side == 0 && r == 0) {
    float* dec = reinterpret_cast<float*>(ws + WS_DECAY);
#pragma unroll
    for (int c = 0; c < 64; ++c) dec[hh * 64 + c] = expf(s_gl[grp * 64 + c]);
  }

  float* s_akk = reinterpret_cast<float*>(sm + S_AKK);
  float* s_tf = reinterpret_cast<float*>(sm + S_TF);
  float a32[32];
  bool ok = true;
  uint32_t phase = 0;
  if (!exact) {
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
      constexpr uint32_t idA = tc::idesc_f16(128, 64, true, false, false);
      const uint32_t ah = tc::smem_u32(sm + S_AROW_HI), al = tc::smem_u32(sm + S_AROW_LO);
      const uint32_t bh = tc::smem_u32(sm + S_BCOL_HI), bl = tc::smem_u32(sm + S_BCOL_LO);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t o = kk * 256;
        tc::mma_f16(tmem, tc::sdesc(ah + o, 128, 2048), tc::sdesc(bh + o, 128, 2048), idA, kk > 0);
        tc::mma_f16(tmem, tc::sdesc(ah + o, 128, 2048), tc::sdesc(bl + o, 128, 2048), idA, true);
        tc::mma_f16(tmem, tc::sdesc(al + o, 128, 2048), tc::sdesc(bh + o, 128, 2048), idA, true);
      }
      tc::mma_commit(&bar);
    }
    ok = cta_wait(&bar, phase);
    phase ^= 1;
    tc::fence_after_sync();
    if (ok) tc::tmem_ld32(tc::tmem_addr(tmem, 64 * side + (warp & 1) * 32, hh * 32), a32);
    tc::fence_before_sync();
    __syncthreads();
  } else {
    // exact element-wise path: stage k, q and G for every row
    bf16* fk = reinterpret_cast<bf16*>(sm + S_FK);
    bf16* fq = reinterpret_cast<bf16*>(sm + S_FQ);
    float* fg = reinterpret_cast<float*>(sm + S_FG);
    float* fakk = reinterpret_cast<float*>(sm + S_FAKK);
    float* faqk = reinterpret_cast<float*>(sm + S_FAQK);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c0 = hh * 64 + 8 * i;
      *reinterpret_cast<uint4*>((side == 0 ? fk : fq) + r * D + c0) = xr[i];
      if (side == 0) {
#pragma unroll
        for (int u = 0; u < 8; ++u) fg[r * D + c0 + u] = G[8 * i + u];
      }
    }
    __syncthreads();
    intra_exact_A(fk, fq, fg, n, fakk, faqk);
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int j = hh * 32 + u;
      a32[u] = side == 0 ? fakk[r * C + j] : faqk[r * C + j];
    }
    __syncthreads();
  }
  if (!ok) {
    if (tid == 0) latch_status(p.dev_status, KDA_DEV_TIMEOUT);
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
    return;
  }
  // ---- A_kk (beta-scaled, strictly lower) to smem; A_qk (lower) to workspace ----
  if (side == 0) {
    const float br = s_beta[r];
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int j = hh * 32 + u;
      s_akk[r * 65 + j] = (j < r) ? br * a32[u] : 0.f;
    }
  } else {
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) {
      float x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = hh * 32 + 8 * g8 + u;
        x[u] = (j <= r && r < n) ? a32[8 * g8 + u] : 0.f;
      }
      *reinterpret_cast<uint4*>(ws + WS_AQK + kmaj(r, hh * 32 + 8 * g8, 1024)) = pack_half8(x);
    }
  }
  for (int i = tid; i < 64 * 65; i += kThreads) s_tf[i] = 0.f;
  __syncthreads();
  // ---- T = (I + A)^-1 : 16x16 diagonal blocks, then off-diagonal blocks ----
  if (tid < 64) {
    const int b = tid >> 4, jj = tid & 15;
    float x[16];
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
      float s = rr == jj ? 1.f : 0.f;
      if (rr > jj) {
        for (int ii = jj; ii < rr; ++ii) s -= s_akk[(16 * b + rr) * 65 + 16 * b + ii] * x[ii];
      }
      x[rr] = rr >= jj ? s : 0.f;
    }
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) s_tf[(16 * b + rr) * 65 + 16 * b + jj] = x[rr];
  }
  __syncthreads();
  float* s_mb = reinterpret_cast<float*>(sm + S_MB);
  for (int dist = 1; dist < 4; ++dist) {
    const int npairs = 4 - dist;
    // M = sum_{bk=bj}^{bi-1} A[bi][bk] T[bk][bj]
    for (int e = tid; e < npairs * 256; e += kThreads) {
      const int pi = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
      const int bj = pi, bi = pi + dist;
      float s = 0.f;
      for (int kk = 16 * bj; kk < 16 * bi; ++kk) s += s_akk[(16 * bi + rr) * 65 + kk] * s_tf[kk * 65 + 16 * bj + cc];
      s_mb[pi * 272 + rr * 17 + cc] = s;
    }
    __syncthreads();
    // T[bi][bj] = -T[bi][bi] M
    for (int e = tid; e < npairs * 256; e += kThreads) {
      const int pi = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
      const int bj = pi, bi = pi + dist;
      float s = 0.f;
#pragma unroll
      for (int l = 0; l < 16; ++l) s += s_tf[(16 * bi + rr) * 65 + 16 * bi + l] * s_mb[pi * 272 + l * 17 + cc];
      s_tf[(16 * bi + rr) * 65 + 16 * bj + cc] = -s;
    }
    __syncthreads();
  }
  // ---- T' = T Diag(beta) -> bf16 K-major [128 x 64] rows 0-63 ----
  if (side == 0) {
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) {
      float x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = hh * 32 + 8 * g8 + u;
        x[u] = s_tf[r * 65 + j] * s_beta[j];
      }
      *reinterpret_cast<uint4*>(sm + S_TP + kmaj(r, hh * 32 + 8 * g8, 1024)) = pack_bf8(x);
    }
  }
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // ---- W = T' (K e^G) -> TMEM cols 0-127 ; U0 = T' V -> cols 128-255 ----
  if (tid == 0) {
    constexpr uint32_t idW = tc::idesc_f16(128, 128, true, false, true);
    const uint32_t ta = tc::smem_u32(sm + S_TP), kw = tc::smem_u32(sm + S_KW), vb = tc::smem_u32(sm + S_VB);
#pragma unroll
    for (int kk = 0; kk < C / 16; ++kk) {
      const uint64_t a = tc::sdesc(ta + kk * 256, 128, 1024);
      tc::mma_f16(tmem, a, tc::sdesc(kw + kk * 4096, 2048, 128), idW, kk > 0);
      tc::mma_f16(tmem + 128, a, tc::sdesc(vb + kk * 4096, 2048, 128), idW, kk > 0);
    }
    tc::mma_commit(&bar);
  }
  ok = cta_wait(&bar, phase);
  tc::fence_after_sync();
  if (ok && side == 0) {
    // W rows 0-63 of [W; Q e^G] (fp16 K-major) and U0 (fp16 row-major)
    float w32[32];
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const int cbase = hh * 64 + part * 32;
      tc::tmem_ld32(tc::tmem_addr(tmem, (warp & 1) * 32, cbase), w32);
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        *reinterpret_cast<uint4*>(ws + WS_PA + kmaj(r, cbase + 8 * g8, 2048)) = pack_half8(w32 + 8 * g8);
      tc::tmem_ld32(tc::tmem_addr(tmem, (warp & 1) * 32, 128 + cbase), w32);
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        *reinterpret_cast<uint4*>(ws + WS_U0 + (r * 128 + cbase + 8 * g8) * 2) = pack_half8(w32 + 8 * g8);
    }
  }
  if (!ok && tid == 0) latch_status(p.dev_status, KDA_DEV_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// =====================================================================
// Kernel 2: state carry, one CTA per (sequence, head)
// =====================================================================
namespace state {
constexpr uint32_t STAGE = 82432;        // PA|KLT|U0 (65536) | ZERO (8192) | AQK (8192) | DECAY (512)
constexpr uint32_t ST_PA = 0, ST_KLT = 32768, ST_U0 = 49152, ST_ZERO = 65536, ST_AQK = 73728,
                   ST_DECAY = 81920;
constexpr uint32_t S_SOP = 2 * STAGE;    // fp16 MN-major [K=c 128 x N=v 128] (K stride 2048)
constexpr uint32_t S_UOP = S_SOP + 32768;  // fp16 MN-major [K=j 64 x N=v 128]
constexpr uint32_t S_NW = S_UOP + 16384;   // fp32 [128]
constexpr uint32_t S_SS = S_NW + 512;      // fp32 [2][64]
constexpr uint32_t SMEM_BYTES = S_SS + 512;
}  // namespace state

template <typename TS>
__device__ __forceinline__ void load_state_row(const TS* src, float* s) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 v = load4(src + 4 * i);
    s[4 * i] = v.x; s[4 * i + 1] = v.y; s[4 * i + 2] = v.z; s[4 * i + 3] = v.w;
  }
}
template <typename TS>
__device__ __forceinline__ void store_state_row(TS* dst, const float* s) {
#pragma unroll
  for (int i = 0; i < 16; ++i) store4(dst + 4 * i, make_float4(s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]));
}

template <typename TS>
__global__ void __launch_bounds__(kThreads, 1) kda_state_kernel(PrefillParams p) {
  using namespace state;
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar_ld[2];
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, hh = warp >> 2;
  const int lrow = 32 * quad + lane;  // TMEM lane == state row c
  const int seq = blockIdx.x, head = blockIdx.y;
  const int H = p.H;

  SeqInfo si;
  if (!seq_prologue(p, seq, head, true, si)) {
    if (si.zero_rows) zero_out_rows<bf16>(p, si.t0, si.t1, head, 0, D, D);
    return;
  }
  const int64_t t0 = si.t0;
  const int len = (int)(si.t1 - si.t0);
  const int nchunks = (len + C - 1) / C;
  const int64_t slot0 = t0 / C + seq;
  const uint8_t* wsb = reinterpret_cast<const uint8_t*>(p.workspace);
  auto ws_block = [&](int k) { return wsb + ((slot0 + k) * H + head) * (int64_t)WS_BYTES; };

  if (warp == 0) tc::tmem_alloc(&s_tmem, 256);
  if (tid == 0) {
    tc::mbar_init(&bar_ld[0], 1);
    tc::mbar_init(&bar_ld[1], 1);
    tc::mbar_init(&bar_mma, 1);
    tc::mbar_fence_init();
  }
  for (int i = tid; i < 8192 / 16; i += kThreads) {
    reinterpret_cast<uint4*>(sm + ST_ZERO)[i] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(sm + STAGE + ST_ZERO)[i] = make_uint4(0, 0, 0, 0);
  }
  float* s_nw = reinterpret_cast<float*>(sm + S_NW);
  float* s_ss = reinterpret_cast<float*>(sm + S_SS);
  if (p.gate && tid < D) s_nw[tid] = __bfloat162float(reinterpret_cast<const bf16*>(p.norm_w)[tid]);
  // state row lrow, columns [64 hh, 64 hh + 64)
  TS* slot_state = reinterpret_cast<TS*>(p.state_pool) + ((int64_t)si.slot * H + head) * (D * D);
  float S[64];
  load_state_row(slot_state + lrow * D + hh * 64, S);
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const uint32_t tP = tmem, tS = tmem + 128;

  auto issue_load = [&](int k) {
    uint8_t* st = sm + (k & 1) * STAGE;
    uint64_t* b = &bar_ld[k & 1];
    tc::mbar_arrive_expect_tx(b, WS_COPY0 + WS_COPY1);
    tc::bulk_g2s(st, ws_block(k), WS_COPY0, b);
    tc::bulk_g2s(st + ST_AQK, ws_block(k) + WS_AQK, WS_COPY1, b);
  };
  if (tid == 0) issue_load(0);
  int last_issued = 0, last_landed = -1;  // bulk copies in flight: (last_landed, last_issued]

  auto write_sop = [&]() {
#pragma unroll
    for (int g8 = 0; g8 < 8; ++g8)
      *reinterpret_cast<uint4*>(sm + S_SOP + mnmaj(hh * 64 + 8 * g8, lrow, 2048)) = pack_half8(S + 8 * g8);
  };
  write_sop();

  const bf16* ggate = reinterpret_cast<const bf16*>(p.gate);
  bf16* gout = reinterpret_cast<bf16*>(p.out);
  uint32_t mma_phase = 0;
  bool ok = true;
  int k = 0;
  for (; k < nchunks; ++k) {
    const int c0 = k * C;
    const int n = min(C, len - c0);
    uint8_t* st = sm + (k & 1) * STAGE;
    tc::fence_proxy_async();
    tc::fence_before_sync();
    ok = cta_wait(&bar_ld[k & 1], (k >> 1) & 1);
    if (!ok) break;
    last_landed = k;
    tc::fence_after_sync();
    if (k + 1 < nchunks) last_issued = k + 1;
    if (tid == 0) {
      if (k + 1 < nchunks) issue_load(k + 1);
      // P = [W; Q e^G] S  -> tP (rows 0-63: W S, rows 64-127: Q e^G S)
      constexpr uint32_t idP = tc::idesc_f16(128, 128, false, false, true);
      const uint32_t pa = tc::smem_u32(st + ST_PA), so = tc::smem_u32(sm + S_SOP);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc::mma_f16(tP, tc::sdesc(pa + kk * 256, 128, 2048), tc::sdesc(so + kk * 4096, 2048, 128), idP, kk > 0);
      tc::mma_commit(&bar_mma);
    }
    // prefetch this chunk's gate row (query-side threads own output rows)
    uint4 graw[8];
    const int orow = lrow - 64;
    const bool qside = quad >= 2;
    if (p.gate && qside) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        graw[i] = orow < n ? __ldg(reinterpret_cast<const uint4*>(ggate + ((t0 + c0 + orow) * H + head) * D + hh * 64) + i)
                           : make_uint4(0, 0, 0, 0);
    }
    ok = cta_wait(&bar_mma, mma_phase & 1);
    ++mma_phase;
    if (!ok) break;
    tc::fence_after_sync();
    // U = U0 - W S (key-side rows 0-63) -> fp16 MN-major B operand
    if (!qside) {
      float ws32[32], u0[8];
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int cb = hh * 64 + part * 32;
        tc::tmem_ld32(tc::tmem_addr(tP, 32 * quad, cb), ws32);
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) {
          unpack_half8(*reinterpret_cast<const uint4*>(st + ST_U0 + (lrow * 128 + cb + 8 * g8) * 2), u0);
#pragma unroll
          for (int u = 0; u < 8; ++u) u0[u] -= ws32[8 * g8 + u];
          *reinterpret_cast<uint4*>(sm + S_UOP + mnmaj(cb + 8 * g8, lrow, 2048)) = pack_half8(u0);
        }
      }
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
      constexpr uint32_t idO = tc::idesc_f16(128, 128, false, false, true);
      constexpr uint32_t idS = tc::idesc_f16(128, 128, false, true, true);
      const uint32_t z = tc::smem_u32(st + ST_ZERO), uo = tc::smem_u32(sm + S_UOP),
                     kl = tc::smem_u32(st + ST_KLT);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk) {
        const uint64_t b = tc::sdesc(uo + kk * 4096, 2048, 128);
        tc::mma_f16(tP, tc::sdesc(z + kk * 256, 128, 1024), b, idO, true);
        tc::mma_f16(tS, tc::sdesc(kl + kk * 4096, 2048, 128), b, idS, kk > 0);
      }
      tc::mma_commit(&bar_mma);
    }
    ok = cta_wait(&bar_mma, mma_phase & 1);
    ++mma_phase;
    if (!ok) break;
    tc::fence_after_sync();
    // ---- output rows (query side): scale, RMSNorm-gate, store ----
    float o[64];
    if (qside) {
      float t32[32];
      tc::tmem_ld32(tc::tmem_addr(tP, 32 * quad, hh * 64), t32);
#pragma unroll
      for (int u = 0; u < 32; ++u) o[u] = p.scale * t32[u];
      tc::tmem_ld32(tc::tmem_addr(tP, 32 * quad, hh * 64 + 32), t32);
#pragma unroll
      for (int u = 0; u < 32; ++u) o[32 + u] = p.scale * t32[u];
      if (p.gate) {
        float ss = 0.f;
#pragma unroll
        for (int u = 0; u < 64; ++u) ss += o[u] * o[u];
        s_ss[hh * 64 + orow] = ss;
      }
    }
    // ---- state carry: S <- Diag(e^G_last) S + (K e^(G_last-G))^T U ----
    {
      const float d = reinterpret_cast<const float*>(st + ST_DECAY)[lrow];
      float t32[32];
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        tc::tmem_ld32(tc::tmem_addr(tS, 32 * quad, hh * 64 + part * 32), t32);
#pragma unroll
        for (int u = 0; u < 32; ++u) S[part * 32 + u] = d * S[part * 32 + u] + t32[u];
      }
    }
    __syncthreads();  // norm partial sums visible
    if (qside && orow < n) {
      bf16* dst = gout + ((t0 + c0 + orow) * H + head) * D + hh * 64;
      float inv = 1.f;
      if (p.gate) inv = rsqrtf((s_ss[orow] + s_ss[64 + orow]) / (float)D + p.eps);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float y[8];
        if (p.gate) {
          float gt[8];
          unpack_bf8(graw[i], gt);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            y[u] = o[8 * i + u] * inv * s_nw[hh * 64 + 8 * i + u] * sigmoidf_(gt[u]);
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) y[u] = o[8 * i + u];
        }
        reinterpret_cast<uint4*>(dst)[i] = pack_bf8(y);
      }
    }
    // checkpoint after every checkpoint_every tokens of this segment
    if (si.ckpt_ok && p.checkpoint_every > 0 && (c0 + n) % p.checkpoint_every == 0) {
      const int64_t mck = si.ckpt_off + (c0 + n) / p.checkpoint_every - 1;
      TS* dst = reinterpret_cast<TS*>(p.checkpoints) + (mck * H + head) * (int64_t)(D * D) + lrow * D + hh * 64;
      store_state_row(dst, S);
    }
    write_sop();
  }
  if (!ok) {
    if (tid == 0) {
      latch_status(p.dev_status, KDA_DEV_TIMEOUT);
      // let the bulk copies still in flight land before the CTA exits
      for (int j = last_landed + 1; j <= last_issued; ++j) tc::mbar_wait(&bar_ld[j & 1], (j >> 1) & 1);
    }
  } else {
    store_state_row(slot_state + lrow * D + hh * 64, S);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

}  // namespace tcp

bool prefill_tc_supported(const PrefillParams& p) {
  return p.dk == tcp::D && p.dv == tcp::D && p.chunk == tcp::C && p.in_dtype == KDA_BF16;
}

size_t prefill_tc_workspace_bytes(int N, int64_t T, int H) {
  return (size_t)tcp::num_slots_bound(T, N) * (size_t)H * tcp::WS_BYTES;
}

cudaError_t launch_prefill_tc(const PrefillParams& p, cudaStream_t stream) {
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(tcp::kda_intra_kernel), (int)tcp::intra::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const void* sk = p.state_dtype == KDA_F32 ? reinterpret_cast<const void*>(tcp::kda_state_kernel<float>)
                                            : reinterpret_cast<const void*>(tcp::kda_state_kernel<bf16>);
  e = set_smem_once(sk, (int)tcp::state::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t slots = tcp::num_slots_bound(p.T, p.N);
  if (p.T > 0 && slots > 0) {
    dim3 g1((unsigned)slots, (unsigned)p.H);
    tcp::kda_intra_kernel<<<g1, tcp::kThreads, tcp::intra::SMEM_BYTES, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  dim3 g2((unsigned)p.N, (unsigned)p.H);
  if (p.state_dtype == KDA_F32)
    tcp::kda_state_kernel<float><<<g2, tcp::kThreads, tcp::state::SMEM_BYTES, stream>>>(p);
  else
    tcp::kda_state_kernel<bf16><<<g2, tcp::kThreads, tcp::state::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
