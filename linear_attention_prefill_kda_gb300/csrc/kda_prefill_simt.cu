// Chunked KDA prefill, CUDA-core (FP32 FMA) variant.
//
// This is the portable reference path of the library: every contraction is
// an fp32 FMA loop, the intra-chunk decay factors are evaluated element by
// element (exp(G_r - G_j) with j <= r, never overflowing), and it supports
// every shape the ABI accepts.  The tensor-core path (kda_prefill_tc.cu)
// handles the large shapes; this one is used where that path does not apply.
//
// Method ("[Feature][KDA] Add Kimi K3 KDA execution", section "KDA
// execution", step 3: chunk prefill over the cumulative gate).  For a chunk of
// rows r = 0..C-1 of one sequence and head, with chunk-start state S
// (dk x dv) and inclusive cumulative log-decay G_r = g_0 + ... + g_r:
//   A[r,j]   = beta_r sum_c k_r[c] k_j[c] exp(G_r[c] - G_j[c])     (j < r)
//   Aqk[r,j] = sum_c q_r[c] k_j[c] exp(G_r[c] - G_j[c])            (j <= r)
//   (I + A) U = Diag(beta) (V - (K * exp(G)) S)       (forward substitution)
//   O        = scale ((Q * exp(G)) S + Aqk U)
//   S       <- Diag(exp(G_last)) S + (K * exp(G_last - G))^T U
// which reproduces the token recurrence S_t = (I - b k k^T) Diag(e^g) S + b k v^T,
// o_t = scale S_t^T q_t exactly in exact arithmetic.  State pool indexing,
// padding and checkpoints follow the ABI contract in kda.h.
//
// Launch: one CTA per (sequence, head, value slab of BV columns); the columns
// of S evolve independently given q, k, g, beta, so slabs need no exchange.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_prefill_shared.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;

template <int DK, int C, int BV>
struct SimtLayout {
  static constexpr int LDK = DK + 4;  // padded row strides (keep 16 B alignment)
  static constexpr int LDV = BV + 4;
  static constexpr int LDA = C + 1;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_Q = OFF_K + C * LDK;
  static constexpr int OFF_G = OFF_Q + C * LDK;
  static constexpr int OFF_V = OFF_G + C * LDK;
  static constexpr int OFF_S = OFF_V + C * LDV;
  static constexpr int OFF_A = OFF_S + DK * LDV;
  static constexpr int OFF_AQ = OFF_A + C * LDA;
  static constexpr int OFF_GL = OFF_AQ + C * LDA;
  static constexpr int OFF_B = OFF_GL + DK;
  static constexpr int FLOATS = OFF_B + C;
  static constexpr size_t BYTES = sizeof(float) * FLOATS;
  static_assert(OFF_V % 4 == 0 && OFF_S % 4 == 0, "float4 alignment of V and S tiles");
};

template <int DK, int DV, int C, int BV, typename TI, typename TS>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(PrefillParams p) {
  using L = SimtLayout<DK, C, BV>;
  constexpr int RN = BV / 16;  // register tile: columns per thread
  static_assert(BV % 16 == 0 && C % 16 == 0 && DK % 16 == 0, "16-multiples");
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  float* sK = sm + L::OFF_K;
  float* sQ = sm + L::OFF_Q;
  float* sG = sm + L::OFF_G;
  float* sV = sm + L::OFF_V;  // V slab, then U
  float* sS = sm + L::OFF_S;
  float* sA = sm + L::OFF_A;
  float* sAq = sm + L::OFF_AQ;
  float* sGl = sm + L::OFF_GL;
  float* sB = sm + L::OFF_B;

  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;
  const int seq = blockIdx.x, head = blockIdx.y, slab = blockIdx.z;
  const int v0 = slab * BV;
  const int H = p.H;

  SeqInfo si;
  if (!seq_prologue(p, seq, head, slab == 0, si)) {
    if (si.zero_rows) zero_out_rows<TI>(p, si.t0, si.t1, head, v0, BV, DV);
    return;
  }
  const int64_t t0 = si.t0;
  const int len = (int)(si.t1 - si.t0);

  const TI* gq = reinterpret_cast<const TI*>(p.q);
  const TI* gk = reinterpret_cast<const TI*>(p.k);
  const TI* gg = reinterpret_cast<const TI*>(p.g);
  const TI* gv = reinterpret_cast<const TI*>(p.v);
  const TI* gb = reinterpret_cast<const TI*>(p.beta);
  TI* gout = reinterpret_cast<TI*>(p.out);
  TS* slot_state = reinterpret_cast<TS*>(p.state_pool) + ((int64_t)si.slot * H + head) * (DK * DV);

  for (int i = tid; i < DK * BV; i += kThreads) {
    const int c = i / BV, v = i % BV;
    sS[c * L::LDV + v] = si.init ? to_f32(slot_state[c * DV + v0 + v]) : 0.f;
  }

  for (int c0 = 0; c0 < len; c0 += C) {
    const int n = min(C, len - c0);
    // ---- load the chunk (rows >= n are zero: they contribute nothing) ----
    for (int i = tid; i < C * DK; i += kThreads) {
      const int r = i / DK, c = i % DK;
      float kv = 0.f, qv = 0.f, gvv = 0.f;
      if (r < n) {
        const int64_t off = ((t0 + c0 + r) * H + head) * DK + c;
        kv = to_f32(gk[off]);
        qv = to_f32(gq[off]);
        gvv = fmaxf(to_f32(gg[off]), kLogDecayFloor);
      }
      sK[r * L::LDK + c] = kv;
      sQ[r * L::LDK + c] = qv;
      sG[r * L::LDK + c] = gvv;
    }
    for (int i = tid; i < C * BV; i += kThreads) {
      const int r = i / BV, v = i % BV;
      sV[r * L::LDV + v] = r < n ? to_f32(gv[((t0 + c0 + r) * H + head) * DV + v0 + v]) : 0.f;
    }
    for (int r = tid; r < C; r += kThreads) sB[r] = r < n ? to_f32(gb[(t0 + c0 + r) * H + head]) : 0.f;
    __syncthreads();
    // ---- in-chunk cumulative gate ----
    for (int c = tid; c < DK; c += kThreads) {
      float run = 0.f;
      for (int r = 0; r < C; ++r) {
        run += sG[r * L::LDK + c];
        sG[r * L::LDK + c] = run;
      }
      sGl[c] = run;  // rows >= n add zero, so this is G at the last valid row
    }
    __syncthreads();
    // ---- decay-weighted K K^T and Q K^T, exact per element ----
    for (int pidx = tid; pidx < C * C; pidx += kThreads) {
      const int r = pidx / C, j = pidx % C;
      float a = 0.f, aq = 0.f;
      if (j <= r) {
        const float* kr = sK + r * L::LDK;
        const float* kj = sK + j * L::LDK;
        const float* qr = sQ + r * L::LDK;
        const float* Gr = sG + r * L::LDK;
        const float* Gj = sG + j * L::LDK;
#pragma unroll 8
        for (int c = 0; c < DK; ++c) {
          const float w = kj[c] * expf(Gr[c] - Gj[c]);
          a += kr[c] * w;
          aq += qr[c] * w;
        }
      }
      sA[r * L::LDA + j] = j < r ? sB[r] * a : 0.f;
      sAq[r * L::LDA + j] = aq;
    }
    __syncthreads();
    // ---- decay-scaled operands: Q*e^G, K*e^G, K*e^(G_last - G) ----
    for (int i = tid; i < C * DK; i += kThreads) {
      const int r = i / DK, c = i % DK;
      const float gam = sG[r * L::LDK + c];
      const float e = expf(gam);
      const float kv = sK[r * L::LDK + c];
      sQ[r * L::LDK + c] *= e;
      sK[r * L::LDK + c] = kv * e;
      sG[r * L::LDK + c] = kv * expf(sGl[c] - gam);
    }
    __syncthreads();
    // ---- right-hand side: beta_r (v_r - S^T (k_r e^G_r)) ----
    {
      constexpr int RM = C / 16;
      float acc[RM][RN];
#pragma unroll
      for (int a = 0; a < RM; ++a)
#pragma unroll
        for (int b = 0; b < RN; ++b) acc[a][b] = 0.f;
      for (int c = 0; c < DK; ++c) {
        float sv[RN];
#pragma unroll
        for (int b = 0; b < RN; ++b) sv[b] = sS[c * L::LDV + tx * RN + b];
#pragma unroll
        for (int a = 0; a < RM; ++a) {
          const float kr = sK[(ty + 16 * a) * L::LDK + c];
#pragma unroll
          for (int b = 0; b < RN; ++b) acc[a][b] += kr * sv[b];
        }
      }
#pragma unroll
      for (int a = 0; a < RM; ++a) {
        const int r = ty + 16 * a;
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          float* dst = sV + r * L::LDV + tx * RN + b;
          *dst = sB[r] * (*dst - acc[a][b]);
        }
      }
    }
    __syncthreads();
    // ---- forward substitution (I + A) U = rhs, row by row ----
    for (int r = 1; r < C; ++r) {
      for (int v = tid; v < BV; v += kThreads) {
        float s = sV[r * L::LDV + v];
        for (int j = 0; j < r; ++j) s -= sA[r * L::LDA + j] * sV[j * L::LDV + v];
        sV[r * L::LDV + v] = s;
      }
      __syncthreads();
    }
    // ---- output: scale ((Q e^G) S + Aqk U) ----
    {
      constexpr int RM = C / 16;
      float acc[RM][RN];
#pragma unroll
      for (int a = 0; a < RM; ++a)
#pragma unroll
        for (int b = 0; b < RN; ++b) acc[a][b] = 0.f;
      for (int c = 0; c < DK; ++c) {
        float sv[RN];
#pragma unroll
        for (int b = 0; b < RN; ++b) sv[b] = sS[c * L::LDV + tx * RN + b];
#pragma unroll
        for (int a = 0; a < RM; ++a) {
          const float qr = sQ[(ty + 16 * a) * L::LDK + c];
#pragma unroll
          for (int b = 0; b < RN; ++b) acc[a][b] += qr * sv[b];
        }
      }
      for (int j = 0; j < C; ++j) {
        float uv[RN];
#pragma unroll
        for (int b = 0; b < RN; ++b) uv[b] = sV[j * L::LDV + tx * RN + b];
#pragma unroll
        for (int a = 0; a < RM; ++a) {
          const float w = sAq[(ty + 16 * a) * L::LDA + j];
#pragma unroll
          for (int b = 0; b < RN; ++b) acc[a][b] += w * uv[b];
        }
      }
#pragma unroll
      for (int a = 0; a < RM; ++a) {
        const int r = ty + 16 * a;
        const int64_t off = ((t0 + c0 + r) * H + head) * DV + v0 + tx * RN;
        float o[RN];
#pragma unroll
        for (int b = 0; b < RN; ++b) o[b] = p.scale * acc[a][b];
        if constexpr (BV == DV) {
          // One slab holds the whole row: the output norm-gate is fused here.
          // Row r's DV columns lie on the 16 threads of this ty (lanes of one
          // half-warp), so its sum of squares is a 16-lane reduction.
          if (p.gate) {
            float ss = 0.f;
#pragma unroll
            for (int b = 0; b < RN; ++b) ss += o[b] * o[b];
#pragma unroll
            for (int m = 8; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
            const float inv = rsqrtf(ss / (float)DV + p.eps);
            if (r < n) {
              const TI* gt = reinterpret_cast<const TI*>(p.gate) + off;
              const TI* wt = reinterpret_cast<const TI*>(p.norm_w) + tx * RN;
#pragma unroll
              for (int b = 0; b < RN; ++b) o[b] *= inv * to_f32(wt[b]) * gate_actf(to_f32(gt[b]), p.gate_act);
            }
          }
        }
        if (r < n) {
          if (p.o_scratch) {
#pragma unroll
            for (int b = 0; b < RN; ++b) p.o_scratch[off + b] = o[b];
          } else {
#pragma unroll
            for (int b = 0; b < RN; ++b) gout[off + b] = from_f32<TI>(o[b]);
          }
        }
      }
    }
    __syncthreads();
    // ---- state carry: S <- Diag(e^G_last) S + (K e^(G_last-G))^T U ----
    {
      constexpr int RM = DK / 16;
      float acc[RM][RN];
#pragma unroll
      for (int a = 0; a < RM; ++a)
#pragma unroll
        for (int b = 0; b < RN; ++b) acc[a][b] = 0.f;
      for (int r = 0; r < C; ++r) {
        float uv[RN];
#pragma unroll
        for (int b = 0; b < RN; ++b) uv[b] = sV[r * L::LDV + tx * RN + b];
#pragma unroll
        for (int a = 0; a < RM; ++a) {
          const float kl = sG[r * L::LDK + ty + 16 * a];
#pragma unroll
          for (int b = 0; b < RN; ++b) acc[a][b] += kl * uv[b];
        }
      }
#pragma unroll
      for (int a = 0; a < RM; ++a) {
        const int c = ty + 16 * a;
        const float d = expf(sGl[c]);
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          float* s = sS + c * L::LDV + tx * RN + b;
          *s = d * (*s) + acc[a][b];
        }
      }
    }
    __syncthreads();
    // ---- checkpoint after every checkpoint_every tokens of this segment ----
    if (si.ckpt_ok && p.checkpoint_every > 0 && (c0 + n) % p.checkpoint_every == 0) {
      const int64_t m = si.ckpt_off + (c0 + n) / p.checkpoint_every - 1;
      TS* dst = reinterpret_cast<TS*>(p.checkpoints) + (m * H + head) * (int64_t)(DK * DV);
      for (int i = tid; i < DK * BV; i += kThreads) {
        const int c = i / BV, v = i % BV;
        dst[c * DV + v0 + v] = from_f32<TS>(sS[c * L::LDV + v]);
      }
    }
  }
  for (int i = tid; i < DK * BV; i += kThreads) {
    const int c = i / BV, v = i % BV;
    slot_state[c * DV + v0 + v] = from_f32<TS>(sS[c * L::LDV + v]);
  }
}

template <int D, int C, typename TI, typename TS>
cudaError_t launch_simt_t(const PrefillParams& p, cudaStream_t stream) {
  constexpr int BV = D >= 64 ? 64 : D;
  using L = SimtLayout<D, C, BV>;
  auto kern = prefill_simt_kernel<D, D, C, BV, TI, TS>;
  const cudaError_t attr = set_smem_once(reinterpret_cast<const void*>(kern), (int)L::BYTES);
  if (attr != cudaSuccess) return attr;
  dim3 grid(p.N, p.H, D / BV);
  kern<<<grid, kThreads, L::BYTES, stream>>>(p);
  return cudaGetLastError();
}

template <int D, int C>
cudaError_t launch_simt_dc(const PrefillParams& p, cudaStream_t stream) {
  if (p.in_dtype == KDA_F32 && p.state_dtype == KDA_F32) return launch_simt_t<D, C, float, float>(p, stream);
  if (p.in_dtype == KDA_F32 && p.state_dtype == KDA_BF16) return launch_simt_t<D, C, float, bf16>(p, stream);
  if (p.in_dtype == KDA_BF16 && p.state_dtype == KDA_F32) return launch_simt_t<D, C, bf16, float>(p, stream);
  return launch_simt_t<D, C, bf16, bf16>(p, stream);
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillParams& p, cudaStream_t stream) {
  const int d = p.dk;
  if (p.chunk == 16) {
    if (d == 16) return launch_simt_dc<16, 16>(p, stream);
    if (d == 64) return launch_simt_dc<64, 16>(p, stream);
    if (d == 128) return launch_simt_dc<128, 16>(p, stream);
  } else if (p.chunk == 64) {
    if (d == 16) return launch_simt_dc<16, 64>(p, stream);
    if (d == 64) return launch_simt_dc<64, 64>(p, stream);
    if (d == 128) return launch_simt_dc<128, 64>(p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kda
