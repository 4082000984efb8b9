// Multi-token recurrent decode for speculative-decoding verification, and the
// commit of the accepted state.
//
// "[Feature][KDA] Add Kimi K3 KDA execution", section "Metadata construction"
// (speculative decode is a separate batch kind), and the FlashKDA summary's
// risk section (checkpoint recovery inside speculative decoding is the case
// its tests leave out): each sequence runs K candidate tokens through the
// recurrence from its pool state, and the state after every token is kept so
// that, once the drafts are verified, the state after the last accepted token
// can be committed to the slot.
//
// kda_decode_multi: per (sequence, head), K steps of the one-token update of
// kda_decode.cu with the state slice held in registers across the steps;
// after step t the state is stored to token_states[sequence, t] (state dtype,
// when token_states is given) and the outputs of step t are written (with the
// optional RMSNorm-gate).
// The pool slot itself is rewritten only when write_back is set.
//
// kda_commit_accepted: pool[slot_i] = token_states[i, a_i - 1] for a_i >= 1
// accepted tokens; a_i == 0 leaves the slot as it was.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

template <int DK, int DV>
struct MultiShape {
  static constexpr int CG = DV / 4;
  static constexpr int RG = (256 / CG) < DK ? (256 / CG) : DK;
  static constexpr int RPT = DK / RG;
  static constexpr int THREADS = CG * RG;
};

constexpr int kTokBlock = 8;  // tokens whose inputs are staged in shared memory at once

template <int DK, int DV, typename TI, typename TS>
__global__ void __launch_bounds__(MultiShape<DK, DV>::THREADS)
decode_multi_kernel(DecodeMultiParams p) {
  using Sh = MultiShape<DK, DV>;
  constexpr int CG = Sh::CG, RG = Sh::RG, RPT = Sh::RPT;
  const int tid = threadIdx.x;
  const int cg = tid % CG, rg = tid / CG;
  const int seq = (int)(blockIdx.x / (unsigned)p.H), head = (int)(blockIdx.x % (unsigned)p.H);
  const int H = p.H, K = p.K;

  // the inputs of up to kTokBlock tokens, loaded together before they are used
  __shared__ float s_q[kTokBlock][DK], s_k[kTokBlock][DK], s_a[kTokBlock][DK];
  __shared__ float s_v[kTokBlock][DV], s_gt[kTokBlock][DV], s_beta[kTokBlock], s_qk[kTokBlock];
  __shared__ float s_pk[RG][DV], s_pq[RG][DV];

  const int32_t slot = p.state_indices[seq];
  if (slot < 0 || slot >= p.num_slots) {
    if (slot != -1 && tid == 0) latch_status(p.dev_status, KDA_DEV_BAD_INDEX);
    for (int t = 0; t < K; ++t) {
      TI* out = reinterpret_cast<TI*>(p.out) + (((int64_t)seq * K + t) * H + head) * DV;
      for (int j = tid; j < DV; j += blockDim.x) out[j] = from_f32<TI>(0.f);
    }
    return;
  }
  if (head == 0) check_duplicate_slot(p.state_indices, seq, slot, p.dev_status);
  TS* S = reinterpret_cast<TS*>(p.state_pool) + ((int64_t)slot * H + head) * (DK * DV);
  float4 st[RPT];
#pragma unroll
  for (int m = 0; m < RPT; ++m) st[m] = load4(S + (rg + m * RG) * DV + cg * 4);

  for (int tb = 0; tb < K; tb += kTokBlock) {
    const int nb = min(kTokBlock, K - tb);
    __syncthreads();  // the previous block's inputs are no longer read
    for (int e = tid; e < nb * DK; e += blockDim.x) {
      const int u = e / DK, i = e % DK;
      const int64_t row = ((int64_t)seq * K + tb + u) * H + head;
      s_q[u][i] = to_f32(reinterpret_cast<const TI*>(p.q)[row * DK + i]);
      s_k[u][i] = to_f32(reinterpret_cast<const TI*>(p.k)[row * DK + i]);
      s_a[u][i] = expf(to_f32(reinterpret_cast<const TI*>(p.g)[row * DK + i]));
    }
    for (int e = tid; e < nb * DV; e += blockDim.x) {
      const int u = e / DV, j = e % DV;
      const int64_t row = ((int64_t)seq * K + tb + u) * H + head;
      s_v[u][j] = to_f32(reinterpret_cast<const TI*>(p.v)[row * DV + j]);
      if (p.gate) s_gt[u][j] = to_f32(reinterpret_cast<const TI*>(p.gate)[row * DV + j]);
    }
    if (tid < nb) s_beta[tid] = to_f32(reinterpret_cast<const TI*>(p.beta)[((int64_t)seq * K + tb + tid) * H + head]);
    __syncthreads();
    // q . k of every token of the block (one warp per token)
    for (int u = tid >> 5; u < nb; u += blockDim.x >> 5) {
      float acc = 0.f;
      for (int i = tid & 31; i < DK; i += 32) acc += s_q[u][i] * s_k[u][i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if ((tid & 31) == 0) s_qk[u] = acc;
    }
    for (int u = 0; u < nb; ++u) {
      const int t = tb + u;
      const int64_t row = ((int64_t)seq * K + t) * H + head;  // token-major [N*K, H, *]
      float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
      for (int m = 0; m < RPT; ++m) {
        const int i = rg + m * RG;
        const float a = s_a[u][i];
        st[m].x *= a; st[m].y *= a; st[m].z *= a; st[m].w *= a;
        const float ki = s_k[u][i], qi = s_q[u][i];
        pk.x += ki * st[m].x; pk.y += ki * st[m].y; pk.z += ki * st[m].z; pk.w += ki * st[m].w;
        pq.x += qi * st[m].x; pq.y += qi * st[m].y; pq.z += qi * st[m].z; pq.w += qi * st[m].w;
      }
      __syncthreads();  // s_pk / s_pq of the previous token read by all (and s_qk ready)
      *reinterpret_cast<float4*>(&s_pk[rg][cg * 4]) = pk;
      *reinterpret_cast<float4*>(&s_pq[rg][cg * 4]) = pq;
      __syncthreads();
      float tk[4] = {0.f, 0.f, 0.f, 0.f}, tq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const float4 a = *reinterpret_cast<const float4*>(&s_pk[r][cg * 4]);
        const float4 b = *reinterpret_cast<const float4*>(&s_pq[r][cg * 4]);
        tk[0] += a.x; tk[1] += a.y; tk[2] += a.z; tk[3] += a.w;
        tq[0] += b.x; tq[1] += b.y; tq[2] += b.z; tq[3] += b.w;
      }
      const float beta = s_beta[u];
      float u4[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) u4[c] = beta * (s_v[u][cg * 4 + c] - tk[c]);
#pragma unroll
      for (int m = 0; m < RPT; ++m) {
        const float ki = s_k[u][rg + m * RG];
        st[m].x += ki * u4[0]; st[m].y += ki * u4[1]; st[m].z += ki * u4[2]; st[m].w += ki * u4[3];
      }
      if (p.token_states) {
        TS* ts = reinterpret_cast<TS*>(p.token_states) + row * (DK * DV);
#pragma unroll
        for (int m = 0; m < RPT; ++m) store4_stream(ts + (rg + m * RG) * DV + cg * 4, st[m]);
      }
      if (rg == 0) {
        const float qk = s_qk[u];
        float o[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) o[c] = p.scale * (tq[c] + qk * u4[c]);
        if (p.gate) {
          float ss = o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3];
          const unsigned mask = CG == 32 ? 0xffffffffu : ((1u << CG) - 1u);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1)
            if (off < CG) ss += __shfl_xor_sync(mask, ss, off);
          const float inv = rsqrtf(ss / (float)DV + p.eps);
          const float4 w = load4(reinterpret_cast<const TI*>(p.norm_w) + cg * 4);
          o[0] *= inv * w.x * gate_actf(s_gt[u][cg * 4 + 0], p.gate_act);
          o[1] *= inv * w.y * gate_actf(s_gt[u][cg * 4 + 1], p.gate_act);
          o[2] *= inv * w.z * gate_actf(s_gt[u][cg * 4 + 2], p.gate_act);
          o[3] *= inv * w.w * gate_actf(s_gt[u][cg * 4 + 3], p.gate_act);
        }
        store4(reinterpret_cast<TI*>(p.out) + row * DV + cg * 4, make_float4(o[0], o[1], o[2], o[3]));
      }
    }
  }
  if (p.write_back) {
#pragma unroll
    for (int m = 0; m < RPT; ++m) store4(S + (rg + m * RG) * DV + cg * 4, st[m]);
  }
}

// pool[slot_i] = token_states[i, a_i - 1]; one CTA per (sequence, head), 16-byte copies.
template <typename TS>
__global__ void __launch_bounds__(256) commit_kernel(CommitParams p) {
  const int seq = (int)(blockIdx.x / (unsigned)p.H), head = (int)(blockIdx.x % (unsigned)p.H);
  const int32_t slot = p.state_indices[seq];
  const int32_t a = p.num_accepted[seq];
  if (slot == -1 || a == 0) return;
  if (slot < -1 || slot >= p.num_slots || a < 0 || a > p.K) {
    if (threadIdx.x == 0) latch_status(p.dev_status, KDA_DEV_BAD_INDEX);
    return;
  }
  if (head == 0)
    check_duplicate_slot(p.state_indices, seq, slot, p.dev_status,
                         [&](int j) { return p.num_accepted[j] > 0; });
  const int64_t elems = (int64_t)p.dk * p.dv;
  const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const TS*>(p.token_states) +
                                                    (((int64_t)seq * p.K + (a - 1)) * p.H + head) * elems);
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<TS*>(p.state_pool) + ((int64_t)slot * p.H + head) * elems);
  const int64_t n16 = elems * (int64_t)sizeof(TS) / 16;
  for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = __ldcs(src + i);
}

template <int D, typename TI, typename TS>
cudaError_t launch_multi_t(const DecodeMultiParams& p, cudaStream_t stream) {
  const int64_t blocks = (int64_t)p.N * p.H;
  decode_multi_kernel<D, D, TI, TS><<<(unsigned)blocks, MultiShape<D, D>::THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_multi_d(const DecodeMultiParams& p, cudaStream_t stream) {
  if (p.in_dtype == KDA_F32 && p.state_dtype == KDA_F32) return launch_multi_t<D, float, float>(p, stream);
  if (p.in_dtype == KDA_F32 && p.state_dtype == KDA_BF16) return launch_multi_t<D, float, bf16>(p, stream);
  if (p.in_dtype == KDA_BF16 && p.state_dtype == KDA_F32) return launch_multi_t<D, bf16, float>(p, stream);
  return launch_multi_t<D, bf16, bf16>(p, stream);
}

}  // namespace

cudaError_t launch_decode_multi(const DecodeMultiParams& p, cudaStream_t stream) {
  switch (p.dk) {
    case 16: return launch_multi_d<16>(p, stream);
    case 64: return launch_multi_d<64>(p, stream);
    case 128: return launch_multi_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_commit(const CommitParams& p, cudaStream_t stream) {
  const int64_t blocks = (int64_t)p.N * p.H;
  if (p.state_dtype == KDA_F32)
    commit_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(p);
  else
    commit_kernel<bf16><<<(unsigned)blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
