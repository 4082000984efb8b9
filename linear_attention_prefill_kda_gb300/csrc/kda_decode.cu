// Recurrent KDA decode step: one token per sequence, state updated in place in
// the indexed pool ("[Feature][KDA] Add Kimi K3 KDA execution", section "KDA
// execution", step 4; pool indexing as in "[KK] Prepare B12X Kimi KDA
// prefill ...", section "Behavior").
//
// Per (sequence, head) and value column j, with alpha = exp(g):
//     p_j = sum_i alpha_i k_i S_ij            (key read of the decayed state)
//     r_j = sum_i alpha_i q_i S_ij            (query read of the decayed state)
//     u_j = beta (v_j - p_j)
//     S_ij <- alpha_i S_ij + k_i u_j
//     o_j = scale (r_j + (q . k) u_j)        (= scale * (S_new^T q)_j)
// then the optional RMSNorm-gate (sigmoid or SiLU gate) over the dv outputs of
// the row.
//
// The step is a pure HBM stream over the state (dk*dv elements read and
// written once): one CTA per (sequence, head); a warp reads whole rows of the
// state with 16-byte vector loads, every thread keeps its slice of the state
// in registers between the read and the write, and the column sums are
// combined through shared memory.
#include <algorithm>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_tc.cuh"

namespace kda {
namespace {

template <int DK, int DV>
struct DecodeShape {
  static constexpr int CG = DV / 4;                                   // 4-column groups
  static constexpr int RG = (256 / CG) < DK ? (256 / CG) : DK;          // row groups
  static constexpr int RPT = DK / RG;                                   // rows per thread
  static constexpr int THREADS = CG * RG;
  static_assert(DV % 4 == 0 && DV / 4 <= 32, "dv must be a multiple of 4 and <= 128");
  static_assert(DK % RG == 0, "row groups must tile dk");
};

// One CTA walks rows (sequence, head) with a stride of the grid; while it
// computes a row from the state in its registers, the next row's state is
// already on its way into shared memory by one bulk copy, so that each SM
// keeps two states in flight per CTA instead of one.
template <int DK, int DV, typename TI, typename TS>
__global__ void __launch_bounds__(DecodeShape<DK, DV>::THREADS)
decode_kernel(DecodeParams p) {
  using Sh = DecodeShape<DK, DV>;
  constexpr int CG = Sh::CG, RG = Sh::RG, RPT = Sh::RPT;
  constexpr uint32_t SBYTES = DK * DV * sizeof(TS);
  const int tid = threadIdx.x;
  const int cg = tid % CG, rg = tid / CG;

  extern __shared__ __align__(16) uint8_t s_next[];  // the next row's state, prefetched
  // q, k and the decay of a row, by row parity: a row's are written before
  // the barrier that starts it, while the previous row's may still be read
  __shared__ float s_qb[2][DK], s_kb[2][DK], s_ab[2][DK];
  __shared__ float s_pk[RG][DV], s_pq[RG][DV];
  __shared__ float s_qk;
  __shared__ __align__(8) uint64_t bar_pf;
  if (tid == 0) {
    tc::mbar_init(&bar_pf, 1);
    tc::mbar_fence_init();
  }
  __syncthreads();

  const int64_t rows = (int64_t)p.N * p.H;
  auto state_block = [&](int32_t slot, int64_t r) {
    return reinterpret_cast<TS*>(p.state_pool) + ((int64_t)slot * p.H + r % p.H) * (DK * DV);
  };
  auto slot_ok = [&](int32_t slot) { return slot >= 0 && slot < p.num_slots; };
  uint32_t parity = 0;       // phase of bar_pf the next prefetch completes
  bool pf = false;           // this row's state is being prefetched into s_next
  bool prefetching = true;   // turned off for good after a wait that gave up
  bool in_flight = false;    // a copy that gave up may still land (drained at the end)
  int par = 0;               // row parity of this CTA's walk
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, par ^= 1) {
    const int seq = (int)(row / p.H), head = (int)(row % p.H);
    const int32_t slot = p.state_indices[seq];
    const bool valid = slot_ok(slot);
    float* s_q = s_qb[par];
    float* s_k = s_kb[par];
    float* s_a = s_ab[par];
    // Issue the state loads first: they are the whole cost of the step.
    float4 st[RPT];
    bool ok = true;
    if (valid) {
      const TS* src = state_block(slot, row);
      if (pf) {
        ok = tc::mbar_wait(&bar_pf, parity);
        parity ^= 1;
        if (ok) src = reinterpret_cast<const TS*>(s_next);
      }
#pragma unroll
      for (int m = 0; m < RPT; ++m) st[m] = load4(src + (rg + m * RG) * DV + cg * 4);
      const TI* q = reinterpret_cast<const TI*>(p.q) + row * DK;
      const TI* k = reinterpret_cast<const TI*>(p.k) + row * DK;
      const TI* g = reinterpret_cast<const TI*>(p.g) + row * DK;
      for (int i = tid; i < DK; i += blockDim.x) {
        s_q[i] = to_f32(q[i]);
        s_k[i] = to_f32(k[i]);
        s_a[i] = expf(to_f32(g[i]));
      }
    }
    // every thread has read s_next and written this row's q, k and decay; a
    // wait that gave up (its copy may still land) ends the prefetching
    const bool all_ok = __syncthreads_and(ok) != 0;
    if (!all_ok && pf) {
      if (tid == 0) latch_status(p.dev_status, KDA_DEV_TIMEOUT);
      prefetching = false;
      in_flight = true;
    }
    pf = false;
    const int64_t nrow = row + gridDim.x;
    if (prefetching && nrow < rows) {
      const int32_t nslot = p.state_indices[nrow / p.H];
      if (slot_ok(nslot)) {
        pf = true;
        if (tid == 0) {
          tc::fence_proxy_async();  // the generic reads of s_next precede the copy's writes
          tc::mbar_arrive_expect_tx(&bar_pf, SBYTES);
          tc::bulk_g2s(s_next, state_block(nslot, nrow), SBYTES, &bar_pf);
        }
      }
    }

    TI* out = reinterpret_cast<TI*>(p.out) + row * DV;
    if (!valid) {
      if (slot != -1 && tid == 0) latch_status(p.dev_status, KDA_DEV_BAD_INDEX);
      for (int j = tid; j < DV; j += blockDim.x) out[j] = from_f32<TI>(0.f);
      continue;
    }
    if (head == 0) check_duplicate_slot(p.state_indices, seq, slot, p.dev_status);
    TS* S = state_block(slot, row);

    if (tid < 32) {
      float acc = 0.f;
      for (int i = tid; i < DK; i += 32) acc += s_q[i] * s_k[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (tid == 0) s_qk = acc;
    }

    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
      const int i = rg + m * RG;
      const float a = s_a[i];
      st[m].x *= a; st[m].y *= a; st[m].z *= a; st[m].w *= a;
      const float ki = s_k[i], qi = s_q[i];
      pk.x += ki * st[m].x; pk.y += ki * st[m].y; pk.z += ki * st[m].z; pk.w += ki * st[m].w;
      pq.x += qi * st[m].x; pq.y += qi * st[m].y; pq.z += qi * st[m].z; pq.w += qi * st[m].w;
    }
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
    const int64_t tok = row;  // one token per sequence: token index == sequence
    const float beta = to_f32(reinterpret_cast<const TI*>(p.beta)[tok]);
    const float4 v4 = load4(reinterpret_cast<const TI*>(p.v) + row * DV + cg * 4);
    float u[4];
    u[0] = beta * (v4.x - tk[0]);
    u[1] = beta * (v4.y - tk[1]);
    u[2] = beta * (v4.z - tk[2]);
    u[3] = beta * (v4.w - tk[3]);

#pragma unroll
    for (int m = 0; m < RPT; ++m) {
      const int i = rg + m * RG;
      const float ki = s_k[i];
      float4 sv = st[m];
      sv.x += ki * u[0]; sv.y += ki * u[1]; sv.z += ki * u[2]; sv.w += ki * u[3];
      store4(S + i * DV + cg * 4, sv);
    }

    if (rg == 0) {  // row group 0 (the first CG threads of warp 0) owns the output
      const float qk = s_qk;
      float o[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) o[c] = p.scale * (tq[c] + qk * u[c]);
      if (p.gate) {
        float ss = o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3];
        const unsigned mask = CG == 32 ? 0xffffffffu : ((1u << CG) - 1u);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          if (off < CG) ss += __shfl_xor_sync(mask, ss, off);
        const float inv = rsqrtf(ss / (float)DV + p.eps);
        const float4 gt = load4(reinterpret_cast<const TI*>(p.gate) + row * DV + cg * 4);
        const float4 w = load4(reinterpret_cast<const TI*>(p.norm_w) + cg * 4);
        o[0] *= inv * w.x * gate_actf(gt.x, p.gate_act);
        o[1] *= inv * w.y * gate_actf(gt.y, p.gate_act);
        o[2] *= inv * w.z * gate_actf(gt.z, p.gate_act);
        o[3] *= inv * w.w * gate_actf(gt.w, p.gate_act);
      }
      store4(out + cg * 4, make_float4(o[0], o[1], o[2], o[3]));
    }
  }
  // a copy whose wait gave up lands (bounded) before the shared memory is released
  if (in_flight && tid == 0) tc::mbar_wait(&bar_pf, parity ^ 1);
}

template <int DK, int DV, typename TI, typename TS>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  using Sh = DecodeShape<DK, DV>;
  constexpr int SBYTES = DK * DV * (int)sizeof(TS);
  void (*kern)(DecodeParams) = decode_kernel<DK, DV, TI, TS>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), SBYTES);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Sh::THREADS, SBYTES)) != cudaSuccess)
    return e;
  const int64_t rows = (int64_t)p.N * p.H;
  const int64_t grid = std::min<int64_t>(rows, (int64_t)std::max(per_sm, 1) * sms);
  kern<<<(unsigned)grid, Sh::THREADS, SBYTES, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecodeParams& p, cudaStream_t stream) {
  if (p.in_dtype == KDA_F32 && p.state_dtype == KDA_F32) return launch_decode_t<D, D, float, float>(p, stream);
  if (p.in_dtype == KDA_F32 && p.state_dtype == KDA_BF16) return launch_decode_t<D, D, float, bf16>(p, stream);
  if (p.in_dtype == KDA_BF16 && p.state_dtype == KDA_F32) return launch_decode_t<D, D, bf16, float>(p, stream);
  return launch_decode_t<D, D, bf16, bf16>(p, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  switch (p.dk) {
    case 16: return launch_decode_d<16>(p, stream);
    case 64: return launch_decode_d<64>(p, stream);
    case 128: return launch_decode_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kda
