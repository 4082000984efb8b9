// Per-sequence prologue shared by the prefill kernels: sequence bounds,
// state-slot validation, padding rows and checkpoint offsets.  These are the
// ABI's boundary rules (kda.h), not method arithmetic:
//  - state_indices[i] == -1 is a graph-padding sequence whose output rows are
//    zeroed ("[Feature][KDA] Add Kimi K3 KDA execution", section "KDA
//    execution", step 5);
//  - a zero-length sequence is a no-op;
//  - a sequence whose has_initial_state flag is 0 starts from a zero state
//    (a new prompt: "[Feature][KDA] ...", section "Metadata construction");
//  - sequence i owns checkpoint entries [off_i, off_i + floor(len_i / I)),
//    off_i the exclusive prefix sum, written to ckpt_offsets.
#pragma once

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

struct SeqInfo {
  int64_t t0, t1;
  int64_t ckpt_off;
  int32_t slot;
  bool zero_rows;
  bool ckpt_ok;
  bool init;  // start from the slot's state (false: from zero, a new prompt)
};

// Must be called by every thread of the block (it contains __syncthreads).
// Returns true when the sequence has work; otherwise si.zero_rows says
// whether the caller should zero its output rows.
__device__ __forceinline__ bool seq_prologue(const PrefillParams& p, int seq, int head,
                                             bool first_slab, SeqInfo& si) {
  __shared__ long long s_off;
  if (threadIdx.x == 0) s_off = 0;
  __syncthreads();
  const int I = p.checkpoint_every;
  if (I > 0) {
    long long part = 0;
    for (int j = threadIdx.x; j < seq; j += blockDim.x) {
      const int32_t a = p.cu_seqlens[j], b = p.cu_seqlens[j + 1];
      part += b > a ? (b - a) / I : 0;
    }
    if (part) atomicAdd(reinterpret_cast<unsigned long long*>(&s_off), (unsigned long long)part);
  }
  __syncthreads();
  si.t0 = p.cu_seqlens[seq];
  si.t1 = p.cu_seqlens[seq + 1];
  si.ckpt_off = s_off;
  si.zero_rows = false;
  si.ckpt_ok = false;
  si.slot = -1;
  si.init = p.has_initial_state == nullptr || p.has_initial_state[seq] != 0;
  const int64_t len = si.t1 - si.t0;
  if (first_slab && head == 0 && threadIdx.x == 0 && p.ckpt_offsets) {
    p.ckpt_offsets[seq] = (int32_t)si.ckpt_off;
    if (seq == p.N - 1) p.ckpt_offsets[p.N] = (int32_t)(si.ckpt_off + (I > 0 && len > 0 ? len / I : 0));
  }
  if (si.t0 < 0 || len < 0 || si.t1 > p.T) {
    if (threadIdx.x == 0) latch_status(p.dev_status, KDA_DEV_BAD_SEQLENS);
    return false;
  }
  si.slot = p.state_indices[seq];
  if (si.slot < 0 || si.slot >= p.num_slots || (p.conv && si.slot >= p.conv_num_slots)) {
    if (si.slot != -1 && threadIdx.x == 0) latch_status(p.dev_status, KDA_DEV_BAD_INDEX);
    si.zero_rows = true;
    return false;
  }
  if (first_slab && head == 0) check_duplicate_slot(p.state_indices, seq, si.slot, p.dev_status);
  if (len == 0) return false;
  if (I > 0) {
    si.ckpt_ok = si.ckpt_off + len / I <= p.checkpoint_capacity;
    if (!si.ckpt_ok && threadIdx.x == 0) latch_status(p.dev_status, KDA_DEV_CKPT_OVERFLOW);
  }
  return true;
}

template <typename TI>
__device__ __forceinline__ void zero_out_rows(const PrefillParams& p, int64_t t0, int64_t t1, int head,
                                              int v0, int bv, int dv) {
  TI* out = reinterpret_cast<TI*>(p.out);
  const int64_t n = (t1 - t0) * bv;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t t = t0 + i / bv;
    const int v = (int)(i % bv);
    out[(t * p.H + head) * dv + v0 + v] = from_f32<TI>(0.f);
  }
}

}  // namespace kda
