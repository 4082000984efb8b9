/*
 * kda_oracle.c -- fp64 CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or table with the CUDA
 * library.
 *
 * What it computes (the gated delta rule with per-channel decay that the
 * pages' KDA operators evaluate -- "[Feature][KDA] Add Kimi K3 KDA
 * execution", section "KDA execution", steps 3 and 4: chunk prefill and
 * recurrent decode):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * evaluated token by token, in the plain order
 *     1. S <- Diag(exp g_t) S            (decay, per key channel)
 *     2. u <- beta_t (v_t - S^T k_t)     (delta-rule residual)
 *     3. S <- S + k_t u^T                (write)
 *     4. o_t <- scale * S^T q_t          (read-out of the post-update state)
 * which expands to exactly the formula above.  No chunking, blocking or
 * reordering.
 *
 * State pool ("[KK] Prepare B12X Kimi KDA prefill ...", section "Behavior":
 * the kernel consumes state-pool indices directly): sequence i starts from
 * pool[state_indices[i]] and its final state is written back to the same
 * slot.  state_indices[i] == -1 marks a graph-padding sequence whose output
 * rows are zeroed and whose pool slot is untouched ("[Feature][KDA] ...",
 * section "KDA execution", step 5).  A zero-length sequence is a no-op.
 *
 * Checkpoint states ("FlashKDA ... bf16 checkpoint", section on the
 * motivation: intermediate breakpoint states that join SSM state across
 * segments): after every `checkpoint_every` tokens of a sequence (counted
 * from the start of this call's segment) a copy of S is appended.  Layout
 * [sum_i floor(len_i/I), H, dk, dv], ordered by sequence then position;
 * ckpt_offsets[i] is the exclusive prefix sum of floor(len_i/I).
 *
 * Output norm-gate ("[Feature][KDA] ...", first section: FusedRMSNormGated,
 * output normalisation and gating; its test coverage names sigmoid and SiLU):
 *     y = o / sqrt(mean_dv(o^2) + eps) * w * act(gate),  act = sigmoid or SiLU
 * per (token, head) row, weight w[dv] shared by the heads.
 *
 * Sequences without initial state ("[Feature][KDA] ...", section "Metadata
 * construction": a one-token prompt without state is still prefill): when a
 * has_initial_state flag is 0 the sequence starts from S = 0 instead of its
 * slot's content.
 *
 * Everything is fp64.  Layouts are row-major, last dimension contiguous:
 *   q,k,g [T,H,dk]   v [T,H,dv]   beta [T,H]   out/gate [T,H,dv]
 *   pool  [num_slots,H,dk,dv]     checkpoints [cap,H,dk,dv]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_INDEX -2
#define ORACLE_ERR_CAPACITY -3
#define ORACLE_ERR_NOMEM -4

/* One token of the recurrence on a [dk, dv] state, steps 1-4 above. */
static void token_step(double* S, int dk, int dv, const double* q, const double* k,
                       const double* v, const double* g, double beta, double scale,
                       double* u /* scratch [dv] */, double* o /* [dv] */) {
  for (int c = 0; c < dk; ++c) {
    const double a = exp(g[c]);
    double* row = S + (size_t)c * dv;
    for (int j = 0; j < dv; ++j) row[j] *= a;
  }
  for (int j = 0; j < dv; ++j) u[j] = 0.0;
  for (int c = 0; c < dk; ++c) {
    const double* row = S + (size_t)c * dv;
    for (int j = 0; j < dv; ++j) u[j] += k[c] * row[j];
  }
  for (int j = 0; j < dv; ++j) u[j] = beta * (v[j] - u[j]);
  for (int c = 0; c < dk; ++c) {
    double* row = S + (size_t)c * dv;
    for (int j = 0; j < dv; ++j) row[j] += k[c] * u[j];
  }
  for (int j = 0; j < dv; ++j) o[j] = 0.0;
  for (int c = 0; c < dk; ++c) {
    const double* row = S + (size_t)c * dv;
    for (int j = 0; j < dv; ++j) o[j] += q[c] * row[j];
  }
  for (int j = 0; j < dv; ++j) o[j] *= scale;
}

/* y = o / sqrt(mean(o^2) + eps) * w * act(gate) over one row of dv, where
 * act is the sigmoid (act == 0) or SiLU, x * sigmoid(x) (act == 1): the two
 * gate activations the pages' norm-gate coverage lists. */
static void norm_gate_row(const double* o, const double* gate, const double* w, double eps,
                          int dv, int act, double* y) {
  double ss = 0.0;
  for (int j = 0; j < dv; ++j) ss += o[j] * o[j];
  const double inv = 1.0 / sqrt(ss / (double)dv + eps);
  for (int j = 0; j < dv; ++j) {
    const double sig = 1.0 / (1.0 + exp(-gate[j]));
    const double a = act == 1 ? gate[j] * sig : sig;
    y[j] = o[j] * inv * w[j] * a;
  }
}

int kda_oracle_norm_gate(const double* o, const double* gate, const double* w, double eps,
                         double* y, int64_t rows, int dv, int act) {
  if (!o || !gate || !w || !y || rows < 0 || dv <= 0 || act < 0 || act > 1) return ORACLE_ERR_ARG;
  for (int64_t r = 0; r < rows; ++r)
    norm_gate_row(o + r * dv, gate + r * dv, w, eps, dv, act, y + r * dv);
  return ORACLE_OK;
}

/*
 * Norm-gate variants covered by the norm-gate tests of "[Feature][KDA] Add
 * Kimi K3 KDA execution" (testing section: fp16/bf16, sigmoid/SiLU, packed
 * gate strides, affine and residual/prenorm paths).  Per (row r, head h):
 *   x = o + residual                      (residual optional)
 *   residual_out = x                      (the prenorm output, optional)
 *   z = x / sqrt(mean(x^2) + eps) * w + b (w optional: 1; b optional: 0)
 *   y = z * act(gate)                     act = sigmoid or SiLU
 * o, residual, y, residual_out are [rows, H, dv]; w, b are [dv]; the gate of
 * (r, h) starts at gate[r * gate_row_stride + h * dv].
 */
int kda_oracle_norm_gate_ex(const double* o, const double* residual, const double* gate,
                            int64_t gate_row_stride, const double* w, const double* b, double eps,
                            int act, double* y, double* residual_out, int64_t rows, int H, int dv) {
  if (!o || !gate || !y || rows < 0 || H <= 0 || dv <= 0 || act < 0 || act > 1) return ORACLE_ERR_ARG;
  if (gate_row_stride < (int64_t)H * dv) return ORACLE_ERR_ARG;
  for (int64_t r = 0; r < rows; ++r) {
    for (int h = 0; h < H; ++h) {
      const int64_t off = (r * H + h) * (int64_t)dv;
      const double* gt = gate + r * gate_row_stride + (int64_t)h * dv;
      double ss = 0.0;
      for (int j = 0; j < dv; ++j) {
        const double x = o[off + j] + (residual ? residual[off + j] : 0.0);
        if (residual_out) residual_out[off + j] = x;
        ss += x * x;
      }
      const double inv = 1.0 / sqrt(ss / (double)dv + eps);
      for (int j = 0; j < dv; ++j) {
        const double x = o[off + j] + (residual ? residual[off + j] : 0.0);
        const double z = x * inv * (w ? w[j] : 1.0) + (b ? b[j] : 0.0);
        const double sig = 1.0 / (1.0 + exp(-gt[j]));
        y[off + j] = z * (act == 1 ? gt[j] * sig : sig);
      }
    }
  }
  return ORACLE_OK;
}

/*
 * Short causal convolution ahead of the recurrence ("[Feature][KDA] Add Kimi
 * K3 KDA execution", section "KDA execution", step 2: run the causal
 * convolution and update its cache).  Depthwise over `channels`, width W, on
 * each sequence's tokens extended on the left by the W-1 cached inputs (zero
 * when the sequence has no initial state):
 *   y[t, c] = act(bias[c] + sum_{i<W} w[c, i] * xe[t - (W-1) + i, c])
 * act = identity (0) or SiLU (1).  The cache of a sequence afterwards holds
 * its last W-1 extended inputs, oldest first: cache[j, c] = xe[t1 - (W-1) + j, c].
 * x, y: [T, channels]; w: [channels, W]; bias: [channels] or NULL; cache pool:
 * [num_slots, W-1, channels], updated in place.  A padding sequence (index -1)
 * gets zero outputs and leaves the pool alone.
 */
int kda_oracle_conv_prefill(const double* x, const double* w, const double* bias,
                            const int32_t* cu_seqlens, int N, const int32_t* state_indices,
                            const int32_t* has_initial_state, double* pool, int64_t num_slots,
                            int channels, int W, int act, double* y) {
  if (!x || !w || !cu_seqlens || !state_indices || !pool || !y || N < 0 || channels <= 0 || W < 1 ||
      act < 0 || act > 1)
    return ORACLE_ERR_ARG;
  const int Wm = W - 1;
  for (int i = 0; i < N; ++i) {
    const int64_t t0 = cu_seqlens[i], t1 = cu_seqlens[i + 1];
    if (t1 < t0) return ORACLE_ERR_ARG;
    const int32_t slot = state_indices[i];
    if (slot < 0) {
      for (int64_t t = t0; t < t1; ++t)
        for (int c = 0; c < channels; ++c) y[t * channels + c] = 0.0;
      continue;
    }
    if (slot >= num_slots) return ORACLE_ERR_ARG;
    if (t1 == t0) continue;
    double* cache = pool + (int64_t)slot * Wm * channels;
    const int init = has_initial_state ? has_initial_state[i] != 0 : 1;
    const int64_t len = t1 - t0;
    for (int c = 0; c < channels; ++c) {
      /* the extended sequence xe[0 .. Wm + len) for this channel */
      double* xe = (double*)malloc(sizeof(double) * (size_t)(Wm + len));
      if (!xe) return ORACLE_ERR_ARG;
      for (int j = 0; j < Wm; ++j) xe[j] = init ? cache[(int64_t)j * channels + c] : 0.0;
      for (int64_t t = 0; t < len; ++t) xe[Wm + t] = x[(t0 + t) * channels + c];
      for (int64_t t = 0; t < len; ++t) {
        double acc = bias ? bias[c] : 0.0;
        for (int k = 0; k < W; ++k) acc += w[(int64_t)c * W + k] * xe[t + k];
        y[(t0 + t) * channels + c] = act == 1 ? acc / (1.0 + exp(-acc)) : acc;
      }
      for (int j = 0; j < Wm; ++j) cache[(int64_t)j * channels + c] = xe[len + j];
      free(xe);
    }
  }
  return ORACLE_OK;
}

/* Exclusive prefix sum of floor(len_i / every); returns the total, or -1 on
 * a malformed cu_seqlens.  every == 0 means no checkpoints. */
int64_t kda_oracle_checkpoint_offsets(const int32_t* cu_seqlens, int N, int every,
                                      int32_t* offsets /* [N+1] or NULL */) {
  int64_t acc = 0;
  for (int i = 0; i < N; ++i) {
    const int64_t len = (int64_t)cu_seqlens[i + 1] - cu_seqlens[i];
    if (len < 0) return -1;
    if (offsets) offsets[i] = (int32_t)acc;
    if (every > 0) acc += len / every;
  }
  if (offsets) offsets[N] = (int32_t)acc;
  return acc;
}

/*
 * Prefill over N packed sequences.  Returns 0, or a negative code when an
 * argument is malformed (nothing is then written).  nthreads <= 0 uses the
 * OpenMP default; the parallel loop is over independent (sequence, head)
 * pairs and does not change any sum's order.
 */
int kda_oracle_prefill(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const int32_t* cu_seqlens, int N,
                       const int32_t* state_indices, const int32_t* has_initial_state,
                       double* pool, int64_t num_slots,
                       double* out, double* checkpoints, int checkpoint_every,
                       int64_t checkpoint_capacity, int32_t* ckpt_offsets,
                       const double* gate, const double* norm_w, double eps, int act, int H,
                       int dk, int dv, double scale, int nthreads) {
  if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || checkpoint_every < 0) return ORACLE_ERR_ARG;
  if (act < 0 || act > 1) return ORACLE_ERR_ARG;
  if (N == 0) return ORACLE_OK;
  if (!cu_seqlens || !state_indices || !pool || !out) return ORACLE_ERR_ARG;
  if (gate && !norm_w) return ORACLE_ERR_ARG;
  if (cu_seqlens[0] != 0) return ORACLE_ERR_ARG;
  int32_t* offs = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N + 1));
  if (!offs) return ORACLE_ERR_NOMEM;
  const int64_t n_ckpt = kda_oracle_checkpoint_offsets(cu_seqlens, N, checkpoint_every, offs);
  if (n_ckpt < 0) { free(offs); return ORACLE_ERR_ARG; }
  if (n_ckpt > 0 && (!checkpoints || n_ckpt > checkpoint_capacity)) {
    free(offs);
    return ORACLE_ERR_CAPACITY;
  }
  for (int i = 0; i < N; ++i) {
    const int32_t s = state_indices[i];
    if (s < -1 || (s >= 0 && s >= num_slots)) { free(offs); return ORACLE_ERR_INDEX; }
  }
  if (ckpt_offsets) memcpy(ckpt_offsets, offs, sizeof(int32_t) * (size_t)(N + 1));

  const size_t sd = (size_t)dk * dv;
  const int64_t pairs = (int64_t)N * H;
#ifdef _OPENMP
  /* a thread count for this call only (the process-wide default is untouched) */
  const int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
#endif
  int failed = 0;
#pragma omp parallel num_threads(nt)
  {
    double* S = (double*)malloc(sizeof(double) * sd);
    double* u = (double*)malloc(sizeof(double) * (size_t)dv);
    double* o = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!S || !u || !o) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t p = 0; p < pairs; ++p) {
      if (!S || !u || !o) continue;
      const int i = (int)(p / H), h = (int)(p % H);
      const int64_t t0 = cu_seqlens[i], t1 = cu_seqlens[i + 1];
      const int32_t slot = state_indices[i];
      if (slot < 0) {
        for (int64_t t = t0; t < t1; ++t) memset(out + ((size_t)t * H + h) * dv, 0, sizeof(double) * dv);
        continue;
      }
      if (t1 == t0) continue;
      double* slot_state = pool + ((size_t)slot * H + h) * sd;
      /* a sequence without initial state (a new prompt) starts from zero; its
       * final state is still written to the slot */
      if (has_initial_state && has_initial_state[i] == 0) memset(S, 0, sizeof(double) * sd);
      else memcpy(S, slot_state, sizeof(double) * sd);
      int64_t m = 0;
      for (int64_t t = t0; t < t1; ++t) {
        const size_t qk = ((size_t)t * H + h) * dk, vo = ((size_t)t * H + h) * dv;
        token_step(S, dk, dv, q + qk, k + qk, v + vo, g + qk, beta[(size_t)t * H + h], scale, u, o);
        if (gate) norm_gate_row(o, gate + vo, norm_w, eps, dv, act, out + vo);
        else memcpy(out + vo, o, sizeof(double) * dv);
        if (checkpoint_every > 0 && (t - t0 + 1) % checkpoint_every == 0) {
          memcpy(checkpoints + (((size_t)offs[i] + m) * H + h) * sd, S, sizeof(double) * sd);
          ++m;
        }
      }
      memcpy(slot_state, S, sizeof(double) * sd);
    }
    free(S); free(u); free(o);
  }
  free(offs);
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * One recurrent decode step ("[Feature][KDA] ...", section "KDA execution",
 * step 4): N sequences of one token each.  q,k,g [N,H,dk], v [N,H,dv],
 * beta [N,H], out [N,H,dv].  The pages' "normalize the recurrent gate"
 * pre-step is the caller's: g arrives in the same log-decay form as for
 * prefill.
 */
int kda_oracle_decode(const double* q, const double* k, const double* v, const double* g,
                      const double* beta, const int32_t* state_indices, int N, double* pool,
                      int64_t num_slots, double* out, const double* gate, const double* norm_w,
                      double eps, int act, int H, int dk, int dv, double scale, int nthreads) {
  if (N < 0) return ORACLE_ERR_ARG;
  if (N == 0) return ORACLE_OK;
  int32_t* cu = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N + 1));
  if (!cu) return ORACLE_ERR_NOMEM;
  for (int i = 0; i <= N; ++i) cu[i] = i;
  const int rc = kda_oracle_prefill(q, k, v, g, beta, cu, N, state_indices, NULL, pool, num_slots,
                                    out, NULL, 0, 0, NULL, gate, norm_w, eps, act, H, dk, dv, scale,
                                    nthreads);
  free(cu);
  return rc;
}

int kda_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
