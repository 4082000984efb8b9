/*
 * kda.h -- C ABI of libkda: Kimi Delta Attention (KDA) prefill, decode and
 * output norm-gate on one NVIDIA GB300 (sm_103a).
 *
 * The method.  KDA is the gated delta rule with a per-channel decay.  For a
 * head with key dimension dk and value dimension dv, token t updates the
 * recurrent state S (dk x dv) and reads it out:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * Sources: "[Feature][KDA] Add Kimi K3 KDA execution" (vllm-ascend PR 14598),
 * section "KDA execution", steps 3 (chunk prefill over a cumulative gate) and
 * 4 (recurrent decode); "[KK] Prepare B12X Kimi KDA prefill ..." (vLLM PR
 * 937), section "Behavior" (state-pool indices consumed in place, reusable
 * caller-owned scratch); the FlashKDA bf16-checkpoint summary (vLLM PR
 * 56485), motivation and implementation sections (intermediate checkpoint
 * states whose dtype follows the state dtype; tolerances 0.03 bf16 / 0.01
 * fp32).
 *
 * Conventions shared by every call.
 *  - All tensors are dense, row-major, last dimension contiguous, and live in
 *    device memory unless stated otherwise.  The caller owns every buffer;
 *    the library allocates nothing and never synchronises.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls are asynchronous on that stream and make no host read of
 *    device data, so they can be captured in a CUDA graph.
 *  - Argument errors are detected on the host and returned; nothing is
 *    launched then.  Errors that need device values (a bad state index, a bad
 *    cu_seqlens entry) are latched into `*dev_status` (an int32 in device
 *    memory, zeroed by the caller; may be NULL), and the affected sequence is
 *    skipped with its output rows zeroed.  Kernels never trap.
 *  - Token-major layouts: q, k, g are [T, H, dk]; v, out, gate are
 *    [T, H, dv]; beta is [T, H].  The state pool is [num_slots, H, dk, dv].
 *  - Supported: dk == dv in {16, 64, 128}; chunk in {16, 64} (prefill);
 *    inputs fp32 or bf16; state fp32 or bf16.  Others -> KDA_ERR_UNSUPPORTED.
 *  - Pointer alignment: 16 bytes for every tensor argument.
 */
#ifndef LIBKDA_KDA_H_
#define LIBKDA_KDA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = -1, /* null/misaligned pointer, negative size, bad combination */
  KDA_ERR_UNSUPPORTED = -2, /* a shape or dtype outside the supported set */
  KDA_ERR_WORKSPACE = -3,   /* workspace smaller than *_workspace_bytes() asks */
  KDA_ERR_CUDA = -4         /* a CUDA launch or attribute call failed */
} kda_status;

/* Element types.  KDA_F16 is accepted by kda_norm_gate_ex only (the pages'
 * norm-gate coverage names fp16 and bf16); the recurrence entry points take
 * KDA_F32 and KDA_BF16. */
typedef enum { KDA_F32 = 0, KDA_BF16 = 1, KDA_F16 = 2 } kda_dtype;

/* Activation of the output gate in the RMSNorm-gate: sigmoid(x) or SiLU,
 * x * sigmoid(x) (the two activations the pages' norm-gate coverage names). */
typedef enum { KDA_GATE_SIGMOID = 0, KDA_GATE_SILU = 1 } kda_gate_act;

/* Codes latched into *dev_status by the kernels (first error wins). */
#define KDA_DEV_OK 0
#define KDA_DEV_BAD_INDEX 1       /* state_indices[i] outside [-1, num_slots) */
#define KDA_DEV_BAD_SEQLENS 2     /* cu_seqlens not non-decreasing within [0, T] */
#define KDA_DEV_TIMEOUT 3         /* a bounded on-chip wait gave up */
#define KDA_DEV_CKPT_OVERFLOW 4   /* checkpoints would exceed checkpoint_capacity */
#define KDA_DEV_DUP_INDEX 5       /* one state slot named by two sequences of a call */

/*
 * Bytes of caller-owned scratch that always suffice for kda_prefill_chunked
 * with these sizes (the pages' "reusable caller-owned scratch"), whatever the
 * dtypes and the gate option.  A call may need less (or none); it returns
 * KDA_ERR_WORKSPACE when what it needs is not provided.  The same workspace
 * can be reused by consecutive calls on one stream.
 */
KDA_API size_t kda_prefill_workspace_bytes(int N, int64_t T, int H, int dk, int dv, int chunk);

/*
 * Chunked varlen prefill over an indexed state pool ("[Feature][KDA] ...",
 * "KDA execution" step 3; "[KK] Prepare B12X ...", "Behavior").
 *
 *  q, k, g      [T, H, dk]  in_dtype.  g is the per-channel log-decay
 *               (alpha = exp(g)); the in-chunk cumulative sum is done here.
 *  v            [T, H, dv]  in_dtype.
 *  beta         [T, H]      in_dtype.
 *  cu_seqlens   int32 [N+1], device.  Sequence i is tokens
 *               [cu_seqlens[i], cu_seqlens[i+1]); cu_seqlens[0] == 0 and
 *               cu_seqlens[N] == T.  Chunks restart at every sequence start;
 *               the last chunk of a sequence may be partial.  A zero-length
 *               sequence is a no-op (its slot is not rewritten).  The entries
 *               must be non-decreasing: a negative length latches
 *               KDA_DEV_BAD_SEQLENS; ranges that overlap an earlier sequence
 *               give undefined values for the sequences involved (every
 *               access still stays inside the buffers).
 *  state_indices int32 [N], device.  Sequence i starts from
 *               state_pool[state_indices[i]] and its final state is written
 *               back to that slot in place.  -1 marks a padding sequence: its
 *               output rows are zeroed and the pool is untouched.  Indices
 *               must be distinct within a call: a repeated index latches
 *               KDA_DEV_DUP_INDEX, and the results of the sequences that
 *               share the slot are undefined.
 *  has_initial_state int32 [N], device, or NULL (every sequence has state).
 *               0 marks a sequence without initial state -- a new prompt
 *               ("[Feature][KDA] ...", section "Metadata construction": a
 *               one-token prompt without state is still prefill): it starts
 *               from S = 0 whatever its slot holds, and its final state is
 *               written to the slot as usual.
 *  state_pool   [num_slots, H, dk, dv] state_dtype, read and written.
 *  out          [T, H, dv] in_dtype.  o_t, or the norm-gated y_t when gate
 *               is non-NULL.
 *  checkpoints  [checkpoint_capacity, H, dk, dv] state_dtype, or NULL when
 *               checkpoint_every == 0.  After every checkpoint_every tokens of
 *               a sequence (counted from the start of this call's segment) the
 *               state is appended; sequence i owns entries
 *               [ckpt_offsets[i], ckpt_offsets[i+1]).  checkpoint_every must be
 *               0 or a multiple of chunk, and checkpoint_capacity must be at
 *               least T / checkpoint_every.
 *  ckpt_offsets int32 [N+1], device, written (may be NULL): the exclusive
 *               prefix sum of floor(len_i / checkpoint_every).
 *  gate, norm_w gate [T, H, dv] in_dtype and norm_w [dv] in_dtype, or both
 *               NULL.  When given, out = o / sqrt(mean(o^2) + eps) * norm_w *
 *               act(gate) per (token, head) row, act chosen by gate_act.
 *  scale        read-out scale; <= 0 selects 1/sqrt(dk).
 *  workspace    caller scratch of at least kda_prefill_workspace_bytes().
 *  dev_status   see the conventions above (may be NULL).
 *
 * State is carried in fp32 inside a call and rounded (to nearest even) to
 * state_dtype only when stored: at checkpoints and at the final write-back.
 *
 * Numerics.  The tensor-core path (bf16 inputs, dk = dv in {64, 128}, chunk
 * 64; kda_prefill_path says which path a shape takes) forms the in-chunk
 * products A_kk, A_qk from split bf16 operands (fp32
 * accuracy) and the state-coupled products from fp16 operands, all with fp32
 * accumulation.  That relies on the method's regime: q and k rows of unit L2
 * norm and beta in [0, 1], where I - beta k k^T is a contraction and the
 * state and the intermediate rows stay O(1).  A chunk whose decay spread
 * exceeds e^60 in some channel is computed by an exact element-wise path.
 */
KDA_API kda_status kda_prefill_chunked(const void* q, const void* k, const void* v, const void* g,
                               const void* beta, kda_dtype in_dtype, const int32_t* cu_seqlens,
                               int N, int64_t T, const int32_t* state_indices,
                               const int32_t* has_initial_state, void* state_pool,
                               int64_t num_slots, kda_dtype state_dtype, void* out,
                               void* checkpoints, int32_t checkpoint_every,
                               int64_t checkpoint_capacity, int32_t* ckpt_offsets,
                               const void* gate, const void* norm_w, float eps,
                               kda_gate_act gate_act, int H, int dk, int dv, int chunk,
                               float scale, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream);

/*
 * One recurrent decode step for N sequences of one token each ("[Feature][KDA]
 * ...", "KDA execution" step 4).  q, k, g [N, H, dk]; v, out, gate [N, H, dv];
 * beta [N, H]; state_indices int32 [N] (device; -1 = padding row, zeroed).
 * g is in the same log-decay form as for prefill (the pages' "normalize the
 * recurrent gate" step is the caller's).  The state is updated in place and
 * rounded to state_dtype at the store.  gate/norm_w as for prefill.
 */
KDA_API kda_status kda_decode_step(const void* q, const void* k, const void* v, const void* g,
                           const void* beta, kda_dtype in_dtype, const int32_t* state_indices,
                           int N, void* state_pool, int64_t num_slots, kda_dtype state_dtype,
                           void* out, const void* gate, const void* norm_w, float eps,
                           kda_gate_act gate_act, int H, int dk, int dv, float scale,
                           int32_t* dev_status, void* stream);

/*
 * K recurrent decode steps per sequence, for verifying K speculative tokens
 * ("[Feature][KDA] Add Kimi K3 KDA execution", section "Metadata
 * construction": speculative decode is its own batch kind; the FlashKDA page,
 * risk section: state recovery inside speculative decoding).  Sequence i runs
 * tokens t = 0..K-1 through the decode step of kda_decode_step, starting from
 * state_pool[state_indices[i]], and the state after token t is stored to
 * token_states[i, t] so that the state after any accepted prefix can be
 * committed afterwards (kda_commit_accepted).
 *  q, k, g      [N, K, H, dk] in_dtype (token t of sequence i at row i*K + t).
 *  v, out, gate [N, K, H, dv]; beta [N, K, H].
 *  state_indices int32 [N] (device); -1 = padding (its K output rows are zeroed,
 *               its token_states left untouched); out of range -> KDA_DEV_BAD_INDEX.
 *  token_states [N, K, H, dk, dv] state_dtype (device, 16-byte aligned), or
 *               NULL to keep no per-token states.
 *  write_back   nonzero: the state after token K-1 is also written to the slot
 *               (every token accepted); zero: the pool is only read.
 * Other arguments as for kda_decode_step.  The state is carried in fp32 across
 * the K tokens and rounded to state_dtype only at the stores.
 */
KDA_API kda_status kda_decode_multi(const void* q, const void* k, const void* v, const void* g,
                            const void* beta, kda_dtype in_dtype, const int32_t* state_indices,
                            int N, int K, void* state_pool, int64_t num_slots,
                            kda_dtype state_dtype, void* out, void* token_states, int write_back,
                            const void* gate, const void* norm_w, float eps,
                            kda_gate_act gate_act, int H, int dk, int dv, float scale,
                            int32_t* dev_status, void* stream);

/*
 * Commit the verified prefix of a kda_decode_multi call: for each sequence i
 * with a_i = num_accepted[i] >= 1, state_pool[state_indices[i]] =
 * token_states[i, a_i - 1]; a_i == 0 or a padding index (-1) leaves the slot
 * unchanged.  num_accepted int32 [N] (device); a_i outside [0, K] or an index
 * out of range latches KDA_DEV_BAD_INDEX and skips the sequence.  token_states
 * as written by kda_decode_multi with the same N, K, H, dk, dv, state_dtype.
 */
KDA_API kda_status kda_commit_accepted(const void* token_states, const int32_t* num_accepted,
                               const int32_t* state_indices, int N, int K, void* state_pool,
                               int64_t num_slots, kda_dtype state_dtype, int H, int dk, int dv,
                               int32_t* dev_status, void* stream);

/*
 * Standalone output RMSNorm-gate ("[Feature][KDA] ...", first section:
 * FusedRMSNormGated output normalisation and gating):
 *     y = o / sqrt(mean_dv(o^2) + eps) * w * act(gate),  act = sigmoid or SiLU
 * o, gate, y are [rows, H, dv] in `dtype`; w is [dv] in `dtype`.  y may alias o
 * (in place); otherwise o is preserved.
 */
KDA_API kda_status kda_norm_gate(const void* o, const void* gate, const void* w, float eps,
                         kda_gate_act gate_act, void* y, int64_t rows, int H, int dv,
                         kda_dtype dtype, void* stream);

/*
 * Norm-gate variants, the coverage list of "[Feature][KDA] ..." (testing
 * section: fp16/bf16, sigmoid/SiLU, packed gate strides, affine and
 * residual/prenorm paths).  Per token row t and head h, over the dv values:
 *     x = o + residual                                  (residual may be NULL)
 *     residual_out = x                                  (the prenorm output; may be NULL)
 *     y = (x / sqrt(mean(x^2) + eps) * w + b) * act(gate)
 * w and b are [dv] (NULL: w = 1, b = 0).  o, residual, residual_out and y are
 * [rows, H, dv]; the gate of (t, h) is the dv values at
 * gate + t * gate_row_stride + h * dv (gate_row_stride in elements, a
 * multiple of 4 and >= H * dv; 0 means H * dv), so a gate that is a slice of
 * a packed projection output can be used without a copy.  Every tensor is in
 * `dtype` (f32, bf16 or f16); x is formed and normalised in fp32 and rounded
 * to dtype at the stores.  y may alias o or residual, residual_out may alias
 * o or residual; y and residual_out must differ.  Inputs not aliased by an
 * output are preserved.
 */
KDA_API kda_status kda_norm_gate_ex(const void* o, const void* residual, void* residual_out,
                            const void* gate, int64_t gate_row_stride, const void* w,
                            const void* b, float eps, kda_gate_act gate_act, void* y, int64_t rows,
                            int H, int dv, kda_dtype dtype, void* stream);

/*
 * Short causal convolution with a per-sequence cache, run on the projections
 * ahead of the recurrence ("[Feature][KDA] Add Kimi K3 KDA execution", section
 * "KDA execution", step 2: run the causal convolution and update its cache).
 * Depthwise over `channels` (a multiple of 8) with width W in {2, 3, 4}:
 *     y[t, c] = act(bias[c] + sum_{i<W} weight[c, i] * xe[t - (W-1) + i, c])
 * where xe is the sequence extended on the left by the W-1 inputs held in its
 * cache slot, oldest first (zeros when has_initial_state[i] == 0).  The slot
 * then holds the sequence's last W-1 extended inputs.  act: identity or SiLU.
 *  x, y         [T, channels] dtype (f32 or bf16); y must not overlap x.
 *  weight       [channels, W] dtype;  bias [channels] dtype or NULL.
 *  cu_seqlens, state_indices, has_initial_state: as for kda_prefill_chunked
 *               (index -1: padding, zero outputs, cache untouched; an empty
 *               sequence leaves its cache alone).
 *  conv_state_pool [num_slots, W-1, channels] dtype, updated in place.
 * Values are formed in fp32 and rounded to dtype when stored.
 * Host-side errors: KDA_ERR_UNSUPPORTED for a width outside {2, 3, 4},
 * channels not a multiple of 8 or a dtype other than f32/bf16;
 * KDA_ERR_INVALID_ARG for a NULL or misaligned pointer, negative sizes,
 * an unknown act, or T/64 + N > 65535 (the prefill's 64-token tile slots;
 * the decode's limit is N <= 65535).  Device-side (dev_status): a bad index
 * or bad cu_seqlens as for kda_prefill_chunked.
 */
typedef enum { KDA_CONV_IDENTITY = 0, KDA_CONV_SILU = 1 } kda_conv_act;
KDA_API kda_status kda_causal_conv1d_prefill(const void* x, const void* weight, const void* bias,
                                     kda_dtype dtype, const int32_t* cu_seqlens, int N, int64_t T,
                                     int channels, int width, const int32_t* state_indices,
                                     const int32_t* has_initial_state, void* conv_state_pool,
                                     int64_t num_slots, kda_conv_act act, void* y,
                                     int32_t* dev_status, void* stream);

/*
 * One token per sequence through the same convolution: x, y [N, channels];
 * the cache of state_indices[i] supplies the W-1 earlier inputs and is
 * shifted by one (x appended).  Other arguments as for the prefill.
 */
KDA_API kda_status kda_causal_conv1d_decode(const void* x, const void* weight, const void* bias,
                                    kda_dtype dtype, int N, int channels, int width,
                                    const int32_t* state_indices, void* conv_state_pool,
                                    int64_t num_slots, kda_conv_act act, void* y,
                                    int32_t* dev_status, void* stream);

/*
 * The short convolution, the L2 normalisation of q and k and the chunked
 * prefill in one pass ("[Feature][KDA] Add Kimi K3 KDA execution", section
 * "KDA execution", steps 2-3: the causal convolution with its cache update,
 * then the chunk prefill on its output).  Per token and head, with the
 * convolution and cache of kda_causal_conv1d_prefill over the packed channels
 * [q | k | v] (channels = 3 H d, head by head within each block):
 *     y        = act(conv(x)) rounded to bf16
 *     q, k     = y_q / sqrt(|y_q|^2 + KDA_CONV_L2_EPS), y_k / ..., rounded to bf16
 *     v        = y_v
 * then everything kda_prefill_chunked does with those q, k, v and the given
 * g, beta (state pool, checkpoints, fused norm-gate).  The results equal
 * kda_causal_conv1d_prefill, a per-(token, head) L2 normalisation stored in
 * bf16, and kda_prefill_chunked, run in sequence -- without the intermediate
 * tensors (q, k, v are never written to memory).
 *  x_q, x_k, x_v  [T, H, d] bf16 rows of x_row_stride elements (a multiple of
 *                 8, at least H d): for a packed projection output [T, 3 H d]
 *                 pass its base, base + H d, base + 2 H d and 3 H d.
 *  conv_w         [3 H d, W] bf16; conv_b [3 H d] bf16 or NULL; W in {2, 3, 4}.
 *  conv_state_pool [conv_num_slots, W-1, 3 H d] bf16, indexed by the same
 *                 state_indices as the state pool and read as initial context
 *                 under the same has_initial_state flag; rewritten with each
 *                 sequence's last W-1 extended inputs (an empty sequence or a
 *                 padding index leaves its slot alone, and so does a sequence
 *                 whose chain latched an error: its state slot and its cache
 *                 slot are both left as they were).
 * Other arguments as for kda_prefill_chunked (same workspace size).  Supported
 * only where kda_prefill_path reports KDA_PATH_TENSOR_CORES (bf16 inputs,
 * dk = dv in {64, 128}, chunk 64); otherwise KDA_ERR_UNSUPPORTED, as for W
 * outside {2, 3, 4}.  KDA_ERR_INVALID_ARG for an unknown act, a bad row
 * stride, conv_num_slots <= 0 or a NULL/misaligned convolution pointer.  An
 * index at or above conv_num_slots latches KDA_DEV_BAD_INDEX like one at or
 * above num_slots.
 */
#define KDA_CONV_L2_EPS 1e-6f
KDA_API kda_status kda_prefill_chunked_conv(
    const void* x_q, const void* x_k, const void* x_v, int64_t x_row_stride, const void* conv_w,
    const void* conv_b, int conv_width, kda_conv_act conv_act, void* conv_state_pool, int64_t conv_num_slots,
    const void* g, const void* beta, kda_dtype in_dtype, const int32_t* cu_seqlens, int N, int64_t T,
    const int32_t* state_indices, const int32_t* has_initial_state, void* state_pool, int64_t num_slots,
    kda_dtype state_dtype, void* out, void* checkpoints, int32_t checkpoint_every, int64_t checkpoint_capacity,
    int32_t* ckpt_offsets, const void* gate, const void* norm_w, float eps, kda_gate_act gate_act, int H, int dk,
    int dv, int chunk, float scale, void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * Chunked prefill without caller scratch.  The pages have no counterpart of
 * this entry point; it serves callers that cannot allocate device memory where
 * they run the prefill (for example code running under strict-mode stream
 * capture, where cudaMalloc is an error, or runtimes confined to a fixed
 * memory arena).  Arguments and results are those of kda_prefill_chunked,
 * minus the workspace: the library uses its own device array of
 * KDA_STATIC_SCRATCH_BYTES bytes instead, which every GPU that loads the
 * library holds until the process exits.  A call whose scratch need
 * (kda_prefill_workspace_bytes bounds it) exceeds that size returns
 * KDA_ERR_WORKSPACE without launching.  The first call on each device looks up
 * the array's device address and caches it for the device's current context,
 * so make that first call before any stream capture starts; after
 * cudaDeviceReset (or from another context) the next call looks it up again,
 * and that call, too, belongs before any capture.  Every call shares the array: calls whose kernels
 * overlap on the GPU (different streams, or different host threads) race on it
 * and must be serialised by the caller.  No allocation happens in this call.
 */
#define KDA_STATIC_SCRATCH_BYTES ((size_t)128 << 20)
KDA_API kda_status kda_prefill_chunked_static_scratch(
    const void* q, const void* k, const void* v, const void* g, const void* beta, kda_dtype in_dtype,
    const int32_t* cu_seqlens, int N, int64_t T, const int32_t* state_indices,
    const int32_t* has_initial_state, void* state_pool, int64_t num_slots, kda_dtype state_dtype,
    void* out, void* checkpoints, int32_t checkpoint_every, int64_t checkpoint_capacity,
    int32_t* ckpt_offsets, const void* gate, const void* norm_w, float eps, kda_gate_act gate_act,
    int H, int dk, int dv, int chunk, float scale, int32_t* dev_status, void* stream);

/*
 * Testing only: the number of polls the first bounded on-chip wait of a
 * tensor-core prefill kernel makes before it gives up (the other waits keep
 * their limit, so the clean-up after a timed-out wait still lets every copy
 * and product in flight finish).  `kernels` selects the kernels the setting
 * applies to: bit 0 the intra-chunk kernel (each CTA's first wait), bit 1 the
 * state kernel (each chain's first wait); tries < 0 restores the default for
 * both.  The setting is process wide and applies to kda_prefill_chunked and
 * kda_prefill_chunked_static_scratch launches made after the call; it exists
 * so that a test can make a wait run out (KDA_DEV_TIMEOUT) without touching
 * any other part of the GPU.  Not for production use.
 */
KDA_API void kda_testing_set_first_wait_tries(int32_t tries, int32_t kernels);

/*
 * Which kernels kda_prefill_chunked runs for this shape: KDA_PATH_TENSOR_CORES
 * (an intra-chunk and a state kernel on tcgen05/TMEM; bf16 inputs, dk = dv in
 * {64, 128}, chunk 64), KDA_PATH_CUDA_CORES (one CUDA-core kernel per
 * (sequence, head, 64-column slab), with the norm-gate fused when dv <= 64
 * and as a second pass when gated with dv = 128), or
 * KDA_PATH_UNSUPPORTED.  A host-side query; no device work.
 */
#define KDA_PATH_UNSUPPORTED 0
#define KDA_PATH_CUDA_CORES 1
#define KDA_PATH_TENSOR_CORES 2
KDA_API int kda_prefill_path(int dk, int dv, int chunk, kda_dtype in_dtype);

/* A static, human-readable name for a kda_status value. */
KDA_API const char* kda_status_string(kda_status status);

/* Library ABI version (major * 100 + minor). */
KDA_API int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBKDA_KDA_H_ */
