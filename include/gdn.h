/*
 * gdn.h -- C ABI of libgdn: batched Gated-DeltaNet decode on one GB300 (sm_103a).
 *
 * What the library computes. For every request b of a decode batch and every
 * head h, the recurrent state S[dk][dv] (fp32, row-major, dv contiguous) of
 * the request's cache slot is advanced by one token:
 *
 *   q, k, v   <- width-4 causal conv1d + SiLU of the projected token (optional),
 *                then q, k L2-normalised per head, q multiplied by q_scale
 *   Sbar       = D(lambda) S_{t-1}                 forget; D(l) = diag(exp(l)) on key rows
 *   b          = beta (v - Sbar^T k)               delta-rule residual on the decayed state
 *   S_t        = Sbar + k b^T                       i.e. S_t = (I - beta k k^T) D(lambda) S_{t-1} + beta k v^T
 *   o          = S_t^T q                            post-update readout
 *
 * Sources, by page title and section:
 *   "深度解析线性注意力机制演进与 AI Infra 实现" (linear-attention evolution article):
 *     "去掉分母引入卷积" -- short conv + SiLU and the conv_state cache rows;
 *     "DeltaNet", "GDN：增加遗忘门", "KDA: By Channel的遗忘门", "KDA实现逻辑概述" --
 *     decay first, residual on the decayed state, outer-product write, readout;
 *     appendix "附2: 为什么要L2 Norm" -- L2 normalisation with an epsilon.
 *   "DeltaLog：延迟物化递归状态以加速线性注意力解码" (DeltaLog reading notes):
 *     Sec. 1.1 Eqs. (2)-(3) -- D(l) S + a b^T interface; Sec. 2.1 -- base + log
 *     layout; Sec. 2.2 Eq. (7) -- invariant; Sec. 2.3 Algorithm 1, Eq. (6) --
 *     append / merge; Sec. 2.4 -- readout from base + log, a_t = k_t,
 *     b_t = beta_t (v_t - vhat_t); Sec. 2.6 Fig. 5 -- one writer per state slice;
 *     Sec. 2.7 -- the three instantiations: GDN (per-head decay), KDA (per-key
 *     decay), both with K log bf16 and U log fp32; RWKV6 (per-key decay, raw
 *     value update, no correction, K and U logs bf16); decay metadata fp32.
 *   "线性注意力与混合架构的推理" (inference handbook): fp32 state, bf16 conv cache,
 *     slot-indexed state pools read by a batched kernel.
 *
 * Two execution modes.
 *   Dense    : gdn_decode_dense reads and rewrites the full state every token.
 *   DeltaLog : the state of a slot-head is held as a base Sbar plus a short log
 *              (K_log, U_log, Lambda_log, ell, L) such that
 *                S = D(ell) Sbar + sum_{i<L} D(ell - Lambda_log[i]) K_log[i] U_log[i]^T.
 *              gdn_decode_append adds one entry and never writes the base;
 *              gdn_decode_merge folds the log and the current token into the base.
 *              With merge interval M the log capacity is C = M - 1: steps with
 *              L < C on entry append, the step with L == C merges.
 *
 * Conventions shared by every entry point.
 *   - All data pointers are DEVICE pointers owned by the caller. The library
 *     allocates no memory, keeps no per-call state, and returns as soon as the
 *     work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - The synchronous return value reports argument errors (nothing is
 *     launched) and launch failures. Conditions found on the device (a slot
 *     index >= num_slots, a log length outside [0, C], an append on a full log)
 *     are never trapped: the affected (request, head) is skipped -- nothing of
 *     it is written -- and a GDN_STATUS_* bit is ORed into *status (a device
 *     int32 the caller zeroes and reads back; status may be NULL).
 *   - A negative slot index marks a padding request: it is skipped silently and
 *     its output row is left unchanged.
 *   - Slot indices of one call must be distinct (two requests on one slot race).
 *   - Supported head sizes. The decode steps (dense, append, merge, step), the log
 *     sizes and the slot reset: dk == dv in {16, 32, 64, 128}, dk = 128 with
 *     dv = 64, and dk = 64 with dv = 128 (GDN_SPLIT_DV: dk == dv in {64, 128}).
 *     The input stage, verify and prefill: dk == dv in {16, 32, 64, 128}. Other
 *     shapes return GDN_ERR_UNSUPPORTED. Pointers that the kernels read or write
 *     as 16-byte vectors (state/base, q, k, v, mixed_qkv, conv_w, o, k_log, u_log)
 *     must be 16-byte aligned.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_API_VERSION 2

/* Synchronous return codes. */
#define GDN_OK 0
#define GDN_ERR_INVALID_ARG 1 /* NULL where a pointer is required, negative sizes, bad flags */
#define GDN_ERR_UNSUPPORTED 2 /* head size, log capacity or flag combination not built; misaligned pointer */
#define GDN_ERR_CUDA 3        /* the kernel launch failed; gdn_last_error() has the CUDA message */

/* Device status bits, ORed into *status by the kernels. */
#define GDN_STATUS_BAD_SLOT 0x1u /* slot >= num_slots: the request was skipped */
#define GDN_STATUS_LOG_FULL 0x2u /* append entered with L == C: the slot-head was skipped */
#define GDN_STATUS_BAD_LEN 0x4u  /* log length outside [0, C]: the slot-head was skipped */
#define GDN_STATUS_TIMEOUT 0x8u  /* a bounded wait for an asynchronous copy gave up */

/* Flags (gdn_dims.flags). */
#define GDN_QKV_BF16 (1u << 0)     /* q/k/v (or mixed_qkv and the conv cache) are bf16; else fp32 */
#define GDN_FUSE_CONV (1u << 1)    /* inputs are mixed_qkv rows passed through the width-4 conv + SiLU */
#define GDN_NO_QK_L2NORM (1u << 2) /* skip the L2 normalisation of q and k (q_scale still applies) */
#define GDN_GATE_RAW (1u << 3)     /* log_decay holds a, beta holds b: lambda = logsigmoid(a), beta = sigmoid(b) */
#define GDN_PLAIN_UPDATE (1u << 4) /* additive update b = beta v (no delta correction); test mode */
#define GDN_KLOG_FP32 (1u << 5)    /* K_log entries are fp32 instead of bf16 */
#define GDN_KLOG_PRENORM (1u << 6) /* K_log keeps the key before L2 normalisation and U_log the
                                      value factor times the key's inverse norm (same product
                                      k b^T, no rounding of the normalised key); requires L2
                                      normalisation and no fused conv */
#define GDN_ULOG_BF16 (1u << 7)    /* U_log entries are bf16 instead of fp32 (the RWKV6 instantiation
                                      of the DeltaLog notes, Sec. 2.7: a raw-value update has no
                                      correction to protect, so both logs are bf16). Exact when
                                      b = v of bf16 inputs (GDN_PLAIN_UPDATE, beta == NULL) */
#define GDN_GATE_KDA (1u << 8)     /* the KDA gate parametrisation (evolution article, "KDA实现逻辑概述"):
                                      log_decay holds the forget pre-activation f, beta the write
                                      logit; lambda = gate_lower_bound * sigmoid(exp(a_log[h]) *
                                      (f + dt_bias[h])), beta = sigmoid(logit). Needs in->a_log and
                                      in->dt_bias; excludes GDN_GATE_RAW */
#define GDN_OUT_NORM_GATE (1u << 9) /* output epilogue of the same section: o <- RMSNorm(o) (.) w (.)
                                      sigmoid(g) per head over dv, RMSNorm(o) = o / sqrt(mean(o^2) +
                                      out_eps); g = in->out_gate, w = in->out_norm_w (NULL: 1) */
#define GDN_SPLIT_DV (1u << 10)    /* decode steps: each (request, head) is handled by two CTAs (one
                                      cluster), each the single writer of half the value columns of
                                      the state tile, of the output row and of the U log (DeltaLog
                                      notes, Sec. 2.6 / Fig. 5: the tile sliced along dv, B_V = dv/2);
                                      the first CTA also commits the head's shared metadata (K_log[L],
                                      Lambda_log[L], ell, L) and the q / k conv cache rows, after the
                                      cluster barrier has seen the second read them. Needs dk == dv in
                                      {64, 128}; excludes GDN_GATE_KDA and GDN_OUT_NORM_GATE. A bounded
                                      wait that runs out skips the slice that saw it: the other slice
                                      of the head may still commit. Same results as without the flag
                                      up to the order of the column sums */
#define GDN_TEST_STARVE_WAIT (1u << 31) /* test only: the decode kernels expect 16 bytes more than
                                           the first tile copy delivers, so that bounded wait runs
                                           out (about a second) and the call reports
                                           GDN_STATUS_TIMEOUT without writing anything; exercises
                                           the timeout path without any fault */

/* Problem description, passed by pointer to every call. */
typedef struct gdn_dims {
  int32_t batch;         /* B: requests in this decode batch (B == 0 is a no-op) */
  int32_t num_heads;     /* H */
  int32_t dk, dv;        /* key / value head size (shapes: see "Supported head sizes" above) */
  int32_t num_slots;     /* rows of the state, conv and log pools */
  int32_t decay_per_key; /* 0: per-head scalar log-decay (GDN); 1: per-key-channel (KDA) */
  int32_t log_capacity;  /* C = M - 1 log entries per slot-head, 0..63 (DeltaLog calls only);
                            larger values are rejected with GDN_ERR_UNSUPPORTED */
  uint32_t flags;        /* GDN_* flags above */
  float q_scale;         /* multiplies q after normalisation (1.0: o = S^T q exactly) */
  float l2_eps;          /* x / sqrt(sum x^2 + l2_eps) */
  float gate_lower_bound; /* GDN_GATE_KDA: lambda lies in (gate_lower_bound, 0) */
  float out_eps;          /* GDN_OUT_NORM_GATE: epsilon of the RMSNorm */
} gdn_dims;

/* Per-token inputs of one decode step. dlam = decay_per_key ? dk : 1. */
typedef struct gdn_inputs {
  const void *q;          /* [B][H][dk], bf16 or fp32 (GDN_QKV_BF16); unused with GDN_FUSE_CONV */
  const void *k;          /* [B][H][dk] */
  const void *v;          /* [B][H][dv] */
  const void *mixed_qkv;  /* GDN_FUSE_CONV: [B][2*H*dk + H*dv], channel order [q heads | k heads | v heads] */
  const float *conv_w;    /* GDN_FUSE_CONV: [channels][4]; column 3 multiplies the current token */
  const float *conv_b;    /* GDN_FUSE_CONV: [channels] or NULL */
  void *conv_pool;        /* GDN_FUSE_CONV: [num_slots][channels][3] pre-conv inputs, column 0 oldest;
                             same dtype as mixed_qkv; updated in place */
  const float *log_decay; /* lambda: [B][H][dlam] (<= 0), or raw gate logits with GDN_GATE_RAW */
  const float *beta;      /* [B][H] write strength in [0, 1], or raw logits with GDN_GATE_RAW;
                             NULL: beta = 1 for every head (the RWKV6 update k v^T with
                             GDN_PLAIN_UPDATE) */
  const int32_t *slot;    /* [B] pool row of each request; < 0 = padding */
  const float *a_log;     /* GDN_GATE_KDA: [H] */
  const float *dt_bias;   /* GDN_GATE_KDA: [H][dlam] */
  const float *out_gate;  /* GDN_OUT_NORM_GATE: [B][H][dv] output-gate logits ([B][T][H][dv] for verify) */
  const float *out_norm_w; /* GDN_OUT_NORM_GATE: [dv] RMSNorm weight shared by the heads, or NULL */
} gdn_inputs;

/* DeltaLog log pools (all [num_slots][H][...], updated in place). */
typedef struct gdn_log {
  void *k_log;      /* [num_slots][H][C][dk] bf16 (or fp32 with GDN_KLOG_FP32): key factors a_i */
  void *u_log;      /* [num_slots][H][C][dv] fp32 (or bf16 with GDN_ULOG_BF16): value factors b_i */
  float *lam_log;   /* [num_slots][H][C][dlam] cumulative log-decay at insertion, Lambda_i */
  float *ell;       /* [num_slots][H][dlam] cumulative log-decay since the last merge */
  int32_t *len;     /* [num_slots][H] log length L, 0 <= L <= C */
} gdn_log;

/* Byte sizes of the log pools for a gdn_dims (see gdn_log_bytes). */
typedef struct gdn_log_sizes {
  size_t k_log, u_log, lam_log, ell, len;
  size_t residency; /* k_log + u_log + lam_log + ell: (M-1) C_entry + C_decay of the DeltaLog notes */
  size_t total;     /* residency + len */
} gdn_log_sizes;

/* Library version (GDN_API_VERSION of the build). */
int gdn_version(void);

/* Human-readable name of a GDN_OK / GDN_ERR_* code. Never NULL. */
const char *gdn_strerror(int code);

/* Message of the most recent GDN_ERR_CUDA (or argument error) on the calling
 * thread; "" if none. Never NULL. */
const char *gdn_last_error(void);

/*
 * gdn_conv_l2norm -- the input stage on its own: width-4 causal conv + SiLU of
 * mixed_qkv (evolution article, "去掉分母引入卷积"), conv_pool row update, then
 * q, k L2-normalised (appendix 附2) and q multiplied by q_scale.
 * Requires GDN_FUSE_CONV in dims->flags (the fused decode calls run the same
 * stage inside their kernel).
 *   q_out, k_out [B][H][dk] fp32, v_out [B][H][dv] fp32 (16-byte aligned).
 * Rows of padding requests are left unchanged. Errors: as above.
 */
int gdn_conv_l2norm(const gdn_dims *dims, const gdn_inputs *in, float *q_out, float *k_out,
                    float *v_out, int32_t *status, void *stream);

/*
 * gdn_decode_dense -- one dense decode step (the recurrence at the top of this
 * file) on state_pool [num_slots][H][dk][dv] fp32, updated in place.
 *   o [B][H][dv] fp32: post-update readout.
 * Each (request, head) is handled by one CTA that is the only writer of its
 * state slice and output row.
 */
int gdn_decode_dense(const gdn_dims *dims, const gdn_inputs *in, float *state_pool, float *o,
                     int32_t *status, void *stream);

/*
 * gdn_decode_append -- one DeltaLog append step (Algorithm 1 with L < C on
 * entry): ell' = ell + lambda; vhat and o are read from base + log (Sec. 2.4);
 * entry L becomes (k, b, ell'), ell = ell', L = L + 1. base_pool is only read.
 * Requires log_capacity >= 1. A slot-head entering with L == C is skipped
 * (GDN_STATUS_LOG_FULL): call gdn_decode_merge or gdn_decode_step for it.
 */
int gdn_decode_append(const gdn_dims *dims, const gdn_inputs *in, const float *base_pool,
                      const gdn_log *log, float *o, int32_t *status, void *stream);

/*
 * gdn_decode_merge -- one DeltaLog merge step (Eq. (6)): same reads and output
 * as append, then base = D(ell') base + sum_{i<L} D(ell' - Lambda_i) K_i U_i^T + k b^T,
 * ell = 0, L = 0. Valid for any 0 <= L <= C (a forced flush before the log is
 * full checkpoints the slot: afterwards the base is the logical state).
 * With log_capacity == 0 (M = 1) the log pointers may be NULL except len and
 * ell, and every step is a merge, identical in arithmetic to a dense step.
 */
int gdn_decode_merge(const gdn_dims *dims, const gdn_inputs *in, float *base_pool,
                     const gdn_log *log, float *o, int32_t *status, void *stream);

/*
 * gdn_decode_step -- one DeltaLog step where every slot-head picks its own
 * phase from its log length: append if L < C on entry, merge otherwise
 * (Algorithm 1). Lets requests at different points of their cycle share one
 * launch (and one captured graph).
 */
int gdn_decode_step(const gdn_dims *dims, const gdn_inputs *in, float *base_pool,
                    const gdn_log *log, float *o, int32_t *status, void *stream);

/*
 * gdn_decode_verify -- speculative-decoding verification on the dense state
 * (inference handbook, "推测解码：验证后如何恢复状态"). T = num_tokens input
 * positions per request ([x0, d1, ..., d_{T-1}]: the last sampled token and the
 * drafts) run through the dense step one after another. The state after every
 * position is kept in its own pool row, so a rejected draft is rolled back by
 * choosing a row, not by copying a state:
 *   state_indices [B][T] int32: pool rows of request b; the state after position
 *       t is written to row state_indices[b][t]. The rows of one request must be
 *       distinct, and no two requests may share a row.
 *   num_accepted [B] int32 in [1, T]: the initial state is read from row
 *       state_indices[b][num_accepted[b] - 1], the column the previous round's
 *       acceptance selects (1 for a request whose state sits in column 0). It is
 *       read in full before any row is written, so it may be one of the rows this
 *       call overwrites.
 *   in->q, in->k, in->v [B][T][H][d] (bf16 or fp32), in->log_decay [B][T][H][dlam],
 *   in->beta [B][T][H] (or NULL: beta = 1); in->slot is not used.
 *   o [B][T][H][dv] fp32: the readout of every position.
 * With GDN_FUSE_CONV, q, k and v come from the width-4 conv + SiLU of
 * in->mixed_qkv [B][T][channels] (channel order and conv_w / conv_b as for the decode
 * calls) through the widened conv window of the same passage:
 *   in->conv_pool [num_slots][channels][T + 2] (bf16 with GDN_QKV_BF16, else fp32):
 *       per channel the last T + 2 pre-conv inputs, column 0 oldest; the request's
 *       window is row state_indices[b][0]. The three inputs before position 0 are read
 *       from columns num_accepted[b] - 1 .. num_accepted[b] + 1, and the row is rewritten
 *       with columns num_accepted[b] and num_accepted[b] + 1 followed by the T inputs of
 *       this call (bit-exact copies). A plain three-column conv state enters as columns
 *       0..2 with num_accepted = 1. Consecutive verify calls on one window pool use the
 *       same num_tokens.
 * A request with state_indices[b][0] < 0 is padding and is skipped. A row outside
 * [0, num_slots) skips the request with GDN_STATUS_BAD_SLOT; num_accepted outside
 * [1, T] skips it with GDN_STATUS_BAD_LEN; a skipped request's rows, window and
 * outputs are untouched. Requires 1 <= num_tokens <= 16; the verify path is the
 * dense recurrence, so the DeltaLog flags are rejected with GDN_ERR_UNSUPPORTED.
 */
int gdn_decode_verify(const gdn_dims *dims, int32_t num_tokens, const gdn_inputs *in,
                      const int32_t *state_indices, const int32_t *num_accepted,
                      float *state_pool, float *o, int32_t *status, void *stream);

/*
 * gdn_prefill -- the prompt of every request through the recurrence, evaluated chunk by
 * chunk with the WY/UT algebra (evolution article, "Prefill中的Chunk微观并行"; same
 * arithmetic per token as gdn_decode_dense). The initial state is the request's pool row
 * (zero it with gdn_slot_reset for a new request); the final state is written back there:
 * the base a DeltaLog decode continues from (DeltaLog notes Sec. 2.8 -- reset the log of
 * the slot as well).
 *   num_tokens T: positions per request in the input arrays.
 *   in->q, in->k, in->v [B][T][H][d] (bf16 or fp32), in->log_decay [B][T][H][dlam],
 *   in->beta [B][T][H] (or NULL: beta = 1), in->slot [B] (< 0: padding).
 *   seq_lens [B] int32 in [0, T]: the prompt length of each request, or NULL (all T).
 *       Positions past it are not read and their o rows are left unchanged; a length
 *       outside [0, T] skips the request with GDN_STATUS_BAD_LEN.
 *   state_pool [num_slots][H][dk][dv] fp32, read and overwritten.
 *   o [B][T][H][dv] fp32: the readout of every position.
 * Flags: GDN_QKV_BF16, GDN_NO_QK_L2NORM, GDN_GATE_RAW, GDN_PLAIN_UPDATE, decay_per_key,
 * and as for the decode calls:
 *   GDN_FUSE_CONV: q, k, v are the width-4 conv + SiLU of in->mixed_qkv [B][T][channels]
 *       (conv_w, conv_b as for decode); the inputs before position 0 come from the slot's
 *       conv state in->conv_pool [num_slots][channels][3], which afterwards holds the last
 *       three inputs of (old state, prompt) -- the state a fused-conv decode continues
 *       from (unchanged for an empty prompt);
 *   GDN_GATE_KDA and GDN_OUT_NORM_GATE (in->out_gate [B][T][H][dv]).
 * The DeltaLog flags are rejected with GDN_ERR_UNSUPPORTED. Requires num_tokens >= 0.
 * Precision and path: the state and every product stay at fp32 accuracy. Head size 128
 * (and B * T below 2^31) runs its matrix products on the tensor cores as three TF32
 * products per fp32 product (hi*hi + lo*hi + hi*lo, relative error about 2^-20 per term):
 * with a per-head decay (bf16 or fp32 q/k/v, or bf16 mixed_qkv through GDN_FUSE_CONV; no
 * KDA flags), or with a per-key decay (bf16 q/k/v without GDN_FUSE_CONV, a 16-byte aligned
 * log_decay, the KDA gate and epilogue included); a chunk whose per-key decay falls below
 * e^-80 forms its pair sums term by term on the CUDA cores. Every other case runs on the
 * FP32 CUDA cores. All agree with token-by-token decode to 1e-4.
 */
int gdn_prefill(const gdn_dims *dims, int32_t num_tokens, const gdn_inputs *in,
                const int32_t *seq_lens, float *state_pool, float *o, int32_t *status, void *stream);

/*
 * gdn_log_bytes -- byte sizes of the log pools for dims (num_slots, num_heads,
 * dk, dv, decay_per_key, log_capacity, GDN_KLOG_FP32, GDN_ULOG_BF16). Host only;
 * no GPU needed. residency equals (M-1) C_entry + C_decay of the DeltaLog notes'
 * capacity table (Sec. 2.5): 21.125 MiB for GDN at M = 8, 17 MiB for KDA at M = 4
 * and 14 MiB for RWKV6 (bf16 U log) at M = 4, with 128 slots, 32 heads and
 * dk = dv = 128.
 */
int gdn_log_bytes(const gdn_dims *dims, gdn_log_sizes *out);

/*
 * gdn_slot_reset -- prepare n cache slots for new requests (DeltaLog notes
 * Sec. 2.8: a reused slot starts with an empty log): L = 0 and ell = 0 for
 * every head; the conv_pool rows are zeroed when conv_pool is not NULL; the
 * state_pool rows are zeroed when state_pool is not NULL (a request that
 * starts from zero state; a prefill would write them instead).
 *   slots [n] device int32; entries < 0 are ignored, entries >= num_slots set
 *   GDN_STATUS_BAD_SLOT. log may be NULL (dense-only callers).
 */
int gdn_slot_reset(const gdn_dims *dims, const gdn_log *log, void *conv_pool, float *state_pool,
                   const int32_t *slots, int32_t n, int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
