/*
 * mtp_rs.h -- C ABI of the GB300 (sm_103a) library for multi-token-prediction
 * rejection-sampling verification, per-position row statistics and the fused
 * forward+backward of the end-to-end TV loss.
 *
 * Method references (page title, section):
 *   [BB] "Breaking Entropy Bounds: Accelerating RL Training via MTP with
 *        Rejection Sampling" -- §2 "Acceptance methods" (accept with
 *        probability min(1, p(y)/q(y)); RS preserves p), §3 and §8 (acceptance
 *        equals the overlap sum_v min(p_v, q_v) = 1 - TV), §4 "End-to-end TV
 *        loss", App. A (TV gradient with S = sum_v 1[q_v <= p_v] q_v),
 *        App. F (fused TV loss kernel), App. G.1 (stop at the first rejection;
 *        residual or bonus token by two-pass CDF inversion).
 *   [EM] "EntMTP: Accelerating LLM Inference with Entropy Guided Multi Token
 *        Prediction", Related Work, "Speculative Decoding" (left-to-right
 *        acceptance; replacement from norm(max(0, p - q)); suffix discarded).
 *
 * Conventions shared by every entry point
 *   - Logits are row-major with the vocabulary contiguous: target
 *     [B, gamma+1, V] (verify, stats) or [N, gamma, V] (TV loss), draft
 *     [B, gamma, V] or [N, gamma, V].  Storage is float32 or bfloat16; all
 *     arithmetic is float32.
 *   - Every pointer is caller-owned DEVICE memory on the current device.  The
 *     library allocates nothing, keeps no per-call state and never modifies
 *     its inputs.  Optional outputs may be NULL.
 *   - Logit base pointers must be 16-byte aligned (MTP_ERR_MISALIGNED
 *     otherwise); any V >= 1 is accepted, and rows that are not 16-byte
 *     aligned (V * element size not a multiple of 16) are handled in-kernel.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream).  The
 *     return value covers argument validation and the launch; an error from
 *     an earlier asynchronous failure surfaces as MTP_ERR_CUDA.
 *   - Bad data never traps: it sets row-flag bits, and the flagged row gets
 *     defined outputs (tokens and accept length -1, statistics and loss NaN,
 *     gradient 0).
 *   - Temperatures scale both target and draft logits: p = softmax(z_t / T),
 *     q = softmax(z_d / T).  -inf logits are allowed (probability 0).
 */
#ifndef MTP_RS_H
#define MTP_RS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same type as cudaStream_t / CUstream). */
typedef struct CUstream_st *mtp_stream_t;

typedef enum {
    MTP_OK = 0,
    MTP_ERR_INVALID_ARG = 1,      /* NULL required pointer, bad size or gamma */
    MTP_ERR_UNSUPPORTED_DTYPE = 2,
    MTP_ERR_MISALIGNED = 3,       /* logit base pointer not 16-byte aligned */
    MTP_ERR_CUDA = 4,             /* CUDA launch / earlier asynchronous error */
    MTP_ERR_TIMEOUT = 5,          /* an on-chip wait gave up.  Calls are asynchronous, so no
                                     call returns it: the device reports the affected rows
                                     with MTP_ROW_TIMEOUT, and the Python binding's
                                     check_row_flags() raises this status for them. */
    MTP_ERR_NO_DEVICE = 6         /* no usable cluster launch configuration */
} mtp_status;

typedef enum { MTP_DTYPE_F32 = 0, MTP_DTYPE_BF16 = 1 } mtp_dtype;

/* Per-row flag bits written by the device. */
enum {
    MTP_ROW_NONFINITE = 1,   /* a read logit is NaN or +inf, or a read row is all -inf */
    MTP_ROW_BAD_ID = 2,      /* a draft id outside [0, V) */
    MTP_ROW_BAD_TEMP = 4,    /* temperature < 0, NaN or inf (0 is greedy where supported) */
    MTP_ROW_ZERO_MASS = 8,   /* residual mass rounded to 0 at a rejection; the
                                token was drawn from p_j instead (outputs valid) */
    MTP_ROW_BAD_UNIFORM = 16,/* a uniform outside [0, 1) or NaN */
    MTP_ROW_TIMEOUT = 32     /* an on-chip wait gave up (bounded waits) */
};

/* Maximum number of draft steps per call. */
#define MTP_MAX_GAMMA 32

/*
 * mtp_rs_verify -- batched MTP rejection-sampling verification [BB §2,
 * App. G.1; EM "Speculative Decoding"].
 *
 * For each sequence b: for i = 0..gamma-1, p_i = softmax(target[b,i]/T_b),
 * q_i = softmax(draft[b,i]/T_b); draft token y_i = draft_ids[b,i] is
 * accepted iff uniforms[b,i] * q_i(y_i) < p_i(y_i) (probability
 * min(1, p/q)).  At the first rejection j the replacement is drawn from
 * norm(max(0, p_j - q_j)) by inverse CDF with uniforms[b,gamma]: the smallest
 * vocabulary index v with C(v) > u * R (ascending index, C the running sum, R
 * the total).  If all gamma drafts are accepted, the bonus token is drawn the
 * same way from p_gamma.  Rows after the stop are not used unless statistics
 * are requested (without statistics the streaming kernel may prefetch a
 * bounded part of the next position's rows before a decision is known; it
 * never reads beyond the caller's arrays).
 *
 * T_b == 0 is greedy decoding: p and q are one-hot at the row's arg max
 * (ties to the smallest index), so y_i is accepted iff it is the target's
 * arg max, and the next token is the target's arg max; statistics need
 * T_b > 0 (a greedy sequence with alpha/entropy requested is flagged
 * MTP_ROW_BAD_TEMP).
 *
 *   target_logits [B, gamma+1, V] dtype     draft_logits [B, gamma, V] dtype
 *   draft_ids     [B, gamma] int32          temperature  [B] float32 (>= 0)
 *   uniforms      [B, gamma+1] float32 in [0, 1)
 *   out_tokens    [B, gamma+1] int32: accepted drafts, then the drawn token,
 *                 then -1 padding.                               (required)
 *   accept_len    [B] int32: number of accepted drafts n in [0, gamma], -1 if
 *                 the row is flagged with an error bit.          (required)
 *   alpha         [B, gamma] float32 or NULL: overlap sum_v min(p_i, q_i)
 *   entropy       [B, gamma+1] float32 or NULL: H(p_i) in nats
 *                 (alpha and entropy must both be given or both NULL; when
 *                 given, every row of the sequence is read.)
 *   row_flags     [B] int32 or NULL.
 * Requirements: B >= 0 (B = 0 is a no-op), 1 <= gamma <= MTP_MAX_GAMMA,
 * V >= 1.
 */
int mtp_rs_verify(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                  const int32_t *draft_ids, const float *temperature, const float *uniforms,
                  int B, int gamma, int V,
                  int32_t *out_tokens, int32_t *accept_len, float *alpha, float *entropy,
                  int32_t *row_flags, mtp_stream_t stream);

/*
 * mtp_to_verify -- batched target-only verification [BB §2 "Acceptance
 * methods", App. D.2 "Target-Only Sampling"].
 *
 * For each sequence b: the draft token of position i is y_i = arg max of
 * draft[b,i] (ties to the smallest index; no draft probability is formed),
 * accepted iff uniforms[b,i] < p_i(y_i) with p_i = softmax(target[b,i]/T_b).
 * At the first rejection j the replacement is drawn by inverse CDF with
 * uniforms[b,gamma] from p_j with y_j removed -- the residual of rejection
 * sampling with a one-hot draft, so the output law stays p.  After gamma
 * accepts the bonus token is drawn from p_gamma.  T_b == 0 is greedy: accept
 * while y_i is the target's arg max, then emit the target's arg max.
 *
 *   target_logits [B, gamma+1, V], draft_logits [B, gamma, V], dtype as above
 *   temperature [B] (>= 0), uniforms [B, gamma+1] in [0, 1)
 *   out_tokens [B, gamma+1], accept_len [B]              (required)
 *   draft_tokens [B, gamma] int32 or NULL: y_i for every position whose
 *                decision was taken, -1 elsewhere
 *   row_flags [B] or NULL
 * Requirements: rows of whole 16-byte vectors (V a multiple of 8 for bf16,
 * 4 for float32; MTP_ERR_MISALIGNED otherwise) and gamma <= 8
 * (MTP_ERR_INVALID_ARG otherwise).
 */
int mtp_to_verify(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                  const float *temperature, const float *uniforms, int B, int gamma, int V,
                  int32_t *out_tokens, int32_t *accept_len, int32_t *draft_tokens, int32_t *row_flags,
                  mtp_stream_t stream);

/*
 * mtp_gumbel_verify -- mtp_rs_verify with the Gumbel-max final draw [BB App.
 * G.2 "Gumbel-Max Trick (vLLM)"]: the acceptance chain is the same (u_i
 * q_i(y_i) < p_i(y_i), stop at the first rejection, T = 0 greedy); the
 * replacement at a rejection j is arg max_v [ln r_v + G_v] over r =
 * max(0, p_j - q_j) (the p_j keys if every r_v rounds to 0, flagged
 * MTP_ROW_ZERO_MASS), and the bonus after gamma accepts is arg max_v [ln
 * p_gamma(v) + G_v].  G_v = -ln(-ln U_v) is standard Gumbel noise drawn in
 * the kernel from Philox4x32-10 (Salmon et al., "Parallel random numbers: as
 * easy as 1, 2, 3", SC 2011): key = seed (low 32 bits first), counter =
 * (v / 4, row, b, offset) with row the position drawn from (j, or gamma for
 * the bonus) and b the sequence, word v mod 4, U_v = (floor(x / 2^8) + 1/2)
 * / 2^24.  The same (seed, offset) gives the same tokens; callers advance
 * offset (or the seed) between calls for fresh noise.
 *
 *   target_logits [B, gamma+1, V], draft_logits [B, gamma, V] dtype
 *   draft_ids [B, gamma] int32, temperature [B] float32 (0 = greedy)
 *   uniforms [B, gamma+1] float32: u[b, 0..gamma-1] are the accept tests,
 *     u[b, gamma] is not read
 *   out_tokens [B, gamma+1], accept_len [B], row_flags [B] or NULL: as for
 *   mtp_rs_verify.
 * Requirements: 1 <= gamma <= 8 (else MTP_ERR_INVALID_ARG); 16-byte aligned
 * logit bases and V a multiple of 16 / esize (else MTP_ERR_MISALIGNED).
 */
int mtp_gumbel_verify(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                      const int32_t *draft_ids, const float *temperature, const float *uniforms, uint64_t seed,
                      uint32_t offset, int B, int gamma, int V, int32_t *out_tokens, int32_t *accept_len,
                      int32_t *row_flags, mtp_stream_t stream);

/*
 * mtp_draft_sample -- the draft stage of production rejection sampling [BB
 * App. G: draft tokens are drawn from q, G.1 multinomial (SGLang), G.2
 * Gumbel-max (vLLM)]: one token per row of draft_logits [R, V] (R = B x gamma
 * rows for a batch of MTP steps, any row order) from q_r = softmax(z_r / T_r).
 *   method 0: inverse CDF with uniforms [R] in [0, 1): the smallest v with
 *             sum_{w <= v} q_w > u_r (ascending index; if rounding leaves
 *             none, the last v with q_v > 0);
 *   method 1: Gumbel-max arg max_v [ln q_v + G_v], the noise of
 *             mtp_gumbel_verify with counter (v / 4, 0, r, offset) under key
 *             seed; uniforms is not read (may be NULL).
 *   T_r = 0: greedy arg max (ties to the smallest index).
 *   out_ids [R] int32 (-1 for a flagged row), row_flags [R] or NULL
 *   (BAD_TEMP, BAD_UNIFORM, NONFINITE).
 * Requirements: 16-byte aligned base and V a multiple of 16 / esize (else
 * MTP_ERR_MISALIGNED).  Inverse CDF: each row is read once from HBM and one
 * chunk of it a second time for the draw.  Gumbel-max: each row is read once
 * (its arg max needs no normaliser); a near-tie of the two best keys
 * re-reads those two logits.
 */
int mtp_draft_sample(const void *draft_logits, mtp_dtype dtype, const float *temperature, const float *uniforms,
                     int method, uint64_t seed, uint32_t offset, int R, int V, int32_t *out_ids,
                     int32_t *row_flags, mtp_stream_t stream);

/*
 * mtp_row_stats -- per-position overlap and target entropy without
 * decisions [BB §3, §8: alpha = sum_v min(p_v, q_v) = 1 - TV; entropy
 * H(p) = -sum_v p_v log p_v in nats].
 *
 *   target_logits [B, gamma+1, V], draft_logits [B, gamma, V], temperature [B]
 *   alpha [B, gamma] float32 (required), entropy [B, gamma+1] float32
 *   (required), row_flags [B] int32 or NULL.
 * Runs on the cluster-resident kernel; mtp_tuning.stats_kernel selects the
 * streaming kernel of mtp_rs_diagnostics or the TMEM-resident kernel
 * (aligned rows, gamma <= 8) instead.
 */
int mtp_row_stats(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                  const float *temperature, int B, int gamma, int V,
                  float *alpha, float *entropy, int32_t *row_flags, mtp_stream_t stream);

/*
 * mtp_rs_diagnostics -- per-position acceptance diagnostics without
 * decisions [BB §2 "Acceptance methods", §8 "Robustness of acceptance
 * methods", App. E "Rejection Sampling Decision Boundary Derivation"].
 *
 * For sequence b and draft position i < gamma, with p = softmax(target[b,i]
 * / T_b) and q = softmax(draft[b,i] / T_b):
 *   alpha[b,i]     = sum_v min(p_v, q_v) = 1 - d_TV(p, q)
 *   ent_q[b,i]     = H(q) in nats
 *   kl[b,i]        = D_KL(q || p) = sum_v q_v ln(q_v / p_v) in nats (rounding
 *                    below 0 is clamped to 0; +inf where some p_v = 0 < q_v)
 *   yhat[b,i]      = arg max_v draft[b,i,v], ties to the smallest index
 *                    (the token target-only acceptance proposes)
 *   p_yhat[b,i]    = p(yhat), the target-only acceptance probability
 *   rs_better[b,i] = 1 if d_TV(p, q) < 1 - p(yhat), else 0: rejection
 *                    sampling then accepts more often than target-only
 *                    acceptance (evaluated as p(yhat) < alpha)
 * and for i <= gamma ent_p[b,i] = H(p_i) in nats.
 *
 *   target_logits [B, gamma+1, V] dtype, draft_logits [B, gamma, V] dtype,
 *   temperature [B] float32 (T_b > 0; otherwise, T = 0 included, the row is
 *   flagged MTP_ROW_BAD_TEMP: these statistics need T > 0).
 *   Outputs, each float32 / int32 in the layout above or NULL (not written):
 *   alpha, ent_p, ent_q, kl, yhat, p_yhat, rs_better; row_flags [B].
 *   A flagged row gets NaN in its float outputs and -1 in yhat and
 *   rs_better.
 * Requirements: 1 <= gamma <= 8 (else MTP_ERR_INVALID_ARG); 16-byte aligned
 * logit bases and V a multiple of 16 / esize (else MTP_ERR_MISALIGNED).
 * Every row is read twice: once from HBM, once more shortly after (L2).
 */
int mtp_rs_diagnostics(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                       const float *temperature, int B, int gamma, int V, float *alpha, float *ent_p,
                       float *ent_q, float *kl, int32_t *yhat, float *p_yhat, int32_t *rs_better,
                       int32_t *row_flags, mtp_stream_t stream);

/*
 * mtp_tv_loss_fwd_bwd -- fused forward and backward of the end-to-end TV
 * loss [BB §4, App. A, App. F].
 *
 * For every token position t and draft step k: p = softmax(target[t,k]/T)
 * (detached), q = softmax(draft[t,k]/T), alpha_k = sum_v min(p_v, q_v),
 * S_k = sum_v 1[q_v <= p_v] q_v.  The loss of position t is
 *     l_t = - sum_{m=1..gamma} prod_{i<=m} alpha_i
 * and the gradient with respect to the draft logits is
 *     grad[t,k,j] = grad_scale * (dl_t/dalpha_k) * (1/T) * q_j (1[q_j <= p_j] - S_k).
 * The pages call the loss "normalised"; a constant normaliser such as 1/gamma
 * is folded into grad_scale by the caller.
 *
 *   target_logits, draft_logits [N, gamma, V] dtype
 *   loss  [N] float32 (required)            alpha [N, gamma] float32 or NULL
 *   grad_draft_logits [N, gamma, V] float32 (required; fully overwritten)
 *   row_flags [N] int32 or NULL.
 * Requirements: N >= 0, 1 <= gamma <= MTP_MAX_GAMMA, V >= 1, temperature > 0
 * (otherwise every position is flagged MTP_ROW_BAD_TEMP).
 */
int mtp_tv_loss_fwd_bwd(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                        float temperature, int N, int gamma, int V, float grad_scale,
                        float *loss, float *alpha, float *grad_draft_logits, int32_t *row_flags,
                        mtp_stream_t stream);

/*
 * mtp_tv_loss_ex -- mtp_tv_loss_fwd_bwd with the layout and loss variants of
 * [BB] App. F:
 *   target_layout 0: target_logits [N, gamma, V] like the draft;
 *   target_layout 1: shared target rows [N + gamma - 1, V]: pair (t, k)
 *     reads row t + k, the target model's distribution at the token draft
 *     step k of position t predicts (consecutive positions share rows);
 *   loss_kind 0: the e2e loss of mtp_tv_loss_fwd_bwd;
 *   loss_kind 1: l_t = sum_k clamp(1 - alpha_k, 0, tau_max), the per-step
 *     clamped loss, with dl_t/dalpha_k = -1 strictly inside the clamp and 0
 *     elsewhere (the subgradient 0 at the kinks); tau_max >= 0.
 * Other arguments, outputs and flags as for mtp_tv_loss_fwd_bwd.  Returns
 * MTP_ERR_INVALID_ARG for another layout or loss kind, or tau_max < 0 or NaN
 * with loss_kind 1.
 */
int mtp_tv_loss_ex(const void *target_logits, const void *draft_logits, mtp_dtype dtype, float temperature,
                   int N, int gamma, int V, float grad_scale, int target_layout, int loss_kind, float tau_max,
                   float *loss, float *alpha, float *grad_draft_logits, int32_t *row_flags, mtp_stream_t stream);

/*
 * mtp_tv_loss_topk -- the top-K path of the fused TV loss [BB App. F: "an
 * optional top-K path reduces memory from O(|V|) to O(K)"]: the detached
 * target of pair (t, k) is given as its K cached logits target_values
 * [N, gamma, K] (dtype) at vocabulary indices target_idx [N, gamma, K]
 * (int32, distinct, in [0, V)).  The target distribution is the softmax of
 * those K logits at temperature T, renormalised over the K entries (zero
 * elsewhere); q = softmax(draft[t,k] / T) over the full row.  Then
 *   alpha~_k = sum_e min(p~_e, q_{idx_e}),  S~_k = sum_{e: q <= p~} q_{idx_e},
 * the loss is the e2e loss (loss_kind 0) or sum_k clamp(1 - alpha~_k, 0,
 * tau_max) (loss_kind 1), and the gradient with respect to the draft logits
 * is that of mtp_tv_loss_fwd_bwd with p~ in place of p.  Outputs and flags
 * as for mtp_tv_loss_fwd_bwd; an index outside [0, V) flags MTP_ROW_BAD_ID.
 * Requirements: 1 <= K <= V and gamma <= 8 (else MTP_ERR_INVALID_ARG);
 * 16-byte aligned draft and gradient bases and V a multiple of 16 / esize
 * (else MTP_ERR_MISALIGNED).  Bytes per pair: the draft row read once
 * (plus a re-read from L2), the gradient row written once, 6 K bytes (bf16)
 * of target entries.
 */
int mtp_tv_loss_topk(const void *target_values, const int32_t *target_idx, const void *draft_logits,
                     mtp_dtype dtype, float temperature, int N, int gamma, int K, int V, float grad_scale,
                     int loss_kind, float tau_max, float *loss, float *alpha, float *grad_draft_logits,
                     int32_t *row_flags, mtp_stream_t stream);

/*
 * mtp_query_plan -- the launch plan a call would use on the current device
 * (diagnostics; launches nothing).  op: 0 = mtp_rs_verify, 1 = mtp_rs_verify
 * with statistics, 2 = mtp_row_stats, 3 = mtp_tv_loss_fwd_bwd, 4 =
 * mtp_rs_verify forced onto the cluster-resident kernel, 5 =
 * mtp_tv_loss_fwd_bwd forced onto the cluster-resident kernel, 6 =
 * mtp_rs_diagnostics, 7 = mtp_row_stats forced onto the cluster-resident
 * kernel, 8 = mtp_to_verify, 9 = mtp_gumbel_verify, 10 = mtp_draft_sample by
 * inverse CDF, 11 = mtp_draft_sample by Gumbel-max (10 and 11: units = rows;
 * gamma is not used but must be valid).  Otherwise units = B
 * (sequences) or N (positions).  Outputs (any may be NULL): cluster_size (C,
 * CTAs per thread-block cluster; the vocabulary is split across them),
 * clusters (persistent clusters launched), smem_bytes (dynamic shared memory
 * per CTA), resident_drafts (cluster-resident TV kernel: draft slices kept on
 * chip; ops 0 and 8-11: chunk slots per warp of the streaming kernel, 0 when the call
 * would use the cluster-resident kernel or, op 11, the one-pass Gumbel-max
 * kernel; else 0).
 * Returns the status the call's planning step would return.
 */
int mtp_query_plan(int op, mtp_dtype dtype, int units, int gamma, int V, int *cluster_size, int *clusters,
                   int *smem_bytes, int *resident_drafts);

/*
 * Kernel choices for mtp_tuning (0 = the planner's choice everywhere).
 */
enum {
    MTP_KERNEL_AUTO = 0,
    MTP_KERNEL_STREAM = 1,      /* per-warp streaming kernels (rows re-read from L2) */
    MTP_KERNEL_RESIDENT = 2,    /* cluster-resident kernels (row slices in shared memory) */
    MTP_KERNEL_TMEM = 3         /* tensor-memory-resident kernels (row slices parked in TMEM) */
};

/*
 * mtp_tuning -- explicit, process-wide overrides of the launch planners, for
 * tests and tuning sweeps.  The library reads no environment variable: the
 * kernel a call runs depends only on its arguments, the device and the last
 * mtp_set_tuning() of the process.  Every field 0 (or a zero-initialised
 * struct, or mtp_set_tuning(NULL)) restores the planners' own choices.  An
 * override that does not fit a call (a cluster size whose shared memory does
 * not fit, say) is ignored for that call or makes the call return
 * MTP_ERR_NO_DEVICE; outputs never depend on it beyond the documented
 * tie-breaking of equal results.
 */
typedef struct mtp_tuning {
    int cluster_size;        /* CTAs per cluster, 1..16 (streaming kernels: a power of two); 0 = planner */
    int ring_slots;          /* streaming kernels: chunk slots per warp, 2..8; 0 = 2 */
    int lookahead;           /* streaming verify: 0 = gamma positions streamed ahead of the last
                                decision; d + 1 = d positions */
    int chunk_vectors;       /* streaming kernels: 16-byte vectors per chunk, 128, 160 or 192; 0 = planner */
    int max_clusters;        /* cap on the persistent clusters launched; 0 = every co-resident one */
    int verify_kernel;       /* mtp_rs_verify without statistics: MTP_KERNEL_AUTO / _STREAM / _RESIDENT */
    int tv_kernel;           /* TV loss: MTP_KERNEL_AUTO / _STREAM / _RESIDENT / _TMEM (_TMEM where a
                                position's draft rows fit in tensor memory, else as _AUTO) */
    int stats_kernel;        /* mtp_row_stats: MTP_KERNEL_AUTO (= _RESIDENT) / _STREAM / _RESIDENT /
                                _TMEM (where two draft row segments fit a warp's tensor memory) */
    int tv_resident_drafts;  /* cluster-resident TV kernel: cap on draft slices kept on chip; 0 = none */
    int tv_l2_mb;            /* streaming TV kernel: cap positions in flight so the rows they re-read
                                fit this many MB; 0 = no cap */
    int pair_l2_mb;          /* streaming row-pair kernel: the same cap for sequences; 0 = no cap */
    int row_streams;         /* cluster-resident row kernel: sequences in flight per CTA, 1 or 2; 0 = planner */
    /* Fault injection for tests of the bounded waits (both 0 in normal use).
     * They act on the TMEM-resident TV kernel only. */
    int fault_wait_us;       /* limit of every on-chip wait in microseconds; 0 = 2 s */
    int fault_skip_position; /* 1 + the position whose first exchange push the cluster's first warp
                                skips: every wait on it gives up, and that position and the later ones
                                of its cluster come back flagged MTP_ROW_TIMEOUT; 0 = none */
} mtp_tuning;

/* Set (t != NULL) or clear (t == NULL) the overrides; affects calls made
 * after it returns, from any thread.  Returns MTP_OK. */
int mtp_set_tuning(const mtp_tuning *t);
/* Copy the current overrides into *t.  MTP_ERR_INVALID_ARG if t is NULL. */
int mtp_get_tuning(mtp_tuning *t);

/* Static description of a status code. */
const char *mtp_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* MTP_RS_H */
