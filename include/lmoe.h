/*
 * lmoe.h -- C ABI of the Stable Latent MoE feed-forward layer on one GB300 (sm_103a).
 *
 * The layer (Kimi K3; sources below) replaces the dense FFN of a decoder block:
 *   lat    = x . W_down^T                          hidden d -> latent L (L = d/2 in K3)
 *   logits = lat . W_r^T,  s = sigmoid(logits)     router over E routed experts
 *   tau[e] = k-th largest s[:, e] in the batch     Quantile-Balancing threshold
 *   top-K of fl32(s - tau) per token               K experts per token, gates s / sum(s)
 *   h      = SiTU(lat . W_g[e]^T, lat . W_v[e]^T)  routed experts work in the latent
 *   u      = sum_j gate_j (h_j . W_ed[e_j]^T)      gate-weighted aggregation
 *   z      = gamma * u / sqrt(mean(u^2) + eps)     RMSNorm before the up-projection
 *   y      = residual + z . W_up^T + sum_s SiTU(x . W_sg[s]^T, x . W_sv[s]^T) . W_sd[s]^T
 * with SiTU(g, v) = silu(c tanh(g/c)) * c tanh(v/c), c = 100.
 *
 * Sources:
 *   [TPP] "The 2.8-Trillion-Parameter Problem: Why Bigger Models Break the Old Playbook"
 *         (aitrending.vip summary), sections "TL;DR" and "Technical Details".
 *   [IK3] The same title, "Part 1 of Inside Kimi K3" (Towards AI article): passages on
 *         Mixture of Experts, Stable LatentMoE, the stabilizers and Quantile Balancing.
 *   [SU]  "苏神复盘 Kimi K3：896 个专家背后，藏着哪些关键技术取舍？" (daily-ai-frontier),
 *         "Merged summary", bullets "LatentMoE" and "Stable LatentMoE".
 * The pages give the structure in words only; the score function, where the threshold
 * acts, the gate normalisation and the SiTU-GLU formula are readings, stated at each call.
 *
 * Conventions for every entry point:
 *   - Every pointer argument is DEVICE memory owned by the caller, unless stated.  The
 *     library allocates nothing, keeps no global state between calls and may be called
 *     concurrently on different streams with disjoint buffers.
 *   - bf16 tensors are raw IEEE bfloat16 bit patterns; all matrices are row-major and
 *     weights are stored [out, in].
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *     asynchronous on that stream and returns after enqueueing its kernels.
 *   - Return value: LMOE_OK, or an LMOE_ERR_* code for a rejected argument or a failed
 *     launch; nothing is enqueued when an argument is rejected.  Errors raised on the
 *     device (a bounded wait that ran out) are read with lmoe_last_device_error after the
 *     stream has synchronised.
 *   - Inputs must be finite.  NaN router logits give an unspecified (but in-bounds)
 *     selection.  Checked mode: with LMOE_CHECK_FINITE=1 in the environment (read at each
 *     call), lmoe_forward scans the router logits it routes on, and a NaN or infinite one
 *     makes lmoe_last_device_error return LMOE_ERR_INVALID_ARG.
 */
#ifndef LMOE_H
#define LMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum lmoe_status {
  LMOE_OK = 0,
  LMOE_ERR_INVALID_ARG = 1,          /* null pointer, negative size, bad combination */
  LMOE_ERR_UNSUPPORTED = 2,          /* shape outside the supported set (see lmoe_forward) */
  LMOE_ERR_CUDA = 3,                 /* a CUDA runtime/driver call or a launch failed */
  LMOE_ERR_DEVICE_TIMEOUT = 4,       /* a device-side wait ran out (from lmoe_last_device_error) */
  LMOE_ERR_WORKSPACE_TOO_SMALL = 5   /* workspace or packed buffer smaller than required */
};

/* Layer sizes.  K3: d=7168, L=3584, E=896, K=16, S=2 ([TPP] Technical Details; [SU]
 * LatentMoE bullet); the pages give no intermediate sizes I and Is. */
typedef struct lmoe_dims {
  int T;      /* tokens in the batch, >= 0 */
  int d;      /* hidden width */
  int L;      /* latent width */
  int E;      /* routed experts */
  int K;      /* routed experts per token */
  int I;      /* routed expert intermediate size */
  int S;      /* shared experts */
  int Is;     /* shared expert intermediate size */
  float c;    /* SiTU-GLU cap (100 for K3) */
  float eps;  /* RMSNorm epsilon (1e-6) */
  int expert_fp8; /* 0: routed experts in bf16; 1: routed experts with e4m3 operands (see
                     below); fixes the packed layout, so pack and forward must agree */
} lmoe_dims;

/* Routed experts in FP8 (lmoe_dims.expert_fp8 = 1).  [SU] Stable LatentMoE bullet:
 * SiTU-GLU soft-caps the outliers that would otherwise blow up the BF16/FP8 dynamic range,
 * i.e. the routed experts are meant to run in FP8; the pages give no recipe.  Reading: both
 * operands of the two routed GEMMs are e4m3 (OCP E4M3: ties to even, saturating at 448)
 * with one fp32 scale per row -- per output feature of each expert's weights (quantised
 * by lmoe_pack_weights), per token for the latent, per (token, expert) pair for the SiTU
 * output -- s = amax/448 and code = e4m3(x/s), every step an IEEE fp32 operation; the GEMM
 * accumulates in fp32 and multiplies its sum by both scales.  The latent and the SiTU
 * output are quantised from their bf16 values.  The dense GEMMs, routing, combine and
 * RMSNorm are unchanged.  Requires L and I multiples of 128. */

/* Unpacked weights as a caller holds them (device pointers, bf16 unless stated). */
typedef struct lmoe_weights {
  const void *w_down;    /* [L, d]      latent down-projection */
  const void *w_router;  /* [E, L]      router */
  const void *w_gate;    /* [E, I, L]   routed experts, gate branch */
  const void *w_value;   /* [E, I, L]   routed experts, value branch */
  const void *w_edown;   /* [E, L, I]   routed experts, down projection */
  const float *gamma;    /* [L] fp32    RMSNorm weight */
  const void *w_up;      /* [d, L]      up-projection */
  const void *w_sgate;   /* [S, Is, d]  shared experts, gate branch */
  const void *w_svalue;  /* [S, Is, d]  shared experts, value branch */
  const void *w_sdown;   /* [S, d, Is]  shared experts, down projection */
} lmoe_weights;

/* Stages of lmoe_forward, in launch order (for lmoe_io.stage_events). */
enum lmoe_stage {
  LMOE_STAGE_LATENT_SHARED = 0, /* x . [W_down ; W_shared_gate/value]^T, SiTU on the shared part */
  LMOE_STAGE_ROUTER = 1,        /* router logits (skipped when logits_in is given) */
  LMOE_STAGE_THRESHOLDS = 2,    /* in-batch Quantile-Balancing thresholds (when solved) */
  LMOE_STAGE_ROUTE = 3,         /* top-K selection and gates */
  LMOE_STAGE_DISPATCH = 4,      /* expert segments: token indices per expert */
  LMOE_STAGE_EXPERT_GATE_UP = 5,/* grouped gate/value GEMM with SiTU-GLU */
  LMOE_STAGE_EXPERT_DOWN = 6,   /* grouped down-projection GEMM */
  LMOE_STAGE_COMBINE = 7,       /* gate-weighted aggregation + RMSNorm */
  LMOE_STAGE_OUTPUT = 8,        /* up-projection + shared down-projection + residual */
  LMOE_NUM_STAGES = 9
};

/* Optional routing inputs and debug outputs of lmoe_forward.  Any pointer may be NULL. */
typedef struct lmoe_io {
  const float *tau_in;   /* [E] thresholds to route against (e.g. from a prefill batch) */
  int balance;           /* used when tau_in == NULL: 1 = solve thresholds from this batch
                            (Quantile Balancing), 0 = plain top-K without thresholds */
  const float *logits_in;/* [T, E] fp32 router logits to route on instead of computing
                            them from the latent (replay, or routing done elsewhere) */
  float *logits_out;     /* [T, E] router logits used */
  float *tau_out;        /* [E] thresholds used (zeros when balance == 0) */
  int32_t *idx_out;      /* [T, K] selected experts, slot order */
  float *gate_out;       /* [T, K] gates */
  int32_t *counts_out;   /* [E] tokens routed to each expert */
  void **stage_events;   /* host array of LMOE_NUM_STAGES + 1 cudaEvent_t handles, or NULL:
                            event i is recorded on the stream before stage i, the last one
                            after the final stage (skipped stages record back to back) */
  int kernel_launches;   /* out: number of kernels this call launched */
  void *aux_stream;      /* optional second cudaStream_t: with it (and T >= LMOE_OVERLAP_MIN_T)
                            the shared experts run on it, on shared_sms SMs, while the routed
                            path runs on `stream` on the others; `stream` waits for it before
                            the output GEMM, so the call stays ordered on `stream` */
  void *aux_events[2];   /* two cudaEvent_t handles (fork, join), required with aux_stream */
  int shared_sms;        /* SMs for the shared experts while they overlap (0: a third) */
  int phase;             /* LMOE_PHASE_*: the whole layer (0), or one of its two halves */
  float *cand_out;       /* LMOE_PHASE_ROUTER only: [cand_k, E] threshold candidates of this
                            batch, as lmoe_threshold_candidates writes them */
  int cand_k;            /* rank the candidates serve (required with cand_out, >= 1) */
  float *tau_ema;        /* [E] streaming thresholds, in/out, or NULL.  With tau_in == NULL
                            and balance == 1: the batch's thresholds are solved, folded into
                            tau_ema by lmoe_tau_ema (ema_beta, ema_first), and the batch is
                            routed against the updated tau_ema (tau_out receives it) */
  float ema_beta;        /* weight of the previous tau_ema, in [0, 1] */
  int ema_first;         /* 1: this step initialises tau_ema to the batch's thresholds */
  unsigned long long *load_stats; /* counters updated with this step's per-expert token
                            counts, as lmoe_load_stats_update does, or NULL */
  void *save_pre;        /* [T*K, 2I] bf16, or NULL: a training step also stores the routed
                            experts' gate/value pre-activations here (slot order; per slot,
                            groups of 16 gate then 16 value features), so that the backward
                            need not recompute them.  bf16 routed experts only. */
  void *save_pre_shared; /* [T, 2 S Is] bf16, or NULL: likewise the shared experts'
                            pre-activations (per token, groups of 16 gate then 16 value
                            features over the S Is concatenated features) */
  float *y_f32_out;      /* [T, d] fp32, or NULL: the output as the up-projection's epilogue
                            computes it in fp32 (accumulator + residual), before the store
                            that rounds it to bf16; y is exactly this value rounded to
                            nearest even.  For checking the arithmetic apart from the final
                            rounding; costs one extra fp32 store of the output */
  const float *logit_bias; /* [E] fp32, or NULL: added to the router logits the layer
                            computes, logits[t, e] = fl32(lat[t] . W_r[e] + logit_bias[e]),
                            in the router GEMM's epilogue; thresholds, selection and gates
                            all see the biased logits.  (A router with a per-expert bias; the
                            skewed-router workload adds a Zipf bias this way.)  Ignored when
                            logits_in is given. */
} lmoe_io;

/* lmoe_io.phase.  The layer splits where its only cross-batch quantity, the thresholds, is
 * needed: a batch spread over several ranks solves one threshold set over all of them by
 * running LMOE_PHASE_ROUTER on each rank (with cand_out), exchanging the candidates (an
 * all-gather), reducing them with lmoe_thresholds, and running LMOE_PHASE_EXPERTS with the
 * result as tau_in.  LMOE_PHASE_EXPERTS continues from the workspace that a
 * LMOE_PHASE_ROUTER call with the same dims, packed weights, io->logits_in, io->aux_stream
 * and io->aux_events left on the same stream; it does not read x (which may be NULL).
 * Together the two phases compute what LMOE_PHASE_ALL computes. */
enum lmoe_phase {
  LMOE_PHASE_ALL = 0,      /* stages LATENT_SHARED .. OUTPUT */
  LMOE_PHASE_ROUTER = 1,   /* stages LATENT_SHARED and ROUTER (+ candidates) */
  LMOE_PHASE_EXPERTS = 2   /* stages THRESHOLDS .. OUTPUT */
};

/* Batches at least this large run the shared experts concurrently when lmoe_io.aux_stream is
 * given; the workspace of such batches holds their fp32 output [T, d]. */
#define LMOE_OVERLAP_MIN_T 512

/* Bytes of the packed weight buffer for `dims` (0 if the dims are invalid). */
size_t lmoe_packed_bytes(const lmoe_dims *dims);

/* Repack unpacked weights into the layout lmoe_forward reads: the shared gate/value rows
 * are stacked under W_down and interleaved in groups of 16 rows, the routed gate/value rows
 * likewise per expert, and W_up and the shared down-projections are concatenated along
 * their input dimension.  `packed` (device, packed_bytes >= lmoe_packed_bytes(dims), 256-byte
 * aligned) is overwritten; the inputs are only read.  Pure function of its inputs. */
int lmoe_pack_weights(const lmoe_dims *dims, const lmoe_weights *w, void *packed,
                      size_t packed_bytes, void *stream);

/* Bytes of device workspace lmoe_forward uses for `dims` (0 if the dims are invalid).  For a
 * batch of at most 128 tokens this includes a 12 MiB region for split-K partial sums of the
 * dense GEMMs (a single M-tile would otherwise leave most SMs idle).  lmoe_forward also runs
 * in a workspace 12 MiB smaller, without splitting them, and only whole-layer calls
 * (LMOE_PHASE_ALL) split: the two phases keep every token's logits and output bit-identical
 * to those of any other batch it is part of. */
size_t lmoe_workspace_bytes(const lmoe_dims *dims);

/* Quantile-Balancing thresholds.  [IK3] Quantile Balancing passage: each step's routing
 * thresholds are read off the distribution of the router scores -- the score an expert
 * needs to stay within its fair share of tokens; [SU] Stable LatentMoE bullet: it solves
 * directly for per-expert Top-K thresholds.  Reading: tau[e] = the k-th largest
 * s[t, e] = sigmoid(logits[t, e]) over the T tokens, with k = k_rank, or, when k_rank <= 0,
 * k = max(1, floor(T*K/E)) (at most T).  Bit-exact: s uses the fp32 sigmoid specified at
 * lmoe_route, and the threshold is one of the s values.
 *   logits [T, E] fp32 (read), tau [E] fp32 (written).  T == 0 writes nothing.
 * Errors: INVALID_ARG for null pointers or T < 0, E < 1, K < 1, k_rank > T. */
int lmoe_thresholds(const float *logits, int T, int E, int K, int k_rank, float *tau,
                    void *stream);

/* The rank k of the Quantile-Balancing threshold among a column's T scores, the fair share
 * of tokens per expert ([IK3] Quantile Balancing passage): k = max(1, floor(T*K/E)), at
 * most T; 0 for T == 0.  lmoe_thresholds (k_rank <= 0) and lmoe_forward use it; a batch
 * spread over ranks passes the whole batch's T.  Returns -1 for K < 1, E < 1, T < 0 or
 * T > 2^40.  Host function; touches no device. */
int lmoe_fair_share_rank(long long T, int K, int E);

/* Threshold candidates of one part of a batch that is spread over several ranks.
 * [IK3] Quantile Balancing passage: the threshold is read off the distribution of the
 * scores of the whole step's batch; the pages do not say how a batch split across devices
 * obtains it.  Reading: the k largest scores of a column over the whole batch lie among the
 * k largest of each part, so each part contributes those.  Column e of cand receives the
 * logits of the min(k, T) tokens with the largest scores s = sigmoid(logit) of expert e
 * (scores above the min(k, T)-th largest first, then tokens whose score equals it, each
 * group in token order), and rows T..k-1, when T < k, receive -FLT_MAX (the lowest score).
 * Stacking the candidates of all parts as [parts * k, E] and calling lmoe_thresholds on
 * them with k_rank = k gives, bit for bit, the thresholds of the whole batch.
 *   logits [T, E] fp32 (read), cand [k, E] fp32 (written).  T == 0 fills cand with -FLT_MAX.
 * Errors: INVALID_ARG for null pointers, T < 0, E < 1, k < 1. */
int lmoe_threshold_candidates(const float *logits, int T, int E, int k, float *cand,
                              void *stream);

/* Streaming thresholds.  [IK3] Quantile Balancing passage: the thresholds are read off the
 * distribution of the router scores at each step; the pages name no cross-step rule.
 * Reading: a threshold that persists across steps (decode batches are too small to carry a
 * quantile) is the exponential moving average of the per-step thresholds, in fp32:
 *   tau_ema[e] = first ? tau_step[e] : fma(beta, tau_ema[e] - tau_step[e], tau_step[e]).
 *   tau_step [E] (read), tau_ema [E] (read and written).
 * Errors: INVALID_ARG for null pointers, E < 0, beta outside [0, 1]. */
int lmoe_tau_ema(const float *tau_step, float *tau_ema, int E, float beta, int first,
                 void *stream);

/* Load statistics over steps ([IK3]: balancing keeps experts from sitting idle while a few
 * take the traffic).  Adds one step's per-expert token counts [E] to the caller's 64-bit
 * counters acc [4 + 4E] (zero them before the first step):
 *   acc[0] steps, acc[1] routed (token, expert) pairs, acc[2] sum over steps of the largest
 *   count, acc[3] largest count of any expert in any step; for each expert e: acc[4 + e] sum
 *   of its counts, acc[4 + E + e] sum of their squares, acc[4 + 2E + e] steps in which it
 *   received no token, acc[4 + 3E + e] its largest count.
 * Errors: INVALID_ARG for null pointers or E < 1. */
int lmoe_load_stats_update(const int32_t *counts, int E, unsigned long long *acc, void *stream);

/* Expert-parallel dispatch and combine, packed and unpacked on one device.  [IK3] Stable
 * LatentMoE and communication passages: the routed experts live on different GPUs, each
 * selected expert receives the token's vector and the outputs travel back to be combined;
 * projecting to the latent first halves the bytes ([TPP] Technical Details: 7168 -> 3584).
 * Readings: R ranks host the E experts in equal contiguous blocks (expert e on rank
 * e / (E/R)); a token's row travels once to every rank hosting at least one of its K
 * experts; the (token, rank) pairs are laid out by rank, then token.  The buffers below are
 * what would cross the interconnect; the transfer (an all-to-all) is not part of the library.
 * Requires 1 <= K <= 32, 1 <= R <= 64, E % R == 0.
 *
 * lmoe_ep_workspace_bytes: scratch (device) that dispatch fills and combine reads again.
 * lmoe_ep_dispatch: idx [T, K] int32 (read); rows [T, W] bf16 or NULL (then only the layout);
 *   outputs send_off [R + 1] (pair offsets per rank; P = send_off[R] <= T * min(K, R)),
 *   send_tok [P] (token of each pair), send_slots [P] (bit j: the token's slot j is served
 *   on that rank), send_rows [T * min(K, R), W] bf16 (row of each pair).  W % 8 == 0,
 *   16-byte-aligned rows.  Slots whose index is outside [0, E) go to no rank.
 * lmoe_ep_combine: the expert side sums, for every pair, gate[t, j] * o[inv[t, j]] over its
 *   slots j in ascending order by fp32 fused multiply-adds and rounds to bf16 into part [P, W];
 *   the source side adds a token's pairs in rank order in fp32 into u [T, W].  o [*, W] bf16
 *   (the experts' outputs, one row per (token, slot) at inv [T, K]), gate [T, K] fp32, and
 *   send_off / send_tok / send_slots / ws from lmoe_ep_dispatch with the same idx.
 * Errors: INVALID_ARG (null pointers, negative sizes, W, alignment), UNSUPPORTED (K, R, E),
 *   WORKSPACE_TOO_SMALL. */
size_t lmoe_ep_workspace_bytes(int T, int K, int E, int R);
int lmoe_ep_dispatch(const int32_t *idx, int T, int K, int E, int R, const void *rows, int W,
                     void *send_rows, int32_t *send_off, int32_t *send_tok,
                     uint32_t *send_slots, void *ws, size_t ws_bytes, void *stream);
int lmoe_ep_combine(const int32_t *idx, int T, int K, int E, int R, const int32_t *send_off,
                    const int32_t *send_tok, const uint32_t *send_slots, const int32_t *inv,
                    const float *gate, const void *o, int W, void *part, float *u,
                    const void *ws, void *stream);

/* Top-K routing.  [TPP] Technical Details: a lightweight router selects 16 of 896 routed
 * experts per token; [SU]: Quantile Balancing replaces the predecessor's bias updates.
 * Readings: s = sigmoid(logits) evaluated in fp32 by a fixed sequence of IEEE operations
 * (clamp to [-88, 88]; Cody-Waite reduction by ln 2 split as 22713/32768 + fl32 remainder;
 * degree-7 Taylor polynomial of exp with fl32(1/k!) coefficients by fma Horner; scaling by
 * two exact powers of two; 1/(1+e) with round-to-nearest add and divide); a[t, e] =
 * fl32(s - tau[e]) (tau == NULL: a = s); the K largest a, ties to the lower expert id, in
 * that order; gate_j = fl32(s_j / sum), sum accumulated in fp32 in slot order.
 *   logits [T, E] fp32, tau [E] or NULL, idx [T, K] int32, gate [T, K] fp32,
 *   scores_out [T, E] fp32 or NULL.  Requires 1 <= K <= min(E, 32), E <= 4096.
 * Errors: INVALID_ARG (null outputs, T < 0), UNSUPPORTED (K or E out of range). */
int lmoe_route(const float *logits, const float *tau, int T, int E, int K, int32_t *idx,
               float *gate, float *scores_out, void *stream);

/* The whole layer, y = FFN(x) (+ residual), as stated at the top of this header.
 *   packed   weights from lmoe_pack_weights for the same dims
 *   x        [T, d] bf16;  residual [T, d] bf16 or NULL (then no residual term)
 *   y        [T, d] bf16 output (may not alias x or residual)
 *   workspace, ws_bytes >= lmoe_workspace_bytes(dims) (less the optional split-K region for
 *            T <= 128, see lmoe_workspace_bytes), 256-byte aligned; its contents are
 *            scratch between calls (its first word carries the device error flag)
 *   io       routing options and debug outputs, or NULL (= in-batch thresholds); only
 *            io->kernel_launches is written
 * Supported shapes: d, L, I, Is multiples of 64 (L and I of 128 with expert_fp8);
 * 1 <= K <= min(E, 32); E <= 4096 and a multiple of 16;
 * L <= 16384; T * K < 2^31.  T == 0 is a no-op.
 * Arithmetic: bf16 operands on the tensor cores with fp32 accumulation; the latent, the
 * expert intermediates and the normalised latent are rounded to bf16 between GEMMs;
 * routing is fp32 and reproduces lmoe_thresholds / lmoe_route on the logits it uses.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA. */
int lmoe_forward(const lmoe_dims *dims, const void *packed, const void *x,
                 const void *residual, void *y, void *workspace, size_t ws_bytes,
                 lmoe_io *io, void *stream);

/* End-to-end calls from host memory, overlapped across consecutive batches.  The pages have
 * no counterpart (this is how batches reach the layer, not the layer).  A pipe is a set of
 * caller-owned resources: `depth` device staging slots (x and y buffers of max_tokens rows),
 * three streams (upload, compute, download) and per-slot events.  lmoe_forward_host enqueues,
 * for one batch in slot k = calls % depth: the copy of x_host into slot k's x buffer on the
 * upload stream (after the forward that last read that buffer), lmoe_forward on the compute
 * stream (after that copy, and after the download of slot k's previous output), and the copy
 * of y into y_host on the download stream; then it increments `calls` and returns.  So batch
 * i + 1's upload and batch i - 1's download run while batch i computes, and the forwards,
 * which share one workspace, stay in order on the compute stream.
 *   x_host, y_host: HOST memory [T, d] bf16 (page-locked, or the copies are not
 *     asynchronous); they must stay valid until the download stream has passed this batch
 *     (synchronise it before reading y_host).
 *   residual_is_x: 1 = the layer's residual is x itself (the FFN's residual connection).
 *   workspace, ws_bytes, io: as lmoe_forward (io->stage_events are recorded on the compute
 *     stream).  Calls on one pipe must come from one host thread, in order.
 * Errors: INVALID_ARG (null pointers, depth outside 1..LMOE_HOST_PIPE_MAX_DEPTH, T above
 * max_tokens, misaligned buffers), and lmoe_forward's; nothing is enqueued when an argument
 * is rejected. */
#define LMOE_HOST_PIPE_MAX_DEPTH 4
typedef struct lmoe_host_pipe {
  int depth;        /* staging slots in use, 1..LMOE_HOST_PIPE_MAX_DEPTH */
  int max_tokens;   /* rows each staging buffer holds */
  void *x_dev[LMOE_HOST_PIPE_MAX_DEPTH];      /* [max_tokens, d] bf16 device buffers */
  void *y_dev[LMOE_HOST_PIPE_MAX_DEPTH];      /* [max_tokens, d] bf16 device buffers */
  void *upload, *compute, *download;          /* cudaStream_t, three distinct streams */
  void *uploaded[LMOE_HOST_PIPE_MAX_DEPTH];   /* cudaEvent_t per slot */
  void *computed[LMOE_HOST_PIPE_MAX_DEPTH];
  void *downloaded[LMOE_HOST_PIPE_MAX_DEPTH];
  unsigned long long calls;  /* batches enqueued on this pipe (start at 0; incremented) */
} lmoe_host_pipe;

int lmoe_forward_host(const lmoe_dims *dims, const void *packed, const void *x_host,
                      int residual_is_x, void *y_host, void *workspace, size_t ws_bytes,
                      lmoe_io *io, lmoe_host_pipe *pipe);

/* Building block of lmoe_forward, exposed for verification: C = A . B^T on the tensor
 * cores (tcgen05, fp32 accumulation in TMEM), with A [M, Kd] and B [N, Kd] bf16 row-major
 * (K-major) and C [M, N] fp32.  Requires Kd % 64 == 0, N % 16 == 0, 16-byte aligned
 * pointers.  dev_flag: one caller-owned device word (zero it first); it receives the same
 * error bits as the forward workspace's flag if a device-side wait runs out. */
int lmoe_gemm_bf16(const void *A, const void *B, float *C, int M, int N, int Kd,
                   uint32_t *dev_flag, void *stream);

/* Building block of lmoe_backward's weight gradients, exposed for verification: C = A^T . B
 * summed over all T rows, with A [T, M] and B [T, N] bf16 row-major (token-major, read as
 * MN-major tcgen05 operands) and C [M, N] fp32.  Requires M % 8 == 0, N % 16 == 0, T >= 0,
 * 16-byte aligned pointers.  dev_words: four caller-owned device words, zeroed: word 0
 * receives the error bits of a device-side wait that ran out, words 2 and 3 the row range
 * {0, T} that the call writes there.  T == 0 writes C = 0. */
int lmoe_gemm_wgrad_bf16(const void *A, const void *B, float *C, int M, int N, int T,
                         uint32_t *dev_words, void *stream);

/* Backward pass of the routed-expert branch.  [IK3] stabilizers passage: SiTU-GLU and the
 * RMSNorm after aggregation were introduced to keep training of the routed branch stable.
 * For the branch  h_j = SiTU(lat W_g[e_j]^T, lat W_v[e_j]^T),  o_j = h_j W_ed[e_j]^T,
 * u = sum_j g_j o_j,  z = gamma u / sqrt(mean(u^2) + eps),  and dz = dLoss/dz, computes
 * dLoss/d(lat, gates, gamma, W_g, W_v, W_ed).  Routing is a discrete choice and is held fixed.
 * It continues from the workspace of the lmoe_forward call (same dims, packed weights and
 * stream) that produced z: the latent, the routing, the SiTU outputs and the expert outputs
 * are read from there; the gate/value pre-activations are recomputed.  Operands of the
 * GEMMs are bf16 with fp32 accumulation, like the forward's.  bf16 routed experts only.
 *   lmoe_pack_backward_weights: transposed copies of the weights into packed_bwd
 *     (lmoe_packed_backward_bytes): the expert weights in tiles, from the same unpacked
 *     weights w as the forward's packing, and the dense weights, from `packed` (the
 *     forward's packed buffer, filled by lmoe_pack_weights with the same dims).
 *   lmoe_routed_backward: dz [T, L] fp32 in; pre: the forward's lmoe_io.save_pre buffer,
 *     or NULL (the pre-activations are then recomputed from the latent and W_g, W_v);
 *     dlat [T, L], dgate [T, K], dgamma [L],
 *     dw_gu [E, 2I, L] (rows 0..I-1: W_g, rows I..2I-1: W_v) and dw_ed [E, L, I], all fp32,
 *     out; bwd_ws: lmoe_routed_backward_workspace_bytes of device scratch.
 * Errors: INVALID_ARG, UNSUPPORTED (expert_fp8), WORKSPACE_TOO_SMALL, CUDA. */
size_t lmoe_packed_backward_bytes(const lmoe_dims *dims);
int lmoe_pack_backward_weights(const lmoe_dims *dims, const lmoe_weights *w, const void *packed,
                               void *packed_bwd, size_t bytes, void *stream);
size_t lmoe_routed_backward_workspace_bytes(const lmoe_dims *dims);
int lmoe_routed_backward(const lmoe_dims *dims, const void *packed, const void *packed_bwd,
                         void *workspace, size_t ws_bytes, const float *dz, const void *pre,
                         float *dlat,
                         float *dgate, float *dgamma, float *dw_gu, float *dw_ed, void *bwd_ws,
                         size_t bwd_ws_bytes, void *stream);

/* Backward pass of the whole layer (the same passages; the layer as lmoe_forward computes
 * it).  Given dy = dLoss/dy [T, d] bf16 for the lmoe_forward call whose workspace is passed
 * (same dims, packed weights and stream), computes, all fp32:
 *   dx [T, d]: the gradient reaching x through the latent (x W_down^T) and the shared
 *     experts.  The residual term adds dy itself, which dx does not include.
 *   dgamma [L];
 *   dw_in [L + 2 S Is, d]: rows 0..L-1 dW_down; then row L + s Is + i for shared expert s's
 *     gate row i; then row L + S Is + s Is + i for its value row i;
 *   dw_router [E, L];
 *   dw_gu [E, 2I, L] and dw_ed [E, L, I] as lmoe_routed_backward;
 *   dw_out [d, L + S Is]: columns 0..L-1 dW_up, columns L + s Is + i dW_sd[s][:, i].
 * The router's part: the gates g_j = s_j / sum_i s_i of the selected experts carry gradient
 * to their scores s = sigmoid(logit), and from there to the latent and W_r; the selection
 * (thresholds and top-K) is held fixed.  logits: the fp32 [T, E] router logits the forward
 * routed on -- required when the forward was given lmoe_io.logits_in, else NULL (the ones
 * it computed into the workspace).  x: the forward's input [T, d] bf16.  pre: as for
 * lmoe_routed_backward; pre_shared: the forward's lmoe_io.save_pre_shared buffer, or NULL
 * (the shared experts' pre-activations are then recomputed from x).
 * bwd_ws: lmoe_backward_workspace_bytes of device scratch.  bf16 routed experts only.
 * Errors: INVALID_ARG (null or misaligned pointers), UNSUPPORTED (expert_fp8),
 * WORKSPACE_TOO_SMALL, CUDA. */
size_t lmoe_backward_workspace_bytes(const lmoe_dims *dims);
int lmoe_backward(const lmoe_dims *dims, const void *packed, const void *packed_bwd,
                  void *workspace, size_t ws_bytes, const void *x, const float *logits,
                  const void *dy, const void *pre, const void *pre_shared, float *dx, float *dgamma, float *dw_in, float *dw_router,
                  float *dw_gu, float *dw_ed, float *dw_out, void *bwd_ws, size_t bwd_ws_bytes,
                  void *stream);

/* Building block of the FP8 routed experts, exposed for verification: per-row e4m3
 * quantisation of x [rows, cols] bf16 (row-major, cols a multiple of 16, 16-byte aligned)
 * into codes [rows, cols] and scales [rows] fp32, by the recipe stated at lmoe_dims.
 * Errors: INVALID_ARG (null pointers, rows < 0), UNSUPPORTED (cols). */
int lmoe_quantize_e4m3(const void *x, long long rows, int cols, uint8_t *codes, float *scales,
                       void *stream);

/* Size in bytes of the fixed device array that lmoe_forward_noalloc uses as its workspace. */
#define LMOE_NOALLOC_SCRATCH_BYTES (24u << 20)

/* lmoe_forward for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point: it concerns how the library is called, not the layer.
 * Who needs it: code that may not call cudaMalloc at the point where it runs the layer -- a
 * plug-in whose host framework owns all device memory through its own pool and gives
 * extensions no raw allocations, a serving loop in which an allocation would synchronise
 * the device and stall the other streams, a deployment whose memory is fixed when the
 * process starts.  Arguments and results are those of lmoe_forward without the workspace.
 * Scratch: a LMOE_NOALLOC_SCRATCH_BYTES (24 MiB) array in the library's device image,
 * reserved on every GPU that loads the library until the process exits.  It covers a K3
 * decode batch of up to 152 tokens (64 tokens need 10.08 MiB, or 22.08 MiB with the split-K
 * region, which is used when it fits).  When the workspace without that region exceeds the
 * array, the call returns LMOE_ERR_WORKSPACE_TOO_SMALL and enqueues nothing.
 * Set-up: the first call in each CUDA context looks up the array's device address in that
 * context (cudaGetSymbolAddress, which may load the library's device code); make that first
 * call before any stream capture.  The address is cached per context, so a second context on
 * the same device, or the new context after cudaDeviceReset, gets its own array.  No call
 * allocates or frees memory.
 * Sharing: every call in a context uses the same array, which keeps the last call's
 * contents; each call clears what must start at zero.  Calls whose work overlaps on the
 * GPU (different streams, or host threads without ordering between them) race on the array
 * and corrupt each other's results: serialise them.  A device-side error of a call (a
 * bounded wait that ran out; checked mode's non-finite logit) is recorded in the array:
 * read it with lmoe_noalloc_last_device_error after the stream has synchronised and before
 * the next call, which clears it. */
int lmoe_forward_noalloc(const lmoe_dims *dims, const void *packed, const void *x,
                         const void *residual, void *y, lmoe_io *io, void *stream);

/* lmoe_last_device_error for lmoe_forward_noalloc: synchronously reads and clears the device
 * error flag in the current context's scratch array (no counterpart in the pages either).
 * Returns what lmoe_last_device_error returns for a workspace, or LMOE_ERR_CUDA if the
 * array cannot be reached. */
int lmoe_noalloc_last_device_error(void);

/* Synchronously read and clear the device error flag that lmoe_forward's kernels write
 * into `workspace`.  Every device-side wait is bounded (2 s by default; the environment
 * variable LMOE_WAIT_LIMIT_MS overrides it), and LMOE_FAULT_INJECT=stall makes the first
 * GEMM of a call wait on a barrier that nothing arrives on, so that this path can be
 * tested: its kernels then give up, free their tensor memory and return.  Returns LMOE_OK,
 * LMOE_ERR_DEVICE_TIMEOUT (a bounded wait ran out; the kernel returned early and y is not
 * valid), or LMOE_ERR_INVALID_ARG (checked mode saw a non-finite router logit, or a device
 * index check failed; y is not specified).  Call after the stream has synchronised. */
int lmoe_last_device_error(void *workspace);

/* Static description of a status code. */
const char *lmoe_error_string(int status);

/* Library version, e.g. "lmoe 0.1 sm_103a". */
const char *lmoe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LMOE_H */
