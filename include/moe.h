/*
 * moe.h -- C ABI of the B300 (sm_103a) top-k Mixture-of-Experts layer forward.
 *
 * The layer: router logits -> softmax / top-k gates (+ balancing statistics)
 * -> per-expert capacity with in-token-order dropping -> permute into
 * expert-contiguous rows -> expert FFNs (GELU with bias, or SwiGLU; optional
 * always-on shared experts) -> gate-weighted combine back into token order.
 * Definitions follow these pages (cited by title and section):
 *   [AIG] "Mixture of Experts" (aigrafen.se): gate formula y = sum_{top-k} g_i E_i(x),
 *         g = softmax(W_r x); auxiliary loss; expert capacity; MoE module code.
 *   [AIE] "Mixture of Experts (MoE)" (wiki.ai-engineering.at): router, softmax, top-k,
 *         weighted combination; "Gather/scatter outputs from experts".
 *   [VAN] "MoE Architecture" (vanos001.github.io): TokenChoiceRouter (top-k on logits,
 *         softmax over k), ExpertChoiceRouter, SwiGLUExpert / StandardExpert,
 *         CapacityManagedMoE, HybridMoE (shared experts), "Efficient Batched MoE".
 *   [STP] "Mixture of Experts (MoE)" (learn.starphix.com): "Key Equations",
 *         "Load Balancing (Critical)" (aux loss, z-loss), "Shared + Specialized".
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major,
 *    16-byte aligned, and stay owned by the caller. The library allocates and
 *    frees nothing and never synchronises the stream (except
 *    moe_get_device_status). Work is enqueued on `stream` (a cudaStream_t;
 *    NULL = the legacy default stream) and the call returns before it runs.
 *  - "dtype" tensors hold fp32 (MOE_DT_F32) or bf16 (MOE_DT_BF16) elements as
 *    cfg->dtype says; index tensors are int32; gates/probabilities fp32.
 *  - Argument errors are detected on the host before anything is launched and
 *    returned synchronously (MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED,
 *    MOE_ERR_WORKSPACE). A launch failure returns MOE_ERR_CUDA. Conditions
 *    found on the device (an index out of range, a pipeline wait that ran out
 *    of time) set a sticky error word in the workspace; read it with
 *    moe_get_device_status. No kernel traps or spins without a bound.
 *  - `ws` is a caller-allocated device workspace of at least
 *    moe_workspace_size() bytes (256-byte aligned), initialised once with
 *    moe_workspace_init(). Every stage call with the same cfg may share one
 *    workspace; calls that run concurrently must not.
 *  - Limits: 1 <= k <= min(E, 32); E <= 512; N*k < 2^31; bf16 layers need
 *    d % 64 == 0, F % 64 == 0 and Fs % 64 == 0; fp32 layers need d % 4 == 0.
 *    SwiGLU experts take no biases. Expert choice needs N <= 1<<20.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 2

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, size out of range          */
  MOE_ERR_UNSUPPORTED = 2,  /* valid layer this build does not run (see Limits)     */
  MOE_ERR_WORKSPACE = 3,    /* ws smaller than moe_workspace_size()                 */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime/driver call or launch failed          */
  MOE_ERR_DEVICE_CHECK = 5, /* a kernel found an out-of-range index (sticky word)   */
  MOE_ERR_TIMEOUT = 6       /* a kernel's bounded pipeline wait ran out (sticky)    */
} moe_status;

/* Gate rule. [AIG] formula / [AIE]: g = top-k of softmax(L) (A, no renormalisation);
 * [AIG] MoE code: the chosen weights divided by their sum (A');
 * [VAN] TokenChoiceRouter / [STP] TopKRouter / [AIE] MoELayer: top-k on the logits,
 * then a softmax over those k (B); [VAN] ExpertChoiceRouter: every expert takes its
 * top-C tokens by softmax probability (EC). Top-k ranks logits descending, equal
 * logits to the lower expert index. */
typedef enum moe_gating {
  MOE_GATE_SOFTMAX_TOPK = 0,
  MOE_GATE_SOFTMAX_TOPK_RENORM = 1,
  MOE_GATE_TOPK_SOFTMAX = 2,
  MOE_GATE_EXPERT_CHOICE = 3
} moe_gating;

/* Expert FFN. [AIG] MoE experts / [VAN] StandardExpert: W2 gelu(W1 x + b1) + b2 (exact
 * erf GELU; biases optional). [VAN] SwiGLUExpert / [STP] Expert: W2 (silu(W1 x) * W3 x). */
typedef enum moe_act { MOE_ACT_GELU = 0, MOE_ACT_SWIGLU = 1 } moe_act;

typedef enum moe_dtype { MOE_DT_F32 = 0, MOE_DT_BF16 = 1 } moe_dtype;

/* moe_config.flags bits.
 * MOE_FLAG_DROP_PASSTHROUGH: a token left with no kept (token, expert) row -- every
 *   one of its k choices dropped over capacity (token choice), or picked by no expert
 *   (expert choice) -- gets its own input x added to its output, so it passes through
 *   the layer unchanged apart from the shared experts. [VAN] CapacityManagedMoE,
 *   "Handle dropped tokens (pass through residual)"; [AIG] "Expert capacity": tokens
 *   above the limit "pass through unchanged". Off: such a token's routed part is 0 and
 *   the residual connection is the caller's. */
#define MOE_FLAG_DROP_PASSTHROUGH 1
/* MOE_FLAG_GATHER_ROWS (bf16 layers, moe_forward / moe_forward_overlap): the routed
 *   up-projection loads its A rows straight from x by the permute's row -> token map
 *   (TMA tile::gather4, four rows per copy) instead of from an expert-contiguous copy,
 *   so the permute writes only row metadata and the workspace has no xp region
 *   (max_rows * d * 2 bytes less: 1.9 GB for 16384 tokens, d = 7168, top-8). It costs
 *   up-projection time: the GEMM re-reads each row tile once per output column tile,
 *   and each re-read is 32 gathers instead of one tile copy (measured on B300: the
 *   8192-token d = 512 layer's up-projection 46 -> 133 us, the 16384-token d = 7168
 *   layer's 8.7 -> 22.2 ms). [AIE] "Gather/scatter outputs from experts". */
#define MOE_FLAG_GATHER_ROWS 2

/* Storage of the routed experts' weight matrices w1, w3, w2 (bf16 layers).
 * MOE_WEIGHTS_MXFP8: the routed experts compute in OCP microscaling "MXFP8". Each
 *   weight matrix [rows, K] is FP8 E4M3 codes (1 byte: sign, 4 exponent bits with bias
 *   7, 3 mantissa bits; max 448) with one E8M0 scale byte s per 32 consecutive codes
 *   along K (value = code * 2^(s - 127)), scales [rows, K / 32] row-major
 *   (moe_weights.w1_scale ...). The experts' inputs are quantised the same way: each
 *   permuted token row and each hidden row H is cut into blocks of 32 values whose
 *   shared exponent is floor(log2(max |v|)) - 8 (at least -127) and whose elements
 *   round to the nearest E4M3 code (ties to even, saturating at 448); both matrix
 *   products run on the tensor cores' block-scaled FP8 path with fp32 accumulation.
 *   xp then holds the rows' codes [max_rows, d] followed, from the next 256-byte
 *   boundary after max_rows * d bytes, by their scales [max_rows, d / 32]; the
 *   workspace's h region holds H the same way ([max_rows, F] codes, then scales).
 *   A decode batch, bound by streaming the expert weights, reads half the bytes of
 *   bf16. Needs d % 512 == 0 and F % 512 == 0 and no MOE_FLAG_GATHER_ROWS. Shared
 *   experts and the router stay bf16. ("Mixture of Experts (MoE)"
 *   (learn.starphix.com), "Quantization": lower-precision experts.) */
typedef enum moe_weight_format { MOE_WEIGHTS_DTYPE = 0, MOE_WEIGHTS_MXFP8 = 1 } moe_weight_format;

/* Layer description (plain data, 96 bytes). */
typedef struct moe_config {
  int64_t n_tokens;      /* N: tokens (B*T flattened)                                 */
  int64_t d_model;       /* d                                                         */
  int64_t d_ff;          /* F: routed expert hidden size                              */
  int64_t n_experts;     /* E: routed experts                                         */
  int64_t n_shared;      /* S: always-on shared experts (0 = none)                    */
  int64_t d_ff_shared;   /* Fs: shared expert hidden size                             */
  int64_t top_k;         /* k (expert choice: average experts per token, sets C)      */
  float capacity_factor; /* cf. Token choice: C = ceil(N*k*cf/E), cf <= 0 = no limit.
                            Expert choice: C = min(N, ceil(N*k*cf/E)), cf <= 0 = 1.
                            [AIG] "Expert capacity"; [VAN] CapacityManagedMoE.        */
  int32_t gating;        /* moe_gating                                                */
  int32_t act;           /* moe_act                                                   */
  int32_t dtype;         /* moe_dtype of x, weights, biases, outputs                  */
  int32_t has_bias;      /* GELU experts: b1/b2 (and bs1/bs2) present                 */
  float aux_alpha;       /* alpha of the auxiliary loss ([AIG]: ~0.01)                */
  int32_t flags;         /* MOE_FLAG_* bits                                           */
  int32_t weight_format; /* moe_weight_format of the routed experts' w1, w3, w2       */
  int64_t n_tokens_total; /* token-sharded batch: tokens of the whole batch over all
                            shards (capacity, statistics and kernel shapes follow it);
                            0 or n_tokens: this call holds the whole batch             */
} moe_config;

/* Weights, nn.Linear [out, in] layout, all device pointers of cfg->dtype except
 * logit_bias (fp32) and, with MOE_WEIGHTS_MXFP8, w1 / w3 / w2 (E4M3 codes, 1 byte)
 * and their scales. Unused entries may be NULL. */
typedef struct moe_weights {
  const void* w_router;    /* [E, d]   router, no bias ([AIG], [VAN], [STP])          */
  const float* logit_bias; /* [E] fp32 constant added to every token's logits, or NULL */
  const void* w1;          /* [E, F, d]                                               */
  const void* w3;          /* [E, F, d] SwiGLU only                                   */
  const void* b1;          /* [E, F]   GELU with bias only                            */
  const void* w2;          /* [E, d, F]                                               */
  const void* b2;          /* [E, d]   GELU with bias only                            */
  const void* ws1;         /* [S, Fs, d] shared experts                               */
  const void* ws3;         /* [S, Fs, d] shared, SwiGLU only                          */
  const void* bs1;         /* [S, Fs]  shared, GELU with bias only                    */
  const void* ws2;         /* [S, d, Fs] shared                                       */
  const void* bs2;         /* [S, d]   shared, GELU with bias only                    */
  const uint8_t* w1_scale; /* MOE_WEIGHTS_MXFP8: E8M0 scales of w1 [E, F, d / 32], else NULL */
  const uint8_t* w3_scale; /* ... of w3 [E, F, d / 32] (SwiGLU)                         */
  const uint8_t* w2_scale; /* ... of w2 [E, d, F / 32]                                  */
} moe_weights;

/* Router statistics, written to a caller-owned DEVICE buffer of
 * moe_stats_bytes(E) bytes: this 32-byte header, then float f[E], float P[E],
 * int32 counts[E], int32 kept[E].
 *   f_e   = share of the N*k assignments routed to e before dropping
 *   P_e   = mean over tokens of softmax(L)[t, e]
 *   aux   = alpha * E * sum_e f_e P_e        ([AIG] L_aux; [STP] load_balancing_loss)
 *   z     = (mean_t logsumexp_e L[t, e])^2   ([STP] z_loss)
 *   mean_lse_sq = mean_t logsumexp^2
 *   dropped = assignments over capacity ([AIG] "dropped_share" = dropped/(N*k))
 * moe_route writes aux, z, mean_lse_sq, f, P, counts; moe_permute writes
 * dropped, dropped_share, capacity, rows, kept. */
typedef struct moe_stats_header {
  float aux_loss;
  float z_loss;
  float mean_lse_sq;
  float dropped_share;
  int32_t dropped;
  int32_t capacity;
  int32_t rows; /* R: kept (token, expert) rows */
  int32_t n_experts;
} moe_stats_header;

/* Byte offsets of the intermediate buffers inside a workspace (for callers and
 * tests that want to read them after moe_forward). */
typedef struct moe_workspace_layout {
  size_t total_bytes;
  size_t status;      /* int32[4] sticky device error word                     */
  size_t logits;      /* fp32 [N, E] router logits                              */
  size_t probs;       /* fp32 [N, E] softmax probabilities (expert choice)      */
  size_t idx;         /* int32 token choice [N, k]; expert choice [E, C]        */
  size_t gate;        /* fp32, same shape as idx                                */
  size_t tok_rows;    /* int32 token choice [N, k] (-1 dropped); EC [E*C]       */
  size_t tok_off;     /* int32 [N+1] (expert choice)                            */
  size_t expert_off;  /* int32 [E+1]                                            */
  size_t row_token;   /* int32 [max_rows]                                       */
  size_t row_gate;    /* fp32 [max_rows]                                        */
  size_t xp;          /* dtype [max_rows, d] permuted tokens (empty with
                         MOE_FLAG_GATHER_ROWS; MXFP8 codes + scales with
                         MOE_WEIGHTS_MXFP8)                                      */
  size_t h;           /* dtype [max_rows, F] routed hidden activations (MXFP8
                         codes + scales with MOE_WEIGHTS_MXFP8)                  */
  size_t hs;          /* dtype [N, S*Fs] shared hidden activations              */
  size_t yp;          /* fp32 [max_rows, d] gate-scaled expert outputs          */
  size_t ys;          /* fp32 [N, d] sum of shared expert outputs               */
  size_t stats;       /* moe_stats_bytes(E) used when the caller passes none    */
  size_t stat_acc;    /* router statistic partial sums, moe_stat_acc_bytes(E):
                         uint64 P_sum[E] (fixed point 2^-40), uint64 lse_sum and
                         lse2_sum (2^-32, 2^-24), int32 counts[E] (before dropping) */
  size_t scratch;     /* per-kernel partial sums and tile counts                */
  int64_t max_rows;   /* token choice N*k; expert choice E*C                    */
  int64_t capacity;   /* C (token choice without a limit: N)                    */
} moe_workspace_layout;

/* ABI version of the loaded library (MOE_ABI_VERSION at build time). */
MOE_API int32_t moe_abi_version(void);

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_string(moe_status s);

/* Bytes of the device statistics buffer for E routed experts. */
MOE_API size_t moe_stats_bytes(int64_t n_experts);

/* Bytes of the router's statistic partial sums for E routed experts (the
 * moe_workspace_layout.stat_acc region; see moe_permute_shard). */
MOE_API size_t moe_stat_acc_bytes(int64_t n_experts);

/* Validates cfg (no CUDA call) and returns the workspace size in *bytes. */
MOE_API moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Validates cfg (no CUDA call) and fills *layout. */
MOE_API moe_status moe_workspace_layout_of(const moe_config* cfg, moe_workspace_layout* layout);

/* Zeroes the workspace's device error word (enqueued on stream). Call once on a
 * freshly allocated workspace. */
MOE_API moe_status moe_workspace_init(const moe_config* cfg, void* ws, size_t ws_bytes, void* stream);

/* Router, gates and balancing statistics (hot-path steps: router GEMM, softmax,
 * log-sum-exp, top-k, gates, statistics). [STP] "Key Equations"; [AIG] formula and
 * MoE code; [VAN] TokenChoiceRouter / ExpertChoiceRouter. With a sharded cfg
 * (n_tokens_total > n_tokens) the statistics stay as partial sums in the workspace
 * for the shards' exchange (see moe_permute_shard) and stats is not written.
 *  x      [N, d] dtype
 *  idx    token choice: [N, k] int32 expert ids, rank order (largest logit first).
 *         expert choice: [E, C] int32 token ids, ascending within each expert.
 *  gate   fp32, same shape as idx: the gate of each choice (expert choice: p[t, e]).
 *  logits [N, E] fp32 or NULL; probs [N, E] fp32 softmax or NULL.
 *  stats  moe_stats buffer or NULL. */
MOE_API moe_status moe_route(const moe_config* cfg, const void* x, const moe_weights* w, int32_t* idx,
                     float* gate, float* logits, float* probs, void* stats, void* ws, size_t ws_bytes,
                     void* stream);

/* Capacity, dropping and permutation ([AIG] "Expert capacity" and MoE code's
 * nonzero()[:capacity]; [AIE] "Gather/scatter"). Kept (token, choice) pairs are
 * numbered expert by expert, in token order inside each expert; row r of xp is
 * x[row_token[r]].
 *  x          [N, d] dtype;  idx / gate as written by moe_route.
 *  xp         [max_rows, d] dtype: rows [0, R) written (MOE_WEIGHTS_MXFP8: their E4M3
 *             codes and E8M0 scales, laid out as that format states).
 *  tok_rows   token choice: [N, k] row of each choice or -1 if dropped.
 *             expert choice: [E*C] rows listed token by token (ascending expert id).
 *  tok_off    expert choice: [N+1] start of each token's list in tok_rows
 *             (token choice: may be NULL, unused).
 *  expert_off [E+1] int32 first row of each expert (exclusive prefix of kept counts).
 *  row_token  [max_rows] int32; row_gate [max_rows] fp32 (the row's gate).
 *  stats      moe_stats buffer or NULL (kept/dropped/rows/capacity). */
MOE_API moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* idx, const float* gate, void* xp,
                       int32_t* tok_rows, int32_t* tok_off, int32_t* expert_off, int32_t* row_token,
                       float* row_gate, void* stats, void* ws, size_t ws_bytes, void* stream);

/* Capacity, dropping and permutation of one shard of a token-sharded batch.
 * [AIG] "Expert capacity" and MoE code: every expert keeps the first C of its
 * assignments in token order over the WHOLE batch, so a shard holding tokens
 * [t0, t0 + N) keeps (t, j) exactly when (assignments to e in earlier shards) +
 * (rank of (t, j) among this shard's assignments to e) < C, with C from the whole
 * batch (cfg->n_tokens_total). Token choice only (expert choice ranks every token of
 * the batch for every expert; sharding it would need a candidate exchange).
 * The sharded layer, shard r of n_shards holding a contiguous token range in rank order:
 *   1. moe_route with the sharded cfg: top-k and gates of the shard's tokens; the
 *      statistic partial sums (moe_workspace_layout.stat_acc: P_sum, lse sums,
 *      counts before dropping) stay in the workspace, nothing is finalised;
 *   2. the caller exchanges them (e.g. NCCL): all-gather the int32 counts[E] of every
 *      shard into shard_counts [n_shards][E] (rank order), and all-reduce (sum) the
 *      stat_acc region in place: the E + 2 uint64 words as 64-bit integers (fixed
 *      point, so the sum is exact and independent of the order) and counts[E] as int32;
 *   3. moe_permute_shard (this call): per-expert rank base from shard_counts, this
 *      shard's rows, and the router statistics of the whole batch from the exchanged
 *      sums (f, P, aux, z over n_tokens_total; counts are the batch's); dropped,
 *      rows and kept in stats are this shard's;
 *   4. moe_expert_ffn and moe_combine on the shard's rows, as for a whole batch.
 * Every token's routing, rows and output equal the unsharded batch's bit for bit for any
 * cut. The statistics' partial sums are fp32 sums over router tiles (8, 16 or 32
 * tokens, chosen from n_tokens_total) before the exact fixed-point addition, so they
 * equal the unsharded batch's bit for bit when every shard starts at a multiple of 32
 * tokens, and otherwise to fp32 rounding.
 *  shard_counts  [n_shards][E] int32 device; shard_rank in [0, n_shards).
 *  Other arguments as moe_permute (tok_rows [N, k], no tok_off). */
MOE_API moe_status moe_permute_shard(const moe_config* cfg, const void* x, const int32_t* idx, const float* gate,
                                     const int32_t* shard_counts, int32_t n_shards, int32_t shard_rank, void* xp,
                                     int32_t* tok_rows, int32_t* expert_off, int32_t* row_token, float* row_gate,
                                     void* stats, void* ws, size_t ws_bytes, void* stream);

/* Grouped expert FFNs over the expert-contiguous rows, and the shared experts
 * over all tokens ([VAN] SwiGLUExpert / StandardExpert / HybridMoE;
 * [VAN] "Efficient Batched MoE": one grouped computation instead of a loop).
 *  xp         [max_rows, d] as moe_permute wrote it (MOE_WEIGHTS_MXFP8: codes + scales);
 *             expert_off [E+1] (device; read on the device only).
 *  row_gate   [max_rows] fp32: yp row r = row_gate[r] * E_e(xp[r]).
 *  x          [N, d] (needed when S > 0).
 *  yp         [max_rows, d] fp32: rows [0, R) written (fp32 for every layer dtype,
 *             so the combine rounds the output once).
 *  ys         [N, d] fp32: sum of the shared experts (written when S > 0). */
MOE_API moe_status moe_expert_ffn(const moe_config* cfg, const void* xp, const int32_t* expert_off,
                          const float* row_gate, const void* x, const moe_weights* w, void* yp, void* ys,
                          void* ws, size_t ws_bytes, void* stream);

/* Combine into token order ([AIG] out[index] += w * expert(x); [VAN] HybridMoE):
 * out[t] = ys[t] + sum of yp over the token's rows, in fixed order (token choice:
 * j = 0..k-1 skipping dropped; expert choice: ascending expert id), fp32
 * accumulation and one rounding. Tokens with no kept row get ys[t] (or 0), plus
 * x[t] when cfg->flags has MOE_FLAG_DROP_PASSTHROUGH.
 *  yp [max_rows, d] fp32 and ys [N, d] fp32 (may be NULL) as written by moe_expert_ffn;
 *  tok_rows / tok_off as written by moe_permute. x [N, d] dtype: the layer input,
 *  required with MOE_FLAG_DROP_PASSTHROUGH, else ignored (may be NULL).
 *  out [N, d] dtype. */
MOE_API moe_status moe_combine(const moe_config* cfg, const void* yp, const int32_t* tok_rows, const int32_t* tok_off,
                       const void* ys, const void* x, void* out, void* stream);

/* The whole layer: moe_route -> moe_permute -> moe_expert_ffn -> moe_combine with
 * every intermediate in ws (see moe_workspace_layout_of). out [N, d] dtype.
 * stats: moe_stats buffer or NULL (then written inside ws). No host sync.
 * A sharded cfg (n_tokens_total > n_tokens) is rejected: see moe_permute_shard. */
MOE_API moe_status moe_forward(const moe_config* cfg, const void* x, const moe_weights* w, void* out, void* stats,
                       void* ws, size_t ws_bytes, void* stream);

/* moe_forward with the shared experts on a second stream: their up- and
 * down-projection launches run on side_stream, forked from `stream` by ev_fork and
 * joined back by ev_join before the combine, so they can overlap the routing and the
 * permute, which they do not depend on ("Mixture of Experts (MoE)"
 * (learn.starphix.com), "Communication Optimization": compute the shared experts
 * while the routed tokens are dispatched). side_ctas > 0 caps the side launches' CTAs
 * (one per SM), leaving the other SMs to the main stream; 0 = no cap.
 *  side_stream: a cudaStream_t other than `stream`; ev_fork, ev_join: caller-created
 *  cudaEvent_t (timing may be disabled), recorded by this call. Same results as
 *  moe_forward. fp32 layers and layers without shared experts run as moe_forward. */
MOE_API moe_status moe_forward_overlap(const moe_config* cfg, const void* x, const moe_weights* w, void* out,
                                       void* stats, void* ws, size_t ws_bytes, void* stream, void* side_stream,
                                       void* ev_fork, void* ev_join, int32_t side_ctas);

/* moe_forward that also records caller-created CUDA events (cudaEvent_t) on
 * `stream`: events[0] before the first kernel and events[i] after the i-th
 * stage (route, permute, expert up-projection, expert down-projection,
 * combine); n_events <= 6 are used, extra ones ignored. For timing stages. */
MOE_API moe_status moe_forward_traced(const moe_config* cfg, const void* x, const moe_weights* w, void* out,
                              void* stats, void* ws, size_t ws_bytes, void* stream, void* const* events,
                              int32_t n_events);

/* moe_route without a workspace, for callers that cannot allocate device memory
 * (a plugin handed only its input and output buffers by a framework that owns all
 * device memory through its own pool; a latency-critical caller that must not
 * enter the CUDA allocator, whose cudaMalloc / cudaFree can synchronise the
 * device). The pages have no counterpart: this is a deployment variant of
 * moe_route with the same arguments and results.
 *  - Scratch (an error word and the router's statistic accumulators, 12*E + 16
 *    bytes) is a fixed 4 KiB device array inside the library, held on every device
 *    that runs this call until the process exits. Layers with more than 318
 *    routed experts need more and return MOE_ERR_UNSUPPORTED before anything is
 *    launched.
 *  - All calls on a device share that array and it keeps the last call's
 *    contents: calls that overlap on the GPU race, so serialise them.
 *  - The first call on each device looks up the array's address and keeps it for
 *    the life of the process; make it before any stream capture, and do not use
 *    the library across a cudaDeviceReset (or any other re-creation of the
 *    device's primary context), after which that address is stale.
 *  - stats is required. Layers routed on the tensor cores (bf16, E > 32) need
 *    logits, and expert choice needs probs (the buffers moe_route would otherwise
 *    keep in its workspace); missing ones give MOE_ERR_INVALID_ARG.
 *  - Arguments are checked on the host as for moe_route. Device-side conditions
 *    go to an error word in the same array, cleared at the start of every call:
 *    read it with moe_get_noalloc_status before the next call on the device. */
MOE_API moe_status moe_route_noalloc(const moe_config* cfg, const void* x, const moe_weights* w, int32_t* idx,
                                     float* gate, float* logits, float* probs, void* stats, void* stream);

/* moe_get_device_status for moe_route_noalloc: synchronises `stream`, reads and
 * clears the error word of the current device's no-alloc scratch array (the
 * last moe_route_noalloc call's). *device_error (may be NULL) receives the raw
 * word (0 = none). Returns MOE_OK, or MOE_ERR_DEVICE_CHECK / MOE_ERR_TIMEOUT when
 * a kernel recorded one; MOE_ERR_CUDA if the stream reports an error. */
MOE_API moe_status moe_get_noalloc_status(void* stream, int32_t* device_error);

/* Synchronises `stream`, reads and clears the workspace's device error word.
 * *device_error receives the raw word (0 = none). Returns MOE_OK, or
 * MOE_ERR_DEVICE_CHECK / MOE_ERR_TIMEOUT when a kernel recorded one. */
MOE_API moe_status moe_get_device_status(const moe_config* cfg, void* ws, size_t ws_bytes, void* stream,
                                 int32_t* device_error);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
