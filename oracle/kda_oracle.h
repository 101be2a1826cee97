/*
 * kda_oracle.h -- plain, slow fp64 CPU oracle for the single-token fused KDA
 * (Kimi Delta Attention) decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library and its Python binding) never calls it and shares no code,
 * header, table or helper with it.
 *
 * Source cited throughout as "P1": the web page "[ROCm][Perf] Kimi-K3 Fused
 * kernel for KDA decode" (vLLM PR #50654 report).  Section names are the
 * page's own: 功能与动机 (motivation), 实现拆解 (implementation breakdown),
 * 关键源码片段 (code excerpts), 风险与影响 (risks and impact).
 *
 * ---------------------------------------------------------------------------
 * FORMULATION ADOPTED
 *
 * P1 (功能与动机) names the three stages a decode step runs for every
 * (sequence, value head): causal conv1d state advance, gated delta-rule
 * recurrence, gated RMSNorm.  P1 never writes the equations; the oracle
 * adopts the standard KDA definition, stated here in full.  Notation:
 * K = key head dim, V = value head dim, W = conv width, H = heads,
 * D_q = D_k = H*K, D_v = H*V, C = D_q + D_k + D_v channels.
 *
 * For each row n in [0,N) and head h in [0,H), with s = slot_idx[n]:
 *
 *  0. Padding.  If s <= 0 the row is CUDA-graph padding (P1 实现拆解 #1 and
 *     the kernel excerpt in 关键源码片段): out[n, h*V + j] = 0 for all j and
 *     nothing else is read or written.  If s >= num_slots the oracle does the
 *     same and counts the row as out of range (library contract, not P1).
 *
 *  1. Conv + SiLU.  For block c in {q, k, v} and channel j of head h, global
 *     channel ch = off_c + h*dim_c + j (blocks laid out q | k | v, each
 *     head-major; off_q = 0, off_k = D_q, off_v = D_q + D_k):
 *        x_t = conv_state[s, ch, t]     t = 0 .. W-2   (oldest .. newest)
 *        x_{W-1} = qkv[n, ch]           (the current token)
 *        y = sum_t Wc_c[t, h*dim_c + j] * x_t  (+ bias[ch] if given)
 *        a = y * sigmoid(y)  (SiLU)
 *     If update_conv_state: conv_state[s, ch, :] <- (x_1, ..., x_{W-1}),
 *     the same bf16 bit patterns (a pure shift, never rounded).
 *     The conv state is stored dim-first ("DS", [slots][C][W-1], the kernel's
 *     (..., dim, width-1) view) or, with conv_state_sd, tap-first ("SD",
 *     [slots][W-1][C], channel contiguous), which P1's model layer otherwise
 *     transposes into the dim-first view (关键源码片段, kda.py).  Element
 *     conv_state[s, ch, t] is at s*C*(W-1) + ch*(W-1) + t (DS) or
 *     s*C*(W-1) + t*C + ch (SD); the values are the same either way.
 *
 *  2. L2 norm.  q^ = q_scale * q~ / sqrt(|q~|^2 + l2_eps),
 *               k^ = k~ / sqrt(|k~|^2 + l2_eps),
 *     q_scale = 1/sqrt(K) unless given, l2_eps = 1e-6.  v~ is used as is.
 *
 *  3. Gated delta rule on S = state[s, h] (K x V, S[i][j], i = key channel,
 *     j = value channel, j contiguous):
 *        alpha_i = exp(g[n, h, i])
 *        S' = (I - beta k^ k^T) Diag(alpha) S + beta k^ v~^T
 *     beta = beta[n, h] (bf16, already activated), g already activated.
 *
 *  4. Readout.  o = S'^T q^ (length V).
 *
 *  5. Output.  out_norm on:  out_j = o_j / sqrt(mean_j(o_j^2) + eps)
 *                                     * norm_weight[j] * sigmoid(gate[n, h*V + j])
 *              out_norm off: out_j = o_j
 *
 *  Fused gate (fused_gate = 1; P1 实现拆解 item 1 "safe gate" template flag and
 *  the op's raw_g / raw_beta / A_log / dt_bias / lower_bound arguments in
 *  关键源码片段; P1 does not print the formula, the standard KDA gate is
 *  adopted, parity unpinned by the pages):
 *        z_i = raw_g[n, h, i] + dt_bias[h*K + i]        (dt_bias may be absent)
 *        lower_bound < 0:  g_i = lower_bound * sigmoid(exp(A_log[h]) * z_i)
 *        otherwise:        g_i = -exp(A_log[h]) * softplus(z_i)
 *        beta = sigmoid(raw_beta[n, h])
 *     softplus(z) = log(1 + exp(z)).  These replace the activated g and beta.
 *
 *  6. Rounding.  Every stored input is widened exactly to fp64; all
 *     arithmetic is fp64; out is rounded to bf16 and S' to fp32, both
 *     round-to-nearest-even, and S' is written back to slot s.
 *
 * The choices P1 leaves open (q scale, the two epsilons' placement, the
 * conv-state tap order, the state's index order, norm weight shared across
 * heads, the gate activation, norm-off output) are taken as above.
 * Parity unpinned by the pages: the q scale (1/sqrt(K)) and the L2-norm
 * epsilon's placement have no passage behind them; both sides follow the
 * formulation written here.
 *
 * ---------------------------------------------------------------------------
 * PREFILL (multi-token sequences)
 *
 * Source cited as "P2": the web page "[ROCm][Perf] Kimi-K3 Remove prefill
 * pipeline stall in chunk KDA" (vLLM PR #51862 report).  P2 feeds a varlen
 * batch of sequences (cu_seqlens) to the chunked KDA prefill kernel together
 * with the (sequence, chunk) metadata (实现拆解 #2, #3); it names the
 * kernel's arguments but prints none of its arithmetic.  The chunked form is
 * a way of evaluating the same recurrence, so the oracle is the recurrence
 * itself, token by token:
 *
 * For each sequence b in [0,B) with tokens r = cu_seqlens[b] .. cu_seqlens[b+1]-1
 * (in order) and s = slot_idx[b], and each head h:
 *   - s <= 0: padding sequence, out rows of all its tokens are zero, nothing
 *     else is read or written; s >= num_slots: the same, counted out of range.
 *   - otherwise steps 1-5 above run for every token r in order, with:
 *       * the conv window sliding over the sequence: for its first token the
 *         W-1 older taps come from conv_state[s] (DS layout), after that from
 *         the sequence's own preceding tokens;
 *       * the state carried from token to token in fp64, never rounded in
 *         between (no intermediate state is ever stored);
 *       * at the end, S (rounded to fp32) is stored to slot s and
 *         conv_state[s] holds the last W-1 inputs of the window (the bit
 *         patterns of the newest W-1 taps, which reach back into the old
 *         conv state when the sequence is shorter than W-1).
 *   - an empty sequence (no tokens) leaves everything unchanged.
 * ---------------------------------------------------------------------------
 * MULTI-TOKEN DECODE (speculative decoding)
 *
 * P1 keeps speculative-decode batches off its fused kernel: the support gate
 * requires num_spec == 0 (实现拆解 item 3), the model layer takes the fused
 * path only without a speculative sequence mask and indexes the
 * non-speculative state indices (实现拆解 item 4; kda.py under 关键源码片段),
 * and 风险与影响 lists spec decode as not covered.  P1 gives no formulation;
 * the oracle adopts the plainest one consistent with a per-token state-index
 * table next to the non-speculative one:
 *   - sequence n carries T = 1 + num_spec tokens, rows n*T + t (t = 0..T-1,
 *     in order) of qkv, g, beta, gate and out;
 *   - src_slot[n] holds the sequence's current recurrent state and conv
 *     window; dst_slots[n*T + t] receives the state and the window after
 *     token t;
 *   - src_slot[n] <= 0: padding sequence, its T output rows are zero and
 *     nothing else is read or written; src_slot[n] >= num_slots: the same,
 *     counted out of range;
 *   - dst_slots[n*T + t] <= 0: token t is absent, its output row is zero and
 *     it advances neither the window nor the recurrence; >= num_slots: the
 *     same, counted out of range;
 *   - every present token runs steps 1-5 in order, the window sliding over
 *     the sequence's present tokens (its first W-1 taps from conv_state[src])
 *     and the state carried in fp64 from token to token, never rounded in
 *     between; after token t, S rounded to fp32 is stored to
 *     state[dst_slots[n*T + t]] and, with update_conv_state, the window's
 *     bit patterns to conv_state[dst_slots[n*T + t]];
 *   - the source is read in full before anything is stored, so a destination
 *     may be the sequence's own source slot; apart from that, the slots of
 *     one call are distinct.
 * With T = 1 and dst_slots = src_slot this is the decode step above.
 * ---------------------------------------------------------------------------
 */
#ifndef KDA_ORACLE_H
#define KDA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Whole-step problem.  All pointers are host memory owned by the caller.
 * bf16 tensors are passed as their raw 16-bit patterns. */
typedef struct {
  int32_t N, H, K, V, W, num_slots;
  const uint16_t* qkv;        /* [N][qkv_row_stride], first C used */
  int64_t qkv_row_stride;     /* elements; >= C */
  const float* conv_weight;   /* q block [W][H*K], k block [W][H*K], v block [W][H*V] */
  const float* conv_bias;     /* [C] or NULL */
  uint16_t* conv_state;       /* [num_slots][C][W-1], or [num_slots][W-1][C] if conv_state_sd */
  float* state;               /* [num_slots][H][K][V] */
  const float* g;             /* [N][H][K] log-decay */
  const uint16_t* beta;       /* [N][H] */
  const uint16_t* gate;       /* [N][H*V]; ignored when out_norm == 0 */
  const float* norm_weight;   /* [V]; ignored when out_norm == 0 */
  const int32_t* slot_idx;    /* [N] */
  uint16_t* out;              /* [N][H*V] */
  double* out_f64;            /* optional [N][H*V]: out before bf16 rounding */
  double eps;                 /* RMSNorm epsilon */
  double l2_eps;              /* L2-norm epsilon */
  double q_scale;             /* 0 => 1/sqrt(K) */
  int32_t out_norm;           /* 1: gated RMSNorm epilogue, 0: raw o */
  int32_t update_conv_state;  /* 1: write the shifted conv state */
  int32_t fused_gate;         /* 1: g and beta hold raw logits (see "Fused gate") */
  const float* A_log;         /* [H]; fused_gate only */
  const float* dt_bias;       /* [H*K] or NULL; fused_gate only */
  double lower_bound;         /* < 0: bounded ("safe") gate; fused_gate only */
  int32_t conv_state_sd;      /* 1: conv_state is [num_slots][W-1][C] (tap-first) */
} kda_oracle_problem;

/* Runs one decode step over every (row, head).  num_threads <= 0 uses the
 * OpenMP default.  Returns the number of rows whose slot was >= num_slots
 * (they are zeroed like padding), or -1 on a bad argument. */
int kda_oracle_decode(const kda_oracle_problem* p, int num_threads);

/* Size of kda_oracle_problem, so a foreign-function caller can check that its
 * mirror of the struct matches. */
int kda_oracle_problem_size(void);

/* Varlen prefill problem (see PREFILL above).  Host memory, caller-owned. */
typedef struct {
  int32_t B, H, K, V, W, num_slots;
  const int32_t* cu_seqlens;  /* [B+1], non-decreasing, cu_seqlens[0] = 0 */
  const uint16_t* qkv;        /* [T][qkv_row_stride] */
  int64_t qkv_row_stride;
  const float* conv_weight;   /* as kda_oracle_problem */
  const float* conv_bias;     /* [C] or NULL */
  uint16_t* conv_state;       /* [num_slots][C][W-1] (DS), or [num_slots][W-1][C] if conv_state_sd */
  float* state;               /* [num_slots][H][K][V] */
  const float* g;             /* [T][H][K] */
  const uint16_t* beta;       /* [T][H] */
  const uint16_t* gate;       /* [T][H*V]; ignored when out_norm == 0 */
  const float* norm_weight;   /* [V]; ignored when out_norm == 0 */
  const int32_t* slot_idx;    /* [B] */
  uint16_t* out;              /* [T][H*V] */
  double* out_f64;            /* optional [T][H*V] */
  double eps, l2_eps, q_scale;
  int32_t out_norm;
  int32_t fused_gate;         /* 1: g and beta hold raw logits (see "Fused gate") */
  const float* A_log;         /* [H]; fused_gate only */
  const float* dt_bias;       /* [H*K] or NULL; fused_gate only */
  double lower_bound;         /* < 0: bounded gate; fused_gate only */
  int32_t conv_state_sd;      /* 1: conv_state is [num_slots][W-1][C] (tap-first) */
} kda_oracle_prefill_problem;

/* Runs the prefill of every sequence.  Returns the number of sequences whose
 * slot was >= num_slots, or -1 on a bad argument. */
int kda_oracle_prefill(const kda_oracle_prefill_problem* p, int num_threads);
int kda_oracle_prefill_problem_size(void);

/* Multi-token decode problem (see MULTI-TOKEN DECODE above).  Host memory,
 * caller-owned. */
typedef struct {
  int32_t N, T, H, K, V, W, num_slots;
  const int32_t* src_slot;    /* [N] */
  const int32_t* dst_slots;   /* [N][T] */
  const uint16_t* qkv;        /* [N*T][qkv_row_stride] */
  int64_t qkv_row_stride;
  const float* conv_weight;   /* as kda_oracle_problem */
  const float* conv_bias;     /* [C] or NULL */
  uint16_t* conv_state;       /* [num_slots][C][W-1] (DS), or [num_slots][W-1][C] if conv_state_sd */
  float* state;               /* [num_slots][H][K][V] */
  const float* g;             /* [N*T][H][K] */
  const uint16_t* beta;       /* [N*T][H] */
  const uint16_t* gate;       /* [N*T][H*V]; ignored when out_norm == 0 */
  const float* norm_weight;   /* [V]; ignored when out_norm == 0 */
  uint16_t* out;              /* [N*T][H*V] */
  double* out_f64;            /* optional [N*T][H*V] */
  double eps, l2_eps, q_scale;
  int32_t out_norm;
  int32_t update_conv_state;
  int32_t fused_gate;
  const float* A_log;
  const float* dt_bias;
  double lower_bound;
  int32_t conv_state_sd;
} kda_oracle_multi_problem;

/* Runs the multi-token decode of every sequence.  Returns the number of
 * out-of-range slot entries met (a source slot, or a destination slot of a
 * sequence whose source is in range), or -1 on a bad argument. */
int kda_oracle_decode_multi(const kda_oracle_multi_problem* p, int num_threads);
int kda_oracle_multi_problem_size(void);

/* ---- the individual steps, fp64, exposed for the fact tests ---- */

/* sigmoid(x) = 1 / (1 + exp(-x)). */
double kda_oracle_sigmoid(double x);

/* Step 1: y = sum_t w[t] * x[t] + bias over a window x[0..W-1], oldest first,
 * x[W-1] the current input; returns y (before SiLU). */
double kda_oracle_causal_conv(const double* x, const double* w, int W, double bias);

/* SiLU(y) = y * sigmoid(y). */
double kda_oracle_silu(double y);

/* Step 2: y = scale * x / sqrt(sum x^2 + eps), length n. */
void kda_oracle_l2norm(const double* x, int n, double eps, double scale, double* y);

/* Step 3: S (K x V, row-major, in place) <- (I - beta k k^T) Diag(alpha) S + beta k v^T. */
void kda_oracle_gated_delta_update(int K, int V, double* S, const double* alpha,
                                   double beta, const double* k, const double* v);

/* Step 4: o = S^T q, S K x V row-major. */
void kda_oracle_readout(int K, int V, const double* S, const double* q, double* o);

/* Step 5: y_j = o_j / sqrt(mean(o^2) + eps) * w_j * sigmoid(gate_j). */
void kda_oracle_gated_rmsnorm(int V, const double* o, const double* w,
                              const double* gate, double eps, double* y);

/* softplus(z) = log(1 + exp(z)). */
double kda_oracle_softplus(double z);

/* Fused gate: g from z = raw + bias (see "Fused gate" above). */
double kda_oracle_kda_gate(double z, double A_log, double lower_bound);

/* Round to bf16, nearest-even, directly from fp64; returns the bit pattern. */
uint16_t kda_oracle_round_bf16(double x);

/* Exact widening of a bf16 bit pattern. */
double kda_oracle_bf16_to_f64(uint16_t b);

#ifdef __cplusplus
}
#endif

#endif /* KDA_ORACLE_H */
