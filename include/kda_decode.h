/*
 * kda_decode.h -- C ABI of the GB300 (sm_103a) fused KDA decode step.
 *
 * One call runs, for every (token row n, value head h) of a decode batch, the
 * three stages that the page "[ROCm][Perf] Kimi-K3 Fused kernel for KDA
 * decode" (vLLM PR #50654 report; cited below as P1) fuses into one launch
 * (P1, section 功能与动机 "motivation" and 实现拆解 "implementation
 * breakdown" item 1):
 *
 *   1. causal conv1d state advance (width 4) + SiLU on the q, k, v channels;
 *   2. gated delta-rule recurrence on the [128, 128] fp32 state:
 *        q^ = q_scale * q / sqrt(|q|^2 + 1e-6),  k^ = k / sqrt(|k|^2 + 1e-6)
 *        S' = (I - beta k^ k^T) Diag(exp(g)) S + beta k^ v^T,  o = S'^T q^
 *   3. gated RMSNorm: out = o / sqrt(mean(o^2) + eps) * norm_weight * sigmoid(gate),
 *      or out = o when KDA_OUT_NORM is not set.
 *
 * P1 does not print the equations; the standard KDA definition above is the
 * one adopted.  Rows whose slot index is <= 0 are CUDA-graph padding: their
 * output is zero and no state is read or written (P1 实现拆解 item 1 and the
 * kernel excerpt under 关键源码片段 "code excerpts").
 *
 * Memory: every pointer is memory owned by the caller that the device current
 * when kda_decode is called can address: device memory, or (for the
 * per-token tensors qkv, g, beta, gate, slot_idx and out) pinned host memory
 * mapped into the device's address space, which the kernel then reads and
 * writes directly over the CPU-GPU link.  The library never allocates, frees,
 * synchronises or reads device memory from the host, so a call may be
 * captured into a CUDA graph (after one eager call on that device, which
 * performs the once-per-device kernel attribute set-up).
 */
#ifndef KDA_DECODE_H
#define KDA_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_DECODE_ABI_VERSION 2

/* Fixed problem geometry (P1 实现拆解 item 3: head_dim 128, conv width 4). */
#define KDA_HEAD_DIM 128
#define KDA_CONV_WIDTH 4
/* Largest tokens_per_seq of a multi-token (speculative) call: 1 + num_spec. */
#define KDA_MAX_TOKENS_PER_SEQ 8

/* flags */
#define KDA_OUT_NORM          1u /* apply the gated RMSNorm epilogue */
#define KDA_UPDATE_CONV_STATE 2u /* write the advanced conv state back */
/* The caller guarantees that the kernel enqueued immediately before this call
 * on the stream writes none of slot_idx, state or conv_state (for example the
 * previous layer's decode, with its own pools).  The call may then start
 * streaming state and conv state while that kernel is still running; all
 * per-token inputs (qkv, g, beta, gate) are still read only after it has
 * completed.  Without this flag nothing is read before it completes. */
#define KDA_EARLY_PREFETCH    4u /* (with src_slot: it too is not written by that kernel) */
/* g and beta hold raw logits and the kernel activates them (the page's
 * "safe gate" variant; formula below, in KdaDecodeArgs.lower_bound). */
#define KDA_FUSED_GATE        8u
/* conv_state is stored tap-first, [num_slots][3][C] with the channel index
 * contiguous (P1 关键源码片段, kda.py: the "SD" layout its model layer would
 * otherwise transpose into the kernel's dim-first view). */
#define KDA_CONV_STATE_SD    16u

/* return codes of kda_decode */
#define KDA_OK            0
#define KDA_ERR_NULLPTR  -1 /* a required pointer is NULL */
#define KDA_ERR_SHAPE    -2 /* head_dim != 128, conv_width != 4, N < 0, H < 1,
                               num_slots < 1, a stride too small, N*H too large, or
                               tokens_per_seq outside 0 .. KDA_MAX_TOKENS_PER_SEQ */
#define KDA_ERR_ALIGN    -3 /* a pointer or row stride breaks the 16-byte rule */
#define KDA_ERR_FLAGS    -4 /* unknown flag bits */
#define KDA_ERR_LAUNCH   -5 /* the CUDA launch failed; see kda_last_error() */
#define KDA_ERR_ABI      -6 /* args->struct_size does not match this library */

/* bits OR-ed into *err_flag by the kernel (never a trap) */
#define KDA_DEVERR_SLOT_RANGE 1 /* a row had slot >= num_slots; its output was zeroed */
#define KDA_DEVERR_TIMEOUT    2 /* an internal pipeline wait gave up after 2 s; the launch
                                   stopped early and its results are incomplete */

/*
 * Arguments.  Shapes use N = rows (tokens), H = heads, D = H * 128,
 * C = 3 * D (q | k | v channel blocks, each head-major).  bf16 tensors are
 * passed as their 16-bit patterns (uint16_t).
 *
 * Alignment: every pointer except beta, slot_idx, err_flag, A_log and dt_bias must be
 * 16-byte aligned, and every row stride must be a multiple of 8 elements.
 */
typedef struct KdaDecodeArgs {
  uint32_t struct_size;        /* = sizeof(KdaDecodeArgs) */
  int32_t N;                   /* rows; 0 is a no-op */
  int32_t H;                   /* value heads (= key heads) */
  int32_t num_slots;           /* state-pool entries; slot 0 is the padding slot */
  int32_t head_dim;            /* must be 128 */
  int32_t conv_width;          /* must be 4 */

  const uint16_t* qkv;         /* bf16 [N][qkv_row_stride], channels [0, C) used */
  int64_t qkv_row_stride;      /* elements, >= C */
  const float* conv_weight;    /* fp32 [3][4][D], width-major, channel contiguous
                                  (P1 实现拆解 item 3) */
  const float* conv_bias;      /* fp32 [C] or NULL */
  uint16_t* conv_state;        /* bf16 [num_slots][C][3] (dim-first, oldest tap first),
                                  or [num_slots][3][C] with KDA_CONV_STATE_SD;
                                  read, and rewritten in place if KDA_UPDATE_CONV_STATE */
  float* state;                /* fp32 [num_slots][H][128][128], S[key][value],
                                  value index contiguous; read and rewritten in place */
  const float* g;              /* fp32 [N][H][128] log-decay, alpha = exp(g) */
  const uint16_t* beta;        /* bf16 [N][H] write strength, already activated */
  const uint16_t* gate;        /* bf16 [N][gate_row_stride], D used; KDA_OUT_NORM only */
  int64_t gate_row_stride;     /* elements, >= D (ignored without KDA_OUT_NORM) */
  const float* norm_weight;    /* fp32 [128], shared by all heads; KDA_OUT_NORM only */
  const int32_t* slot_idx;     /* int32 [N]; <= 0 marks a padding row.  Positive
                                  slots must be distinct within one call. */
  uint16_t* out;               /* bf16 [N][out_row_stride], D written per row */
  int64_t out_row_stride;      /* elements, >= D */
  float eps;                   /* RMSNorm epsilon (e.g. 1e-6) */
  float q_scale;               /* 0 => 1/sqrt(128) */
  uint32_t flags;              /* KDA_OUT_NORM | KDA_UPDATE_CONV_STATE | KDA_EARLY_PREFETCH |
                                  KDA_FUSED_GATE | KDA_CONV_STATE_SD */
  int32_t* err_flag;           /* device int32 or NULL; KDA_DEVERR_* bits are OR-ed in */

  /* KDA_FUSED_GATE only (P1 关键源码片段: the op's A_log, dt_bias, lower_bound;
   * the formula is the standard KDA gate, not printed on P1).  With
   * z = g[n][h][i] + dt_bias[h*128 + i] (raw logits plus bias):
   *   lower_bound < 0:  g' = lower_bound * sigmoid(exp(A_log[h]) * z)
   *   otherwise:        g' = -exp(A_log[h]) * softplus(z)
   * and beta' = sigmoid(beta[n][h]); alpha = exp(g').  Scalar loads only, so
   * these two pointers need 4-byte alignment. */
  const float* A_log;          /* fp32 [H] */
  const float* dt_bias;        /* fp32 [H*128] or NULL */
  float lower_bound;

  /* Optional work queue: device int32[2], zero before the call; every call
   * leaves it zero again.  With it, units beyond each CTA's first few are
   * handed out dynamically so that all SMs finish together; NULL keeps a
   * static round-robin schedule.  Calls that may overlap on the GPU (for
   * example on different streams) need different queues; calls ordered on
   * one stream may share one.  4-byte alignment. */
  int32_t* work_queue;

  /* Multi-token (speculative) decode.  P1 keeps speculative batches off its
   * fused kernel (实现拆解 items 3-4: the support gate wants num_spec == 0 and
   * the model layer indexes the non-speculative state indices; 风险与影响:
   * spec decode not covered) and gives no formulation; this library adopts
   * the one below.  It is selected by tokens_per_seq >= 2 or by a non-NULL
   * src_slot.  Then N counts sequences, and sequence n carries
   * T = max(tokens_per_seq, 1) tokens, rows n*T + t (t = 0 .. T-1, in order)
   * of qkv, g, beta, gate and out (so those tensors have N*T rows), and
   * slot_idx is int32 [N][T]:
   *   - the sequence starts from the recurrent state and conv window of
   *     src_slot[n] (slot_idx[n*T] when src_slot is NULL);
   *   - after token t its state and window are stored to slot_idx[n*T + t]
   *     (the window only with KDA_UPDATE_CONV_STATE); the state is carried
   *     on chip from token to token;
   *   - a source slot <= 0 marks a padding sequence: its T output rows are
   *     zero and nothing else is read or written;
   *   - a destination slot <= 0 marks an absent token: its output row is
   *     zero and it advances neither the state nor the window;
   *   - slots >= num_slots are treated as padding / absent and raise
   *     KDA_DEVERR_SLOT_RANGE;
   *   - the source is read in full before anything is stored, so a
   *     destination may equal its own sequence's source; apart from that all
   *     slots of a call must be distinct.
   * With tokens_per_seq <= 1 and src_slot NULL a call is the single-token
   * step above (one row per sequence, slot_idx both source and destination). */
  int32_t tokens_per_seq;      /* 0 or 1: single-token step; 2 .. KDA_MAX_TOKENS_PER_SEQ */
  const int32_t* src_slot;     /* int32 [N] or NULL; 4-byte alignment */
} KdaDecodeArgs;

/*
 * Enqueue one fused decode step on `stream` (a cudaStream_t; NULL = the
 * legacy default stream).  The launch is a programmatic dependent launch:
 * it may become resident while the previous kernel on the stream drains and
 * waits for that kernel's completion before reading anything it could have
 * written (see KDA_EARLY_PREFETCH for the one exception the caller can allow).  Returns KDA_OK or a negative KDA_ERR_* code; on an
 * argument error nothing is launched.  Asynchronous: results are visible
 * after the stream reaches this point.  Rows with slot >= num_slots are
 * treated as padding and raise KDA_DEVERR_SLOT_RANGE in *err_flag.
 * Duplicate positive slots within one call give undefined state.
 */
int kda_decode(const KdaDecodeArgs* args, void* stream);

/*
 * Test hook for the bounded-wait path (no counterpart on the page; it exists
 * so that the failure handling can be exercised without faulting a GPU).
 * Same as kda_decode, except that every internal pipeline wait gives up after
 * `wait_limit_ns` (> 0) instead of 2 s, and the inputs of unit
 * `withhold_unit` (= row * H + head; -1 for none) are never signalled as
 * loaded, so the waits that depend on them run out.  The kernel then sets
 * KDA_DEVERR_TIMEOUT in *err_flag, stops early and returns; the context stays
 * usable.  Results of such a launch are incomplete.
 */
int kda_decode_wait_test(const KdaDecodeArgs* args, void* stream, uint64_t wait_limit_ns,
                         int32_t withhold_unit);

/*
 * kda_decode_noalloc: the same decode step for callers that cannot allocate
 * device memory (no counterpart on the page; it exists for integration).
 * Plugin interfaces whose enqueue step must not allocate, serving loops with
 * a device-memory budget fixed at start-up, and callers that reach the
 * library only through this C ABI and hold no device allocator cannot hand
 * the kernel a work queue of their own.  This entry point runs the dynamic
 * schedule with the queue kept in a file-scope device array of 256 bytes
 * inside the library (every GPU that loads the library holds it until the
 * process exits).  One call uses 8 bytes of it, a fixed need whatever N and
 * H, checked against the array's size when the library is compiled.
 * args->work_queue is ignored.  The caller still passes all inputs and
 * outputs.  It allocates nothing: it calls no cudaMalloc, cudaFree or
 * allocating library routine.
 *
 * Every argument is checked first, with the codes of kda_decode; on an error
 * nothing is enqueued.  Then the call clears the queue with an asynchronous
 * memset on `stream` and launches as kda_decode.  Every call shares the one
 * array: calls that overlap on the GPU (other streams, other host threads)
 * race on it and give wrong results; calls ordered on one stream are safe.
 * The first call on a device looks up the array's device address (and does
 * kda_decode's once-per-device set-up); make that first call before any
 * stream capture on that device.  The looked-up address is kept for the life
 * of the process: the library assumes the device's primary context is never
 * reset (no cudaDeviceReset) while it is loaded.
 */
int kda_decode_noalloc(const KdaDecodeArgs* args, void* stream);

/* Static text for a KDA_* return code. */
const char* kda_status_string(int status);

/* Detail of the last failing call on the calling host thread ("" if none). */
const char* kda_last_error(void);

/* KDA_DECODE_ABI_VERSION of the loaded library. */
int kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_DECODE_H */
