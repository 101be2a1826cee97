/*
 * kda_prefill.h -- C ABI of the GB300 (sm_103a) chunked KDA prefill over a
 * varlen batch of sequences.
 *
 * Source: the page "[ROCm][Perf] Kimi-K3 Remove prefill pipeline stall in
 * chunk KDA" (vLLM PR #51862 report; "P2"), section 实现拆解 (implementation
 * breakdown) items 2-3: prefill runs the KDA layer over whole sequences of a
 * varlen batch (cumulative starts `cu_seqlens`) with a chunked kernel.  P2
 * names the kernel's arguments but prints none of its arithmetic; the
 * chunked evaluation is a way of computing the same recurrence as the decode
 * step applied token by token, which is what this call computes:
 *
 * For sequence b with tokens r = cu_seqlens[b] .. cu_seqlens[b+1]-1 (in
 * order), slot s = slot_idx[b], and every head h:
 *   - s <= 0: padding sequence; its output rows (head h) are zero and nothing
 *     else is read or written.  s >= num_slots: the same, and
 *     KDA_DEVERR_SLOT_RANGE is set.
 *   - otherwise, per token: width-4 causal conv + SiLU of the q, k, v channels
 *     (the window's three older taps come from conv_state[s] for the first
 *     token, then from the sequence itself); q^ = q_scale q / sqrt(|q|^2 +
 *     1e-6), k^ = k / sqrt(|k|^2 + 1e-6);
 *       S <- (I - beta k^ k^T) Diag(exp(g)) S + beta k^ v^T,  o = S^T q^;
 *     out = o / sqrt(mean(o^2) + eps) * norm_weight * sigmoid(gate) with
 *     KDA_OUT_NORM, else out = o.  At the end S is stored to state[s, h] and
 *     conv_state[s] holds the last three inputs of the window (the conv state
 *     is always advanced).
 *   - an empty sequence leaves everything unchanged.
 * This is the definition in the decode header (kda_decode.h) applied to a
 * sequence; the state between tokens is never stored, so it is not rounded.
 *
 * Method (device side): one CTA per (sequence, head) walks the sequence in
 * chunks of 32 tokens.  Within a chunk the recurrence is solved in closed
 * form (cumulative decays, a lower-triangular solve for the chunk's deltas);
 * the contractions with the state and between tokens run on the tensor cores
 * (tf32 operands split into high and low parts, three products per
 * contraction, fp32 accumulation), the state stays in registers for the whole
 * sequence.
 *
 * Memory: all pointers are caller-owned device memory; the library allocates,
 * frees and synchronises nothing and reads no device memory from the host, so
 * a call can be captured into a CUDA graph.
 */
#ifndef KDA_PREFILL_H
#define KDA_PREFILL_H

#include <stddef.h>
#include <stdint.h>

#include "kda_chunk_metadata.h" /* KDA_DEVERR_SEQLENS */
#include "kda_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

/* chunk length of the device algorithm (tokens) */
#define KDA_PREFILL_CHUNK 32

/*
 * Arguments.  B = sequences, T = token rows of the batch, H = heads,
 * D = H * 128, C = 3 * D.  bf16 tensors are passed as 16-bit words.
 *
 *   qkv          bf16 [T][qkv_row_stride], channels q | k | v (each H*128,
 *                head-major); row stride >= C, a multiple of 8 elements
 *   conv_weight  fp32 [3][4][D] (block, tap oldest..current, channel)
 *   conv_bias    fp32 [C] or NULL
 *   conv_state   bf16 [num_slots][C][3], oldest tap first (dim-first)
 *   state        fp32 [num_slots][H][128][128], S[key][value], value contiguous
 *   g            fp32 [T][H][128] log-decay, already activated (alpha = exp(g))
 *   beta         bf16 [T][H], already activated
 *   gate         bf16 [T][gate_row_stride] (KDA_OUT_NORM only; stride >= D,
 *                a multiple of 8)
 *   norm_weight  fp32 [128] (KDA_OUT_NORM only)
 *   cu_seqlens   int32 [B+1] on the device: cu_seqlens[0] = 0, non-decreasing,
 *                cu_seqlens[B] <= T.  A sequence whose bounds break this is
 *                skipped and KDA_DEVERR_SEQLENS is set.
 *   slot_idx     int32 [B] (one slot per sequence, distinct among the active
 *                sequences of a call)
 *   out          bf16 [T][out_row_stride] (stride >= D, a multiple of 4);
 *                rows outside every sequence are not written
 *   err_flag     int32 or NULL: device-side error bits (KDA_DEVERR_*)
 *
 * Alignment: state, g and norm_weight 16 bytes; qkv, gate, out 16 / 16 / 8
 * bytes with row strides as stated; cu_seqlens, slot_idx, err_flag 4 bytes.
 */
typedef struct KdaPrefillArgs {
  size_t struct_size; /* sizeof(KdaPrefillArgs) */
  int32_t B, H, num_slots, head_dim, conv_width;
  int64_t T;
  const int32_t* cu_seqlens;
  const uint16_t* qkv;
  int64_t qkv_row_stride;
  const float* conv_weight;
  const float* conv_bias;
  uint16_t* conv_state;
  float* state;
  const float* g;
  const uint16_t* beta;
  const uint16_t* gate;
  int64_t gate_row_stride;
  const float* norm_weight;
  const int32_t* slot_idx;
  uint16_t* out;
  int64_t out_row_stride;
  float eps;     /* RMSNorm epsilon */
  float q_scale; /* 0 => 1/sqrt(128) */
  uint32_t flags; /* KDA_OUT_NORM or 0; other bits are rejected */
  int32_t* err_flag;
} KdaPrefillArgs;

/*
 * Enqueue the prefill on `stream` (a cudaStream_t; NULL = legacy default).
 * Returns KDA_OK or a negative KDA_ERR_* code of kda_decode.h; on an error
 * nothing is launched and kda_last_error() describes it.  B == 0 or T == 0
 * is a no-op.
 */
int kda_prefill(const KdaPrefillArgs* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_PREFILL_H */
