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
 * Method (device side), two kernels per call:
 *   1. chunk-parallel: one CTA per (chunk, head), the chunks taken from the
 *      (sequence, chunk) metadata of kda_chunk_metadata.h (P2 实现拆解 item
 *      2) built with chunk size KDA_PREFILL_CHUNK.  Each CTA does the work of
 *      its chunk that does not depend on the state entering it (conv, norms,
 *      cumulative decays, the chunk's lower-triangular solve) and writes it
 *      to the workspace;
 *   2. scan: one CTA per (sequence, head) walks that sequence's chunks in
 *      order (its rows in the workspace start at chunk_offsets[b]) with the
 *      state held in tensor memory, and applies each chunk to the state and
 *      the outputs.  The CTAs take the sequences in the order seq_order
 *      gives (longest first balances ragged batches), else in index order.
 * The contractions with the state and between tokens run on the tensor cores
 * (tf32 operands split into high and low parts, three products per
 * contraction, fp32 accumulation).
 *
 * Memory: every pointer of KdaPrefillArgs is caller-owned device memory; the
 * library allocates, frees and synchronises nothing and reads no device
 * memory from the host, so a kda_prefill call can be captured into a CUDA
 * graph.  kda_prefill_longest_first works on host memory only.
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
 *   conv_state   bf16 [num_slots][C][3], oldest tap first (dim-first), or
 *                [num_slots][3][C] with KDA_CONV_STATE_SD (tap-first)
 *   state        fp32 [num_slots][H][128][128], S[key][value], value contiguous
 *   g            fp32 [T][H][128] log-decay, already activated (alpha = exp(g)),
 *                or raw logits with KDA_FUSED_GATE
 *   beta         bf16 [T][H], already activated, or raw with KDA_FUSED_GATE
 *   gate         bf16 [T][gate_row_stride] (KDA_OUT_NORM only; stride >= D,
 *                a multiple of 4)
 *   norm_weight  fp32 [128] (KDA_OUT_NORM only)
 *   cu_seqlens   int32 [B+1] on the device: cu_seqlens[0] = 0, non-decreasing,
 *                cu_seqlens[B] <= T.  A sequence whose bounds break this is
 *                skipped and KDA_DEVERR_SEQLENS is set.
 *   slot_idx     int32 [B] (one slot per sequence, distinct among the active
 *                sequences of a call)
 *   out          bf16 [T][out_row_stride] (stride >= D, a multiple of 4);
 *                rows outside every sequence are not written
 *   chunk_indices int32 [num_chunks][2] and chunk_offsets int64 [B+1]: the
 *                output of kda_chunk_metadata(cu_seqlens, B, KDA_PREFILL_CHUNK,
 *                ...) for this batch (enqueued before this call on the same
 *                stream); num_chunks is their row count, known on the host
 *                from the sequence lengths.  If chunk_offsets does not match
 *                cu_seqlens, the sequence is skipped and KDA_DEVERR_SEQLENS set.
 *   workspace    device scratch of workspace_bytes >=
 *                kda_prefill_workspace_bytes(num_chunks, H) bytes
 *   err_flag     int32 or NULL: device-side error bits (KDA_DEVERR_*)
 *
 * Alignment: state, g, norm_weight and workspace 16 bytes; qkv 16 bytes with
 * a row stride that is a multiple of 8 elements; gate and out 8 bytes with row
 * strides that are multiples of 4; chunk_indices and chunk_offsets 8 bytes;
 * cu_seqlens, slot_idx, seq_order, err_flag 4 bytes.
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
  uint32_t flags; /* KDA_OUT_NORM, KDA_FUSED_GATE, KDA_CONV_STATE_SD; other bits are rejected */
  int32_t* err_flag;
  const int32_t* chunk_indices;
  const int64_t* chunk_offsets;
  int64_t num_chunks;
  void* workspace;
  int64_t workspace_bytes;
  /* KDA_FUSED_GATE only (as in KdaDecodeArgs): g and beta hold raw logits;
   * A_log fp32 [H], dt_bias fp32 [H*128] or NULL, lower_bound < 0 selects the
   * bounded gate.  P2's prefill kernel is this variant
   * (chunk_kda_with_fused_gate, 实现拆解 item 3). */
  const float* A_log;
  const float* dt_bias;
  float lower_bound;
  /* int32 [B] on the device, or NULL for index order: the order in which the
   * scan kernel's CTAs take the sequences, a permutation of 0 .. B-1.  The
   * scan runs one CTA per (sequence, head) and a sequence's chunks one after
   * another, so with ragged lengths the longest sequences should start first
   * (kda_prefill_longest_first builds that order on the host).  The order
   * changes no result: every (sequence, head) is computed the same way
   * wherever it runs.  An entry outside [0, B) sets KDA_DEVERR_ORDER and its
   * CTAs do nothing; a repeated entry is a caller error (undefined results,
   * as for repeated slots). */
  const int32_t* seq_order;
} KdaPrefillArgs;

/* bit OR-ed into *err_flag (the KDA_DEVERR_* space of kda_decode.h) */
#define KDA_DEVERR_ORDER 16 /* seq_order held an entry outside [0, B); those CTAs did nothing */

/* Host helper: fill order[0 .. B-1] (host memory) with the sequence indices
 * sorted by length, longest first, equal lengths in index order, from the
 * host copy of cu_seqlens [B+1] (a negative length counts as 0).  Returns
 * KDA_OK, KDA_ERR_NULLPTR (a NULL pointer with B > 0) or KDA_ERR_SHAPE
 * (B < 0). */
int kda_prefill_longest_first(const int32_t* cu_seqlens, int32_t B, int32_t* order);

/* Workspace bytes a call with `num_chunks` chunks and H heads needs (about
 * 84.5 KiB, 86,528 bytes, per (chunk, head)); -1 for a negative count or H < 1. */
int64_t kda_prefill_workspace_bytes(int64_t num_chunks, int32_t H);

/*
 * Enqueue the prefill on `stream` (a cudaStream_t; NULL = legacy default).
 * Returns KDA_OK or a negative KDA_ERR_* code of kda_decode.h; on an error
 * nothing is launched and kda_last_error() describes it.  B == 0 or T == 0
 * is a no-op.  The chunk kernel reads the slots' old conv state; the scan
 * kernel, which runs after it, writes the new one.
 */
int kda_prefill(const KdaPrefillArgs* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_PREFILL_H */
