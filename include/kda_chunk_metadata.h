/*
 * kda_chunk_metadata.h -- C ABI of the device-side chunk metadata used by
 * chunked prefill of KDA layers.
 *
 * Source: the page "[ROCm][Perf] Kimi-K3 Remove prefill pipeline stall in
 * chunk KDA" (vLLM PR #51862 report), section 实现拆解 (implementation
 * breakdown) item 2: the (sequence, chunk) index pairs and per-sequence
 * chunk offsets are built on the GPU straight from the cumulative sequence
 * starts, so the host never waits for the device (the stall that page
 * removes came from a device-to-host read of those starts).
 *
 * Definition, for N sequences with starts cu_seqlens[0..N] (cu_seqlens[0] =
 * 0, non-decreasing) and chunk size BT:
 *   n_i              = ceil((cu_seqlens[i+1] - cu_seqlens[i]) / BT)
 *   chunk_offsets[i] = n_0 + ... + n_{i-1}      for i = 0 .. N
 *   chunk_indices    = rows (i, c) for c = 0 .. n_i - 1, i = 0 .. N-1, in
 *                      that order, as int32 pairs [total][2]
 */
#ifndef KDA_CHUNK_METADATA_H
#define KDA_CHUNK_METADATA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* bits OR-ed into *err_flag (the KDA_DEVERR_* space of kda_decode.h) */
#define KDA_DEVERR_SEQLENS   4 /* cu_seqlens decreased somewhere; that sequence got 0 chunks */
#define KDA_DEVERR_CAPACITY  8 /* more chunks than `capacity`; rows past it were not written */

/*
 * Enqueue the metadata build on `stream` (a cudaStream_t).  All pointers are
 * caller-owned device memory:
 *   cu_seqlens     int32 [num_seqs + 1], 4-byte aligned
 *   chunk_indices  int32 [capacity][2], 8-byte aligned (may be NULL if capacity == 0)
 *   chunk_offsets  int64 [num_seqs + 1], 8-byte aligned
 *   err_flag       int32 or NULL
 * The caller sizes `capacity` from its host copy of the sequence lengths (no
 * device read is needed).  Returns 0 or a negative KDA_ERR_* code of
 * kda_decode.h (nothing is launched on an argument error).  One CTA of 1024
 * threads does a block-wide scan over the sequences and then expands the
 * rows; it allocates and synchronises nothing.
 */
int kda_chunk_metadata(const int32_t* cu_seqlens, int32_t num_seqs, int32_t chunk_size,
                       int32_t* chunk_indices, int64_t capacity, int64_t* chunk_offsets,
                       int32_t* err_flag, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_CHUNK_METADATA_H */
