// kda_chunk_metadata.cu -- device-side chunk metadata for chunked prefill
// (the page "[ROCm][Perf] Kimi-K3 Remove prefill pipeline stall in chunk
// KDA", 实现拆解 item 2; definition in include/kda_chunk_metadata.h).
//
// One CTA: a block-wide exclusive scan of the per-sequence chunk counts in
// tiles of 1024 sequences writes chunk_offsets (and, for up to 4096
// sequences, a shared-memory copy), then each warp takes sequences
// i = warp, warp + 32, ... and its lanes write that sequence's rows
// off[i] + c, c = lane, lane + 32, ... (coalesced 8-byte rows).
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_chunk_metadata.h"
#include "kda_decode.h"

namespace {

constexpr int kThreads = 1024;
constexpr int kSharedOffsets = 4097;  // offsets kept on chip for up to 4096 sequences

__global__ void __launch_bounds__(kThreads) chunk_metadata_kernel(const int32_t* __restrict__ cu, int n_seqs,
                                                                   int bt, int32_t* __restrict__ idx,
                                                                   int64_t capacity, int64_t* __restrict__ off,
                                                                   int32_t* err) {
  __shared__ int64_t warp_tot[kThreads / 32];
  __shared__ int64_t carry_s;
  __shared__ int64_t off_s[kSharedOffsets];
  const bool on_chip = n_seqs < kSharedOffsets;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry_s = 0;
  __syncthreads();
  bool bad = false;
  for (int base = 0; base < n_seqs; base += kThreads) {
    const int i = base + tid;
    int64_t nt = 0;
    if (i < n_seqs) {
      const int64_t len = static_cast<int64_t>(cu[i + 1]) - cu[i];
      if (len < 0) bad = true;
      nt = len > 0 ? (len + bt - 1) / bt : 0;
    }
    // inclusive scan within the warp, then across warps
    int64_t x = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int64_t t = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      warp_tot[lane] = t;  // inclusive totals of warps 0..lane
    }
    __syncthreads();
    const int64_t carry = carry_s;
    const int64_t excl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x - nt;
    if (i < n_seqs) {
      off[i] = excl;
      if (on_chip) off_s[i] = excl;
    }
    __syncthreads();
    if (tid == 0) carry_s = carry + warp_tot[kThreads / 32 - 1];
    __syncthreads();
  }
  const int64_t total = carry_s;
  if (tid == 0) {
    off[n_seqs] = total;
    if (on_chip) off_s[n_seqs] = total;
  }
  if (bad && err) atomicOr(err, KDA_DEVERR_SEQLENS);
  if (tid == 0 && total > capacity && err) atomicOr(err, KDA_DEVERR_CAPACITY);
  __syncthreads();  // offsets written by this CTA are visible to it from here on
  const int64_t* offs = on_chip ? off_s : off;
  for (int i = warp; i < n_seqs; i += kThreads / 32) {
    const int64_t first = offs[i], last = offs[i + 1] < capacity ? offs[i + 1] : capacity;
    for (int64_t r = first + lane; r < last; r += 32) {
      int2 row;
      row.x = i;
      row.y = static_cast<int32_t>(r - first);
      reinterpret_cast<int2*>(idx)[r] = row;
    }
  }
}

}  // namespace

extern "C" int kda_chunk_metadata(const int32_t* cu_seqlens, int32_t num_seqs, int32_t chunk_size,
                                  int32_t* chunk_indices, int64_t capacity, int64_t* chunk_offsets,
                                  int32_t* err_flag, void* stream) {
  if (!cu_seqlens || !chunk_offsets || (capacity > 0 && !chunk_indices)) return KDA_ERR_NULLPTR;
  if (num_seqs < 0 || chunk_size <= 0 || capacity < 0) return KDA_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) || (reinterpret_cast<uintptr_t>(chunk_offsets) & 7u) ||
      (reinterpret_cast<uintptr_t>(chunk_indices) & 7u) || (reinterpret_cast<uintptr_t>(err_flag) & 3u))
    return KDA_ERR_ALIGN;
  chunk_metadata_kernel<<<1, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      cu_seqlens, num_seqs, chunk_size, chunk_indices, capacity, chunk_offsets, err_flag);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}
