"""Reference for the device-side chunk metadata of chunked prefill.

TEST INFRASTRUCTURE ONLY (tests and the benchmark's CPU leg; the product
never imports it).

Source: the page "[ROCm][Perf] Kimi-K3 Remove prefill pipeline stall in
chunk KDA" (vLLM PR #51862 report), 实现拆解 item 2: from the cumulative
sequence starts `cu_seqlens` (length N+1, cu_seqlens[0] = 0, non-decreasing)
and a chunk size BT, build
  chunk_offsets[i] = number of chunks of sequences 0 .. i-1, for i = 0 .. N
                     (so chunk_offsets[N] is the total), where sequence j has
                     ceil((cu_seqlens[j+1] - cu_seqlens[j]) / BT) chunks;
  chunk_indices    = one row (seq_idx, chunk_idx) per chunk, sequences in
                     order and chunks in order within a sequence.
Plain loops, written from that definition.
"""
from __future__ import annotations


def chunk_metadata(cu_seqlens, chunk_size: int):
    """Returns (chunk_indices as a list of (seq, chunk) pairs, chunk_offsets list)."""
    assert chunk_size > 0
    n = len(cu_seqlens) - 1
    offsets = [0]
    indices = []
    for i in range(n):
        length = int(cu_seqlens[i + 1]) - int(cu_seqlens[i])
        assert length >= 0, "cu_seqlens must be non-decreasing"
        chunks = (length + chunk_size - 1) // chunk_size
        for c in range(chunks):
            indices.append((i, c))
        offsets.append(offsets[-1] + chunks)
    return indices, offsets
