"""Pins of the chunk-metadata reference (CPU): facts the definition fixes,
and agreement with an independent numpy construction."""
import numpy as np
import pytest

from oracle.chunk_metadata import chunk_metadata


def _numpy_construction(cu, bt):
    lens = np.diff(np.asarray(cu, dtype=np.int64))
    nt = -(-lens // bt)
    offsets = np.concatenate([[0], np.cumsum(nt)])
    seq = np.repeat(np.arange(len(lens)), nt)
    chunk = np.arange(offsets[-1]) - np.repeat(offsets[:-1], nt)
    return np.stack([seq, chunk], axis=1), offsets


def test_worked_example_by_hand():
    # lengths 64, 1, 0, 130 with BT = 64 -> 1, 1, 0, 3 chunks
    idx, off = chunk_metadata([0, 64, 65, 65, 195], 64)
    assert off == [0, 1, 2, 2, 5]
    assert idx == [(0, 0), (1, 0), (3, 0), (3, 1), (3, 2)]


def test_empty_batch_and_empty_sequences():
    assert chunk_metadata([0], 64) == ([], [0])
    assert chunk_metadata([0, 0, 0], 16) == ([], [0, 0, 0])


@pytest.mark.parametrize("bt", [1, 16, 64, 100])
def test_random_against_numpy(bt):
    rng = np.random.default_rng(bt)
    for n in (1, 2, 7, 300, 2500):
        lens = rng.integers(0, 500, n) * (rng.random(n) > 0.1)
        cu = np.concatenate([[0], np.cumsum(lens)])
        idx, off = chunk_metadata(cu.tolist(), bt)
        want_idx, want_off = _numpy_construction(cu, bt)
        assert off == want_off.tolist()
        assert np.array_equal(np.asarray(idx, dtype=np.int64).reshape(-1, 2), want_idx)
        # every chunk covers tokens inside its sequence
        for s, c in idx[:: max(1, len(idx) // 50)]:
            assert cu[s] + c * bt < cu[s + 1]
