"""Device-side chunk metadata (chunked prefill) against the reference,
bit-exact (integer work), through the C ABI."""
import numpy as np
import pytest
import torch

from linear_attention_decode_04_gb300 import binding, kda_chunk_metadata
from oracle.chunk_metadata import chunk_metadata

pytestmark = pytest.mark.gpu


def _case(lens, bt, dev):
    cu = np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))]).astype(np.int32)
    cu_cpu = torch.from_numpy(cu)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    idx, off = kda_chunk_metadata(cu_cpu.to(dev), cu_cpu, bt, err_flag=err)
    torch.cuda.synchronize()
    want_idx, want_off = chunk_metadata(cu.tolist(), bt)
    assert off.cpu().tolist() == want_off
    got = idx.cpu().numpy()
    assert np.array_equal(got, np.asarray(want_idx, dtype=np.int32).reshape(-1, 2))
    assert int(err.item()) == 0


@pytest.mark.parametrize("bt", [16, 64])
def test_random_batches(bt, cuda_device):
    rng = np.random.default_rng(bt)
    for n in (1, 5, 31, 1023, 1024, 1025, 5000):   # across the 1024-sequence scan tiles
        lens = rng.integers(0, 700, n) * (rng.random(n) > 0.15)   # some empty sequences
        _case(lens, bt, cuda_device)


def test_edge_cases(cuda_device):
    _case([], 64, cuda_device)                 # no sequences
    _case([0, 0, 0], 64, cuda_device)          # only empty sequences
    _case([64, 1, 0, 130], 64, cuda_device)    # exact multiple, single token, empty, ragged
    _case([1] * 3000, 1, cuda_device)          # chunk size 1


def test_capacity_and_bad_lengths_set_error_bits(cuda_device):
    lib = binding.load_library()
    cu = torch.tensor([0, 100, 90, 300], dtype=torch.int32, device=cuda_device)   # sequence 1 decreases
    idx = torch.full((2, 2), -7, dtype=torch.int32, device=cuda_device)
    off = torch.empty(4, dtype=torch.int64, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    import ctypes
    rc = lib.kda_chunk_metadata(cu.data_ptr(), 3, 64, idx.data_ptr(), 2, off.data_ptr(), err.data_ptr(),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0
    # lengths 100, -10 (-> 0 chunks), 210 -> 2 + 0 + 4 = 6 chunks, capacity 2
    assert off.cpu().tolist() == [0, 2, 2, 6]
    assert idx.cpu().tolist() == [[0, 0], [0, 1]]
    assert int(err.item()) == (4 | 8)
