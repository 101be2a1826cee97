"""The C-ABI library builds, loads without a GPU and exports every function
``include/*.h`` declares; its host-side argument checks answer with the right
codes before any CUDA call (fake, never-dereferenced pointers)."""
import ctypes
import glob
import os
import re

import pytest

from linear_attention_decode_04_gb300 import binding
from linear_attention_decode_04_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return binding.load_library()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(kda_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    assert {"kda_decode", "kda_status_string", "kda_last_error", "kda_abi_version"} <= set(declared_functions())


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(binding.library_path())
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared but not exported"


def test_struct_layout_matches_header(lib):
    # every field of the C struct, in order, in the Python mirror
    text = open(os.path.join(ROOT, "include", "kda_decode.h")).read()
    body = text[text.index("typedef struct KdaDecodeArgs {"):text.index("} KdaDecodeArgs;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"(\w+)\s*;", body)
    assert fields == [f for f, _ in binding.KdaDecodeArgs._fields_]


def test_prefill_struct_layout_matches_header(lib):
    text = open(os.path.join(ROOT, "include", "kda_prefill.h")).read()
    body = text[text.index("typedef struct KdaPrefillArgs {"):text.index("} KdaPrefillArgs;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = []
    for decl in re.findall(r"([^;{]+);", body):   # "int32_t B, H, num_slots" declares three
        first, *rest = decl.split(",")
        fields += [first.split()[-1].lstrip("*")] + [r.strip().lstrip("*") for r in rest]
    assert fields == [f for f, _ in binding.KdaPrefillArgs._fields_]


def _pargs(**kw):
    a = binding.KdaPrefillArgs(struct_size=ctypes.sizeof(binding.KdaPrefillArgs), B=3, H=4,
                               num_slots=8, head_dim=128, conv_width=4, T=40, eps=1e-6, flags=1)
    fake = 0x10000
    for f in ("cu_seqlens", "qkv", "conv_weight", "conv_state", "state", "g", "beta", "gate",
              "norm_weight", "slot_idx", "out", "chunk_indices", "chunk_offsets", "workspace"):
        setattr(a, f, fake)
        fake += 0x100000
    a.num_chunks = 3
    a.workspace_bytes = 1 << 30
    a.qkv_row_stride = 3 * 4 * 128
    a.gate_row_stride = a.out_row_stride = 4 * 128
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_prefill_host_validation_codes(lib):
    L = binding.load_library()
    call = lambda a: L.kda_prefill(ctypes.byref(a), None)  # noqa: E731
    assert L.kda_prefill(None, None) == -1
    assert call(_pargs(struct_size=8)) == -6
    assert call(_pargs(head_dim=64)) == -2
    assert call(_pargs(B=-1)) == -2
    assert call(_pargs(T=-1)) == -2
    assert call(_pargs(flags=2)) == -4                  # the conv state is always advanced by prefill
    assert call(_pargs(flags=32)) == -4
    assert call(_pargs(B=0)) == 0                       # no-op, no launch
    assert call(_pargs(T=0)) == 0
    assert call(_pargs(cu_seqlens=None)) == -1
    assert call(_pargs(gate=None)) == -1                # norm on needs the gate
    assert call(_pargs(qkv_row_stride=100)) == -2
    assert call(_pargs(qkv_row_stride=3 * 4 * 128 + 4)) == -3
    assert call(_pargs(state=0x10004)) == -3
    assert call(_pargs(out=0x10004)) == -3
    assert b"aligned" in L.kda_last_error()
    assert call(_pargs(workspace=0x10008)) == -3        # workspace needs 16-byte alignment
    assert call(_pargs(chunk_offsets=None)) == -1
    assert call(_pargs(workspace_bytes=1000)) == -2     # smaller than the chunks need
    assert b"workspace" in L.kda_last_error()
    assert call(_pargs(num_chunks=-1)) == -2
    assert call(_pargs(flags=1 | 8)) == -1              # fused gate needs A_log
    assert call(_pargs(flags=1 | 8, A_log=0x20002)) == -3
    assert call(_pargs(seq_order=0x20002)) == -3        # seq_order needs 4-byte alignment
    L.kda_prefill_workspace_bytes.restype = ctypes.c_int64
    L.kda_prefill_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32]
    assert L.kda_prefill_workspace_bytes(10, 4) == 10 * 4 * 86528
    assert L.kda_prefill_workspace_bytes(-1, 4) == -1


def _args(**kw):
    a = binding.KdaDecodeArgs(struct_size=ctypes.sizeof(binding.KdaDecodeArgs), N=4, H=12,
                              num_slots=8, head_dim=128, conv_width=4, eps=1e-6, flags=3)
    fake = 0x10000
    for f in ("qkv", "conv_weight", "conv_state", "state", "g", "beta", "gate", "norm_weight",
              "slot_idx", "out"):
        setattr(a, f, fake)
        fake += 0x100000
    a.qkv_row_stride = 3 * 12 * 128
    a.gate_row_stride = a.out_row_stride = 12 * 128
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _call(lib, a):
    return lib.kda_decode(ctypes.byref(a), None)


def test_host_validation_codes(lib):
    assert lib.kda_decode(None, None) == -1
    assert _call(lib, _args(struct_size=8)) == -6
    assert _call(lib, _args(head_dim=64)) == -2
    assert _call(lib, _args(conv_width=3)) == -2
    assert _call(lib, _args(H=0)) == -2
    assert _call(lib, _args(N=-1)) == -2
    assert _call(lib, _args(flags=32)) == -4
    assert _call(lib, _args(flags=3 | 8)) == -1            # fused gate needs A_log
    assert _call(lib, _args(flags=3 | 8, A_log=0x20002)) == -3
    assert _call(lib, _args(N=0)) == 0          # no-op, no launch
    assert _call(lib, _args(qkv=None)) == -1
    assert _call(lib, _args(gate=None)) == -1    # norm on needs the gate
    assert _call(lib, _args(qkv_row_stride=100)) == -2
    assert _call(lib, _args(qkv_row_stride=3 * 12 * 128 + 4)) == -3
    assert _call(lib, _args(state=0x10004)) == -3
    assert b"aligned" in lib.kda_last_error()
    # multi-token (speculative) form
    assert _call(lib, _args(tokens_per_seq=9)) == -2
    assert _call(lib, _args(tokens_per_seq=-1)) == -2
    assert _call(lib, _args(tokens_per_seq=4, src_slot=0x10002)) == -3
    assert _call(lib, _args(tokens_per_seq=4, N=0)) == 0
    assert lib.kda_status_string(-3).decode().startswith("pointer")


def test_noalloc_validates_before_enqueueing(lib):
    """kda_decode_noalloc answers every argument error with the same code as
    kda_decode before it makes any CUDA call: on this host, with no GPU, a
    call that got as far as the scratch look-up or its memset would answer
    KDA_ERR_LAUNCH instead."""
    fn = lib.kda_decode_noalloc
    fn.argtypes = [ctypes.POINTER(binding.KdaDecodeArgs), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    assert fn(None, None) == -1
    for kw, code in ((dict(struct_size=8), -6), (dict(head_dim=64), -2), (dict(N=-1), -2),
                     (dict(flags=32), -4), (dict(qkv=None), -1), (dict(state=0x10004), -3),
                     (dict(qkv_row_stride=100), -2), (dict(N=0), 0)):
        assert fn(ctypes.byref(_args(**kw)), None) == code, kw
        assert _call(lib, _args(**kw)) == code, kw
    # work_queue is ignored by the allocation-free entry (kda_decode checks it)
    assert _call(lib, _args(work_queue=0x10003)) == -3
    assert fn(ctypes.byref(_args(work_queue=0x10003)), None) == -5


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(FileNotFoundError):
        binding.load_library()


def test_oracle_builds():
    import oracle
    assert os.path.exists(oracle.build())


def test_chunk_metadata_validation_codes(lib):
    L = ctypes.CDLL(binding.library_path())
    f = L.kda_chunk_metadata
    f.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(None, 4, 64, 0x1000, 8, 0x2000, None, None) == -1      # no cu_seqlens
    assert f(0x1000, 4, 64, None, 8, 0x2000, None, None) == -1      # rows wanted, no buffer
    assert f(0x1000, 4, 0, 0x2000, 8, 0x3000, None, None) == -2     # chunk size 0
    assert f(0x1000, -1, 64, 0x2000, 8, 0x3000, None, None) == -2   # negative count
    assert f(0x1002, 4, 64, 0x2000, 8, 0x3000, None, None) == -3    # cu_seqlens misaligned
    assert f(0x1000, 4, 64, 0x2004, 8, 0x3000, None, None) == -3    # indices not 8-byte aligned


def test_prefill_longest_first_order(lib):
    # host helper: a stable sort by length, longest first; negative lengths count as 0
    import numpy as np
    import torch
    rng = np.random.default_rng(7)
    for B in (1, 2, 5, 16, 300):
        lens = rng.integers(-3, 90, B)
        lens[rng.integers(0, B, B // 3)] = 40        # ties
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        got = binding.longest_first_order(torch.from_numpy(cu)).tolist()
        want = sorted(range(B), key=lambda b: -max(int(lens[b]), 0))
        assert got == want
    assert binding.longest_first_order(torch.zeros(1, dtype=torch.int32)).numel() == 0
    L = binding.load_library()
    assert L.kda_prefill_longest_first(None, 0, None) == 0
    assert L.kda_prefill_longest_first(None, 3, None) == -1
    assert L.kda_prefill_longest_first(None, -1, None) == -2


def test_device_error_bits_are_distinct():
    # the KDA_DEVERR_* bits of all headers share one err_flag word
    bits = {}
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        for name, val in re.findall(r"#define\s+(KDA_DEVERR_\w+)\s+(\d+)", open(h).read()):
            bits[name] = int(val)
    assert {"KDA_DEVERR_SLOT_RANGE", "KDA_DEVERR_TIMEOUT", "KDA_DEVERR_SEQLENS", "KDA_DEVERR_CAPACITY",
            "KDA_DEVERR_ORDER"} <= set(bits)
    vals = list(bits.values())
    assert all(v > 0 and v & (v - 1) == 0 for v in vals) and len(set(vals)) == len(vals)
