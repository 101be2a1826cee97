"""Python binding of the C ABI in ``include/kda_decode.h``.

Argument marshalling only: tensors are checked for device, dtype and layout,
their pointers are packed into ``KdaDecodeArgs`` and ``kda_decode`` in
``lib/libkda_decode.so`` runs every step of the decode on the GPU.  There is
no other code path: a missing library, a CPU tensor or a failing call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HEAD_DIM = 128
CONV_WIDTH = 4
KDA_OUT_NORM = 1
KDA_UPDATE_CONV_STATE = 2
KDA_EARLY_PREFETCH = 4
KDA_FUSED_GATE = 8
KDA_CONV_STATE_SD = 16
KDA_DEVERR_SLOT_RANGE = 1
KDA_DEVERR_TIMEOUT = 2
ABI_VERSION = 2
MAX_TOKENS_PER_SEQ = 8

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
# KDA_DECODE_TIMELINE=1 in the environment (read when the library is first
# loaded) selects the build with the decode kernel's per-CTA timeline
# compiled in; results are identical, the kernel also records timestamps.
_LIB_PATH = os.path.join(_PKG_DIR, "lib", "libkda_decode_timeline.so"
                         if os.environ.get("KDA_DECODE_TIMELINE") == "1" else "libkda_decode.so")
_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"kda_decode failed with status {status}: {detail}")
        self.status = status


class KdaDecodeArgs(ctypes.Structure):
    """Mirror of ``struct KdaDecodeArgs`` (field order and types must match)."""
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("N", ctypes.c_int32), ("H", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("conv_width", ctypes.c_int32),
        ("qkv", ctypes.c_void_p), ("qkv_row_stride", ctypes.c_int64),
        ("conv_weight", ctypes.c_void_p), ("conv_bias", ctypes.c_void_p),
        ("conv_state", ctypes.c_void_p), ("state", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("gate", ctypes.c_void_p), ("gate_row_stride", ctypes.c_int64),
        ("norm_weight", ctypes.c_void_p), ("slot_idx", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("out_row_stride", ctypes.c_int64),
        ("eps", ctypes.c_float), ("q_scale", ctypes.c_float),
        ("flags", ctypes.c_uint32), ("err_flag", ctypes.c_void_p),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p), ("lower_bound", ctypes.c_float),
        ("work_queue", ctypes.c_void_p),
        ("tokens_per_seq", ctypes.c_int32), ("src_slot", ctypes.c_void_p),
    ]


class KdaPrefillArgs(ctypes.Structure):
    """Mirror of ``KdaPrefillArgs`` in ``include/kda_prefill.h`` (field order matters)."""
    _fields_ = [
        ("struct_size", ctypes.c_size_t),
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("conv_width", ctypes.c_int32),
        ("T", ctypes.c_int64),
        ("cu_seqlens", ctypes.c_void_p),
        ("qkv", ctypes.c_void_p), ("qkv_row_stride", ctypes.c_int64),
        ("conv_weight", ctypes.c_void_p), ("conv_bias", ctypes.c_void_p),
        ("conv_state", ctypes.c_void_p), ("state", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("gate", ctypes.c_void_p), ("gate_row_stride", ctypes.c_int64),
        ("norm_weight", ctypes.c_void_p), ("slot_idx", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("out_row_stride", ctypes.c_int64),
        ("eps", ctypes.c_float), ("q_scale", ctypes.c_float),
        ("flags", ctypes.c_uint32), ("err_flag", ctypes.c_void_p),
        ("chunk_indices", ctypes.c_void_p), ("chunk_offsets", ctypes.c_void_p),
        ("num_chunks", ctypes.c_int64), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_int64),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p), ("lower_bound", ctypes.c_float),
        ("seq_order", ctypes.c_void_p),
    ]


PREFILL_CHUNK = 32  # KDA_PREFILL_CHUNK


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load the CUDA library once; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise FileNotFoundError(
                    f"{_LIB_PATH} is missing: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(_LIB_PATH)
            L.kda_decode.argtypes = [ctypes.POINTER(KdaDecodeArgs), ctypes.c_void_p]
            L.kda_decode.restype = ctypes.c_int
            L.kda_status_string.argtypes = [ctypes.c_int]
            L.kda_status_string.restype = ctypes.c_char_p
            L.kda_last_error.argtypes = []
            L.kda_last_error.restype = ctypes.c_char_p
            L.kda_decode_wait_test.argtypes = [ctypes.POINTER(KdaDecodeArgs), ctypes.c_void_p,
                                               ctypes.c_uint64, ctypes.c_int32]
            L.kda_decode_wait_test.restype = ctypes.c_int
            L.kda_chunk_metadata.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p]
            L.kda_chunk_metadata.restype = ctypes.c_int
            L.kda_prefill.argtypes = [ctypes.POINTER(KdaPrefillArgs), ctypes.c_void_p]
            L.kda_prefill.restype = ctypes.c_int
            L.kda_prefill_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32]
            L.kda_prefill_workspace_bytes.restype = ctypes.c_int64
            L.kda_prefill_longest_first.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
            L.kda_prefill_longest_first.restype = ctypes.c_int
            L.kda_abi_version.argtypes = []
            L.kda_abi_version.restype = ctypes.c_int
            if L.kda_abi_version() != ABI_VERSION:
                raise RuntimeError(f"{_LIB_PATH}: ABI version {L.kda_abi_version()} != {ABI_VERSION}")
            _lib = L
    return _lib


def timeline_read(max_records: int = 1 << 16):
    """Per-CTA records of the decode kernel since the last reset (timeline
    build only): int64 [n, 8] = block, SM, start ns, first unit ready ns, end
    ns, units, consumer compute ns, consumer wait ns."""
    import numpy as np
    lib = load_library()
    if not hasattr(lib, "kda_timeline_read"):
        raise RuntimeError("the loaded library has no timeline (set KDA_DECODE_TIMELINE=1 before loading)")
    buf = np.zeros((max_records, 8), np.uint64)
    total = ctypes.c_uint(0)
    fn = lib.kda_timeline_read
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_uint)]
    fn.restype = ctypes.c_int
    n = fn(buf.ctypes.data, max_records, ctypes.byref(total))
    if n < 0:
        raise KdaError(n, lib.kda_last_error().decode())
    return buf[:n].astype(np.int64)


def timeline_reset() -> None:
    lib = load_library()
    rc = lib.kda_timeline_reset()
    if rc != 0:
        raise KdaError(rc, lib.kda_last_error().decode())


def kda_status_string(status: int) -> str:
    return load_library().kda_status_string(int(status)).decode()


def _check(t: torch.Tensor, name: str, dtype: torch.dtype, device: torch.device | None,
           host_ok: bool = False):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if host_ok and t.device.type == "cpu":
        # pinned host memory is mapped into the GPU's address space: the
        # kernel reads or writes it directly over the CPU-GPU link
        if not t.is_pinned():
            raise ValueError(f"{name} is a CPU tensor: it must be pinned (tensor.pin_memory())")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
        return
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _dense(t: torch.Tensor, name: str):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _rows(t: torch.Tensor, name: str, N: int, width: int) -> int:
    """Row-strided 2-D view [N, >= width] with unit inner stride; returns the row stride."""
    if t.dim() != 2 or t.shape[0] != N or t.shape[1] < width:
        raise ValueError(f"{name} must be [N={N}, >={width}] (got {tuple(t.shape)})")
    if t.stride(1) != 1:
        raise ValueError(f"{name} needs a unit inner stride")
    return t.stride(0) if N > 1 else max(t.stride(0), width)


class KdaDecodeCall:
    """A prepared ``kda_decode`` call: validates and packs the arguments once;
    each ``__call__`` is one C call (cheap enough for eager loops and CUDA
    graph capture).  Keeps references to the tensors it points at.

    ``host_token_io=True`` lets the per-token tensors (qkv, g, beta, gate,
    slot_idx, out) be pinned host tensors: the kernel then reads them and
    writes the output straight over the CPU-GPU link, with no copy step.
    The host must not rewrite them while a launch that uses them may run.

    Multi-token (speculative) decode: with ``tokens_per_seq`` = T >= 2 or a
    ``src_slot`` tensor (int32 [N]), the per-token tensors hold N*T rows
    (sequence n's tokens at rows n*T .. n*T + T - 1), ``slot_idx`` is int32
    [N, T] (the destination of each token's state and conv window; <= 0 =
    absent token) and each sequence starts from ``src_slot[n]`` (default
    ``slot_idx[n, 0]``)."""

    def __init__(self, qkv, conv_weight, conv_state, state, g, beta, slot_idx, out, *,
                 gate=None, norm_weight=None, conv_bias=None, eps: float = 1e-6,
                 q_scale: float = 0.0, out_norm: bool = True, update_conv_state: bool = True,
                 err_flag=None, early_prefetch: bool = False, A_log=None, dt_bias=None,
                 lower_bound: float = 0.0, work_queue=None, conv_state_layout: str = "DS",
                 host_token_io: bool = False, tokens_per_seq: int = 1, src_slot=None):
        self._lib = load_library()
        dev = state.device
        _check(state, "state", torch.float32, None)
        if state.dim() != 4 or state.shape[2:] != (HEAD_DIM, HEAD_DIM):
            raise ValueError(f"state must be [slots, H, 128, 128] (got {tuple(state.shape)})")
        _dense(state, "state")
        num_slots, H = int(state.shape[0]), int(state.shape[1])
        D = H * HEAD_DIM
        C = 3 * D
        _check(qkv, "qkv", torch.bfloat16, dev, host_token_io)
        T = int(tokens_per_seq)
        if not 1 <= T <= MAX_TOKENS_PER_SEQ:
            raise ValueError(f"tokens_per_seq must be 1 .. {MAX_TOKENS_PER_SEQ} (got {T})")
        multi = T > 1 or src_slot is not None
        R = int(qkv.shape[0])                # token rows
        if R % T:
            raise ValueError(f"qkv has {R} rows, not a multiple of tokens_per_seq={T}")
        N = R // T                           # sequences (= rows when T = 1)
        qkv_stride = _rows(qkv, "qkv", R, C)
        _check(conv_weight, "conv_weight", torch.float32, dev)
        if tuple(conv_weight.shape) != (3, CONV_WIDTH, D):
            raise ValueError(f"conv_weight must be [3, 4, {D}] (got {tuple(conv_weight.shape)})")
        _dense(conv_weight, "conv_weight")
        _check(conv_state, "conv_state", torch.bfloat16, dev)
        if conv_state_layout not in ("DS", "SD"):
            raise ValueError("conv_state_layout is 'DS' ([slots, C, 3]) or 'SD' ([slots, 3, C])")
        want_cs = (num_slots, C, CONV_WIDTH - 1) if conv_state_layout == "DS" else (num_slots, CONV_WIDTH - 1, C)
        if tuple(conv_state.shape) != want_cs:
            raise ValueError(f"conv_state ({conv_state_layout}) must be {list(want_cs)} (got {tuple(conv_state.shape)})")
        _dense(conv_state, "conv_state")
        _check(g, "g", torch.float32, dev, host_token_io)
        if tuple(g.shape) != (R, H, HEAD_DIM):
            raise ValueError(f"g must be [{R}, {H}, 128] (got {tuple(g.shape)})")
        _dense(g, "g")
        _check(beta, "beta", torch.bfloat16, dev, host_token_io)
        if tuple(beta.shape) != (R, H):
            raise ValueError(f"beta must be [{R}, {H}] (got {tuple(beta.shape)})")
        _dense(beta, "beta")
        _check(slot_idx, "slot_idx", torch.int32, dev, host_token_io)
        if slot_idx.numel() != R or (multi and tuple(slot_idx.shape) not in ((N, T), (R,))) or \
                (not multi and tuple(slot_idx.shape) != (N,)):
            want = f"[{N}, {T}]" if multi else f"[{N}]"
            raise ValueError(f"slot_idx must be {want} (got {tuple(slot_idx.shape)})")
        _dense(slot_idx, "slot_idx")
        src_ptr = None
        if src_slot is not None:
            _check(src_slot, "src_slot", torch.int32, dev, host_token_io)
            if tuple(src_slot.shape) != (N,):
                raise ValueError(f"src_slot must be [{N}] (got {tuple(src_slot.shape)})")
            _dense(src_slot, "src_slot")
            src_ptr = src_slot.data_ptr()
        _check(out, "out", torch.bfloat16, dev, host_token_io)
        out_stride = _rows(out, "out", R, D)
        fused_gate = A_log is not None
        flags = ((KDA_OUT_NORM if out_norm else 0) | (KDA_UPDATE_CONV_STATE if update_conv_state else 0)
                 | (KDA_EARLY_PREFETCH if early_prefetch else 0) | (KDA_FUSED_GATE if fused_gate else 0)
                 | (KDA_CONV_STATE_SD if conv_state_layout == "SD" else 0))
        alog_ptr = dtb_ptr = None
        if fused_gate:
            _check(A_log, "A_log", torch.float32, dev)
            if tuple(A_log.shape) != (H,):
                raise ValueError(f"A_log must be [{H}]")
            alog_ptr = A_log.data_ptr()
            if dt_bias is not None:
                _check(dt_bias, "dt_bias", torch.float32, dev)
                if tuple(dt_bias.shape) != (H * HEAD_DIM,):
                    raise ValueError(f"dt_bias must be [{H * HEAD_DIM}]")
                _dense(dt_bias, "dt_bias")
                dtb_ptr = dt_bias.data_ptr()
        gate_ptr = nw_ptr = None
        gate_stride = 0
        if out_norm:
            if gate is None or norm_weight is None:
                raise ValueError("out_norm needs gate and norm_weight")
            _check(gate, "gate", torch.bfloat16, dev, host_token_io)
            gate_stride = _rows(gate, "gate", R, D)
            _check(norm_weight, "norm_weight", torch.float32, dev)
            if tuple(norm_weight.shape) != (HEAD_DIM,):
                raise ValueError("norm_weight must be [128]")
            gate_ptr, nw_ptr = gate.data_ptr(), norm_weight.data_ptr()
        bias_ptr = None
        if conv_bias is not None:
            _check(conv_bias, "conv_bias", torch.float32, dev)
            if tuple(conv_bias.shape) != (C,):
                raise ValueError(f"conv_bias must be [{C}]")
            bias_ptr = conv_bias.data_ptr()
        queue_ptr = None
        if work_queue is not None:
            _check(work_queue, "work_queue", torch.int32, dev)
            if work_queue.numel() < 2:
                raise ValueError("work_queue needs 2 int32")
            queue_ptr = work_queue.data_ptr()
        err_ptr = None
        if err_flag is not None:
            _check(err_flag, "err_flag", torch.int32, dev)
            err_ptr = err_flag.data_ptr()
        self.device = dev
        self.N, self.H, self.num_slots, self.T = N, H, num_slots, T
        self._keep = (qkv, conv_weight, conv_state, state, g, beta, slot_idx, out, gate,
                      norm_weight, conv_bias, err_flag, A_log, dt_bias, work_queue, src_slot)
        self.args = KdaDecodeArgs(
            struct_size=ctypes.sizeof(KdaDecodeArgs), N=N, H=H, num_slots=num_slots,
            head_dim=HEAD_DIM, conv_width=CONV_WIDTH,
            qkv=qkv.data_ptr(), qkv_row_stride=qkv_stride,
            conv_weight=conv_weight.data_ptr(), conv_bias=bias_ptr,
            conv_state=conv_state.data_ptr(), state=state.data_ptr(),
            g=g.data_ptr(), beta=beta.data_ptr(), gate=gate_ptr, gate_row_stride=gate_stride,
            norm_weight=nw_ptr, slot_idx=slot_idx.data_ptr(),
            out=out.data_ptr(), out_row_stride=out_stride,
            eps=float(eps), q_scale=float(q_scale), flags=flags, err_flag=err_ptr,
            A_log=alog_ptr, dt_bias=dtb_ptr, lower_bound=float(lower_bound), work_queue=queue_ptr,
            tokens_per_seq=T if multi else 0, src_slot=src_ptr)
        self._argp = ctypes.byref(self.args)

    def __call__(self, stream: torch.cuda.Stream | None = None) -> None:
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        rc = self._lib.kda_decode(self._argp, ctypes.c_void_p(stream.cuda_stream))
        if rc != 0:
            raise KdaError(rc, f"{kda_status_string(rc)}: {self._lib.kda_last_error().decode()}")

    def wait_test(self, wait_limit_ns: int, withhold_unit: int,
                  stream: torch.cuda.Stream | None = None) -> None:
        """``kda_decode_wait_test``: exercise the bounded-wait failure path."""
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        rc = self._lib.kda_decode_wait_test(self._argp, ctypes.c_void_p(stream.cuda_stream),
                                            int(wait_limit_ns), int(withhold_unit))
        if rc != 0:
            raise KdaError(rc, f"{kda_status_string(rc)}: {self._lib.kda_last_error().decode()}")


def kda_decode(qkv, conv_weight, conv_state, state, g, beta, slot_idx, out, *,
               gate=None, norm_weight=None, conv_bias=None, eps: float = 1e-6,
               q_scale: float = 0.0, out_norm: bool = True, update_conv_state: bool = True,
               err_flag=None, early_prefetch: bool = False, A_log=None, dt_bias=None,
               lower_bound: float = 0.0, work_queue=None, conv_state_layout: str = "DS",
               tokens_per_seq: int = 1, src_slot=None,
               stream: torch.cuda.Stream | None = None) -> None:
    """One fused decode step (see ``include/kda_decode.h``).  ``conv_state``,
    ``state`` and ``out`` are written in place on ``stream`` (default: the
    current stream of the state's device).  ``early_prefetch`` sets
    KDA_EARLY_PREFETCH: only when the kernel enqueued just before on the
    stream writes none of slot_idx, state and conv_state.  Passing ``A_log``
    sets KDA_FUSED_GATE: ``g`` and ``beta`` are then raw logits.
    ``work_queue`` (int32[2], zero) enables the dynamic schedule.
    ``conv_state_layout`` is "DS" ([slots, C, 3]) or "SD" ([slots, 3, C]).
    ``tokens_per_seq`` / ``src_slot`` select the multi-token (speculative)
    form described on ``KdaDecodeCall``."""
    KdaDecodeCall(qkv, conv_weight, conv_state, state, g, beta, slot_idx, out, gate=gate,
                  norm_weight=norm_weight, conv_bias=conv_bias, eps=eps, q_scale=q_scale,
                  out_norm=out_norm, update_conv_state=update_conv_state,
                  err_flag=err_flag, early_prefetch=early_prefetch, A_log=A_log, dt_bias=dt_bias,
                  lower_bound=lower_bound, work_queue=work_queue,
                  conv_state_layout=conv_state_layout, tokens_per_seq=tokens_per_seq,
                  src_slot=src_slot)(stream)


def kda_chunk_metadata(cu_seqlens: torch.Tensor, cu_seqlens_cpu: torch.Tensor, chunk_size: int,
                       err_flag=None, stream: torch.cuda.Stream | None = None):
    """Device-side chunk metadata for chunked prefill (``include/kda_chunk_metadata.h``):
    returns ``(chunk_indices int32 [total, 2], chunk_offsets int64 [N + 1])``.
    The output size comes from the host copy ``cu_seqlens_cpu``, so nothing
    waits for the device; the values are computed by the GPU from
    ``cu_seqlens`` (int32, on the GPU)."""
    lib = load_library()
    _check(cu_seqlens, "cu_seqlens", torch.int32, None)
    _dense(cu_seqlens, "cu_seqlens")
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must be [N + 1]")
    n = cu_seqlens.numel() - 1
    lens = (cu_seqlens_cpu[1:] - cu_seqlens_cpu[:-1]).to(torch.int64).clamp(min=0)
    total = int(((lens + chunk_size - 1) // chunk_size).sum()) if n > 0 else 0
    dev = cu_seqlens.device
    idx = torch.empty(max(total, 1), 2, dtype=torch.int32, device=dev)
    off = torch.empty(n + 1, dtype=torch.int64, device=dev)
    if err_flag is not None:
        _check(err_flag, "err_flag", torch.int32, dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    rc = lib.kda_chunk_metadata(cu_seqlens.data_ptr(), n, int(chunk_size), idx.data_ptr(), total,
                                off.data_ptr(), None if err_flag is None else err_flag.data_ptr(),
                                ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise KdaError(rc, kda_status_string(rc))
    return idx[:total], off


class KdaPrefillCall:
    """A prepared ``kda_prefill`` call (``include/kda_prefill.h``): validates
    and packs the arguments once, allocates the chunk metadata and the
    workspace (sized from ``cu_seqlens_cpu``, the host copy of the sequence
    starts, so nothing waits for the device); each ``__call__`` enqueues the
    device-side metadata build and the prefill.  Keeps references to the
    tensors it points at.  With ``longest_first`` (the default) the scan takes
    the sequences longest first (``seq_order``), which shortens the tail of
    a batch with ragged lengths and changes no result.

    Shapes: T token rows, B sequences, H heads, D = H * 128.
      qkv [T, >=3D] bf16, conv_weight [3, 4, D] f32, conv_state [slots, 3D, 3]
      bf16, state [slots, H, 128, 128] f32, g [T, H, 128] f32, beta [T, H]
      bf16, cu_seqlens [B + 1] int32 (device), slot_idx [B] int32, out
      [T, >=D] bf16, gate [T, >=D] bf16 and norm_weight [128] f32 with
      out_norm."""

    def __init__(self, qkv, conv_weight, conv_state, state, g, beta, cu_seqlens, slot_idx, out, *,
                 cu_seqlens_cpu=None, gate=None, norm_weight=None, conv_bias=None, eps: float = 1e-6,
                 q_scale: float = 0.0, out_norm: bool = True, err_flag=None, A_log=None, dt_bias=None,
                 lower_bound: float = 0.0, conv_state_layout: str = "DS", longest_first: bool = True):
        self._lib = load_library()
        dev = state.device
        _check(state, "state", torch.float32, None)
        _dense(state, "state")
        if state.dim() != 4 or state.shape[2:] != (128, 128):
            raise ValueError(f"state must be [slots, H, 128, 128] (got {tuple(state.shape)})")
        num_slots, H = state.shape[0], state.shape[1]
        D = H * 128
        T = qkv.shape[0]
        _check(qkv, "qkv", torch.bfloat16, dev)
        qkv_stride = _rows(qkv, "qkv", T, 3 * D)
        for name, t, dt in (("conv_weight", conv_weight, torch.float32),
                            ("conv_state", conv_state, torch.bfloat16), ("g", g, torch.float32),
                            ("beta", beta, torch.bfloat16), ("cu_seqlens", cu_seqlens, torch.int32),
                            ("slot_idx", slot_idx, torch.int32)):
            _check(t, name, dt, dev)
            _dense(t, name)
        if conv_weight.numel() != 3 * 4 * D:
            raise ValueError("conv_weight must be [3, 4, H*128]")
        if conv_state.numel() != num_slots * 3 * D * 3:
            raise ValueError("conv_state must be [slots, 3*H*128, 3]")
        if g.numel() != T * D or beta.numel() != T * H:
            raise ValueError("g must be [T, H, 128] and beta [T, H]")
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
            raise ValueError("cu_seqlens must be [B + 1]")
        B = cu_seqlens.numel() - 1
        if slot_idx.numel() != B:
            raise ValueError(f"slot_idx must have one entry per sequence ({B})")
        if cu_seqlens_cpu is None:
            cu_seqlens_cpu = cu_seqlens.cpu()  # a device read; pass the host copy to avoid it
        cu_cpu = torch.as_tensor(cu_seqlens_cpu).to(torch.int64).reshape(-1)
        if cu_cpu.numel() != B + 1:
            raise ValueError("cu_seqlens_cpu must match cu_seqlens")
        lens = (cu_cpu[1:] - cu_cpu[:-1]).clamp(min=0)
        num_chunks = int(((lens + PREFILL_CHUNK - 1) // PREFILL_CHUNK).sum()) if B > 0 else 0
        _check(out, "out", torch.bfloat16, dev)
        out_stride = _rows(out, "out", T, D)
        gate_stride = 0
        if out_norm:
            if gate is None or norm_weight is None:
                raise ValueError("out_norm needs gate and norm_weight")
            _check(gate, "gate", torch.bfloat16, dev)
            gate_stride = _rows(gate, "gate", T, D)
            _check(norm_weight, "norm_weight", torch.float32, dev)
            _dense(norm_weight, "norm_weight")
            if norm_weight.numel() != 128:
                raise ValueError("norm_weight must be [128]")
        if conv_bias is not None:
            _check(conv_bias, "conv_bias", torch.float32, dev)
            _dense(conv_bias, "conv_bias")
            if conv_bias.numel() != 3 * D:
                raise ValueError("conv_bias must be [3*H*128]")
        if err_flag is not None:
            _check(err_flag, "err_flag", torch.int32, dev)
        flags = KDA_OUT_NORM if out_norm else 0
        if conv_state_layout not in ("DS", "SD"):
            raise ValueError('conv_state_layout must be "DS" or "SD"')
        if conv_state_layout == "SD":
            flags |= KDA_CONV_STATE_SD
        if A_log is not None:  # g and beta are raw logits
            _check(A_log, "A_log", torch.float32, dev)
            _dense(A_log, "A_log")
            if A_log.numel() != H:
                raise ValueError("A_log must be [H]")
            if dt_bias is not None:
                _check(dt_bias, "dt_bias", torch.float32, dev)
                _dense(dt_bias, "dt_bias")
                if dt_bias.numel() != D:
                    raise ValueError("dt_bias must be [H*128]")
            flags |= KDA_FUSED_GATE
        elif dt_bias is not None:
            raise ValueError("dt_bias needs A_log (the fused gate)")
        ws_bytes = int(self._lib.kda_prefill_workspace_bytes(num_chunks, H))
        self.num_chunks, self.B = num_chunks, B
        self.chunk_indices = torch.empty(max(num_chunks, 1), 2, dtype=torch.int32, device=dev)
        self.chunk_offsets = torch.empty(B + 1, dtype=torch.int64, device=dev)
        self.workspace = torch.empty(max(ws_bytes // 4, 4), dtype=torch.float32, device=dev)
        self.device = dev
        # the scan takes the longest sequences first; the order is computed on
        # the host and uploaded once, and left out where it is the index order
        # or where the upload would fall inside a stream capture
        self.seq_order = None
        if longest_first and B > 1 and not torch.cuda.is_current_stream_capturing():
            order = longest_first_order(cu_cpu.to(torch.int32))
            if not torch.equal(order, torch.arange(B, dtype=torch.int32)):
                self.seq_order = order.to(dev)
        self._keep = (qkv, conv_weight, conv_state, state, g, beta, cu_seqlens, slot_idx, out, gate,
                      norm_weight, conv_bias, err_flag, A_log, dt_bias)
        self._cu, self._err = cu_seqlens, err_flag
        ptr = (lambda t: None if t is None else t.data_ptr())
        self.args = KdaPrefillArgs(
            struct_size=ctypes.sizeof(KdaPrefillArgs), B=B, H=H, num_slots=num_slots,
            head_dim=128, conv_width=4, T=T, cu_seqlens=ptr(cu_seqlens), qkv=ptr(qkv),
            qkv_row_stride=qkv_stride, conv_weight=ptr(conv_weight), conv_bias=ptr(conv_bias),
            conv_state=ptr(conv_state), state=ptr(state), g=ptr(g), beta=ptr(beta),
            gate=ptr(gate) if out_norm else None, gate_row_stride=gate_stride,
            norm_weight=ptr(norm_weight) if out_norm else None, slot_idx=ptr(slot_idx), out=ptr(out),
            out_row_stride=out_stride, eps=eps, q_scale=q_scale,
            flags=flags, err_flag=ptr(err_flag),
            chunk_indices=ptr(self.chunk_indices), chunk_offsets=ptr(self.chunk_offsets),
            num_chunks=num_chunks, workspace=ptr(self.workspace), workspace_bytes=ws_bytes,
            A_log=ptr(A_log), dt_bias=ptr(dt_bias), lower_bound=lower_bound, seq_order=ptr(self.seq_order))

    def __call__(self, stream: torch.cuda.Stream | None = None) -> None:
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        if self.B == 0:
            return
        sp = ctypes.c_void_p(stream.cuda_stream)
        rc = self._lib.kda_chunk_metadata(self._cu.data_ptr(), self.B, PREFILL_CHUNK,
                                          self.chunk_indices.data_ptr(), self.num_chunks,
                                          self.chunk_offsets.data_ptr(),
                                          None if self._err is None else self._err.data_ptr(), sp)
        if rc != 0:
            raise KdaError(rc, kda_status_string(rc))
        rc = self._lib.kda_prefill(ctypes.byref(self.args), sp)
        if rc != 0:
            raise KdaError(rc, f"{kda_status_string(rc)}: {self._lib.kda_last_error().decode()}")


def longest_first_order(cu_seqlens_cpu) -> torch.Tensor:
    """Sequence indices longest first (equal lengths in index order) from the
    host copy of ``cu_seqlens``, by ``kda_prefill_longest_first``."""
    cu = torch.as_tensor(cu_seqlens_cpu, dtype=torch.int32).contiguous().reshape(-1)
    B = max(cu.numel() - 1, 0)
    order = torch.empty(B, dtype=torch.int32)
    rc = load_library().kda_prefill_longest_first(cu.data_ptr(), B, order.data_ptr())
    if rc != 0:
        raise KdaError(rc, kda_status_string(rc))
    return order


def kda_prefill(qkv, conv_weight, conv_state, state, g, beta, cu_seqlens, slot_idx, out, *,
                cu_seqlens_cpu=None, gate=None, norm_weight=None, conv_bias=None, eps: float = 1e-6,
                q_scale: float = 0.0, out_norm: bool = True, err_flag=None, A_log=None, dt_bias=None,
                lower_bound: float = 0.0, conv_state_layout: str = "DS",
                stream: torch.cuda.Stream | None = None) -> None:
    """Chunked prefill of a varlen batch (see ``include/kda_prefill.h``):
    ``out``, ``state`` and ``conv_state`` are written in place.  Pass
    ``cu_seqlens_cpu`` (the host copy of ``cu_seqlens``) to keep the call free
    of device reads.  Passing ``A_log`` sets KDA_FUSED_GATE: ``g`` and
    ``beta`` are then raw logits."""
    KdaPrefillCall(qkv, conv_weight, conv_state, state, g, beta, cu_seqlens, slot_idx, out,
                   cu_seqlens_cpu=cu_seqlens_cpu, gate=gate, norm_weight=norm_weight,
                   conv_bias=conv_bias, eps=eps, q_scale=q_scale, out_norm=out_norm,
                   err_flag=err_flag, A_log=A_log, dt_bias=dt_bias, lower_bound=lower_bound,
                   conv_state_layout=conv_state_layout)(stream)
