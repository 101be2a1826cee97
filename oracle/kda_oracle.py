"""ctypes wrapper of the C oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE ONLY.  ``build()`` compiles the C source with the host's
gcc into ``oracle/_build/`` (plain C, OpenMP, ``-ffp-contract=off`` so x86 and
Arm produce the same bits).  Arrays are numpy; bf16 tensors travel as their
uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_HDR = os.path.join(_HERE, "kda_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libkda_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle library if it is missing or older than its source."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest_src:
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


class _Problem(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int32), ("H", ctypes.c_int32), ("K", ctypes.c_int32),
        ("V", ctypes.c_int32), ("W", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("qkv", ctypes.c_void_p), ("qkv_row_stride", ctypes.c_int64),
        ("conv_weight", ctypes.c_void_p), ("conv_bias", ctypes.c_void_p),
        ("conv_state", ctypes.c_void_p), ("state", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("gate", ctypes.c_void_p),
        ("norm_weight", ctypes.c_void_p), ("slot_idx", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("out_f64", ctypes.c_void_p),
        ("eps", ctypes.c_double), ("l2_eps", ctypes.c_double), ("q_scale", ctypes.c_double),
        ("out_norm", ctypes.c_int32), ("update_conv_state", ctypes.c_int32),
        ("fused_gate", ctypes.c_int32), ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("lower_bound", ctypes.c_double), ("conv_state_sd", ctypes.c_int32),
    ]


class _PrefillProblem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("K", ctypes.c_int32),
        ("V", ctypes.c_int32), ("W", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p),
        ("qkv", ctypes.c_void_p), ("qkv_row_stride", ctypes.c_int64),
        ("conv_weight", ctypes.c_void_p), ("conv_bias", ctypes.c_void_p),
        ("conv_state", ctypes.c_void_p), ("state", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("gate", ctypes.c_void_p),
        ("norm_weight", ctypes.c_void_p), ("slot_idx", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("out_f64", ctypes.c_void_p),
        ("eps", ctypes.c_double), ("l2_eps", ctypes.c_double), ("q_scale", ctypes.c_double),
        ("out_norm", ctypes.c_int32), ("fused_gate", ctypes.c_int32), ("A_log", ctypes.c_void_p),
        ("dt_bias", ctypes.c_void_p), ("lower_bound", ctypes.c_double),
        ("conv_state_sd", ctypes.c_int32),
    ]


class _MultiProblem(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32), ("K", ctypes.c_int32),
        ("V", ctypes.c_int32), ("W", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("src_slot", ctypes.c_void_p), ("dst_slots", ctypes.c_void_p),
        ("qkv", ctypes.c_void_p), ("qkv_row_stride", ctypes.c_int64),
        ("conv_weight", ctypes.c_void_p), ("conv_bias", ctypes.c_void_p),
        ("conv_state", ctypes.c_void_p), ("state", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("gate", ctypes.c_void_p),
        ("norm_weight", ctypes.c_void_p), ("out", ctypes.c_void_p), ("out_f64", ctypes.c_void_p),
        ("eps", ctypes.c_double), ("l2_eps", ctypes.c_double), ("q_scale", ctypes.c_double),
        ("out_norm", ctypes.c_int32), ("update_conv_state", ctypes.c_int32),
        ("fused_gate", ctypes.c_int32), ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("lower_bound", ctypes.c_double), ("conv_state_sd", ctypes.c_int32),
    ]


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            # KDA_ORACLE_SO points the pins at another build of the oracle
            # (the planted-mistake tests use it); normally unset.
            so = os.environ.get("KDA_ORACLE_SO") or build()
            L = ctypes.CDLL(so)
            dp = ctypes.POINTER(ctypes.c_double)
            L.kda_oracle_decode.argtypes = [ctypes.POINTER(_Problem), ctypes.c_int]
            L.kda_oracle_decode.restype = ctypes.c_int
            L.kda_oracle_problem_size.restype = ctypes.c_int
            L.kda_oracle_sigmoid.argtypes = [ctypes.c_double]
            L.kda_oracle_sigmoid.restype = ctypes.c_double
            L.kda_oracle_silu.argtypes = [ctypes.c_double]
            L.kda_oracle_silu.restype = ctypes.c_double
            L.kda_oracle_causal_conv.argtypes = [dp, dp, ctypes.c_int, ctypes.c_double]
            L.kda_oracle_causal_conv.restype = ctypes.c_double
            L.kda_oracle_l2norm.argtypes = [dp, ctypes.c_int, ctypes.c_double, ctypes.c_double, dp]
            L.kda_oracle_gated_delta_update.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp,
                                                        ctypes.c_double, dp, dp]
            L.kda_oracle_readout.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp, dp]
            L.kda_oracle_gated_rmsnorm.argtypes = [ctypes.c_int, dp, dp, dp, ctypes.c_double, dp]
            L.kda_oracle_softplus.argtypes = [ctypes.c_double]
            L.kda_oracle_softplus.restype = ctypes.c_double
            L.kda_oracle_kda_gate.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_double]
            L.kda_oracle_kda_gate.restype = ctypes.c_double
            L.kda_oracle_round_bf16.argtypes = [ctypes.c_double]
            L.kda_oracle_round_bf16.restype = ctypes.c_uint16
            L.kda_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.kda_oracle_bf16_to_f64.restype = ctypes.c_double
            L.kda_oracle_prefill.argtypes = [ctypes.POINTER(_PrefillProblem), ctypes.c_int]
            L.kda_oracle_prefill.restype = ctypes.c_int
            L.kda_oracle_prefill_problem_size.restype = ctypes.c_int
            L.kda_oracle_decode_multi.argtypes = [ctypes.POINTER(_MultiProblem), ctypes.c_int]
            L.kda_oracle_decode_multi.restype = ctypes.c_int
            L.kda_oracle_multi_problem_size.restype = ctypes.c_int
            if L.kda_oracle_multi_problem_size() != ctypes.sizeof(_MultiProblem):
                raise RuntimeError("oracle multi-token struct layout mismatch")
            if L.kda_oracle_problem_size() != ctypes.sizeof(_Problem):
                raise RuntimeError("oracle struct layout mismatch")
            if L.kda_oracle_prefill_problem_size() != ctypes.sizeof(_PrefillProblem):
                raise RuntimeError("oracle prefill struct layout mismatch")
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


# ------------------------------------------------------------ step functions

def sigmoid(x: float) -> float:
    return lib().kda_oracle_sigmoid(float(x))


def silu(y: float) -> float:
    return lib().kda_oracle_silu(float(y))


def causal_conv(x, w, bias: float = 0.0) -> float:
    x, w = _f64(x), _f64(w)
    assert x.shape == w.shape and x.ndim == 1
    return lib().kda_oracle_causal_conv(_dp(x), _dp(w), x.size, float(bias))


def l2norm(x, eps: float = 1e-6, scale: float = 1.0) -> np.ndarray:
    x = _f64(x)
    y = np.empty_like(x)
    lib().kda_oracle_l2norm(_dp(x), x.size, float(eps), float(scale), _dp(y))
    return y


def gated_delta_update(S, alpha, beta: float, k, v) -> np.ndarray:
    S = _f64(S).copy()
    K, V = S.shape
    alpha, k, v = _f64(alpha), _f64(k), _f64(v)
    assert alpha.shape == (K,) and k.shape == (K,) and v.shape == (V,)
    lib().kda_oracle_gated_delta_update(K, V, _dp(S), _dp(alpha), float(beta), _dp(k), _dp(v))
    return S


def readout(S, q) -> np.ndarray:
    S, q = _f64(S), _f64(q)
    K, V = S.shape
    o = np.empty(V)
    lib().kda_oracle_readout(K, V, _dp(S), _dp(q), _dp(o))
    return o


def gated_rmsnorm(o, w, gate, eps: float = 1e-6) -> np.ndarray:
    o, w, gate = _f64(o), _f64(w), _f64(gate)
    y = np.empty_like(o)
    lib().kda_oracle_gated_rmsnorm(o.size, _dp(o), _dp(w), _dp(gate), float(eps), _dp(y))
    return y


def softplus(z: float) -> float:
    return lib().kda_oracle_softplus(float(z))


def kda_gate(z: float, A_log: float, lower_bound: float = 0.0) -> float:
    return lib().kda_oracle_kda_gate(float(z), float(A_log), float(lower_bound))


def round_bf16(x: float) -> int:
    return int(lib().kda_oracle_round_bf16(float(x)))


def bf16_to_f64(b: int) -> float:
    return lib().kda_oracle_bf16_to_f64(int(b))


# ------------------------------------------------------------ whole step

@dataclass
class OracleResult:
    out: np.ndarray            # uint16 bf16 bits [N, H*V]
    out_f64: np.ndarray | None  # fp64 [N, H*V] before rounding
    conv_state: np.ndarray     # uint16 [slots, C, W-1] after the step
    state: np.ndarray          # float32 [slots, H, K, V] after the step
    n_out_of_range: int


def decode(*, qkv, conv_weight, conv_state, state, g, beta, slot_idx, H: int,
           K: int = 128, V: int = 128, W: int = 4, gate=None, norm_weight=None,
           conv_bias=None, eps: float = 1e-6, l2_eps: float = 1e-6, q_scale: float = 0.0,
           out_norm: bool = True, update_conv_state: bool = True, threads: int = 0,
           want_f64: bool = True, in_place: bool = False, fused_gate: bool = False,
           A_log=None, dt_bias=None, lower_bound: float = 0.0,
           conv_state_sd: bool = False) -> OracleResult:
    """One decode step over all rows.  ``conv_state``/``state`` are copied
    unless ``in_place``; the updated arrays come back in the result.  With
    ``fused_gate``, ``g`` and ``beta`` hold raw logits and are activated with
    ``A_log``, ``dt_bias`` and ``lower_bound``.  ``conv_state_sd``: the conv
    state is [slots, W-1, C] (tap-first) instead of [slots, C, W-1]."""
    qkv = np.ascontiguousarray(qkv, dtype=np.uint16)
    N = qkv.shape[0]
    C = 2 * H * K + H * V
    conv_weight = np.ascontiguousarray(conv_weight, dtype=np.float32)
    assert conv_weight.size == W * C, conv_weight.shape
    if in_place:
        assert conv_state.dtype == np.uint16 and conv_state.flags.c_contiguous
        assert state.dtype == np.float32 and state.flags.c_contiguous
        cs, st = conv_state, state
    else:
        cs = np.array(conv_state, dtype=np.uint16, order="C", copy=True)
        st = np.array(state, dtype=np.float32, order="C", copy=True)
    num_slots = st.shape[0]
    assert st.size == num_slots * H * K * V
    assert cs.size == num_slots * C * max(W - 1, 0) or W == 1
    g = np.ascontiguousarray(g, dtype=np.float32)
    beta = np.ascontiguousarray(beta, dtype=np.uint16)
    slot_idx = np.ascontiguousarray(slot_idx, dtype=np.int32)
    assert g.size == N * H * K and beta.size == N * H and slot_idx.size == N
    if out_norm:
        gate = np.ascontiguousarray(gate, dtype=np.uint16)
        norm_weight = np.ascontiguousarray(norm_weight, dtype=np.float32)
        assert gate.size == N * H * V and norm_weight.size == V
    else:
        gate = norm_weight = None
    if conv_bias is not None:
        conv_bias = np.ascontiguousarray(conv_bias, dtype=np.float32)
        assert conv_bias.size == C
    if fused_gate:
        A_log = np.ascontiguousarray(A_log, dtype=np.float32)
        assert A_log.size == H
        if dt_bias is not None:
            dt_bias = np.ascontiguousarray(dt_bias, dtype=np.float32)
            assert dt_bias.size == H * K
    else:
        A_log = dt_bias = None
    out = np.zeros((N, H * V), dtype=np.uint16)
    out64 = np.zeros((N, H * V), dtype=np.float64) if want_f64 else None
    p = _Problem(N=N, H=H, K=K, V=V, W=W, num_slots=num_slots,
                 qkv=_ptr(qkv), qkv_row_stride=qkv.shape[1] if qkv.ndim == 2 else C,
                 conv_weight=_ptr(conv_weight), conv_bias=_ptr(conv_bias),
                 conv_state=_ptr(cs), state=_ptr(st), g=_ptr(g), beta=_ptr(beta),
                 gate=_ptr(gate), norm_weight=_ptr(norm_weight), slot_idx=_ptr(slot_idx),
                 out=_ptr(out), out_f64=_ptr(out64), eps=eps, l2_eps=l2_eps,
                 q_scale=q_scale, out_norm=int(bool(out_norm)),
                 update_conv_state=int(bool(update_conv_state)), fused_gate=int(bool(fused_gate)),
                 A_log=_ptr(A_log), dt_bias=_ptr(dt_bias), lower_bound=float(lower_bound),
                 conv_state_sd=int(bool(conv_state_sd)))
    rc = lib().kda_oracle_decode(ctypes.byref(p), int(threads))
    if rc < 0:
        raise ValueError("kda_oracle_decode rejected its arguments")
    return OracleResult(out=out, out_f64=out64, conv_state=cs, state=st, n_out_of_range=rc)


def prefill(*, qkv, conv_weight, conv_state, state, g, beta, slot_idx, cu_seqlens, H: int,
            K: int = 128, V: int = 128, W: int = 4, gate=None, norm_weight=None,
            conv_bias=None, eps: float = 1e-6, l2_eps: float = 1e-6, q_scale: float = 0.0,
            out_norm: bool = True, threads: int = 0, want_f64: bool = True,
            in_place: bool = False, fused_gate: bool = False, A_log=None, dt_bias=None,
            lower_bound: float = 0.0, conv_state_sd: bool = False) -> OracleResult:
    """Prefill of a varlen batch: every sequence's tokens run through the
    decode steps in order (window and state carried along, state never
    rounded in between); final state and conv window stored to the
    sequence's slot.  With ``fused_gate``, ``g`` and ``beta`` hold raw
    logits activated with ``A_log``, ``dt_bias`` and ``lower_bound``;
    ``conv_state_sd``: the conv state is [slots, W-1, C] (tap-first).  ``slot_idx`` has one entry per sequence; ``qkv``, ``g``,
    ``beta``, ``gate`` one row per token.  Pools are copied unless
    ``in_place``."""
    qkv = np.ascontiguousarray(qkv, dtype=np.uint16)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    B = cu.size - 1
    T = int(cu[-1]) if B > 0 else 0
    C = 2 * H * K + H * V
    conv_weight = np.ascontiguousarray(conv_weight, dtype=np.float32)
    assert conv_weight.size == W * C
    if in_place:
        assert conv_state.dtype == np.uint16 and conv_state.flags.c_contiguous
        assert state.dtype == np.float32 and state.flags.c_contiguous
        cs, st = conv_state, state
    else:
        cs = np.array(conv_state, dtype=np.uint16, order="C", copy=True)
        st = np.array(state, dtype=np.float32, order="C", copy=True)
    num_slots = st.shape[0]
    g = np.ascontiguousarray(g, dtype=np.float32)
    beta = np.ascontiguousarray(beta, dtype=np.uint16)
    slot_idx = np.ascontiguousarray(slot_idx, dtype=np.int32)
    assert qkv.shape[0] >= T and g.size >= T * H * K and beta.size >= T * H and slot_idx.size == B
    if out_norm:
        gate = np.ascontiguousarray(gate, dtype=np.uint16)
        norm_weight = np.ascontiguousarray(norm_weight, dtype=np.float32)
        assert gate.size >= T * H * V and norm_weight.size == V
    else:
        gate = norm_weight = None
    if conv_bias is not None:
        conv_bias = np.ascontiguousarray(conv_bias, dtype=np.float32)
    if fused_gate:
        A_log = np.ascontiguousarray(A_log, dtype=np.float32)
        assert A_log.size == H
        if dt_bias is not None:
            dt_bias = np.ascontiguousarray(dt_bias, dtype=np.float32)
            assert dt_bias.size == H * K
    else:
        A_log = dt_bias = None
    out = np.zeros((T, H * V), dtype=np.uint16)
    out64 = np.zeros((T, H * V), dtype=np.float64) if want_f64 else None
    p = _PrefillProblem(B=B, H=H, K=K, V=V, W=W, num_slots=num_slots, cu_seqlens=_ptr(cu),
                        qkv=_ptr(qkv), qkv_row_stride=qkv.shape[1] if qkv.ndim == 2 else C,
                        conv_weight=_ptr(conv_weight), conv_bias=_ptr(conv_bias),
                        conv_state=_ptr(cs), state=_ptr(st), g=_ptr(g), beta=_ptr(beta),
                        gate=_ptr(gate), norm_weight=_ptr(norm_weight), slot_idx=_ptr(slot_idx),
                        out=_ptr(out), out_f64=_ptr(out64), eps=eps, l2_eps=l2_eps,
                        q_scale=q_scale, out_norm=int(bool(out_norm)), fused_gate=int(bool(fused_gate)),
                        A_log=_ptr(A_log), dt_bias=_ptr(dt_bias), lower_bound=float(lower_bound),
                        conv_state_sd=int(bool(conv_state_sd)))
    rc = lib().kda_oracle_prefill(ctypes.byref(p), int(threads))
    if rc < 0:
        raise ValueError("kda_oracle_prefill rejected its arguments")
    return OracleResult(out=out, out_f64=out64, conv_state=cs, state=st, n_out_of_range=rc)


def decode_multi(*, qkv, conv_weight, conv_state, state, g, beta, src_slot, dst_slots, H: int,
                 K: int = 128, V: int = 128, W: int = 4, gate=None, norm_weight=None,
                 conv_bias=None, eps: float = 1e-6, l2_eps: float = 1e-6, q_scale: float = 0.0,
                 out_norm: bool = True, update_conv_state: bool = True, threads: int = 0,
                 want_f64: bool = True, in_place: bool = False, fused_gate: bool = False,
                 A_log=None, dt_bias=None, lower_bound: float = 0.0,
                 conv_state_sd: bool = False) -> OracleResult:
    """Multi-token (speculative) decode: sequence n starts from the window and
    state in ``src_slot[n]`` and runs its T tokens (rows n*T + t of ``qkv``,
    ``g``, ``beta``, ``gate``) in order; the state and window after token t go
    to ``dst_slots[n, t]`` (an entry <= 0 marks an absent token).  ``dst_slots``
    is [N, T].  Pools are copied unless ``in_place``."""
    dst = np.ascontiguousarray(dst_slots, dtype=np.int32)
    assert dst.ndim == 2
    N, T = dst.shape
    src = np.ascontiguousarray(src_slot, dtype=np.int32)
    assert src.shape == (N,)
    qkv = np.ascontiguousarray(qkv, dtype=np.uint16)
    C = 2 * H * K + H * V
    assert qkv.shape[0] == N * T
    conv_weight = np.ascontiguousarray(conv_weight, dtype=np.float32)
    assert conv_weight.size == W * C
    if in_place:
        assert conv_state.dtype == np.uint16 and conv_state.flags.c_contiguous
        assert state.dtype == np.float32 and state.flags.c_contiguous
        cs, st = conv_state, state
    else:
        cs = np.array(conv_state, dtype=np.uint16, order="C", copy=True)
        st = np.array(state, dtype=np.float32, order="C", copy=True)
    num_slots = st.shape[0]
    g = np.ascontiguousarray(g, dtype=np.float32)
    beta = np.ascontiguousarray(beta, dtype=np.uint16)
    assert g.size == N * T * H * K and beta.size == N * T * H
    if out_norm:
        gate = np.ascontiguousarray(gate, dtype=np.uint16)
        norm_weight = np.ascontiguousarray(norm_weight, dtype=np.float32)
        assert gate.size == N * T * H * V and norm_weight.size == V
    else:
        gate = norm_weight = None
    if conv_bias is not None:
        conv_bias = np.ascontiguousarray(conv_bias, dtype=np.float32)
        assert conv_bias.size == C
    if fused_gate:
        A_log = np.ascontiguousarray(A_log, dtype=np.float32)
        assert A_log.size == H
        if dt_bias is not None:
            dt_bias = np.ascontiguousarray(dt_bias, dtype=np.float32)
            assert dt_bias.size == H * K
    else:
        A_log = dt_bias = None
    out = np.zeros((N * T, H * V), dtype=np.uint16)
    out64 = np.zeros((N * T, H * V), dtype=np.float64) if want_f64 else None
    p = _MultiProblem(N=N, T=T, H=H, K=K, V=V, W=W, num_slots=num_slots, src_slot=_ptr(src),
                      dst_slots=_ptr(dst), qkv=_ptr(qkv),
                      qkv_row_stride=qkv.shape[1] if qkv.ndim == 2 else C,
                      conv_weight=_ptr(conv_weight), conv_bias=_ptr(conv_bias),
                      conv_state=_ptr(cs), state=_ptr(st), g=_ptr(g), beta=_ptr(beta),
                      gate=_ptr(gate), norm_weight=_ptr(norm_weight),
                      out=_ptr(out), out_f64=_ptr(out64), eps=eps, l2_eps=l2_eps,
                      q_scale=q_scale, out_norm=int(bool(out_norm)),
                      update_conv_state=int(bool(update_conv_state)), fused_gate=int(bool(fused_gate)),
                      A_log=_ptr(A_log), dt_bias=_ptr(dt_bias), lower_bound=float(lower_bound),
                      conv_state_sd=int(bool(conv_state_sd)))
    rc = lib().kda_oracle_decode_multi(ctypes.byref(p), int(threads))
    if rc < 0:
        raise ValueError("kda_oracle_decode_multi rejected its arguments")
    return OracleResult(out=out, out_f64=out64, conv_state=cs, state=st, n_out_of_range=rc)
