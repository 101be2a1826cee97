"""Seeded synthetic inputs for the fused KDA decode step and the varlen prefill.

This module only draws random numbers and lays them out in the storage
dtypes and shapes of the decode step (one row per sequence) and of the
prefill (one row per token, sequences given by their lengths); it holds none
of the method's arithmetic.
Both the CUDA path (through the tests and the benchmark) and the fp64 oracle
consume the same arrays it returns.

bf16 tensors are returned as numpy ``uint16`` bit patterns (round-to-nearest-
even from the fp32 draw).  Every tensor has its own seed stream
``SeedSequence([seed, tag, ...])``; the recurrent and conv state pools are
drawn slot by slot (``SeedSequence([seed, tag, slot])``), so any slot can be
regenerated on its own and large pools can be drawn by several threads.

Value distributions (sigma is the standard deviation):
  mixed qkv      bf16  N(0, 1)                      [N, 3*H*128]
  conv weight    fp32  N(0, 0.5)                    [3, 4, H*128] width-major
  conv state     bf16  N(0, 1)                      [slots, 3*H*128, 3]
  state          fp32  N(0, 0.02)                   [slots, H, 128, 128]
  g (log-decay)  fp32  -softplus(N(0, 1))           [N, H, 128]
                  or   -5 * (1 - U[0,1))  (decays in [exp(-5), 1))
  beta           bf16  sigmoid(N(0, 1))             [N, H]
  output gate    bf16  N(0, 1)                      [N, H*128]
  norm weight    fp32  1 + N(0, 0.1)                [128]
  slot indices   int32 distinct draws from 1..slots-1, padding rows 0
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field, replace

import numpy as np

HEAD_DIM = 128
CONV_WIDTH = 4

# seed-stream tags, one per tensor
_T_QKV, _T_CW, _T_CS, _T_STATE, _T_G, _T_BETA, _T_GATE, _T_NW, _T_SLOT, _T_BIAS = range(1, 11)


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Spec:
    """One synthetic decode-step problem."""
    name: str
    N: int
    H: int
    num_slots: int
    seed: int
    out_norm: bool = True
    update_conv_state: bool = True
    pad_tail: int = 0                 # last rows set to slot 0
    slots: tuple | None = None        # explicit slot list overrides the draw
    g_mode: str = "softplus"          # "softplus" | "uniform5"
    eps: float = 1e-6
    with_bias: bool = False
    qkv_row_pad: int = 0              # extra bf16 elements per qkv row


# The workloads the decode step is measured and checked on.
PR1_REF = Spec("n4_h12_pool8", N=4, H=12, num_slots=8, seed=0, slots=(1, 3, 5, 7))
PAD_TAIL = Spec("n32_h24_pool64_pad8", N=32, H=24, num_slots=64, seed=1, pad_tail=8)
NORM_OFF = Spec("n128_h48_pool512_normoff", N=128, H=48, num_slots=512, seed=2,
                out_norm=False, g_mode="uniform5")
ROOFLINE = Spec("n256_h96_pool1024", N=256, H=96, num_slots=1024, seed=3)
# 69 independent layers, each its own weights and state pool.
STACK_LAYERS = 69
STACK_LAYER = Spec("stack69_n64_h48_pool96_pad4", N=64, H=48, num_slots=96, seed=4000, pad_tail=4)

SPECS = {s.name: s for s in (PR1_REF, PAD_TAIL, NORM_OFF, ROOFLINE)}


def stack_layer_spec(layer: int) -> Spec:
    return replace(STACK_LAYER, seed=STACK_LAYER.seed + layer)


@dataclass
class Inputs:
    """Host arrays of one problem (bf16 as uint16 bits)."""
    spec: Spec
    qkv: np.ndarray
    conv_weight: np.ndarray
    conv_bias: np.ndarray | None
    conv_state: np.ndarray
    state: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    gate: np.ndarray
    norm_weight: np.ndarray
    slot_idx: np.ndarray
    extra: dict = field(default_factory=dict)

    @property
    def N(self) -> int: return self.spec.N

    @property
    def H(self) -> int: return self.spec.H

    @property
    def C(self) -> int: return 3 * self.spec.H * HEAD_DIM

    def active_rows(self) -> np.ndarray:
        s = self.slot_idx
        return np.nonzero((s > 0) & (s < self.spec.num_slots))[0]


def draw_slots(spec: Spec) -> np.ndarray:
    if spec.slots is not None:
        s = np.asarray(spec.slots, dtype=np.int32)
        assert s.size == spec.N
        return s
    n_act = spec.N - spec.pad_tail
    assert 0 <= n_act <= spec.num_slots - 1, "not enough distinct slots"
    perm = _rng(spec.seed, _T_SLOT).permutation(np.arange(1, spec.num_slots, dtype=np.int32))
    s = np.zeros(spec.N, dtype=np.int32)
    s[:n_act] = perm[:n_act]
    return s


def _fill_pool(shape_per_slot, num_slots, seed, tag, sigma, dtype_out, threads):
    """Draw a [num_slots, *shape_per_slot] pool slot by slot (one seed stream per slot)."""
    out_dtype = np.float32 if dtype_out == "f32" else np.uint16
    pool = np.empty((num_slots,) + tuple(shape_per_slot), dtype=out_dtype)

    def one(slot):
        x = _rng(seed, tag, slot).standard_normal(shape_per_slot, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        pool[slot] = x if dtype_out == "f32" else f32_to_bf16_bits(x)

    if threads <= 1 or num_slots < 8:
        for s in range(num_slots):
            one(s)
    else:
        with _cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(num_slots)))
    return pool


def draw_step_inputs(spec: Spec, variant: int = 0) -> dict:
    """Per-token inputs (qkv, g, beta, gate) of one step; ``variant`` selects
    another independent draw with the same distributions."""
    N, H, D = spec.N, spec.H, spec.H * HEAD_DIM
    key = (spec.seed,) if variant == 0 else (spec.seed, 1000 + variant)
    qkv = f32_to_bf16_bits(_rng(*key, _T_QKV).standard_normal((N, 3 * D + spec.qkv_row_pad),
                                                               dtype=np.float32))
    if spec.g_mode == "softplus":
        z = _rng(*key, _T_G).standard_normal((N, H, HEAD_DIM))
        g = (-np.logaddexp(0.0, z)).astype(np.float32)
    elif spec.g_mode == "uniform5":
        u = _rng(*key, _T_G).random((N, H, HEAD_DIM))
        g = (-5.0 * (1.0 - u)).astype(np.float32)
    else:
        raise ValueError(spec.g_mode)
    zb = _rng(*key, _T_BETA).standard_normal((N, H))
    beta = f32_to_bf16_bits((1.0 / (1.0 + np.exp(-zb))).astype(np.float32))
    gate = f32_to_bf16_bits(_rng(*key, _T_GATE).standard_normal((N, D), dtype=np.float32))
    return dict(qkv=qkv, g=g, beta=beta, gate=gate)


def make_inputs(spec: Spec, threads: int | None = None) -> Inputs:
    """Draw every tensor of ``spec``."""
    if threads is None:
        threads = min(16, os.cpu_count() or 1)
    H, D = spec.H, spec.H * HEAD_DIM
    C = 3 * D
    step = draw_step_inputs(spec, 0)
    cw = _rng(spec.seed, _T_CW).standard_normal((3, CONV_WIDTH, D), dtype=np.float32)
    cw *= np.float32(0.5)
    bias = None
    if spec.with_bias:
        bias = _rng(spec.seed, _T_BIAS).standard_normal(C, dtype=np.float32) * np.float32(0.1)
    cs = _fill_pool((C, CONV_WIDTH - 1), spec.num_slots, spec.seed, _T_CS, 1.0, "bf16", threads)
    st = _fill_pool((H, HEAD_DIM, HEAD_DIM), spec.num_slots, spec.seed, _T_STATE, 0.02, "f32",
                    threads)
    nw = (1.0 + 0.1 * _rng(spec.seed, _T_NW).standard_normal(HEAD_DIM)).astype(np.float32)
    return Inputs(spec=spec, qkv=step["qkv"], conv_weight=cw, conv_bias=bias, conv_state=cs,
                  state=st, g=step["g"], beta=step["beta"], gate=step["gate"],
                  norm_weight=nw, slot_idx=draw_slots(spec))


# ------------------------------------------------- multi-token (speculative)

@dataclass(frozen=True)
class MultiSpec:
    """One synthetic multi-token (speculative) decode batch: N sequences of
    T = 1 + num_spec tokens, with the decode step's value distributions, one
    row per token.  Slots: N distinct source slots, then N*T distinct
    destination slots, all drawn from 1..slots-1 without repetition.
    ``pad_seqs`` get source slot 0; ``absent`` lists (n, t) tokens whose
    destination is 0; ``alias_last`` stores each sequence's last token back
    into its own source slot."""
    name: str
    N: int
    T: int
    H: int
    num_slots: int
    seed: int
    out_norm: bool = True
    update_conv_state: bool = True
    pad_seqs: tuple = ()
    absent: tuple = ()
    alias_last: bool = False
    g_mode: str = "softplus"
    eps: float = 1e-6

    def rows_spec(self) -> Spec:
        """The per-token draw as a decode Spec with N*T rows."""
        return Spec(self.name, N=self.N * self.T, H=self.H, num_slots=self.num_slots, seed=self.seed,
                    out_norm=self.out_norm, update_conv_state=self.update_conv_state,
                    slots=(0,) * (self.N * self.T), g_mode=self.g_mode, eps=self.eps)


@dataclass
class MultiInputs:
    spec: MultiSpec
    qkv: np.ndarray          # uint16 [N*T, 3D]
    conv_weight: np.ndarray  # f32 [3, 4, D]
    conv_state: np.ndarray   # uint16 [slots, 3D, 3]
    state: np.ndarray        # f32 [slots, H, 128, 128]
    g: np.ndarray            # f32 [N*T, H, 128]
    beta: np.ndarray         # uint16 [N*T, H]
    gate: np.ndarray         # uint16 [N*T, D]
    norm_weight: np.ndarray  # f32 [128]
    src_slot: np.ndarray     # int32 [N]
    dst_slots: np.ndarray    # int32 [N, T]
    conv_bias: np.ndarray | None = None

    @property
    def N(self) -> int: return self.spec.N

    @property
    def T(self) -> int: return self.spec.T

    @property
    def H(self) -> int: return self.spec.H


_T_MULTI = 200  # seed-stream tag of the multi-token slot draw


def make_multi_inputs(spec: MultiSpec, threads: int | None = None) -> MultiInputs:
    x = make_inputs(spec.rows_spec(), threads)
    N, T = spec.N, spec.T
    need = N + N * T
    assert need <= spec.num_slots - 1, "not enough distinct slots"
    perm = _rng(spec.seed, _T_MULTI).permutation(np.arange(1, spec.num_slots, dtype=np.int32))
    src = perm[:N].copy()
    dst = perm[N:need].reshape(N, T).copy()
    if spec.alias_last:
        dst[:, T - 1] = src
    for n, t in spec.absent:
        dst[n, t] = 0
    for n in spec.pad_seqs:
        src[n] = 0
    return MultiInputs(spec=spec, qkv=x.qkv, conv_weight=x.conv_weight, conv_state=x.conv_state,
                       state=x.state, g=x.g, beta=x.beta, gate=x.gate, norm_weight=x.norm_weight,
                       src_slot=src, dst_slots=dst)


def multi_algorithmic_bytes(spec: MultiSpec, src_slot: np.ndarray, dst_slots: np.ndarray) -> int:
    """Bytes one multi-token launch must move at minimum: per active
    (sequence, head) the source state and window read once, and per present
    token its state (and, with the flag, window) written, its q/k/v inputs,
    g, beta, gate and output; per zero output row (padding sequence or
    absent token) 256 B per head; per launch the conv weight, norm weight and
    slot indices."""
    K = V = HEAD_DIM
    H = spec.H
    valid = lambda s: 0 < s < spec.num_slots  # noqa: E731
    per_tok = 3 * K * 2 + K * 4 + 2 + V * 2 + (V * 2 if spec.out_norm else 0) + K * V * 4 \
        + (3 * K * 3 * 2 if spec.update_conv_state else 0)
    per_src = K * V * 4 + 3 * K * 3 * 2
    total = 0
    for n in range(spec.N):
        present = [t for t in range(spec.T) if valid(src_slot[n]) and valid(dst_slots[n, t])]
        if present:
            total += per_src + len(present) * per_tok
        total += (spec.T - len(present)) * V * 2
    fixed = 3 * CONV_WIDTH * H * K * 4 + (V * 4 if spec.out_norm else 0) + 4 * spec.N * (spec.T + 1)
    return H * total + fixed


# The measured multi-token batch: the stack layer's shape with three draft
# tokens per sequence (T = 4), 60 sequences and 4 padding sequences.
MULTI_BENCH = MultiSpec("spec_n64_t4_h48_pool336_pad4", N=64, T=4, H=48, num_slots=336, seed=300,
                        pad_seqs=(60, 61, 62, 63))


# ----------------------------------------------------------------- prefill

_T_PREFILL = 100  # seed-stream tags of the prefill inputs start here


@dataclass(frozen=True)
class PrefillSpec:
    """One synthetic varlen prefill batch: ``lens`` tokens per sequence (0 =
    empty sequence); sequences listed in ``pad_seqs`` get slot 0 (padding).
    Same value distributions as the decode step, one row per token; ``g_mode``
    "uniform20" draws g = -20 (1 - U) (decays down to e^-20 per token)."""
    name: str
    lens: tuple
    H: int
    num_slots: int
    seed: int
    out_norm: bool = True
    pad_seqs: tuple = ()
    g_mode: str = "softplus"          # "softplus" | "uniform5" | "uniform20"
    eps: float = 1e-6
    with_bias: bool = False

    @property
    def B(self) -> int: return len(self.lens)

    @property
    def T(self) -> int: return int(sum(self.lens))


# Ragged lengths: partial chunks, exact multiples of the 32-token chunk, a
# one-token and an empty sequence, a padding sequence.
PREFILL_SMALL = PrefillSpec("prefill_b6_h3_pool12", lens=(37, 1, 0, 64, 5, 96), H=3, num_slots=12,
                            seed=50, pad_seqs=(4,), with_bias=True)
PREFILL_NORM_OFF = PrefillSpec("prefill_b2_h2_pool6_normoff", lens=(70, 33), H=2, num_slots=6, seed=51,
                               out_norm=False, g_mode="uniform5")
PREFILL_STRONG_DECAY = PrefillSpec("prefill_b2_h2_pool5_decay20", lens=(45, 96), H=2, num_slots=5,
                                   seed=52, g_mode="uniform20")
# The measured prefill batch: 16 sequences, 16,384 tokens, H = 48.
PREFILL_BENCH = PrefillSpec("prefill_b16_t16384_h48_pool64",
                            lens=(2900, 1, 1800, 417, 64, 2048, 999, 17, 1500, 700, 2345, 100, 33,
                                  1210, 230, 2020),
                            H=48, num_slots=64, seed=53)
# A quarter of that for profiler captures: 4 sequences, 4,096 tokens, H = 48
# (inputs and workspace still larger than L2, under 1 GB on the device).
PREFILL_PROFILE = PrefillSpec("prefill_b4_t4096_h48_pool16", lens=(1500, 1024, 900, 672), H=48,
                              num_slots=16, seed=54)


@dataclass
class PrefillInputs:
    spec: PrefillSpec
    qkv: np.ndarray          # uint16 [T, 3D]
    conv_weight: np.ndarray  # f32 [3, 4, D]
    conv_bias: np.ndarray | None
    conv_state: np.ndarray   # uint16 [slots, 3D, 3]
    state: np.ndarray        # f32 [slots, H, 128, 128]
    g: np.ndarray            # f32 [T, H, 128]
    beta: np.ndarray         # uint16 [T, H]
    gate: np.ndarray         # uint16 [T, D]
    norm_weight: np.ndarray  # f32 [128]
    slot_idx: np.ndarray     # int32 [B]
    cu_seqlens: np.ndarray   # int32 [B + 1]


def make_prefill_inputs(spec: PrefillSpec, threads: int | None = None) -> PrefillInputs:
    if threads is None:
        threads = min(16, os.cpu_count() or 1)
    H, D, T, B = spec.H, spec.H * HEAD_DIM, spec.T, spec.B
    C = 3 * D
    base = _T_PREFILL
    qkv = f32_to_bf16_bits(_rng(spec.seed, base + _T_QKV).standard_normal((T, C), dtype=np.float32))
    if spec.g_mode == "softplus":
        g = (-np.logaddexp(0.0, _rng(spec.seed, base + _T_G).standard_normal((T, H, HEAD_DIM)))).astype(np.float32)
    elif spec.g_mode in ("uniform5", "uniform20"):
        a = 5.0 if spec.g_mode == "uniform5" else 20.0
        g = (-a * (1.0 - _rng(spec.seed, base + _T_G).random((T, H, HEAD_DIM)))).astype(np.float32)
    else:
        raise ValueError(spec.g_mode)
    zb = _rng(spec.seed, base + _T_BETA).standard_normal((T, H))
    beta = f32_to_bf16_bits((1.0 / (1.0 + np.exp(-zb))).astype(np.float32))
    gate = f32_to_bf16_bits(_rng(spec.seed, base + _T_GATE).standard_normal((T, D), dtype=np.float32))
    cw = _rng(spec.seed, base + _T_CW).standard_normal((3, CONV_WIDTH, D), dtype=np.float32) * np.float32(0.5)
    bias = None
    if spec.with_bias:
        bias = _rng(spec.seed, base + _T_BIAS).standard_normal(C, dtype=np.float32) * np.float32(0.1)
    cs = _fill_pool((C, CONV_WIDTH - 1), spec.num_slots, spec.seed, base + _T_CS, 1.0, "bf16", threads)
    st = _fill_pool((H, HEAD_DIM, HEAD_DIM), spec.num_slots, spec.seed, base + _T_STATE, 0.02, "f32", threads)
    nw = (1.0 + 0.1 * _rng(spec.seed, base + _T_NW).standard_normal(HEAD_DIM)).astype(np.float32)
    assert B <= spec.num_slots - 1, "not enough distinct slots"
    perm = _rng(spec.seed, base + _T_SLOT).permutation(np.arange(1, spec.num_slots, dtype=np.int32))
    slots = perm[:B].copy()
    for b in spec.pad_seqs:
        slots[b] = 0
    cu = np.concatenate([[0], np.cumsum(spec.lens)]).astype(np.int32)
    return PrefillInputs(spec=spec, qkv=qkv, conv_weight=cw, conv_bias=bias, conv_state=cs, state=st,
                         g=g, beta=beta, gate=gate, norm_weight=nw, slot_idx=slots, cu_seqlens=cu)


def prefill_algorithmic_bytes(spec: PrefillSpec) -> int:
    """Bytes a prefill launch must move at minimum: per token of an active
    sequence and head its q/k/v inputs, g, beta, gate (norm on) and output;
    per token of a padding sequence its zeroed output; per active (sequence,
    head) the state read and write and the conv state read and write; the
    conv weights, norm weight, slots and sequence starts once."""
    K = V = HEAD_DIM
    H = spec.H
    per_tok = 3 * K * 2 + K * 4 + 2 + V * 2 + (V * 2 if spec.out_norm else 0)
    per_seq_head = 2 * K * V * 4 + 2 * 3 * K * 3 * 2
    act = [n for b, n in enumerate(spec.lens) if b not in spec.pad_seqs and n > 0]
    pad_tokens = sum(n for b, n in enumerate(spec.lens) if b in spec.pad_seqs)
    fixed = 3 * CONV_WIDTH * H * K * 4 + (V * 4 if spec.out_norm else 0) + 4 * spec.B + 4 * (spec.B + 1)
    return H * (sum(act) * per_tok + len(act) * per_seq_head + pad_tokens * V * 2) + fixed


def prefill_algorithmic_flops(spec: PrefillSpec, chunk: int = 32) -> int:
    """Dense-contraction FLOPs of the chunked form per active (sequence, head),
    counted once (2 per multiply-add): for each chunk of c tokens
    W S0 and Q_G S0 (c x 128 x 128 each), K_E^T Delta (128 x c x 128),
    R Delta (c x c x 128), P and R (c x c x 128 each)."""
    K = HEAD_DIM
    total = 0
    for b, n in enumerate(spec.lens):
        if b in spec.pad_seqs or n == 0:
            continue
        for t0 in range(0, n, chunk):
            c = min(chunk, n - t0)
            total += 2 * (3 * c * K * K + 3 * c * c * K)
    return spec.H * total


def algorithmic_bytes(N: int, H: int, n_active_rows: int, out_norm: bool = True) -> int:
    """Bytes one decode launch must move at minimum (DRAM or L2), counting
    each tensor once: per active (row, head) the fp32 state read and write
    (2 * 64 KiB), its q/k/v inputs, conv-state read and write, g, beta, gate
    and output; per padding (row, head) its zeroed output; per launch the conv
    weight, norm weight and slot indices."""
    K = V = HEAD_DIM
    per_active = (2 * K * V * 4          # state read + write
                  + 3 * K * 2            # qkv slice
                  + 2 * 3 * K * 3 * 2    # conv state read + write
                  + K * 4                # g
                  + 2                    # beta
                  + V * 2)               # out
    if out_norm:
        per_active += V * 2              # gate
    per_pad = V * 2
    fixed = 3 * CONV_WIDTH * H * K * 4 + 4 * N
    if out_norm:
        fixed += V * 4
    n_pad = N - n_active_rows
    return H * (n_active_rows * per_active + n_pad * per_pad) + fixed
