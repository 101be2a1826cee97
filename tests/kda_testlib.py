"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the binding, run the oracle on the same inputs, and
compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from linear_attention_decode_04_gb300 import kda_decode
from linear_attention_decode_04_gb300 import workloads as W

# Tolerances of the decode step:
STATE_ATOL = 1e-4        # recurrent state: |d| <= 1e-4 + 1e-4 |ref|
STATE_RTOL = 1e-4
OUT_ATOL = 3e-2          # bf16 output: |d| <= 3e-2 (the pages' tolerance)
# A tighter bound the fp32 kernel meets: within one bf16 ulp of the exact
# (fp64) output, plus 1e-5 absolute for outputs near zero.
TIGHT_ABS = 1e-5


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def to_device(x: W.Inputs, device, out_row_pad: int = 0, gate_row_pad: int = 0) -> dict:
    d = dict(
        qkv=bf16_tensor(x.qkv, device),
        conv_weight=torch.from_numpy(x.conv_weight).to(device),
        conv_state=bf16_tensor(x.conv_state, device),
        state=torch.from_numpy(x.state).to(device),
        g=torch.from_numpy(x.g).to(device),
        beta=bf16_tensor(x.beta, device),
        slot_idx=torch.from_numpy(x.slot_idx).to(device),
        norm_weight=torch.from_numpy(x.norm_weight).to(device),
        conv_bias=None if x.conv_bias is None else torch.from_numpy(x.conv_bias).to(device),
    )
    D = x.H * W.HEAD_DIM
    if gate_row_pad:
        gate = np.zeros((x.N, D + gate_row_pad), np.uint16)
        gate[:, :D] = x.gate
        d["gate"] = bf16_tensor(gate, device)[:, :D]
    else:
        d["gate"] = bf16_tensor(x.gate, device)
    # NaN-filled so that any element the kernel fails to write is caught
    d["out_full"] = torch.full((x.N, D + out_row_pad), float("nan"), dtype=torch.bfloat16,
                               device=device)
    d["out"] = d["out_full"][:, :D]
    d["err_flag"] = torch.zeros(1, dtype=torch.int32, device=device)
    return d


def run_gpu(x: W.Inputs, d: dict, out_norm=None, update_conv_state=None, q_scale=0.0,
            early_prefetch=False, work_queue=None):
    out_norm = x.spec.out_norm if out_norm is None else out_norm
    upd = x.spec.update_conv_state if update_conv_state is None else update_conv_state
    kda_decode(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"],
               d["slot_idx"], d["out"], gate=d["gate"], norm_weight=d["norm_weight"],
               conv_bias=d["conv_bias"], eps=x.spec.eps, q_scale=q_scale, out_norm=out_norm,
               update_conv_state=upd, err_flag=d["err_flag"], early_prefetch=early_prefetch,
               work_queue=work_queue)


def run_oracle(x: W.Inputs, out_norm=None, update_conv_state=None, q_scale=0.0, in_place=False):
    out_norm = x.spec.out_norm if out_norm is None else out_norm
    upd = x.spec.update_conv_state if update_conv_state is None else update_conv_state
    return oracle.decode(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=x.conv_state,
                         state=x.state, g=x.g, beta=x.beta, slot_idx=x.slot_idx, H=x.H,
                         gate=x.gate, norm_weight=x.norm_weight, conv_bias=x.conv_bias,
                         eps=x.spec.eps, q_scale=q_scale, out_norm=out_norm,
                         update_conv_state=upd, in_place=in_place)


def bf16_ulp(y: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(y), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def check_out(gpu_bits: np.ndarray, ref: oracle.OracleResult, what: str = "out"):
    got = W.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    want = W.bf16_bits_to_f32(ref.out).astype(np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU output"
    err = np.abs(got - want)
    assert err.max(initial=0.0) <= OUT_ATOL, f"{what}: max |d| {err.max()} > {OUT_ATOL}"
    exact = ref.out_f64
    tight = np.abs(got - exact) <= bf16_ulp(exact) + TIGHT_ABS
    assert tight.all(), (f"{what}: {np.count_nonzero(~tight)} outputs further than one bf16 ulp "
                         f"from the exact value; worst {np.abs(got - exact).max()}")
    return float(err.max(initial=0.0))


def check_state_slot(got: np.ndarray, want: np.ndarray, what: str):
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    lim = STATE_ATOL + STATE_RTOL * np.abs(want.astype(np.float64))
    assert np.all(err <= lim), f"{what}: state |d| max {err.max()} beyond 1e-4 + 1e-4|ref|"
    return float(err.max(initial=0.0))


def compare_all(x: W.Inputs, d: dict, ref: oracle.OracleResult, init_state: np.ndarray | None = None,
                init_conv: np.ndarray | None = None) -> dict:
    """Output within tolerance; conv state bit-exact over the whole pool;
    state within tolerance on touched slots and bit-exact on all others."""
    out_err = check_out(bf16_bits(d["out"]), ref)
    cs = bf16_bits(d["conv_state"])
    assert np.array_equal(cs, ref.conv_state), "conv state not bit-exact"
    st = d["state"]
    active = set(int(s) for s in x.slot_idx if 0 < s < x.spec.num_slots)
    worst = 0.0
    for s in range(x.spec.num_slots):
        got = st[s].cpu().numpy()
        if s in active:
            worst = max(worst, check_state_slot(got, ref.state[s], f"slot {s}"))
        else:
            assert np.array_equal(got, ref.state[s]), f"untouched slot {s} changed"
            if init_state is not None:
                assert np.array_equal(got, init_state[s])
    if init_conv is not None:
        for s in range(x.spec.num_slots):
            if s not in active:
                assert np.array_equal(cs[s], init_conv[s])
    return dict(out_max_abs=out_err, state_max_abs=worst)


def cancellation_inputs(sigma: float, v_scale: float, seed: int = 5, N: int = 6, H: int = 4,
                        out_norm: bool = True) -> W.Inputs:
    """A decode step whose readout is far smaller than the matvec it comes
    from.  The q and k channels get identical conv weights, taps and inputs
    (so q~ = k~ exactly), beta = 1, g = 0, the state is scaled to N(0, sigma)
    and the v conv weights by ``v_scale``.  Then o = S'^T q^ is about
    v~ / sqrt(128) while w = A^T q^ grows with sigma: |o| << |w|."""
    spec = W.Spec(f"cancel_s{sigma:g}_v{v_scale:g}", N=N, H=H, num_slots=N + 2, seed=seed,
                  out_norm=out_norm)
    x = W.make_inputs(spec)
    D = H * W.HEAD_DIM
    x.conv_weight[1] = x.conv_weight[0]
    x.conv_weight[2] *= np.float32(v_scale)
    x.qkv[:, D:2 * D] = x.qkv[:, 0:D]
    x.conv_state[:, D:2 * D, :] = x.conv_state[:, 0:D, :]
    x.beta[:] = W.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    x.g[:] = 0.0
    x.state *= np.float32(sigma / 0.02)
    return x
