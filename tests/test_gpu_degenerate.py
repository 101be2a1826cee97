"""Degenerate and extreme inputs against the oracle: no write (beta = 0), no
decay (g = 0), decay to nothing (g = -80), an all-zero state, all-zero q/k/v
inputs (the L2 and RMS epsilons decide the result), large-magnitude inputs,
and a large batch (N=1024, H=96: 98,304 units, every slot distinct)."""
import numpy as np
import pytest
import torch

import kda_testlib as T
from linear_attention_decode_04_gb300 import workloads as W

pytestmark = pytest.mark.gpu

BASE = W.Spec("degenerate_n24_h12_pool32", N=24, H=12, num_slots=32, seed=71, pad_tail=2)


def _run(x, dev, **kw):
    d = T.to_device(x, dev)
    T.run_gpu(x, d, **kw)
    torch.cuda.synchronize()
    ref = T.run_oracle(x, **kw)
    T.compare_all(x, d, ref, init_state=x.state, init_conv=x.conv_state)
    assert int(d["err_flag"].item()) == 0
    return d, ref


def test_beta_zero_is_pure_decay(cuda_device):
    x = W.make_inputs(BASE)
    x.beta[:] = 0
    d, ref = _run(x, cuda_device)
    # the state of every active slot is Diag(alpha) S, to fp32 rounding
    n, s = 0, int(x.slot_idx[0])
    alpha = np.exp(x.g[n].astype(np.float64))            # [H, 128]
    want = alpha[:, :, None] * x.state[s].astype(np.float64)
    assert np.allclose(d["state"][s].cpu().numpy(), want, rtol=1e-6, atol=1e-9)


def test_no_decay(cuda_device):
    x = W.make_inputs(BASE)
    x.g[:] = 0.0
    _run(x, cuda_device)


def test_decay_to_nothing(cuda_device):
    x = W.make_inputs(BASE)
    x.g[:] = -80.0          # alpha = exp(-80) ~ 1.8e-35: the old state vanishes
    _run(x, cuda_device)


def test_zero_state(cuda_device):
    x = W.make_inputs(BASE)
    x.state[:] = 0.0
    _run(x, cuda_device)


@pytest.mark.parametrize("norm", [True, False])
def test_zero_inputs_epsilons_decide(norm, cuda_device):
    """q = k = v = 0 after the conv: q^ = k^ = 0, so S' = Diag(alpha) S and
    o = 0; the RMSNorm of a zero row is 0.  Done by zeroing the conv state,
    the token and the conv weights."""
    x = W.make_inputs(BASE)
    x.qkv[:] = 0
    x.conv_state[:] = 0
    d, ref = _run(x, cuda_device, out_norm=norm)
    assert not np.any(W.bf16_bits_to_f32(T.bf16_bits(d["out"])))


def test_large_magnitude_inputs(cuda_device):
    x = W.make_inputs(BASE)
    big = W.bf16_bits_to_f32(x.qkv) * 64.0             # conv outputs in the hundreds
    x.qkv = W.f32_to_bf16_bits(big)
    x.state *= 50.0
    _run(x, cuda_device)


def test_large_batch_n1024_h96(cuda_device):
    spec = W.Spec("large_n1024_h96_pool1100", N=1024, H=96, num_slots=1100, seed=72, pad_tail=16)
    x = W.make_inputs(spec)
    d = T.to_device(x, cuda_device)
    T.run_gpu(x, d)
    torch.cuda.synchronize()
    ref = T.run_oracle(x, in_place=False)
    T.check_out(T.bf16_bits(d["out"]), ref, "large batch")
    assert np.array_equal(T.bf16_bits(d["conv_state"]), ref.conv_state)
    rng = np.random.default_rng(0)
    for s in rng.choice(spec.num_slots, 64, replace=False):   # sampled slots of the 6.9 GB pool
        got = d["state"][int(s)].cpu().numpy()
        if s in set(x.slot_idx.tolist()) and s > 0:
            T.check_state_slot(got, ref.state[s], f"slot {s}")
        else:
            assert np.array_equal(got, x.state[s])
