"""Host-side checks of the seeded input generator (no method arithmetic)."""
import numpy as np

from linear_attention_decode_04_gb300 import workloads as W


def test_bf16_round_trip_and_rne():
    x = np.array([1.0, -2.5, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 3.14159], np.float32)
    b = W.f32_to_bf16_bits(x)
    assert list(b[:2]) == [0x3F80, 0xC020]
    assert b[2] == 0x3F80          # tie -> even
    assert b[3] == 0x3F82          # tie -> even (up)
    assert np.allclose(W.bf16_bits_to_f32(b), x, rtol=2 ** -8)


def test_pr1_reference_shapes_and_slots():
    x = W.make_inputs(W.PR1_REF)
    assert x.qkv.shape == (4, 3 * 12 * 128) and x.qkv.dtype == np.uint16
    assert x.conv_weight.shape == (3, 4, 1536) and x.conv_weight.dtype == np.float32
    assert x.conv_state.shape == (8, 4608, 3) and x.conv_state.dtype == np.uint16
    assert x.state.shape == (8, 12, 128, 128) and x.state.dtype == np.float32
    assert x.g.shape == (4, 12, 128) and x.beta.shape == (4, 12) and x.gate.shape == (4, 1536)
    assert list(x.slot_idx) == [1, 3, 5, 7]


def test_deterministic_and_slotwise_pools():
    a, b = W.make_inputs(W.PAD_TAIL, threads=1), W.make_inputs(W.PAD_TAIL, threads=4)
    for f in ("qkv", "conv_weight", "conv_state", "state", "g", "beta", "gate", "norm_weight",
              "slot_idx"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    s = a.slot_idx
    assert (s[24:] == 0).all() and len(set(s[:24])) == 24 and (s[:24] > 0).all()


def test_distributions():
    x = W.make_inputs(W.NORM_OFF)
    assert np.all(x.g >= -5.0) and np.all(x.g < 0.0)
    y = W.make_inputs(W.PR1_REF)
    assert np.all(y.g < 0)
    assert abs(np.std(y.state) - 0.02) < 0.001
    beta = W.bf16_bits_to_f32(y.beta)
    assert np.all((beta > 0) & (beta < 1))
    assert abs(np.mean(y.norm_weight) - 1.0) < 0.05


def test_algorithmic_bytes_per_unit():
    assert W.algorithmic_bytes(1, 1, 1) - W.algorithmic_bytes(1, 1, 0) == 137474 - 256
    assert W.algorithmic_bytes(1, 1, 1, out_norm=False) - W.algorithmic_bytes(1, 1, 0, out_norm=False) == 137218 - 256
