"""Pins of the fp64 prefill oracle against facts that are not the oracle:
a dense-matrix brute force with the conv taken by torch's conv1d over the
whole padded sequence, a closed form (orthonormal keys written into an empty
memory), the separately pinned decode oracle chained token by token, and the
padding / empty-sequence / split-sequence invariants.

Head sizes are unequal (K != V) so a transposed state cannot pass by symmetry.
"""
import numpy as np
import torch
import torch.nn.functional as F

import oracle


def bf16_bits(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def widen(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def tiny_prefill(seed=0, lens=(5, 1, 0, 3), H=2, K=3, V=5, W=4, num_slots=7, slots=None,
                 out_norm=True, bias=False):
    rng = np.random.default_rng(seed)
    B = len(lens)
    T = int(sum(lens))
    C = 2 * H * K + H * V
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    p = dict(
        H=H, K=K, V=V, W=W, out_norm=out_norm, cu_seqlens=cu,
        qkv=bf16_bits(rng.standard_normal((T, C))),
        conv_weight=(0.5 * rng.standard_normal(W * C)).astype(np.float32),
        conv_state=bf16_bits(rng.standard_normal((num_slots, C, W - 1))),
        state=(0.3 * rng.standard_normal((num_slots, H, K, V))).astype(np.float32),
        g=(-np.logaddexp(0, rng.standard_normal((T, H, K)))).astype(np.float32),
        beta=bf16_bits(1 / (1 + np.exp(-rng.standard_normal((T, H))))),
        gate=bf16_bits(rng.standard_normal((T, H * V))),
        norm_weight=(1 + 0.1 * rng.standard_normal(V)).astype(np.float32),
        slot_idx=np.asarray(slots if slots is not None else rng.permutation(np.arange(1, num_slots))[:B],
                            dtype=np.int32),
    )
    p["conv_bias"] = (0.1 * rng.standard_normal(C)).astype(np.float32) if bias else None
    return p


def run(p, **kw):
    a = dict(p)
    a.update(kw)
    return oracle.prefill(**a)


def brute_force(p, q_scale=None, l2_eps=1e-6, eps=1e-6, gate=None):
    """Dense-matrix evaluation: conv by torch conv1d over [conv state | tokens]
    per channel, S <- (I - b k k^T) Diag(a) S + b k v^T as explicit matrices.
    ``gate`` = (A_log, dt_bias or None, lower_bound): g and beta are raw
    logits, activated here with numpy (log1p / exp)."""
    H, K, V, W = p["H"], p["K"], p["V"], p["W"]
    Dq, Dv = H * K, H * V
    C = 2 * Dq + Dv
    cu = p["cu_seqlens"]
    T = int(cu[-1])
    cw = p["conv_weight"].astype(np.float64)
    taps = np.concatenate([cw[0:W * Dq].reshape(W, Dq), cw[W * Dq:2 * W * Dq].reshape(W, Dq),
                           cw[2 * W * Dq:].reshape(W, Dv)], axis=1).T  # [C, W]
    bias = p["conv_bias"].astype(np.float64) if p["conv_bias"] is not None else np.zeros(C)
    scale = 1 / np.sqrt(K) if q_scale is None else q_scale
    out = np.zeros((T, Dv))
    state = p["state"].astype(np.float64).copy()
    cs = p["conv_state"].copy()
    for b in range(len(cu) - 1):
        r0, r1 = int(cu[b]), int(cu[b + 1])
        s = int(p["slot_idx"][b])
        if r1 == r0 or s <= 0 or s >= state.shape[0]:
            continue
        seq = np.concatenate([widen(cs[s]).T, widen(p["qkv"][r0:r1, :C])], axis=0)  # [W-1+L, C]
        y = F.conv1d(torch.from_numpy(seq.T[None]), torch.from_numpy(taps[:, None, :]),
                     torch.from_numpy(bias), groups=C)[0].numpy().T  # [L, C]
        a = y / (1 + np.exp(-y))
        for h in range(H):
            S = state[s, h]
            for t in range(r1 - r0):
                r = r0 + t
                q = a[t, h * K:(h + 1) * K]
                k = a[t, Dq + h * K:Dq + (h + 1) * K]
                v = a[t, 2 * Dq + h * V:2 * Dq + (h + 1) * V]
                qh = scale * q / np.sqrt(q @ q + l2_eps)
                kh = k / np.sqrt(k @ k + l2_eps)
                al = np.exp(p["g"][r, h].astype(np.float64))
                be = widen(p["beta"][r, h])
                if gate is not None:
                    A_log, dt_bias, lb = gate
                    z = p["g"][r, h].astype(np.float64)
                    if dt_bias is not None:
                        z = z + dt_bias[h * K:(h + 1) * K].astype(np.float64)
                    ea = np.exp(np.float64(A_log[h]))
                    if lb < 0:
                        gg = lb / (1.0 + np.exp(-ea * z))
                    else:
                        gg = -ea * (np.maximum(z, 0) + np.log1p(np.exp(-np.abs(z))))
                    al = np.exp(gg)
                    be = 1.0 / (1.0 + np.exp(-be))
                S = (np.eye(K) - be * np.outer(kh, kh)) @ np.diag(al) @ S + be * np.outer(kh, v)
                o = S.T @ qh
                if p["out_norm"]:
                    gt = widen(p["gate"][r, h * V:(h + 1) * V])
                    o = o / np.sqrt(np.mean(o * o) + eps) * p["norm_weight"] / (1 + np.exp(-gt))
                out[r, h * V:(h + 1) * V] = o
            state[s, h] = S
        cs[s] = bf16_bits(seq[-(W - 1):].T.astype(np.float32))
    return out, state.astype(np.float32), cs


def test_prefill_matches_dense_brute_force():
    # catches: window not slid / wrong tap order across tokens, state reset or
    # not carried, per-token indices of g/beta/gate taken from the wrong row,
    # final window or state not stored, transposed update
    for seed, kw in ((0, {}), (1, dict(out_norm=False)), (2, dict(bias=True)),
                     (3, dict(lens=(2, 7, 1), W=4))):
        p = tiny_prefill(seed=seed, **kw)
        r = run(p)
        want_out, want_state, want_cs = brute_force(p)
        np.testing.assert_allclose(r.out_f64, want_out, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(r.state, want_state, rtol=1e-6, atol=1e-7)
        assert np.array_equal(r.conv_state, want_cs)


def test_prefill_associative_memory_closed_form():
    # Orthonormal keys written with beta = 1 and no decay into an empty state:
    # S_T = sum_m k^_m v~_m^T, and the readout with q = k_t returns the stored
    # value scaled by |k^|^2 * q_scale.  Catches a state that is not carried
    # from token to token and a decay or beta taken from the wrong token.
    H, K, V, W, L = 1, 8, 6, 4, 5
    C = 2 * H * K + H * V
    rng = np.random.default_rng(7)
    qkv = np.zeros((L, C), np.float32)
    for m in range(L):
        qkv[m, m] = 4.0                 # q input along e_m
        qkv[m, K + m] = 4.0             # k input along e_m
    qkv[:, 2 * K:] = rng.standard_normal((L, V))
    conv_weight = np.zeros(W * C, np.float32)
    # identity on the current token (last tap) for every channel of every block
    conv_weight[(W - 1) * K:W * K] = 1.0
    conv_weight[W * K + (W - 1) * K:W * K + W * K] = 1.0
    conv_weight[2 * W * K + (W - 1) * V:2 * W * K + W * V] = 1.0
    p = dict(H=H, K=K, V=V, W=W, out_norm=False, cu_seqlens=np.array([0, L], np.int32),
             qkv=bf16_bits(qkv), conv_weight=conv_weight,
             conv_state=np.zeros((2, C, W - 1), np.uint16),
             state=np.zeros((2, H, K, V), np.float32),
             g=np.zeros((L, H, K), np.float32), beta=bf16_bits(np.ones((L, H))),
             gate=None, norm_weight=None, slot_idx=np.array([1], np.int32), conv_bias=None)
    r = run(p)
    silu4 = 4.0 / (1 + np.exp(-4.0))
    c = silu4 / np.sqrt(silu4 ** 2 + 1e-6)          # |k^| after the L2 norm
    vt = widen(bf16_bits(qkv[:, 2 * K:]))
    vt = vt / (1 + np.exp(-vt))
    want_S = np.zeros((K, V))
    want_S[:L] = c * vt
    np.testing.assert_allclose(r.state[1, 0], want_S, rtol=1e-6, atol=1e-7)
    want_o = (c * c / np.sqrt(K)) * vt
    np.testing.assert_allclose(r.out_f64, want_o, rtol=1e-9, atol=1e-12)


def test_prefill_equals_decode_chained_token_by_token():
    # the decode oracle is pinned on its own; prefill must agree with it up to
    # the fp32 rounding the chained decode applies to the state after every token
    p = tiny_prefill(seed=11, lens=(6, 3, 1, 4))
    r = run(p)
    cs, st = p["conv_state"].copy(), p["state"].copy()
    out = np.zeros_like(r.out_f64)
    cu = p["cu_seqlens"]
    for b in range(len(cu) - 1):
        for t in range(int(cu[b]), int(cu[b + 1])):
            d = oracle.decode(qkv=p["qkv"][t:t + 1], conv_weight=p["conv_weight"], conv_state=cs,
                              state=st, g=p["g"][t:t + 1], beta=p["beta"][t:t + 1],
                              slot_idx=p["slot_idx"][b:b + 1], H=p["H"], K=p["K"], V=p["V"],
                              W=p["W"], gate=p["gate"][t:t + 1], norm_weight=p["norm_weight"],
                              in_place=True)
            out[t] = d.out_f64[0]
    np.testing.assert_allclose(r.out_f64, out, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(r.state, st, rtol=1e-5, atol=1e-7)
    assert np.array_equal(r.conv_state, cs)


def test_prefill_padding_empty_and_out_of_range():
    p = tiny_prefill(seed=4, lens=(3, 2, 0, 4), slots=(0, 2, 5, 9), num_slots=7)
    r = run(p)
    assert r.n_out_of_range == 1                      # slot 9 >= 7
    assert np.all(r.out[0:3] == 0) and np.all(r.out_f64[0:3] == 0.0)   # padding sequence
    assert np.all(r.out[5:9] == 0)                    # out-of-range sequence
    assert np.any(r.out[3:5] != 0)
    for s in (0, 1, 3, 4, 5, 6):                      # only slot 2 is written (slot 5's sequence is empty)
        assert np.array_equal(r.state[s], p["state"][s])
        assert np.array_equal(r.conv_state[s], p["conv_state"][s])
    assert not np.array_equal(r.state[2], p["state"][2])


def test_prefill_split_sequence_invariance():
    # one sequence in one call == its two halves in two calls on the same slot
    # (catches a final window or state stored from the wrong tokens)
    p = tiny_prefill(seed=5, lens=(7,), slots=(3,))
    whole = run(p)
    for m in (1, 2, 5):
        a = dict(p, cu_seqlens=np.array([0, m], np.int32))
        first = run(a)
        b = dict(p, cu_seqlens=np.array([0, 7 - m], np.int32), qkv=p["qkv"][m:], g=p["g"][m:],
                 beta=p["beta"][m:], gate=p["gate"][m:], conv_state=first.conv_state,
                 state=first.state)
        second = run(b)
        np.testing.assert_allclose(np.concatenate([first.out_f64[:m], second.out_f64]), whole.out_f64,
                                   rtol=1e-5, atol=1e-6)
        assert np.array_equal(second.conv_state, whole.conv_state)
        np.testing.assert_allclose(second.state, whole.state, rtol=1e-5, atol=1e-7)


def test_prefill_length_one_is_decode():
    p = tiny_prefill(seed=6, lens=(1, 1, 1), num_slots=5)
    r = run(p)
    d = oracle.decode(qkv=p["qkv"], conv_weight=p["conv_weight"], conv_state=p["conv_state"],
                      state=p["state"], g=p["g"], beta=p["beta"], slot_idx=p["slot_idx"], H=p["H"],
                      K=p["K"], V=p["V"], W=p["W"], gate=p["gate"], norm_weight=p["norm_weight"])
    assert np.array_equal(r.out, d.out)
    assert np.array_equal(r.state, d.state)
    assert np.array_equal(r.conv_state, d.conv_state)


def test_prefill_fused_gate_matches_brute_force():
    # raw g / beta logits activated inside the prefill (both gate forms, with
    # and without dt_bias) against the brute force's own numpy activation
    for seed, lb, with_dt in ((21, -5.0, True), (22, 0.0, True), (23, 0.0, False)):
        p = tiny_prefill(seed=seed, lens=(6, 3))
        rng = np.random.default_rng(seed + 100)
        p["g"] = rng.standard_normal(p["g"].shape).astype(np.float32)
        p["beta"] = bf16_bits(rng.standard_normal(p["beta"].shape))
        A_log = (0.5 * rng.standard_normal(p["H"])).astype(np.float32)
        dt_bias = (0.5 * rng.standard_normal(p["H"] * p["K"])).astype(np.float32) if with_dt else None
        r = run(p, fused_gate=True, A_log=A_log, dt_bias=dt_bias, lower_bound=lb)
        want_out, want_state, want_cs = brute_force(p, gate=(A_log, dt_bias, lb))
        np.testing.assert_allclose(r.out_f64, want_out, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(r.state, want_state, rtol=1e-6, atol=1e-7)
        assert np.array_equal(r.conv_state, want_cs)


def test_prefill_sd_conv_state_is_the_transposed_ds_result():
    # the tap-first layout holds the same values: running on the transposed
    # pool gives the transposed final pool and the same outputs and state
    p = tiny_prefill(seed=31, lens=(5, 1, 2, 0))
    ds = run(p)
    sd_in = np.ascontiguousarray(p["conv_state"].transpose(0, 2, 1))
    sd = run(p, conv_state=sd_in, conv_state_sd=True)
    assert np.array_equal(sd.conv_state, ds.conv_state.transpose(0, 2, 1))
    assert np.array_equal(sd.out, ds.out)
    assert np.array_equal(sd.state, ds.state)
