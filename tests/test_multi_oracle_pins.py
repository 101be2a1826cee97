"""Pins of the fp64 multi-token (speculative) decode oracle against facts
that are not that oracle:
  - T = 1 with the destination equal to the source is the decode step, bit
    for bit (the decode oracle is pinned on its own);
  - a dense-matrix brute force: the conv by torch's conv1d over
    [source window | present tokens], S <- (I - b k k^T) Diag(a) S + b k v^T
    as explicit matrices, each present token's state and window stored to
    its own destination;
  - the decode oracle chained token by token on fresh slots (its state is
    rounded to fp32 between calls, so states agree to fp32 rounding, windows
    bit for bit);
  - invariants: an absent token equals the same call without it, a padding
    sequence touches nothing, a source that is also a destination reads the
    old contents, the conv-state flag only gates the window stores.

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


def tiny_multi(seed=0, N=3, T=3, H=2, K=3, V=5, W=4, num_slots=14, src=None, dst=None,
               out_norm=True, bias=False):
    rng = np.random.default_rng(seed)
    C = 2 * H * K + H * V
    R = N * T
    if src is None or dst is None:
        perm = rng.permutation(np.arange(1, num_slots))
        src = perm[:N] if src is None else src
        dst = perm[N:N + N * T].reshape(N, T) if dst is None else dst
    p = dict(
        H=H, K=K, V=V, W=W, out_norm=out_norm,
        qkv=bf16_bits(rng.standard_normal((R, C))),
        conv_weight=(0.5 * rng.standard_normal(W * C)).astype(np.float32),
        conv_state=bf16_bits(rng.standard_normal((num_slots, C, W - 1))),
        state=(0.3 * rng.standard_normal((num_slots, H, K, V))).astype(np.float32),
        g=(-np.logaddexp(0, rng.standard_normal((R, H, K)))).astype(np.float32),
        beta=bf16_bits(1 / (1 + np.exp(-rng.standard_normal((R, H))))),
        gate=bf16_bits(rng.standard_normal((R, H * V))),
        norm_weight=(1 + 0.1 * rng.standard_normal(V)).astype(np.float32),
        src_slot=np.asarray(src, np.int32),
        dst_slots=np.asarray(dst, np.int32).reshape(N, T),
    )
    p["conv_bias"] = (0.1 * rng.standard_normal(C)).astype(np.float32) if bias else None
    return p


def run(p, **kw):
    a = dict(p)
    a.update(kw)
    return oracle.decode_multi(**a)


def brute_force(p, update_conv_state=True, eps=1e-6, l2_eps=1e-6):
    H, K, V, W = p["H"], p["K"], p["V"], p["W"]
    Dq, Dv = H * K, H * V
    C = 2 * Dq + Dv
    N, T = p["dst_slots"].shape
    num_slots = p["state"].shape[0]
    cw = p["conv_weight"].astype(np.float64)
    taps = np.concatenate([cw[0:W * Dq].reshape(W, Dq), cw[W * Dq:2 * W * Dq].reshape(W, Dq),
                           cw[2 * W * Dq:].reshape(W, Dv)], axis=1).T  # [C, W]
    bias = p["conv_bias"].astype(np.float64) if p["conv_bias"] is not None else np.zeros(C)
    out = np.zeros((N * T, Dv))
    state = p["state"].copy()
    cs = p["conv_state"].copy()
    src_state = p["state"].astype(np.float64)
    src_cs = p["conv_state"]
    for n in range(N):
        s = int(p["src_slot"][n])
        if s <= 0 or s >= num_slots:
            continue
        present = [t for t in range(T) if 0 < p["dst_slots"][n, t] < num_slots]
        if not present:
            continue
        rows = [n * T + t for t in present]
        seq = np.concatenate([widen(src_cs[s]).T, widen(p["qkv"][rows, :C])], axis=0)  # [W-1+L, C]
        y = F.conv1d(torch.from_numpy(seq.T[None]), torch.from_numpy(taps[:, None, :]),
                     torch.from_numpy(bias), groups=C)[0].numpy().T  # [L, C]
        a = y / (1 + np.exp(-y))
        for h in range(H):
            S = src_state[s, h].copy()
            for m, (t, r) in enumerate(zip(present, rows)):
                q = a[m, h * K:(h + 1) * K]
                k = a[m, Dq + h * K:Dq + (h + 1) * K]
                v = a[m, 2 * Dq + h * V:2 * Dq + (h + 1) * V]
                qh = q / np.sqrt(K) / np.sqrt(q @ q + l2_eps)
                kh = k / np.sqrt(k @ k + l2_eps)
                al = np.exp(p["g"][r, h].astype(np.float64))
                be = widen(p["beta"][r, h])
                S = (np.eye(K) - be * np.outer(kh, kh)) @ np.diag(al) @ S + be * np.outer(kh, v)
                o = S.T @ qh
                if p["out_norm"]:
                    gt = widen(p["gate"][r, h * V:(h + 1) * V])
                    o = o / np.sqrt(np.mean(o * o) + eps) * p["norm_weight"] / (1 + np.exp(-gt))
                out[r, h * V:(h + 1) * V] = o
                state[p["dst_slots"][n, t], h] = S.astype(np.float32)
        if update_conv_state:
            for m, t in enumerate(present):
                cs[p["dst_slots"][n, t]] = bf16_bits(seq[m + 1:m + W].T.astype(np.float32))
    return out, state, cs


def _close_out(got64, want64, rel=1e-11):
    assert np.allclose(got64, want64, rtol=rel, atol=1e-13), np.abs(got64 - want64).max()


def test_t1_with_destination_equal_to_source_is_the_decode_step():
    for seed, kw in ((0, {}), (1, dict(out_norm=False)), (2, dict(bias=True))):
        p = tiny_multi(seed=seed, N=4, T=1, num_slots=9, **kw)
        p["dst_slots"] = p["src_slot"].reshape(-1, 1).copy()
        m = run(p)
        d = oracle.decode(qkv=p["qkv"], conv_weight=p["conv_weight"], conv_state=p["conv_state"],
                          state=p["state"], g=p["g"], beta=p["beta"], slot_idx=p["src_slot"], H=p["H"],
                          K=p["K"], V=p["V"], W=p["W"], gate=p["gate"], norm_weight=p["norm_weight"],
                          conv_bias=p["conv_bias"], out_norm=p["out_norm"])
        assert np.array_equal(m.out, d.out) and np.array_equal(m.out_f64, d.out_f64)
        assert np.array_equal(m.state, d.state) and np.array_equal(m.conv_state, d.conv_state)


def test_matches_dense_brute_force():
    # catches: window not slid between tokens, state re-read from the source,
    # a token's state or window stored to the wrong destination, per-token
    # rows of g / beta / gate taken from the wrong token, a transposed update
    for seed, kw in ((0, {}), (1, dict(out_norm=False)), (2, dict(bias=True)), (3, dict(T=5, N=2))):
        p = tiny_multi(seed=seed, **kw)
        out, state, cs = brute_force(p)
        r = run(p)
        _close_out(r.out_f64, out)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(out), 2.0 ** -126))) - 8)
        assert np.all(np.abs(widen(r.out) - out) <= ulp)  # bf16 rounding of the same value
        assert np.allclose(r.state, state, rtol=1e-6, atol=1e-7)
        assert np.array_equal(r.conv_state, cs)


def test_chained_decode_calls_on_fresh_slots():
    """Token t of sequence n equals one decode call on slot dst[n, t] after
    copying in the previous token's slot (the source for t = 0)."""
    p = tiny_multi(seed=5, N=3, T=4, num_slots=20, bias=True)
    r = run(p)
    cs, st = p["conv_state"].copy(), p["state"].copy()
    N, T = p["dst_slots"].shape
    for t in range(T):
        prev = p["src_slot"] if t == 0 else p["dst_slots"][:, t - 1]
        dst = p["dst_slots"][:, t]
        cs[dst], st[dst] = cs[prev], st[prev]
        rows = np.arange(N) * T + t
        d = oracle.decode(qkv=p["qkv"][rows], conv_weight=p["conv_weight"], conv_state=cs, state=st,
                          g=p["g"][rows], beta=p["beta"][rows], slot_idx=dst, H=p["H"], K=p["K"], V=p["V"],
                          W=p["W"], gate=p["gate"][rows], norm_weight=p["norm_weight"],
                          conv_bias=p["conv_bias"], in_place=True)
        assert np.allclose(r.out_f64[rows], d.out_f64, rtol=1e-6, atol=1e-7)
    touched = np.concatenate([p["dst_slots"].ravel()])
    assert np.array_equal(r.conv_state, cs)
    assert np.allclose(r.state[touched], st[touched], rtol=1e-6, atol=1e-7)


def test_absent_token_equals_the_call_without_it():
    p = tiny_multi(seed=6, N=2, T=4, num_slots=16)
    p["dst_slots"][0, 1] = 0          # sequence 0: token 1 absent
    p["dst_slots"][1, 3] = -2         # sequence 1: last token absent
    r = run(p)
    for rr in (1, 7):
        assert not r.out[rr].any() and not r.out_f64[rr].any()
    # the same sequences with the absent tokens removed
    keep = {0: [0, 2, 3], 1: [0, 1, 2]}
    for n, ts in keep.items():
        q = tiny_multi(seed=6, N=2, T=4, num_slots=16)
        sub = dict(p)
        rows = [n * 4 + t for t in ts]
        for key in ("qkv", "g", "beta", "gate"):
            sub[key] = p[key][rows]
        sub["src_slot"] = p["src_slot"][n:n + 1]
        sub["dst_slots"] = p["dst_slots"][n, ts].reshape(1, 3)
        sub["conv_state"], sub["state"] = q["conv_state"], q["state"]
        s = run(sub)
        assert np.array_equal(s.out, r.out[rows]) and np.array_equal(s.out_f64, r.out_f64[rows])
        for d in sub["dst_slots"].ravel():
            assert np.array_equal(s.state[d], r.state[d]) and np.array_equal(s.conv_state[d], r.conv_state[d])


def test_padding_sequence_and_out_of_range_slots():
    p = tiny_multi(seed=7, N=3, T=2, num_slots=12)
    p["src_slot"][0] = 0              # padding sequence
    p["src_slot"][1] = 40             # out of range: treated like padding, counted
    p["dst_slots"][2, 0] = 99         # out-of-range destination: absent, counted
    r = run(p)
    assert r.n_out_of_range == 2
    assert not r.out[0:4].any()       # both tokens of sequences 0 and 1
    assert not r.out[4].any() and r.out[5].any()
    untouched = set(range(12)) - {int(p["dst_slots"][2, 1])}
    for s in untouched:
        assert np.array_equal(r.state[s], p["state"][s]) and np.array_equal(r.conv_state[s], p["conv_state"][s])


def test_source_may_be_one_of_its_destinations():
    """Destinations may include the source slot (the accepted-token slot of a
    speculative step is rewritten): the result equals reading a copy."""
    p = tiny_multi(seed=8, N=2, T=3, num_slots=14)
    q = dict(p, state=p["state"].copy(), conv_state=p["conv_state"].copy())
    spare = [s for s in range(1, 14) if s not in p["src_slot"] and s not in p["dst_slots"]]
    q["dst_slots"] = p["dst_slots"].copy()
    q["dst_slots"][0, 2] = p["src_slot"][0]          # alias: the last token rewrites the source
    q["dst_slots"][1, 0] = p["src_slot"][1]          # alias: the first token rewrites the source
    r = run(q)
    c = dict(q, state=q["state"].copy(), conv_state=q["conv_state"].copy(), src_slot=np.array(spare[:2], np.int32))
    c["state"][spare[:2]] = q["state"][q["src_slot"]]
    c["conv_state"][spare[:2]] = q["conv_state"][q["src_slot"]]
    rc = run(c)
    assert np.array_equal(r.out, rc.out)
    for d in q["dst_slots"].ravel():
        assert np.array_equal(r.state[d], rc.state[d]) and np.array_equal(r.conv_state[d], rc.conv_state[d])


def test_update_off_only_gates_the_window_stores():
    p = tiny_multi(seed=9, N=2, T=3, num_slots=12)
    on, off = run(p), run(p, update_conv_state=False)
    assert np.array_equal(on.out, off.out) and np.array_equal(on.state, off.state)
    assert np.array_equal(off.conv_state, p["conv_state"])
    out, state, cs = brute_force(p, update_conv_state=False)
    assert np.array_equal(off.conv_state, cs)


def test_realistic_head_size_t1_chain_against_decode():
    """K = V = 128 and the workload's distributions: two tokens per sequence
    equal two chained decode calls."""
    from linear_attention_decode_04_gb300 import workloads as Wl
    x = Wl.make_inputs(Wl.Spec("multi_pin_n6_h2", N=6, H=2, num_slots=16, seed=11))
    N, T = 3, 2
    src = np.array([2, 5, 9], np.int32)
    dst = np.array([[3, 4], [6, 7], [10, 11]], np.int32)
    r = oracle.decode_multi(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=x.conv_state, state=x.state,
                            g=x.g, beta=x.beta, src_slot=src, dst_slots=dst, H=2, gate=x.gate,
                            norm_weight=x.norm_weight)
    cs, st = x.conv_state.copy(), x.state.copy()
    for t in range(T):
        prev = src if t == 0 else dst[:, t - 1]
        cs[dst[:, t]], st[dst[:, t]] = cs[prev], st[prev]
        rows = np.arange(N) * T + t
        d = oracle.decode(qkv=x.qkv[rows], conv_weight=x.conv_weight, conv_state=cs, state=st, g=x.g[rows],
                          beta=x.beta[rows], slot_idx=dst[:, t], H=2, gate=x.gate[rows],
                          norm_weight=x.norm_weight, in_place=True)
        assert np.allclose(r.out_f64[rows], d.out_f64, rtol=1e-5, atol=1e-6)
    assert np.array_equal(r.conv_state, cs)
    assert np.allclose(r.state, st, rtol=1e-6, atol=1e-8)
