"""Pins of the fp64 oracle against facts fixed by the mathematics, the pages
and independent library routines -- never against the CUDA path.

Each test names the plausible oracle mistake it would catch.  Head sizes are
kept unequal (K != V) wherever a layout is involved, so a transposed state or
readout cannot pass by symmetry.
"""
import math
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

# ----------------------------------------------------------------- helpers


def bf16_bits(x):
    """Test-side fp32 -> bf16 RNE for building inputs (not the oracle's)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def widen(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def tiny_problem(seed=0, N=3, H=2, K=3, V=5, W=4, num_slots=6, slots=None, out_norm=True,
                 bias=False, state_scale=0.3, qkv_pad=0):
    rng = np.random.default_rng(seed)
    C = 2 * H * K + H * V
    p = dict(
        H=H, K=K, V=V, W=W, out_norm=out_norm,
        qkv=bf16_bits(rng.standard_normal((N, C + qkv_pad))),
        conv_weight=(0.5 * rng.standard_normal(W * C)).astype(np.float32),
        conv_state=bf16_bits(rng.standard_normal((num_slots, C, W - 1))),
        state=(state_scale * rng.standard_normal((num_slots, H, K, V))).astype(np.float32),
        g=(-np.logaddexp(0, rng.standard_normal((N, H, K)))).astype(np.float32),
        beta=bf16_bits(1 / (1 + np.exp(-rng.standard_normal((N, H))))),
        gate=bf16_bits(rng.standard_normal((N, H * V))),
        norm_weight=(1 + 0.1 * rng.standard_normal(V)).astype(np.float32),
        slot_idx=np.asarray(slots if slots is not None else rng.permutation(np.arange(1, num_slots))[:N],
                            dtype=np.int32),
    )
    p["conv_bias"] = (0.1 * rng.standard_normal(C)).astype(np.float32) if bias else None
    return p


def run(p, **kw):
    args = dict(p)
    args.update(kw)
    return oracle.decode(**args)


def channel_weights(p):
    """[C, W] per-channel taps from the block layout q [W][H*K] | k [W][H*K] | v [W][H*V]."""
    H, K, V, W = p["H"], p["K"], p["V"], p["W"]
    cw = p["conv_weight"].astype(np.float64)
    Dq, Dv = H * K, H * V
    q = cw[: W * Dq].reshape(W, Dq).T
    k = cw[W * Dq: 2 * W * Dq].reshape(W, Dq).T
    v = cw[2 * W * Dq:].reshape(W, Dv).T
    return np.concatenate([q, k, v], axis=0)


def torch_reference(p, eps=1e-6, l2_eps=1e-6, q_scale=None):
    """Whole step in float64 torch, built from library routines: depthwise
    conv1d, silu, dense matrix products, rms_norm, sigmoid."""
    H, K, V, W = p["H"], p["K"], p["V"], p["W"]
    Dq, Dv = H * K, H * V
    C = 2 * Dq + Dv
    qkv = torch.from_numpy(widen(p["qkv"]))[:, :C]
    wts = torch.from_numpy(channel_weights(p)).unsqueeze(1)          # [C, 1, W]
    bias = None if p.get("conv_bias") is None else torch.from_numpy(p["conv_bias"].astype(np.float64))
    cs = torch.from_numpy(widen(p["conv_state"]))                    # [slots, C, W-1]
    S_all = torch.from_numpy(p["state"].astype(np.float64))
    g = torch.from_numpy(p["g"].astype(np.float64))
    beta = torch.from_numpy(widen(p["beta"]))
    gate = torch.from_numpy(widen(p["gate"]))
    nw = torch.from_numpy(p["norm_weight"].astype(np.float64))
    scale = q_scale if q_scale else 1.0 / math.sqrt(K)
    N = qkv.shape[0]
    out = torch.zeros(N, Dv, dtype=torch.float64)
    new_state = {}
    for n in range(N):
        s = int(p["slot_idx"][n])
        if s <= 0 or s >= S_all.shape[0]:
            continue
        window = torch.cat([cs[s], qkv[n].unsqueeze(1)], dim=1)      # [C, W] oldest first
        y = F.conv1d(window.unsqueeze(0), wts, bias=bias, groups=C)[0, :, 0]
        a = F.silu(y)
        for h in range(H):
            qt = a[h * K:(h + 1) * K]
            kt = a[Dq + h * K: Dq + (h + 1) * K]
            vt = a[2 * Dq + h * V: 2 * Dq + (h + 1) * V]
            qh = scale * qt / torch.sqrt((qt * qt).sum() + l2_eps)
            kh = kt / torch.sqrt((kt * kt).sum() + l2_eps)
            b = beta[n, h]
            M = torch.eye(K, dtype=torch.float64) - b * torch.outer(kh, kh)
            Sn = M @ torch.diag(torch.exp(g[n, h])) @ S_all[s, h] + b * torch.outer(kh, vt)
            o = Sn.T @ qh
            if p["out_norm"]:
                o = F.rms_norm(o, (V,), weight=nw, eps=eps) * torch.sigmoid(gate[n, h * V:(h + 1) * V])
            out[n, h * V:(h + 1) * V] = o
            new_state[(s, h)] = Sn.numpy()
    return out.numpy(), new_state


# ----------------------------------------------------------------- dtypes


def _all_bf16_finite():
    b = np.arange(0, 0x7F80, dtype=np.uint32)  # +0 .. max finite
    return (b << 16).view(np.float32).astype(np.float64)


def test_round_bf16_is_nearest_even_by_brute_force():
    """Catches a truncating / round-half-up / double-rounding bf16 store: the
    nearest of all finite bf16 values, ties to the even pattern."""
    grid = _all_bf16_finite()
    rng = np.random.default_rng(1)
    xs = list(rng.standard_normal(2000) * 10.0 ** rng.integers(-40, 38, 2000))
    mids = (grid[1000:1200] + grid[1001:1201]) / 2      # exact ties
    xs += list(mids) + list(-mids) + [1e-45, 5e-41, 3.3e38, 3.4e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9]
    for x in xs:
        a = abs(x)
        i = np.searchsorted(grid, a)
        cands = [j for j in (i - 1, i) if 0 <= j < grid.size]
        if a > grid[-1] + (grid[-1] - grid[-2]) / 2:
            want = 0x7F80
        else:
            d = [abs(grid[j] - a) for j in cands]
            best = [cands[t] for t in range(len(cands)) if d[t] == min(d)]
            want = best[0] if len(best) == 1 else [j for j in best if j % 2 == 0][0]
        if x < 0:
            want |= 0x8000
        assert oracle.round_bf16(x) == want, (x, hex(oracle.round_bf16(x)), hex(want))


def test_bf16_widening_exact():
    for b in (0x0000, 0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F):
        assert oracle.bf16_to_f64(b) == float(widen(np.uint16(b)))


# ----------------------------------------------------------------- step 1


def test_causal_conv_is_library_depthwise_conv():
    """Catches reversed taps or a dropped bias: the 4-tap window dot equals
    torch's conv1d (cross-correlation) and numpy's convolve with flipped taps."""
    rng = np.random.default_rng(2)
    for _ in range(20):
        x, w, b = rng.standard_normal(4), rng.standard_normal(4), rng.standard_normal()
        got = oracle.causal_conv(x, w, b)
        ref = F.conv1d(torch.tensor(x).view(1, 1, 4), torch.tensor(w).view(1, 1, 4),
                       bias=torch.tensor([b], dtype=torch.float64)).item()
        assert abs(got - ref) < 1e-12
        assert abs(got - (np.convolve(x, w[::-1], "valid")[0] + b)) < 1e-12


def test_silu_sigmoid_library():
    for y in (-30.0, -2.5, -1e-3, 0.0, 0.7, 4.0, 25.0):
        assert abs(oracle.silu(y) - F.silu(torch.tensor(y, dtype=torch.float64)).item()) < 1e-15
        assert abs(oracle.sigmoid(y) - torch.sigmoid(torch.tensor(y, dtype=torch.float64)).item()) < 1e-15
    assert oracle.sigmoid(0.0) == 0.5


def test_conv_state_is_input_shifted_by_one():
    """Catches a conv state that shifts the wrong way or stores rounded
    values: after the step each active channel holds (x1, x2, x_new) bitwise."""
    p = tiny_problem(seed=3, N=3, slots=[2, 0, 5])
    r = run(p)
    C = p["conv_state"].shape[1]
    for n, s in enumerate(p["slot_idx"]):
        if s <= 0:
            continue
        old = p["conv_state"][s]
        assert np.array_equal(r.conv_state[s, :, 0], old[:, 1])
        assert np.array_equal(r.conv_state[s, :, 1], old[:, 2])
        assert np.array_equal(r.conv_state[s, :, 2], p["qkv"][n, :C])
    untouched = [s for s in range(p["conv_state"].shape[0]) if s not in (2, 5)]
    assert np.array_equal(r.conv_state[untouched], p["conv_state"][untouched])


def test_conv_state_update_off_leaves_it_and_keeps_recurrence():
    p = tiny_problem(seed=4)
    on, off = run(p), run(p, update_conv_state=False)
    assert np.array_equal(off.conv_state, p["conv_state"])
    assert np.array_equal(off.state, on.state)
    assert np.array_equal(off.out, on.out)


# ----------------------------------------------------------------- step 2


def test_l2norm_length_and_scale():
    """Catches the epsilon outside the square root or a missing scale."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(128)
    ss = float(np.dot(x, x))
    y = oracle.l2norm(x, eps=1e-6, scale=1.0)
    assert abs(np.linalg.norm(y) - math.sqrt(ss / (ss + 1e-6))) < 1e-14
    y2 = oracle.l2norm(x, eps=1e-6, scale=0.25)
    assert np.allclose(y2, 0.25 * y, rtol=0, atol=1e-16)
    tiny = np.full(4, 1e-4)     # |x|^2 = 4e-8 << eps: eps dominates
    assert np.allclose(oracle.l2norm(tiny, 1e-6), tiny / math.sqrt(4e-8 + 1e-6), rtol=1e-14)


# ----------------------------------------------------------------- step 3


def _unit(rng, K):
    k = rng.standard_normal(K)
    return k / np.linalg.norm(k)


@pytest.mark.parametrize("K,V", [(3, 5), (7, 2), (128, 128)])
def test_delta_rule_writes_value_under_unit_key(K, V):
    """beta = 1, alpha = 1, |k| = 1  =>  S'^T k = v  (a wrong sign or a
    dropped beta k v^T term breaks it)."""
    rng = np.random.default_rng(6)
    S = rng.standard_normal((K, V))
    k, v = _unit(rng, K), rng.standard_normal(V)
    Sn = oracle.gated_delta_update(S, np.ones(K), 1.0, k, v)
    assert np.allclose(Sn.T @ k, v, atol=1e-12)


@pytest.mark.parametrize("K,V", [(3, 5), (128, 128)])
def test_delta_rule_beta_zero_is_pure_decay(K, V):
    """beta = 0  =>  S' = Diag(alpha) S  (decay applied along the key index)."""
    rng = np.random.default_rng(7)
    S, alpha = rng.standard_normal((K, V)), np.exp(-rng.random(K))
    Sn = oracle.gated_delta_update(S, alpha, 0.0, rng.standard_normal(K), rng.standard_normal(V))
    assert np.array_equal(Sn, alpha[:, None] * S)


def test_delta_rule_from_zero_state_closed_form():
    """S = 0  =>  S' = beta k v^T and o = beta (q.k) v."""
    rng = np.random.default_rng(8)
    K, V = 4, 6
    k, v, q = rng.standard_normal(K), rng.standard_normal(V), rng.standard_normal(K)
    Sn = oracle.gated_delta_update(np.zeros((K, V)), np.exp(-rng.random(K)), 0.375, k, v)
    assert np.allclose(Sn, 0.375 * np.outer(k, v), atol=1e-15)
    assert np.allclose(oracle.readout(Sn, q), 0.375 * np.dot(q, k) * v, atol=1e-14)


def test_delta_rule_associative_memory():
    """Writing m orthonormal keys in turn (beta = 1, alpha = 1) recalls every
    stored value: S'^T k_i = v_i for all i."""
    rng = np.random.default_rng(9)
    K, V, m = 8, 5, 6
    Q, _ = np.linalg.qr(rng.standard_normal((K, K)))
    keys, vals = Q[:, :m].T, rng.standard_normal((m, V))
    S = rng.standard_normal((K, V))
    for k, v in zip(keys, vals):
        S = oracle.gated_delta_update(S, np.ones(K), 1.0, k, v)
    for k, v in zip(keys, vals):
        assert np.allclose(S.T @ k, v, atol=1e-12)


@pytest.mark.parametrize("K,V", [(3, 5), (9, 4), (128, 128)])
def test_delta_rule_dense_matrix_form(K, V):
    """Brute force: (I - beta k k^T) Diag(alpha) S + beta k v^T by explicit
    K x K matrix products."""
    rng = np.random.default_rng(10)
    S, alpha = rng.standard_normal((K, V)), np.exp(-rng.random(K))
    k, v, beta = rng.standard_normal(K), rng.standard_normal(V), 0.6
    want = (np.eye(K) - beta * np.outer(k, k)) @ np.diag(alpha) @ S + beta * np.outer(k, v)
    assert np.allclose(oracle.gated_delta_update(S, alpha, beta, k, v), want, atol=1e-12)


def test_readout_is_transpose_product():
    rng = np.random.default_rng(11)
    S, q = rng.standard_normal((3, 7)), rng.standard_normal(3)
    assert np.allclose(oracle.readout(S, q), S.T @ q, atol=1e-14)


# ----------------------------------------------------------------- step 5


def test_gated_rmsnorm_unit_rms_and_gate_half():
    """Unit RMS before the weight (eps inside the root), sigmoid gate
    (gate = 0 gives exactly half), weight applied per channel; and equality
    with torch's rms_norm."""
    rng = np.random.default_rng(12)
    o, w = rng.standard_normal(128), 1 + 0.1 * rng.standard_normal(128)
    ms = float(np.mean(o * o))
    y = oracle.gated_rmsnorm(o, np.ones(128), np.full(128, 50.0), eps=1e-6)
    assert abs(math.sqrt(np.mean(y * y)) - math.sqrt(ms / (ms + 1e-6))) < 1e-13
    y0 = oracle.gated_rmsnorm(o, w, np.zeros(128), eps=1e-6)
    assert np.allclose(y0, 0.5 * w * o / math.sqrt(ms + 1e-6), atol=1e-14)
    gate = rng.standard_normal(128)
    ref = F.rms_norm(torch.tensor(o), (128,), weight=torch.tensor(w), eps=1e-6) * torch.sigmoid(torch.tensor(gate))
    assert np.allclose(oracle.gated_rmsnorm(o, w, gate, 1e-6), ref.numpy(), atol=1e-14)


# ----------------------------------------------------------------- whole step


@pytest.mark.parametrize("out_norm", [True, False])
@pytest.mark.parametrize("bias", [False, True])
def test_whole_step_matches_library_composition(out_norm, bias):
    """The full step against a float64 torch composition of library routines
    (depthwise conv1d, silu, dense matrix products, rms_norm, sigmoid) with
    its own indexing of the q | k | v blocks.  Catches wrong channel offsets,
    a swapped k/v block, a transposed state and a readout from the old state."""
    p = tiny_problem(seed=13, N=4, H=3, K=3, V=5, num_slots=8, slots=[3, 0, 7, 1],
                     out_norm=out_norm, bias=bias, qkv_pad=6)
    r = run(p)
    ref_out, ref_state = torch_reference(p)
    assert np.allclose(r.out_f64, ref_out, rtol=0, atol=1e-12)
    for (s, h), Sn in ref_state.items():
        assert np.array_equal(r.state[s, h], Sn.astype(np.float32))
    want_bits = np.vectorize(oracle.round_bf16)(r.out_f64).astype(np.uint16)
    assert np.array_equal(r.out, want_bits)


def test_whole_step_at_head_dim_128():
    p = tiny_problem(seed=14, N=2, H=2, K=128, V=128, num_slots=4, slots=[2, 3], state_scale=0.02)
    r = run(p)
    ref_out, ref_state = torch_reference(p)
    assert np.allclose(r.out_f64, ref_out, rtol=0, atol=1e-12)
    for (s, h), Sn in ref_state.items():
        # fp32 store of the fp64 value: within half an fp32 ulp
        assert np.all(np.abs(r.state[s, h] - Sn) <= np.abs(Sn) * 2.0 ** -24 + 1e-15)


def _decimal_step(p, prec=50):
    """Pure-Python, 50-digit Decimal brute force of the whole step (dense
    matrix form), with its own loops over the layout.  Small shapes only."""
    getcontext().prec = prec
    D = Decimal
    H, K, V, W = p["H"], p["K"], p["V"], p["W"]
    Dq, Dv = H * K, H * V
    C = 2 * Dq + Dv
    w = channel_weights(p)
    qkv, cs = widen(p["qkv"]), widen(p["conv_state"])
    eps = D("1e-6")
    sig = lambda x: 1 / (1 + (-x).exp())  # noqa: E731
    res = {}
    for n, s in enumerate(p["slot_idx"]):
        s = int(s)
        if s <= 0:
            continue
        a = []
        for ch in range(C):
            xs = [D(float(cs[s, ch, t])) for t in range(W - 1)] + [D(float(qkv[n, ch]))]
            y = sum(D(float(w[ch, t])) * xs[t] for t in range(W))
            a.append(y * sig(y))
        for h in range(H):
            qt, kt = a[h * K:(h + 1) * K], a[Dq + h * K: Dq + (h + 1) * K]
            vt = a[2 * Dq + h * V: 2 * Dq + (h + 1) * V]
            rq = 1 / (sum(x * x for x in qt) + eps).sqrt() / D(K).sqrt()
            rk = 1 / (sum(x * x for x in kt) + eps).sqrt()
            qh, kh = [x * rq for x in qt], [x * rk for x in kt]
            b = D(float(widen(p["beta"][n, h])))
            al = [D(float(p["g"][n, h, i])).exp() for i in range(K)]
            S = [[D(float(p["state"][s, h, i, j])) for j in range(V)] for i in range(K)]
            M = [[(1 if i == m else 0) - b * kh[i] * kh[m] for m in range(K)] for i in range(K)]
            Sn = [[sum(M[i][m] * al[m] * S[m][j] for m in range(K)) + b * kh[i] * vt[j]
                   for j in range(V)] for i in range(K)]
            o = [sum(Sn[i][j] * qh[i] for i in range(K)) for j in range(V)]
            ms = sum(x * x for x in o) / V
            r = 1 / (ms + eps).sqrt()
            gt = [D(float(widen(p["gate"][n, h * V + j]))) for j in range(V)]
            nw = [D(float(p["norm_weight"][j])) for j in range(V)]
            res[(n, h)] = ([float(o[j] * r * nw[j] * sig(gt[j])) for j in range(V)],
                           [[float(x) for x in row] for row in Sn])
    return res


def test_whole_step_decimal_brute_force():
    """50-digit brute force agrees with the fp64 oracle to ~1e-13."""
    p = tiny_problem(seed=15, N=3, H=2, K=3, V=5, num_slots=6, slots=[4, 0, 1])
    r = run(p)
    ref = _decimal_step(p)
    for (n, h), (o, Sn) in ref.items():
        got = r.out_f64[n, h * 5:(h + 1) * 5]
        assert np.allclose(got, o, rtol=1e-13, atol=1e-15)
        s = p["slot_idx"][n]
        assert np.array_equal(r.state[s, h], np.asarray(Sn).astype(np.float32))


# ----------------------------------------------------------------- padding


def test_padding_rows_zero_and_slot0_untouched():
    """slot <= 0 (including negative): zero output row for every head; slot 0
    and every unreferenced slot keep their exact bits (P1 padding rule)."""
    p = tiny_problem(seed=16, N=5, H=2, num_slots=7, slots=[0, 3, -2, 0, 6])
    r = run(p)
    HV = p["H"] * p["V"]
    for n in (0, 2, 3):
        assert np.array_equal(r.out[n], np.zeros(HV, np.uint16))
        assert np.array_equal(r.out_f64[n], np.zeros(HV))
    for s in (0, 1, 2, 4, 5):
        assert np.array_equal(r.state[s], p["state"][s])
        assert np.array_equal(r.conv_state[s], p["conv_state"][s])
    assert not np.array_equal(r.state[3], p["state"][3])
    assert r.n_out_of_range == 0


def test_out_of_range_slot_is_zeroed_and_counted():
    p = tiny_problem(seed=17, N=3, H=2, num_slots=5, slots=[2, 5, 99])
    r = run(p)
    assert r.n_out_of_range == 2
    assert not r.out[1].any() and not r.out[2].any()
    untouched = [0, 1, 3, 4]
    assert np.array_equal(r.state[untouched], p["state"][untouched])


def test_all_padding_batch_changes_nothing():
    p = tiny_problem(seed=18, N=4, slots=[0, 0, -1, 0])
    r = run(p)
    assert not r.out.any()
    assert np.array_equal(r.state, p["state"]) and np.array_equal(r.conv_state, p["conv_state"])


def test_norm_off_is_linear_in_q_scale():
    """Norm off returns the raw readout: doubling q_scale doubles it exactly,
    and q_scale = 0 means 1/sqrt(K)."""
    p = tiny_problem(seed=19, out_norm=False, K=4, V=6)
    a = run(p, q_scale=0.125).out_f64
    b = run(p, q_scale=0.25).out_f64
    assert np.array_equal(2 * a, b)
    d = run(p, q_scale=0.0).out_f64
    e = run(p, q_scale=1 / math.sqrt(4)).out_f64
    assert np.array_equal(d, e)


def test_threads_do_not_change_bits():
    p = tiny_problem(seed=20, N=6, H=4, num_slots=9)
    a, b = run(p, threads=1), run(p, threads=4)
    assert np.array_equal(a.out, b.out) and np.array_equal(a.state, b.state)


# ----------------------------------------------------------------- fused gate


def test_softplus_library_and_stability():
    for z in (-700.0, -30.0, -1.5, 0.0, 0.25, 3.0, 30.0, 700.0):
        want = F.softplus(torch.tensor(z, dtype=torch.float64), threshold=1e9).item()
        got = oracle.softplus(z)
        assert math.isfinite(got)
        assert abs(got - want) <= 1e-15 * max(1.0, abs(want)), (z, got, want)
    assert oracle.softplus(0.0) == math.log(2.0)


def test_kda_gate_closed_forms():
    """Bounded gate: z=0 gives lower_bound/2, the range is (lower_bound, 0),
    decreasing in z, slope lower_bound*e^A/4 at 0.  Unbounded gate:
    -e^A log 2 at z=0 and -e^A softplus(z) in general (torch softplus)."""
    lb, A = -5.0, 0.3
    assert oracle.kda_gate(0.0, A, lb) == lb / 2
    assert abs(oracle.kda_gate(60.0, A, lb) - lb) < 1e-12 and abs(oracle.kda_gate(-60.0, A, lb)) < 1e-12
    zs = np.linspace(-6, 6, 41)
    gs = [oracle.kda_gate(z, A, lb) for z in zs]
    assert all(lb < g < 0 for g in gs) and all(a > b for a, b in zip(gs, gs[1:]))
    h = 1e-6
    slope = (oracle.kda_gate(h, A, lb) - oracle.kda_gate(-h, A, lb)) / (2 * h)
    assert abs(slope - lb * math.exp(A) / 4) < 1e-6
    assert abs(oracle.kda_gate(0.0, A, 0.0) + math.exp(A) * math.log(2)) < 1e-15
    for z in (-3.0, 0.7, 9.0):
        want = -math.exp(A) * F.softplus(torch.tensor(z, dtype=torch.float64), threshold=1e9).item()
        assert abs(oracle.kda_gate(z, A, 0.0) - want) < 1e-14


def _gate_problem(seed, lower_bound, with_bias=True):
    p = tiny_problem(seed=seed, N=4, H=3, K=3, V=5, num_slots=8, slots=[3, 0, 7, 1])
    rng = np.random.default_rng(seed + 1000)
    p["g"] = rng.standard_normal(p["g"].shape).astype(np.float32)             # raw logits
    p["beta"] = bf16_bits(rng.standard_normal(p["beta"].shape))               # raw logits
    p.update(fused_gate=True, A_log=rng.standard_normal(3).astype(np.float32) * 0.5,
             dt_bias=(rng.standard_normal(3 * 3).astype(np.float32) if with_bias else None),
             lower_bound=lower_bound)
    return p


@pytest.mark.parametrize("lower_bound", [-5.0, 0.0])
@pytest.mark.parametrize("with_bias", [True, False])
def test_fused_gate_whole_step_equals_preactivated(lower_bound, with_bias):
    """The fused-gate step equals the plain step fed with g and beta that
    torch activates from the same raw logits (library softplus / sigmoid)."""
    p = _gate_problem(71, lower_bound, with_bias)
    r = run(p)
    H, K = p["H"], p["K"]
    z = torch.from_numpy(p["g"].astype(np.float64))
    if with_bias:
        z = z + torch.from_numpy(p["dt_bias"].astype(np.float64)).view(H, K)
    A = torch.from_numpy(p["A_log"].astype(np.float64)).view(1, H, 1).exp()
    if lower_bound < 0:
        g = lower_bound * torch.sigmoid(A * z)
    else:
        g = -A * F.softplus(z, threshold=1e9)
    beta = torch.sigmoid(torch.from_numpy(widen(p["beta"])))
    # Feed the activated values through the float64 library composition.
    q = dict(p)
    q["g"], q["beta"] = g.numpy(), beta.numpy()
    ref_out, ref_state = _torch_reference_f64_gate(q)
    assert np.allclose(r.out_f64, ref_out, rtol=0, atol=1e-12)
    for (s, h), Sn in ref_state.items():
        assert np.array_equal(r.state[s, h], Sn.astype(np.float32))


def _torch_reference_f64_gate(p):
    """torch_reference with g and beta given as float64 activated values."""
    q = dict(p)
    g64, b64 = q.pop("g"), q.pop("beta")
    q["g"] = np.zeros(g64.shape, np.float32)
    q["beta"] = np.zeros(b64.shape, np.uint16)
    # re-run the composition with exact activated values
    H, K, V, W = q["H"], q["K"], q["V"], q["W"]
    Dq, Dv = H * K, H * V
    C = 2 * Dq + Dv
    qkv = torch.from_numpy(widen(q["qkv"]))[:, :C]
    wts = torch.from_numpy(channel_weights(q)).unsqueeze(1)
    cs = torch.from_numpy(widen(q["conv_state"]))
    S_all = torch.from_numpy(q["state"].astype(np.float64))
    gate = torch.from_numpy(widen(q["gate"]))
    nw = torch.from_numpy(q["norm_weight"].astype(np.float64))
    out = torch.zeros(qkv.shape[0], Dv, dtype=torch.float64)
    new_state = {}
    for n in range(qkv.shape[0]):
        s = int(q["slot_idx"][n])
        if s <= 0:
            continue
        window = torch.cat([cs[s], qkv[n].unsqueeze(1)], dim=1)
        a = F.silu(F.conv1d(window.unsqueeze(0), wts, groups=C)[0, :, 0])
        for h in range(H):
            qt, kt = a[h * K:(h + 1) * K], a[Dq + h * K: Dq + (h + 1) * K]
            vt = a[2 * Dq + h * V: 2 * Dq + (h + 1) * V]
            qh = qt / torch.sqrt((qt * qt).sum() + 1e-6) / math.sqrt(K)
            kh = kt / torch.sqrt((kt * kt).sum() + 1e-6)
            b = float(b64[n, h])
            M = torch.eye(K, dtype=torch.float64) - b * torch.outer(kh, kh)
            Sn = M @ torch.diag(torch.exp(torch.from_numpy(np.asarray(g64[n, h])))) @ S_all[s, h] \
                + b * torch.outer(kh, vt)
            o = F.rms_norm(Sn.T @ qh, (V,), weight=nw, eps=1e-6) * torch.sigmoid(gate[n, h * V:(h + 1) * V])
            out[n, h * V:(h + 1) * V] = o
            new_state[(s, h)] = Sn.numpy()
    return out.numpy(), new_state


# ----------------------------------------------------------------- SD layout


@pytest.mark.parametrize("update", [True, False])
def test_sd_conv_state_layout_is_a_transpose(update):
    """The tap-first (SD) conv state gives the same step as the dim-first one
    on the transposed array, and its update is the transpose of the DS
    update (catches SD strides mixed up with DS ones)."""
    p = tiny_problem(seed=81, N=4, H=3, K=3, V=5, num_slots=7, slots=[2, 0, 6, 3])
    ds = run(p, update_conv_state=update)
    q = dict(p)
    q["conv_state"] = np.ascontiguousarray(p["conv_state"].transpose(0, 2, 1))  # [slots, W-1, C]
    sd = run(q, update_conv_state=update, conv_state_sd=True)
    assert np.array_equal(sd.out, ds.out) and np.array_equal(sd.out_f64, ds.out_f64)
    assert np.array_equal(sd.state, ds.state)
    assert np.array_equal(sd.conv_state, np.ascontiguousarray(ds.conv_state.transpose(0, 2, 1)))
    # and the SD update is the shift, read in the SD layout
    C = p["conv_state"].shape[1]
    for n, s in enumerate(p["slot_idx"]):
        if s <= 0 or not update:
            continue
        assert np.array_equal(sd.conv_state[s, 0], q["conv_state"][s, 1])
        assert np.array_equal(sd.conv_state[s, 1], q["conv_state"][s, 2])
        assert np.array_equal(sd.conv_state[s, 2], p["qkv"][n, :C])
