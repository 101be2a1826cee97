"""The decode readout in the regime where it cancels: q~ parallel to k~,
beta = 1, no decay, a large state and a small v.  Then o = S'^T q^ is tiny
while w = A^T q^ is not, and how the fp32 kernel forms o and the RMSNorm sum
decides whether the output survives.

An fp32 numpy restatement of the decode kernel's arithmetic (same
association of the sums over 16-row warp blocks, same rounding points; numpy
cannot fuse multiply-adds, so it rounds a little more often) is run in three
forms against the fp64 oracle:
  - "expansion": o = w + (q^.k^) delta with sum o^2 expanded as
    sum w^2 + 2 (q^.k^) sum w delta + (q^.k^)^2 sum delta^2;
  - "direct": the same o, sum o^2 taken from o;
  - "rearranged": the kernel's form, o = rq ((w~ - u~) + m u~) + beta (q^.k^) v
    with m = (|k~|^2 + 1e-6 - beta q~.k~) rk^2, sum o^2 taken from o.
The expansion must miss the pages' 3e-2 output tolerance on these inputs
(which shows they reach the regime), the rearranged form must meet it and
stay within one bf16 ulp of the exact output.  The GPU test with the same
inputs is in test_gpu_parity.py.
"""
import numpy as np
import pytest

import kda_testlib as T
from linear_attention_decode_04_gb300 import workloads as W

f32 = np.float32


def _emulate(x, form: str) -> np.ndarray:
    """Output (fp32, before bf16 rounding) of every row, padding rows zero."""
    N, H = x.N, x.H
    D = H * 128
    out = np.zeros((N, D), f32)
    cs_all = W.bf16_bits_to_f32(x.conv_state)
    xin_all = W.bf16_bits_to_f32(x.qkv)
    nw = x.norm_weight.astype(f32)
    for n in range(N):
        s = int(x.slot_idx[n])
        if s <= 0:
            continue
        for h in range(H):
            act = []
            for c in range(3):
                sl = slice(c * D + h * 128, c * D + (h + 1) * 128)
                wc = x.conv_weight[c, :, h * 128:(h + 1) * 128]
                y = np.zeros(128, f32)
                for t in range(3):
                    y = (y + wc[t] * cs_all[s, sl, t]).astype(f32)
                y = (y + wc[3] * xin_all[n, sl]).astype(f32)
                act.append((y / (f32(1) + np.exp(-y))).astype(f32))
            qt, kt, vt = act
            A = (x.state[s, h] * np.exp(x.g[n, h]).astype(f32)[:, None]).astype(f32)
            ut = np.zeros(128, f32)
            wt = np.zeros(128, f32)
            pq, pk, pqk = [], [], []
            for wp in range(8):
                rows = range(16 * wp, 16 * wp + 16)
                pu = np.zeros(128, f32)
                pw = np.zeros(128, f32)
                for i in rows:
                    pu = (pu + kt[i] * A[i]).astype(f32)
                    pw = (pw + qt[i] * A[i]).astype(f32)
                ut = (ut + pu).astype(f32)
                wt = (wt + pw).astype(f32)
                idx = np.array(rows)
                pq.append(f32(np.sum(qt[idx] * qt[idx], dtype=f32)))
                pk.append(f32(np.sum(kt[idx] * kt[idx], dtype=f32)))
                pqk.append(f32(np.sum(qt[idx] * kt[idx], dtype=f32)))
            ssq = f32(sum(pq, f32(0)))
            ssk = f32(sum(pk, f32(0)))
            sqk = f32(sum(pqk, f32(0)))
            rq = f32(f32(128 ** -0.5) / np.sqrt(ssq + f32(1e-6)))
            rk = f32(f32(1) / np.sqrt(ssk + f32(1e-6)))
            beta = W.bf16_bits_to_f32(x.beta[n, h])
            d = (beta * (vt - rk * ut)).astype(f32)
            if form == "rearranged":
                m = f32(f32(np.float64(ssk) - np.float64(beta) * np.float64(sqk)) + f32(1e-6)) * rk * rk
                bqk = f32(beta * sqk * rq * rk)
                inner = (np.float64(m) * ut.astype(np.float64) + (wt - ut).astype(np.float64)).astype(f32)
                o = (np.float64(bqk) * vt.astype(np.float64) + (rq * inner).astype(np.float64)).astype(f32)
            else:
                w = (rq * wt).astype(f32)
                qk = f32(sqk * rq * rk)
                o = (w + qk * d).astype(f32)
            if not x.spec.out_norm:
                y = o
            else:
                if form == "expansion":
                    w = (rq * wt).astype(f32)
                    qk = f32(sqk * rq * rk)
                    sww = np.sum(w * w, dtype=f32)
                    swd = np.sum(w * d, dtype=f32)
                    sdd = np.sum(d * d, dtype=f32)
                    ss = f32(sww + qk * (f32(2) * swd + qk * sdd))
                else:
                    ss = f32(np.sum(o * o, dtype=f32))
                rr = f32(f32(1) / np.sqrt(max(ss, f32(0)) / f32(128) + f32(x.spec.eps)))
                gate = W.bf16_bits_to_f32(x.gate[n, h * 128:(h + 1) * 128])
                y = (o * rr * nw * (f32(1) / (f32(1) + np.exp(-gate)))).astype(f32)
            out[n, h * 128:(h + 1) * 128] = y
    return out


def _errors(x, ref, form):
    got = W.bf16_bits_to_f32(W.f32_to_bf16_bits(_emulate(x, form))).astype(np.float64)
    want = W.bf16_bits_to_f32(ref.out).astype(np.float64)
    exact = ref.out_f64
    worst = float(np.abs(got - want).max())
    n_beyond_ulp = int(np.count_nonzero(np.abs(got - exact) > T.bf16_ulp(exact) + T.TIGHT_ABS))
    return worst, n_beyond_ulp


@pytest.mark.parametrize("sigma,v_scale", [(10.0, 1e-2), (100.0, 1e-1)])
def test_rearranged_readout_survives_where_expansion_fails(sigma, v_scale):
    x = T.cancellation_inputs(sigma, v_scale, N=3, H=2)
    ref = T.run_oracle(x)
    exp_worst, _ = _errors(x, ref, "expansion")
    assert exp_worst > T.OUT_ATOL, f"inputs do not reach the cancelling regime ({exp_worst})"
    worst, beyond = _errors(x, ref, "rearranged")
    assert worst <= T.OUT_ATOL and beyond == 0, (worst, beyond)
    # the direct sum alone passes the pages' tolerance but not the ulp bound
    d_worst, _ = _errors(x, ref, "direct")
    assert d_worst <= T.OUT_ATOL


def test_rearranged_readout_norm_off():
    x = T.cancellation_inputs(30.0, 3e-3, N=3, H=2, out_norm=False)
    ref = T.run_oracle(x)
    worst, beyond = _errors(x, ref, "rearranged")
    assert worst <= T.OUT_ATOL and beyond == 0, (worst, beyond)


def test_rearranged_readout_on_the_ordinary_workload():
    """On the pages' value distributions all three forms agree with the oracle."""
    x = W.make_inputs(W.PR1_REF)
    ref = T.run_oracle(x)
    for form in ("expansion", "direct", "rearranged"):
        worst, beyond = _errors(x, ref, form)
        assert worst <= T.OUT_ATOL and beyond == 0, (form, worst, beyond)
