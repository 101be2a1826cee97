"""The chunk form the prefill kernels evaluate equals the token-by-token
recurrence (fp64, CPU).

The prefill computes the decode recurrence over whole sequences
("[ROCm][Perf] Kimi-K3 Remove prefill pipeline stall in chunk KDA",
实现拆解): per token
    S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = S_t^T q_t.
The device path rearranges a chunk of L tokens (cumulative decays G, the
intra-chunk matrices P and R, one triangular solve for [U | W], the state
carried as S_L = Diag(exp G_{L-1}) S0 + K_E^T Delta) and splits each decay
factor exp(G_t - G_s) around a reference token m as exp(G_t - G_m)
exp(G_m - G_s).  This file writes that rearrangement in numpy, independently
of the device code and of the oracle, and checks it against the plain
recurrence (also written here) to fp64 rounding: the algebra the kernels rely
on, pinned without a GPU.
"""
import numpy as np
import pytest

K = V = 16  # head dims of the check (the algebra does not depend on 128)


def recurrence(q, k, v, g, beta, S0):
    S = S0.copy()
    out = np.empty((len(q), V))
    for t in range(len(q)):
        A = np.exp(g[t])[:, None] * S
        S = A + beta[t] * np.outer(k[t], v[t] - A.T @ k[t])
        out[t] = S.T @ q[t]
    return out, S


def chunk_form(q, k, v, g, beta, S0, L, ref=None, mistake=None):
    """The chunk-by-chunk evaluation; `ref` = reference token of the split
    factors (None: exp(G_t - G_s) taken element by element).  `mistake`
    plants one slip (test of the test)."""
    S = S0.copy()
    out = np.empty((len(q), V))
    for c0 in range(0, len(q), L):
        c1 = min(c0 + L, len(q))
        n = c1 - c0
        G = np.cumsum(g[c0:c1], axis=0)                          # [n, K]
        kc, qc, vc, bc = k[c0:c1], q[c0:c1], v[c0:c1], beta[c0:c1]
        if ref is None:
            E = np.exp(G[:, None, :] - G[None, :, :])             # [t, s, K]
            P = np.einsum("ti,si,tsi->ts", kc, kc, E)
            R = np.einsum("ti,si,tsi->ts", qc, kc, E)
        else:
            m = min(ref, n - 1)
            ek = np.exp(G - G[m]) * kc                            # exp(G_t - G_m) k_t
            fk = np.exp(G[m] - G) * kc                            # exp(G_m - G_s) k_s
            eq = np.exp(G - G[m]) * qc
            P, R = ek @ fk.T, eq @ fk.T
        P = np.tril(P, 0 if mistake == "p_with_diagonal" else -1)
        R = np.tril(R, -1 if mistake == "r_without_diagonal" else 0)
        KG, QG = np.exp(G) * kc, np.exp(G) * qc
        KE = (np.exp(G) if mistake == "k_e_forward_decay" else np.exp(G[-1] - G)) * kc
        if mistake == "beta_on_columns":
            M = np.eye(n) + P * bc[None, :]
        else:
            M = np.eye(n) + bc[:, None] * P                       # unit lower triangular
        X = np.empty((n, V + K))
        Y = bc[:, None] * np.concatenate([vc, KG], axis=1)
        for t in range(n):                                        # forward substitution
            X[t] = (Y[t] - M[t, :t] @ X[:t]) / M[t, t]
        U, W = X[:, :V], X[:, V:]
        Delta = U + W @ S if mistake == "delta_sign" else U - W @ S
        out[c0:c1] = QG @ S + R @ Delta
        carry = np.ones(K) if mistake == "no_carry_decay" else np.exp(G[-1])
        S = carry[:, None] * S + KE.T @ Delta
    return out, S


def inputs(rng, T, decay="mild"):
    def unit(x):
        return x / np.linalg.norm(x, axis=1, keepdims=True)
    q = unit(rng.standard_normal((T, K))) * K ** -0.5
    k = unit(rng.standard_normal((T, K)))
    v = rng.standard_normal((T, V))
    if decay == "mild":
        g = -np.log1p(np.exp(rng.standard_normal((T, K))))      # -softplus(N(0,1))
    else:
        g = -20.0 * rng.random((T, K))                           # strong decay
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    S0 = 0.1 * rng.standard_normal((K, V))
    return q, k, v, g, beta, S0


@pytest.mark.parametrize("T", [1, 5, 32, 33, 97])
@pytest.mark.parametrize("ref", [None, 15])
def test_chunk_form_equals_recurrence(T, ref):
    rng = np.random.default_rng(100 + T)
    q, k, v, g, beta, S0 = inputs(rng, T)
    o_ref, S_ref = recurrence(q, k, v, g, beta, S0)
    o, S = chunk_form(q, k, v, g, beta, S0, L=32, ref=ref)
    assert np.allclose(o, o_ref, rtol=0, atol=1e-11)
    assert np.allclose(S, S_ref, rtol=0, atol=1e-11)


@pytest.mark.parametrize("L", [1, 4, 8, 16, 32])
def test_chunk_size_does_not_change_the_result(L):
    rng = np.random.default_rng(7)
    q, k, v, g, beta, S0 = inputs(rng, 70)
    o_ref, S_ref = recurrence(q, k, v, g, beta, S0)
    o, S = chunk_form(q, k, v, g, beta, S0, L=L, ref=None)
    assert np.allclose(o, o_ref, rtol=0, atol=1e-11)
    assert np.allclose(S, S_ref, rtol=0, atol=1e-11)


def test_strong_decay_element_wise_path():
    # cumulative decays of several hundred: the split factors around the
    # reference token would overflow (exp(G_m - G_s) ~ e^300), which is why the
    # device takes such chunks element by element; that path stays exact
    rng = np.random.default_rng(11)
    q, k, v, g, beta, S0 = inputs(rng, 64, decay="strong")
    G = np.cumsum(g[:32], axis=0)
    assert np.abs(G - G[15]).max() > 80.0
    o_ref, S_ref = recurrence(q, k, v, g, beta, S0)
    o, S = chunk_form(q, k, v, g, beta, S0, L=32, ref=None)
    assert np.allclose(o, o_ref, rtol=0, atol=1e-11)
    assert np.allclose(S, S_ref, rtol=0, atol=1e-11)


@pytest.mark.parametrize("mistake", ["p_with_diagonal", "r_without_diagonal", "k_e_forward_decay",
                                     "beta_on_columns", "delta_sign", "no_carry_decay"])
def test_planted_mistakes_are_caught(mistake):
    # each plausible slip in the rearrangement fails the comparison
    rng = np.random.default_rng(5)
    q, k, v, g, beta, S0 = inputs(rng, 70)
    o_ref, S_ref = recurrence(q, k, v, g, beta, S0)
    for ref in (None, 15):
        o, S = chunk_form(q, k, v, g, beta, S0, 32, ref=ref, mistake=mistake)
        assert not (np.allclose(o, o_ref, atol=1e-6) and np.allclose(S, S_ref, atol=1e-6)), mistake


# ---------------------------------------------------------------------------
# The cancellation-safe readout of the chunk form.  With unnormalised q~, k~
# (q^ = r_q q~, k^ = r_k k~, r_q = s / sqrt(|q~|^2 + eps), r_k = 1 / sqrt(|k~|^2
# + eps)) the decode step's own rearrangement of o_t = S_t^T q^_t reads
#     o_t = A_t^T q'_t + c_t v_t,   q'_t = r_q ((q~_t - k~_t) + m_t k~_t),
#     m_t = (|k~_t|^2 + eps - beta_t q~_t.k~_t) r_k^2,  c_t = beta_t (q^_t . k^_t),
# where A_t = Diag(exp g_t) S_{t-1} is the state before token t's update.
# In the chunk form that is: q^ replaced by q', R strictly lower (token t's
# own update enters through c_t v_t), and c_t v_t added to the output.  When
# q~ = k~, q' = r_q m k~ is tiny and nothing of the size of the state cancels.

EPS = 1e-6


def safe_terms(qt, kt, beta, scale, dtype=np.float64):
    sq = np.einsum("ti,ti->t", qt, qt)
    sk = np.einsum("ti,ti->t", kt, kt)
    sqk = np.einsum("ti,ti->t", qt, kt)
    rq = (scale / np.sqrt(sq + EPS)).astype(dtype)
    rk = (1.0 / np.sqrt(sk + EPS)).astype(dtype)
    m = ((sk + EPS - beta * sqk) * rk * rk).astype(dtype)
    c = (beta * sqk * rq * rk).astype(dtype)
    qp = (rq[:, None] * ((qt - kt) + m[:, None] * kt)).astype(dtype)
    return qp, rk[:, None] * kt, rq[:, None] * qt, c


def chunk_form_safe(qt, kt, v, g, beta, S0, L, scale, ref=None, mistake=None, dtype=np.float64):
    """The chunk form with the rearranged readout, in `dtype` arithmetic."""
    qp, kh, _, c = safe_terms(qt, kt, beta, scale, dtype)
    v, g, beta, S = (a.astype(dtype) for a in (v, g, beta, S0.copy()))
    out = np.empty((len(qt), V), dtype)
    for c0 in range(0, len(qt), L):
        c1 = min(c0 + L, len(qt))
        n = c1 - c0
        G = np.cumsum(g[c0:c1], axis=0)
        kc, qc, vc, bc, cc = kh[c0:c1], qp[c0:c1], v[c0:c1], beta[c0:c1], c[c0:c1]
        if ref is None:
            E = np.exp(G[:, None, :] - G[None, :, :])
            P = np.einsum("ti,si,tsi->ts", kc, kc, E)
            R = np.einsum("ti,si,tsi->ts", qc, kc, E)
        else:
            mm = min(ref, n - 1)
            fk = np.exp(G[mm] - G) * kc
            P, R = (np.exp(G - G[mm]) * kc) @ fk.T, (np.exp(G - G[mm]) * qc) @ fk.T
        P = np.tril(P, -1)
        R = np.tril(R, 0 if mistake == "r_with_diagonal" else -1)
        KG, QG = np.exp(G) * kc, np.exp(G) * qc
        KE = np.exp(G[-1] - G) * kc
        M = np.eye(n, dtype=dtype) + bc[:, None] * P
        X = np.empty((n, V + K), dtype)
        Y = bc[:, None] * np.concatenate([vc, KG], axis=1)
        for t in range(n):
            X[t] = Y[t] - M[t, :t] @ X[:t]
        U, W = X[:, :V], X[:, V:]
        Delta = U - W @ S
        diag = 0.0 if mistake == "no_diagonal_term" else cc[:, None] * vc
        out[c0:c1] = QG @ S + R @ Delta + diag
        S = np.exp(G[-1])[:, None] * S + KE.T @ Delta
    return out, S


def unnormalised_inputs(rng, T, cancel=False, sigma=0.1, v_scale=1.0):
    qt = rng.standard_normal((T, K))
    kt = qt.copy() if cancel else rng.standard_normal((T, K))
    v = v_scale * rng.standard_normal((T, V))
    g = np.zeros((T, K)) if cancel else -np.log1p(np.exp(rng.standard_normal((T, K))))
    beta = np.ones(T) if cancel else 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    S0 = sigma * rng.standard_normal((K, V))
    return qt, kt, v, g, beta, S0


@pytest.mark.parametrize("T", [1, 5, 33, 97])
@pytest.mark.parametrize("ref", [None, 15])
def test_safe_readout_chunk_form_equals_recurrence(T, ref):
    rng = np.random.default_rng(300 + T)
    qt, kt, v, g, beta, S0 = unnormalised_inputs(rng, T)
    _, kh, qh, _ = safe_terms(qt, kt, beta, K ** -0.5)
    o_ref, S_ref = recurrence(qh, kh, v, g, beta, S0)
    o, S = chunk_form_safe(qt, kt, v, g, beta, S0, 32, K ** -0.5, ref=ref)
    assert np.allclose(o, o_ref, rtol=0, atol=1e-11)
    assert np.allclose(S, S_ref, rtol=0, atol=1e-11)


@pytest.mark.parametrize("mistake", ["r_with_diagonal", "no_diagonal_term"])
def test_safe_readout_planted_mistakes_are_caught(mistake):
    rng = np.random.default_rng(9)
    qt, kt, v, g, beta, S0 = unnormalised_inputs(rng, 70)
    _, kh, qh, _ = safe_terms(qt, kt, beta, K ** -0.5)
    o_ref, _ = recurrence(qh, kh, v, g, beta, S0)
    o, _ = chunk_form_safe(qt, kt, v, g, beta, S0, 32, K ** -0.5, ref=15, mistake=mistake)
    assert not np.allclose(o, o_ref, atol=1e-6), mistake


def test_safe_readout_keeps_the_output_where_the_plain_one_cancels():
    # q~ = k~, beta = 1, g = 0, a state of N(0, 100), small v: every o_t is
    # orders of magnitude below Q_G S0.  In fp32 arithmetic the plain chunk
    # readout (Q_G S0 + R Delta) loses o_t; the rearranged one keeps it to a
    # small fraction of a bf16 ulp (2^-8 relative).
    rng = np.random.default_rng(21)
    qt, kt, v, g, beta, S0 = unnormalised_inputs(rng, 64, cancel=True, sigma=100.0, v_scale=1e-3)
    scale = K ** -0.5
    _, kh, qh, _ = safe_terms(qt, kt, beta, scale)
    o_ref, _ = recurrence(qh, kh, v, g, beta, S0)
    rel = lambda o: np.max(np.abs(o - o_ref)) / np.max(np.abs(o_ref))  # noqa: E731
    f32 = np.float32
    o_plain, _ = chunk_form(qh.astype(f32), kh.astype(f32), v.astype(f32), g.astype(f32), beta.astype(f32),
                            S0.astype(f32), 32, ref=15)
    o_safe, _ = chunk_form_safe(qt, kt, v, g, beta, S0, 32, scale, ref=15, dtype=f32)
    assert rel(o_plain) > 2.0 ** -8
    assert rel(o_safe) < 2.0 ** -12
