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
