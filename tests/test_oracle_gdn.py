"""Pins for the oracle's linear branch: the GDN state update and the
fixed-budget routing that feeds it.

Source: page "迈向线性的关键：分析驱动的 Transformer 线性化", section
线性注意力替换机制 (the GDN equation with a scalar gate) and section
填补近似缺口的实用设计 (tokens outside the sink + window budget go to the
linear path).
"""
import numpy as np
import pytest


def _unit_rows(rng, n, d):
    x = rng.standard_normal((n, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def _product_form_state(K, V, alpha, beta, absorbed, d):
    """S = sum_i beta_i [prod_{j in absorbed, j > i} alpha_j (I - beta_j k_j k_j^T)] k_i v_i^T,
    later tokens on the left: the unrolled effective-weight form, built by brute force."""
    S = np.zeros((d, d))
    for i in absorbed:
        M = np.eye(d)
        for j in absorbed:
            if j > i:
                M = alpha[j] * (np.eye(d) - beta[j] * np.outer(K[j], K[j])) @ M
        S += beta[i] * M @ np.outer(K[i], V[i])
    return S


@pytest.mark.parametrize("n_sinks,window,T,d", [(0, 1, 16, 8), (3, 2, 16, 8), (2, 5, 14, 6), (0, 4, 9, 4)])
def test_recurrence_equals_explicit_product_form(oracle_mod, n_sinks, window, T, d):
    rng = np.random.default_rng(10 + T + window)
    Q = rng.standard_normal((T, d))
    K = _unit_rows(rng, T, d)
    V = rng.standard_normal((T, d))
    g = -0.1 * np.log1p(np.exp(rng.standard_normal(T)))
    beta = 1 / (1 + np.exp(-rng.standard_normal(T)))
    alpha = np.exp(g)
    o, S = oracle_mod.gdn_delayed(Q, K, V, g, beta, n_sinks, window)
    for p in range(T):
        absorbed = [j for j in range(T) if n_sinks <= j <= p - window]
        Sp = _product_form_state(K, V, alpha, beta, absorbed, d)
        np.testing.assert_allclose(o[p], Q[p] @ Sp, rtol=1e-12, atol=1e-13)
    final = [j for j in range(T) if n_sinks <= j <= T - 1 - window]
    np.testing.assert_allclose(S, _product_form_state(K, V, alpha, beta, final, d), rtol=1e-12,
                               atol=1e-13)


def test_delta_rule_step_identity(oracle_mod):
    # With a unit key, k^T S_t = (1 - beta) alpha k^T S_{t-1} + beta v^T for any history.
    rng = np.random.default_rng(11)
    d, T = 16, 30
    K = _unit_rows(rng, T, d)
    V = rng.standard_normal((T, d))
    g = -0.2 * rng.random(T)
    beta = rng.random(T)
    beta[5] = 1.0
    # one extra trailing row: with no sinks and a 1-token window, a run over the
    # first t+1 rows absorbs tokens 0..t-1
    Q1 = np.zeros((T + 1, d))
    K1, V1 = np.vstack([K, K[:1]]), np.vstack([V, V[:1]])
    g1, b1 = np.append(g, 0.0), np.append(beta, 0.0)
    states = [np.zeros((d, d))]
    for t in range(1, T + 1):
        _, S = oracle_mod.gdn_delayed(Q1[: t + 1], K1[: t + 1], V1[: t + 1], g1[: t + 1],
                                      b1[: t + 1], 0, 1)
        states.append(S)  # states[t]: after absorbing tokens 0..t-1
    states = states[1:]   # states[t]: after absorbing tokens 0..t
    for t in range(1, T):
        lhs = K[t] @ states[t]
        rhs = (1 - beta[t]) * np.exp(g[t]) * (K[t] @ states[t - 1]) + beta[t] * V[t]
        np.testing.assert_allclose(lhs, rhs, rtol=1e-11, atol=1e-12)
    # beta = 1 stores the value exactly: querying with the key returns it
    np.testing.assert_allclose(K[5] @ states[5], V[5], rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_with_unit_gates_recall_values(oracle_mod):
    rng = np.random.default_rng(12)
    d, T = 8, 8
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    K = Qm.T[:T]
    V = rng.standard_normal((T + 1, d))
    K1 = np.vstack([K, K[:1]])
    o, S = oracle_mod.gdn_delayed(np.zeros((T + 1, d)), K1, V, np.zeros(T + 1), np.ones(T + 1), 0, 1)
    for i in range(T):
        np.testing.assert_allclose(K[i] @ S, V[i], rtol=1e-12, atol=1e-12)


def test_beta_zero_keeps_state_empty(oracle_mod):
    rng = np.random.default_rng(13)
    d, T = 8, 20
    o, S = oracle_mod.gdn_delayed(rng.standard_normal((T, d)), _unit_rows(rng, T, d),
                                  rng.standard_normal((T, d)), -0.1 * rng.random(T), np.zeros(T), 2, 3)
    assert np.abs(o).max() == 0.0 and np.abs(S).max() == 0.0


def test_erase_off_is_gated_linear_accumulation(oracle_mod):
    # Test switch: the GLA update S_t = alpha_t S_{t-1} + k_t v_t^T has the closed form
    # S_T = sum_i (prod_{j>i} alpha_j) k_i v_i^T.
    rng = np.random.default_rng(14)
    d, T = 6, 12
    K = rng.standard_normal((T, d))
    V = rng.standard_normal((T, d))
    g = -0.3 * rng.random(T)
    _, S = oracle_mod.gdn_delayed(np.zeros((T, d)), K, V, g, rng.random(T), 0, 1, erase_off=True)
    ref = np.zeros((d, d))
    for i in range(T - 1):
        ref += np.exp(g[i + 1: T - 1].sum()) * np.outer(K[i], V[i])
    np.testing.assert_allclose(S, ref, rtol=1e-12, atol=1e-13)


def _routing_rows():
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", "budget_routing.txt")
    rows = []
    for line in open(path, encoding="utf-8"):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(tuple(int(x) for x in line.split()))
    return rows


@pytest.mark.parametrize("n_sinks,window,p,n_keys,n_absorbed", _routing_rows())
def test_budget_routing_golden(oracle_mod, n_sinks, window, p, n_keys, n_absorbed):
    # Softmax key count from the visibility predicate.
    assert sum(oracle_mod.key_visible(p, j, n_sinks, window) for j in range(p + 1)) == n_keys
    # Absorbed-token count from the linear branch itself: GLA switch, unit gates,
    # one-hot keys and values, so o_lin[p] counts the tokens held in the state.
    T = p + 1
    d = T
    K = np.eye(T)
    V = np.eye(T)
    Q = np.ones((T, d))
    o, _ = oracle_mod.gdn_delayed(Q, K, V, np.zeros(T), np.ones(T), n_sinks, window, erase_off=True)
    held = o[p]
    assert held.sum() == n_absorbed
    # exactly the non-sink tokens that have left the window
    np.testing.assert_array_equal(np.nonzero(held)[0], np.arange(n_sinks, n_sinks + n_absorbed))
