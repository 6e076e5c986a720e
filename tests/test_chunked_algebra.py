"""The chunked (UT-transform) form of the delayed GDN branch, restated in
numpy fp64 and checked against the oracle's token-by-token recurrence.

This pins the algebra the chunked CUDA kernel implements.  Within a chunk of
C tokens with gates cumulated as G_r = sum_{i<=r} g_i:
  A[r,i] = beta_r e^{G_r - G_i} k_r . k_i  (i < r),   T = (I + A)^{-1}
  U~ = T diag(beta) V,   Wm = T diag(beta e^G) K,    U = U~ - Wm S0
  O  = diag(e^G) Q S0 + (Q K^T (.) M) U,  M[r,i] = e^{G_r - G_i} (i <= r)
  S1 = e^{G_C} S0 + (diag(e^{G_C - G}) K)^T U
where Q holds the queries shifted by the window (query p reads the state
after token p - W).  GDN equation: page "迈向线性的关键：分析驱动的 Transformer
线性化", section 线性注意力替换机制.
"""
import numpy as np
import pytest


def chunked_delayed_gdn(Qh, Kh, Vh, g, beta, n_sinks, window, C=64):
    L, d = Qh.shape
    o = np.zeros((L, d))
    S = np.zeros((d, d))
    start, stop = n_sinks, L - window  # GDN token range; query of token t is t + window
    for c0 in range(start, max(stop, start), C):
        c1 = min(c0 + C, stop)
        K, V, Q = Kh[c0:c1], Vh[c0:c1], Qh[c0 + window:c1 + window]
        b = beta[c0:c1]
        G = np.cumsum(g[c0:c1])
        n = c1 - c0
        decay = np.exp(G[:, None] - G[None, :])
        A = np.tril(b[:, None] * decay * (K @ K.T), -1)
        T = np.linalg.inv(np.eye(n) + A)
        Ut = T @ (b[:, None] * V)
        Wm = T @ ((b * np.exp(G))[:, None] * K)
        U = Ut - Wm @ S
        P = np.tril(Q @ K.T * decay)
        o[c0 + window:c1 + window] = np.exp(G)[:, None] * (Q @ S) + P @ U
        S = np.exp(G[-1]) * S + (np.exp(G[-1] - G)[:, None] * K).T @ U
    return o, S


@pytest.mark.parametrize("L,n_sinks,window,C", [(512, 8, 56, 64), (300, 8, 56, 64), (700, 8, 120, 64),
                                                (130, 0, 1, 16), (40, 8, 56, 64), (1000, 8, 888, 64)])
def test_chunked_form_equals_recurrence(oracle_mod, L, n_sinks, window, C):
    rng = np.random.default_rng(L + window)
    d = 32
    mu = rng.standard_normal(d)
    mu /= np.linalg.norm(mu)
    K = mu + 0.3 * rng.standard_normal((L, d))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    Q = rng.standard_normal((L, d))
    Q /= np.linalg.norm(Q, axis=1, keepdims=True)
    V = rng.standard_normal((L, d))
    g = -0.1 * np.log1p(np.exp(rng.standard_normal(L)))
    beta = 1 / (1 + np.exp(-rng.standard_normal(L)))
    o_ref, S_ref = oracle_mod.gdn_delayed(Q, K, V, g, beta, n_sinks, window)
    o, S = chunked_delayed_gdn(Q, K, V, g, beta, n_sinks, window, C)
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S, S_ref, rtol=1e-11, atol=1e-12)
