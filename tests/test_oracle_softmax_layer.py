"""Pins for the oracle's exact branch (sink + sliding-window softmax) and for
the composed layer.

Sources: page "迈向线性的关键：分析驱动的 Transformer 线性化", section
填补近似缺口的实用设计 (8 sinks + sliding window keep exact attention) and
Lemma 1 in section 从 softmax 到 delta 规则的一阶近似 (the 1/sqrt(d) scale);
page "Untangling Component Imbalance in Hybrid Linear Attention Conversion",
section 关键设计 (1) (inference-time weighting of the two branches).
"""
import numpy as np
import pytest
import scipy.special
import torch

from linearized_attention_rope_gb300 import synth


def test_wide_window_is_full_causal_softmax(oracle_mod):
    rng = np.random.default_rng(20)
    T, d = 40, 16
    q, k, v = (rng.standard_normal((T, d)) for _ in range(3))
    o = oracle_mod.window_softmax(q, k, v, 0, T)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        is_causal=True)[0].numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)


def test_window_of_one_returns_current_value(oracle_mod):
    rng = np.random.default_rng(21)
    T, d = 25, 8
    q, k, v = (rng.standard_normal((T, d)) for _ in range(3))
    np.testing.assert_allclose(oracle_mod.window_softmax(q, k, v, 0, 1), v, rtol=1e-15)


@pytest.mark.parametrize("n_sinks,window", [(8, 56), (3, 5), (0, 7), (8, 1)])
def test_attention_support_and_weights(oracle_mod, n_sinks, window):
    # One-hot values turn the output row into the attention distribution itself.
    rng = np.random.default_rng(22 + window)
    T = d = 90  # one-hot values need d = T
    q, k = rng.standard_normal((T, d)), rng.standard_normal((T, d))
    o = oracle_mod.window_softmax(q, k, np.eye(T), n_sinks, window)
    for p in range(T):
        support = [j for j in range(p + 1) if j < n_sinks or j > p - window]
        np.testing.assert_array_equal(np.nonzero(o[p])[0], support)
        logits = (k[support] @ q[p]) / np.sqrt(d)
        np.testing.assert_allclose(o[p, support], scipy.special.softmax(logits), rtol=1e-12)


def _unit_inputs(L=80, d=16, seed=30):
    rng = np.random.default_rng(seed)
    mu = rng.standard_normal(d)
    mu /= np.linalg.norm(mu)
    return dict(q=rng.standard_normal((L, d)), k=mu + 0.3 * rng.standard_normal((L, d)),
                v=rng.standard_normal((L, d)), g=-0.1 * np.log1p(np.exp(rng.standard_normal(L))),
                beta=1 / (1 + np.exp(-rng.standard_normal(L))),
                wq=rng.standard_normal((d, 8)) / np.sqrt(8), wk=rng.standard_normal((d, 8)) / np.sqrt(8),
                wv=rng.standard_normal((d, 8)) / np.sqrt(8))


def _run(oracle_mod, cfg, x, lam, want=()):
    return oracle_mod.layer_unit(cfg, x["q"], x["k"], x["v"], x["g"], x["beta"], lam, x["wq"],
                                 x["wk"], x["wv"], want=want)


def test_layer_wiring_follows_the_feature_path(oracle_mod):
    x = _unit_inputs()
    cfg = oracle_mod.OracleCfg(d=16, n_sinks=4, window=10, rope_base=500000.0)
    r = _run(oracle_mod, cfg, x, 0.7, want=("qr", "kr", "qhat", "khat", "vhat", "o_sm", "o_lin"))
    qr, kr = oracle_mod.rope(x["q"], 500000.0), oracle_mod.rope(x["k"], 500000.0)
    np.testing.assert_allclose(r["qr"], qr, rtol=1e-15)
    np.testing.assert_allclose(r["qhat"], oracle_mod.l2norm(oracle_mod.conv(qr, x["wq"])), rtol=1e-14)
    np.testing.assert_allclose(r["khat"], oracle_mod.l2norm(oracle_mod.conv(kr, x["wk"])), rtol=1e-14)
    np.testing.assert_allclose(r["vhat"], oracle_mod.conv(x["v"], x["wv"]), rtol=1e-14)
    # the exact branch sees RoPE'd q, k and the raw v, not the convolved features
    np.testing.assert_allclose(r["o_sm"], oracle_mod.window_softmax(qr, kr, x["v"], 4, 10), rtol=1e-14)
    o_lin, S = oracle_mod.gdn_delayed(r["qhat"], r["khat"], r["vhat"], x["g"], x["beta"], 4, 10)
    np.testing.assert_allclose(r["o_lin"], o_lin, rtol=1e-14)
    np.testing.assert_allclose(r["S"], S, rtol=1e-14)
    np.testing.assert_allclose(r["o"], r["o_sm"] + 0.7 * r["o_lin"], rtol=1e-14)


def test_lambda_zero_and_softmax_off_isolate_branches(oracle_mod):
    x = _unit_inputs(seed=31)
    cfg = oracle_mod.OracleCfg(d=16, n_sinks=2, window=6)
    full = _run(oracle_mod, cfg, x, 1.3, want=("o_sm", "o_lin"))
    assert np.abs(full["o_lin"]).max() > 0.05  # the linear branch is really used
    only_sm = _run(oracle_mod, cfg, x, 0.0)
    np.testing.assert_array_equal(only_sm["o"], full["o_sm"])
    cfg_off = oracle_mod.OracleCfg(d=16, n_sinks=2, window=6, softmax_off=True)
    only_lin = _run(oracle_mod, cfg_off, x, 1.3)
    np.testing.assert_allclose(only_lin["o"], 1.3 * full["o_lin"], rtol=1e-15)


def test_budget_covering_sequence_leaves_state_empty(oracle_mod):
    x = _unit_inputs(L=40, seed=32)
    cfg = oracle_mod.OracleCfg(d=16, n_sinks=8, window=32)  # budget 40 >= length
    r = _run(oracle_mod, cfg, x, 1.0, want=("o_sm", "o_lin"))
    assert np.abs(r["S"]).max() == 0.0 and np.abs(r["o_lin"]).max() == 0.0
    np.testing.assert_array_equal(r["o"], r["o_sm"])


def test_first_absorption_happens_at_budget(oracle_mod):
    x = _unit_inputs(L=30, seed=33)
    cfg = oracle_mod.OracleCfg(d=16, n_sinks=3, window=5)
    r = _run(oracle_mod, cfg, x, 1.0, want=("o_lin",))
    assert np.abs(r["o_lin"][:8]).max() == 0.0  # positions < n_sinks + window
    assert np.abs(r["o_lin"][8]).max() > 0.0


def test_synthetic_recipe_shapes():
    wl = synth.small("t", [5, 9], n_q_heads=4, n_kv_heads=2, head_dim=8, decode_steps=3)
    x = synth.make_inputs(wl)
    assert x["q"].shape == (14, 4, 8) and x["k"].shape == (14, 2, 8)
    assert x["cu_seqlens"].tolist() == [0, 5, 14]
    assert x["dq"].shape == (3, 2, 4, 8) and x["dg"].shape == (3, 2, 4)
    assert float(x["g"].max()) < 0 and 0 < float(x["beta"].min()) and float(x["beta"].max()) < 1
    again = synth.make_inputs(wl)
    assert torch.equal(x["k"], again["k"])  # seeded
