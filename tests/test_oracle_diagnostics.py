"""Pins for the oracle's component-usage diagnostics: key concentration and
projection residual of page "迈向线性的关键：分析驱动的 Transformer 线性化",
sections 从 softmax 到 delta 规则的一阶近似 (Lemma 2: projection onto the
orthogonal complement of the mean key) and 填补近似缺口的实用设计 (the
residual grows when keys do not share one direction).  Each case has a closed
form."""
import math

import numpy as np


def test_identical_keys_are_fully_concentrated(oracle_mod):
    kr = np.tile(np.array([3.0, -1.0, 2.0, 0.5]), (20, 1))
    conc, res = oracle_mod.key_stats(kr)
    np.testing.assert_allclose(conc, 1.0, rtol=1e-14)
    np.testing.assert_allclose(res, 0.0, atol=1e-14)


def test_orthonormal_keys_follow_the_closed_form(oracle_mod):
    # u_p = e_p: m_p = (e_0 + .. + e_p)/(p+1), |m_p| = 1/sqrt(p+1), mhat.u_p = 1/sqrt(p+1), so the
    # residual is sqrt(1 - 1/(p+1)); scaling a key changes nothing (keys are normalised)
    d = 12
    kr = np.eye(d) * np.arange(1, d + 1)[:, None]
    conc, res = oracle_mod.key_stats(kr)
    p = np.arange(d)
    np.testing.assert_allclose(conc, 1.0 / np.sqrt(p + 1), rtol=1e-13)
    np.testing.assert_allclose(res, np.sqrt(1.0 - 1.0 / (p + 1)), rtol=1e-13, atol=1e-15)


def test_residual_is_the_sine_to_the_mean_direction(oracle_mod):
    # two unit keys at angle phi: the mean bisects them, so each makes phi/2 with it; the residual at
    # p = 1 is sin(phi/2) and the concentration cos(phi/2)
    for phi in (0.1, 0.7, 2.0, 3.0):
        kr = np.array([[1.0, 0.0, 0.0], [math.cos(phi), math.sin(phi), 0.0]])
        conc, res = oracle_mod.key_stats(kr)
        assert res[0] == 0.0 and conc[0] == 1.0
        assert res[1] == pytest_approx(math.sin(phi / 2))
        assert conc[1] == pytest_approx(math.cos(phi / 2))


def test_opposite_keys_leave_no_mean_direction(oracle_mod):
    kr = np.array([[0.0, 2.0], [0.0, -5.0]])
    conc, res = oracle_mod.key_stats(kr)
    assert conc[1] == 0.0 and res[1] == 1.0


def test_random_keys_match_a_direct_restatement_with_library_routines(oracle_mod):
    rng = np.random.default_rng(7)
    kr = rng.standard_normal((50, 16)) + 2.0 * np.eye(16)[3]
    conc, res = oracle_mod.key_stats(kr)
    u = kr / np.linalg.norm(kr, axis=1, keepdims=True)
    m = np.cumsum(u, axis=0) / np.arange(1, 51)[:, None]
    mh = m / np.linalg.norm(m, axis=1, keepdims=True)
    resid = u - np.sum(mh * u, axis=1, keepdims=True) * mh
    np.testing.assert_allclose(conc, np.linalg.norm(m, axis=1), rtol=1e-12)
    np.testing.assert_allclose(res, np.linalg.norm(resid, axis=1), rtol=1e-10, atol=1e-12)


def pytest_approx(x):
    import pytest

    return pytest.approx(x, rel=1e-12, abs=1e-14)
