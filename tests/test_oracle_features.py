"""Pins for the oracle's feature path (RoPE -> short conv -> L2 norm).

Each check compares the oracle with something other than itself: closed
forms, invariants, or a library routine.  Source: page "迈向线性的关键：分析驱动的
Transformer 线性化", section 实践建议 item 3 (short conv of width 8 after RoPE
and before L2 normalisation); RoPE base 500000 is the workload's.
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore")
BASE = 500000.0


def test_rope_position_zero_is_identity(oracle_mod):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((1, 16))
    np.testing.assert_allclose(oracle_mod.rope(x, BASE), x, rtol=0, atol=1e-15)


def test_rope_preserves_norm_of_every_pair(oracle_mod):
    rng = np.random.default_rng(2)
    d = 64
    x = rng.standard_normal((300, d))
    y = oracle_mod.rope(x, BASE)
    h = d // 2
    np.testing.assert_allclose(x[:, :h] ** 2 + x[:, h:] ** 2, y[:, :h] ** 2 + y[:, h:] ** 2,
                               rtol=1e-12)


def test_rope_first_pair_turns_one_radian_per_position(oracle_mod):
    # theta_0 = base^0 = 1: unit vector e_0 at position p becomes (cos p) e_0 + (sin p) e_{d/2}.
    d = 8
    L = 40
    x = np.zeros((L, d))
    x[:, 0] = 1.0
    y = oracle_mod.rope(x, BASE)
    p = np.arange(L)
    np.testing.assert_allclose(y[:, 0], np.cos(p), atol=1e-13)
    np.testing.assert_allclose(y[:, d // 2], np.sin(p), atol=1e-13)
    others = np.delete(y, [0, d // 2], axis=1)
    assert np.abs(others).max() == 0.0


def test_rope_pair_frequencies_form_geometric_spectrum(oracle_mod):
    # Pair i turns by base^(-2i/d) per position: consecutive pairs differ by the
    # constant ratio base^(-2/d), the last pair turns by base^(-(d-2)/d).
    d = 16
    x = np.zeros((2, d))
    x[:, : d // 2] = 1.0
    y = oracle_mod.rope(x, BASE)
    ang = np.arctan2(y[1, d // 2:], y[1, : d // 2])
    ratio = ang[1:] / ang[:-1]
    np.testing.assert_allclose(ratio, BASE ** (-2.0 / d), rtol=1e-10)
    assert ang[0] == pytest.approx(1.0, abs=1e-14)


def test_rope_scores_depend_only_on_relative_position(oracle_mod):
    rng = np.random.default_rng(3)
    d = 32
    qv, kv = rng.standard_normal(d), rng.standard_normal(d)
    L = 200
    Q = np.tile(qv, (L, 1))
    K = np.tile(kv, (L, 1))
    Qr, Kr = oracle_mod.rope(Q, BASE), oracle_mod.rope(K, BASE)
    for m, n, s in [(10, 3, 50), (7, 7, 120), (100, 0, 99), (5, 60, 17)]:
        a = Qr[m] @ Kr[n]
        b = Qr[m + s] @ Kr[n + s]
        assert a == pytest.approx(b, rel=1e-10, abs=1e-12)
    # ... and do change with the offset
    assert abs(Qr[10] @ Kr[3] - Qr[10] @ Kr[4]) > 1e-6


def test_rope_matches_complex_multiplication(oracle_mod):
    # A second formulation: pair (a, b) as the complex number a + ib times e^{i p theta}.
    rng = np.random.default_rng(4)
    d, L = 16, 33
    x = rng.standard_normal((L, d))
    y = oracle_mod.rope(x, BASE)
    h = d // 2
    z = x[:, :h] + 1j * x[:, h:]
    spectrum = np.logspace(0, -(d - 2) / d, h, base=BASE)  # base^0 .. base^(-(d-2)/d)
    zr = z * np.exp(1j * np.outer(np.arange(L), spectrum))
    np.testing.assert_allclose(y[:, :h], zr.real, atol=1e-12)
    np.testing.assert_allclose(y[:, h:], zr.imag, atol=1e-12)


def test_conv_last_tap_is_identity(oracle_mod):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((50, 12))
    w = np.zeros((12, 8))
    w[:, 7] = 1.0
    np.testing.assert_array_equal(oracle_mod.conv(x, w), x)


def test_conv_first_tap_delays_by_seven_with_zero_padding(oracle_mod):
    rng = np.random.default_rng(6)
    x = rng.standard_normal((50, 12))
    w = np.zeros((12, 8))
    w[:, 0] = 1.0
    y = oracle_mod.conv(x, w)
    np.testing.assert_array_equal(y[:7], 0.0)
    np.testing.assert_array_equal(y[7:], x[:-7])


def test_conv_matches_numpy_convolve(oracle_mod):
    rng = np.random.default_rng(7)
    L, d = 40, 6
    x = rng.standard_normal((L, d))
    w = rng.standard_normal((d, 8)) * math.sqrt(1 / 8)
    y = oracle_mod.conv(x, w)
    for c in range(d):
        ref = np.convolve(x[:, c], w[c, ::-1], mode="full")[:L]
        np.testing.assert_allclose(y[:, c], ref, rtol=1e-12, atol=1e-14)


def test_conv_is_causal(oracle_mod):
    rng = np.random.default_rng(8)
    x = rng.standard_normal((30, 4))
    w = rng.standard_normal((4, 8))
    y1 = oracle_mod.conv(x, w)
    x2 = x.copy()
    x2[20:] += 5.0
    y2 = oracle_mod.conv(x2, w)
    np.testing.assert_array_equal(y1[:20], y2[:20])
    assert np.abs(y1[20:] - y2[20:]).min() > 0


def test_l2norm_gives_unit_rows_parallel_to_input(oracle_mod):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((20, 64)) * 3.0
    y = oracle_mod.l2norm(x, 0.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), 1.0, rtol=1e-14)
    cos = np.sum(x * y, axis=1) / np.linalg.norm(x, axis=1)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-14)
    # eps sits inside the square root: a zero row stays zero
    z = oracle_mod.l2norm(np.zeros((1, 8)), 1e-6)
    np.testing.assert_array_equal(z, 0.0)
    small = oracle_mod.l2norm(np.full((1, 4), 1e-3), 1e-6)
    np.testing.assert_allclose(small, 1e-3 / np.sqrt(4e-6 + 1e-6), rtol=1e-14)
