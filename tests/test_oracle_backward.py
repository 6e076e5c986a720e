"""Pins for the fp64 autograd restatement of the layer (oracle/backward.py):
its forward equals the C oracle's on the same inputs (two independent
restatements of the pages' steps), its gradients equal central finite
differences of the C oracle's forward along random directions, the lambda
gradient is the closed form sum(dO . o_lin), and tokens that never enter the
state get zero gate gradients."""
import numpy as np
import pytest

from oracle import backward as bw

CFGS = [
    dict(L=70, d=8, n_sinks=3, window=10, l2norm_q=True, erase_off=False),
    dict(L=45, d=16, n_sinks=0, window=5, l2norm_q=False, erase_off=False),
    dict(L=60, d=8, n_sinks=8, window=7, l2norm_q=True, erase_off=True),
]


def _job(rng, L, d):
    mu = rng.standard_normal(d)
    mu /= np.linalg.norm(mu)
    return dict(q=rng.standard_normal((L, d)), k=mu + 0.3 * rng.standard_normal((L, d)),
                v=rng.standard_normal((L, d)), g=-0.1 * np.log1p(np.exp(rng.standard_normal(L))),
                beta=1.0 / (1.0 + np.exp(-rng.standard_normal(L))), lam=0.5 + rng.random(),
                wq=rng.standard_normal((d, 8)) / np.sqrt(8), wk=rng.standard_normal((d, 8)) / np.sqrt(8),
                wv=rng.standard_normal((d, 8)) / np.sqrt(8))


def _c_forward(oracle_mod, cfg, job, want=()):
    c = oracle_mod.OracleCfg(d=cfg["d"], n_sinks=cfg["n_sinks"], window=cfg["window"], l2norm_q=cfg["l2norm_q"],
                             erase_off=cfg["erase_off"])
    return oracle_mod.layer_unit(c, job["q"], job["k"], job["v"], job["g"], job["beta"], job["lam"], job["wq"],
                                 job["wk"], job["wv"], want=want)


@pytest.mark.parametrize("cfg", CFGS)
def test_forward_matches_the_c_oracle(oracle_mod, cfg):
    rng = np.random.default_rng(11)
    job = _job(rng, cfg["L"], cfg["d"])
    dout = rng.standard_normal((cfg["L"], cfg["d"]))
    got = bw.grads(job, dout, n_sinks=cfg["n_sinks"], window=cfg["window"], l2norm_q=cfg["l2norm_q"],
                   erase_off=cfg["erase_off"])["o"]
    np.testing.assert_allclose(got, _c_forward(oracle_mod, cfg, job)["o"], rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("cfg", CFGS)
def test_gradients_match_finite_differences_of_the_c_oracle(oracle_mod, cfg):
    rng = np.random.default_rng(12)
    job = _job(rng, cfg["L"], cfg["d"])
    dout = rng.standard_normal((cfg["L"], cfg["d"]))
    gr = bw.grads(job, dout, n_sinks=cfg["n_sinks"], window=cfg["window"], l2norm_q=cfg["l2norm_q"],
                  erase_off=cfg["erase_off"])
    loss = lambda j: float(np.sum(dout * _c_forward(oracle_mod, cfg, j)["o"]))  # noqa: E731
    eps = 1e-6
    for trial in range(3):
        # one random direction over every input at once, and one per input
        names = list(bw.NAMES) if trial == 0 else [bw.NAMES[(trial * 4 + i) % len(bw.NAMES)] for i in range(3)]
        delta = {n: rng.standard_normal(np.shape(job[n])) for n in names}
        plus = {n: (job[n] + eps * delta[n] if n in delta else job[n]) for n in job}
        minus = {n: (job[n] - eps * delta[n] if n in delta else job[n]) for n in job}
        fd = (loss(plus) - loss(minus)) / (2 * eps)
        an = sum(float(np.sum(gr[n] * delta[n])) for n in names)
        assert fd == pytest.approx(an, rel=2e-6, abs=1e-7), (trial, names)


def test_lambda_gradient_is_the_linear_branch_projection(oracle_mod):
    cfg = CFGS[0]
    rng = np.random.default_rng(13)
    job = _job(rng, cfg["L"], cfg["d"])
    dout = rng.standard_normal((cfg["L"], cfg["d"]))
    gr = bw.grads(job, dout, n_sinks=cfg["n_sinks"], window=cfg["window"])
    o_lin = _c_forward(oracle_mod, cfg, job, want=("o_lin",))["o_lin"]
    assert float(gr["lam"]) == pytest.approx(float(np.sum(dout * o_lin)), rel=1e-12, abs=1e-14)


def test_tokens_that_never_enter_the_state_have_zero_gate_gradients():
    # budget n_sinks + W >= L: nothing is absorbed, so g and beta do not reach the output
    rng = np.random.default_rng(14)
    job = _job(rng, 30, 8)
    gr = bw.grads(job, rng.standard_normal((30, 8)), n_sinks=8, window=22)
    assert np.all(gr["g"] == 0.0) and np.all(gr["beta"] == 0.0)
    # with a smaller window only tokens n_sinks .. L - 1 - W are absorbed; the first of them meets an
    # empty state, so its gate multiplies zero and gets no gradient either
    gr = bw.grads(job, rng.standard_normal((30, 8)), n_sinks=8, window=10)
    gated = np.zeros(30, dtype=bool)
    gated[9:30 - 10] = True
    assert np.all(gr["g"][~gated] == 0.0) and np.all(gr["g"][gated] != 0.0)
    assert np.all(gr["beta"][8:20] != 0.0) and np.all(gr["beta"][:8] == 0.0) and np.all(gr["beta"][20:] == 0.0)
