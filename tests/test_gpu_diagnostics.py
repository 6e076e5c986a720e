"""GPU parity of the component-usage diagnostics (hla_prefill_diagnostics)
against the oracle: per (sequence, q-head) the summed squares of the two
branch outputs, from the oracle's o_sm and o_lin intermediates, and per
position and kv head the key concentration and projection residual, from the
oracle's key statistics over its own RoPE'd keys."""
import numpy as np
import pytest
import torch

from linearized_attention_rope_gb300 import hla, synth
from gpu_cases import oracle_cfg, params_for, unit_job, unit_rows

pytestmark = pytest.mark.gpu

# bf16 layers: branch outputs rounded to bf16 before squaring (relative 2^-8 per element at most) and
# fp16 RoPE'd keys; fp32 layer: fp32 throughout
TOL = {"bf16": dict(sq_rel=1e-2, stat_abs=3e-3), "f32": dict(sq_rel=1e-4, stat_abs=1e-5)}


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    from linearized_attention_rope_gb300 import build

    build.build()


@pytest.mark.parametrize("dtype,d,seqlens,hq,hkv,sigma", [
    ("bf16", 128, [333, 70, 1, 200], 4, 2, 0.3),    # tensor-core path, varlen with a one-token sequence
    ("bf16", 128, [260], 8, 2, 1.5),                # dispersed keys
    ("f32", 64, [512, 90], 2, 1, 0.3),              # token-serial fp32 path
])
def test_diagnostics_match_the_oracle(oracle_mod, dtype, d, seqlens, hq, hkv, sigma):
    wl = synth.small(f"diag {dtype} d{d}", seqlens, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, dtype=dtype,
                     sigma=sigma)
    x = synth.make_inputs(wl, "cuda")
    prm = params_for(wl)
    sq, stats = hla.prefill_diagnostics(prm, x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"],
                                        x["wv"], x["cu_seqlens"])
    torch.cuda.synchronize()
    sq, stats = sq.cpu().numpy(), stats.cpu().numpy()
    units = [(n, h) for n in range(wl.n_seqs) for h in range(wl.n_q_heads)]
    refs = oracle_mod.layer_units(oracle_cfg(wl, oracle_mod), [unit_job(wl, x, n, h) for n, h in units],
                                  want=("o_sm", "o_lin", "kr"))
    tol = TOL[dtype]
    G = hq // hkv
    for (n, h), ref in zip(units, refs):
        lam = float(x["lam"][h])
        want = np.array([np.sum(ref["o_sm"] ** 2), np.sum((lam * ref["o_lin"]) ** 2)])
        got = sq[n, h].astype(np.float64)
        np.testing.assert_allclose(got, want, rtol=tol["sq_rel"], atol=1e-6, err_msg=f"branch sums seq {n} head {h}")
        if h % G == 0:  # the key statistics belong to the kv head
            conc, res = oracle_mod.key_stats(ref["kr"])
            a, b = unit_rows(x, n)
            np.testing.assert_allclose(stats[a:b, h // G, 0], conc, rtol=0, atol=tol["stat_abs"],
                                       err_msg=f"concentration seq {n} kv {h // G}")
            np.testing.assert_allclose(stats[a:b, h // G, 1], res, rtol=0, atol=tol["stat_abs"],
                                       err_msg=f"residual seq {n} kv {h // G}")


def test_concentrated_keys_have_small_residuals_dispersed_keys_large():
    # the regime the analysis describes: a key noise scale of 0.1 around one direction against 3.0
    out = {}
    for sigma in (0.1, 3.0):
        wl = synth.small(f"conc {sigma}", [400], n_q_heads=2, n_kv_heads=1, head_dim=128, sigma=sigma)
        x = synth.make_inputs(wl, "cuda")
        _, stats = hla.prefill_diagnostics(params_for(wl), x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"],
                                           x["wq"], x["wk"], x["wv"], x["cu_seqlens"])
        out[sigma] = stats.cpu().numpy()[:, 0, :]
    assert out[0.1][:, 1].mean() < out[3.0][:, 1].mean()
    assert out[0.1][:, 0].mean() > out[3.0][:, 0].mean()
