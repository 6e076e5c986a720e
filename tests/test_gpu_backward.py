"""GPU parity of the layer's backward (hla_backward) against the fp64 autograd
restatement of the layer (oracle/backward.py), unit by unit: every
(sequence, q-head) unit's gradients come from the oracle, the kv heads'
gradients (k, v and their conv filters) are the sums over the q-heads of the
group, and lambda's and the filters' over the sequences.

Tolerance: the backward computes in fp32 from the stored inputs (bf16 values
upcast), so the only error is fp32 rounding; the bound is the fp32 layer's,
relative L2 <= 1e-4 per gradient tensor, with max |diff| <= 1e-3 max |ref|.

Cases: both head dims, GQA groups of 1, 2 and 4, varlen batches with ragged
tails and sequences shorter than the budget (no absorption at all), several
checkpoint segments, the GLA update, q without L2 norm, no sinks, a
full-size LLaMA-3.1-8B-shaped layer (4096 tokens, 32/8 heads, d 128) on one
sampled kv group, the branch-off flags, zero tokens, determinism and
argument errors."""
import numpy as np
import pytest
import torch

from linearized_attention_rope_gb300 import hla, synth
from gpu_cases import params_for

pytestmark = pytest.mark.gpu

TOL = dict(rel_l2=1e-4, max_abs=1e-3)


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    from linearized_attention_rope_gb300 import build

    build.build()


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _args(x):
    return (x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"], x["wv"], x["cu_seqlens"])


def run_backward(wl, x, dout, flags=hla.FLAG_L2NORM_Q):
    prm = params_for(wl, flags)
    ws = torch.empty(hla.backward_workspace_bytes(prm, x["q"].shape[0], wl.n_seqs), dtype=torch.uint8,
                     device="cuda")
    gr = hla.backward(prm, *_args(x), dout, ws=ws)
    torch.cuda.synchronize()
    assert hla.check_workspace_error(ws) == 0
    return {n: _np(t) for n, t in gr.items()}


def oracle_grads(wl, x, dout, seqs, groups, oracle_bw, **kw):
    """Expected gradients over sequences `seqs` and kv groups `groups` (full-shaped arrays; only the
    covered rows are filled)."""
    G, d = wl.n_q_heads // wl.n_kv_heads, wl.head_dim
    cu = x["cu_seqlens"].tolist()
    T = cu[-1]
    e = dict(q=np.zeros((T, wl.n_q_heads, d)), k=np.zeros((T, wl.n_kv_heads, d)),
             v=np.zeros((T, wl.n_kv_heads, d)), g=np.zeros((T, wl.n_q_heads)), beta=np.zeros((T, wl.n_q_heads)),
             lam=np.zeros(wl.n_q_heads), wq=np.zeros((wl.n_q_heads * d, 8)), wk=np.zeros((wl.n_kv_heads * d, 8)),
             wv=np.zeros((wl.n_kv_heads * d, 8)))
    for n in seqs:
        a, b = cu[n], cu[n + 1]
        for kv in groups:
            for h in range(kv * G, kv * G + G):
                job = dict(q=_np(x["q"][a:b, h]), k=_np(x["k"][a:b, kv]), v=_np(x["v"][a:b, kv]),
                           g=_np(x["g"][a:b, h]), beta=_np(x["beta"][a:b, h]), lam=float(x["lam"][h]),
                           wq=_np(x["wq"][h * d:(h + 1) * d]), wk=_np(x["wk"][kv * d:(kv + 1) * d]),
                           wv=_np(x["wv"][kv * d:(kv + 1) * d]))
                r = oracle_bw.grads(job, _np(dout[a:b, h]), n_sinks=wl.n_sinks, window=wl.window, **kw)
                e["q"][a:b, h] = r["q"]
                e["g"][a:b, h] = r["g"]
                e["beta"][a:b, h] = r["beta"]
                e["k"][a:b, kv] += r["k"]
                e["v"][a:b, kv] += r["v"]
                e["lam"][h] += r["lam"]
                e["wq"][h * d:(h + 1) * d] += r["wq"]
                e["wk"][kv * d:(kv + 1) * d] += r["wk"]
                e["wv"][kv * d:(kv + 1) * d] += r["wv"]
    return e


def _close(got, ref, what):
    diff = got - ref
    nref = float(np.linalg.norm(ref))
    if nref == 0.0:
        assert float(np.abs(got).max(initial=0.0)) == 0.0, f"{what}: expected exact zeros"
        return
    rel = float(np.linalg.norm(diff)) / nref
    mx, rmax = float(np.abs(diff).max()), float(np.abs(ref).max())
    assert rel <= TOL["rel_l2"], f"{what}: rel_l2 {rel:.3g}"
    assert mx <= TOL["max_abs"] * rmax, f"{what}: max_abs {mx:.3g} vs max|ref| {rmax:.3g}"


def compare(wl, got, exp, seqs, groups):
    """seqs: {sequence: (first row, end row)} of the sequences the oracle ran."""
    G, d = wl.n_q_heads // wl.n_kv_heads, wl.head_dim
    heads = [h for kv in groups for h in range(kv * G, kv * G + G)]
    all_seqs = len(seqs) == wl.n_seqs
    rows = np.concatenate([np.arange(a, b) for a, b in seqs.values()])
    for name in ("q", "g", "beta"):
        _close(got[name][rows][:, heads], exp[name][rows][:, heads], f"d{name}")
    for name in ("k", "v"):
        _close(got[name][rows][:, groups], exp[name][rows][:, groups], f"d{name}")
    if all_seqs:
        _close(got["lam"][heads], exp["lam"][heads], "dlambda")
        hq = np.concatenate([np.arange(h * d, (h + 1) * d) for h in heads])
        hk = np.concatenate([np.arange(kv * d, (kv + 1) * d) for kv in groups])
        _close(got["wq"].reshape(-1, 8)[hq], exp["wq"][hq], "dconv_wq")
        _close(got["wk"].reshape(-1, 8)[hk], exp["wk"][hk], "dconv_wk")
        _close(got["wv"].reshape(-1, 8)[hk], exp["wv"][hk], "dconv_wv")


def check(wl, oracle_bw, flags=hla.FLAG_L2NORM_Q, seqs=None, groups=None, **kw):
    x = synth.make_inputs(wl, "cuda")
    dout = synth.cotangent(wl, "cuda")
    got = run_backward(wl, x, dout, flags)
    seqs = list(range(wl.n_seqs)) if seqs is None else seqs
    groups = list(range(wl.n_kv_heads)) if groups is None else groups
    exp = oracle_grads(wl, x, dout, seqs, groups, oracle_bw, **kw)
    cu = x["cu_seqlens"].tolist()
    compare(wl, got, exp, {n: (cu[n], cu[n + 1]) for n in seqs}, groups)
    return got, exp


@pytest.fixture(scope="module")
def oracle_bw():
    from oracle import backward

    return backward


def test_bf16_d64_varlen_gqa2(oracle_bw):
    # 200 tokens: 136 absorptions (three checkpoint segments); 131: ragged; 40: shorter than the budget
    wl = synth.small("bwd-a", [200, 131, 40], n_q_heads=4, n_kv_heads=2, head_dim=64, seed=synth.BASE_SEED + 300)
    check(wl, oracle_bw)


def test_bf16_d128_gqa4(oracle_bw):
    wl = synth.small("bwd-b", [300], n_q_heads=4, n_kv_heads=1, head_dim=128, seed=synth.BASE_SEED + 301)
    check(wl, oracle_bw)


def test_f32_d64_small_budget(oracle_bw):
    wl = synth.small("bwd-c", [150, 70, 5], n_q_heads=2, n_kv_heads=1, head_dim=64, dtype="f32", n_sinks=4,
                     window=16, seed=synth.BASE_SEED + 302, lam="one")
    check(wl, oracle_bw)


def test_bf16_d128_group8_short_sequences(oracle_bw):
    # 8 q-heads per kv head (8 units per 8-token block in the feature backward); sequences shorter than
    # one 8-token block and than the budget, and boundaries inside blocks
    wl = synth.small("bwd-g8", [37, 200, 5, 64, 3, 71], n_q_heads=8, n_kv_heads=1, head_dim=128,
                     seed=synth.BASE_SEED + 307)
    check(wl, oracle_bw)


def test_f32_d64_group8(oracle_bw):
    wl = synth.small("bwd-g8f", [90, 7, 130], n_q_heads=16, n_kv_heads=2, head_dim=64, dtype="f32",
                     seed=synth.BASE_SEED + 308)
    check(wl, oracle_bw)


def test_gla_variant(oracle_bw):
    wl = synth.small("bwd-gla", [180, 97], n_q_heads=4, n_kv_heads=2, head_dim=64, seed=synth.BASE_SEED + 303)
    got, _ = check(wl, oracle_bw, flags=hla.FLAG_L2NORM_Q | hla.FLAG_GLA, erase_off=True)
    assert np.all(got["beta"] == 0.0)  # beta does not enter the GLA update


def test_q_without_l2_norm_no_sinks(oracle_bw):
    wl = synth.small("bwd-nol2", [160], n_q_heads=2, n_kv_heads=2, head_dim=64, dtype="f32", n_sinks=0,
                     window=24, seed=synth.BASE_SEED + 304)
    check(wl, oracle_bw, flags=0, l2norm_q=False)


def test_llama_shaped_full_size_sampled_group(oracle_bw):
    # 4096 tokens, 32 q / 8 kv heads, d 128, bf16, 8 sinks + 56 window; the oracle on kv group 3 (4 q-heads)
    wl = synth.workloads()["c1"]
    check(wl, oracle_bw, groups=[3])


def test_branch_off_flags(oracle_bw):
    """SOFTMAX_OFF: the linear branch alone; LINEAR_OFF: the softmax branch alone.  Their sum is the
    full layer's backward (the layer is the sum of its branches), and LINEAR_OFF's equals the full
    backward with lambda = 0 except for lambda's own gradient, which is zero."""
    wl = synth.small("bwd-flags", [150, 90], n_q_heads=4, n_kv_heads=2, head_dim=64, dtype="f32",
                     seed=synth.BASE_SEED + 305)
    x = synth.make_inputs(wl, "cuda")
    dout = synth.cotangent(wl, "cuda")
    full = run_backward(wl, x, dout)
    sm = run_backward(wl, x, dout, hla.FLAG_L2NORM_Q | hla.FLAG_LINEAR_OFF)
    lin = run_backward(wl, x, dout, hla.FLAG_L2NORM_Q | hla.FLAG_SOFTMAX_OFF)
    for n in hla.BACKWARD_GRADS:
        np.testing.assert_allclose(sm[n] + lin[n], full[n], rtol=1e-5, atol=1e-5 * np.abs(full[n]).max())
    assert np.all(sm["lam"] == 0.0)
    assert np.all(sm["g"] == 0.0) and np.all(sm["beta"] == 0.0)
    x0 = dict(x, lam=torch.zeros_like(x["lam"]))
    zero_lam = run_backward(wl, x0, dout)
    for n in hla.BACKWARD_GRADS:
        if n != "lam":
            np.testing.assert_array_equal(sm[n], zero_lam[n])


def test_deterministic():
    wl = synth.small("bwd-det", [260, 77], n_q_heads=4, n_kv_heads=2, head_dim=128, seed=synth.BASE_SEED + 306)
    x = synth.make_inputs(wl, "cuda")
    dout = synth.cotangent(wl, "cuda")
    a, b = run_backward(wl, x, dout), run_backward(wl, x, dout)
    for n in hla.BACKWARD_GRADS:
        np.testing.assert_array_equal(a[n], b[n])


def test_zero_tokens_and_errors():
    wl = synth.small("bwd-zero", [0, 0], n_q_heads=4, n_kv_heads=2, head_dim=64)
    prm = params_for(wl)
    x = synth.make_inputs(wl, "cuda")
    gr = {n: torch.full(t.shape, 7.0, device="cuda") for n, t in
          zip(hla.BACKWARD_GRADS, (x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"], x["wv"]))}
    hla.backward(prm, *_args(x), synth.cotangent(wl, "cuda"), grads=gr)  # per-token tensors: empty (NULL)
    torch.cuda.synchronize()
    for n in ("lam", "wq", "wk", "wv"):
        assert torch.all(gr[n] == 0)
    # the test-stall hook has no meaning here, and a short workspace is refused before any launch
    wl = synth.small("bwd-err", [40], n_q_heads=2, n_kv_heads=1, head_dim=64)
    x = synth.make_inputs(wl, "cuda")
    dout = synth.cotangent(wl, "cuda")
    with pytest.raises(hla.HlaError) as e:
        hla.backward(params_for(wl, hla.FLAG_L2NORM_Q | hla.FLAG_TEST_STALL), *_args(x), dout)
    assert e.value.status == hla.HLA_ERR_INVALID_ARG
    small_ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(hla.HlaError) as e:
        hla.backward(params_for(wl), *_args(x), dout, ws=small_ws)
    assert e.value.status == hla.HLA_ERR_WORKSPACE


def test_malformed_seqlens_are_flagged_not_faulting():
    # the table ends at 40 although 64 tokens are passed: tokens 40..63 belong to no sequence; every access
    # stays clamped inside [0, total) and the workspace's error word reports the table
    wl = synth.small("bwd bad cu", [40, 24], n_q_heads=2, n_kv_heads=1, head_dim=64)
    x = synth.make_inputs(wl, "cuda")
    x["cu_seqlens"] = torch.tensor([0, 20, 40], dtype=torch.int32, device="cuda")
    prm = params_for(wl)
    ws = torch.empty(hla.backward_workspace_bytes(prm, 64, 2), dtype=torch.uint8, device="cuda")
    hla.backward(prm, *_args(x), synth.cotangent(wl, "cuda"), ws=ws)
    torch.cuda.synchronize()
    assert hla.check_workspace_error(ws) != 0
