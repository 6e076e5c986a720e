"""GPU parity of the prefill path (C ABI -> CUDA kernels) against the fp64
oracle, on the same seeded inputs: small cases with every unit checked and
ragged tails, the fp32 reference workload in full, and the LLaMA/Qwen-shaped
workloads at full size on sampled (sequence, q-head) units."""
import numpy as np
import pytest
import torch

from linearized_attention_rope_gb300 import hla, synth
from gpu_cases import assert_close, oracle_cfg, run_prefill, strided_units, unit_job, unit_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    from linearized_attention_rope_gb300 import build

    build.build()


def check_prefill(wl, x, out, st, units, oracle, flags=hla.FLAG_L2NORM_Q, **cfg_kw):
    jobs = [unit_job(wl, x, n, h) for n, h in units]
    if flags & hla.FLAG_LINEAR_OFF:
        for j in jobs:
            j["lam"] = 0.0
    cfg = oracle_cfg(wl, oracle, softmax_off=bool(flags & hla.FLAG_SOFTMAX_OFF), **cfg_kw)
    refs = oracle.layer_units(cfg, jobs)
    worst = 0.0
    d = wl.head_dim
    for (n, h), ref in zip(units, refs):
        a, b = unit_rows(x, n)
        m = assert_close(out[a:b, h].float().cpu().numpy(), ref["o"], wl.dtype, f"o seq {n} head {h}")
        worst = max(worst, m["rel_l2"])
        if st is not None:
            S = st.view("S").view(wl.n_seqs, wl.n_q_heads, d, d)[n, h].cpu().numpy()
            assert_close(S, ref["S"], wl.dtype, f"S seq {n} head {h}")
    return worst


def all_units(wl):
    return [(n, h) for n in range(wl.n_seqs) for h in range(wl.n_q_heads)]


RAGGED = [1, 5, 8, 63, 64, 65, 120, 200, 333]


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 64), ("f32", 128)])
def test_small_ragged_all_units(oracle_mod, dtype, d):
    wl = synth.small(f"ragged {dtype} d{d}", RAGGED, n_q_heads=4, n_kv_heads=2, head_dim=d, dtype=dtype)
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, with_state=True)
    check_prefill(wl, x, out, st, all_units(wl), oracle_mod)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n_sinks,window", [(0, 1), (0, 40), (8, 1), (3, 7), (8, 120), (16, 400)])
def test_budget_variants(oracle_mod, n_sinks, window, d):
    # windows over 128 keys make the tensor-core softmax merge several key groups
    wl = synth.small(f"budget {n_sinks}+{window}", [300, 77, 530], n_q_heads=4, n_kv_heads=1, head_dim=d,
                     n_sinks=n_sinks, window=window)
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, with_state=True)
    check_prefill(wl, x, out, st, all_units(wl), oracle_mod)


@pytest.mark.parametrize("flags", [hla.FLAG_L2NORM_Q | hla.FLAG_LINEAR_OFF,
                                   hla.FLAG_L2NORM_Q | hla.FLAG_SOFTMAX_OFF])
def test_each_branch_alone(oracle_mod, flags):
    # a broken branch cannot hide under the other one
    wl = synth.small("branches", [260, 130], n_q_heads=4, n_kv_heads=2, head_dim=128)
    x = synth.make_inputs(wl, "cuda")
    out, _ = run_prefill(wl, x, flags=flags)
    check_prefill(wl, x, out, None, all_units(wl), oracle_mod, flags=flags)


def test_without_q_normalisation(oracle_mod):
    wl = synth.small("no q norm", [200], n_q_heads=2, n_kv_heads=1, head_dim=64)
    x = synth.make_inputs(wl, "cuda")
    out, _ = run_prefill(wl, x, flags=0)
    check_prefill(wl, x, out, None, all_units(wl), oracle_mod, l2norm_q=False)


@pytest.mark.parametrize("dtype,d,seqlens", [("f32", 64, [512, 77]), ("bf16", 128, [700, 64, 333]),
                                             ("bf16", 64, [300, 65])])
def test_gla_variant(oracle_mod, dtype, d, seqlens):
    # gated linear attention in place of the delta rule (no erase term, write gain 1), on the
    # token-serial path (fp32 layer, bf16 d64) and on the tensor-core path (bf16 d128)
    wl = synth.small(f"gla {dtype} d{d}", seqlens, n_q_heads=4, n_kv_heads=2, head_dim=d, dtype=dtype)
    x = synth.make_inputs(wl, "cuda")
    flags = hla.FLAG_L2NORM_Q | hla.FLAG_GLA
    out, st = run_prefill(wl, x, flags=flags, with_state=True)
    check_prefill(wl, x, out, st, all_units(wl), oracle_mod, flags=flags, erase_off=True)


def test_recurrent_kernel_selected_by_flag(oracle_mod):
    wl = synth.small("recurrent flag", [333, 64], n_q_heads=4, n_kv_heads=1, head_dim=128)
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, flags=hla.FLAG_L2NORM_Q | hla.FLAG_GDN_RECURRENT, with_state=True)
    check_prefill(wl, x, out, st, all_units(wl), oracle_mod)


def test_c0_reference_workload_fp32(oracle_mod):
    wl = synth.workloads()["c0"]
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, with_state=True)
    worst = check_prefill(wl, x, out, st, all_units(wl), oracle_mod)
    assert worst <= 1e-4


def test_c1_llama8b_prefill_all_units(oracle_mod):
    wl = synth.workloads()["c1"]
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, with_state=True)
    check_prefill(wl, x, out, st, all_units(wl), oracle_mod)


def test_c4_qwen32b_varlen_sampled(oracle_mod):
    wl = synth.workloads()["c4"]
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, with_state=True)
    units = strided_units(wl.n_seqs, wl.n_q_heads, 64)  # 8 of the 64 heads of every sequence
    check_prefill(wl, x, out, st, units, oracle_mod)


@pytest.mark.slow
def test_c2_llama8b_long_prefill_sampled(oracle_mod):
    wl = synth.workloads()["c2"]
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, with_state=True)
    units = strided_units(wl.n_seqs, wl.n_q_heads, 32, offset=3)  # 4 of the 32 heads of every sequence
    check_prefill(wl, x, out, st, units, oracle_mod)


def test_varlen_packing_matches_separate_runs():
    wl = synth.small("packed", [70, 1, 190, 64], n_q_heads=4, n_kv_heads=2, head_dim=128)
    x = synth.make_inputs(wl, "cuda")
    out, _ = run_prefill(wl, x)
    cu = x["cu_seqlens"].tolist()
    for n in range(wl.n_seqs):
        a, b = cu[n], cu[n + 1]
        sub = dict(x)
        for key in ("q", "k", "v", "g", "beta"):
            sub[key] = x[key][a:b].contiguous()
        sub["cu_seqlens"] = torch.tensor([0, b - a], dtype=torch.int32, device="cuda")
        wl1 = synth.small("one", [b - a], n_q_heads=4, n_kv_heads=2, head_dim=128)
        o1, _ = run_prefill(wl1, sub)
        # same arithmetic per row; only the tensor-core summation order over key
        # slots differs (blocks follow the global token index), so compare to rounding
        assert_close(o1.float().cpu().numpy(), out[a:b].float().cpu().numpy(), "bf16", f"sequence {n}")
        assert (o1.float() - out[a:b].float()).abs().max().item() <= 2e-2


def test_gqa_equals_mha_with_repeated_kv():
    wl = synth.small("gqa", [150, 90], n_q_heads=4, n_kv_heads=2, head_dim=64)
    x = synth.make_inputs(wl, "cuda")
    out, _ = run_prefill(wl, x)
    mha = dict(x)
    mha["k"] = x["k"].repeat_interleave(2, dim=1).contiguous()
    mha["v"] = x["v"].repeat_interleave(2, dim=1).contiguous()
    mha["wk"] = x["wk"].view(2, 64, 8).repeat_interleave(2, dim=0).reshape(256, 8).contiguous()
    mha["wv"] = x["wv"].view(2, 64, 8).repeat_interleave(2, dim=0).reshape(256, 8).contiguous()
    wl2 = synth.small("mha", [150, 90], n_q_heads=4, n_kv_heads=4, head_dim=64)
    out2, _ = run_prefill(wl2, mha)
    assert torch.equal(out, out2)


def test_empty_sequences_and_zero_tokens(oracle_mod):
    wl = synth.small("empties", [0, 40, 0, 100, 0], n_q_heads=2, n_kv_heads=1, head_dim=64)
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, with_state=True)
    check_prefill(wl, x, out, st, [(1, 0), (3, 1)], oracle_mod)
    pos = st.view("pos").cpu().tolist()
    assert pos == [0, 40, 0, 100, 0]
    # no tokens at all
    prm = hla.Params(2, 1, 64, 8, 56)
    z = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    hla.prefill(prm, z, z[:, :1], z[:, :1], torch.empty((0, 2), device="cuda"),
                torch.empty((0, 2), device="cuda"), x["lam"], x["wq"], x["wk"], x["wv"], cu, z)
    torch.cuda.synchronize()


def test_malformed_seqlens_are_flagged_not_faulting():
    wl = synth.small("bad cu", [40, 24], n_q_heads=2, n_kv_heads=1, head_dim=64)
    x = synth.make_inputs(wl, "cuda")
    # the table ends at 40 although 64 tokens are passed: tokens 40..63 belong to
    # no sequence; every access stays clamped inside [0, total)
    x["cu_seqlens"] = torch.tensor([0, 20, 40], dtype=torch.int32, device="cuda")
    prm = hla.Params(2, 1, 64, 8, 56)
    out = torch.zeros_like(x["q"])
    ws = hla.prefill(prm, x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"],
                     x["wv"], x["cu_seqlens"], out)
    torch.cuda.synchronize()
    assert hla.check_workspace_error(ws) != 0


@pytest.mark.parametrize("d", [64, 128])
def test_large_magnitude_activations(oracle_mod, d):
    # q and k at 4x the unit scale (attention logits 16x larger) and v at 300x: the bf16 layer keeps its
    # RoPE'd q and k, the conv outputs, the softmax rows, U and the state images in fp16, whose range
    # (65,504) holds these values and whose rounding (2^-11) perturbs a logit by about
    # 2^-11 sqrt(2) |q| |k| / d (see the design notes for the bound)
    wl = synth.small(f"large d{d}", [333, 140], n_q_heads=4, n_kv_heads=2, head_dim=d)
    x = synth.make_inputs(wl, "cuda")
    x["q"] = (x["q"].float() * 4.0).to(torch.bfloat16)
    x["k"] = (x["k"].float() * 4.0).to(torch.bfloat16)
    x["v"] = (x["v"].float() * 300.0).to(torch.bfloat16)
    out, st = run_prefill(wl, x, with_state=True)
    check_prefill(wl, x, out, st, all_units(wl), oracle_mod)


def test_many_sequences_keep_index_order(oracle_mod):
    # 70 sequences of mixed lengths: more than the state kernel ranks by length, so its grid rows take the
    # sequences in index order (the ranked order is covered by every other varlen case)
    lens = [65, 130, 7, 200, 64, 129, 1]
    wl = synth.small("many seqs", [lens[i % len(lens)] for i in range(70)], n_q_heads=2, n_kv_heads=1,
                     head_dim=128, seed=synth.BASE_SEED + 431)
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, with_state=True)
    check_prefill(wl, x, out, st, all_units(wl), oracle_mod)


@pytest.mark.parametrize("gate_scale", [2.0, 30.0])
def test_strong_and_mixed_gates(oracle_mod, gate_scale):
    # gates 20x and 300x the unit recipe (log-gate per token about -1.6 and -24 on average): a 64-token
    # chunk then spans far more than 100 powers of two, where the chunk-local kernel forms e^(G_r - G_i)
    # entry by entry instead of as a product of row and column factors; the second sequence keeps the
    # unit gates, so one launch holds chunks of both kinds
    wl = synth.small(f"gates x{gate_scale}", [700, 300], n_q_heads=4, n_kv_heads=2, head_dim=128,
                     seed=synth.BASE_SEED + 430)
    x = synth.make_inputs(wl, "cuda")
    cu = x["cu_seqlens"].tolist()
    x["g"][cu[0]:cu[1]] *= 10.0 * gate_scale
    out, st = run_prefill(wl, x, with_state=True)
    check_prefill(wl, x, out, st, all_units(wl), oracle_mod)
