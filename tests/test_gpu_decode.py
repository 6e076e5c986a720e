"""GPU parity of prefill -> decode against the fp64 oracle run over the whole
token stream (prefill tokens followed by the decode tokens), plus decode
invariants: prefill(T) + decode(n) matches prefill(T + n), and saving and
restoring the state buffers resumes decoding exactly."""
import pytest
import torch

from linearized_attention_rope_gb300 import hla, synth
from gpu_cases import (assert_close, oracle_cfg, params_for, run_decode, run_prefill, strided_units, unit_job)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    from linearized_attention_rope_gb300 import build

    build.build()


def check_decode(wl, x, st, outs, units, oracle, steps, **cfg_kw):
    jobs = [unit_job(wl, x, n, h, decode_steps=steps) for n, h in units]
    refs = oracle.layer_units(oracle_cfg(wl, oracle, **cfg_kw), jobs)
    d = wl.head_dim
    for (n, h), ref in zip(units, refs):
        L = wl.seqlens[n]
        got = outs[:steps, n, h].float().cpu().numpy()
        assert_close(got, ref["o"][L:L + steps], wl.dtype, f"decode outputs seq {n} head {h}")
        S = st.view("S").view(wl.n_seqs, wl.n_q_heads, d, d)[n, h].cpu().numpy()
        assert_close(S, ref["S"], wl.dtype, f"final S seq {n} head {h}")


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 64)])
def test_decode_small_all_units(oracle_mod, dtype, d):
    # prefill lengths below, at and above the budget, then 40 steps that cross
    # the start of absorption for the short sequences
    wl = synth.small(f"decode {dtype} d{d}", [3, 20, 24, 70, 150], n_q_heads=4, n_kv_heads=2,
                     head_dim=d, dtype=dtype, n_sinks=8, window=16, decode_steps=40)
    x = synth.make_inputs(wl, "cuda")
    _, st = run_prefill(wl, x, with_state=True)
    outs = run_decode(wl, x, st)
    units = [(n, h) for n in range(wl.n_seqs) for h in range(wl.n_q_heads)]
    check_decode(wl, x, st, outs, units, oracle_mod, wl.decode_steps)
    assert st.view("pos").cpu().tolist() == [L + 40 for L in wl.seqlens]


@pytest.mark.parametrize("dtype,hq,hkv,d,n_sinks,window", [
    ("bf16", 8, 1, 128, 0, 70),   # G = 8, no sinks, two key splits
    ("bf16", 2, 2, 64, 3, 130),   # G = 1, three key splits
    ("bf16", 6, 2, 128, 8, 40),   # G = 3 (padded to four heads per group)
    ("f32", 8, 2, 64, 0, 20),     # fp32 layer, no sinks
])
def test_decode_head_groups_and_budgets(oracle_mod, dtype, hq, hkv, d, n_sinks, window):
    # group sizes and budgets beside the ones above: every head-group width of the decode softmax,
    # windows over several 64-key splits, no sinks at all (four sequences, so that every step's slice
    # of g and beta, n_seqs x Hq fp32, starts on the 16-byte boundary the C ABI asks for)
    wl = synth.small(f"decode G{hq // hkv} {n_sinks}+{window}", [5, 60, 150, 33], n_q_heads=hq,
                     n_kv_heads=hkv, head_dim=d, dtype=dtype, n_sinks=n_sinks, window=window, decode_steps=30)
    x = synth.make_inputs(wl, "cuda")
    _, st = run_prefill(wl, x, with_state=True)
    outs = run_decode(wl, x, st)
    units = [(n, h) for n in range(wl.n_seqs) for h in range(wl.n_q_heads)]
    check_decode(wl, x, st, outs, units, oracle_mod, wl.decode_steps)
    assert st.view("pos").cpu().tolist() == [L + 30 for L in wl.seqlens]


def test_decode_from_empty_state(oracle_mod):
    wl = synth.small("decode only", [0, 0], n_q_heads=2, n_kv_heads=1, head_dim=64, n_sinks=2,
                     window=5, decode_steps=30)
    x = synth.make_inputs(wl, "cuda")
    st = hla.State(params_for(wl), wl.n_seqs).init()
    outs = run_decode(wl, x, st)
    check_decode(wl, x, st, outs, [(0, 0), (0, 1), (1, 0), (1, 1)], oracle_mod, 30)


def test_c3_decode_workload_sampled(oracle_mod):
    # 64 sequences prefilled to 8192, then 512 steps with a ring of 8 + 888
    wl = synth.workloads()["c3"]
    x = synth.make_inputs(wl, "cuda")
    _, st = run_prefill(wl, x, with_state=True)
    outs = run_decode(wl, x, st)
    units = strided_units(wl.n_seqs, wl.n_q_heads, 32, offset=5)  # 32 of the 64 sequences
    check_decode(wl, x, st, outs, units, oracle_mod, wl.decode_steps)


def test_prefill_then_decode_matches_longer_prefill():
    wl = synth.small("split", [100, 137], n_q_heads=4, n_kv_heads=2, head_dim=128, n_sinks=8,
                     window=24, decode_steps=30)
    x = synth.make_inputs(wl, "cuda")
    _, st = run_prefill(wl, x, with_state=True)
    outs = run_decode(wl, x, st)
    # the same tokens as one longer prefill
    full = synth.small("joined", [130, 167], n_q_heads=4, n_kv_heads=2, head_dim=128, n_sinks=8,
                       window=24)
    y = dict(x)
    cu = x["cu_seqlens"].tolist()
    for key, dkey in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta")):
        parts = []
        for n in range(2):
            parts += [x[key][cu[n]:cu[n + 1]], x[dkey][:, n]]
        y[key] = torch.cat(parts).contiguous()
    y["cu_seqlens"] = torch.tensor([0, 130, 297], dtype=torch.int32, device="cuda")
    out_full, st_full = run_prefill(full, y, with_state=True)
    for n, (a, L) in enumerate(((0, 100), (130, 137))):
        assert_close(outs[:, n].float().cpu().numpy(), out_full[a + L:a + L + 30].float().cpu().numpy(),
                     "bf16", f"seq {n}")
    assert_close(st.view("S").cpu().numpy(), st_full.view("S").cpu().numpy(), "bf16", "state")


def test_state_save_and_restore_resumes_exactly():
    wl = synth.small("resume", [90, 40], n_q_heads=4, n_kv_heads=2, head_dim=64, n_sinks=4, window=12,
                     decode_steps=12)
    x = synth.make_inputs(wl, "cuda")
    _, st = run_prefill(wl, x, with_state=True)
    run_decode(wl, x, st, steps=4)
    saved = {k: b.cpu().clone() for k, b in st.buffers.items()}  # checkpoint to host
    a = run_decode(wl, x, st, steps=8, first=4)
    for k, b in st.buffers.items():
        b.copy_(saved[k].to(b.device))  # restore
    b2 = run_decode(wl, x, st, steps=8, first=4)
    assert torch.equal(a, b2)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_decode_gla_variant(oracle_mod, dtype, d):
    # gated linear attention (no erase term): prefill on the tensor-core path (bf16 d128) or the
    # token-serial path (fp32), then decode steps that absorb a token each
    wl = synth.small(f"decode gla {dtype} d{d}", [10, 90, 200, 64], n_q_heads=4, n_kv_heads=2, head_dim=d,
                     dtype=dtype, n_sinks=8, window=24, decode_steps=30)
    x = synth.make_inputs(wl, "cuda")
    flags = hla.FLAG_L2NORM_Q | hla.FLAG_GLA
    _, st = run_prefill(wl, x, flags=flags, with_state=True)
    outs = run_decode(wl, x, st, flags=flags)
    units = [(n, h) for n in range(wl.n_seqs) for h in range(wl.n_q_heads)]
    check_decode(wl, x, st, outs, units, oracle_mod, wl.decode_steps, erase_off=True)
