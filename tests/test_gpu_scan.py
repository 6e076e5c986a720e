"""GPU parity of the context-parallel token-serial GDN (HLA_FLAG_GDN_SCAN): the
absorptions of every sequence are cut into parts, each part's state map
S -> P S + R is formed at once, a scan over the parts gives their start
states, and all parts run at once.  The layer's outputs and final states must
be the oracle's (fp32 layer: rel-L2 <= 1e-4; bf16: rel-L2 <= 5e-3, max-abs <=
1e-2 max|ref|).  Cases: fp32 and bf16 (token-serial path by flag), head dims
64 and 128, GQA, varlen batches with sequences that have no absorption or a
single part, the GLA update, a long single sequence cut into many parts, and
the launch count."""
import numpy as np
import pytest
import torch

from linearized_attention_rope_gb300 import hla, synth
from gpu_cases import run_prefill
from test_gpu_prefill import all_units, check_prefill

pytestmark = pytest.mark.gpu

SCAN = hla.FLAG_L2NORM_Q | hla.FLAG_GDN_SCAN


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    from linearized_attention_rope_gb300 import build

    build.build()


@pytest.mark.parametrize("dtype,d,flags", [("f32", 64, SCAN), ("f32", 128, SCAN),
                                           ("bf16", 128, SCAN | hla.FLAG_GDN_RECURRENT),
                                           ("bf16", 64, SCAN)])
def test_scan_varlen_all_units(oracle_mod, dtype, d, flags):
    # 1 and 70 tokens: no absorption (8 sinks + 56 window); 130: one part; 700 and 1500: several parts
    wl = synth.small(f"scan {dtype} d{d}", [1, 700, 70, 1500, 130], n_q_heads=4, n_kv_heads=2, head_dim=d,
                     dtype=dtype, seed=synth.BASE_SEED + 400 + d)
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, flags=flags, with_state=True)
    check_prefill(wl, x, out, st, all_units(wl), oracle_mod)


def test_scan_gla(oracle_mod):
    wl = synth.small("scan gla", [900, 333], n_q_heads=2, n_kv_heads=1, head_dim=64, dtype="f32",
                     seed=synth.BASE_SEED + 410)
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, flags=SCAN | hla.FLAG_GLA, with_state=True)
    check_prefill(wl, x, out, st, all_units(wl), oracle_mod, erase_off=True)


def test_scan_long_sequence_many_parts(oracle_mod):
    # one 8192-token sequence, 2 q-heads: parts of 64 absorptions, 127 of them chained by the scan
    wl = synth.small("scan long", [8192], n_q_heads=2, n_kv_heads=1, head_dim=64, dtype="f32",
                     seed=synth.BASE_SEED + 411, lam="one")
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, flags=SCAN, with_state=True)
    check_prefill(wl, x, out, st, all_units(wl), oracle_mod)


def test_scan_matches_the_single_pass():
    wl = synth.small("scan vs whole", [2000, 517], n_q_heads=4, n_kv_heads=1, head_dim=128, dtype="f32",
                     seed=synth.BASE_SEED + 412)
    x = synth.make_inputs(wl, "cuda")
    a, sa = run_prefill(wl, x, with_state=True)
    b, sb = run_prefill(wl, x, flags=SCAN, with_state=True)
    for u, v in ((a, b), (sa.view("S"), sb.view("S"))):
        u, v = u.double().cpu().numpy(), v.double().cpu().numpy()
        assert np.linalg.norm(u - v) <= 1e-5 * np.linalg.norm(u)


def test_scan_launch_count():
    p = hla.Params(2, 1, 64, 8, 56, dtype=hla.DTYPE_F32)
    assert hla.prefill_launch_count(p) == 4
    p.flags |= hla.FLAG_GDN_SCAN
    assert hla.prefill_launch_count(p) == 6
    assert hla.prefill_launch_count(p, with_state=True) == 7
    # no effect on the tensor-core path
    q = hla.Params(32, 8, 128, 8, 56, flags=hla.FLAG_L2NORM_Q | hla.FLAG_GDN_SCAN)
    assert hla.prefill_launch_count(q) == hla.prefill_launch_count(hla.Params(32, 8, 128, 8, 56))
