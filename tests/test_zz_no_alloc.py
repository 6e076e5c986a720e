"""hla_prefill_noalloc, the prefill for callers that cannot allocate device
memory (a plugin whose host framework owns all device memory and hands it no
allocator, or a latency-critical caller that cannot pay for cudaMalloc's
implicit synchronisation).  It must give the results of hla_prefill, which
uses a caller-allocated workspace, on consecutive calls that share the
library's one static scratch buffer, and refuse prefills that need more
scratch than that buffer holds.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process
(the first call on the device sets the buffer up)."""
import ctypes

import pytest
import torch

from linearized_attention_rope_gb300 import hla, synth
from gpu_cases import assert_close, params_for

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 64 << 20


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    from linearized_attention_rope_gb300 import build

    build.build()


CASES = {
    "fp32 reference shape": dict(seqlens=[512], n_q_heads=2, n_kv_heads=1, head_dim=64, dtype="f32"),
    "bf16 LLaMA-8B heads, varlen": dict(seqlens=[700, 61, 263], n_q_heads=32, n_kv_heads=8,
                                        head_dim=128, dtype="bf16"),
}


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_workspace_prefill_on_consecutive_calls(case):
    spec = CASES[case]
    for call in range(2):  # two calls in a row through the shared static scratch
        wl = synth.small(f"{case} call {call}", seed=synth.BASE_SEED + 500 + call, **spec)
        prm = params_for(wl)
        assert hla.workspace_bytes(prm, wl.total_tokens, wl.n_seqs) <= STATIC_SCRATCH_BYTES
        x = synth.make_inputs(wl, "cuda")
        args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"], x["wv"],
                x["cu_seqlens"])
        ref = torch.empty_like(x["q"])
        st_ref = hla.State(prm, wl.n_seqs).init()
        hla.prefill(prm, *args, ref, state=st_ref)
        got = torch.full_like(x["q"], float("nan"))
        st = hla.State(prm, wl.n_seqs).init()
        hla.prefill_noalloc(prm, *args, got, state=st)
        torch.cuda.synchronize()
        assert_close(got.float().cpu().numpy(), ref.float().cpu().numpy(), wl.dtype, f"{case} call {call}")
        assert_close(st.view("S").cpu().numpy(), st_ref.view("S").cpu().numpy(), wl.dtype,
                     f"{case} call {call} state")


def test_noalloc_refuses_prefills_beyond_the_static_scratch():
    prm = hla.Params(32, 8, 128, 8, 56)
    total = 4096
    assert hla.workspace_bytes(prm, total, 1) > STATIC_SCRATCH_BYTES
    # The size check comes before any other work: with the per-token pointers
    # left NULL the call can only ever return a status, never launch.
    lam = torch.ones(32, device="cuda")
    w = torch.zeros(4096, 8, device="cuda")
    cu = torch.tensor([0, total], dtype=torch.int32, device="cuda")
    rc = hla.load().hla_prefill_noalloc(ctypes.byref(prm.c()), None, None, None, None, None,
                                        ctypes.c_void_p(lam.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                        ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                        ctypes.c_void_p(cu.data_ptr()), 1, total, None, None, None)
    assert rc == hla.HLA_ERR_WORKSPACE


def test_noalloc_error_word_is_readable_and_cleared():
    # A cu_seqlens table that ends short of the tokens passed is clamped on the device and flagged
    # in the error word at the head of the library's buffer; the accessor reads it back (allocating
    # nothing) and clears it, and a correct call afterwards leaves it clear.
    wl = synth.small("bad cu noalloc", [40, 24], n_q_heads=2, n_kv_heads=1, head_dim=64)
    x = synth.make_inputs(wl, "cuda")
    prm = params_for(wl)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"], x["wv"])
    out = torch.zeros_like(x["q"])
    bad = torch.tensor([0, 20, 40], dtype=torch.int32, device="cuda")
    hla.prefill_noalloc(prm, *args, bad, out)
    assert hla.prefill_noalloc_check_error() != 0
    assert hla.prefill_noalloc_check_error() == 0
    hla.prefill_noalloc(prm, *args, x["cu_seqlens"], out)
    assert hla.prefill_noalloc_check_error() == 0
