"""GPU checks of the failure paths of the C ABI, none of which faults, traps
or hangs the device: a bounded wait that runs out (the stall test hook, whose
state kernel issues no copy and no MMA, so its waits end after about a
millisecond) is reported as HLA_ERR_TIMEOUT and the next prefill is correct;
a decode state that is not fresh is flagged by the prefill; a negative decode
position is flagged and left alone."""
import pytest
import torch

from linearized_attention_rope_gb300 import hla, synth
from gpu_cases import assert_close, oracle_cfg, params_for, run_prefill, unit_job, unit_rows

pytestmark = pytest.mark.gpu

ERR_STATE, ERR_TIMEOUT = 3, 2  # device error word codes


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    from linearized_attention_rope_gb300 import build

    build.build()


def _args(x):
    return (x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"], x["wv"], x["cu_seqlens"])


def test_bounded_wait_runs_out_then_next_prefill_is_correct(oracle_mod):
    wl = synth.small("stall", [300, 140], n_q_heads=4, n_kv_heads=2, head_dim=128)
    x = synth.make_inputs(wl, "cuda")
    prm = params_for(wl, hla.FLAG_L2NORM_Q | hla.FLAG_TEST_STALL)
    out = torch.zeros_like(x["q"])
    ws = hla.prefill(prm, *_args(x), out)
    assert hla.check_workspace_error(ws) == ERR_TIMEOUT  # synchronises, reads, clears
    assert hla.check_workspace_error(ws) == 0
    # the context is still usable: the same workspace serves a normal prefill that matches the oracle
    prm = params_for(wl)
    out2 = torch.empty_like(x["q"])
    hla.prefill(prm, *_args(x), out2, ws=ws)
    torch.cuda.synchronize()
    assert hla.check_workspace_error(ws) == 0
    jobs = [unit_job(wl, x, n, h) for n in range(wl.n_seqs) for h in range(wl.n_q_heads)]
    refs = oracle_mod.layer_units(oracle_cfg(wl, oracle_mod), jobs)
    i = 0
    for n in range(wl.n_seqs):
        a, b = unit_rows(x, n)
        for h in range(wl.n_q_heads):
            assert_close(out2[a:b, h].float().cpu().numpy(), refs[i]["o"], wl.dtype, f"seq {n} head {h}")
            i += 1


def test_status_of_a_timed_out_call_through_the_c_abi():
    import ctypes

    wl = synth.small("stall status", [200], n_q_heads=2, n_kv_heads=1, head_dim=128)
    x = synth.make_inputs(wl, "cuda")
    prm = params_for(wl, hla.FLAG_L2NORM_Q | hla.FLAG_TEST_STALL)
    out = torch.zeros_like(x["q"])
    ws = hla.prefill(prm, *_args(x), out)
    code = ctypes.c_int32(-1)
    rc = hla.load().hla_check_workspace_error(ctypes.c_void_p(ws.data_ptr()),
                                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                              ctypes.byref(code))
    assert rc == hla.HLA_ERR_TIMEOUT and code.value == ERR_TIMEOUT


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f32")])
def test_prefill_flags_a_state_that_is_not_fresh(d, dtype):
    wl = synth.small("not fresh", [90, 30], n_q_heads=2, n_kv_heads=1, head_dim=d, dtype=dtype)
    x = synth.make_inputs(wl, "cuda")
    out, st = run_prefill(wl, x, with_state=True)  # fills the state: positions 90 and 30
    assert st.check_error() == 0
    prm = params_for(wl)
    out2 = torch.empty_like(x["q"])
    ws = hla.prefill(prm, *_args(x), out2, state=st)
    torch.cuda.synchronize()
    assert st.check_error() == ERR_STATE
    assert hla.check_workspace_error(ws) == 0
    assert torch.equal(out, out2)  # the outputs do not depend on the state


def test_negative_decode_position_is_flagged_and_left_alone():
    wl = synth.small("bad pos", [40, 70], n_q_heads=4, n_kv_heads=2, head_dim=64, decode_steps=1)
    x = synth.make_inputs(wl, "cuda")
    _, st = run_prefill(wl, x, with_state=True)
    st.view("pos")[0] = -5
    prm = params_for(wl)
    out = torch.empty(x["dq"].shape[1:], dtype=x["dq"].dtype, device="cuda")
    hla.decode_step(prm, x["dq"][0], x["dk"][0], x["dv"][0], x["dg"][0], x["dbeta"][0], x["lam"], x["wq"],
                    x["wk"], x["wv"], st, out)
    torch.cuda.synchronize()
    assert st.check_error() == ERR_STATE
    assert st.view("pos").cpu().tolist() == [-5, 71]
