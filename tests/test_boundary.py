"""CPU checks of the C ABI: the library loads, exports every entry point that
include/hla.h declares, and rejects bad arguments on the host (no GPU call is
made on any of these paths)."""
import ctypes
import os
import re

import pytest

from linearized_attention_rope_gb300 import hla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from linearized_attention_rope_gb300 import build

    build.build()
    return hla.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "hla.h"), encoding="utf-8").read()
    return re.findall(r"HLA_API\s+[\w\s\*]+?\b(hla_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    assert {"hla_state_init", "hla_prefill", "hla_decode_step"} <= names
    assert {"hla_state_bytes", "hla_prefill_workspace_bytes", "hla_status_string",
            "hla_check_device_error", "hla_check_workspace_error"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def declared_arities():
    """{entry point: number of parameters} from the declarations in include/hla.h."""
    text = open(os.path.join(ROOT, "include", "hla.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for name, args in re.findall(r"HLA_API\s+[\w\s\*]+?\b(hla_\w+)\s*\(([^)]*)\)", text):
        args = args.strip()
        out[name] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_argument_counts_match_header(lib):
    # every entry point the binding declares argtypes for passes exactly the header's parameters
    ar = declared_arities()
    checked = 0
    for name, n in ar.items():
        argtypes = getattr(lib, name).argtypes
        if argtypes is not None:
            assert len(argtypes) == n, f"{name}: binding passes {len(argtypes)}, header declares {n}"
            checked += 1
    assert checked == len(ar)


def test_struct_layouts_match_header():
    assert ctypes.sizeof(hla.CParams) == 9 * 4
    assert ctypes.sizeof(hla.CState) == 13 * 8
    assert ctypes.sizeof(hla.CStateSizes) == 13 * 8


def test_status_strings(lib):
    assert hla.status_string(hla.HLA_OK) == "ok"
    assert "workspace" in hla.status_string(hla.HLA_ERR_WORKSPACE)
    assert hla.status_string(99) == "unknown status"


def _p(**kw):
    base = dict(n_q_heads=32, n_kv_heads=8, head_dim=128, n_sinks=8, window=56)
    base.update(kw)
    return hla.Params(**base)


def test_state_sizes(lib):
    sz = hla.state_sizes(_p(window=888), 64)
    assert sz["S"] == 64 * 32 * 128 * 128 * 4
    assert sz["k_ring"] == 64 * 8 * 896 * 128 * 2
    assert sz["pend_k"] == 64 * 8 * 889 * 128 * 4
    assert sz["pend_g"] == 64 * 32 * 889 * 4
    assert sz["conv_q"] == 64 * 7 * 32 * 128 * 4
    assert sz["pos"] == 64 * 8
    # per-step decode scratch: q rot, qhat, o_lin [N, Hq, d]; per split of 64 key slots
    # (14 for an 896-slot ring) the running max, sum and P V
    assert sz["scratch"] == 4 * (3 * 64 * 32 * 128 + 2 * 64 * 32 * 14 + 64 * 32 * 14 * 128)
    f32 = hla.state_sizes(_p(dtype=hla.DTYPE_F32, head_dim=64), 1)
    assert f32["k_ring"] == 8 * 64 * 64 * 4


def test_prefill_launch_count(lib):
    # tensor-core path: one table launch, features, softmax, then a chunk-local and a state launch
    # for each of the two parts of the chunk slots; plus the decode-state hand-off when asked
    assert hla.prefill_launch_count(_p()) == 7
    assert hla.prefill_launch_count(_p(), with_state=True) == 8
    # token-serial path (fp32 layer): tables, features, recurrent GDN, softmax + combine
    assert hla.prefill_launch_count(_p(dtype=hla.DTYPE_F32, head_dim=64)) == 4


def test_workspace_grows_with_tokens(lib):
    a = hla.workspace_bytes(_p(), 4096, 1)
    b = hla.workspace_bytes(_p(), 8192, 1)
    assert 0 < a < b
    assert hla.workspace_bytes(_p(), 0, 1) > 0


@pytest.mark.parametrize("kw,code", [
    (dict(n_q_heads=30), hla.HLA_ERR_INVALID_ARG),   # not a multiple of n_kv_heads
    (dict(head_dim=96), hla.HLA_ERR_UNSUPPORTED),
    (dict(window=0), hla.HLA_ERR_INVALID_ARG),
    (dict(n_sinks=-1), hla.HLA_ERR_INVALID_ARG),
    (dict(conv_width=4), hla.HLA_ERR_UNSUPPORTED),
    (dict(dtype=7), hla.HLA_ERR_UNSUPPORTED),
    (dict(flags=0x100), hla.HLA_ERR_INVALID_ARG),
])
def test_bad_params_rejected_on_host(lib, kw, code):
    with pytest.raises(hla.HlaError) as e:
        hla.workspace_bytes(_p(**kw), 16, 1)
    assert e.value.status == code


def test_prefill_rejects_null_and_misaligned_pointers_without_gpu(lib):
    prm = _p().c()
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1001)
    args = [fake] * 10
    rc = lib.hla_prefill(ctypes.byref(prm), None, *args[1:], 1, 16, fake, None, fake, 1 << 30, None)
    assert rc == hla.HLA_ERR_INVALID_ARG
    rc = lib.hla_prefill(ctypes.byref(prm), odd, *args[1:], 1, 16, fake, None, fake, 1 << 30, None)
    assert rc == hla.HLA_ERR_INVALID_ARG
    rc = lib.hla_prefill(ctypes.byref(prm), *args, 0, 16, fake, None, fake, 1 << 30, None)
    assert rc == hla.HLA_ERR_INVALID_ARG  # no sequences
    rc = lib.hla_prefill(ctypes.byref(prm), *args, 1, 16, fake, None, fake, 16, None)
    assert rc == hla.HLA_ERR_WORKSPACE
    bad_state = hla.CState(*([0x1000] * 11 + [0] + [0x1000]))  # no error word
    rc = lib.hla_prefill(ctypes.byref(prm), *args, 1, 16, fake, ctypes.byref(bad_state), fake,
                         1 << 30, None)
    assert rc == hla.HLA_ERR_INVALID_ARG


def test_decode_rejects_bad_state_without_gpu(lib):
    prm = _p().c()
    fake = ctypes.c_void_p(0x1000)
    bad_state = hla.CState(*([0x1000] * 5 + [0x1008] + [0x1000] * 7))  # misaligned pend_g
    rc = lib.hla_decode_step(ctypes.byref(prm), 4, *([fake] * 9), ctypes.byref(bad_state), fake, None)
    assert rc == hla.HLA_ERR_INVALID_ARG
    rc = lib.hla_decode_step(ctypes.byref(prm), -1, *([fake] * 9), ctypes.byref(bad_state), fake, None)
    assert rc == hla.HLA_ERR_INVALID_ARG
    rc = lib.hla_state_init(ctypes.byref(prm), 4, None, None)
    assert rc == hla.HLA_ERR_INVALID_ARG


def test_decode_rejects_head_groups_over_eight_without_gpu(lib):
    # 16 query heads per kv head: refused on the host before any pointer is looked at
    prm = _p(n_q_heads=32, n_kv_heads=2).c()
    fake = ctypes.c_void_p(0x1000)
    state = hla.CState(*([0x1000] * 13))
    rc = lib.hla_decode_step(ctypes.byref(prm), 4, *([fake] * 9), ctypes.byref(state), fake, None)
    assert rc == hla.HLA_ERR_UNSUPPORTED


def test_scan_flag_sizes_its_buffers_on_the_token_serial_path_only(lib):
    f32 = dict(n_q_heads=2, n_kv_heads=1, head_dim=64, dtype=hla.DTYPE_F32)
    plain = hla.workspace_bytes(_p(**f32), 8192, 1)
    scan = hla.workspace_bytes(_p(flags=hla.FLAG_L2NORM_Q | hla.FLAG_GDN_SCAN, **f32), 8192, 1)
    # 127 parts of 64 absorptions (plus the bound's slack): maps (R, P) and start states of d x d fp32
    assert scan - plain >= 127 * 2 * 3 * 64 * 64 * 4
    tc = hla.workspace_bytes(_p(), 4096, 1)
    assert hla.workspace_bytes(_p(flags=hla.FLAG_L2NORM_Q | hla.FLAG_GDN_SCAN), 4096, 1) == tc


def test_gla_and_stall_flags_are_known(lib):
    assert hla.workspace_bytes(_p(flags=hla.FLAG_L2NORM_Q | hla.FLAG_GLA), 16, 1) > 0
    assert hla.workspace_bytes(_p(flags=hla.FLAG_L2NORM_Q | hla.FLAG_TEST_STALL), 16, 1) > 0


def test_continue_workspace_covers_the_cached_rows(lib):
    # tensor-core path: the prefill's workspace for the new tokens plus every sequence's n_sinks + window
    # cached rows, and the extended rows' v, g, beta and output; token-serial path: the prefill's
    tc = _p()
    assert hla.continue_workspace_bytes(tc, 1000, 4) >= hla.workspace_bytes(tc, 1000 + 4 * 64, 4)
    assert hla.continue_workspace_bytes(tc, 1000, 4) > hla.continue_workspace_bytes(tc, 1000, 1)
    serial = _p(head_dim=64)
    assert hla.continue_workspace_bytes(serial, 1000, 4) == hla.workspace_bytes(serial, 1000, 4)
