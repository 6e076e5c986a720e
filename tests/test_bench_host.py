"""Host logic of bench.py (no GPU): the decode step's algorithmic bytes and the parser that turns an
ncu raw-page CSV into the per-kernel DRAM traffic bench.py reports."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from linearized_attention_rope_gb300 import synth  # noqa: E402


def test_decode_bytes_of_the_c3_step():
    wl = synth.workloads()["c3"]
    N, Hq, Hkv, d = 64, 32, 8, 128
    state = N * Hq * d * d * 4 * 2                 # fp32 state read and written once
    ring = N * Hkv * 896 * d * 2 * 2               # bf16 K and V over the full 8 + 888 slots
    assert state == 268_435_456 and ring == 234_881_024
    got = bench.decode_bytes(wl, 8192 + 100)
    rest = got - state - ring
    assert 20e6 < rest < 30e6                      # new-token writes, pending ring, conv caches, q/k/v/out
    # a position below the budget reads only the valid slots
    assert bench.decode_bytes(wl, 100) < got


def _csv(rows):
    head = ["ID", "Kernel Name", "dram__bytes_read.sum", "dram__bytes_write.sum", "gpu__time_duration.sum"]
    units = ["", "", "Mbyte", "Kbyte", "us"]
    lines = [head, units] + rows
    return "\n".join(",".join('"%s"' % c for c in r) for r in lines) + "\n"


def test_traffic_parser_sums_launches_per_kernel_and_converts_units():
    raw = _csv([
        ["0", "void features_kernel<__nv_bfloat16, __half, 128>(LayerDims, const T1 *)", "50", "30", "40.5"],
        ["1", "hla::<unnamed>::gdn_inverse_kernel(LayerDims, const __half *)", "20", "1", "38"],
        ["2", "hla::<unnamed>::gdn_inverse_kernel(LayerDims, const __half *)", "22", "3", "36"],
        ["3", "void at::vectorized_elementwise_kernel<4>(int)", "900", "900", "99"],
    ])
    out = bench.traffic_from_csv(raw)
    f = out["features_kernel"]
    assert f["launches_per_step"] == 1
    assert f["dram_bytes_read"] == 50e6 and f["dram_bytes_write"] == 30e3
    assert f["dram_bytes_per_step"] == 50e6 + 30e3 and f["duration_us_ncu"] == 40.5
    g = out["gdn_inverse_kernel"]
    assert g["launches_per_step"] == 2
    assert g["dram_bytes_per_step"] == 42e6 + 4e3 and g["duration_us_ncu"] == 74.0
    # keyed by the hash of the kernel's current sources; kernels absent from the report are left out
    assert g["source_sha256"] == bench.source_hash(bench.GDN_PREP_SOURCES)
    assert "gdn_chunked_kernel" not in out and "window_softmax_tc_kernel" not in out
