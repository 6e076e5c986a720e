#!/usr/bin/env python
"""Benchmark of the hybrid GDN + sink/SWA layer on GB300.

Default: prefill of the LLaMA-3.1-8B-shaped layer (B=1, T=4096, 32 q / 8 kv
heads, head_dim 128, bf16, 8 sinks + 56 window) -> tokens/s, plus the decode
workload (64 sequences prefilled to 8192, ring 8 + 888) -> decode steps/s,
both through the libhla C ABI on synthetic seeded inputs.

One JSON line on stdout (rank 0).  ``--impl reference`` times the fp64 CPU
oracle instead (the reference arm).  Under torchrun every rank runs its own
replica of the workload (the layer shards into independent sequences, so
there is no data-path collective): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "hybrid GDN+sink/SWA layer prefill tokens/s & decode steps/s on 1 GB300; % roofline"
L2_FLUSH_BYTES = 512 << 20
FP32_ALU_TFLOPS_DERIVATION = "152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz"
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000,
                    help="timed steps of the headline prefill workload (about 0.5 s of c1 steps)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c1", choices=["c1", "c2", "c4"],
                    help="prefill workload of the headline line")
    ap.add_argument("--extra", default="c2,c4",
                    help="further prefill workloads reported as prefill_<name> objects ('' for none)")
    ap.add_argument("--extra-seconds", type=float, default=0.5,
                    help="approximate timed region of each further workload (steps derived from a trial)")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode measurement")
    ap.add_argument("--scan", type=int, default=1,
                    help="1: also time the context-parallel token-serial GDN on a long fp32 sequence and the "
                         "prefill continuation (chunked prefill)")
    ap.add_argument("--only", default="", choices=["", "backward", "scan", "continue", "diagnostics", "gla"],
                    help="run one secondary measurement alone with few calls (--warmup warm-up calls; --steps timed "
                         "calls for continue; 3 for backward and scan): the form the profiler captures use")
    ap.add_argument("--backward", default="c1", choices=["", "c1", "c2", "c4"],
                    help="workload of the backward (hla_backward) measurement; empty to skip")
    ap.add_argument("--backward-seconds", type=float, default=2.0,
                    help="about how long the backward's timed region runs")
    ap.add_argument("--decode-only", action="store_true",
                    help="only the decode measurement (one JSON line with its results)")
    ap.add_argument("--traffic-from", metavar="NCU_REP", default=None,
                    help="write the counters of an ncu report into profiles/traffic.json under --traffic-key "
                         "and exit; runs here, without a GPU")
    ap.add_argument("--traffic-key", default="c1", help="workload key of the report given to --traffic-from")
    ap.add_argument("--traffic-calls", type=int, default=1,
                    help="calls (prefill calls or decode steps) each report given to --traffic-from covers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-steps", type=int, default=4000,
                    help="timed decode steps (step s feeds the inputs of synthetic step s mod 512)")
    ap.add_argument("--e2e-steps", type=int, default=200, help="timed steps of each end-to-end measurement")
    ap.add_argument("--stage-steps", type=int, default=50, help="instrumented steps for per-kernel times")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing: one process per GPU, max over ranks
class Dist:
    def __init__(self):
        import torch

        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist

            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist
        if torch.cuda.is_available():
            torch.cuda.set_device(self.local)

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def max_over_ranks(dist, value: float) -> float:
    return dist.max(value)


# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        p["source"] = "measured"
        return p
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_traffic(kernel: str, source_files, workload: str = "c1") -> float | None:
    """DRAM bytes per step (summed over the kernel's launches in one call)
    recorded for `workload` from an ncu capture of `kernel`, if the kernel's
    sources are unchanged since (hash match); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(workload, {}).get(kernel)
    if not rec:
        return None
    h = hashlib.sha256()
    for s in source_files:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("source_sha256"):
        return None
    return rec.get("dram_bytes_per_step")


def source_hash(files) -> str:
    h = hashlib.sha256()
    for s in files:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ---------------------------------------------------------------------------
# prefill
GDN_RECURRENT_SOURCES = ["linearized_attention_rope_gb300/csrc/gdn_recurrent.cu",
                         "linearized_attention_rope_gb300/csrc/hla_common.cuh"]
CSRC = "linearized_attention_rope_gb300/csrc/"
GDN_PREP_SOURCES = [CSRC + "gdn_inverse.cu", CSRC + "umma.cuh", CSRC + "hla_common.cuh"]
GDN_CHUNKED_SOURCES = [CSRC + "gdn_chunked.cu", CSRC + "umma.cuh", CSRC + "tma.cuh", CSRC + "hla_common.cuh"]
SOFTMAX_TC_SOURCES = [CSRC + "window_softmax_tc.cu", CSRC + "umma.cuh", CSRC + "tma.cuh", CSRC + "hla_common.cuh"]
FEATURES_SOURCES = [CSRC + "features.cu", CSRC + "hla_common.cuh"]


def chunked_gdn_flops_per_token_head(d: int = 128, C: int = 64) -> dict:
    """Useful flops of the chunked GDN per absorbed token and q-head, split by
    kernel (triangles halved).  Chunk-local kernel: the Gram triangle K K^T,
    the masked Q K^T and the triangular solve for T.  State kernel: the three
    d x d products (W S0, Q S0, Kt^T U) and U~ = T diag(b) V, Wm = T diag(b g) K,
    P U."""
    prep = (C - 1) * d / 2 + (C + 1) * d / 2 + (C * C - 1) / 6
    state = 3 * d * d + 3 * (C + 1) * d / 2
    return {"prep": 2.0 * prep, "state": 2.0 * state, "total": 2.0 * (prep + state)}


def prefill_work(wl):
    """Algorithmic work of one prefill launch per stage."""
    d, Hq, Hkv = wl.head_dim, wl.n_q_heads, wl.n_kv_heads
    T = wl.total_tokens
    absorbed = sum(max(0, L - wl.window - wl.n_sinks) for L in wl.seqlens)
    keys = sum(visible_keys(L, wl.n_sinks, wl.window) for L in wl.seqlens)
    eb = 2 if wl.dtype == "bf16" else 4
    if wl.dtype == "bf16" and d == 128:
        f = chunked_gdn_flops_per_token_head(d)
        gdn_state = {"bound": "tensor", "flops": f["state"] * absorbed * Hq,
                     "unit": "TFLOP/s", "sources": GDN_CHUNKED_SOURCES, "kernel": "gdn_chunked_kernel"}
        gdn_prep = {"bound": "tensor", "flops": f["prep"] * absorbed * Hq,
                    "unit": "TFLOP/s", "sources": GDN_PREP_SOURCES, "kernel": "gdn_inverse_kernel"}
    else:
        # token-serial delta rule: k^T S, the rank-1 update, q^T S -> 6 d^2 flops per token-head
        gdn_state = {"bound": "alu", "flops": 6.0 * d * d * absorbed * Hq, "peak": FP32_ALU_TFLOPS,
                     "unit": "TFLOP/s", "sources": GDN_RECURRENT_SOURCES, "kernel": "gdn_recurrent_kernel"}
        gdn_prep = None
    return {
        "gdn_prep": gdn_prep,
        "gdn_state": gdn_state,
        # q.k and p.v over the visible keys of every (token, q-head)
        "softmax": ({"bound": "tensor", "flops": 4.0 * d * keys * Hq, "unit": "TFLOP/s",
                     "sources": SOFTMAX_TC_SOURCES,
                     "kernel": "window_softmax_tc_kernel"}
                    if wl.dtype == "bf16" and d == 128 else
                    {"bound": "alu", "flops": 4.0 * d * keys * Hq, "peak": FP32_ALU_TFLOPS,
                     "unit": "TFLOP/s", "sources": ["linearized_attention_rope_gb300/csrc/window_softmax.cu"],
                     "kernel": "window_softmax_kernel"}),
        # read q, k, v; write RoPE'd q, k and qhat, khat, vhat
        "features": {"bound": "hbm", "bytes": float(T * d * ((Hq + 2 * Hkv) * eb + (2 * Hq + 3 * Hkv) * eb)),
                     "unit": "GB/s", "sources": FEATURES_SOURCES,
                     "kernel": "features_kernel"},
        "absorbed_token_heads": absorbed * Hq,
    }


def run_prefill_bench(key, steps, warmup, dist, peaks, e2e_steps=200, stage_steps=50, trial_seconds=None):
    """Prefill of workload `key`: `steps` timed steps (or, with trial_seconds, as many as fill about that
    long after a short trial), per-kernel times, the roofline of the dominant kernel, and the end-to-end
    number through the C ABI with host buffers."""
    import torch

    from linearized_attention_rope_gb300 import hla, synth

    wl = synth.workloads()[key]
    x = synth.make_inputs(wl, "cuda")
    prm = hla.Params(wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.n_sinks, wl.window,
                     dtype=hla.DTYPE_BF16 if wl.dtype == "bf16" else hla.DTYPE_F32)
    out = torch.empty_like(x["q"])
    ws = hla.alloc_workspace(prm, wl.total_tokens, wl.n_seqs)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        hla.prefill(prm, x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"],
                    x["wv"], x["cu_seqlens"], out, ws=ws)

    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if trial_seconds:  # size the timed region from a short trial
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(3):
            step()
        b.record(stream)
        b.synchronize()
        per = a.elapsed_time(b) / 3 / 1e3
        steps = max(10, int(trial_seconds / max(per, 1e-6)))
        steps = int(dist.max(float(steps)))
    assert hla.check_workspace_error(ws) == 0
    n_stage = 23
    chunked = wl.dtype == "bf16" and wl.head_dim == 128 and wl.n_q_heads // wl.n_kv_heads in (1, 2, 4, 8)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with ClockSampler(dist.local) as clocks:
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    dist.barrier()
    step_ms = [starts[i].elapsed_time(ends[i]) for i in range(steps)]
    # Per-kernel durations: further steps with the library's stage events on, right after the timed
    # region (with the hook on every launch runs alone; events inside the timed region would serialise
    # the launches that overlap there).
    n_inst = max(1, min(stage_steps, steps))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_stage)] for _ in range(n_inst)]
    for row in ev:  # materialise the event handles
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(n_inst):
        flush.zero_()
        hla.set_prefill_stage_events(ev[i])
        step()
    hla.set_prefill_stage_events(None)
    torch.cuda.synchronize()

    def stages(row):
        t = [0.0] + [row[0].elapsed_time(row[j]) for j in range(1, n_stage)]  # ms from mark 0
        if chunked:  # each GDN kernel runs once per part of the chunk slots: a stage sums its launches
            return {"features": t[1], "softmax": t[2] - t[1],
                    "gdn_prep": sum(t[8 + 4 * p] - t[7 + 4 * p] for p in range(4)),
                    "gdn_state": sum(t[10 + 4 * p] - t[9 + 4 * p] for p in range(4))}
        return {"features": t[1], "gdn_state": t[4] - t[3], "softmax": t[5] - t[4]}

    per_step = [stages(ev[i]) for i in range(n_inst)]
    stage_ms = {k: statistics.mean(st[k] for st in per_step) for k in per_step[0]}
    device_s = dist.max(sum(step_ms) / 1e3)
    launches_per_step = hla.prefill_launch_count(prm)

    work = prefill_work(wl)

    def roof(name):
        w, sec = work[name], stage_ms[name] / 1e3
        if w["bound"] == "hbm":
            achieved, peak = w["bytes"] / sec / 1e9, peaks["hbm_gbs"]
        elif w["bound"] == "tensor":
            achieved, peak = w["flops"] / sec / 1e12, peaks["bf16_tflops"]
        else:
            achieved, peak = w["flops"] / sec / 1e12, w["peak"]
        return {"kernel": w["kernel"], "bound": w["bound"], "achieved": round(achieved, 3), "peak": peak,
                "unit": w["unit"], "frac": round(achieved / peak, 5),
                "traffic": kernel_traffic(w["kernel"], w["sources"], key),
                "algorithmic": w.get("bytes", w.get("flops")),
                "peak_source": (peaks["source"] + " burst" if w["bound"] == "tensor" else peaks["source"])
                if w["bound"] != "alu" else FP32_ALU_TFLOPS_DERIVATION}

    measured = [k for k in stage_ms if work.get(k)]
    roofline = roof(max(measured, key=stage_ms.get))  # the dominant kernel
    stage_roofline = {k: {kk: v for kk, v in roof(k).items() if kk in ("kernel", "bound", "achieved", "unit",
                                                                         "frac")}
                      for k in measured}
    # the whole layer against its own bound: the larger of the HBM time of the algorithmic bytes and the
    # tensor time of the algorithmic flops
    layer = layer_work(wl)
    t_bound = max(layer["bytes"] / (peaks["hbm_gbs"] * 1e9), layer["flops"] / (peaks["bf16_tflops"] * 1e12))
    layer_roof = {"bytes": layer["bytes"], "flops": layer["flops"], "bound_ms": round(t_bound * 1e3, 5),
                  "frac": round(t_bound / (device_s / steps), 5)}

    # end to end through the C ABI: every step's inputs copied in from pinned host memory and its result
    # copied back to pinned host memory, inside the timed region
    host = {k: x[k].cpu().pin_memory() for k in ("q", "k", "v", "g", "beta", "cu_seqlens")}
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = host_out.numel() * host_out.element_size()
    e2e_n = max(1, min(e2e_steps, steps))
    # (a) serial: copy in, prefill, copy out on one stream, one step at a time (L2 flushed before each)
    serial_n = max(1, min(e2e_n, 20))
    e2e_ms = []
    for i in range(2 + serial_n):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for k in host:
            x[k].copy_(host[k], non_blocking=True)
        step()
        host_out.copy_(out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= 2:
            e2e_ms.append(a.elapsed_time(b))
    serial_s = dist.max(sum(e2e_ms) / 1e3)
    # (b) pipelined, as a serving loop runs it: step i's inputs are copied in on one stream while step i - 1
    # computes and step i - 2's result is copied out on a third; two device input sets and outputs
    # alternate, each reused only once the step two back has finished with it (events)
    xs = [x, dict(x, **{k: torch.empty_like(x[k]) for k in host})]
    outs = [out, torch.empty_like(out)]
    host_outs = [host_out, torch.empty(out.shape, dtype=out.dtype, pin_memory=True)]
    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in, ev_c, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def pipe(i):
        bi = i & 1
        xb = xs[bi]
        if i >= 2:
            s_in.wait_event(ev_c[bi])  # step i - 2 has read this input set
        with torch.cuda.stream(s_in):
            for k in host:
                xb[k].copy_(host[k], non_blocking=True)
        ev_in[bi].record(s_in)
        s_c.wait_event(ev_in[bi])
        if i >= 2:
            s_c.wait_event(ev_out[bi])  # step i - 2's result has been copied out of this output
        hla.prefill(prm, xb["q"], xb["k"], xb["v"], xb["g"], xb["beta"], xb["lam"], xb["wq"], xb["wk"],
                    xb["wv"], xb["cu_seqlens"], outs[bi], ws=ws, stream=s_c)
        ev_c[bi].record(s_c)
        s_out.wait_event(ev_c[bi])
        with torch.cuda.stream(s_out):
            host_outs[bi].copy_(outs[bi], non_blocking=True)
        ev_out[bi].record(s_out)

    for i in range(4):
        pipe(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(e2e_n):
        pipe(i)
    b.record(s_out)
    b.synchronize()
    e2e_s = dist.max(a.elapsed_time(b) / 1e3)
    assert hla.check_workspace_error(ws) == 0
    del host, host_out, host_outs, xs, outs
    tokens = wl.total_tokens * dist.world
    res = {
        "value": tokens * steps / device_s, "unit": "tokens/s", "steps": steps, "warmup": warmup,
        "ms_per_step": device_s * 1e3 / steps, "wall_s": wall,
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()}, "roofline": roofline,
        "stage_roofline": stage_roofline, "layer_roofline": layer_roof,
        "clocks": clocks.summary(), "gpu_launches": launches_per_step * steps,
        "e2e": {"value": tokens * e2e_n / e2e_s, "unit": "tokens/s", "steps": e2e_n,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "mode": "pipelined: step i's inputs copied in while step i-1 computes and step i-2's result is "
                        "copied out (three streams, two device input sets and outputs); no L2 flush, every step's "
                        "inputs arrive by copy",
                "serial_value": tokens * serial_n / serial_s, "serial_steps": serial_n},
        "workload": wl, "inputs": x,
    }
    del ws, out, flush
    return res


BWD_SOURCES = [CSRC + "backward.cu", CSRC + "hla_common.cuh"]
# hla_backward's stages, in order (stage marks 1 .. 8 follow them; the L2 backward runs inside the
# feat_out launch, so its interval is empty)
BWD_STAGES = ("rope", "conv", "gdn", "softmax", "l2", "feat_out", "conv_filters", "lambda")


def bwd_launches(wl) -> int:
    """Kernels one hla_backward call launches."""
    return 10 + (1 if wl.n_sinks > 0 else 0)


def backward_work(wl) -> dict:
    """Algorithmic work of the backward's stages: fp32 flops of the two compute stages, bytes of the three
    streaming ones (counted per entry below).  GDN, per absorbed token and
    q-head (every such token is also a read-out position): the forward's absorption (k^T S and the
    rank-1 update, 4 d^2) and read-out (2 d^2, for lambda's gradient), the read-out backward (S dO and
    q dO^T, 4 d^2) and the absorption backward (k^T S again, k^T dS, <dS, S_prev>, dS u, S_prev du and
    the dS update, 12 d^2): 22 d^2; the checkpoint recompute is overhead, not counted.  Softmax, per
    visible (query, key) pair and q-head: the logit, dP = dO . v, and the three products into dq, dk,
    dv, 2 d each: 10 d."""
    d, Hq, Hkv, T = wl.head_dim, wl.n_q_heads, wl.n_kv_heads, wl.total_tokens
    absorbed = sum(max(0, L - wl.window - wl.n_sinks) for L in wl.seqlens) * Hq
    keys = sum(visible_keys(L, wl.n_sinks, wl.window) for L in wl.seqlens) * Hq
    vb = 2 if wl.dtype == "bf16" else 4
    row = 4.0 * d  # one fp32 row of the workspace
    return {"gdn": {"bound": "alu", "flops": 22.0 * d * d * absorbed, "kernel": "bwd_gdn_kernel"},
            "softmax": {"bound": "alu", "flops": 10.0 * d * keys, "kernel": "bwd_softmax_kernel"},
            # the streaming launches, HBM-bound, per token: reads RoPE'd q and k and v; writes q~, qhat, k~,
            # khat, vhat (fp32)
            "conv": {"bound": "hbm", "kernel": "bwd_conv_kernel",
                     "bytes": T * (row * (Hq + Hkv) + vb * d * Hkv + row * (2 * Hq + 3 * Hkv))},
            # reads dqhat, the group's per-head dkhat, dvhat and softmax gradients (each Hq rows), q~ and k~,
            # the RoPE angles; writes the conv-output gradients and dq, dk, dv
            "feat_out": {"bound": "hbm", "kernel": "bwd_feat_out_kernel",
                         "bytes": T * (row * (6 * Hq + Hq + Hkv) + row + 2 * row * (Hq + 2 * Hkv))},
            # reads the conv inputs and the conv-output gradients (the partial sums are small)
            "conv_filters": {"bound": "hbm", "kernel": "bwd_convw_part_kernel",
                             "bytes": T * (row * (Hq + Hkv) + vb * d * Hkv + row * (Hq + 2 * Hkv))}}


def run_backward_bench(key, dist, peaks, trial_seconds=2.0, warmup=3, stage_steps=5, e2e_steps=5):
    """hla_backward on workload `key`: as many timed steps as fill about trial_seconds, per-launch
    times, the roofline of the dominant kernel, and the end-to-end number with host buffers."""
    import torch

    from linearized_attention_rope_gb300 import hla, synth

    wl = synth.workloads()[key]
    x = synth.make_inputs(wl, "cuda")
    dout = synth.cotangent(wl, "cuda")
    prm = hla.Params(wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.n_sinks, wl.window,
                     dtype=hla.DTYPE_BF16 if wl.dtype == "bf16" else hla.DTYPE_F32)
    ws = torch.empty(hla.backward_workspace_bytes(prm, wl.total_tokens, wl.n_seqs), dtype=torch.uint8,
                     device="cuda")
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"], x["wv"], x["cu_seqlens"])
    grads = hla.backward(prm, *args, dout, ws=ws)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        hla.backward(prm, *args, dout, grads=grads, ws=ws)

    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert hla.check_workspace_error(ws) == 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    step()
    b.record(stream)
    b.synchronize()
    steps = int(dist.max(float(max(3, int(trial_seconds / max(a.elapsed_time(b) / 1e3, 1e-6))))))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dist.local) as clocks:
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    dist.barrier()
    device_s = dist.max(sum(starts[i].elapsed_time(ends[i]) for i in range(steps)) / 1e3)
    # per-launch times from the library's stage marks (the launches run one after another anyway)
    n_marks = len(BWD_STAGES) + 1
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_marks)] for _ in range(stage_steps)]
    for row in ev:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(stage_steps):
        flush.zero_()
        hla.set_prefill_stage_events(ev[i])
        step()
    hla.set_prefill_stage_events(None)
    torch.cuda.synchronize()
    stage_ms = {name: statistics.mean(row[j].elapsed_time(row[j + 1]) for row in ev)
                for j, name in enumerate(BWD_STAGES)}
    work = backward_work(wl)

    def roof(name):
        w = work[name]
        sec = stage_ms[name] / 1e3
        traffic = kernel_traffic(w["kernel"], BWD_SOURCES, key + "_backward")
        if w["bound"] == "hbm":
            achieved = w["bytes"] / sec / 1e9
            return {"kernel": w["kernel"], "bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 5), "traffic": traffic,
                    "algorithmic": w["bytes"], "peak_source": peaks["source"]}
        achieved = w["flops"] / sec / 1e12
        return {"kernel": w["kernel"], "bound": "alu", "achieved": round(achieved, 4), "peak": FP32_ALU_TFLOPS,
                "unit": "TFLOP/s", "frac": round(achieved / FP32_ALU_TFLOPS, 5), "traffic": traffic,
                "algorithmic": w["flops"], "peak_source": FP32_ALU_TFLOPS_DERIVATION}

    dominant = max(work, key=lambda n: stage_ms[n])
    # end to end: inputs and dO from pinned host memory, every gradient back to pinned host memory
    host = {k: x[k].cpu().pin_memory() for k in ("q", "k", "v", "g", "beta", "cu_seqlens")}
    host["dout"] = dout.cpu().pin_memory()
    dev = dict(x, dout=dout)
    host_g = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in grads.items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_g.values())
    e2e_ms = []
    for i in range(1 + e2e_steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for k in host:
            dev[k].copy_(host[k], non_blocking=True)
        step()
        for n in grads:
            host_g[n].copy_(grads[n], non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= 1:
            e2e_ms.append(a.elapsed_time(b))
    e2e_s = dist.max(sum(e2e_ms) / 1e3)
    tokens = wl.total_tokens * dist.world
    res = {"value": tokens * steps / device_s, "unit": "tokens/s", "steps": steps, "warmup": warmup,
           "ms_per_step": device_s * 1e3 / steps,
           "config": {"workload": wl.name, "key": key, "l2": "flushed between steps (512 MiB write)",
                      "precision": "fp32 recompute and gradients from the stored bf16/fp32 inputs"},
           "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
           "roofline": roof(dominant), "stage_roofline": {n: roof(n) for n in work},
           "clocks": clocks.summary(), "gpu_launches": bwd_launches(wl) * steps,
           "gpu_launches_note": "per call: the block table, RoPE, conv, GDN, softmax query and key (and the "
                                "sink keys' sums where there are sinks), feature backward, filter partial "
                                "sums and their reduction, lambda",
           "e2e": {"value": tokens * e2e_steps / e2e_s, "unit": "tokens/s", "steps": e2e_steps,
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}}
    del ws, grads, flush, host, host_g
    return res


SCAN_SEQ = 32768


def scan_traffic(key):
    """DRAM bytes per prefill of the token-serial GDN launches (and the scan's) recorded under `key`."""
    parts = [kernel_traffic(k, GDN_RECURRENT_SOURCES, key) for k in ("gdn_recurrent_kernel", "gdn_part_scan_kernel")]
    return None if parts[0] is None else parts[0] + (parts[1] or 0.0)


def run_scan_bench(dist, trial_seconds=0.5, warmup=3):
    """The context-parallel token-serial GDN (HLA_FLAG_GDN_SCAN) against the single pass, on an fp32 layer
    of the reference config's head shape (2 q / 1 kv heads, d 64, 8 sinks + 56 window) over one long
    sequence: prefill tokens/s both ways and the GDN launches' time (stage marks 3 -> 4)."""
    import torch

    from linearized_attention_rope_gb300 import hla, synth

    wl = synth.small(f"fp32 layer, 2 q / 1 kv heads, d 64, 8 sinks + 56 window, one {SCAN_SEQ}-token sequence",
                     [SCAN_SEQ], n_q_heads=2, n_kv_heads=1, head_dim=64, dtype="f32", seed=synth.BASE_SEED + 500)
    x = synth.make_inputs(wl, "cuda")
    out = torch.empty_like(x["q"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    absorbed = sum(max(0, L - wl.window - wl.n_sinks) for L in wl.seqlens) * wl.n_q_heads
    res = {"config": {"workload": wl.name, "l2": "flushed between steps (512 MiB write)"}}
    for name, flags in (("single_pass", hla.FLAG_L2NORM_Q), ("scan", hla.FLAG_L2NORM_Q | hla.FLAG_GDN_SCAN)):
        prm = hla.Params(wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.n_sinks, wl.window, dtype=hla.DTYPE_F32,
                         flags=flags)
        ws = hla.alloc_workspace(prm, wl.total_tokens, wl.n_seqs)

        def step():
            hla.prefill(prm, x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"], x["wv"],
                        x["cu_seqlens"], out, ws=ws)

        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        assert hla.check_workspace_error(ws) == 0
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
        for e in ev:
            e.record(stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        b.synchronize()
        steps = int(dist.max(float(max(3, int(trial_seconds / max(a.elapsed_time(b) / 1e3, 1e-6))))))
        ms = []
        for _ in range(steps):
            flush.zero_()
            a.record(stream)
            step()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        flush.zero_()
        hla.set_prefill_stage_events(ev)
        step()
        hla.set_prefill_stage_events(None)
        torch.cuda.synchronize()
        gdn_ms = ev[3].elapsed_time(ev[4])
        dev_s = dist.max(sum(ms) / 1e3)
        flops = 6.0 * wl.head_dim ** 2 * absorbed
        res[name] = {"value": wl.total_tokens * dist.world * steps / dev_s, "unit": "tokens/s", "steps": steps,
                     "ms_per_step": dev_s * 1e3 / steps, "gdn_ms": round(gdn_ms, 4),
                     "gpu_launches": hla.prefill_launch_count(prm) * steps,
                     "roofline": {"kernel": "gdn_recurrent_kernel" + (" (+ gdn_part_scan_kernel)" if name == "scan"
                                                                      else ""),
                                  "bound": "alu", "achieved": round(flops / (gdn_ms / 1e3) / 1e12, 4),
                                  "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s",
                                  "frac": round(flops / (gdn_ms / 1e3) / 1e12 / FP32_ALU_TFLOPS, 5),
                                  "algorithmic": flops, "peak_source": FP32_ALU_TFLOPS_DERIVATION,
                                  "traffic": scan_traffic("scan_fp32" if name == "scan" else "scan_fp32_single")}}
        del ws
    return res


def run_gla_bench(dist, steps=200, warmup=5):
    """The LLaMA-3.1-8B-shaped prefill (4096 tokens) with the gated-linear-attention update
    (HLA_FLAG_GLA: S <- alpha S + k v^T, no erase) in place of the delta rule; each call timed with CUDA
    events (L2 flushed between calls)."""
    import torch

    from linearized_attention_rope_gb300 import hla, synth

    wl = synth.workloads()["c1"]
    x = synth.make_inputs(wl, "cuda")
    prm = hla.Params(wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.n_sinks, wl.window,
                     flags=hla.FLAG_L2NORM_Q | hla.FLAG_GLA)
    ws = hla.alloc_workspace(prm, wl.total_tokens, wl.n_seqs)
    out = torch.empty_like(x["q"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def call():
        hla.prefill(prm, x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"], x["wv"],
                    x["cu_seqlens"], out, ws=ws)

    for _ in range(warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    assert hla.check_workspace_error(ws) == 0
    ms = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    dev_s = dist.max(sum(ms) / 1e3)
    del ws, out, flush
    return {"value": wl.total_tokens * dist.world * steps / dev_s, "unit": "tokens/s", "steps": steps,
            "warmup": warmup, "ms_per_step": dev_s * 1e3 / steps,
            "config": {"workload": "LLaMA-3.1-8B layer shape (32q/8kv d128 bf16, 8 sinks + 56 window), B1 T4096, "
                                   "gated linear attention update (no erase)",
                       "l2": "flushed between calls (512 MiB write)"}}


def run_diagnostics_bench(dist, steps=30, warmup=3):
    """hla_prefill_diagnostics on the LLaMA-3.1-8B-shaped layer (4096 tokens): the prefill run with each
    branch alone, the two branch sums and the key statistics; each call timed with CUDA events (L2 flushed
    between calls)."""
    import torch

    from linearized_attention_rope_gb300 import hla, synth

    wl = synth.workloads()["c1"]
    x = synth.make_inputs(wl, "cuda")
    prm = hla.Params(wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.n_sinks, wl.window)
    ws = hla.alloc_workspace(prm, wl.total_tokens, wl.n_seqs)
    out = torch.empty_like(x["q"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def call():
        return hla.prefill_diagnostics(prm, x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"],
                                       x["wv"], x["cu_seqlens"], out=out, ws=ws)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    assert hla.check_workspace_error(ws) == 0
    ms = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    dev_s = dist.max(sum(ms) / 1e3)
    del ws, out, flush
    return {"value": wl.total_tokens * dist.world * steps / dev_s, "unit": "tokens/s", "steps": steps,
            "warmup": warmup, "ms_per_step": dev_s * 1e3 / steps,
            "config": {"workload": "LLaMA-3.1-8B layer shape (32q/8kv d128 bf16, 8 sinks + 56 window), B1 T4096: "
                                   "branch sums per (sequence, head) and key statistics per (position, kv head)",
                       "l2": "flushed between calls (512 MiB write)"}}


def run_continue_bench(dist, steps=30, warmup=3):
    """hla_prefill_continue on the LLaMA-3.1-8B-shaped layer: a 4096-token prefill with a decode state, then
    chunks of 4096 tokens appended one after another (chunked prefill), each call timed with CUDA events
    (L2 flushed between calls)."""
    import torch

    from linearized_attention_rope_gb300 import hla, synth

    wl = synth.workloads()["c1"]
    x0 = synth.make_inputs(wl, "cuda")
    x1 = synth.make_inputs(synth.small("chunk", [4096], n_q_heads=32, n_kv_heads=8, head_dim=128,
                                       seed=synth.BASE_SEED + 601), "cuda")
    for kk in ("wq", "wk", "wv", "lam"):
        x1[kk] = x0[kk]
    prm = hla.Params(wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.n_sinks, wl.window)
    args = lambda x: [x[k] for k in ("q", "k", "v", "g", "beta", "lam", "wq", "wk", "wv", "cu_seqlens")]  # noqa: E731
    st = hla.State(prm, 1).init()
    hla.prefill(prm, *args(x0), torch.empty_like(x0["q"]), state=st)
    out = torch.empty_like(x1["q"])
    ws = torch.empty(hla.continue_workspace_bytes(prm, 4096, 1), dtype=torch.uint8, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    for _ in range(warmup):
        hla.prefill_continue(prm, *args(x1), out, st, ws=ws)
    torch.cuda.synchronize()
    assert st.check_error() == 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ms = []
    for _ in range(steps):
        flush.zero_()
        a.record()
        hla.prefill_continue(prm, *args(x1), out, st, ws=ws)
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    dev_s = dist.max(sum(ms) / 1e3)
    del ws, flush
    return {"value": 4096 * dist.world * steps / dev_s, "unit": "tokens/s", "steps": steps, "warmup": warmup,
            "ms_per_step": dev_s * 1e3 / steps,
            "config": {"workload": "LLaMA-3.1-8B layer shape (32q/8kv d128 bf16, 8 sinks + 56 window): 4096-token "
                                   "chunks appended to one sequence after a 4096-token prefill",
                       "l2": "flushed between calls (512 MiB write)"}}


def layer_work(wl) -> dict:
    """Algorithmic work of the whole layer per prefill: bytes = q and o in the layer dtype, k and v per kv
    head, g and beta fp32 (intermediates excluded); flops = the chunked GDN's useful flops per absorbed
    token-head plus 4 d per visible key per (token, q-head) of the softmax."""
    d, Hq, Hkv = wl.head_dim, wl.n_q_heads, wl.n_kv_heads
    eb = 2 if wl.dtype == "bf16" else 4
    T = wl.total_tokens
    absorbed = sum(max(0, L - wl.window - wl.n_sinks) for L in wl.seqlens)
    keys = sum(visible_keys(L, wl.n_sinks, wl.window) for L in wl.seqlens)
    nbytes = T * (2 * Hq * d * eb + 2 * Hkv * d * eb + 2 * Hq * 4)
    flops = chunked_gdn_flops_per_token_head(d)["total"] * absorbed * Hq + 4.0 * d * keys * Hq
    return {"bytes": float(nbytes), "flops": float(flops)}


def visible_keys(L: int, n_sinks: int, window: int) -> int:
    """Keys the softmax branch visits over a sequence of L positions: min(p + 1, n_sinks) sinks plus
    the window positions after the sinks, for every position p."""
    total = 0
    for p in range(L):
        total += min(p + 1, n_sinks) + max(0, min(window, p + 1 - n_sinks))
    return total


# ---------------------------------------------------------------------------
# decode
def decode_bytes(wl, pos_mean: float) -> float:
    """Algorithmic HBM bytes of one decode step over all sequences."""
    N, Hq, Hkv, d = wl.n_seqs, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    eb = 2 if wl.dtype == "bf16" else 4
    keys = min(pos_mean + 1, wl.n_sinks + wl.window)
    b = N * Hq * d * d * 4 * 2                     # state read + write
    b += N * Hkv * keys * d * eb * 2               # ring K and V read
    b += N * Hkv * d * eb * 2                      # ring K and V write (new token)
    b += N * Hkv * d * 4 * 2 * 2                   # pending khat/vhat: one read, one write
    b += N * 7 * (Hq + 2 * Hkv) * d * 4 * 2        # conv caches read + write
    b += N * (Hq + 2 * Hkv) * d * eb + N * Hq * d * eb   # q, k, v in; out
    return float(b)


DECODE_SOURCES = [CSRC + "decode.cu", CSRC + "hla_common.cuh"]
DECODE_KERNELS = ("decode_features_kernel", "decode_attn_state_kernel", "decode_combine_kernel")


def decode_traffic() -> float | None:
    """DRAM bytes of one decode step (all its launches) from the committed capture, if decode.cu is
    unchanged since."""
    parts = [kernel_traffic(k, DECODE_SOURCES, "c3") for k in DECODE_KERNELS]
    return None if any(p is None for p in parts) else float(sum(parts))


def run_decode_bench(args, dist, peaks):
    import torch

    from linearized_attention_rope_gb300 import hla, synth

    wl = synth.workloads()["c3"]
    x = synth.make_inputs(wl, "cuda")
    prm = hla.Params(wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.n_sinks, wl.window)
    out = torch.empty_like(x["q"])
    st = hla.State(prm, wl.n_seqs).init()
    hla.prefill(prm, x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"], x["wv"],
                x["cu_seqlens"], out, state=st)
    del out
    for key in ("q", "k", "v", "g", "beta"):  # the prefill inputs (~6.5 GB) are not needed any more
        x.pop(key)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    K = args.decode_steps
    W = args.warmup
    n_in = wl.decode_steps  # synthetic step inputs; step s feeds those of step s mod n_in
    dout = torch.empty(x["dq"].shape[1:], dtype=x["dq"].dtype, device="cuda")
    stream = torch.cuda.current_stream()

    def step(s):
        s %= n_in
        hla.decode_step(prm, x["dq"][s], x["dk"][s], x["dv"][s], x["dg"][s], x["dbeta"][s], x["lam"],
                        x["wq"], x["wk"], x["wv"], st, dout)

    for s in range(W):
        step(s)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    dist.barrier()
    with ClockSampler(dist.local) as clocks:
        for i in range(K):
            evs[i][0].record(stream)
            step(W + i)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    dist.barrier()
    assert st.check_error() == 0
    ms = [a.elapsed_time(b) for a, b in evs]
    dev_s = dist.max(sum(ms) / 1e3)
    per_step = dev_s / K
    nbytes = decode_bytes(wl, 8192 + W + K / 2)  # the ring is full from the first step on
    achieved = nbytes / per_step / 1e9
    # end to end: this step's q, k, v, g, beta from pinned host memory, the output back
    keys = ("dq", "dk", "dv", "dg", "dbeta")
    host = {k: x[k][:8].cpu().pin_memory() for k in keys}
    dev_in = {k: torch.empty_like(x[k][0]) for k in keys}
    host_out = torch.empty(dout.shape, dtype=dout.dtype, pin_memory=True)
    h2d = sum(dev_in[k].numel() * dev_in[k].element_size() for k in keys)
    d2h = host_out.numel() * host_out.element_size()
    e2e_n = min(K, 1000)
    # pipelined, as a serving loop runs it: step i's inputs are copied in on one stream while step i - 1
    # runs and step i - 2's output is copied out on a third (two device input sets and outputs, each reused
    # once the step two back is done with it); the steps themselves stay in order on one stream
    dev_ins = [dev_in, {k: torch.empty_like(x[k][0]) for k in keys}]
    douts = [dout, torch.empty_like(dout)]
    host_outs = [host_out, torch.empty(dout.shape, dtype=dout.dtype, pin_memory=True)]
    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in, ev_c, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(e2e_n):
        bi = i & 1
        if i >= 2:
            s_in.wait_event(ev_c[bi])
        with torch.cuda.stream(s_in):
            for k in keys:
                dev_ins[bi][k].copy_(host[k][i % 8], non_blocking=True)
        ev_in[bi].record(s_in)
        s_c.wait_event(ev_in[bi])
        if i >= 2:
            s_c.wait_event(ev_out[bi])
        d = dev_ins[bi]
        hla.decode_step(prm, d["dq"], d["dk"], d["dv"], d["dg"], d["dbeta"], x["lam"], x["wq"], x["wk"], x["wv"],
                        st, douts[bi], stream=s_c)
        ev_c[bi].record(s_c)
        s_out.wait_event(ev_c[bi])
        with torch.cuda.stream(s_out):
            host_outs[bi].copy_(douts[bi], non_blocking=True)
        ev_out[bi].record(s_out)
    b.record(s_out)
    b.synchronize()
    e2e_s = dist.max(a.elapsed_time(b) / 1e3)
    assert st.check_error() == 0
    traffic = decode_traffic()
    return {"value": K * dist.world / dev_s, "unit": "steps/s", "steps": K, "warmup": W,
            "ms_per_step": per_step * 1e3, "tokens_per_s": K * dist.world * wl.n_seqs / dev_s,
            "config": {"workload": wl.name, "sequences": wl.n_seqs, "prefill_len": 8192,
                       "ring": wl.n_sinks + wl.window, "l2": "working set (state + ring) > L2",
                       "inputs": f"step s feeds the synthetic inputs of step s mod {n_in}"},
            "roofline": {"kernel": "decode_step", "bound": "hbm", "achieved": round(achieved, 2),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": traffic, "algorithmic_bytes_per_step": nbytes,
                         "peak_source": peaks["source"]},
            "e2e": {"value": e2e_n * dist.world / e2e_s, "unit": "steps/s", "steps": e2e_n,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "mode": "pipelined: step i's inputs copied in while step i-1 runs and step i-2's output is "
                            "copied out (three streams, two device input sets and outputs)"},
            "clocks": clocks.summary(), "gpu_launches": DECODE_LAUNCHES * K}


DECODE_LAUNCHES = 3  # features; state + softmax; combine


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and reference arm)
def oracle_jobs(wl, x, units):
    """Oracle inputs of the (sequence, q-head) units, cut from the input tensors x (any device)."""
    import torch

    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    cu = x["cu_seqlens"].tolist()
    d, G = wl.head_dim, wl.n_q_heads // wl.n_kv_heads
    jobs = []
    for n, h in units:
        a, b = cu[n], cu[n + 1]
        kv = h // G
        jobs.append(dict(q=f64(x["q"][a:b, h]), k=f64(x["k"][a:b, kv]), v=f64(x["v"][a:b, kv]),
                         g=f64(x["g"][a:b, h]), beta=f64(x["beta"][a:b, h]),
                         lam=float(x["lam"][h]), wq=f64(x["wq"][h * d:(h + 1) * d]),
                         wk=f64(x["wk"][kv * d:(kv + 1) * d]), wv=f64(x["wv"][kv * d:(kv + 1) * d])))
    return jobs


def oracle_units(wl, target_token_heads: float):
    """A strided sample of (sequence, q-head) units whose token-heads add up to about the target
    (all units if they add up to less): every sequence, q-heads spread evenly."""
    total = wl.total_tokens * wl.n_q_heads
    frac = min(1.0, target_token_heads / total)
    per_seq = max(1, round(wl.n_q_heads * frac))
    stride = wl.n_q_heads / per_seq
    return [(n, int(i * stride)) for n in range(wl.n_seqs) for i in range(per_seq)]


# fp64 oracle token-heads per second and core, for sizing the samples (about 10-30 s of CPU work)
ORACLE_TOKEN_HEADS_PER_CORE_S = 1.7e4


def time_oracle(wl, x, units, reps=1):
    """Wall times of the oracle over `units` of wl, on all host cores."""
    import oracle

    oracle.build()
    jobs = oracle_jobs(wl, x, units)
    cfg = oracle.OracleCfg(d=wl.head_dim, n_sinks=wl.n_sinks, window=wl.window)
    cores = min(os.cpu_count() or 1, len(jobs))
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.layer_units(cfg, jobs, threads=cores)
        times.append(time.perf_counter() - t0)
    return times, cores


def cpu_baseline(wl, x, seconds: float = 10.0):
    """The oracle as it stands, on the host cores, over a strided sample of units sized to about
    `seconds`; reported in token-equivalents (a token needs all q-heads) per second."""
    cores = os.cpu_count() or 1
    units = oracle_units(wl, seconds * cores * ORACLE_TOKEN_HEADS_PER_CORE_S)
    times, used = time_oracle(wl, x, units)
    if times[0] < seconds / 2:  # the whole workload is a short sample: repeat it up to about `seconds`
        more, _ = time_oracle(wl, x, units, reps=max(0, min(30, int(seconds / max(times[0], 1e-3))) - 1))
        times += more
    seqlens = wl.seqlens
    token_heads = sum(seqlens[n] for n, _ in units)
    tokens = token_heads / wl.n_q_heads
    return {"value": tokens * len(times) / sum(times), "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"{wl.name}: {len(units)} (sequence, q-head) units, q-heads strided evenly over every "
                      f"sequence ({token_heads} token-heads = {tokens:.0f} token-equivalents), {len(times)} "
                      f"pass(es), fp64 C oracle, {used} threads, {sum(times):.1f} s"}


def run_reference(args, dist):
    from linearized_attention_rope_gb300 import synth

    if dist.rank != 0:
        return None
    wl = synth.workloads()[args.workload]
    x = synth.make_inputs(wl, "cpu")
    cores = os.cpu_count() or 1
    # each step a bounded sample: about 1 s of oracle work per step
    units = oracle_units(wl, 1.0 * cores * ORACLE_TOKEN_HEADS_PER_CORE_S)
    times, used = time_oracle(wl, x, units, reps=args.warmup + args.steps)
    timed = times[args.warmup:]
    token_heads = sum(wl.seqlens[n] for n, _ in units)
    tokens = token_heads / wl.n_q_heads
    value = tokens * len(timed) / sum(timed)
    sample = (f"{wl.name}: {len(units)} (sequence, q-head) units per step, q-heads strided evenly over every "
              f"sequence ({tokens:.0f} token-equivalents), fp64 C oracle, {used} threads")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(timed) / len(timed),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "tokens": wl.total_tokens},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


TRAFFIC_KERNELS = {  # kernel name -> the sources its counters are keyed by
    "features_kernel": FEATURES_SOURCES,
    "window_softmax_tc_kernel": SOFTMAX_TC_SOURCES,
    "gdn_inverse_kernel": GDN_PREP_SOURCES,
    "gdn_chunked_kernel": GDN_CHUNKED_SOURCES,
    "decode_features_kernel": DECODE_SOURCES,
    "decode_attn_state_kernel": DECODE_SOURCES,
    "decode_combine_kernel": DECODE_SOURCES,
    "bwd_gdn_kernel": BWD_SOURCES,
    "bwd_sm_query_kernel": BWD_SOURCES,
    "bwd_sm_key_kernel": BWD_SOURCES,
    "bwd_conv_kernel": BWD_SOURCES,
    "bwd_feat_out_kernel": BWD_SOURCES,
    "bwd_convw_part_kernel": BWD_SOURCES,
    "gdn_recurrent_kernel": GDN_RECURRENT_SOURCES,
    "gdn_part_scan_kernel": GDN_RECURRENT_SOURCES,
}


def write_traffic(reps: str, key: str, calls: int = 1):
    """Stores the counters of ncu reports (comma-separated paths of reports, or of their
    `ncu -i rep --page raw --csv` exports ending in .csv) in
    profiles/traffic.json under workload `key`; each report holds the launches of `calls` calls (prefill
    calls or decode steps) of the kernels it captured.  A kernel in several reports keeps the last."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    data = {}
    if os.path.exists(path):
        with open(path) as f:
            data = json.load(f)
    entry = {}
    for rep in reps.split(","):
        if rep.endswith(".csv"):  # an export of `ncu -i <report> --page raw --csv`
            with open(rep) as f:
                raw = f.read()
        else:
            raw = subprocess.run(["ncu", "-i", rep, "--page", "raw", "--csv"], check=True, capture_output=True,
                                 text=True).stdout
        entry.update(traffic_from_csv(raw, calls))
    if "_command" in data.get(key, {}):  # the capture command recorded with the earlier counters
        entry["_command"] = data[key]["_command"]
    data[key] = entry
    data[key]["_reports"] = [os.path.basename(r) for r in reps.split(",")]
    with open(path, "w") as f:
        json.dump(data, f, indent=1)
        f.write("\n")


def traffic_from_csv(raw: str, calls: int = 1) -> dict:
    """Per kernel of TRAFFIC_KERNELS, the DRAM bytes and ncu durations of its launches in an ncu raw-page
    CSV, summed and divided by the number of calls the capture covers (per call: the GDN kernels run once
    per part of the chunk slots), keyed by a hash of the kernel's sources."""
    import csv
    import io

    rows = list(csv.reader(io.StringIO(raw)))
    head, body = rows[0], [r for r in rows[2:] if r]  # rows[1] holds the units
    col = {k: head.index(k) for k in ("Kernel Name", "dram__bytes_read.sum", "dram__bytes_write.sum",
                                      "gpu__time_duration.sum")}
    units = rows[1]
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "ns": 1e-3, "nsecond": 1e-3, "us": 1.0,
             "usecond": 1.0, "ms": 1e3, "msecond": 1e3}  # to bytes and microseconds
    out = {"_note": "per step = the kernel's launches in one call (cold caches: ncu flushes them before "
                    "each pass)"}
    for name, srcs in TRAFFIC_KERNELS.items():
        mine = [r for r in body if re.search(r"(^|[\s:])" + name + r"[<(]", r[col["Kernel Name"]])]
        if not mine:
            continue
        val = lambda r, k: float(r[col[k]].replace(",", "")) * scale[units[col[k]]]
        rd = sum(val(r, "dram__bytes_read.sum") for r in mine) / calls
        wr = sum(val(r, "dram__bytes_write.sum") for r in mine) / calls
        out[name] = {"source_sha256": source_hash(srcs), "launches_per_step": len(mine) / calls,
                     "dram_bytes_read": rd, "dram_bytes_write": wr, "dram_bytes_per_step": rd + wr,
                     "duration_us_ncu": round(sum(val(r, "gpu__time_duration.sum") for r in mine) / calls, 3)}
    return out


def prefill_line(pre: dict, key: str, dist, with_cpu: bool) -> dict:
    """The reported object of one prefill workload."""
    wl = pre.pop("workload")
    x = pre.pop("inputs")
    obj = {"value": pre["value"], "unit": "tokens/s", "steps": pre["steps"], "warmup": pre["warmup"],
           "ms_per_step": pre["ms_per_step"],
           "config": {"workload": wl.name, "key": key, "global_batch": wl.n_seqs * dist.world,
                      "seq_len": max(wl.seqlens), "tokens_per_rank": wl.total_tokens,
                      "l2": "flushed between steps (512 MiB write)"},
           "roofline": pre["roofline"], "layer_roofline": pre["layer_roofline"], "stage_ms": pre["stage_ms"],
           "stage_roofline": pre["stage_roofline"], "clocks": pre["clocks"], "e2e": pre["e2e"],
           "gpu_launches": pre["gpu_launches"], "wall_s": round(pre["wall_s"], 3)}
    if with_cpu:
        obj["cpu_baseline"] = cpu_baseline(wl, x)
    return obj


def main():
    args = parse()
    if args.traffic_from:
        write_traffic(args.traffic_from, args.traffic_key, args.traffic_calls)
        return
    dist = Dist()
    if args.impl == "reference":
        line = run_reference(args, dist)
        if line is not None:
            print(json.dumps(line), flush=True)
        dist.close()
        return
    import torch

    from linearized_attention_rope_gb300 import build as _build
    from linearized_attention_rope_gb300 import hla

    if dist.rank == 0 or not os.path.exists(hla.LIB_PATH):
        _build.build()
    dist.barrier()
    hla.load()
    peaks = measured_peaks()
    if args.decode_only:
        dec = run_decode_bench(args, dist, peaks)
        if dist.rank == 0:
            print(json.dumps({"decode": dec}), flush=True)
        dist.close()
        return
    if args.only:  # one secondary measurement alone, with few calls (for profiler captures)
        if args.only == "backward":
            part = run_backward_bench(args.backward or "c1", dist, peaks, trial_seconds=0.0, warmup=args.warmup,
                                      stage_steps=1, e2e_steps=1)
        elif args.only == "scan":
            part = run_scan_bench(dist, trial_seconds=0.0, warmup=args.warmup)
        elif args.only == "diagnostics":
            part = run_diagnostics_bench(dist, steps=args.steps, warmup=args.warmup)
        elif args.only == "gla":
            part = run_gla_bench(dist, steps=args.steps, warmup=args.warmup)
        else:
            part = run_continue_bench(dist, steps=args.steps, warmup=args.warmup)
        if dist.rank == 0:
            print(json.dumps({args.only: part}), flush=True)
        dist.close()
        return
    with_cpu = dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline
    pre = run_prefill_bench(args.workload, args.steps, args.warmup, dist, peaks, args.e2e_steps, args.stage_steps)
    wl = pre["workload"]
    head = prefill_line(pre, args.workload, dist, with_cpu)
    del pre
    torch.cuda.empty_cache()
    extras = {}
    for key in [k for k in args.extra.split(",") if k and k != args.workload]:
        p = run_prefill_bench(key, 0, 3, dist, peaks, min(args.e2e_steps, 10), min(args.stage_steps, 10),
                              trial_seconds=args.extra_seconds)
        extras["prefill_" + key] = prefill_line(p, key, dist, with_cpu)
        del p
        torch.cuda.empty_cache()
    scan = run_scan_bench(dist) if args.scan else None
    cont = run_continue_bench(dist) if args.scan else None
    diag = run_diagnostics_bench(dist) if args.scan else None
    gla = run_gla_bench(dist) if args.scan else None
    torch.cuda.empty_cache()
    bwd = None
    if args.backward:
        bwd = run_backward_bench(args.backward, dist, peaks, trial_seconds=args.backward_seconds)
        torch.cuda.empty_cache()
    dec = None if args.no_decode else run_decode_bench(args, dist, peaks)
    torch.cuda.synchronize()
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded; shapes of the named layer, no trained weights)",
        "config": dict(head["config"], parallelism=f"replicas x{dist.world}",
                       precision="bf16 in/out, fp16 MMA operands, fp32 state and accumulation"),
        "roofline": head["roofline"], "layer_roofline": head["layer_roofline"], "stage_ms": head["stage_ms"],
        "stage_ms_source": "each kernel's launches timed on their stream over --stage-steps instrumented steps "
                           "run right after the timed region (every launch alone)",
        "stage_roofline": head["stage_roofline"],
        "clocks": head["clocks"], "e2e": head["e2e"], "gpu_launches": head["gpu_launches"],
        "wall_s": head["wall_s"],
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    line.update(extras)
    if bwd:
        line["backward_" + args.backward] = bwd
    if scan:
        line["prefill_scan_fp32"] = scan
    if cont:
        line["prefill_continue_c1"] = cont
    if diag:
        line["prefill_diagnostics_c1"] = diag
    if gla:
        line["prefill_gla_c1"] = gla
    if dec:
        line["decode"] = dec
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
