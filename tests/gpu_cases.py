"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
cut (sequence, q-head) units out of the same seeded inputs for the oracle,
and compare.

Tolerances: fp32 layer: relative L2 <= 1e-4; bf16 layer: relative L2 <= 5e-3
and max |diff| <= 1e-2 * max |ref|, on outputs and on final states.
"""
from __future__ import annotations

import numpy as np
import torch

from linearized_attention_rope_gb300 import hla, synth

TOL = {"f32": dict(rel_l2=1e-4, max_abs=None), "bf16": dict(rel_l2=5e-3, max_abs=1e-2)}


def params_for(wl: synth.Workload, flags: int = hla.FLAG_L2NORM_Q) -> hla.Params:
    return hla.Params(wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.n_sinks, wl.window,
                      dtype=hla.DTYPE_F32 if wl.dtype == "f32" else hla.DTYPE_BF16, flags=flags)


def run_prefill(wl, x, flags=hla.FLAG_L2NORM_Q, with_state=False):
    prm = params_for(wl, flags)
    out = torch.empty_like(x["q"])
    st = hla.State(prm, wl.n_seqs).init() if with_state else None
    ws = hla.prefill(prm, x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["wq"], x["wk"], x["wv"],
                     x["cu_seqlens"], out, state=st)
    torch.cuda.synchronize()
    assert hla.check_workspace_error(ws) == 0
    return out, st


def run_decode(wl, x, st, steps=None, flags=hla.FLAG_L2NORM_Q, first=0):
    """Runs decode steps [first, first+steps); returns outputs [steps, N, Hq, d]."""
    prm = params_for(wl, flags)
    steps = wl.decode_steps if steps is None else steps
    outs = torch.empty((steps,) + tuple(x["dq"].shape[1:]), dtype=x["dq"].dtype, device=x["dq"].device)
    for i in range(steps):
        s = first + i
        hla.decode_step(prm, x["dq"][s], x["dk"][s], x["dv"][s], x["dg"][s], x["dbeta"][s], x["lam"],
                        x["wq"], x["wk"], x["wv"], st, outs[i])
    torch.cuda.synchronize()
    assert st.check_error() == 0
    return outs


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def unit_job(wl, x, n, h, decode_steps=0):
    """Oracle inputs of (sequence n, q-head h): the prefill rows of that
    sequence, followed by its first `decode_steps` decode tokens."""
    cu = x["cu_seqlens"].tolist()
    a, b = cu[n], cu[n + 1]
    d, kv = wl.head_dim, h // (wl.n_q_heads // wl.n_kv_heads)
    q, k, v = x["q"][a:b, h], x["k"][a:b, kv], x["v"][a:b, kv]
    g, be = x["g"][a:b, h], x["beta"][a:b, h]
    if decode_steps:
        q = torch.cat([q, x["dq"][:decode_steps, n, h]])
        k = torch.cat([k, x["dk"][:decode_steps, n, kv]])
        v = torch.cat([v, x["dv"][:decode_steps, n, kv]])
        g = torch.cat([g, x["dg"][:decode_steps, n, h]])
        be = torch.cat([be, x["dbeta"][:decode_steps, n, h]])
    return dict(q=_np(q), k=_np(k), v=_np(v), g=_np(g), beta=_np(be), lam=float(x["lam"][h]),
                wq=_np(x["wq"][h * d:(h + 1) * d]), wk=_np(x["wk"][kv * d:(kv + 1) * d]),
                wv=_np(x["wv"][kv * d:(kv + 1) * d]))


def oracle_cfg(wl, oracle, **kw):
    return oracle.OracleCfg(d=wl.head_dim, n_sinks=wl.n_sinks, window=wl.window, **kw)


def metrics(got: np.ndarray, ref: np.ndarray) -> dict:
    diff = got - ref
    nref = float(np.linalg.norm(ref))
    return dict(rel_l2=float(np.linalg.norm(diff)) / max(nref, 1e-300),
                max_abs=float(np.abs(diff).max()) if diff.size else 0.0,
                ref_max=float(np.abs(ref).max()) if ref.size else 0.0, ref_norm=nref)


def assert_close(got, ref, dtype: str, what: str):
    m = metrics(np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64))
    tol = TOL[dtype]
    if m["ref_norm"] == 0.0:
        assert m["max_abs"] == 0.0, f"{what}: expected exact zeros, {m}"
        return m
    assert m["rel_l2"] <= tol["rel_l2"], f"{what}: {m}"
    if tol["max_abs"] is not None:
        assert m["max_abs"] <= tol["max_abs"] * m["ref_max"], f"{what}: {m}"
    return m


def unit_rows(x, n):
    cu = x["cu_seqlens"].tolist()
    return cu[n], cu[n + 1]


def strided_units(n_seqs: int, n_heads: int, count: int, offset: int = 0):
    """`count` (sequence, q-head) units spread over every sequence and over the heads: unit i takes
    sequence i mod n_seqs and head (offset + 7 i) mod n_heads (7 is coprime with the head counts
    used, so the heads of a sequence differ)."""
    return [(i % n_seqs, (offset + 7 * i) % n_heads) for i in range(count)]
