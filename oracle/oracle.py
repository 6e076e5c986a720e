"""ctypes wrapper around the fp64 C oracle (``hla_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Marshals numpy float64 arrays into the C
functions; no arithmetic of the method lives here.  ``layer_units`` runs many
(sequence, query-head) units on a thread pool: ctypes releases the GIL for
the duration of each C call, so the threads run on separate host cores.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hla_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math) into oracle/liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int),
        ("n_sinks", ctypes.c_int),
        ("window", ctypes.c_int),
        ("conv_width", ctypes.c_int),
        ("rope_base", ctypes.c_double),
        ("l2_eps", ctypes.c_double),
        ("l2norm_q", ctypes.c_int),
        ("erase_off", ctypes.c_int),
        ("softmax_off", ctypes.c_int),
    ]


@dataclass
class OracleCfg:
    d: int
    n_sinks: int
    window: int
    conv_width: int = 8
    rope_base: float = 500000.0
    l2_eps: float = 1e-6
    l2norm_q: bool = True
    erase_off: bool = False
    softmax_off: bool = False

    def c(self) -> _Cfg:
        return _Cfg(self.d, self.n_sinks, self.window, self.conv_width, self.rope_base,
                    self.l2_eps, int(self.l2norm_q), int(self.erase_off), int(self.softmax_off))


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_rope.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, _dp, _dp]
            lib.oracle_short_conv.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp, _dp, _dp]
            lib.oracle_l2norm.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, _dp, _dp]
            lib.oracle_gdn_delayed.argtypes = [ctypes.c_int] * 4 + [_dp] * 5 + [ctypes.c_int, _dp, _dp]
            lib.oracle_key_visible.argtypes = [ctypes.c_int] * 4
            lib.oracle_key_visible.restype = ctypes.c_int
            lib.oracle_window_softmax.argtypes = [ctypes.c_int] * 4 + [_dp] * 4
            lib.oracle_layer_unit.argtypes = (
                [ctypes.POINTER(_Cfg), ctypes.c_int] + [_dp] * 5 + [ctypes.c_double] + [_dp] * 3
                + [_dp] * 9
            )
            lib.oracle_layer_unit.restype = ctypes.c_int
            lib.oracle_key_stats.argtypes = [ctypes.c_int, ctypes.c_int, _dp, _dp, _dp]
            _lib = lib
    return _lib


def _in(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(_dp)


def rope(x, base: float) -> np.ndarray:
    x = _in(x)
    y = np.empty_like(x)
    _load().oracle_rope(x.shape[0], x.shape[1], base, _p(x), _p(y))
    return y


def conv(x, w) -> np.ndarray:
    x, w = _in(x), _in(w)
    y = np.empty_like(x)
    _load().oracle_short_conv(x.shape[0], x.shape[1], w.shape[1], _p(x), _p(w), _p(y))
    return y


def l2norm(x, eps: float = 1e-6) -> np.ndarray:
    x = _in(x)
    y = np.empty_like(x)
    _load().oracle_l2norm(x.shape[0], x.shape[1], eps, _p(x), _p(y))
    return y


def gdn_delayed(qhat, khat, vhat, g, beta, n_sinks: int, window: int, erase_off: bool = False):
    """Returns (o_lin [len, d], S_final [d, d])."""
    qhat, khat, vhat, g, beta = map(_in, (qhat, khat, vhat, g, beta))
    L, d = qhat.shape
    o = np.empty((L, d))
    S = np.empty((d, d))
    _load().oracle_gdn_delayed(L, d, n_sinks, window, _p(qhat), _p(khat), _p(vhat), _p(g),
                               _p(beta), int(erase_off), _p(o), _p(S))
    return o, S


def key_visible(p: int, j: int, n_sinks: int, window: int) -> bool:
    return bool(_load().oracle_key_visible(p, j, n_sinks, window))


def window_softmax(qr, kr, v, n_sinks: int, window: int) -> np.ndarray:
    qr, kr, v = map(_in, (qr, kr, v))
    o = np.empty_like(qr)
    _load().oracle_window_softmax(qr.shape[0], qr.shape[1], n_sinks, window, _p(qr), _p(kr),
                                  _p(v), _p(o))
    return o


_INTERMEDIATES = ("qr", "kr", "qhat", "khat", "vhat", "o_sm", "o_lin")


def layer_unit(cfg: OracleCfg, q, k, v, g, beta, lam: float, wq, wk, wv, want=()) -> dict:
    """The layer for one (sequence, query head).

    q [len, d] (this q-head), k, v [len, d] (its kv-head), g, beta [len],
    wq/wk/wv [d, width].  Returns {"o", "S"} plus any intermediates named in
    ``want`` (qr, kr, qhat, khat, vhat, o_sm, o_lin), all float64."""
    q, k, v, g, beta, wq, wk, wv = map(_in, (q, k, v, g, beta, wq, wk, wv))
    L, d = q.shape
    assert d == cfg.d
    out = {"o": np.empty((L, d)), "S": np.empty((d, d))}
    extra = []
    for name in _INTERMEDIATES:
        if name in want:
            out[name] = np.empty((L, d))
            extra.append(out[name])
        else:
            extra.append(None)
    c = cfg.c()
    rc = _load().oracle_layer_unit(ctypes.byref(c), L, _p(q), _p(k), _p(v), _p(g), _p(beta),
                                   float(lam), _p(wq), _p(wk), _p(wv), _p(out["o"]),
                                   _p(out["S"]), *[_p(a) for a in extra])
    if rc != 0:
        raise MemoryError("oracle_layer_unit failed to allocate")
    return out


def layer_units(cfg: OracleCfg, jobs, threads: int | None = None, want=()) -> list:
    """Runs ``layer_unit`` over a list of job dicts (keys q,k,v,g,beta,lam,wq,wk,wv,
    each a per-unit array) on a thread pool; returns the results in order."""
    threads = threads or os.cpu_count() or 1
    _load()

    def one(job):
        return layer_unit(cfg, job["q"], job["k"], job["v"], job["g"], job["beta"], job["lam"],
                          job["wq"], job["wk"], job["wv"], want=want)

    if threads <= 1 or len(jobs) <= 1:
        return [one(j) for j in jobs]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(one, jobs))


def key_stats(kr):
    """Key concentration |m_p| and projection residual at every position of one
    sequence and head (rows of kr, the RoPE'd keys); returns two float64 arrays."""
    kr = _in(kr)
    L, d = kr.shape
    conc = np.empty(L)
    res = np.empty(L)
    _load().oracle_key_stats(L, d, _p(kr), _p(conc), _p(res))
    return conc, res
