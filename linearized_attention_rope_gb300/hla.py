"""ctypes binding of libhla (include/hla.h).

Argument marshalling only: tensors are passed as ``data_ptr()`` and the
stream as ``torch.cuda.current_stream().cuda_stream``.  Every step of the
layer runs in libhla's CUDA kernels; there is no Python or CPU fallback, and
calling into the library without a built ``libhla.so`` raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhla.so")

HLA_OK = 0
HLA_ERR_INVALID_ARG = 1
HLA_ERR_UNSUPPORTED = 2
HLA_ERR_STATE = 3
HLA_ERR_CUDA = 4
HLA_ERR_TIMEOUT = 5
HLA_ERR_WORKSPACE = 6

DTYPE_F32 = 0
DTYPE_BF16 = 1
FLAG_L2NORM_Q = 0x1
FLAG_SOFTMAX_OFF = 0x2
FLAG_LINEAR_OFF = 0x4
FLAG_GDN_RECURRENT = 0x8
FLAG_GLA = 0x10
FLAG_TEST_STALL = 0x20
FLAG_GDN_SCAN = 0x40

STATE_FIELDS = ("S", "k_ring", "v_ring", "pend_k", "pend_v", "pend_g", "pend_beta", "conv_q",
                "conv_k", "conv_v", "pos", "err", "scratch")


class HlaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


class CParams(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("n_sinks", ctypes.c_int), ("window", ctypes.c_int),
                ("conv_width", ctypes.c_int), ("rope_base", ctypes.c_float),
                ("dtype", ctypes.c_int), ("flags", ctypes.c_uint)]


class CState(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in STATE_FIELDS]


class CStateSizes(ctypes.Structure):
    _fields_ = [(name, ctypes.c_size_t) for name in STATE_FIELDS]


_vp = ctypes.c_void_p
_lib = None


def load():
    """Loads libhla.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libhla.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(CParams)
        S = ctypes.POINTER(CState)
        lib.hla_status_string.argtypes = [ctypes.c_int]
        lib.hla_status_string.restype = ctypes.c_char_p
        lib.hla_state_bytes.argtypes = [P, ctypes.c_int, ctypes.POINTER(CStateSizes)]
        lib.hla_prefill_workspace_bytes.argtypes = [P, ctypes.c_int64, ctypes.c_int,
                                                    ctypes.POINTER(ctypes.c_size_t)]
        lib.hla_state_init.argtypes = [P, ctypes.c_int, S, _vp]
        lib.hla_prefill.argtypes = [P] + [_vp] * 10 + [ctypes.c_int, ctypes.c_int64, _vp, S, _vp,
                                                       ctypes.c_size_t, _vp]
        lib.hla_decode_step.argtypes = [P, ctypes.c_int] + [_vp] * 9 + [S, _vp, _vp]
        lib.hla_check_device_error.argtypes = [S, _vp, ctypes.POINTER(ctypes.c_int32)]
        lib.hla_check_workspace_error.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int32)]
        lib.hla_prefill_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
        lib.hla_prefill_launch_count.argtypes = [P, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
        lib.hla_prefill_noalloc.argtypes = [P] + [_vp] * 10 + [ctypes.c_int, ctypes.c_int64, _vp, S, _vp]
        lib.hla_prefill_noalloc.restype = ctypes.c_int
        lib.hla_prefill_continue.argtypes = [P] + [_vp] * 10 + [ctypes.c_int, ctypes.c_int64, _vp, S, _vp,
                                                                ctypes.c_size_t, _vp]
        lib.hla_prefill_continue.restype = ctypes.c_int
        lib.hla_prefill_continue_workspace_bytes.argtypes = [P, ctypes.c_int64, ctypes.c_int,
                                                             ctypes.POINTER(ctypes.c_size_t)]
        lib.hla_prefill_continue_workspace_bytes.restype = ctypes.c_int
        lib.hla_prefill_diagnostics.argtypes = [P] + [_vp] * 10 + [ctypes.c_int, ctypes.c_int64, _vp, _vp, _vp,
                                                                   _vp, ctypes.c_size_t, _vp]
        lib.hla_prefill_diagnostics.restype = ctypes.c_int
        lib.hla_backward_workspace_bytes.argtypes = [P, ctypes.c_int64, ctypes.c_int,
                                                     ctypes.POINTER(ctypes.c_size_t)]
        lib.hla_backward_workspace_bytes.restype = ctypes.c_int
        lib.hla_backward.argtypes = [P] + [_vp] * 10 + [ctypes.c_int, ctypes.c_int64] + [_vp] * 10 + [
            _vp, ctypes.c_size_t, _vp]
        lib.hla_backward.restype = ctypes.c_int
        lib.hla_prefill_noalloc_check_error.argtypes = [_vp, ctypes.POINTER(ctypes.c_int32)]
        lib.hla_prefill_noalloc_check_error.restype = ctypes.c_int
        for fn in ("hla_state_bytes", "hla_prefill_workspace_bytes", "hla_state_init", "hla_prefill",
                   "hla_decode_step", "hla_check_device_error", "hla_check_workspace_error",
                   "hla_prefill_stage_events", "hla_prefill_launch_count"):
            getattr(lib, fn).restype = ctypes.c_int
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().hla_status_string(status).decode()


def _check(rc: int, what: str):
    if rc != HLA_OK:
        raise HlaError(rc, what)


@dataclass
class Params:
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_sinks: int
    window: int
    dtype: int = DTYPE_BF16
    rope_base: float = 500000.0
    flags: int = FLAG_L2NORM_Q
    conv_width: int = 8

    def c(self) -> CParams:
        return CParams(self.n_q_heads, self.n_kv_heads, self.head_dim, self.n_sinks, self.window,
                       self.conv_width, self.rope_base, self.dtype, self.flags)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == DTYPE_F32 else torch.bfloat16


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def workspace_bytes(params: Params, total_tokens: int, n_seqs: int) -> int:
    n = ctypes.c_size_t()
    _check(load().hla_prefill_workspace_bytes(ctypes.byref(params.c()), total_tokens, n_seqs,
                                              ctypes.byref(n)), "hla_prefill_workspace_bytes")
    return n.value


def state_sizes(params: Params, n_seqs: int) -> dict:
    s = CStateSizes()
    _check(load().hla_state_bytes(ctypes.byref(params.c()), n_seqs, ctypes.byref(s)),
           "hla_state_bytes")
    return {name: getattr(s, name) for name in STATE_FIELDS}


class State:
    """Decode state of n_seqs sequences; the buffers are torch uint8 tensors."""

    def __init__(self, params: Params, n_seqs: int, device="cuda"):
        self.params, self.n_seqs = params, n_seqs
        self.buffers = {name: torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
                        for name, nbytes in state_sizes(params, n_seqs).items()}
        self.c = CState(*[b.data_ptr() for b in self.buffers.values()])

    def view(self, name: str):
        """Typed view of one buffer (S, pend_* and conv_* fp32; rings in the layer dtype;
        pos int64; err int32)."""
        b = self.buffers[name]
        dt = {"k_ring": self.params.torch_dtype, "v_ring": self.params.torch_dtype,
              "pos": torch.int64, "err": torch.int32}.get(name, torch.float32)
        n = state_sizes(self.params, self.n_seqs)[name] // torch.tensor([], dtype=dt).element_size()
        return b.view(dt)[:n]

    def init(self, stream=None):
        _check(load().hla_state_init(ctypes.byref(self.params.c()), self.n_seqs,
                                     ctypes.byref(self.c), _stream(stream)), "hla_state_init")
        return self

    def check_error(self, stream=None) -> int:
        """Synchronises, reads and clears the device error word; returns it (0 = fine)."""
        code = ctypes.c_int32()
        rc = load().hla_check_device_error(ctypes.byref(self.c), _stream(stream), ctypes.byref(code))
        if rc not in (HLA_OK, HLA_ERR_STATE, HLA_ERR_TIMEOUT):
            _check(rc, "device error word")
        return code.value


def alloc_workspace(params: Params, total_tokens: int, n_seqs: int, device="cuda"):
    return torch.empty(workspace_bytes(params, total_tokens, n_seqs), dtype=torch.uint8,
                       device=device)


def prefill(params: Params, q, k, v, g, beta, lam, wq, wk, wv, cu_seqlens, out, state=None,
            ws=None, stream=None):
    """hla_prefill on torch tensors (all on the GPU, contiguous)."""
    n_seqs = cu_seqlens.numel() - 1
    total = q.shape[0]
    if ws is None:
        ws = alloc_workspace(params, total, n_seqs, q.device)
    rc = load().hla_prefill(ctypes.byref(params.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                            _ptr(lam), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(cu_seqlens), n_seqs, total,
                            _ptr(out), None if state is None else ctypes.byref(state.c), _ptr(ws),
                            ws.numel(), _stream(stream))
    _check(rc, "hla_prefill")
    return ws


def continue_workspace_bytes(params: Params, total_tokens: int, n_seqs: int) -> int:
    n = ctypes.c_size_t()
    _check(load().hla_prefill_continue_workspace_bytes(ctypes.byref(params.c()), total_tokens, n_seqs,
                                                       ctypes.byref(n)), "hla_prefill_continue_workspace_bytes")
    return n.value


def prefill_continue(params: Params, q, k, v, g, beta, lam, wq, wk, wv, cu_seqlens, out, state: State, ws=None,
                     stream=None):
    """hla_prefill_continue: appends the tokens of every sequence to the context `state` holds."""
    n_seqs = cu_seqlens.numel() - 1
    total = q.shape[0]
    if ws is None:
        ws = torch.empty(continue_workspace_bytes(params, total, n_seqs), dtype=torch.uint8, device=q.device)
    rc = load().hla_prefill_continue(ctypes.byref(params.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(lam), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(cu_seqlens), n_seqs, total,
                                     _ptr(out), ctypes.byref(state.c), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "hla_prefill_continue")
    return ws


def prefill_diagnostics(params: Params, q, k, v, g, beta, lam, wq, wk, wv, cu_seqlens, out=None, ws=None,
                        stream=None):
    """hla_prefill_diagnostics: returns (branch_sq [n_seqs, Hq, 2], key_stats [total, Hkv, 2]), fp32
    tensors on the GPU (|o_sm|^2 and |lambda o_lin|^2 summed per sequence and head; key concentration
    and projection residual per position and kv head)."""
    n_seqs = cu_seqlens.numel() - 1
    total = q.shape[0]
    if ws is None:
        ws = alloc_workspace(params, total, n_seqs, q.device)
    if out is None:
        out = torch.empty_like(q)
    branch_sq = torch.empty((n_seqs, params.n_q_heads, 2), dtype=torch.float32, device=q.device)
    key_stats = torch.empty((total, params.n_kv_heads, 2), dtype=torch.float32, device=q.device)
    rc = load().hla_prefill_diagnostics(ctypes.byref(params.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                        _ptr(lam), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(cu_seqlens), n_seqs, total,
                                        _ptr(out), _ptr(branch_sq), _ptr(key_stats), _ptr(ws), ws.numel(),
                                        _stream(stream))
    _check(rc, "hla_prefill_diagnostics")
    return branch_sq, key_stats


def backward_workspace_bytes(params: Params, total_tokens: int, n_seqs: int) -> int:
    n = ctypes.c_size_t()
    _check(load().hla_backward_workspace_bytes(ctypes.byref(params.c()), total_tokens, n_seqs, ctypes.byref(n)),
           "hla_backward_workspace_bytes")
    return n.value


BACKWARD_GRADS = ("q", "k", "v", "g", "beta", "lam", "wq", "wk", "wv")


def backward(params: Params, q, k, v, g, beta, lam, wq, wk, wv, cu_seqlens, dout, grads=None, ws=None,
             stream=None):
    """hla_backward: the gradients of sum(dout * o) as a dict of fp32 GPU tensors named as in
    BACKWARD_GRADS, shaped like the inputs (q [total, Hq, d]; k, v [total, Hkv, d]; g, beta
    [total, Hq]; lam [Hq]; wq [Hq * d, 8]; wk, wv [Hkv * d, 8]).  `grads` (same dict) and `ws`
    (a uint8 tensor of backward_workspace_bytes) may be passed in to be reused."""
    n_seqs = cu_seqlens.numel() - 1
    total = q.shape[0]
    if ws is None:
        ws = torch.empty(backward_workspace_bytes(params, total, n_seqs), dtype=torch.uint8, device=q.device)
    if grads is None:
        src = dict(zip(BACKWARD_GRADS, (q, k, v, g, beta, lam, wq, wk, wv)))
        grads = {n: torch.empty(t.shape, dtype=torch.float32, device=q.device) for n, t in src.items()}
    rc = load().hla_backward(ctypes.byref(params.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(lam),
                             _ptr(wq), _ptr(wk), _ptr(wv), _ptr(cu_seqlens), n_seqs, total, _ptr(dout),
                             *[_ptr(grads[n]) for n in BACKWARD_GRADS], _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "hla_backward")
    return grads


def decode_step(params: Params, q, k, v, g, beta, lam, wq, wk, wv, state: State, out, stream=None):
    """hla_decode_step on torch tensors: q [N,Hq,d], k, v [N,Hkv,d], g, beta [N,Hq]."""
    rc = load().hla_decode_step(ctypes.byref(params.c()), state.n_seqs, _ptr(q), _ptr(k), _ptr(v),
                                _ptr(g), _ptr(beta), _ptr(lam), _ptr(wq), _ptr(wk), _ptr(wv),
                                ctypes.byref(state.c), _ptr(out), _stream(stream))
    _check(rc, "hla_decode_step")


def check_workspace_error(ws, stream=None) -> int:
    """Synchronises, reads and clears a prefill workspace's error word; returns it."""
    code = ctypes.c_int32()
    rc = load().hla_check_workspace_error(_ptr(ws), _stream(stream), ctypes.byref(code))
    if rc not in (HLA_OK, HLA_ERR_STATE, HLA_ERR_TIMEOUT):
        _check(rc, "workspace error word")
    return code.value


PREFILL_STAGES = ("features", "gdn", "softmax", "state_fill")
_stage_handles = None


def set_prefill_stage_events(events):
    """Makes hla_prefill record the given torch.cuda.Event objects (already
    recorded once, so their handles exist) at its stage boundaries on this
    thread; None switches the hook off."""
    global _stage_handles
    if events is None:
        _stage_handles = None
        _check(load().hla_prefill_stage_events(None, 0), "hla_prefill_stage_events")
        return
    _stage_handles = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(load().hla_prefill_stage_events(_stage_handles, len(events)), "hla_prefill_stage_events")


def prefill_launch_count(params: Params, with_state: bool = False) -> int:
    """hla_prefill_launch_count: kernels launched by one prefill call."""
    n = ctypes.c_int(0)
    _check(load().hla_prefill_launch_count(ctypes.byref(params.c()), int(with_state), ctypes.byref(n)),
           "hla_prefill_launch_count")
    return n.value


def prefill_noalloc(params: Params, q, k, v, g, beta, lam, wq, wk, wv, cu_seqlens, out, state=None,
                    stream=None):
    """hla_prefill_noalloc: the prefill with the library's own 64 MiB scratch, for
    callers that cannot allocate device memory; raises HlaError(HLA_ERR_WORKSPACE)
    for prefills that need more scratch than that."""
    rc = load().hla_prefill_noalloc(ctypes.byref(params.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                    _ptr(beta), _ptr(lam), _ptr(wq), _ptr(wk), _ptr(wv),
                                    _ptr(cu_seqlens), cu_seqlens.numel() - 1, q.shape[0], _ptr(out),
                                    None if state is None else ctypes.byref(state.c), _stream(stream))
    _check(rc, "hla_prefill_noalloc")


def prefill_noalloc_check_error(stream=None) -> int:
    """hla_prefill_noalloc_check_error: synchronises, reads and clears the error
    word of the library's own prefill buffer on the current device; returns it."""
    code = ctypes.c_int32()
    rc = load().hla_prefill_noalloc_check_error(_stream(stream), ctypes.byref(code))
    if rc not in (HLA_OK, HLA_ERR_STATE, HLA_ERR_TIMEOUT):
        _check(rc, "hla_prefill_noalloc_check_error")
    return code.value
