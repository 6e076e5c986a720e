"""Gradients of the hybrid layer for one (sequence, query head), in fp64.

TEST INFRASTRUCTURE ONLY: the tests may use it; the CUDA library never does.
It shares no code with the CUDA path or with the C oracle: the layer is
restated here with plain PyTorch CPU ops in float64, step by step in the
pages' order, and torch.autograd differentiates it.  The restatement is
pinned to the C oracle's forward (same outputs on the same inputs) and the
gradients to central finite differences of the C oracle (tests).

Steps (page "迈向线性的关键：分析驱动的 Transformer 线性化"):
  - RoPE, rotate-half pairs (i, i + d/2), angle p * base^(-2i/d);
  - causal depthwise conv of width 8 (tap 7 on the current token) of the
    RoPE'd q and k and of the raw v (section 实践建议, item 3);
  - L2 normalisation of q~ and k~ (eps 1e-6 inside the root);
  - GDN update S <- alpha S - beta alpha k (k^T S) + beta k v^T (section
    线性注意力替换机制), token j absorbed at position j + W if j >= n_sinks
    (section 填补近似缺口的实用设计), read-out o_lin = S^T qhat;
    with erase_off the GLA update S <- alpha S + k v^T;
  - softmax over the sinks and the window with scale 1/sqrt(d) on the RoPE'd
    q, k and the raw v;
  - o = o_sm + lambda o_lin ("Untangling Component Imbalance in Hybrid Linear
    Attention Conversion", section 关键设计 (1)).
"""
from __future__ import annotations

import math

import numpy as np
import torch


def _rope(x: torch.Tensor, base: float) -> torch.Tensor:
    L, d = x.shape
    half = d // 2
    i = torch.arange(half, dtype=torch.float64)
    theta = base ** (-2.0 * i / d)
    ang = torch.arange(L, dtype=torch.float64)[:, None] * theta[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    x1, x2 = x[:, :half], x[:, half:]
    return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=1)


def _conv(x: torch.Tensor, w: torch.Tensor) -> torch.Tensor:
    # y_p[c] = sum_m w[c][m] x_{p-7+m}[c], zero before the sequence start
    L, d = x.shape
    width = w.shape[1]
    xp = torch.cat([torch.zeros(width - 1, d, dtype=x.dtype), x], dim=0)
    y = torch.zeros(L, d, dtype=x.dtype)
    for m in range(width):
        y = y + w[:, m][None, :] * xp[m:m + L]
    return y


def _l2(x: torch.Tensor, eps: float) -> torch.Tensor:
    return x / torch.sqrt((x * x).sum(dim=1, keepdim=True) + eps)


def _visible(p: int, j: int, n_sinks: int, window: int) -> bool:
    return j <= p and (j < n_sinks or j >= p - window + 1)


def layer(q, k, v, g, beta, lam, wq, wk, wv, *, n_sinks, window, base=500000.0, eps=1e-6, l2norm_q=True,
          erase_off=False):
    """o [L, d] of one unit from float64 torch tensors (autograd-ready)."""
    L, d = q.shape
    qr, kr = _rope(q, base), _rope(k, base)
    qt, kt, vh = _conv(qr, wq), _conv(kr, wk), _conv(v, wv)
    qh = _l2(qt, eps) if l2norm_q else qt
    kh = _l2(kt, eps)
    S = torch.zeros(d, d, dtype=torch.float64)
    o_lin = []
    for p in range(L):
        j = p - window
        if j >= n_sinks:
            a = torch.exp(g[j])
            kj, vj = kh[j], vh[j]
            if erase_off:
                S = a * S + torch.outer(kj, vj)
            else:
                x = kj @ S
                S = a * S - beta[j] * a * torch.outer(kj, x) + beta[j] * torch.outer(kj, vj)
        o_lin.append(S.T @ qh[p])
    o_lin = torch.stack(o_lin) if L else torch.zeros(0, d, dtype=torch.float64)
    mask = torch.tensor([[_visible(p, j, n_sinks, window) for j in range(L)] for p in range(L)], dtype=torch.bool)
    logits = (qr @ kr.T) / math.sqrt(d)
    logits = logits.masked_fill(~mask, float("-inf"))
    o_sm = torch.softmax(logits, dim=1) @ v
    return o_sm + lam * o_lin


NAMES = ("q", "k", "v", "g", "beta", "lam", "wq", "wk", "wv")


def grads(job: dict, dout, *, n_sinks, window, l2norm_q=True, erase_off=False) -> dict:
    """Gradients of sum(dout * o) with respect to every input of one unit (float64 numpy arrays);
    `job` holds q, k, v [L, d], g, beta [L], lam, wq, wk, wv [d, 8]."""
    t = {n: torch.tensor(np.asarray(job[n], dtype=np.float64), requires_grad=True) for n in NAMES}
    o = layer(*[t[n] for n in NAMES], n_sinks=n_sinks, window=window, l2norm_q=l2norm_q, erase_off=erase_off)
    loss = (o * torch.tensor(np.asarray(dout, dtype=np.float64))).sum()
    gr = torch.autograd.grad(loss, [t[n] for n in NAMES], allow_unused=True)
    return {n: (np.zeros_like(job[n], dtype=np.float64) if x is None else x.detach().numpy())
            for n, x in zip(NAMES, gr)} | {"o": o.detach().numpy()}
