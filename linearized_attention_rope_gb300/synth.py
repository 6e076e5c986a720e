"""Seeded synthetic inputs shaped like the attention layers of LLaMA-3.1-8B and
Qwen3-32B.  No trained weights and no dataset are used.

This module only draws random tensors; it holds none of the layer's
arithmetic, so both the CUDA path and the oracle can consume its output.

Value recipe (every workload):
  q, v ~ N(0, 1); k = mu_h + sigma * N(0, I) with mu_h a random unit vector
  per kv head (keys concentrated around one direction, the regime the
  linearisation analysis assumes); conv filters ~ N(0, 1/8);
  beta = sigmoid(N(0, 1)); g = log(alpha) = -0.1 * softplus(N(0, 1));
  lambda_h = 1 or U(0.5, 1.5).
Tensors are drawn in fp32 from a seeded generator and rounded to the storage
dtype once; consumers read back exactly those bits.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

BASE_SEED = 20261202


@dataclass
class Workload:
    name: str
    seqlens: list            # one entry per independent sequence
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str               # "f32" or "bf16"
    n_sinks: int
    window: int
    lam: str = "uniform"     # "one" or "uniform"
    sigma: object = 0.3      # float, or (lo, hi) drawn per kv head
    decode_steps: int = 0
    seed: int = BASE_SEED
    rows: list = field(default_factory=list)  # packing note (varlen batch rows)

    @property
    def n_seqs(self) -> int:
        return len(self.seqlens)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


def workloads() -> dict:
    """The five reference workloads (c0 is the small parity case)."""
    return {
        "c0": Workload("PR1 ref: B1 T512 2q/1kv d64 fp32, 8 sinks + 56 window", [512], 2, 1, 64,
                       "f32", 8, 56, lam="one", seed=BASE_SEED + 0),
        "c1": Workload("LLaMA-3.1-8B layer prefill: B1 T4096 32q/8kv d128 bf16, 8 sinks + 56 window",
                       [4096], 32, 8, 128, "bf16", 8, 56, seed=BASE_SEED + 1),
        "c2": Workload("LLaMA-3.1-8B long prefill: B8 T32768 32q/8kv d128 bf16, 8 sinks + 120 window",
                       [32768] * 8, 32, 8, 128, "bf16", 8, 120, sigma=(0.1, 1.0), seed=BASE_SEED + 2),
        "c3": Workload("Decode: 64 seqs prefilled to 8192 then 512 steps, 32q/8kv d128 bf16, "
                       "ring 8 sinks + 888 window", [8192] * 64, 32, 8, 128, "bf16", 8, 888,
                       decode_steps=512, seed=BASE_SEED + 3),
        "c4": Workload("Qwen3-32B layer prefill: B2 T16384 varlen 1024/3072/4096/8192, 64q/8kv d128 bf16, "
                       "8 sinks + 56 window", [1024, 3072, 4096, 8192] * 2, 64, 8, 128, "bf16", 8, 56,
                       seed=BASE_SEED + 4, rows=[[1024, 3072, 4096, 8192]] * 2),
    }


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, device, seed):
    return torch.randn(*shape, generator=_gen(device, seed), device=device, dtype=torch.float32)


def _rand(shape, device, seed):
    return torch.rand(*shape, generator=_gen(device, seed), device=device, dtype=torch.float32)


def _keys(n_tok, wl: Workload, mu, sigma, device, seed):
    noise = _randn((n_tok, wl.n_kv_heads, wl.head_dim), device, seed)
    return mu[None] + sigma[None, :, None] * noise


def make_inputs(wl: Workload, device="cpu") -> dict:
    """Draws every input of ``wl`` on ``device``.

    Returns q [T,Hq,d], k, v [T,Hkv,d] (storage dtype); g, beta [T,Hq] fp32;
    lam [Hq]; wq [Hq*d,8], wk, wv [Hkv*d,8] fp32; cu_seqlens int32 [n+1]; and,
    for decode workloads, dq/dk/dv/dg/dbeta with a leading [steps, n_seqs] shape.
    """
    s = wl.seed * 64
    T, Hq, Hkv, d = wl.total_tokens, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    dt = wl.torch_dtype
    mu = _randn((Hkv, d), device, s + 1)
    mu = mu / mu.norm(dim=-1, keepdim=True)
    if isinstance(wl.sigma, tuple):
        lo, hi = wl.sigma
        sigma = lo + (hi - lo) * _rand((Hkv,), device, s + 2)
    else:
        sigma = torch.full((Hkv,), float(wl.sigma), device=device)
    out = {
        "q": _randn((T, Hq, d), device, s + 3).to(dt),
        "k": _keys(T, wl, mu, sigma, device, s + 4).to(dt),
        "v": _randn((T, Hkv, d), device, s + 5).to(dt),
        "g": -0.1 * torch.nn.functional.softplus(_randn((T, Hq), device, s + 6)),
        "beta": torch.sigmoid(_randn((T, Hq), device, s + 7)),
        "wq": _randn((Hq * d, 8), device, s + 8) * (1.0 / 8) ** 0.5,
        "wk": _randn((Hkv * d, 8), device, s + 9) * (1.0 / 8) ** 0.5,
        "wv": _randn((Hkv * d, 8), device, s + 10) * (1.0 / 8) ** 0.5,
    }
    if wl.lam == "one":
        out["lam"] = torch.ones(Hq, device=device)
    else:
        out["lam"] = 0.5 + _rand((Hq,), device, s + 11)
    cu = [0]
    for L in wl.seqlens:
        cu.append(cu[-1] + int(L))
    out["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32, device=device)
    if wl.decode_steps:
        n, st = wl.n_seqs, wl.decode_steps
        out["dq"] = _randn((st, n, Hq, d), device, s + 12).to(dt)
        out["dk"] = _keys(st * n, wl, mu, sigma, device, s + 13).reshape(st, n, Hkv, d).to(dt)
        out["dv"] = _randn((st, n, Hkv, d), device, s + 14).to(dt)
        out["dg"] = -0.1 * torch.nn.functional.softplus(_randn((st, n, Hq), device, s + 15))
        out["dbeta"] = torch.sigmoid(_randn((st, n, Hq), device, s + 16))
    return out


def cotangent(wl: Workload, device="cpu", seed_offset: int = 0) -> torch.Tensor:
    """dO [T, Hq, d] ~ N(0, 1) in the storage dtype: the output gradient a backward pass receives."""
    T, Hq, d = wl.total_tokens, wl.n_q_heads, wl.head_dim
    return _randn((T, Hq, d), device, wl.seed * 64 + 40 + seed_offset).to(wl.torch_dtype)


def small(name: str, seqlens, n_q_heads=4, n_kv_heads=2, head_dim=64, dtype="bf16", n_sinks=8,
          window=56, decode_steps=0, seed=BASE_SEED + 100, sigma=0.3, lam="uniform") -> Workload:
    """A reduced workload with the same value recipe (for parity and edge cases)."""
    return Workload(name, list(seqlens), n_q_heads, n_kv_heads, head_dim, dtype, n_sinks, window,
                    lam=lam, sigma=sigma, decode_steps=decode_steps, seed=seed)
