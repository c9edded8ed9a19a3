"""Seeded synthetic Muon inputs: the five workload configurations.

This module holds no arithmetic of the method.  It only draws parameters,
gradients and momenta, and it is the one module that both the oracle's
callers (tests, bench's CPU baseline) and the CUDA path's callers use, so
both sides see the same bytes.

The workloads of the DMuon evaluation (Wall-OSS-0.5, Pi0, Wall-WM,
Qwen2.5-7B; gist.science summary, section 4) need trained weights and data
that are not available; these sets stand in for them with the layer shapes of
a small transformer, of Llama-3-8B, of a heterogeneous embodied/VLA model and
of a large-layer stress case.

Per matrix i of configuration c, one torch generator seeded with
``seed_c * 1_000_003 + i`` draws, in this order and in fp32: W ~ N(0, 0.02^2),
then the gradient, then (when not zero) the momentum; each is cast to the
storage dtype with round-to-nearest-even.  Small sets are drawn on the CPU;
``device='cuda'`` draws on the GPU (different stream of numbers, same
recipe), which the large sets need.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

__all__ = ["Config", "CONFIGS", "get", "make_matrix", "make_set", "random_shapes"]


@dataclass(frozen=True)
class Config:
    name: str
    title: str
    dtype: str                  # 'bf16' | 'fp32'
    seed: int
    shapes: tuple               # ((rows, cols), ...)
    grad: str                   # 'normal' | 'heavy' | 'logscale'
    grad_scale: float = 1.0
    mom_std: float = 0.0        # 0 => zero momentum
    lr: float = 0.02
    beta: float = 0.95
    wd: float = 0.01
    ns_steps: int = 5
    precision: str = "bf16"     # 'bf16' | 'fp32'
    logscale: tuple = field(default=(0.0, 0.0))   # per-matrix 10**U(lo, hi)
    budget_gb: float = 0.0      # workspace per wave (0 = the whole set in one wave)


def _layers(n, per_layer):
    return tuple(s for _ in range(n) for s in per_layer)


def _vla_shapes(seed: int, count: int = 2000):
    g = torch.Generator().manual_seed(seed)
    rows = [64 << int(k) for k in torch.randint(0, 5, (count,), generator=g)]
    cols = [64 << int(k) for k in torch.randint(0, 7, (count,), generator=g)]
    return tuple(zip(rows, cols))


CONFIGS = {
    "c1": Config("c1", "single matrix 256x1024 fp32", "fp32", 0, ((256, 1024),), "normal",
                 precision="fp32"),
    "c2": Config("c2", "small-transformer set, 12 x {768x2304, 768x768, 768x3072, 3072x768}",
                 "bf16", 1, _layers(12, ((768, 2304), (768, 768), (768, 3072), (3072, 768))),
                 "normal", grad_scale=1e-3, mom_std=1e-3),
    "c3": Config("c3", "Llama-3-8B-shaped set, 32 x {q, k, v, o, gate, up, down}", "bf16", 2,
                 _layers(32, ((4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096),
                              (14336, 4096), (14336, 4096), (4096, 14336))),
                 "heavy", grad_scale=1e-3),
    # two layers of the c3 shapes: the same kernels on a few GB, for profiler captures
    "c3x2": Config("c3x2", "Llama-3-8B-shaped set, 2 x {q, k, v, o, gate, up, down}", "bf16", 2,
                   _layers(2, ((4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096),
                               (14336, 4096), (14336, 4096), (4096, 14336))),
                   "heavy", grad_scale=1e-3),
    "c4": Config("c4", "embodied/VLA-like heterogeneous set, 2000 matrices", "bf16", 3,
                 _vla_shapes(3), "logscale", logscale=(-5.0, -1.0)),
    "c5": Config("c5", "large-layer stress, 80 x {8192x8192, 28672x8192, 8192x28672}", "bf16", 4,
                 _layers(80, ((8192, 8192), (28672, 8192), (8192, 28672))), "normal",
                 grad_scale=1e-3, budget_gb=16.0),
}


def get(name: str) -> Config:
    return CONFIGS[name]


def _storage(dtype: str):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def make_matrix(cfg: Config, i: int, device="cpu", rows=None, cols=None):
    """(W, grad, mom) of matrix i of ``cfg`` in the storage dtype on ``device``."""
    if rows is None:
        rows, cols = cfg.shapes[i]
    g = torch.Generator(device=device).manual_seed(cfg.seed * 1_000_003 + i)
    kw = dict(generator=g, device=device, dtype=torch.float32)
    w = torch.randn(rows, cols, **kw) * 0.02
    grad = torch.randn(rows, cols, **kw)
    if cfg.grad == "heavy":
        mask = torch.rand(rows, cols, **kw) < 0.01
        grad = torch.where(mask, grad * 100.0, grad)
    if cfg.grad == "logscale":
        lo, hi = cfg.logscale
        u = torch.rand(1, **kw).item()
        grad = grad * (10.0 ** (lo + (hi - lo) * u))
    else:
        grad = grad * cfg.grad_scale
    if cfg.mom_std > 0:
        mom = torch.randn(rows, cols, **kw) * cfg.mom_std
    else:
        mom = torch.zeros(rows, cols, device=device, dtype=torch.float32)
    st = _storage(cfg.dtype)
    return w.to(st), grad.to(st), mom.to(st)


def make_set(cfg: Config, device="cpu", indices=None):
    """Lists (Ws, grads, moms) for the given matrix indices (default: all)."""
    if indices is None:
        indices = range(len(cfg.shapes))
    ws, gs, ms = [], [], []
    for i in indices:
        w, g, m = make_matrix(cfg, i, device)
        ws.append(w)
        gs.append(g)
        ms.append(m)
    return ws, gs, ms


def random_shapes(seed: int, count: int, lo: int = 1, hi: int = 300):
    """Arbitrary (rows, cols) pairs for planner and edge-case tests."""
    g = torch.Generator().manual_seed(seed)
    r = torch.randint(lo, hi + 1, (count,), generator=g)
    c = torch.randint(lo, hi + 1, (count,), generator=g)
    return [(int(a), int(b)) for a, b in zip(r, c)]


def total_elements(cfg: Config) -> int:
    return sum(r * c for r, c in cfg.shapes)


def describe(cfg: Config) -> str:
    return f"{cfg.name}: {cfg.title}; {len(cfg.shapes)} matrices, {total_elements(cfg) / 1e9:.3f} G elements"

