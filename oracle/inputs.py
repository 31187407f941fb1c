"""Adapters from the seeded workload tensors (``workloads``) to the numpy arrays
the oracle takes.  TEST INFRASTRUCTURE ONLY.

bf16 tensors become uint16 bit patterns; fp32 stays fp32; experts are produced
lazily on the CPU, one at a time, so a sampled check needs only the experts its
tokens select.
"""
from __future__ import annotations

from typing import Dict

import numpy as np
import torch

import workloads as wl

from .moe_oracle import LayerParams


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def expert_arrays(w: wl.Workload, e: int) -> Dict[str, np.ndarray]:
    ex = wl.gen_expert(w, e, "cpu")
    out = {}
    for name, t in ex.items():
        out[name] = bf16_bits(t) if t.dtype == torch.bfloat16 else t.numpy()
    return out


class LazyExperts:
    """e -> expert arrays, generated on first use and kept (bounded cache)."""

    def __init__(self, w: wl.Workload, keep: int = 64):
        self.w = w
        self.keep = keep
        self._cache: Dict[int, Dict[str, np.ndarray]] = {}

    def __call__(self, e: int) -> Dict[str, np.ndarray]:
        if e not in self._cache:
            if len(self._cache) >= self.keep:
                self._cache.pop(next(iter(self._cache)))
            self._cache[e] = expert_arrays(self.w, e)
        return self._cache[e]


def layer_params(w: wl.Workload, router=None, latent=None, experts=None) -> LayerParams:
    """Oracle parameters of workload ``w`` (router, experts, latent projections)."""
    if router is None:
        router = wl.gen_router(w)
    W, b = router
    if latent is None and w.L:
        latent = wl.gen_latent(w)
    p = LayerParams(k=w.k, renorm=w.renorm, act_bits=w.act_bits,
                    w_router=W.numpy().astype(np.float64), bias=b.numpy().astype(np.float64),
                    expert=experts if experts is not None else LazyExperts(w), E=w.E, eps=w.eps)
    if latent is not None:
        p.lat_down = bf16_bits(latent["lat_down"])
        p.lat_norm = bf16_bits(latent["lat_norm"])
        p.lat_up = bf16_bits(latent["lat_up"])
    return p


def x_f64(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.float64).numpy()
