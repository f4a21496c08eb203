"""Moves seeded workloads (numpy payloads, see workloads.py) into torch device
tensors and adapter pools.

Marshalling only: bf16 bit patterns are reinterpreted, never converted, and every
step of the layer runs in libmlora.so.  Used by the benchmark and the tests.
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def to_device(payload: np.ndarray, dtype: str, device="cuda"):
    """A bf16 payload (uint16 bit patterns) or fp32 array as a torch tensor on `device`."""
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(payload).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(payload, np.float32))
    return t.to(device)


def to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def make_pool(layer, max_tokens: Optional[int] = None, rank_budget: Optional[int] = None,
              max_rank: Optional[int] = None, host_sources: bool = False):
    """A pool shaped for `layer` (workloads.LayerData) with its adapters loaded in their slots."""
    from .mlora import Pool
    budget = sum((a.rank + 7) // 8 * 8 for a in layer.adapters) if rank_budget is None else rank_budget
    pool = Pool(layer.max_slots, budget, max_rank or layer.max_rank, layer.din, layer.dout, layer.dtype,
                max_tokens or max(layer.T, 1))
    dev = "cpu" if host_sources else "cuda"
    for a in layer.adapters:
        pool.load(a.slot, to_device(a.down, layer.dtype, dev), to_device(a.up, layer.dtype, dev), a.scale)
    return pool


def make_fused_pool(din: int, modules, tenants, T: int):
    """A bf16 pool for a fused projection (modules stacked by rows) with each slot's
    per-module adapters loaded as one combined adapter.  `tenants[s][m]` is None or
    (down, up, scale) of module m, torch tensors (host or device)."""
    from .mlora import Pool
    dout = sum(n for _, n in modules)
    rank_of = [sum(-(-int(t[0].shape[0]) // 16) * 16 for t in row if t is not None) for row in tenants]
    budget = sum(rank_of)
    pool = Pool(len(tenants), max(budget, 0), max(rank_of + [16]), din, dout, "bf16", T)
    for s_, row in enumerate(tenants):
        mods = []
        for (off, n), t in zip(modules, row):
            mods.append((off, n, t[0], t[1], t[2]) if t is not None else (off, n, None, None, 0.0))
        pool.load_modules(s_, mods)
    return pool
