"""Moves seeded workloads onto the GPU and runs them through the C ABI binding.

Test infrastructure: torch allocates device memory and provides the stream; the
forward itself is one ``mlora_forward`` call into libmlora.so.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

import workloads as wl


def to_device(payload: np.ndarray, dtype: str, device="cuda"):
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(payload).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(payload, np.float32))
    return t.to(device)


def to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def make_pool(layer: wl.LayerData, max_tokens: Optional[int] = None, rank_budget: Optional[int] = None,
              max_rank: Optional[int] = None, host_sources: bool = False):
    from heterogeneous_lora_gemm_gb300 import Pool
    budget = sum((a.rank + 7) // 8 * 8 for a in layer.adapters) if rank_budget is None else rank_budget
    pool = Pool(layer.max_slots, budget, max_rank or layer.max_rank, layer.din, layer.dout, layer.dtype,
                max_tokens or max(layer.T, 1))
    for a in layer.adapters:
        if host_sources:
            import torch
            down = to_device(a.down, layer.dtype, "cpu")
            up = to_device(a.up, layer.dtype, "cpu")
        else:
            down = to_device(a.down, layer.dtype)
            up = to_device(a.up, layer.dtype)
        pool.load(a.slot, down, up, a.scale)
    return pool


def upload(layer: wl.LayerData):
    import torch
    X = to_device(layer.X, layer.dtype)
    W = to_device(layer.W, layer.dtype)
    ra = torch.from_numpy(layer.row_adapter.astype(np.int32)).cuda()
    tdt = torch.bfloat16 if layer.dtype == "bf16" else torch.float32
    Y = torch.full((layer.T, layer.dout), float("nan"), dtype=tdt, device="cuda")
    return X, W, ra, Y


def run_layer(layer: wl.LayerData, pool=None, with_row_adapter: bool = True,
              check_status: bool = True) -> np.ndarray:
    """Y of one forward, as fp64 numpy; by default also requires a clean device status."""
    import torch
    from heterogeneous_lora_gemm_gb300 import mlora
    own = pool is None
    if own:
        pool = make_pool(layer)
    X, W, ra, Y = upload(layer)
    pool.forward(X, W, ra if with_row_adapter else None, Y)
    torch.cuda.synchronize()
    if check_status:
        st = pool.status()
        assert st == mlora.MLORA_OK, f"device status {st}: {mlora.status_string(st)}"
    out = to_f64(Y)
    if own:
        pool.close()
    return out
