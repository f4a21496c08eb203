"""Moves seeded workloads onto the GPU and runs them through the C ABI binding.

Test infrastructure: torch allocates device memory and provides the stream; the
forward itself is one ``mlora_forward`` call into libmlora.so.
"""
from __future__ import annotations

import numpy as np

import workloads as wl
from heterogeneous_lora_gemm_gb300.torch_io import make_pool, to_device, to_f64  # noqa: F401


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
