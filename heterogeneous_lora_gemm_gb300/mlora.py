"""ctypes binding of libmlora.so -- argument marshalling only.

The functions below carry the names and signatures of include/mlora.h; every
step of the forward, the segment builder and the merge runs in the library's
CUDA kernels.  ``Pool`` wraps a pool handle for callers that hold torch tensors
(``tensor.data_ptr()`` and the current torch stream are passed through).

The library must have been built (``__graft_entry__.build()`` or
``python -m heterogeneous_lora_gemm_gb300.build``); importing a missing library
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmlora.so")

MLORA_OK = 0
MLORA_ERR_INVALID_ARG = 1
MLORA_ERR_BAD_SLOT = 2
MLORA_ERR_RANK = 3
MLORA_ERR_NOT_LOADED = 4
MLORA_ERR_OOM = 5
MLORA_ERR_CUDA = 6
MLORA_ERR_DEVICE_ROW = 7
MLORA_ERR_UNSUPPORTED = 8
MLORA_ERR_DEVICE_TIMEOUT = 9
MLORA_F32 = 0
MLORA_BF16 = 1


class MloraError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {status_string(status)} [{status}] {detail}")
        self.status = status


class PoolInfo(ctypes.Structure):
    _fields_ = [("din", ctypes.c_int32), ("dout", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("max_slots", ctypes.c_int32), ("max_rank", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("rank_units", ctypes.c_int32), ("rank_units_used", ctypes.c_int32), ("loaded", ctypes.c_int32),
                ("device", ctypes.c_int32), ("arena_bytes", ctypes.c_uint64), ("table_bytes", ctypes.c_uint64),
                ("workspace_bytes", ctypes.c_uint64), ("ext_run_stride", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int

# name -> (restype, argtypes), in header order
_SIGNATURES = {
    "mlora_status_string": (ctypes.c_char_p, [_I]),
    "mlora_last_error": (ctypes.c_char_p, []),
    "mlora_pool_create": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_P)]),
    "mlora_pool_destroy": (_I, [_P]),
    "mlora_load_adapter": (_I, [_P, _I, _P, _P, _I, ctypes.c_float]),
    "mlora_unload_adapter": (_I, [_P, _I]),
    "mlora_load_adapter_modules": (_I, [_P, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_P),
                                        ctypes.POINTER(_P), ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_float)]),
    "mlora_adapter_version": (_I, [_P, _I, ctypes.POINTER(ctypes.c_uint64)]),
    "mlora_host_adapter_add": (_I, [_P, _I, _P, _P, _I, ctypes.c_float]),
    "mlora_host_adapter_remove": (_I, [_P, _I]),
    "mlora_prefetch": (_I, [_P, _I, _I, _P]),
    "mlora_forward": (_I, [_P, _P, _P, _P, _I, _P, _P]),
    "mlora_merge": (_I, [_P, _P, _I, _P]),
    "mlora_unmerge": (_I, [_P, _P, _I, _P]),
    "mlora_dequantize": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "mlora_forward_quantized": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P]),
    "mlora_merge_quantized": (_I, [_P, _P, _P, _I, _P]),
    "mlora_dequantize_nf4": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "mlora_forward_nf4": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P, _P]),
    "mlora_merge_nf4": (_I, [_P, _P, _P, _P, _I, _P]),
    "mlora_pool_status": (_I, [_P, _P]),
    "mlora_pool_info": (_I, [_P, ctypes.POINTER(PoolInfo)]),
    "mlora_debug_segments": (_I, [_P, _P, _I, _P, _P, _P]),
    "mlora_debug_last_segments": (_I, [_P, _I, _P, _P, _P]),
    "mlora_profile_stamps": (_I, [_P, _P, _I]),
    "mlora_project_noalloc": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "mlora_project_noalloc_status": (_I, [_P]),
    "mlora_debug_noalloc_expire_wait": (_I, [ctypes.c_longlong, _P]),
    "mlora_arena_new": (_P, [_I]),
    "mlora_arena_delete": (None, [_P]),
    "mlora_arena_alloc": (_I, [_P, _I, _I]),
    "mlora_arena_free": (_I, [_P, _I]),
    "mlora_arena_rename": (_I, [_P, _I, _I]),
    "mlora_arena_compact": (_I, [_P, _P, _I]),
    "mlora_arena_used": (_I, [_P]),
    "mlora_arena_largest_hole": (_I, [_P]),
}


def lib() -> ctypes.CDLL:
    """The loaded libmlora.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().mlora_status_string(status).decode()


def last_error() -> str:
    return lib().mlora_last_error().decode()


def check(status: int, where: str) -> None:
    if status != MLORA_OK:
        raise MloraError(status, where, last_error())


# ---- the C entry points, same names -------------------------------------- #
def mlora_pool_create(max_slots: int, rank_budget: int, max_rank: int, din: int, dout: int, dtype: int,
                      max_tokens: int) -> int:
    h = _P()
    check(lib().mlora_pool_create(max_slots, rank_budget, max_rank, din, dout, dtype, max_tokens, ctypes.byref(h)),
          "mlora_pool_create")
    return h.value


def mlora_pool_destroy(pool: int) -> None:
    check(lib().mlora_pool_destroy(pool), "mlora_pool_destroy")


def mlora_load_adapter(pool: int, slot: int, down_ptr: int, up_ptr: int, rank: int, scale: float) -> None:
    check(lib().mlora_load_adapter(pool, slot, down_ptr, up_ptr, rank, scale), "mlora_load_adapter")


def mlora_unload_adapter(pool: int, slot: int) -> None:
    check(lib().mlora_unload_adapter(pool, slot), "mlora_unload_adapter")


def mlora_adapter_version(pool: int, slot: int) -> int:
    v = ctypes.c_uint64()
    check(lib().mlora_adapter_version(pool, slot, ctypes.byref(v)), "mlora_adapter_version")
    return int(v.value)


def mlora_forward(pool: int, X_ptr: int, W_ptr: int, row_adapter_ptr: Optional[int], T: int, Y_ptr: int,
                  stream: int) -> None:
    check(lib().mlora_forward(pool, X_ptr, W_ptr, row_adapter_ptr or None, T, Y_ptr, stream or None),
          "mlora_forward")


def mlora_load_adapter_modules(pool: int, slot: int, row_offset, rows, down_ptrs, up_ptrs, ranks, scales) -> None:
    """One tenant's adapters of several row ranges (modules) of a fused projection; see include/mlora.h."""
    n = len(ranks)
    arr = lambda t, v: (t * n)(*v)   # noqa: E731
    check(lib().mlora_load_adapter_modules(pool, slot, n, arr(_I, row_offset), arr(_I, rows),
                                           arr(_P, [p or None for p in down_ptrs]),
                                           arr(_P, [p or None for p in up_ptrs]), arr(_I, ranks),
                                           arr(ctypes.c_float, scales)), "mlora_load_adapter_modules")


def mlora_host_adapter_add(pool: int, id_: int, down_ptr: int, up_ptr: int, rank: int, scale: float) -> None:
    check(lib().mlora_host_adapter_add(pool, id_, down_ptr, up_ptr, rank, scale), "mlora_host_adapter_add")


def mlora_host_adapter_remove(pool: int, id_: int) -> None:
    check(lib().mlora_host_adapter_remove(pool, id_), "mlora_host_adapter_remove")


def mlora_prefetch(pool: int, slot: int, id_: int, stream: int) -> None:
    check(lib().mlora_prefetch(pool, slot, id_, stream or None), "mlora_prefetch")


def mlora_merge(pool: int, W_ptr: int, slot: int, stream: int) -> None:
    check(lib().mlora_merge(pool, W_ptr, slot, stream or None), "mlora_merge")


def mlora_dequantize(Wq_ptr: int, scale_ptr: int, dout: int, din: int, dtype: int, W_ptr: int, stream: int) -> None:
    check(lib().mlora_dequantize(Wq_ptr, scale_ptr, dout, din, dtype, W_ptr, stream or None), "mlora_dequantize")


def mlora_unmerge(pool: int, W_ptr: int, slot: int, stream: int) -> None:
    check(lib().mlora_unmerge(pool, W_ptr, slot, stream or None), "mlora_unmerge")


def mlora_pool_status(pool: int, stream: int) -> int:
    """Returns MLORA_OK, MLORA_ERR_DEVICE_ROW or MLORA_ERR_DEVICE_TIMEOUT; raises on CUDA errors."""
    s = lib().mlora_pool_status(pool, stream or None)
    if s not in (MLORA_OK, MLORA_ERR_DEVICE_ROW, MLORA_ERR_DEVICE_TIMEOUT):
        check(s, "mlora_pool_status")
    return s


def mlora_pool_info(pool: int) -> PoolInfo:
    info = PoolInfo()
    check(lib().mlora_pool_info(pool, ctypes.byref(info)), "mlora_pool_info")
    return info


def mlora_debug_segments(pool: int, row_adapter_ptr: Optional[int], T: int, perm_ptr: int, offsets_ptr: int,
                         stream: int) -> None:
    check(lib().mlora_debug_segments(pool, row_adapter_ptr or None, T, perm_ptr, offsets_ptr, stream or None),
          "mlora_debug_segments")


def mlora_debug_last_segments(pool: int, T: int, perm_ptr: int, offsets_ptr: int, stream: int) -> None:
    check(lib().mlora_debug_last_segments(pool, T, perm_ptr or None, offsets_ptr, stream or None),
          "mlora_debug_last_segments")


def mlora_profile_stamps(pool: int, records_ptr: int, cap: int) -> None:
    """records_ptr: device buffer of 4 + 4 cap uint64 words (0 / cap 0 turns recording off)."""
    check(lib().mlora_profile_stamps(pool, records_ptr or None, cap), "mlora_profile_stamps")


def mlora_project_noalloc(X_ptr: int, W_ptr: int, T: int, din: int, dout: int, Y_ptr: int, stream: int) -> None:
    """Y = X W^T (bf16, T <= 256) without any device allocation; see include/mlora.h."""
    check(lib().mlora_project_noalloc(X_ptr, W_ptr, T, din, dout, Y_ptr, stream or None), "mlora_project_noalloc")


def mlora_project_noalloc_status(stream: int) -> int:
    """Reads and clears the allocation-free calls' status word: MLORA_OK or
    MLORA_ERR_DEVICE_TIMEOUT; raises on other errors."""
    s = int(lib().mlora_project_noalloc_status(stream or None))
    if s not in (MLORA_OK, MLORA_ERR_DEVICE_TIMEOUT):
        check(s, "mlora_project_noalloc_status")
    return s


def mlora_debug_noalloc_expire_wait(cycles: int, stream: int) -> None:
    check(lib().mlora_debug_noalloc_expire_wait(int(cycles), stream or None), "mlora_debug_noalloc_expire_wait")


def _codebook(values) -> "ctypes.Array":
    """16 floats as a C array (host memory, copied by the callee)."""
    vals = [float(v) for v in values]
    if len(vals) != 16:
        raise ValueError("a codebook has 16 values")
    return (ctypes.c_float * 16)(*vals)


def mlora_dequantize_nf4(codes_ptr: int, absmax_ptr: int, codebook, dout: int, din: int, dtype: int, W_ptr: int,
                         stream: int) -> None:
    check(lib().mlora_dequantize_nf4(codes_ptr, absmax_ptr, _codebook(codebook), dout, din, dtype, W_ptr,
                                     stream or None), "mlora_dequantize_nf4")


# ---- torch-facing convenience ------------------------------------------- #
def _stream_handle(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


class Pool:
    """A pool handle driven with torch tensors (device memory and streams only)."""

    def __init__(self, max_slots: int, rank_budget: int, max_rank: int, din: int, dout: int, dtype: str,
                 max_tokens: int):
        self.dtype = dtype
        self.din, self.dout = din, dout
        self.max_slots = max_slots
        code = MLORA_BF16 if dtype == "bf16" else MLORA_F32
        self.handle = mlora_pool_create(max_slots, rank_budget, max_rank, din, dout, code, max_tokens)

    def close(self) -> None:
        if getattr(self, "handle", None):
            mlora_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load(self, slot: int, down, up, scale: float) -> None:
        """down [r x din], up [dout x r]: torch tensors (host or device) of the pool dtype."""
        down = down.contiguous()
        up = up.contiguous()
        mlora_load_adapter(self.handle, slot, down.data_ptr(), up.data_ptr(), int(down.shape[0]), float(scale))

    def unload(self, slot: int) -> None:
        mlora_unload_adapter(self.handle, slot)

    def load_modules(self, slot: int, modules) -> None:
        """modules: list of (row_offset, rows, down, up, scale) with torch tensors, or
        (row_offset, rows, None, None, 0.0) for a module the tenant does not adapt."""
        keep = [(d.contiguous(), u.contiguous()) if d is not None else (None, None) for _, _, d, u, _ in modules]
        mlora_load_adapter_modules(self.handle, slot, [m[0] for m in modules], [m[1] for m in modules],
                                   [d.data_ptr() if d is not None else 0 for d, _ in keep],
                                   [u.data_ptr() if u is not None else 0 for _, u in keep],
                                   [int(d.shape[0]) if d is not None else 0 for d, _ in keep],
                                   [float(m[4]) for m in modules])

    def host_add(self, id_: int, down, up, scale: float) -> None:
        """Copies an adapter (torch tensors, host or device) into the pool's pinned host tier."""
        down = down.contiguous()
        up = up.contiguous()
        mlora_host_adapter_add(self.handle, id_, down.data_ptr(), up.data_ptr(), int(down.shape[0]), float(scale))

    def host_remove(self, id_: int) -> None:
        mlora_host_adapter_remove(self.handle, id_)

    def prefetch(self, slot: int, id_: int, stream=None) -> None:
        mlora_prefetch(self.handle, slot, id_, _stream_handle(stream))

    def version(self, slot: int) -> int:
        return mlora_adapter_version(self.handle, slot)

    def forward(self, X, W, row_adapter, Y, stream=None) -> None:
        ra = None if row_adapter is None else row_adapter.data_ptr()
        mlora_forward(self.handle, X.data_ptr(), W.data_ptr(), ra, int(X.shape[0]), Y.data_ptr(),
                      _stream_handle(stream))

    def merge(self, W, slot: int, stream=None) -> None:
        mlora_merge(self.handle, W.data_ptr(), slot, _stream_handle(stream))

    def unmerge(self, W, slot: int, stream=None) -> None:
        mlora_unmerge(self.handle, W.data_ptr(), slot, _stream_handle(stream))

    def forward_quantized(self, X, Wq, row_scale, W_scratch, row_adapter, Y, stream=None) -> None:
        """The dynamic branch over an int8 base (codes Wq [dout x din] int8, row_scale [dout] fp32)."""
        ra = None if row_adapter is None else row_adapter.data_ptr()
        check(lib().mlora_forward_quantized(self.handle, X.data_ptr(), Wq.data_ptr(), row_scale.data_ptr(),
                                            W_scratch.data_ptr(), ra, int(X.shape[0]), Y.data_ptr(),
                                            _stream_handle(stream)), "mlora_forward_quantized")

    def merge_quantized(self, Wq, row_scale, slot: int, stream=None) -> None:
        check(lib().mlora_merge_quantized(self.handle, Wq.data_ptr(), row_scale.data_ptr(), slot,
                                          _stream_handle(stream)), "mlora_merge_quantized")

    def forward_nf4(self, X, codes, absmax, codebook, W_scratch, row_adapter, Y, stream=None) -> None:
        """The dynamic branch over an NF4 base (codes uint8 [dout x din/2], absmax fp32
        [din/64 x dout], codebook: 16 host floats)."""
        ra = None if row_adapter is None else row_adapter.data_ptr()
        cb = _codebook(codebook)
        check(lib().mlora_forward_nf4(self.handle, X.data_ptr(), codes.data_ptr(), absmax.data_ptr(), cb,
                                      None if W_scratch is None else W_scratch.data_ptr(), ra, int(X.shape[0]),
                                      Y.data_ptr(), _stream_handle(stream)), "mlora_forward_nf4")

    def merge_nf4(self, codes, absmax, codebook, slot: int, stream=None) -> None:
        check(lib().mlora_merge_nf4(self.handle, codes.data_ptr(), absmax.data_ptr(), _codebook(codebook), slot,
                                    _stream_handle(stream)), "mlora_merge_nf4")

    def status(self, stream=None) -> int:
        return mlora_pool_status(self.handle, _stream_handle(stream))

    def info(self) -> PoolInfo:
        return mlora_pool_info(self.handle)

    def profile_stamps(self, records, cap: int) -> None:
        """records: a device torch tensor of >= 4 + 4 cap int64/uint64 words; cap 0 turns recording off."""
        mlora_profile_stamps(self.handle, records.data_ptr() if cap > 0 else 0, cap)

    def last_segments(self, perm, offsets, stream=None) -> None:
        """The segments the last forward with a row map built (perm [T], offsets [max_slots + 1], device int32)."""
        mlora_debug_last_segments(self.handle, int(perm.shape[0]), perm.data_ptr(), offsets.data_ptr(),
                                  _stream_handle(stream))

    def segments(self, row_adapter, perm, offsets, stream=None) -> None:
        ra = None if row_adapter is None else row_adapter.data_ptr()
        mlora_debug_segments(self.handle, ra, int(perm.shape[0]), perm.data_ptr(), offsets.data_ptr(),
                             _stream_handle(stream))
