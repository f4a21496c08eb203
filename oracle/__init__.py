"""TEST INFRASTRUCTURE -- the fp64 CPU oracle of the multi-LoRA linear layer.

Not part of the product.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` leg of ``bench.py`` may import this
package.  It shares no code with the CUDA path and imports nothing from it.

The arithmetic lives in ``mlora_oracle.c`` (plain per-row fp64 loops); this
module only marshals numpy arrays into it.  Sources, by page:

* ai-infra-kb "M031" multi-LoRA tutorial, §02 (shared base plus per-row
  Down->Up branch, original row order), §03 (group order P/R/Q, low-rank FLOP
  count and the max-rank padded budget), §04 (merge W + scale*Up@Down, valid for
  that adapter only).
* airsota interview card "multi-LoRA serving vs merging", part 三 (per-row
  y_k = x_k W0 + alpha/r ((x_k A) B)); with A = Down^T and B = Up^T this is the
  same map.

Pins: every function is checked by ``tests/test_oracle_pins.py`` against what
the pages print (worked example routing, 32 + 32 = 64 and 128 FLOP) and
against independent mathematics (library matmul on special cases, the merge
identity, rank-padding invariance, permutation equivariance, rank-1 closed
forms, brute force on the worked example).  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mlora_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain -O2, OpenMP over rows)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        lib.oracle_segments.restype = i64
        lib.oracle_segments.argtypes = [i64, p, i32, p, p, p, p, p]
        lib.oracle_forward.restype = None
        lib.oracle_forward.argtypes = [i64, i64, i64, p, p, p, i32, p, p, p, p, p, p, p, i64, p]
        lib.oracle_merge.restype = None
        lib.oracle_merge.argtypes = [i64, i64, p, i32, ctypes.c_double, p, p, p]
        lib.oracle_unmerge.restype = None
        lib.oracle_unmerge.argtypes = [i64, i64, p, i32, ctypes.c_double, p, p, p]
        lib.oracle_lora_flops.restype = None
        lib.oracle_lora_flops.argtypes = [i64, i64, i64, p, i32, p, p, p]
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_threads.argtypes = []
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class OracleAdapter:
    """One loaded slot: Down [r x din], Up [dout x r] (fp64 values), scale."""
    down: np.ndarray
    up: np.ndarray
    scale: float

    @property
    def rank(self) -> int:
        return int(self.down.shape[0])


def _pack(adapters: Sequence[Optional[OracleAdapter]], din: int, dout: int):
    S = len(adapters)
    ranks = np.zeros(max(S, 1), np.int32)
    scales = np.zeros(max(S, 1), np.float64)
    down_off = np.zeros(max(S, 1), np.int64)
    up_off = np.zeros(max(S, 1), np.int64)
    downs, ups = [], []
    dpos = upos = 0
    for s, ad in enumerate(adapters):
        if ad is None:
            continue
        r = ad.rank
        assert ad.down.shape == (r, din) and ad.up.shape == (dout, r)
        ranks[s] = r
        scales[s] = ad.scale
        down_off[s] = dpos
        up_off[s] = upos
        downs.append(np.ascontiguousarray(ad.down, np.float64).ravel())
        ups.append(np.ascontiguousarray(ad.up, np.float64).ravel())
        dpos += r * din
        upos += dout * r
    down_all = np.concatenate(downs) if downs else np.zeros(1)
    up_all = np.concatenate(ups) if ups else np.zeros(1)
    return S, ranks, scales, down_off, up_off, down_all, up_all


def slot_ranks(adapters: Sequence[Optional[OracleAdapter]]) -> np.ndarray:
    return np.array([0 if a is None else a.rank for a in adapters] or [0], np.int32)


def segments(row_adapter: np.ndarray, ranks: np.ndarray, S: Optional[int] = None):
    """Group rows by slot (stable).  Returns (counts[S], offsets[S+1], perm, n_invalid)."""
    lib = _load()
    row_adapter = np.ascontiguousarray(row_adapter, np.int32)
    ranks = np.ascontiguousarray(ranks, np.int32)
    S = len(ranks) if S is None else S
    T = row_adapter.shape[0]
    counts = np.zeros(max(S, 1), np.int32)
    offsets = np.zeros(S + 1, np.int32)
    perm = np.zeros(max(T, 1), np.int32)
    bad = np.zeros(1, np.int64)
    n = lib.oracle_segments(T, _ptr(row_adapter), S, _ptr(ranks), _ptr(counts), _ptr(offsets),
                            _ptr(perm), _ptr(bad))
    return counts[:S].copy(), offsets, perm[:n].copy(), int(bad[0])


def forward(X: np.ndarray, W: np.ndarray, row_adapter: Optional[np.ndarray],
            adapters: Sequence[Optional[OracleAdapter]], rows: Optional[np.ndarray] = None) -> np.ndarray:
    """fp64 multi-LoRA forward for all rows (or only ``rows``), original row order."""
    lib = _load()
    X = np.ascontiguousarray(X, np.float64)
    W = np.ascontiguousarray(W, np.float64)
    T, din = X.shape
    dout = W.shape[0]
    assert W.shape == (dout, din)
    ra = None if row_adapter is None else np.ascontiguousarray(row_adapter, np.int32)
    S, ranks, scales, down_off, up_off, down_all, up_all = _pack(adapters, din, dout)
    if rows is None:
        n_rows = T
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, np.int64)
        n_rows = rows_arr.shape[0]
    Y = np.zeros((max(n_rows, 1), dout), np.float64)
    if n_rows > 0:
        lib.oracle_forward(T, din, dout, _ptr(X), _ptr(W), _ptr(ra), S, _ptr(ranks), _ptr(scales),
                           _ptr(down_off), _ptr(up_off), _ptr(down_all), _ptr(up_all),
                           _ptr(rows_arr), n_rows, _ptr(Y))
    return Y[:n_rows]


def merge(W: np.ndarray, adapter: OracleAdapter) -> np.ndarray:
    """W + scale * Up @ Down in fp64 (valid for rows of this adapter only)."""
    lib = _load()
    W = np.ascontiguousarray(W, np.float64)
    dout, din = W.shape
    out = np.empty_like(W)
    lib.oracle_merge(din, dout, _ptr(W), adapter.rank, float(adapter.scale),
                     _ptr(np.ascontiguousarray(adapter.down, np.float64)),
                     _ptr(np.ascontiguousarray(adapter.up, np.float64)), _ptr(out))
    return out


def forward_modules(X: np.ndarray, W: np.ndarray, row_adapter: np.ndarray, modules, tenants,
                    rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Fused projection of several modules (airsota card "multi-LoRA serving vs
    merging", section 四 item ④): W stacks the modules' weights by rows, module m
    owning output rows modules[m] = (row_offset, rows); tenants[s][m] is slot s's
    adapter of module m (or None).  By definition, the rows of module m are the
    single-module layer over W's rows of m with each slot's module-m adapter; rows
    outside every module are the base product.  ``rows`` selects output rows of the
    batch (all by default), in the given order."""
    X = np.asarray(X, np.float64)
    W = np.asarray(W, np.float64)
    sel = np.arange(X.shape[0]) if rows is None else np.asarray(rows, np.int64)
    Y = X[sel] @ W.T
    for m, (off, n) in enumerate(modules):
        ads = [None if t is None else t[m] for t in tenants]
        Y[:, off:off + n] = forward(X, W[off:off + n], row_adapter, ads, rows=rows)
    return Y


def dequantize(codes: np.ndarray, row_scale: np.ndarray) -> np.ndarray:
    """The logical matrix of an int8 base (M031 §05): W[o, i] = code[o, i] * scale[o]."""
    return np.asarray(codes, np.float64) * np.asarray(row_scale, np.float64)[:, None]


def quantize(W: np.ndarray):
    """Symmetric per-row int8 quantization, decided in fp32 (the precision the kernel
    decides in): scale[o] = max_i |w[o, i]| / 127, code = rint(w / scale[o]) (ties to
    even) clamped to [-127, 127]; an all-zero row gets scale 0 and codes 0."""
    w = np.asarray(W, np.float64).astype(np.float32)
    scale = (np.abs(w).max(axis=1) / np.float32(127)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1))
    codes = np.clip(np.rint(w / safe[:, None]), -127, 127)
    codes = np.where(scale[:, None] > 0, codes, 0).astype(np.int8)
    return codes, scale


def merge_quantized(codes: np.ndarray, row_scale: np.ndarray, adapter: OracleAdapter):
    """The merge on a quantized base (M031 §05): restore W, add scale * Up Down, and
    quantize the merged matrix again -- never the update added to the codes."""
    return quantize(merge(dequantize(codes, row_scale), adapter))


NF4_BLOCK = 64   # input columns that share one absmax scale


def nf4_unpack(packed: np.ndarray) -> np.ndarray:
    """4-bit codes [dout x din] from bytes [dout x din/2]: column 2m is the low nibble of
    byte m, column 2m + 1 the high nibble."""
    packed = np.asarray(packed, np.uint8)
    codes = np.empty((packed.shape[0], 2 * packed.shape[1]), np.uint8)
    codes[:, 0::2] = packed & 15
    codes[:, 1::2] = packed >> 4
    return codes


def nf4_pack(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def nf4_dequantize(packed: np.ndarray, absmax: np.ndarray, codebook: np.ndarray) -> np.ndarray:
    """The logical matrix of an NF4 base (M031 §05: W restored by scale and codebook):
    W[o, i] = codebook[code[o, i]] * absmax[i // 64, o], in fp64."""
    codes = nf4_unpack(packed)
    cb = np.asarray(codebook, np.float32).astype(np.float64)
    scale = np.repeat(np.asarray(absmax, np.float32).astype(np.float64).T, NF4_BLOCK, axis=1)
    return cb[codes] * scale


def nf4_quantize(W: np.ndarray, codebook: np.ndarray):
    """NF4 quantization, decided in fp32 (the precision the kernel decides in): per row
    and block of 64 columns, absmax = max |w|; each w / absmax (fp32 division) takes the
    code of the nearest codebook value (fp32 distances, ties to the lower code); an
    all-zero block gets absmax 0 and the code of the value nearest 0.  Returns packed
    codes [dout x din/2] and absmax [din/64 x dout]."""
    w = np.asarray(W, np.float64).astype(np.float32)
    dout, din = w.shape
    blocks = w.reshape(dout, din // NF4_BLOCK, NF4_BLOCK)
    absmax = np.abs(blocks).max(axis=2).astype(np.float32)                    # [dout, nb]
    safe = np.where(absmax > 0, absmax, np.float32(1))
    v = np.where(absmax[:, :, None] > 0, blocks / safe[:, :, None], np.float32(0)).astype(np.float32)
    cb = np.asarray(codebook, np.float32)
    dist = np.abs(v[..., None] - cb).astype(np.float32)                        # fp32 distances
    codes = np.argmin(dist, axis=-1).astype(np.uint8).reshape(dout, din)       # first minimum wins
    return nf4_pack(codes), np.ascontiguousarray(absmax.T)


def nf4_restore_f32(packed: np.ndarray, absmax: np.ndarray, codebook: np.ndarray) -> np.ndarray:
    """The restored values as fp32 products codebook[code] * absmax (the merge's input)."""
    codes = nf4_unpack(packed)
    cb = np.asarray(codebook, np.float32)
    scale = np.repeat(np.asarray(absmax, np.float32).T, NF4_BLOCK, axis=1)
    return (cb[codes] * scale).astype(np.float32)


def nf4_merge(packed: np.ndarray, absmax: np.ndarray, codebook: np.ndarray, adapter: OracleAdapter):
    """The merge on an NF4 base (M031 §05): restore W, add scale * Up Down, quantize the
    merged matrix again -- never the update added to the codes.  The merged value is
    the fp64 sum of the fp32 restored value and the update, rounded to fp32."""
    merged = merge(nf4_restore_f32(packed, absmax, codebook).astype(np.float64), adapter)
    return nf4_quantize(merged.astype(np.float32), codebook)


def unmerge(W: np.ndarray, adapter: OracleAdapter) -> np.ndarray:
    """W - scale * Up @ Down in fp64: the un-merge that switches a merged weight back
    (airsota card "multi-LoRA serving vs merging", section 四 item ③)."""
    lib = _load()
    W = np.ascontiguousarray(W, np.float64)
    dout, din = W.shape
    out = np.empty_like(W)
    lib.oracle_unmerge(din, dout, _ptr(W), adapter.rank, float(adapter.scale),
                       _ptr(np.ascontiguousarray(adapter.down, np.float64)),
                       _ptr(np.ascontiguousarray(adapter.up, np.float64)), _ptr(out))
    return out


def lora_flops(row_adapter: np.ndarray, ranks: np.ndarray, din: int, dout: int):
    """(exact grouped low-rank FLOPs, max-rank padded budget)."""
    lib = _load()
    ra = np.ascontiguousarray(row_adapter, np.int32)
    ranks = np.ascontiguousarray(ranks, np.int32)
    e = np.zeros(1, np.int64)
    p = np.zeros(1, np.int64)
    lib.oracle_lora_flops(ra.shape[0], din, dout, _ptr(ra), len(ranks), _ptr(ranks), _ptr(e), _ptr(p))
    return int(e[0]), int(p[0])


def threads() -> int:
    """OpenMP threads the oracle's row loop uses."""
    return int(_load().oracle_threads())
