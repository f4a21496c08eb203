"""CPU checks of the C ABI boundary: the library loads, exports every symbol the
header declares, rejects bad arguments before touching CUDA, and its arena
allocator places, frees and compacts blocks as documented."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mlora.h")


@pytest.fixture(scope="module")
def lib():
    from heterogeneous_lora_gemm_gb300 import build as b
    b.build()
    from heterogeneous_lora_gemm_gb300 import mlora
    return mlora


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mlora_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(lib):
    names = declared_functions()
    assert "mlora_forward" in names and "mlora_pool_create" in names and "mlora_merge" in names
    L = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    # the binding covers every declared entry point under the same name
    assert set(names) <= set(lib._SIGNATURES)


def test_library_has_no_libcuda_link_dependency(lib):
    import subprocess
    out = subprocess.run(["ldd", lib.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def test_status_strings(lib):
    for code in range(10):
        assert lib.status_string(code)
    assert lib.status_string(0) == "ok"


@pytest.mark.parametrize("args,code", [
    ((-1, 16, 16, 64, 64, 1, 8), 1),
    ((4097, 16, 16, 64, 64, 1, 8), 1),
    ((4, -8, 16, 64, 64, 1, 8), 1),
    ((4, 16, 0, 64, 64, 1, 8), 1),
    ((4, 16, 300, 64, 64, 1, 8), 1),
    ((4, 16, 16, 0, 64, 1, 8), 1),
    ((4, 16, 16, 64, 64, 1, 0), 1),
    ((4, 16, 16, 64, 64, 7, 8), 1),
    ((4, 16, 16, 60, 64, 1, 8), 8),      # bf16 needs din % 8 == 0
])
def test_pool_create_rejects_bad_arguments_before_cuda(lib, args, code):
    h = ctypes.c_void_p(123)
    s = lib.lib().mlora_pool_create(*args, ctypes.byref(h))
    assert s == code and h.value is None
    assert lib.last_error()


def test_null_pool_is_invalid_arg(lib):
    L = lib.lib()
    assert L.mlora_forward(None, None, None, None, 4, None, None) == 1
    assert L.mlora_merge(None, None, 0, None) == 1
    assert L.mlora_load_adapter(None, 0, None, None, 8, 1.0) == 1
    assert L.mlora_unload_adapter(None, 0) == 1
    assert L.mlora_pool_status(None, None) == 1
    assert L.mlora_pool_destroy(None) == 0


class ArenaModel:
    """Plain model of the documented placement rule: first fit at multiples of 8."""

    def __init__(self, units):
        self.units = units
        self.blocks = {}     # id -> (off, size)

    def alloc(self, i, n):
        size = (n + 7) // 8 * 8
        cur = 0
        for off, sz in sorted(self.blocks.values()):
            if off - cur >= size:
                break
            cur = off + sz
        if cur + size > self.units:
            return -1
        self.blocks[i] = (cur, size)
        return cur

    def free(self, i):
        return 0 if self.blocks.pop(i, None) else -1

    def compact(self):
        moves, cur = [], 0
        for i, (off, sz) in sorted(self.blocks.items(), key=lambda kv: kv[1][0]):
            if off != cur:
                moves.append((i, off, cur))
            self.blocks[i] = (cur, sz)
            cur += sz
        return moves


def test_arena_matches_model(lib):
    L = lib.lib()
    rng = np.random.default_rng(0)
    for trial in range(20):
        units = int(rng.integers(1, 40)) * 8
        a = L.mlora_arena_new(units)
        m = ArenaModel(units)
        for step in range(200):
            op = rng.integers(0, 10)
            i = int(rng.integers(0, 12))
            if op < 6:
                n = int(rng.choice([1, 2, 8, 16, 24, 64]))
                if i in m.blocks:
                    assert L.mlora_arena_alloc(a, i, n) == -1
                    continue
                assert L.mlora_arena_alloc(a, i, n) == m.alloc(i, n)
            elif op < 9:
                assert L.mlora_arena_free(a, i) == m.free(i)
            else:
                buf = (ctypes.c_int32 * 300)()
                n = L.mlora_arena_compact(a, buf, 100)
                want = m.compact()
                assert n == len(want)
                assert [tuple(buf[3 * k:3 * k + 3]) for k in range(n)] == want
            assert L.mlora_arena_used(a) == sum(sz for _, sz in m.blocks.values())
        L.mlora_arena_delete(a)


def test_arena_compaction_recovers_fragmented_space(lib):
    L = lib.lib()
    a = L.mlora_arena_new(64)
    for i in range(8):
        assert L.mlora_arena_alloc(a, i, 8) == 8 * i
    for i in (1, 3, 5, 7):
        assert L.mlora_arena_free(a, i) == 0
    assert L.mlora_arena_largest_hole(a) == 8
    assert L.mlora_arena_alloc(a, 20, 32) == -1
    buf = (ctypes.c_int32 * 30)()
    assert L.mlora_arena_compact(a, buf, 10) == 3
    assert L.mlora_arena_largest_hole(a) == 32
    assert L.mlora_arena_alloc(a, 20, 32) == 32
    L.mlora_arena_delete(a)


def test_arena_rename_keeps_the_block_in_place(lib):
    """An evicted adapter's block is renamed to a quarantine id, not freed: a new
    allocation must land elsewhere until the quarantine is released."""
    L = lib.lib()
    a = L.mlora_arena_new(48)
    assert L.mlora_arena_alloc(a, 0, 16) == 0
    assert L.mlora_arena_alloc(a, 1, 16) == 16
    assert L.mlora_arena_rename(a, 0, 1000) == 0
    assert L.mlora_arena_rename(a, 0, 1001) == -1      # 0 holds nothing now
    assert L.mlora_arena_rename(a, 1, 1000) == -1      # 1000 holds a block already
    assert L.mlora_arena_used(a) == 32
    assert L.mlora_arena_alloc(a, 0, 16) == 32         # not the quarantined units 0..15
    assert L.mlora_arena_alloc(a, 2, 8) == -1
    assert L.mlora_arena_free(a, 1000) == 0
    assert L.mlora_arena_alloc(a, 2, 8) == 0
    L.mlora_arena_delete(a)
