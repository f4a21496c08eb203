"""Plants plausible mistakes in a copy of the oracle (on the CPU) and checks that
the pins of tests/test_oracle_pins.py catch every one of them.

Each mutant is the oracle's C source with one edit (a dropped term, a wrong
sign or index, a transposed operand, an unstable group order), compiled into a
temporary library and swapped in for the duration of the pin run.  The oracle's
numpy functions get the same treatment: one edit to a function's source, run in
the oracle module's namespace and swapped in for the pins.
"""
import ctypes
import inspect
import os
import subprocess
import tempfile
import textwrap

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mlora_oracle.c")

MUTANTS = {
    "scale dropped": ("y[o] += scales[a] * acc;", "y[o] += acc;"),
    "delta sign flipped": ("y[o] += scales[a] * acc;", "y[o] -= scales[a] * acc;"),
    "Up transposed": ("acc += u[k] * v[k];", "acc += up[(int64_t)k * dout + o] * v[k];"),
    "Down row stride": ("const double* d = down + (int64_t)k * din;", "const double* d = down + k;"),
    "base uses W transposed": ("const double* w = W + o * din;", "const double* w = W + o;"),
    "groups not stable": ("if (a->row != b->row) return a->row < b->row ? -1 : 1;",
                          "if (a->row != b->row) return a->row > b->row ? -1 : 1;"),
    "merge drops scale": ("W_out[o * din + i] = W[o * din + i] + scale * acc;",
                          "W_out[o * din + i] = W[o * din + i] + acc;"),
    "merge transposed": ("acc += up[o * rank + k] * down[(int64_t)k * din + i];",
                         "acc += up[o * rank + k] * down[(int64_t)k + i * rank];"),
    "unmerge adds": ("W_out[o * din + i] = W[o * din + i] - scale * acc;",
                     "W_out[o * din + i] = W[o * din + i] + scale * acc;"),
    "unmerge Down transposed": ("acc += u[k] * down[(int64_t)k * din + i];",
                                "acc += u[k] * down[(int64_t)k + i * rank];"),
    "flops count din only": ("e += 2 * (int64_t)ranks[a] * (din + dout);", "e += 2 * (int64_t)ranks[a] * din;"),
    "padded budget uses valid rows": ("*padded = 2 * T * (int64_t)r_max * (din + dout);",
                                      "*padded = e / (r_max > 0 ? 1 : 1);"),
}

PIN_TESTS = [
    pins.test_worked_example_group_order,
    pins.test_worked_example_flops,
    pins.test_worked_example_writeback_rows,
    pins.test_worked_example_brute_force_exact,
    pins.test_rows_without_adapter_equal_library_matmul,
    lambda: pins.test_single_adapter_batch_equals_merged_weight(2),
    pins.test_merge_matches_library,
    pins.test_unmerge_subtracts_the_update,
    pins.test_unmerge_after_merge_restores_only_with_the_same_adapter,
    pins.test_rank_padding_leaves_output_unchanged,
    pins.test_rank1_unit_adapter_closed_form,
    pins.test_segments_match_sorted_definition,
]


def _build_mutant(name, tmpdir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site of {name!r} not found exactly once"
    path = os.path.join(tmpdir, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(tmpdir, "libmutant.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", lib, path])
    return lib


def _run_pins_with(lib_path):
    saved_lib, saved_path = oracle._lib, oracle._LIB_PATH
    oracle._lib = None
    oracle._LIB_PATH = lib_path
    try:
        failures = 0
        for t in PIN_TESTS:
            try:
                t()
            except AssertionError:
                failures += 1
        return failures
    finally:
        oracle._lib = saved_lib
        oracle._LIB_PATH = saved_path


def test_pins_pass_on_the_real_oracle():
    assert _run_pins_with(oracle.build()) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_planted_mistake_is_caught(name, monkeypatch):
    monkeypatch.setattr(oracle, "build", lambda force=False: oracle._LIB_PATH)
    with tempfile.TemporaryDirectory() as d:
        lib = _build_mutant(name, d)
        assert _run_pins_with(lib) > 0, f"no pin caught the mutant {name!r}"


# numpy parts of the oracle: (function, text replaced, replacement)
PY_MUTANTS = {
    "quantize ties away from zero": ("quantize", "np.rint(w / safe[:, None])",
                                     "np.trunc(w / safe[:, None] + np.copysign(0.5, w))"),
    "quantize scale from 128 levels": ("quantize", "np.float32(127)", "np.float32(128)"),
    "quantized merge adds to the codes": ("merge_quantized", "quantize(merge(dequantize(codes, row_scale), adapter))",
                                          "(np.clip(codes + np.rint(adapter.scale * adapter.up @ adapter.down), "
                                          "-127, 127).astype(np.int8), row_scale)"),
    "nf4 nibbles swapped": ("nf4_unpack", "codes[:, 0::2] = packed & 15\n    codes[:, 1::2] = packed >> 4",
                            "codes[:, 0::2] = packed >> 4\n    codes[:, 1::2] = packed & 15"),
    "nf4 restore ignores the block scale": ("nf4_dequantize", "return cb[codes] * scale",
                                            "return cb[codes] * np.ones_like(scale)"),
    "nf4 ties to the upper code": ("nf4_quantize", "np.argmin(dist, axis=-1)",
                                   "(15 - np.argmin(dist[..., ::-1], axis=-1))"),
    "nf4 absmax without the magnitude": ("nf4_quantize", "absmax = np.abs(blocks).max(axis=2)",
                                         "absmax = blocks.max(axis=2)"),
    "nf4 merge adds to the codes": ("nf4_merge", "return nf4_quantize(merged.astype(np.float32), codebook)",
                                    "return nf4_pack(np.clip(nf4_unpack(packed) + np.rint(adapter.scale * adapter.up "
                                    "@ adapter.down), 0, 15).astype(np.uint8)), absmax"),
}

PY_PIN_TESTS = [
    pins.test_quantize_recovers_an_exact_grid,
    pins.test_quantize_sends_exact_ties_to_the_even_code,
    pins.test_quantization_error_is_at_most_half_a_step,
    pins.test_merge_on_a_quantized_base_three_ways,
    pins.test_nf4_packing_puts_even_columns_in_the_low_nibble,
    pins.test_nf4_quantize_recovers_an_exact_grid,
    pins.test_nf4_ties_go_to_the_lower_code,
    pins.test_nf4_error_is_at_most_half_the_widest_gap,
    pins.test_nf4_merge_three_ways,
]


def _count_failures(tests):
    failures = 0
    for t in tests:
        try:
            t()
        except AssertionError:
            failures += 1
    return failures


def test_numpy_pins_pass_on_the_real_oracle():
    assert _count_failures(PY_PIN_TESTS) == 0


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_every_planted_numpy_mistake_is_caught(name, monkeypatch):
    fn, old, new = PY_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(getattr(oracle, fn)))
    assert src.count(old) == 1, f"mutation site of {name!r} not found exactly once"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, fn, ns[fn])
    assert _count_failures(PY_PIN_TESTS) > 0, f"no pin caught the mutant {name!r}"
