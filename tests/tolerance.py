"""Element-wise acceptance rule shared by the parity tests.

bf16 in / fp32 accumulate / bf16 out:  |gpu - oracle| <= 1e-2 * (1 + |oracle|)
fp32 throughout:                       |gpu - oracle| <= 1e-5 * (1 + |oracle|)
Integer and index outputs are compared for exact equality.
"""
import numpy as np

RTOL = {"bf16": 1e-2, "f32": 1e-5}


def within(got: np.ndarray, want: np.ndarray, dtype: str) -> np.ndarray:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return np.abs(got - want) <= RTOL[dtype] * (1.0 + np.abs(want))


def assert_within(got, want, dtype: str, what: str = ""):
    ok = within(got, want, dtype)
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        g = np.asarray(got, np.float64)[i]
        w = np.asarray(want, np.float64)[i]
        raise AssertionError(f"{what}: {bad.shape[0]} of {ok.size} elements out of tolerance "
                             f"(first at {i}: got {g!r}, want {w!r})")
