"""The allocation-free projection entry point, through the C ABI.

mlora_project_noalloc serves callers that may not allocate device memory when
they need a projection (inside a host runtime that owns the memory budget, in
loops that cannot take an allocation's synchronisation).
Its output must match the fp64 oracle's projection X W^T, and what the
pool-based entry point (mlora_forward with no row map) produces for the same X
and W, call after call: the shared scratch array keeps the previous call's
contents, so two calls in a row are checked.  Its status word reports a pipeline
wait that gave up, and keeps it until read.

This file is named to be collected last, so that a failure here stops a run only
after every other test has run.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.tolerance import assert_within

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():   # pragma: no cover - CPU machine
    pytest.skip("needs a GPU", allow_module_level=True)

from heterogeneous_lora_gemm_gb300 import mlora  # noqa: E402
from tests.gpu_harness import make_pool, to_f64, upload  # noqa: E402


@pytest.mark.parametrize("T,din,dout", [(32, 4096, 4096), (1, 64, 200), (256, 512, 1000), (77, 4096, 11008)])
def test_noalloc_matches_oracle_and_pool_forward_twice(T, din, dout):
    layer = wl.random_layer(40 + T, T=T, din=din, dout=dout, ranks=[16])
    pool = make_pool(layer)
    X, W, _, Y_ref = upload(layer)
    stream = torch.cuda.current_stream()
    pool.forward(X, W, None, Y_ref, stream=stream)      # existing entry point: Y = X W^T
    torch.cuda.synchronize()
    from_pool = to_f64(Y_ref)
    want = oracle.forward(layer.X_f64, layer.W_f64, None, [])
    assert_within(from_pool, want, "bf16", "pool forward without row map")
    for call in range(2):
        Y = torch.full_like(Y_ref, float("nan"))
        mlora.mlora_project_noalloc(X.data_ptr(), W.data_ptr(), T, din, dout, Y.data_ptr(), stream.cuda_stream)
        torch.cuda.synchronize()
        got = to_f64(Y)
        assert_within(got, want, "bf16", f"no-alloc projection against the oracle, call {call}")
        assert_within(got, from_pool, "bf16", f"no-alloc projection against mlora_forward, call {call}")
    assert mlora.mlora_project_noalloc_status(stream.cuda_stream) == mlora.MLORA_OK
    pool.close()


def test_noalloc_status_reports_an_expired_wait_until_read():
    """A pipeline wait that gives up (here: one that nothing completes, bounded to
    about a millisecond) sets the status bit; later projections leave it set, the
    status call reports and clears it."""
    stream = torch.cuda.current_stream()
    assert mlora.mlora_project_noalloc_status(stream.cuda_stream) == mlora.MLORA_OK
    mlora.mlora_debug_noalloc_expire_wait(2_000_000, stream.cuda_stream)
    X = torch.ones((16, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.ones((64, 64), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    mlora.mlora_project_noalloc(X.data_ptr(), W.data_ptr(), 16, 64, 64, Y.data_ptr(), stream.cuda_stream)
    assert mlora.mlora_project_noalloc_status(stream.cuda_stream) == mlora.MLORA_ERR_DEVICE_TIMEOUT
    assert mlora.mlora_project_noalloc_status(stream.cuda_stream) == mlora.MLORA_OK   # read-and-clear
    assert np.all(to_f64(Y) == 64.0)
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_debug_noalloc_expire_wait(0, stream.cuda_stream)
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG


def test_noalloc_rejects_sizes_beyond_its_scratch():
    X = torch.zeros((300, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((300, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_project_noalloc(X.data_ptr(), W.data_ptr(), 257, 64, 64, Y.data_ptr(), 0)
    assert e.value.status == mlora.MLORA_ERR_UNSUPPORTED
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_project_noalloc(X.data_ptr(), W.data_ptr(), 4, 64, 262145, Y.data_ptr(), 0)
    assert e.value.status == mlora.MLORA_ERR_UNSUPPORTED
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_project_noalloc(X.data_ptr() + 2, W.data_ptr(), 4, 64, 64, Y.data_ptr(), 0)
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    mlora.mlora_project_noalloc(X.data_ptr(), W.data_ptr(), 0, 64, 64, Y.data_ptr(), 0)   # T = 0: nothing to do
    assert np.all(to_f64(Y) == 0.0)
