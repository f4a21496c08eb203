"""Parity of the NF4 base (ai-infra-kb "M031" §05: W restored by scale and codebook)
through the C ABI against the fp64 oracle: restore, the dynamic branch over the
restored base (decode batches read the codes in the projection kernel), and the
merge that quantizes again (codes decided in fp32 on both sides)."""
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
from tests.gpu_harness import make_pool, to_device, to_f64, upload  # noqa: E402


def ora_adapters(layer):
    return [None if a is None else oracle.OracleAdapter(a.down_f64, a.up_f64, a.scale) for a in layer.slot_list()]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_nf4_restore_matches_oracle(dtype):
    cb = wl.nf4_codebook()
    packed, absmax = wl.nf4_random_base(1, 200, 320)
    q, am = torch.from_numpy(packed).cuda(), torch.from_numpy(absmax).cuda()
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    W = torch.empty((200, 320), dtype=tdt, device="cuda")
    mlora.mlora_dequantize_nf4(q.data_ptr(), am.data_ptr(), cb, 200, 320,
                               mlora.MLORA_BF16 if dtype == "bf16" else mlora.MLORA_F32, W.data_ptr(), 0)
    torch.cuda.synchronize()
    assert_within(to_f64(W), oracle.nf4_dequantize(packed, absmax, cb), dtype, "NF4 restore")


@pytest.mark.parametrize("T,din,dout,ranks", [
    (40, 256, 192, [16, 8]),          # decode: the projection reads the codes (push reduction)
    (128, 1024, 640, [16] * 100),     # decode, many adapters (CUDA-core shrink), staged reduction
    (300, 256, 192, [16, 8]),         # prefill: restore pass into W_scratch, then the forward
    (40, 256, 198, [16, 8]),          # decode, dout not a multiple of 4: restore pass (scales not by TMA)
    (40, 192, 256, [16, 8]),          # decode, 3 K blocks: the second step's second block past din
    (256, 512, 384, [16, 8, 16]),     # decode, 256 tokens: the widest token tile over codes
])
def test_forward_over_an_nf4_base(T, din, dout, ranks):
    cb = wl.nf4_codebook()
    layer = wl.random_layer(61, T=T, din=din, dout=dout, ranks=ranks)
    packed, absmax = oracle.nf4_quantize(layer.W_f64, cb)
    pool = make_pool(layer)
    X, _, ra, Y = upload(layer)
    q, am = torch.from_numpy(packed).cuda(), torch.from_numpy(absmax).cuda()
    W_scratch = torch.zeros((dout, din), dtype=torch.bfloat16, device="cuda")
    pool.forward_nf4(X, q, am, cb, W_scratch, ra, Y)
    torch.cuda.synchronize()
    Wd = oracle.nf4_dequantize(packed, absmax, cb)
    assert_within(to_f64(Y), oracle.forward(layer.X_f64, Wd, layer.row_adapter, ora_adapters(layer)), "bf16",
                  "forward over the NF4 base")
    W_rest = torch.empty_like(W_scratch)
    mlora.mlora_dequantize_nf4(q.data_ptr(), am.data_ptr(), cb, dout, din, mlora.MLORA_BF16, W_rest.data_ptr(), 0)
    Y2 = torch.empty_like(Y)
    pool.forward(X, W_rest, ra, Y2)
    torch.cuda.synchronize()
    assert_within(to_f64(Y), to_f64(Y2), "bf16", "codes read by the projection vs restore + forward")
    if T <= 256 and dout % 4 == 0:   # the projection read the codes
        assert torch.count_nonzero(W_scratch) == 0
    else:
        assert torch.equal(W_scratch, W_rest)
    assert pool.status() == mlora.MLORA_OK


def _exact_grid_case(seed):
    """A codebook of eighths, power-of-two block scales, and an adapter of few-bit
    dyadic values: every fp32 step of the merge is exact, so both sides decide the
    same codes (the division and the distances round identically)."""
    rng = np.random.default_rng(seed)
    cb = (np.arange(-8, 8) / 8.0).astype(np.float32)
    dout, din, r = 96, 192, 4
    codes = rng.integers(0, 16, size=(dout, din)).astype(np.uint8)
    absmax = (2.0 ** rng.integers(-6, -3, size=(din // 64, dout))).astype(np.float32)
    down = rng.choice(np.array([0.0, 2.0 ** -4, -2.0 ** -4, 2.0 ** -5]), size=(r, din))
    up = rng.choice(np.array([0.0, 2.0 ** -3, -2.0 ** -3]), size=(dout, r))
    return cb, oracle.nf4_pack(codes), absmax, down, up, 2.0


def test_merge_nf4_is_bit_exact_on_an_exact_grid():
    cb, packed, absmax, down, up, s = _exact_grid_case(71)
    dout, din = packed.shape[0], packed.shape[1] * 2
    from heterogeneous_lora_gemm_gb300 import Pool
    pool = Pool(2, 8, 4, din, dout, "bf16", 4)
    pool.load(1, to_device(wl.f32_to_bf16_bits(down), "bf16"), to_device(wl.f32_to_bf16_bits(up), "bf16"), s)
    q, am = torch.from_numpy(packed.copy()).cuda(), torch.from_numpy(absmax.copy()).cuda()
    pool.merge_nf4(q, am, cb, 1)
    torch.cuda.synchronize()
    want_q, want_am = oracle.nf4_merge(packed, absmax, cb, oracle.OracleAdapter(down, up, s))
    np.testing.assert_array_equal(am.cpu().numpy(), want_am)
    np.testing.assert_array_equal(q.cpu().numpy(), want_q)
    # merging again moves the base on (the update adds up, codes are not restored)
    pool.merge_nf4(q, am, cb, 1)
    torch.cuda.synchronize()
    want_q2, want_am2 = oracle.nf4_merge(want_q, want_am, cb, oracle.OracleAdapter(down, up, s))
    np.testing.assert_array_equal(am.cpu().numpy(), want_am2)
    np.testing.assert_array_equal(q.cpu().numpy(), want_q2)
    assert pool.status() == mlora.MLORA_OK


def test_merge_nf4_random_within_one_code():
    """Random base and adapter (the NormalFloat codebook): the kernel's fp32 update sum
    can land on the other side of a decision boundary only when the merged value is
    within a few fp32 ulps of it -- then the code differs by one; absmax to fp32 rounding."""
    cb = wl.nf4_codebook()
    layer = wl.random_layer(72, T=4, din=512, dout=320, ranks=[24])
    packed, absmax = oracle.nf4_quantize(layer.W_f64, cb)
    pool = make_pool(layer)
    q, am = torch.from_numpy(packed.copy()).cuda(), torch.from_numpy(absmax.copy()).cuda()
    pool.merge_nf4(q, am, cb, 0)
    torch.cuda.synchronize()
    a = layer.adapters[0]
    want_q, want_am = oracle.nf4_merge(packed, absmax, cb, oracle.OracleAdapter(a.down_f64, a.up_f64, a.scale))
    got_am = am.cpu().numpy()
    np.testing.assert_allclose(got_am, want_am, rtol=2.0 ** -20, atol=0)
    got_c, want_c = oracle.nf4_unpack(q.cpu().numpy()), oracle.nf4_unpack(want_q)
    diff = got_c.astype(int) - want_c.astype(int)
    assert np.abs(diff).max() <= 1
    assert np.count_nonzero(diff) <= max(2, diff.size // 1000)
    # the merged base serves the adapter's rows: the dynamic branch's output within the
    # NF4 bound of the merged float weight
    Wm = oracle.nf4_dequantize(q.cpu().numpy(), got_am, cb)
    Wf = oracle.nf4_dequantize(packed, absmax, cb) + a.scale * a.up_f64 @ a.down_f64
    half_gap = np.max(np.diff(cb.astype(np.float64))) / 2
    bound = np.repeat(got_am.T.astype(np.float64), 64, axis=1) * half_gap * 1.001 + 1e-7
    assert (np.abs(Wm - Wf) <= bound).all()
    assert pool.status() == mlora.MLORA_OK


def test_nf4_argument_errors():
    cb = wl.nf4_codebook()
    layer = wl.random_layer(73, T=4, din=96, dout=64, ranks=[8])   # din not a multiple of 64
    pool = make_pool(layer)
    X, _, ra, Y = upload(layer)
    q = torch.zeros((64, 48), dtype=torch.uint8, device="cuda")
    am = torch.ones((2, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(mlora.MloraError) as e:
        pool.forward_nf4(X, q, am, cb, None, ra, Y)
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    with pytest.raises(mlora.MloraError) as e:
        pool.merge_nf4(q, am, cb, 0)
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        pool.merge_nf4(q, am, cb[:15], 0)
