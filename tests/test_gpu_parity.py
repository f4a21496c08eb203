"""Parity of the CUDA path (through the C ABI) against the fp64 oracle.

Values: |gpu - oracle| <= 1e-2 (1 + |oracle|) for bf16, 1e-5 (1 + |oracle|) for fp32.
Indices (perm, offsets): bit-exact.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.tolerance import assert_within, within

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():   # pragma: no cover - CPU machine
    pytest.skip("needs a GPU", allow_module_level=True)

from heterogeneous_lora_gemm_gb300 import mlora  # noqa: E402
from tests.gpu_harness import make_pool, run_layer, to_device, to_f64, upload  # noqa: E402


def ora_adapters(layer):
    return [None if a is None else oracle.OracleAdapter(a.down_f64, a.up_f64, a.scale) for a in layer.slot_list()]


def want_of(layer, rows=None, row_adapter=None):
    ra = layer.row_adapter if row_adapter is None else row_adapter
    return oracle.forward(layer.X_f64, layer.W_f64, ra, ora_adapters(layer), rows=rows)


def gpu_segments(layer, pool, row_adapter=None):
    ra = torch.from_numpy((layer.row_adapter if row_adapter is None else row_adapter).astype(np.int32)).cuda()
    T = ra.shape[0]
    perm = torch.full((max(T, 1),), -7, dtype=torch.int32, device="cuda")
    offs = torch.full((layer.max_slots + 1,), -7, dtype=torch.int32, device="cuda")
    pool.segments(ra, perm[:T], offs)
    torch.cuda.synchronize()
    return perm[:T].cpu().numpy(), offs.cpu().numpy()


def check_segments(layer, pool, row_adapter=None):
    ra = layer.row_adapter if row_adapter is None else row_adapter
    perm, offs = gpu_segments(layer, pool, ra)
    counts, w_offs, w_perm, _ = oracle.segments(ra, oracle.slot_ranks(ora_adapters(layer)), layer.max_slots)
    assert np.array_equal(offs, w_offs), (offs, w_offs)
    n = w_perm.size
    assert np.array_equal(perm[:n], w_perm)
    assert np.all(perm[n:] == -1)


def check_forward_segments(layer, pool, row_adapter=None):
    """The segments the forward's own builder produced (on the bf16 path, the builder
    inside the shrink kernel) equal the oracle's, bit for bit."""
    ra = layer.row_adapter if row_adapter is None else row_adapter
    T = ra.shape[0]
    perm = torch.full((max(T, 1),), -7, dtype=torch.int32, device="cuda")
    offs = torch.full((layer.max_slots + 1,), -7, dtype=torch.int32, device="cuda")
    pool.last_segments(perm[:T], offs)
    torch.cuda.synchronize()
    perm, offs = perm[:T].cpu().numpy(), offs.cpu().numpy()
    counts, w_offs, w_perm, _ = oracle.segments(ra, oracle.slot_ranks(ora_adapters(layer)), layer.max_slots)
    assert np.array_equal(offs, w_offs), (offs, w_offs)
    n = w_perm.size
    assert np.array_equal(perm[:n], w_perm)
    assert np.all(perm[n:] == -1)


# --------------------------------------------------------------------------- #
def test_worked_example_fp32():
    layer = wl.worked_example(0)
    pool = make_pool(layer)
    Y = run_layer(layer, pool)
    assert_within(Y, want_of(layer), "f32", "worked example")
    check_forward_segments(layer, pool)
    check_segments(layer, pool)


@pytest.mark.parametrize("seed", [0, 1])
def test_decode_step(seed):
    layer = wl.decode_step(seed)
    pool = make_pool(layer)
    assert_within(run_layer(layer, pool), want_of(layer), "bf16", "decode_step")
    check_forward_segments(layer, pool)


def test_fragmented_decode():
    layer = wl.fragmented_decode(0)
    pool = make_pool(layer)
    check_segments(layer, pool)
    assert_within(run_layer(layer, pool), want_of(layer), "bf16", "fragmented_decode")
    check_forward_segments(layer, pool)


def prefill_sample_rows(seed):
    lengths = wl.prefill_lengths(seed)
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    rng = np.random.default_rng(1000 + seed)
    rows = []
    for s, n in zip(starts, lengths):
        rows += [s, s + n - 1] + list(s + rng.choice(n, size=8, replace=False))
    return np.array(sorted(set(int(r) for r in rows)), np.int64)


def test_prefill_sampled_rows():
    layer = wl.prefill(0)
    pool = make_pool(layer)
    check_segments(layer, pool)
    Y = run_layer(layer, pool)
    check_forward_segments(layer, pool)
    rows = prefill_sample_rows(0)
    assert_within(Y[rows], want_of(layer, rows=rows), "bf16", "prefill")
    assert np.isfinite(Y).all()


@pytest.mark.parametrize("module", ["q", "k", "v", "down", "gate"])
def test_stack7b_projection(module):
    layer = wl.stack7b_projection(0, 0 if module in "qkv" else 17, module)
    Y = run_layer(layer)
    rows = None if module in ("q", "k", "v") else np.arange(0, 128, 9)
    want = want_of(layer, rows=rows)
    assert_within(Y if rows is None else Y[rows], want, "bf16", f"stack7b {module}")


# --------------------------------------------------------------------------- #
# edge cases
@pytest.mark.parametrize("T,din,dout,ranks", [
    (1, 64, 64, [16]),
    (37, 72, 200, [8, 0, 24, 64, 1]),
    (300, 128, 136, [16, 8, 64]),
    (129, 4096, 256, [16, 64, 8]),
    (5, 8, 8, [3, 5]),
    (64, 1024, 5120, [16, 8]),     # 40 row tiles: 6 K splits, two CTAs per SM
    (200, 512, 384, [16, 8, 64]),  # two token tiles of the projection, the second ragged (72)
    (250, 64, 128, [8, 16]),       # two token tiles, one K step, no K split
    (100, 256, 7200, [16, 8]),     # 57 row tiles (odd), two K splits, ragged last tile
    (256, 256, 3600, [16, 64]),    # two token tiles over 29 row tiles, ragged last tile
])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_shapes(T, din, dout, ranks, dtype):
    layer = wl.random_layer(T * 7 + din, T=T, din=din, dout=dout, ranks=ranks, dtype=dtype)
    pool = make_pool(layer)
    check_segments(layer, pool)
    assert_within(run_layer(layer, pool), want_of(layer), dtype, f"ragged {T}x{din}x{dout}")


@pytest.mark.parametrize("T,din,dout,row_map", [
    (100, 1024, 20000, False),   # 157 row tiles: two per CTA, the last 256-row block ragged (32 rows)
    (128, 4096, 22016, True),    # the 7B layer's gate|up shape, row map of rows without adapter
])
def test_two_row_tiles_per_cta(T, din, dout, row_map):
    """More 128-row W tiles than SMs and no adapters: each CTA takes two row tiles that
    share its X stages (two accumulators, a 256-row partial tile in the split-K sums)."""
    layer = wl.random_layer(T + dout, T=T, din=din, dout=dout, ranks=[])
    pool = make_pool(layer)
    X, W, ra, Y = upload(layer)
    pool.forward(X, W, ra if row_map else None, Y)
    torch.cuda.synchronize()
    assert_within(to_f64(Y), want_of(layer), "bf16", f"two row tiles per CTA, {T}x{din}x{dout}")
    assert pool.status() == mlora.MLORA_OK


def test_many_loaded_slots_few_used():
    """300 loaded rank-16 slots, a batch that uses three of them: the shrink and the
    expand skip the unused chunks, and one projection CTA holds more chunks (300,
    din = 64 gives a single K split) than it keeps in shared memory."""
    ra = np.random.default_rng(11).choice(np.array([3, 150, 299, -1], np.int32), size=64).astype(np.int32)
    layer = wl.random_layer(11, T=64, din=64, dout=256, ranks=[16] * 300, row_adapter=ra)
    pool = make_pool(layer)
    check_segments(layer, pool)
    assert_within(run_layer(layer, pool), want_of(layer), "bf16", "300 slots, 3 used")
    check_forward_segments(layer, pool)


@pytest.mark.parametrize("T,din,n_slots,choices", [
    (200, 1000, 120, (5, 16, 24, 8)), (100, 1000, 120, (5, 16, 24, 8)), (128, 11008, 90, (5, 16, 24, 8)),
    (200, 1000, 120, (5, 16, 8)),     # every adapter one chunk (the second 8-column Up block unused at 5 and 8)
    (128, 4096, 100, (16,)),
])
def test_many_adapters_few_rows_each(T, din, n_slots, choices):
    """Decode batches with at most two rows per loaded adapter on average take the
    CUDA-core shrink: ranks that are not multiples of 16 (partial chunks), one slot
    with more rows than one pass over its Down rows holds, rows without adapter,
    din not a multiple of 256 (and 11008, two rows per pass), with and without the
    L2 prefetch before the wait (T >= loaded slots or not)."""
    rng = np.random.default_rng(T + din)
    ranks = list(rng.choice(np.array(choices), size=n_slots))
    ra = rng.integers(0, n_slots, size=T).astype(np.int32)
    ra[: 20] = 3                                  # slot 3: 20 rows (three passes of 8)
    ra[rng.random(T) < 0.1] = -1
    layer = wl.random_layer(T, T=T, din=din, dout=384, ranks=ranks, row_adapter=ra)
    pool = make_pool(layer)
    assert_within(run_layer(layer, pool), want_of(layer), "bf16", f"many adapters, T = {T}, din = {din}")
    check_forward_segments(layer, pool)


def test_chained_forwards_read_the_previous_output():
    """Each forward's X is the previous forward's Y, enqueued back to back on one
    stream: the kernels of a forward start while the previous forward's kernels may
    still run, and must read X only once it is written.  The kernels are
    deterministic (fixed split order), so the chain must equal, bit for bit, the same
    chain with a device synchronisation after every forward."""
    # the last two: CUDA-core shrink, with a rank-24 adapter spanning two chunks of the
    # same rows, and with 24 adapters of one chunk each
    for shape in ((1024, [16, 8]), (4096, [16, 16, 16]), (1024, [16, 8, 24] * 7), (1024, [16, 8] * 12)):
        chain_case(*shape)


def chain_case(d, ranks):
    layer = wl.random_layer(14, T=32, din=d, dout=d, ranks=ranks)
    pool = make_pool(layer)
    X0, W, ra, _ = upload(layer)
    for row_map in (ra, None):
        synced, x = [], X0
        for _ in range(4):
            y = torch.empty_like(x)
            pool.forward(x, W, row_map, y)
            torch.cuda.synchronize()
            synced.append(y.clone())
            x = y
        chained, x = [], X0
        ys = [torch.empty_like(X0) for _ in range(4)]
        for y in ys:
            pool.forward(x, W, row_map, y)
            chained.append(y)
            x = y
        torch.cuda.synchronize()
        for k, (a, b) in enumerate(zip(synced, chained)):
            assert torch.equal(a, b), f"forward {k} of the chain (row map {'on' if row_map is not None else 'off'})"
    assert pool.status() == mlora.MLORA_OK


def test_arena_holes_use_one_box_per_chunk():
    """Slots 1..8 unloaded leave a hole of 128 rank rows between slots 0 and 9: their
    chunks no longer fit one 128-row window, so the shrink loads each chunk alone."""
    ra = np.random.default_rng(13).choice(np.array([0, 9, -1], np.int32), size=48).astype(np.int32)
    layer = wl.random_layer(13, T=48, din=256, dout=192, ranks=[16] * 10, row_adapter=ra)
    pool = make_pool(layer)
    for slot in range(1, 9):
        pool.unload(slot)
    assert_within(run_layer(layer, pool), want_of(layer), "bf16", "arena holes")


def test_prefill_runs_with_multichunk_ranks():
    """Request-ordered runs over slots whose ranks span 1..4 chunks: every 256-token
    tile of the shrink, and every 128-token tile of the projection, uses its own
    subset of the chunks."""
    runs = [(0, 180), (2, 90), (-1, 40), (4, 300), (1, 70), (3, 120), (0, 30)]
    ra = np.concatenate([np.full(n, s, np.int32) for s, n in runs])
    layer = wl.random_layer(12, T=int(ra.shape[0]), din=256, dout=512, ranks=[64, 8, 40, 16, 1], row_adapter=ra)
    pool = make_pool(layer)
    check_segments(layer, pool)
    assert_within(run_layer(layer, pool), want_of(layer), "bf16", "prefill runs")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_all_rows_without_adapter_and_null_map(dtype):
    layer = wl.random_layer(3, T=33, din=64, dout=48, ranks=[16, 8], dtype=dtype,
                            row_adapter=np.full(33, -1, np.int32))
    pool = make_pool(layer)
    assert_within(run_layer(layer, pool), want_of(layer), dtype, "all -1")
    assert_within(run_layer(layer, pool, with_row_adapter=False), want_of(layer), dtype, "NULL map")
    check_segments(layer, pool)


def test_all_rows_one_adapter_equals_merged():
    layer = wl.random_layer(4, T=64, din=256, dout=128, ranks=[0, 32], row_adapter=np.full(64, 1, np.int32))
    Y = run_layer(layer)
    a = layer.slot_list()[1]
    Wm = layer.W_f64 + a.scale * (a.up_f64 @ a.down_f64)
    assert_within(Y, layer.X_f64 @ Wm.T, "bf16", "single adapter")


def test_invalid_ids_set_status_and_act_as_none():
    ra = np.array([0, 5, 1, -3, 2, 0, 9, -1], np.int32)   # 5, 9 out of range, -3 bad, slot 1 empty
    layer = wl.random_layer(5, T=8, din=64, dout=32, ranks=[8, 0, 16], row_adapter=ra)
    pool = make_pool(layer)
    assert pool.status() == mlora.MLORA_OK
    Y = run_layer(layer, pool, check_status=False)
    assert pool.status() == mlora.MLORA_ERR_DEVICE_ROW
    assert pool.status() == mlora.MLORA_OK           # read-and-clear
    assert_within(Y, want_of(layer), "bf16", "invalid ids")
    base = layer.X_f64 @ layer.W_f64.T
    assert_within(Y[[1, 2, 3, 6, 7]], base[[1, 2, 3, 6, 7]], "bf16", "invalid rows keep base")
    check_forward_segments(layer, pool)
    check_segments(layer, pool)
    with pytest.raises(mlora.MloraError):   # the standalone builder replaced the forward's segments
        check_forward_segments(layer, pool)


def test_zero_rows_is_noop():
    layer = wl.random_layer(6, T=4, din=64, dout=32, ranks=[8])
    pool = make_pool(layer)
    X, W, ra, Y = upload(layer)
    mlora.mlora_forward(pool.handle, X.data_ptr(), W.data_ptr(), ra.data_ptr(), 0, Y.data_ptr(), 0)
    torch.cuda.synchronize()
    assert torch.isnan(Y.float()).all()


def test_max_tokens_boundary_and_errors():
    layer = wl.random_layer(7, T=48, din=64, dout=64, ranks=[16, 16])
    pool = make_pool(layer, max_tokens=48)
    assert_within(run_layer(layer, pool), want_of(layer), "bf16", "T = max_tokens")
    X, W, ra, Y = upload(layer)
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_forward(pool.handle, X.data_ptr(), W.data_ptr(), ra.data_ptr(), 49, Y.data_ptr(), 0)
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_forward(pool.handle, X.data_ptr() + 2, W.data_ptr(), ra.data_ptr(), 4, Y.data_ptr(), 0)
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    with pytest.raises(mlora.MloraError) as e:
        pool.load(0, to_device(layer.adapters[0].down, "bf16")[:0], to_device(layer.adapters[0].up, "bf16"), 1.0)
    assert e.value.status == mlora.MLORA_ERR_RANK


# --------------------------------------------------------------------------- #
# merge (M031 §04)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_merge_matches_oracle(dtype):
    layer = wl.random_layer(8, T=1, din=512, dout=384, ranks=[16, 64], dtype=dtype)
    pool = make_pool(layer)
    for slot in (0, 1):
        W = to_device(layer.W, dtype)
        pool.merge(W, slot)
        torch.cuda.synchronize()
        a = ora_adapters(layer)[slot]
        assert_within(to_f64(W), oracle.merge(layer.W_f64, a), dtype, f"merge slot {slot}")


@pytest.mark.parametrize("din,dout,ranks", [
    (72, 200, [8, 5, 24, 1]),      # ragged tiles; ranks 8, 5, 1 leave the second half of their chunk to the next adapter
    (4096, 4096, [16, 64, 40]),    # the decode shapes, several chunks per adapter
    (256, 136, [256]),             # the largest rank, one adapter filling the arena
])
def test_merge_ranks_and_ragged_tiles(din, dout, ranks):
    layer = wl.random_layer(din + dout, T=1, din=din, dout=dout, ranks=ranks)
    pool = make_pool(layer)
    for slot in range(len(ranks)):
        W = to_device(layer.W, "bf16")
        pool.merge(W, slot)
        torch.cuda.synchronize()
        a = ora_adapters(layer)[slot]
        assert_within(to_f64(W), oracle.merge(layer.W_f64, a), "bf16", f"merge {din}x{dout} slot {slot} rank {ranks[slot]}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_unmerge_matches_oracle_and_bounds_the_round_trip(dtype):
    """airsota card "multi-LoRA serving vs merging", section 四 item ③: a merge
    overwrites the base and switching back re-subtracts the update.  The un-merge
    matches the oracle's W - s Up Down; after a merge, it returns the original W up
    to the two roundings, |W'' - W| <= u (|W'| + |W''|), with the fp32 error of the
    update sum on top.  Ragged tiles; ranks 16, 40 (three chunks) and 5."""
    layer = wl.random_layer(21, T=1, din=200, dout=136, ranks=[16, 40, 5], dtype=dtype)
    pool = make_pool(layer)
    u = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -24   # unit roundoff: 8 and 24 significant bits
    u32 = 2.0 ** -24
    for slot, a in enumerate(ora_adapters(layer)):
        W = to_device(layer.W, dtype)
        pool.unmerge(W, slot)
        torch.cuda.synchronize()
        assert_within(to_f64(W), oracle.unmerge(layer.W_f64, a), dtype, f"unmerge slot {slot}")
        W = to_device(layer.W, dtype)
        pool.merge(W, slot)
        torch.cuda.synchronize()
        Wm = to_f64(W)
        pool.unmerge(W, slot)
        torch.cuda.synchronize()
        Wu = to_f64(W)
        W0 = layer.W_f64
        delta_abs = abs(a.scale) * (np.abs(a.up) @ np.abs(a.down))
        bound = (u * (np.abs(Wm) + np.abs(Wu)) * (1 + 2.0 ** -7)
                 + 2 * a.rank * u32 * delta_abs + 4 * u32 * (np.abs(W0) + np.abs(Wm)))
        err = np.abs(Wu - W0)
        assert (err <= bound).all(), f"slot {slot}: round trip error {err.max()} above its bound"
        assert np.abs(Wm - W0).max() > 10 * err.max(), "the merge changed W"
    assert pool.status() == mlora.MLORA_OK


def test_merged_weight_serves_only_its_adapter():
    layer = wl.decode_step(0)
    pool = make_pool(layer)
    W = to_device(layer.W, "bf16")
    pool.merge(W, 0)
    X, _, ra, Y = upload(layer)
    pool.forward(X, W, None, Y)        # merged weight, no branch
    torch.cuda.synchronize()
    Ym = to_f64(Y)
    want = want_of(layer)
    rows_a = layer.row_adapter == 0
    assert_within(Ym[rows_a], want[rows_a], "bf16", "merged A on A rows")
    assert not within(Ym[layer.row_adapter == 1], want[layer.row_adapter == 1], "bf16").all()


# --------------------------------------------------------------------------- #
# pool lifecycle (M031 §06/§07)
def test_load_waits_for_last_reader_and_versions():
    layer = wl.random_layer(9, T=256, din=1024, dout=1024, ranks=[16, 16], p_none=0.0)
    other = wl.random_layer(10, T=256, din=1024, dout=1024, ranks=[16, 16], p_none=0.0)
    pool = make_pool(layer)
    assert pool.version(0) == 1
    X, W, ra, Y = upload(layer)
    pool.forward(X, W, ra, Y)                       # enqueued, not waited for
    b = other.adapters[0]
    pool.load(0, to_device(b.down, "bf16"), to_device(b.up, "bf16"), b.scale)   # replaces slot 0
    assert pool.version(0) == 2
    torch.cuda.synchronize()
    assert_within(to_f64(Y), want_of(layer), "bf16", "forward before the load keeps old weights")
    Y2 = torch.empty_like(Y)
    pool.forward(X, W, ra, Y2)
    torch.cuda.synchronize()
    swapped = [oracle.OracleAdapter(b.down_f64, b.up_f64, b.scale), ora_adapters(layer)[1]]
    assert_within(to_f64(Y2), oracle.forward(layer.X_f64, layer.W_f64, layer.row_adapter, swapped), "bf16",
                  "forward after the load uses new weights")
    pool.unload(1)
    assert pool.version(1) == 2
    with pytest.raises(mlora.MloraError) as e:
        pool.unload(1)
    assert e.value.status == mlora.MLORA_ERR_NOT_LOADED


# --------------------------------------------------------------------------- #
# quantized base (M031 §05)
@pytest.mark.parametrize("T,din,dout,ranks", [
    (40, 256, 192, [16, 8]),          # decode: the projection reads the codes (push reduction)
    (200, 1024, 640, [16] * 120),     # decode, many adapters (CUDA-core shrink), staged reduction
    (128, 512, 7200, [16, 8]),        # decode, 57 row tiles (odd), two K splits
    (40, 192, 256, [16, 8]),          # decode, 3 K chunks: the second step's second chunk past din
    (300, 256, 192, [16, 8]),         # prefill: restore pass into W_scratch, then the forward
    (40, 136, 192, [16, 8]),          # din not a multiple of 64: restore pass
    (256, 512, 384, [16, 8, 16]),     # decode, 256 tokens: one K chunk per stage (two do not fit)
    (224, 320, 256, [16, 8]),         # decode, 224 tokens, 5 K chunks
])
def test_forward_over_a_quantized_base(T, din, dout, ranks):
    """The dynamic branch over an int8 base (codes x row scale, one rounding of the
    restored value): against the oracle over the restored W, and against the restore
    pass followed by the ordinary forward."""
    layer = wl.random_layer(51, T=T, din=din, dout=dout, ranks=ranks)
    codes, scale = oracle.quantize(layer.W_f64)
    pool = make_pool(layer)
    X, _, ra, Y = upload(layer)
    Wq, sc = torch.from_numpy(codes).cuda(), torch.from_numpy(scale).cuda()
    W_scratch = torch.zeros((layer.dout, layer.din), dtype=torch.bfloat16, device="cuda")
    pool.forward_quantized(X, Wq, sc, W_scratch, ra, Y)
    torch.cuda.synchronize()
    Wd = oracle.dequantize(codes, scale)
    want = oracle.forward(layer.X_f64, Wd, layer.row_adapter, ora_adapters(layer))
    assert_within(to_f64(Y), want, "bf16", "forward over the quantized base")
    W_rest = torch.empty_like(W_scratch)
    mlora.mlora_dequantize(Wq.data_ptr(), sc.data_ptr(), dout, din, mlora.MLORA_BF16, W_rest.data_ptr(), 0)
    Y2 = torch.empty_like(Y)
    pool.forward(X, W_rest, ra, Y2)
    torch.cuda.synchronize()
    assert_within(to_f64(W_rest), Wd, "bf16", "restored base")
    assert_within(to_f64(Y), to_f64(Y2), "bf16", "codes read by the projection vs restore + forward")
    if T <= 256 and din % 64 == 0:
        assert torch.count_nonzero(W_scratch) == 0   # the decode path does not use the scratch
    else:
        assert torch.equal(W_scratch, W_rest)
    assert pool.status() == mlora.MLORA_OK


def test_merge_quantized_is_bit_exact_on_an_exact_grid():
    """Codes, row scales, adapter entries and scale chosen so that every fp32 step of
    the merge is exact: the re-quantized codes and scales equal the oracle's bit for
    bit (both decide in fp32)."""
    from heterogeneous_lora_gemm_gb300 import Pool
    rng = np.random.default_rng(52)
    din, dout, r = 128, 136, 16
    codes = rng.integers(-127, 128, size=(dout, din)).astype(np.int8)
    scale = (2.0 ** rng.integers(-9, -5, size=dout)).astype(np.float32)
    down = rng.integers(-8, 9, size=(r, din)) / 16.0
    up = rng.integers(-8, 9, size=(dout, r)) / 16.0
    pool = Pool(1, 16, 16, din, dout, "bf16", 1)
    pool.load(0, to_device(wl.f32_to_bf16_bits(down), "bf16"), to_device(wl.f32_to_bf16_bits(up), "bf16"), 0.5)
    Wq, sc = torch.from_numpy(codes).cuda(), torch.from_numpy(scale).cuda()
    pool.merge_quantized(Wq, sc, 0)
    torch.cuda.synchronize()
    want_c, want_s = oracle.merge_quantized(codes, scale, oracle.OracleAdapter(down, up, 0.5))
    np.testing.assert_array_equal(sc.cpu().numpy(), want_s)
    np.testing.assert_array_equal(Wq.cpu().numpy(), want_c)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_merge_quantized_random_within_one_step(dtype):
    """Random base and adapter (ragged sizes): row scales to fp32 rounding, codes equal
    but for rare ties decided on an fp32 sum that differs in its last bit."""
    layer = wl.random_layer(53, T=1, din=200, dout=72, ranks=[24], dtype=dtype)
    codes, scale = oracle.quantize(layer.W_f64)
    pool = make_pool(layer)
    Wq, sc = torch.from_numpy(codes).cuda(), torch.from_numpy(scale).cuda()
    pool.merge_quantized(Wq, sc, 0)
    torch.cuda.synchronize()
    want_c, want_s = oracle.merge_quantized(codes, scale, ora_adapters(layer)[0])
    got_c, got_s = Wq.cpu().numpy().astype(np.int32), sc.cpu().numpy()
    np.testing.assert_allclose(got_s, want_s, rtol=1e-6, atol=0)
    diff = np.abs(got_c - want_c.astype(np.int32))
    assert diff.max() <= 1 and (diff > 0).mean() < 1e-3, (diff.max(), (diff > 0).mean())


def test_merge_quantized_ties_round_to_even():
    """Every merged value but one per row lands exactly halfway between two codes
    (w / new scale = code + 1/2 in exact arithmetic): the codes must be the even
    neighbours, as the oracle's fp32 division and rint give."""
    from heterogeneous_lora_gemm_gb300 import Pool
    rng = np.random.default_rng(55)
    din, dout, r = 256, 136, 16
    codes = rng.integers(-127, 127, size=(dout, din)).astype(np.int8)
    codes[:, 0] = 127                     # w[o, 0] = 127 * 2^-6: the row max, new scale 2^-6
    scale = np.full(dout, 2.0 ** -6, dtype=np.float32)
    down = np.zeros((r, din))
    down[0, 1:] = 2.0 ** -7               # update 2^-7 = half a step everywhere but column 0
    up = np.zeros((dout, r))
    up[:, 0] = 1.0
    pool = Pool(1, 16, 16, din, dout, "bf16", 1)
    pool.load(0, to_device(wl.f32_to_bf16_bits(down), "bf16"), to_device(wl.f32_to_bf16_bits(up), "bf16"), 1.0)
    Wq, sc = torch.from_numpy(codes).cuda(), torch.from_numpy(scale).cuda()
    pool.merge_quantized(Wq, sc, 0)
    torch.cuda.synchronize()
    want_c, want_s = oracle.merge_quantized(codes, scale, oracle.OracleAdapter(down, up, 1.0))
    np.testing.assert_array_equal(sc.cpu().numpy(), want_s)
    np.testing.assert_array_equal(Wq.cpu().numpy(), want_c)
    assert (want_c[:, 1:].astype(np.int32) % 2 == 0).all()   # the ties went to the even codes


@pytest.mark.parametrize("din,dout,ranks", [(208, 200, [24]), (1024, 520, [40])])
def test_merge_quantized_tensor_cores_ragged_and_repeated(din, dout, ranks):
    """A bf16 pool whose code rows are whole 16-byte units merges on the tensor cores:
    ragged tiles in both directions, a last rank chunk half used, and a second merge
    after the first (the per-row scratch is cleared between calls).  Each merge is
    checked against the oracle applied to the codes and scales it started from."""
    layer = wl.random_layer(54, T=1, din=din, dout=dout, ranks=ranks, dtype="bf16")
    codes, scale = oracle.quantize(layer.W_f64)
    pool = make_pool(layer)
    Wq, sc = torch.from_numpy(codes).cuda(), torch.from_numpy(scale).cuda()
    ad = ora_adapters(layer)[0]
    for k in range(2):
        start_c, start_s = Wq.cpu().numpy().copy(), sc.cpu().numpy().copy()
        pool.merge_quantized(Wq, sc, 0)
        torch.cuda.synchronize()
        want_c, want_s = oracle.merge_quantized(start_c, start_s, ad)
        got_c, got_s = Wq.cpu().numpy().astype(np.int32), sc.cpu().numpy()
        np.testing.assert_allclose(got_s, want_s, rtol=1e-6, atol=0, err_msg=f"merge {k}: row scales")
        diff = np.abs(got_c - want_c.astype(np.int32))
        assert diff.max() <= 1 and (diff > 0).mean() < 1e-3, (k, diff.max(), (diff > 0).mean())
    assert pool.status() == mlora.MLORA_OK


# --------------------------------------------------------------------------- #
# several modules of a fused projection in one launch (airsota card, section 四 item ④)
@pytest.mark.parametrize("T", [48, 300])
def test_fused_projection_with_per_module_adapters(T):
    """q, k, v rows of one fused projection (boundaries inside 128-row tiles), four
    tenants: q+v with one scale, q alone, k+v with different scales (folded into Up),
    and an adapter of the whole layer; decode (T = 48) and prefill (T = 300) paths."""
    from heterogeneous_lora_gemm_gb300 import Pool
    rng = np.random.default_rng(41)
    din, modules = 256, [(0, 200), (200, 90), (290, 170)]
    dout = 460
    def rnd(shape, std):   # bf16 bit patterns
        return wl.f32_to_bf16_bits(rng.standard_normal(shape) * std)
    spec = {0: [(0, 8, 2.0), (2, 16, 2.0)], 1: [(0, 24, 1.5)], 2: [(1, 16, 3.0), (2, 4, 0.5)]}
    ads = {s_: {m: (rnd((r, din), 1 / 16), rnd((modules[m][1], r), 0.05), sc) for m, r, sc in mods}
           for s_, mods in spec.items()}
    plain = (rnd((16, din), 1 / 16), rnd((dout, 16), 0.05), 2.0)
    W = rnd((dout, din), 0.02)
    X = rnd((T, din), 1.0)
    ra = rng.choice(np.array([0, 1, 2, 3, -1], np.int32), size=T).astype(np.int32)
    pool = Pool(4, 32 + 32 + 32 + 16, 32, din, dout, "bf16", T)
    for s_ in spec:
        mods = []
        for m, (off, n) in enumerate(modules):
            if m in ads[s_]:
                d, u, sc = ads[s_][m]
                mods.append((off, n, to_device(d, "bf16"), to_device(u, "bf16", "cpu"), sc))
            else:
                mods.append((off, n, None, None, 0.0))
        pool.load_modules(s_, mods)
    pool.load(3, to_device(plain[0], "bf16"), to_device(plain[1], "bf16"), plain[2])
    f64 = wl.bf16_bits_to_f64
    tenants = []
    for s_ in range(4):
        row = []
        for m, (off, n) in enumerate(modules):
            if s_ == 3:
                row.append(oracle.OracleAdapter(f64(plain[0]), f64(plain[1])[off:off + n], plain[2]))
            elif m in ads[s_]:
                d, u, sc = ads[s_][m]
                row.append(oracle.OracleAdapter(f64(d), f64(u), sc))
            else:
                row.append(None)
        tenants.append(row)
    Xd, Wd = to_device(X, "bf16"), to_device(W, "bf16")
    Y = torch.empty((T, dout), dtype=torch.bfloat16, device="cuda")
    pool.forward(Xd, Wd, torch.from_numpy(ra).cuda(), Y)
    torch.cuda.synchronize()
    want = oracle.forward_modules(f64(X), f64(W), ra, modules, tenants)
    assert_within(to_f64(Y), want, "bf16", f"fused projection, T = {T}")
    assert pool.status() == mlora.MLORA_OK
    with pytest.raises(mlora.MloraError) as e:   # combined rank 16 + 32 > max_rank 32
        pool.load_modules(0, [(0, 200, to_device(ads[1][0][0], "bf16"), to_device(ads[1][0][1], "bf16"), 1.0),
                              (200, 90, to_device(ads[2][1][0], "bf16"), to_device(ads[2][1][1], "bf16"), 1.0)])
    assert e.value.status == mlora.MLORA_ERR_RANK


@pytest.mark.parametrize("T,layout", [(128, "uniform"), (96, "mixed"), (48, "mixed"),
                                      (200, "mixed"), (256, "uniform")])   # two token tiles
def test_fused_projection_up_runs(T, layout):
    """Tenants that each hold a q and a v adapter of rank 16 put consecutive tenants' q
    (and v) chunks 32 rank columns apart in the arena: a K-extension step of 4 such
    chunks loads their Up tiles in one box.  'mixed' breaks some of those runs with
    tenants of other shapes (q alone, rank 8, rank 32, v alone) between them.  The v rows
    start inside a 128-row tile, and the last tenants' chunks end the arena."""
    from heterogeneous_lora_gemm_gb300 import Pool
    rng = np.random.default_rng(61 + T)
    din, modules = 512, [(0, 320), (320, 320)]   # q rows, v rows
    dout = 640
    n = 37
    shapes = [(16, 16)] * n                      # (rank of q, rank of v) per tenant
    if layout == "mixed":
        shapes = list(shapes)
        for s_, sh in ((5, (8, 0)), (13, (32, 16)), (14, (16, 0)), (29, (0, 24))):
            shapes[s_] = sh
    def rnd(shape, std):   # bf16 bit patterns
        return wl.f32_to_bf16_bits(rng.standard_normal(shape) * std)
    ads = [[(rnd((r, din), 1 / 16), rnd((modules[m][1], r), 0.05), 1.0 + 0.25 * m) if r else None
            for m, r in enumerate(sh)] for sh in shapes]
    budget = sum((r + 15) // 16 * 16 for sh in shapes for r in sh)   # a module takes whole chunks
    pool = Pool(n, budget, 48, din, dout, "bf16", T)
    for s_ in range(n):
        mods = []
        for m, (off, rows) in enumerate(modules):
            a = ads[s_][m]
            mods.append((off, rows, to_device(a[0], "bf16"), to_device(a[1], "bf16", "cpu"), a[2]) if a
                        else (off, rows, None, None, 0.0))
        pool.load_modules(s_, mods)
    assert pool.info().ext_run_stride == 32
    W = rnd((dout, din), 0.02)
    X = rnd((T, din), 1.0)
    ra = rng.choice(np.arange(-1, n, dtype=np.int32), size=T).astype(np.int32)
    f64 = wl.bf16_bits_to_f64
    tenants = [[oracle.OracleAdapter(f64(a[0]), f64(a[1]), a[2]) if a else None for a in row] for row in ads]
    Y = torch.empty((T, dout), dtype=torch.bfloat16, device="cuda")
    pool.forward(to_device(X, "bf16"), to_device(W, "bf16"), torch.from_numpy(ra).cuda(), Y)
    torch.cuda.synchronize()
    want = oracle.forward_modules(f64(X), f64(W), ra, modules, tenants)
    assert_within(to_f64(Y), want, "bf16", f"fused projection with Up runs, T = {T}, {layout}")
    assert pool.status() == mlora.MLORA_OK


# --------------------------------------------------------------------------- #
# host (cold) tier and asynchronous prefetch (M031 §06)
def _host_tier_pool(layer, extra_budget=0, max_rank=None):
    from heterogeneous_lora_gemm_gb300 import Pool
    budget = sum((a.rank + 7) // 8 * 8 for a in layer.adapters) + extra_budget
    return Pool(layer.max_slots, budget, max_rank or layer.max_rank, layer.din, layer.dout, layer.dtype,
                max(layer.T, 1))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefetch_from_host_tier_matches_oracle(dtype):
    """Adapters registered in the pinned host tier and prefetched into their slots
    on the forward's stream: the forward enqueued right after sees them in place."""
    layer = wl.random_layer(31, T=48, din=256, dout=192, ranks=[16, 8, 24, 40], dtype=dtype)
    pool = _host_tier_pool(layer)
    stream = torch.cuda.Stream()
    for a in layer.adapters:   # host sources, ids unrelated to the slots
        pool.host_add(1000 + a.slot, to_device(a.down, dtype, "cpu"), to_device(a.up, dtype, "cpu"), a.scale)
    X, W, ra, Y = upload(layer)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for a in layer.adapters:
            pool.prefetch(a.slot, 1000 + a.slot, stream=stream)
        pool.forward(X, W, ra, Y, stream=stream)
    torch.cuda.synchronize()
    assert_within(to_f64(Y), want_of(layer), dtype, "forward after prefetches")
    assert all(pool.version(a.slot) == 1 for a in layer.adapters)
    check_segments(layer, pool)
    assert pool.status() == mlora.MLORA_OK


def test_prefetch_replaces_a_slot_only_after_its_readers():
    """Forwards enqueued before a prefetch into their slot read the old adapter, the
    ones after it the new one, with no host wait in between (the new weights go to
    free units, the tables change behind the earlier forwards).  Repeated swaps
    recycle the evicted blocks through the quarantine."""
    layer = wl.random_layer(32, T=64, din=1024, dout=1024, ranks=[16, 16], p_none=0.0)
    other = wl.random_layer(33, T=64, din=1024, dout=1024, ranks=[16, 16], p_none=0.0)
    pool = _host_tier_pool(layer, extra_budget=32)   # room for the new copies beside the old
    a0, a1 = layer.adapters
    b0 = other.adapters[0]
    for id_, a in ((0, a0), (1, a1), (2, b0)):
        pool.host_add(id_, to_device(a.down, "bf16", "cpu"), to_device(a.up, "bf16", "cpu"), a.scale)
    stream = torch.cuda.Stream()
    X, W, ra, _ = upload(layer)
    with torch.cuda.stream(stream):
        pool.prefetch(0, 0, stream=stream)
        pool.prefetch(1, 1, stream=stream)
    want_a = want_of(layer)
    swapped = [oracle.OracleAdapter(b0.down_f64, b0.up_f64, b0.scale), ora_adapters(layer)[1]]
    want_b = oracle.forward(layer.X_f64, layer.W_f64, layer.row_adapter, swapped)
    outs = []
    with torch.cuda.stream(stream):
        for rep in range(6):
            ys_a = [torch.empty((layer.T, layer.dout), dtype=torch.bfloat16, device="cuda") for _ in range(8)]
            for y in ys_a:
                pool.forward(X, W, ra, y, stream=stream)
            pool.prefetch(0, 2 if rep % 2 == 0 else 0, stream=stream)   # B, then A back, ...
            y_b = torch.empty_like(ys_a[0])
            pool.forward(X, W, ra, y_b, stream=stream)
            outs.append((ys_a, y_b, rep))
    torch.cuda.synchronize()
    for ys_a, y_b, rep in outs:
        before, after = (want_a, want_b) if rep % 2 == 0 else (want_b, want_a)
        for k, y in enumerate(ys_a):
            assert_within(to_f64(y), before, "bf16", f"swap {rep}: forward {k} before the prefetch")
        assert_within(to_f64(y_b), after, "bf16", f"swap {rep}: forward after the prefetch")
    assert pool.version(0) == 7
    assert pool.status() == mlora.MLORA_OK


def test_prefetch_into_a_slot_that_held_module_adapters():
    """A slot loaded with per-module adapters (chunks that reach only their module's
    rows), then given a whole-layer adapter by prefetch: the new chunks reach every
    row again, and a plain load after that as well."""
    layer = wl.random_layer(36, T=40, din=128, dout=256, ranks=[16, 16], p_none=0.0)
    pool = _host_tier_pool(layer, extra_budget=64, max_rank=32)
    a0, a1 = layer.adapters
    half = layer.dout // 2
    pool.load_modules(0, [(0, half, to_device(a0.down, "bf16"), to_device(a0.up[:half], "bf16"), a0.scale),
                          (half, half, None, None, 0.0)])
    pool.load(1, to_device(a1.down, "bf16"), to_device(a1.up, "bf16"), a1.scale)
    pool.host_add(9, to_device(a0.down, "bf16", "cpu"), to_device(a0.up, "bf16", "cpu"), a0.scale)
    pool.prefetch(0, 9)
    assert_within(run_layer(layer, pool), want_of(layer), "bf16", "whole-layer adapter after module adapters")
    pool.load_modules(0, [(0, half, to_device(a0.down, "bf16"), to_device(a0.up[:half], "bf16"), a0.scale),
                          (half, half, None, None, 0.0)])
    pool.load(0, to_device(a0.down, "bf16"), to_device(a0.up, "bf16"), a0.scale)
    assert_within(run_layer(layer, pool), want_of(layer), "bf16", "plain load after module adapters")


def test_prefetch_errors_and_host_tier_lifecycle():
    layer = wl.random_layer(34, T=8, din=64, dout=64, ranks=[16])
    pool = _host_tier_pool(layer, max_rank=64)
    a = layer.adapters[0]
    down, up = to_device(a.down, "bf16", "cpu"), to_device(a.up, "bf16", "cpu")
    with pytest.raises(mlora.MloraError) as e:
        pool.prefetch(0, 5)
    assert e.value.status == mlora.MLORA_ERR_NOT_LOADED
    pool.host_add(5, down, up, a.scale)
    with pytest.raises(mlora.MloraError) as e:
        pool.prefetch(layer.max_slots, 5)
    assert e.value.status == mlora.MLORA_ERR_BAD_SLOT
    big = wl.random_layer(35, T=8, din=64, dout=64, ranks=[64]).adapters[0]
    pool.host_add(6, to_device(big.down, "bf16", "cpu"), to_device(big.up, "bf16", "cpu"), big.scale)
    with pytest.raises(mlora.MloraError) as e:     # 64 units against a budget of 16
        pool.prefetch(0, 6)
    assert e.value.status == mlora.MLORA_ERR_OOM
    with pytest.raises(mlora.MloraError) as e:
        pool.host_add(7, down[:0], up[:, :0], 1.0)
    assert e.value.status == mlora.MLORA_ERR_RANK
    pool.prefetch(0, 5)
    pool.host_add(5, down, up, 2 * a.scale)          # replaced in the host tier, not in the slot
    pool.host_remove(5)
    with pytest.raises(mlora.MloraError) as e:
        pool.host_remove(5)
    assert e.value.status == mlora.MLORA_ERR_NOT_LOADED
    torch.cuda.synchronize()
    assert_within(run_layer(layer, pool), want_of(layer), "bf16", "slot keeps the prefetched copy")


def test_arena_compaction_keeps_adapters_correct():
    ranks = [16, 64, 8, 24, 16, 8]
    layer = wl.random_layer(11, T=96, din=256, dout=192, ranks=ranks, p_none=0.1)
    budget = sum((r + 7) // 8 * 8 for r in ranks)
    pool = make_pool(layer, rank_budget=budget, max_rank=64)
    info = pool.info()
    assert info.rank_units == budget and info.rank_units_used == budget
    pool.unload(0)
    pool.unload(2)
    pool.unload(4)           # holes of 16, 8, 16 units: 40 free, largest hole 16
    big = wl.random_layer(12, T=1, din=256, dout=192, ranks=[40])
    a = big.adapters[0]
    pool.load(0, to_device(a.down, "bf16"), to_device(a.up, "bf16"), a.scale)    # needs compaction
    assert pool.info().rank_units_used == budget
    slots = ora_adapters(layer)
    slots[0] = oracle.OracleAdapter(a.down_f64, a.up_f64, a.scale)
    slots[2] = slots[4] = None
    ra = layer.row_adapter.copy()
    ra[(ra == 2) | (ra == 4)] = -1
    lay2 = wl.LayerData(layer.name, "bf16", layer.din, layer.dout, layer.X, layer.W, ra, layer.max_slots, [])
    Y = run_layer(lay2, pool)
    assert_within(Y, oracle.forward(layer.X_f64, layer.W_f64, ra, slots), "bf16", "after compaction")
    with pytest.raises(mlora.MloraError) as e:
        pool.load(2, to_device(a.down, "bf16"), to_device(a.up, "bf16"), a.scale)
    assert e.value.status == mlora.MLORA_ERR_OOM


def test_host_sources_for_load():
    layer = wl.random_layer(13, T=20, din=128, dout=96, ranks=[8, 16])
    pool = make_pool(layer, host_sources=True)
    assert_within(run_layer(layer, pool), want_of(layer), "bf16", "host sources")


# --------------------------------------------------------------------------- #
# the checker catches wrong routings on real GPU output (M031 §03)
def test_wrong_routing_is_detected_on_gpu_output():
    layer = wl.decode_step(0)
    Y = run_layer(layer)
    ads = ora_adapters(layer)
    swapped = oracle.forward(layer.X_f64, layer.W_f64, layer.row_adapter, [ads[1], ads[0], ads[2]])
    assert not within(Y, swapped, "bf16").all()
    assert within(Y, want_of(layer), "bf16").all()
