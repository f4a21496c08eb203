"""Pins of the fp64 oracle against facts other than the oracle itself (CPU only).

Each test names what it is pinned to: a fact the pages print (tests/golden/), a
library routine on a special case, an identity of the mathematics, or brute
force on a tiny case.  Together they make a dropped term, a wrong sign or index,
a transposed operand or a mis-ordered writeback in the oracle fail at least one
test.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.tolerance import within

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("=", 1))
                out[k] = v
    return out


def adapters_of(layer):
    return [None if a is None else oracle.OracleAdapter(a.down_f64, a.up_f64, a.scale)
            for a in layer.slot_list()]


def run(layer, rows=None, adapters=None, row_adapter=None):
    ads = adapters_of(layer) if adapters is None else adapters
    ra = layer.row_adapter if row_adapter is None else row_adapter
    return oracle.forward(layer.X_f64, layer.W_f64, ra, ads, rows=rows)


# --------------------------------------------------------------------------- #
# worked example (M031 §02/§03): values printed on the page
def _worked_golden():
    g = read_golden("worked_example.txt")
    names = g["rows"].split()
    slot = {"A": 0, "B": 1}
    ra = np.array([slot.get(a, -1) for a in g["row_adapter"].split()], np.int32)
    ranks = {k: int(v) for k, v in (kv.split(":") for kv in g["rank"].split())}
    return g, names, ra, ranks


def test_worked_example_matches_generator():
    g, names, ra, ranks = _worked_golden()
    layer = wl.worked_example(0)
    assert layer.din == int(g["din"]) and layer.dout == int(g["dout"])
    assert np.array_equal(layer.row_adapter, ra)
    assert [a.rank for a in layer.adapters] == [ranks["A"], ranks["B"]]


def test_worked_example_group_order():
    g, names, ra, ranks = _worked_golden()
    counts, offsets, perm, bad = oracle.segments(ra, np.array([ranks["A"], ranks["B"]], np.int32))
    assert [names[i] for i in perm] == g["group_order"].split()
    assert list(counts) == [2, 1] and list(offsets) == [0, 2, 3] and bad == 0


def test_worked_example_flops():
    g, names, ra, ranks = _worked_golden()
    r = np.array([ranks["A"], ranks["B"]], np.int32)
    exact, padded = oracle.lora_flops(ra, r, int(g["din"]), int(g["dout"]))
    assert exact == int(g["flops_total"])
    assert padded == int(g["flops_padded"])
    per = dict(kv.split(":") for kv in g["flops_group"].split())
    for name, s in (("A", 0), ("B", 1)):
        only = np.where(ra == s, ra, -1).astype(np.int32)
        assert oracle.lora_flops(only, r, 4, 4)[0] == int(per[name])


def test_worked_example_writeback_rows():
    """A's delta lands on rows 0 and 2, B's on row 1, row 3 keeps the base output."""
    g, names, ra, ranks = _worked_golden()
    layer = wl.worked_example(0)
    Y = run(layer)
    base = layer.X_f64 @ layer.W_f64.T
    delta = Y - base
    wb = dict(kv.split(":") for kv in g["writeback"].split())
    rows_of = {k: [int(x) for x in v.split(",")] for k, v in wb.items()}
    assert np.all(delta[rows_of["-"]] == 0.0)
    A, B = layer.adapters
    for name, ad in (("A", A), ("B", B)):
        for t in rows_of[name]:
            want = ad.scale * ad.up_f64 @ (ad.down_f64 @ layer.X_f64[t])
            np.testing.assert_allclose(delta[t], want, rtol=1e-12, atol=1e-14)


def test_worked_example_brute_force_exact():
    """Exact rational arithmetic through the merged weight of each row's adapter (M031 §04)."""
    layer = wl.worked_example(3)
    Y = run(layer)
    X = [[Fraction(float(v)) for v in row] for row in layer.X_f64]
    W = [[Fraction(float(v)) for v in row] for row in layer.W_f64]
    slots = layer.slot_list()
    for t in range(layer.T):
        a = int(layer.row_adapter[t])
        Wt = [row[:] for row in W]
        if a >= 0:
            ad = slots[a]
            D = [[Fraction(float(v)) for v in row] for row in ad.down_f64]
            U = [[Fraction(float(v)) for v in row] for row in ad.up_f64]
            s = Fraction(ad.scale)
            for o in range(layer.dout):
                for i in range(layer.din):
                    Wt[o][i] += s * sum(U[o][k] * D[k][i] for k in range(ad.rank))
        for o in range(layer.dout):
            exact = sum(Wt[o][i] * X[t][i] for i in range(layer.din))
            assert abs(Fraction(Y[t, o]) - exact) <= Fraction(1, 10 ** 14) * (1 + abs(exact))


# --------------------------------------------------------------------------- #
# special cases that reduce to a library routine
def test_rows_without_adapter_equal_library_matmul():
    layer = wl.random_layer(11, T=37, din=72, dout=56, ranks=[8, 0, 16, 24], p_none=0.4)
    Y = run(layer)
    none = layer.row_adapter < 0
    assert none.any() and (~none).any()
    ref = layer.X_f64 @ layer.W_f64.T
    np.testing.assert_allclose(Y[none], ref[none], rtol=1e-12, atol=1e-12)
    assert not np.allclose(Y[~none], ref[~none], rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("slot", [0, 2, 3])
def test_single_adapter_batch_equals_merged_weight(slot):
    """M031 §04: W_merged_a x = W x + s_a Up_a (Down_a x); checked with numpy's matmul."""
    layer = wl.random_layer(12, T=19, din=64, dout=40, ranks=[8, 0, 16, 24],
                            row_adapter=np.full(19, slot, np.int32))
    ad = layer.slot_list()[slot]
    Wm = layer.W_f64 + ad.scale * (ad.up_f64 @ ad.down_f64)
    np.testing.assert_allclose(run(layer), layer.X_f64 @ Wm.T, rtol=1e-11, atol=1e-11)


def test_merge_matches_library():
    layer = wl.random_layer(13, T=1, din=48, dout=24, ranks=[16])
    ad = layer.adapters[0]
    got = oracle.merge(layer.W_f64, oracle.OracleAdapter(ad.down_f64, ad.up_f64, ad.scale))
    want = layer.W_f64 + ad.scale * (ad.up_f64 @ ad.down_f64)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-14)


def test_merge_serves_only_its_adapter():
    """M031 §04: the merged A weight reproduces A's rows and gets B's rows wrong."""
    layer = wl.decode_step(0)
    ads = adapters_of(layer)
    Wa = oracle.merge(layer.W_f64, ads[0])
    rows_a = np.flatnonzero(layer.row_adapter == 0)
    rows_b = np.flatnonzero(layer.row_adapter == 1)
    Y = run(layer)
    Xa = layer.X_f64
    assert within(Xa[rows_a] @ Wa.T, Y[rows_a], "bf16").all()
    assert np.allclose(Xa[rows_a] @ Wa.T, Y[rows_a], rtol=1e-9, atol=1e-9)
    assert not within(Xa[rows_b] @ Wa.T, Y[rows_b], "bf16").all()


def test_unmerge_subtracts_the_update():
    """airsota card, section 四 item ③: switching a merged weight back re-subtracts the
    adapter's update: unmerge(W) x = W x - s Up (Down x), checked with numpy's matmul
    on a random vector (a wrong sign, a transposed Up or Down, or a dropped scale fails)."""
    layer = wl.random_layer(15, T=1, din=56, dout=36, ranks=[12])
    ad = layer.adapters[0]
    Wu = oracle.unmerge(layer.W_f64, oracle.OracleAdapter(ad.down_f64, ad.up_f64, ad.scale))
    x = np.random.default_rng(3).standard_normal(56)
    want = layer.W_f64 @ x - ad.scale * (ad.up_f64 @ (ad.down_f64 @ x))
    np.testing.assert_allclose(Wu @ x, want, rtol=1e-12, atol=1e-12)


def test_unmerge_after_merge_restores_only_with_the_same_adapter():
    """The un-merge of the adapter that was merged returns the original weight (fp64:
    to rounding); un-merging another adapter does not."""
    layer = wl.random_layer(16, T=1, din=40, dout=24, ranks=[16, 8])
    a, b = adapters_of(layer)
    Wm = oracle.merge(layer.W_f64, a)
    np.testing.assert_allclose(oracle.unmerge(Wm, a), layer.W_f64, rtol=0, atol=1e-13)
    assert np.abs(oracle.unmerge(Wm, b) - layer.W_f64).max() > 1e-3


def _module_case():
    rng = np.random.default_rng(17)
    din, modules = 24, [(0, 10), (10, 7), (17, 11)]          # q, k, v rows of a 28-row fused projection
    W = rng.standard_normal((28, din))
    X = rng.standard_normal((9, din))
    def ad(r, n, s):
        return oracle.OracleAdapter(rng.standard_normal((r, din)), rng.standard_normal((n, r)), s)
    tenants = [[ad(2, 10, 2.0), None, ad(3, 11, 0.5)],       # q and v
               [None, ad(4, 7, 1.5), None],                   # k only
               None]                                          # slot 2 empty
    ra = np.array([0, 1, -1, 0, 2, 1, 0, -1, 1], np.int32)
    return X, W, ra, modules, tenants


def test_module_rows_follow_their_own_adapters():
    """airsota card, section 四 item ④ (adapters of different target modules): in a
    fused projection, each module's rows get that module's own update, checked row by
    row with numpy; rows of other modules, invalid or empty slots keep the base."""
    X, W, ra, modules, tenants = _module_case()
    Y = oracle.forward_modules(X, W, ra, modules, tenants)
    want = X @ W.T
    for t, s in enumerate(ra):
        if s < 0 or tenants[s] is None:
            continue
        for (off, n), a in zip(modules, tenants[s]):
            if a is not None:
                want[t, off:off + n] += a.scale * (a.up @ (a.down @ X[t]))
    np.testing.assert_allclose(Y, want, rtol=1e-12, atol=1e-12)


def test_one_module_over_all_rows_is_the_plain_layer():
    X, W, ra, _, tenants = _module_case()
    a = oracle.OracleAdapter(tenants[0][0].down, np.random.default_rng(5).standard_normal((28, 2)), 2.0)
    np.testing.assert_array_equal(oracle.forward_modules(X, W, ra, [(0, 28)], [[a], None, None]),
                                  oracle.forward(X, W, ra, [a, None, None]))


def test_quantize_recovers_an_exact_grid():
    """M031 §05 (a quantized base is codes times a scale): codes whose row maximum is
    127, times power-of-two row scales, quantize back to themselves exactly; an
    all-zero row gets scale 0 and codes 0."""
    rng = np.random.default_rng(21)
    codes = rng.integers(-127, 128, size=(6, 40)).astype(np.int8)
    codes[:, 3] = 127
    codes[5] = 0
    scale = 2.0 ** rng.integers(-9, -2, size=6)
    scale[5] = 0.0
    c2, s2 = oracle.quantize(oracle.dequantize(codes, scale))
    np.testing.assert_array_equal(c2, codes)
    np.testing.assert_array_equal(s2, scale.astype(np.float32))


def test_quantize_sends_exact_ties_to_the_even_code():
    """Rounding to nearest with ties to even (IEEE 754 roundTiesToEven, the rule the
    kernels' fp32 rounding uses): a row whose maximum is 127 units and whose other
    weights sit exactly halfway between two units gets the even neighbour for each --
    2.5 -> 2, 3.5 -> 4, -0.5 -> 0, -1.5 -> -2."""
    unit = 2.0 ** -6
    row = np.array([127.0, 2.5, 3.5, -0.5, -1.5, 126.5, -126.5, 0.5]) * unit
    codes, scale = oracle.quantize(row[None, :])
    assert scale[0] == np.float32(unit)
    np.testing.assert_array_equal(codes[0], [127, 2, 4, 0, -2, 126, -126, 0])


def test_quantization_error_is_at_most_half_a_step():
    W = np.random.default_rng(22).standard_normal((9, 70)) * 0.02
    codes, scale = oracle.quantize(W)
    err = np.abs(oracle.dequantize(codes, scale) - W)
    assert (err <= scale[:, None] / 2 * (1 + 2.0 ** -20) + 2.0 ** -23 * np.abs(W)).all()
    assert np.abs(codes).max() == 127


def test_merge_on_a_quantized_base_three_ways():
    """M031 §05 acceptance: the dynamic branch over the restored base equals the merged
    float weight (fp64), the re-quantized merge stays within half a step per weight,
    and adding the update to the codes (ignoring the scale) does not."""
    rng = np.random.default_rng(23)
    codes, scale = oracle.quantize(rng.standard_normal((24, 32)) * 0.02)
    a = oracle.OracleAdapter(rng.standard_normal((4, 32)) / 8, rng.standard_normal((24, 4)) * 0.05, 2.0)
    X = rng.standard_normal((5, 32))
    Wd = oracle.dequantize(codes, scale)
    dynamic = oracle.forward(X, Wd, np.zeros(5, np.int32), [a])
    merged_float = X @ (Wd + a.scale * a.up @ a.down).T
    np.testing.assert_allclose(dynamic, merged_float, rtol=1e-12, atol=1e-12)
    c2, s2 = oracle.merge_quantized(codes, scale, a)
    quantized = X @ oracle.dequantize(c2, s2).T
    bound = np.abs(X) @ np.broadcast_to(s2[:, None] / 2 * (1 + 2.0 ** -20), (24, 32)).T + 1e-9
    assert (np.abs(quantized - merged_float) <= bound).all()
    wrong = oracle.dequantize(np.clip(np.rint(codes + a.scale * a.up @ a.down), -127, 127), scale)
    assert np.abs(X @ wrong.T - merged_float).max() > 10 * bound.max()


# --------------------------------------------------------------------------- #
# invariants and closed forms
# --------------------------------------------------------------------------- #
# NF4 base (M031 §05: W restored "by scale/codebook"; the NF4 codebook)
def test_nf4_codebook_is_the_normal_float_definition():
    """16 ascending values with an exact 0 and ends -1 and 1; under the normal CDF the
    positive values (times the top quantile) sit at evenly spaced probabilities between
    1/2 and 1 - delta, 8 steps, and the negative ones at 7 such steps (the NormalFloat
    construction the pages' source defines)."""
    from scipy.stats import norm
    cb = wl.nf4_codebook().astype(np.float64)
    assert cb.shape == (16,) and np.all(np.diff(cb) > 0)
    assert cb[0] == -1.0 and cb[15] == 1.0 and cb[7] == 0.0
    p_max = 1.0 - 0.5 * (1.0 / 32 + 1.0 / 30)
    top = norm.ppf(p_max)
    pos = norm.cdf(cb[8:] * top)
    neg = norm.cdf(-cb[:7][::-1] * top)
    np.testing.assert_allclose(np.diff(np.concatenate([[0.5], pos])), (p_max - 0.5) / 8, rtol=1e-5)
    np.testing.assert_allclose(np.diff(np.concatenate([[0.5], neg])), (p_max - 0.5) / 7, rtol=1e-5)


def test_nf4_packing_puts_even_columns_in_the_low_nibble():
    codes = np.array([[1, 2, 15, 0, 7, 9]], np.uint8)
    packed = oracle.nf4_pack(codes)
    np.testing.assert_array_equal(packed, [[0x21, 0x0F, 0x97]])
    np.testing.assert_array_equal(oracle.nf4_unpack(packed), codes)


def test_nf4_quantize_recovers_an_exact_grid():
    """Codebook values times power-of-two block scales, with a +-1 entry in every block
    (so that the block's absmax is its scale), quantize back to the same codes and
    scales; restoring gives the weights exactly.  An all-zero block gets absmax 0 and
    the code of 0."""
    cb = wl.nf4_codebook()
    rng = np.random.default_rng(31)
    codes = rng.integers(0, 16, size=(5, 192)).astype(np.uint8)
    codes[:, ::64] = rng.choice([0, 15], size=(5, 3))
    scale = (2.0 ** rng.integers(-9, -3, size=(3, 5))).astype(np.float32)
    codes[4, 64:128] = 7
    scale[1, 4] = 0.0
    W = oracle.nf4_dequantize(oracle.nf4_pack(codes), scale, cb)
    pk, am = oracle.nf4_quantize(W, cb)
    np.testing.assert_array_equal(oracle.nf4_unpack(pk), codes)
    np.testing.assert_array_equal(am, scale)
    np.testing.assert_array_equal(oracle.nf4_dequantize(pk, am, cb), W)
    assert np.all(W[4, 64:128] == 0.0)


def test_nf4_ties_go_to_the_lower_code():
    """A value exactly halfway between two codebook entries takes the lower code; the
    next fp32 value above it, the upper one (a synthetic codebook of eighths, where the
    halfway points and the distances are exact in fp32)."""
    cb = (np.arange(-8, 8) / 8.0).astype(np.float32)
    row = np.zeros((1, 64), np.float64)
    row[0, 0] = 1.0                                                    # absmax 1: w / absmax = w exactly
    row[0, 1] = -0.5625                                                # halfway between -0.625 (3) and -0.5 (4)
    row[0, 2] = np.nextafter(np.float32(-0.5625), np.float32(1))
    row[0, 3] = 0.0625                                                 # halfway between 0 (8) and 0.125 (9)
    pk, am = oracle.nf4_quantize(row, cb)
    c = oracle.nf4_unpack(pk)[0]
    assert am[0, 0] == 1.0
    assert (c[0], c[1], c[2], c[3]) == (15, 3, 4, 8)


def test_nf4_error_is_at_most_half_the_widest_gap():
    cb = wl.nf4_codebook()
    W = np.random.default_rng(32).standard_normal((7, 256)) * 0.02
    pk, am = oracle.nf4_quantize(W, cb)
    err = np.abs(oracle.nf4_dequantize(pk, am, cb) - W)
    half_gap = np.max(np.diff(cb.astype(np.float64))) / 2
    bound = np.repeat(am.T.astype(np.float64), 64, axis=1) * half_gap * (1 + 2.0 ** -18) + 2.0 ** -23 * np.abs(W)
    assert (err <= bound).all()


def test_nf4_merge_three_ways():
    """M031 §05 acceptance on an NF4 base: the dynamic branch over the restored base
    equals the merged float weight (fp64), the re-quantized merge stays within half the
    widest codebook gap per weight, and adding the update to the codes does not."""
    cb = wl.nf4_codebook()
    rng = np.random.default_rng(33)
    pk, am = oracle.nf4_quantize(rng.standard_normal((24, 128)) * 0.02, cb)
    a = oracle.OracleAdapter(rng.standard_normal((4, 128)) / 8, rng.standard_normal((24, 4)) * 0.05, 2.0)
    X = rng.standard_normal((5, 128))
    Wd = oracle.nf4_dequantize(pk, am, cb)
    dynamic = oracle.forward(X, Wd, np.zeros(5, np.int32), [a])
    merged_float = X @ (Wd + a.scale * a.up @ a.down).T
    np.testing.assert_allclose(dynamic, merged_float, rtol=1e-12, atol=1e-12)
    pk2, am2 = oracle.nf4_merge(pk, am, cb, a)
    half_gap = np.max(np.diff(cb.astype(np.float64))) / 2
    per_w = np.repeat(am2.T.astype(np.float64), 64, axis=1) * half_gap * (1 + 2.0 ** -18) + 1e-9
    assert (np.abs(oracle.nf4_dequantize(pk2, am2, cb) - (Wd + a.scale * a.up @ a.down)) <= per_w).all()
    # the update added to the codes (ignoring scale and codebook) rounds away: most weights
    # then miss the merged value by more than the bound the right way keeps
    wrong = oracle.nf4_dequantize(oracle.nf4_pack(np.clip(np.rint(
        oracle.nf4_unpack(pk) + a.scale * a.up @ a.down), 0, 15).astype(np.uint8)), am, cb)
    assert np.mean(np.abs(wrong - (Wd + a.scale * a.up @ a.down)) > per_w) > 0.2


def test_rank_padding_leaves_output_unchanged():
    """M031 §03: giving an adapter zero rows/columns up to the max rank costs FLOPs, not values."""
    layer = wl.random_layer(14, T=23, din=40, dout=32, ranks=[4, 12, 16], p_none=0.2)
    ads = adapters_of(layer)
    r_max = max(a.rank for a in ads if a is not None)
    padded = []
    for a in ads:
        d = np.zeros((r_max, layer.din)); d[:a.rank] = a.down
        u = np.zeros((layer.dout, r_max)); u[:, :a.rank] = a.up
        padded.append(oracle.OracleAdapter(d, u, a.scale))
    np.testing.assert_allclose(run(layer, adapters=padded), run(layer), rtol=1e-13, atol=1e-13)


def test_permutation_equivariance():
    layer = wl.random_layer(15, T=29, din=24, dout=20, ranks=[8, 16, 0, 8], p_none=0.25)
    Y = run(layer)
    p = np.random.default_rng(0).permutation(layer.T)
    ads = adapters_of(layer)
    Yp = oracle.forward(layer.X_f64[p], layer.W_f64, layer.row_adapter[p], ads)
    np.testing.assert_array_equal(Yp, Y[p])
    ranks = oracle.slot_ranks(ads)
    _, off, perm, _ = oracle.segments(layer.row_adapter, ranks)
    _, offp, permp, _ = oracle.segments(layer.row_adapter[p], ranks)
    assert np.array_equal(off, offp)
    inv = np.argsort(p)
    for s in range(len(ads)):   # each segment holds the same rows, renamed, in ascending order
        assert sorted(p[permp[offp[s]:offp[s + 1]]].tolist()) == perm[off[s]:off[s + 1]].tolist()
        assert np.all(np.diff(permp[offp[s]:offp[s + 1]]) > 0)
    del inv


def test_rank1_unit_adapter_closed_form():
    """Down = e_j (rank 1), Up = u  =>  delta_t = s * u * x_t[j]; integer data, exact."""
    rng = np.random.default_rng(5)
    T, din, dout, j, s = 6, 9, 7, 4, 0.75
    X = rng.integers(-5, 6, (T, din)).astype(np.float64)
    W = rng.integers(-3, 4, (dout, din)).astype(np.float64)
    u = rng.integers(-4, 5, (dout, 1)).astype(np.float64)
    d = np.zeros((1, din)); d[0, j] = 1.0
    ra = np.array([0, -1, 0, 0, -1, 0], np.int32)
    Y = oracle.forward(X, W, ra, [oracle.OracleAdapter(d, u, s)])
    want = X @ W.T
    want[ra == 0] += s * np.outer(X[ra == 0, j], u[:, 0])
    np.testing.assert_array_equal(Y, want)
    # a basis base weight picks one input coordinate per output
    E = np.zeros((dout, din)); E[2, 5] = 1.0
    Y0 = oracle.forward(X, E, None, [])
    assert np.array_equal(Y0[:, 2], X[:, 5]) and np.count_nonzero(Y0[:, [0, 1, 3, 4, 5, 6]]) == 0


def test_zero_scale_and_zero_input():
    layer = wl.random_layer(16, T=10, din=16, dout=8, ranks=[8, 8], p_none=0.0)
    ads = [oracle.OracleAdapter(a.down, a.up, 0.0) for a in adapters_of(layer)]
    np.testing.assert_allclose(run(layer, adapters=ads), layer.X_f64 @ layer.W_f64.T, rtol=1e-13, atol=1e-13)
    Z = oracle.forward(np.zeros((3, 16)), layer.W_f64, np.array([0, 1, -1], np.int32), adapters_of(layer))
    assert np.all(Z == 0.0)


def test_segments_match_sorted_definition():
    rng = np.random.default_rng(7)
    for trial in range(200):
        S = int(rng.integers(0, 9))
        T = int(rng.integers(0, 60))
        ranks = rng.integers(0, 3, S).astype(np.int32) * 8
        ra = rng.integers(-2, S + 2, T).astype(np.int32)
        counts, offsets, perm, bad = oracle.segments(ra, ranks, S)
        valid = [t for t in range(T) if 0 <= ra[t] < S and ranks[ra[t]] > 0]
        want = sorted(valid, key=lambda t: (ra[t], t))
        assert perm.tolist() == want
        assert bad == sum(1 for t in range(T) if ra[t] != -1 and t not in valid)
        for s in range(S):
            assert counts[s] == sum(1 for t in valid if ra[t] == s)
            assert offsets[s + 1] - offsets[s] == counts[s]
        assert offsets[0] == 0 and offsets[S] == len(valid)


def test_invalid_ids_keep_base_output():
    layer = wl.random_layer(17, T=8, din=16, dout=8, ranks=[8, 0, 8],
                            row_adapter=np.array([0, 1, 2, 3, -1, 7, -5, 2], np.int32))
    Y = run(layer)
    base = layer.X_f64 @ layer.W_f64.T
    for t in (1, 3, 4, 5, 6):     # unloaded slot 1, out of range 3/7/-5, and -1
        np.testing.assert_allclose(Y[t], base[t], rtol=1e-13, atol=1e-13)
    _, _, perm, bad = oracle.segments(layer.row_adapter, oracle.slot_ranks(adapters_of(layer)))
    assert perm.tolist() == [0, 2, 7] and bad == 4


# --------------------------------------------------------------------------- #
# wrong routings must be caught by the acceptance rule (M031 §03, wiblog naive mixing)
def test_wrong_routings_fail_tolerance():
    layer = wl.decode_step(0)
    Y = run(layer)
    ads = adapters_of(layer)
    # (i) adapters A and B swapped in their slots
    swapped = [ads[1], ads[0], ads[2]]
    assert not within(run(layer, adapters=swapped), Y, "bf16").all()
    # (ii) compacted writeback: grouped outputs written to the first rows instead of their own
    _, _, perm, _ = oracle.segments(layer.row_adapter, oracle.slot_ranks(ads))
    compact = Y.copy()
    compact[: perm.size] = Y[perm]
    assert not within(compact, Y, "bf16").all()
    # (iii) one shared adapter for the whole mixed batch
    shared = run(layer, row_adapter=np.zeros(layer.T, np.int32))
    assert not within(shared, Y, "bf16").all()
    # and the delta is well above the tolerance, so a dropped branch is caught too
    base = layer.X_f64 @ layer.W_f64.T
    ok = within(base, Y, "bf16")[layer.row_adapter >= 0]
    assert not ok.all(axis=1).any()          # every adapted row fails somewhere
    assert ok.mean() < 0.5                   # most of its elements fail


# --------------------------------------------------------------------------- #
# the generator's recipes
def test_adapter_sizes_golden():
    g = read_golden("adapter_sizes.txt")
    p = wl.stack7b_projection(0, 0, "q")
    a = p.adapters[0]
    per_proj = (a.down.nbytes + a.up.nbytes) / 2 ** 20
    assert a.rank == int(g["rank"]) and a.down.itemsize == int(g["bytes_per_param"])
    assert per_proj == float(g["mib_per_projection"])
    per_adapter = per_proj * int(g["layers"]) * int(g["projections_per_layer"])
    assert per_adapter == float(g["mib_per_adapter"])
    assert per_adapter * int(g["resident_adapters"]) == float(g["mib_resident"])
    assert len(p.adapters) == int(g["resident_adapters"])


def test_workload_recipes():
    d = wl.decode_step(0)
    assert d.T == 32 and sorted(np.bincount(d.row_adapter).tolist()) == [4, 8, 20]
    f = wl.fragmented_decode(0)
    assert f.T == 256 and int((f.row_adapter < 0).sum()) == 26
    assert set(a.rank for a in f.adapters) <= {8, 16, 64} and len(f.adapters) == 64
    lengths = wl.prefill_lengths(0)
    assert lengths.size == 16 and lengths.min() >= 256 and lengths.max() <= 1024
    ra = wl.prefill_row_adapter(0)
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    assert all(ra[s] == j % 8 for j, s in enumerate(starts))
    s7 = wl.stack7b_row_adapter(0)
    assert s7.size == 128 and len(set(s7.tolist())) == 100
    assert sorted(np.bincount(s7).tolist()).count(2) == 28


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.140625, 1e-3], np.float32)
    got = wl.bf16_bits_to_f64(wl.f32_to_bf16_bits(vals))
    assert got[0] == 1.0 and got[1] == 1.0            # tie -> even
    assert got[2] == 1.0 + 4 * 2 ** -8                 # tie -> even (up)
    assert got[3] == -2.5 and got[4] == 3.140625
    assert abs(got[5] - 1e-3) <= 2 ** -9 * 1e-3
