"""Seeded synthetic multi-LoRA batches shaped like the pages' workloads.

Input generation only: random draws, rounding of the draws to the storage dtype
(bf16 round-to-nearest-even or fp32), and the row -> adapter mapping recipes.  It
holds none of the layer's arithmetic.  Both sides consume it: the fp64 oracle
reads the exact fp64 value of every stored element (``*_f64``), the CUDA path
reads the stored payload (bf16 bit patterns as uint16, or float32).

Workloads (the pages publish no dataset; all inputs are synthetic):

* ``worked_example``   -- the four-row example of the ai-infra-kb "M031" tutorial,
  §02/§03: din = dout = 4, rows P(A), Q(B), R(A), S(none), adapter A rank 1,
  adapter B rank 2; values U[-1, 1] in fp32; scale_A = 0.5, scale_B = 2.0.
* ``decode_step``      -- a 32-token decode step split 20/8/4 over three adapters
  (wiblog "vLLM LoRA adapter batch scheduling", section on batch fragmentation);
  4096 -> 4096, rank 16, scale = alpha / r with alpha = 32.
* ``fragmented_decode``-- 256 rows over 64 resident adapters of mixed rank
  8/16/64 (airsota card 四④ lists these ranks), Zipf(1.1) adapter popularity,
  10 % of rows without adapter.
* ``prefill``          -- fused qkv 4096 -> 12288, 16 prompts of 256..1024 tokens
  (wiblog: prompts of hundreds to thousands of tokens) on 8 rank-16 adapters,
  rows in request order.
* ``stack7b``          -- a 7B-shaped decode stack: 32 layers of q, k, v, o
  (4096 -> 4096), gate, up (4096 -> 11008), down (11008 -> 4096); 100 resident
  rank-16 adapters on q and v only (M031 §06 sizes: 0.25 MiB per projection,
  16 MiB per adapter); 128 rows.  As in a transformer layer, q, k and v read one
  input (the attention input) and gate and up another (the MLP input), so a layer
  runs as four projections: fused q|k|v (4096 -> 12288, the q and v adapters of a
  tenant in one slot), o, fused gate|up (4096 -> 22016) and down.

Value distributions for the bf16 workloads: W ~ N(0, 0.02^2), X ~ N(0, 1),
Down ~ N(0, 1/din) (variance 1/din, so that Down @ x has unit scale),
Up ~ N(0, 0.02^2).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

CONFIG_NAMES = ("worked_example", "decode_step", "fragmented_decode", "prefill", "stack7b")
STACK7B_MODULES = (("q", 4096, 4096, True), ("k", 4096, 4096, False), ("v", 4096, 4096, True),
                   ("o", 4096, 4096, False), ("gate", 4096, 11008, False),
                   ("up", 4096, 11008, False), ("down", 11008, 4096, False))
STACK7B_LAYERS = 32
STACK7B_ADAPTERS = 100
STACK7B_T = 128
# the projections of a layer that share an input, in order: (group, din, modules)
STACK7B_GROUPS = (("qkv", 4096, ("q", "k", "v")), ("o", 4096, ("o",)), ("gate_up", 4096, ("gate", "up")),
                  ("down", 11008, ("down",)))


# --------------------------------------------------------------------------- #
# storage rounding
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round to bf16 (round to nearest, ties to even) and return the bit patterns."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact fp64 value of bf16 bit patterns."""
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def payload_to_f64(p: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f64(p)
    return np.asarray(p, np.float32).astype(np.float64)


def _store(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(a)
    return np.ascontiguousarray(a, np.float32)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(entropy=int(seed), spawn_key=tuple(int(k) for k in key)))


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(std)


# --------------------------------------------------------------------------- #
@dataclass
class AdapterData:
    slot: int
    rank: int
    scale: float
    down: np.ndarray          # payload [rank x din]
    up: np.ndarray            # payload [dout x rank]
    dtype: str = "bf16"

    @property
    def down_f64(self) -> np.ndarray:
        return payload_to_f64(self.down, self.dtype)

    @property
    def up_f64(self) -> np.ndarray:
        return payload_to_f64(self.up, self.dtype)


@dataclass
class LayerData:
    """One multi-LoRA linear layer call: Y = X W^T + per-row adapter deltas."""
    name: str
    dtype: str                # "bf16" or "f32"
    din: int
    dout: int
    X: np.ndarray             # payload [T x din]
    W: np.ndarray             # payload [dout x din]
    row_adapter: np.ndarray   # int32 [T], -1 = none
    max_slots: int
    adapters: List[AdapterData] = field(default_factory=list)

    @property
    def T(self) -> int:
        return int(self.X.shape[0])

    @property
    def X_f64(self) -> np.ndarray:
        return payload_to_f64(self.X, self.dtype)

    @property
    def W_f64(self) -> np.ndarray:
        return payload_to_f64(self.W, self.dtype)

    def slot_list(self) -> List[Optional[AdapterData]]:
        out: List[Optional[AdapterData]] = [None] * self.max_slots
        for a in self.adapters:
            out[a.slot] = a
        return out

    @property
    def rank_budget(self) -> int:
        return int(sum(a.rank for a in self.adapters))

    @property
    def max_rank(self) -> int:
        return int(max([a.rank for a in self.adapters] or [1]))


def make_layer(name: str, seed: int, key: Sequence[int], T: int, din: int, dout: int,
               ranks: Sequence[int], scales: Sequence[float], row_adapter: np.ndarray,
               dtype: str = "bf16", max_slots: Optional[int] = None,
               w_std: float = 0.02, x_std: float = 1.0, up_std: float = 0.02,
               down_std: Optional[float] = None, uniform: bool = False) -> LayerData:
    """Draw X, W and one adapter per entry of ``ranks`` (slot = position; rank 0 = empty slot)."""
    S = len(ranks) if max_slots is None else max_slots
    if down_std is None:
        down_std = 1.0 / np.sqrt(din)
    if uniform:
        def draw(rng, shape, std):
            return rng.uniform(-1.0, 1.0, size=shape).astype(np.float32)
    else:
        draw = _normal
    W = _store(draw(_rng(seed, *key, 1), (dout, din), w_std), dtype)
    X = _store(draw(_rng(seed, *key, 2), (T, din), x_std), dtype)
    adapters = []
    for s, (r, sc) in enumerate(zip(ranks, scales)):
        if r <= 0:
            continue
        rng = _rng(seed, *key, 3, s)
        down = _store(draw(rng, (r, din), down_std), dtype)
        up = _store(draw(rng, (dout, r), up_std), dtype)
        adapters.append(AdapterData(slot=s, rank=int(r), scale=float(sc), down=down, up=up, dtype=dtype))
    return LayerData(name=name, dtype=dtype, din=din, dout=dout, X=X, W=W,
                     row_adapter=np.ascontiguousarray(row_adapter, np.int32), max_slots=S,
                     adapters=adapters)


# --------------------------------------------------------------------------- #
# the five workloads
def worked_example(seed: int = 0) -> LayerData:
    """M031 §02/§03: rows P(A), Q(B), R(A), S(none); A rank 1 (slot 0), B rank 2 (slot 1)."""
    return make_layer("worked_example", seed, (0,), T=4, din=4, dout=4, ranks=[1, 2],
                      scales=[0.5, 2.0], row_adapter=np.array([0, 1, 0, -1], np.int32),
                      dtype="f32", uniform=True)


def decode_row_adapter(seed: int) -> np.ndarray:
    ra = np.array([0] * 20 + [1] * 8 + [2] * 4, np.int32)
    return ra[_rng(seed, 1, 0).permutation(ra.shape[0])]


def decode_step(seed: int = 0) -> LayerData:
    """32 decode tokens, adapter counts 20/8/4 over slots 0/1/2, rank 16, scale 32/16."""
    return make_layer("decode_step", seed, (1,), T=32, din=4096, dout=4096, ranks=[16, 16, 16],
                      scales=[2.0, 2.0, 2.0], row_adapter=decode_row_adapter(seed))


def fragmented_ranks(seed: int) -> np.ndarray:
    return _rng(seed, 2, 0).choice(np.array([8, 16, 64]), size=64, p=[0.4, 0.4, 0.2]).astype(np.int32)


def fragmented_row_adapter(seed: int, T: int = 256, n_slots: int = 64, s_zipf: float = 1.1) -> np.ndarray:
    rng = _rng(seed, 2, 1)
    k = np.arange(1, n_slots + 1, dtype=np.float64)
    p = k ** (-s_zipf)
    p /= p.sum()
    ra = (rng.choice(n_slots, size=T, p=p)).astype(np.int32)   # slot = k - 1
    n_none = int(round(0.1 * T))
    ra[rng.choice(T, size=n_none, replace=False)] = -1
    return ra


def fragmented_decode(seed: int = 0) -> LayerData:
    """256 rows, 64 slots with ranks from {8,16,64} (p = .4/.4/.2), Zipf(1.1) ids, 10 % none."""
    ranks = fragmented_ranks(seed)
    return make_layer("fragmented_decode", seed, (2,), T=256, din=4096, dout=4096, ranks=list(ranks),
                      scales=[32.0 / r for r in ranks], row_adapter=fragmented_row_adapter(seed))


def prefill_lengths(seed: int) -> np.ndarray:
    return _rng(seed, 3, 0).integers(256, 1025, size=16).astype(np.int64)


def prefill_row_adapter(seed: int) -> np.ndarray:
    lengths = prefill_lengths(seed)
    return np.concatenate([np.full(int(n), j % 8, np.int32) for j, n in enumerate(lengths)])


def prefill(seed: int = 0) -> LayerData:
    """Fused qkv 4096 -> 12288; 16 prompts of U{256..1024} tokens in request order; request j -> slot j mod 8."""
    ra = prefill_row_adapter(seed)
    return make_layer("prefill", seed, (3,), T=int(ra.shape[0]), din=4096, dout=12288, ranks=[16] * 8,
                      scales=[2.0] * 8, row_adapter=ra)


def stack7b_row_adapter(seed: int) -> np.ndarray:
    """Row t -> slot pi(t mod 100): all 100 adapters used, 28 of them by two rows."""
    pi = _rng(seed, 4, 0).permutation(STACK7B_ADAPTERS).astype(np.int32)
    return pi[np.arange(STACK7B_T) % STACK7B_ADAPTERS]


def stack7b_group_of(module: str) -> int:
    return [i for i, g in enumerate(STACK7B_GROUPS) if module in g[2]][0]


def stack7b_input(seed: int, layer: int, group: int) -> np.ndarray:
    """The input rows [T x din] that the projections of one group of a layer share (bf16 payload)."""
    din = STACK7B_GROUPS[group][1]
    return _store(_normal(_rng(seed, 4, layer, 100 + group), (STACK7B_T, din), 1.0), "bf16")


def stack7b_projection(seed: int, layer: int, module: str) -> LayerData:
    """One projection of the 7B-shaped stack; q and v carry the 100 rank-16 adapters."""
    idx = [m[0] for m in STACK7B_MODULES].index(module)
    _, din, dout, adapted = STACK7B_MODULES[idx]
    ra = stack7b_row_adapter(seed) if adapted else np.full(STACK7B_T, -1, np.int32)
    ranks = [16] * STACK7B_ADAPTERS if adapted else []
    L = make_layer(f"stack7b.L{layer}.{module}", seed, (4, layer, idx), T=STACK7B_T, din=din,
                   dout=dout, ranks=ranks, scales=[2.0] * len(ranks), row_adapter=ra,
                   max_slots=STACK7B_ADAPTERS if adapted else 0)
    L.X = stack7b_input(seed, layer, stack7b_group_of(module))
    return L


@dataclass
class FusedLayerData:
    """Several projections that read one input, run as one projection over their weights
    stacked by rows: module m owns output rows [row_offset[m], row_offset[m] + rows[m]).
    ``tenants[s][m]`` is slot s's adapter of module m (None: not adapted)."""
    name: str
    din: int
    X: np.ndarray                       # payload [T x din]
    W: np.ndarray                       # payload [sum(rows) x din]
    row_adapter: np.ndarray
    modules: List[tuple]                # (row_offset, rows) per module
    tenants: List[List[Optional[AdapterData]]]
    dtype: str = "bf16"

    @property
    def T(self) -> int:
        return int(self.X.shape[0])

    @property
    def dout(self) -> int:
        return int(self.W.shape[0])

    @property
    def max_slots(self) -> int:
        return len(self.tenants)


def stack7b_group(seed: int, layer: int, group: int) -> FusedLayerData:
    """One input group of a 7B-shaped layer as a fused projection (q|k|v, o, gate|up or down)."""
    name, din, mods = STACK7B_GROUPS[group]
    parts = [stack7b_projection(seed, layer, m) for m in mods]
    offsets = np.concatenate([[0], np.cumsum([P.dout for P in parts])[:-1]]).astype(int)
    adapted = any(P.max_slots > 0 for P in parts)
    n_slots = STACK7B_ADAPTERS if adapted else 0
    tenants = []
    for s_ in range(n_slots):
        tenants.append([P.slot_list()[s_] if P.max_slots > 0 else None for P in parts])
    ra = stack7b_row_adapter(seed) if adapted else np.full(STACK7B_T, -1, np.int32)
    return FusedLayerData(name=f"stack7b.L{layer}.{name}", din=din, X=parts[0].X,
                          W=np.ascontiguousarray(np.concatenate([P.W for P in parts], 0)), row_adapter=ra,
                          modules=[(int(o), P.dout) for o, P in zip(offsets, parts)], tenants=tenants)


def by_name(name: str, seed: int = 0) -> LayerData:
    return {"worked_example": worked_example, "decode_step": decode_step,
            "fragmented_decode": fragmented_decode, "prefill": prefill}[name](seed)


def random_layer(seed: int, T: int, din: int, dout: int, ranks: Sequence[int],
                 dtype: str = "bf16", p_none: float = 0.1, scales: Optional[Sequence[float]] = None,
                 row_adapter: Optional[np.ndarray] = None) -> LayerData:
    """A generic seeded case (ragged sizes, mixed ranks) for edge-case tests."""
    S = len(ranks)
    loaded = [s for s, r in enumerate(ranks) if r > 0]
    if row_adapter is None:
        rng = _rng(seed, 9, 0)
        if loaded:
            row_adapter = rng.choice(np.array(loaded, np.int32), size=T).astype(np.int32)
            row_adapter[rng.random(T) < p_none] = -1
        else:
            row_adapter = np.full(T, -1, np.int32)
    if scales is None:
        scales = [(32.0 / r if r > 0 else 0.0) for r in ranks]
    return make_layer(f"random.T{T}.{din}x{dout}", seed, (9, T, din, dout), T=T, din=din, dout=dout,
                      ranks=list(ranks), scales=list(scales), row_adapter=row_adapter, dtype=dtype,
                      max_slots=S)


def oracle_adapters(layer: LayerData):
    """(down_f64, up_f64, scale) per slot, None for empty slots, for the oracle's marshalling."""
    out = []
    for a in layer.slot_list():
        out.append(None if a is None else (a.down_f64, a.up_f64, a.scale))
    return out


# --------------------------------------------------------------------------- #
# device draws for the full 7B-shaped stack (about 13 GB of weights): the same
# recipe and distributions as stack7b_group, drawn by torch's counter-based
# generator on the device instead of numpy on the host (which would take minutes);
# the values differ from the host draws, the shapes and distributions do not.
def _device_gen(device, seed: int, *key: int):
    import torch
    h = int(np.random.SeedSequence(entropy=int(seed), spawn_key=tuple(int(k) for k in key)).generate_state(1)[0])
    g = torch.Generator(device=device)
    g.manual_seed(h)
    return g


def _device_normal(device, shape, std: float, seed: int, *key: int):
    import torch
    g = _device_gen(device, seed, *key)
    return (torch.randn(shape, device=device, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def stack7b_group_device(seed: int, layer: int, group: int, device):
    """Device tensors of one input group of a 7B-shaped layer: X [T x din], the stacked
    W, module row ranges, and per slot the (down, up, scale) of each adapted module."""
    name, din, mods = STACK7B_GROUPS[group]
    X = _device_normal(device, (STACK7B_T, din), 1.0, seed, 5, layer, group, 0)
    Ws, modules, tenants_mods, off = [], [], [], 0
    for m in mods:
        idx = [x[0] for x in STACK7B_MODULES].index(m)
        _, _, dout, adapted = STACK7B_MODULES[idx]
        Ws.append(_device_normal(device, (dout, din), 0.02, seed, 5, layer, group, 1, idx))
        modules.append((off, dout))
        off += dout
        tenants_mods.append(adapted)
    import torch
    W = torch.cat(Ws, 0) if len(Ws) > 1 else Ws[0]
    del Ws
    tenants = []
    if any(tenants_mods):
        for s_ in range(STACK7B_ADAPTERS):
            row = []
            for mi, adapted in enumerate(tenants_mods):
                if not adapted:
                    row.append(None)
                    continue
                rows = modules[mi][1]
                down = _device_normal(device, (16, din), 1.0 / np.sqrt(din), seed, 5, layer, group, 2, mi, s_)
                up = _device_normal(device, (rows, 16), 0.02, seed, 5, layer, group, 3, mi, s_)
                row.append((down, up, 2.0))
            tenants.append(row)
    ra = stack7b_row_adapter(seed) if tenants else np.full(STACK7B_T, -1, np.int32)
    return {"name": f"stack7b.L{layer}.{name}", "X": X, "W": W, "modules": modules, "tenants": tenants,
            "row_adapter": ra, "din": din, "dout": off}


# --------------------------------------------------------------------------- #
# 4-bit NormalFloat base (ai-infra-kb "M031" §05 names restoring W "by scale/codebook"
# and the NF4 codebook; the pages cite the QLoRA paper, which defines the data type)
NF4_BLOCK = 64          # input columns that share one absmax scale


def nf4_codebook() -> np.ndarray:
    """The 16 NormalFloat values, ascending, in fp32: quantiles of the standard normal
    at evenly spaced probabilities from 1/2 up to 1 - delta (delta = (1/32 + 1/30) / 2),
    8 of them on the positive side and 7 on the negative side, each side divided by its
    largest quantile so that the values end at -1 and 1, plus an exact 0."""
    from scipy.stats import norm
    p_max = 1.0 - 0.5 * (1.0 / 32 + 1.0 / 30)
    top = norm.ppf(p_max)
    pos = norm.ppf(np.linspace(0.5, p_max, 9)[1:]) / top
    neg = -norm.ppf(np.linspace(0.5, p_max, 8)[1:]) / top
    return np.sort(np.concatenate([neg, [0.0], pos])).astype(np.float32)


def nf4_random_base(seed: int, dout: int, din: int, key: int = 0):
    """A seeded NF4 base: packed codes [dout x din/2] (column 2m in the low nibble of byte
    m, 2m+1 in the high one) and fp32 block scales [din/64 x dout] ~ |N(0, 0.02)| * 3."""
    rng = _rng(seed, 7, key)
    codes = rng.integers(0, 16, size=(dout, din)).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    absmax = (np.abs(rng.standard_normal((din // NF4_BLOCK, dout))) * 0.06 + 1e-3).astype(np.float32)
    return packed, absmax
