"""Decode step over a paged K/V cache (attn_decode_paged) against the fp64
oracle's decode: one or several new tokens per sequence, context lengths from
0 to several key tiles, GQA groups from 1 to 64 heads, window / soft-cap /
ALiBi; plus determinism, independence of the block placement and the
device-side bounds report."""
import numpy as np
import pytest
import torch

import attn_inputs as gen
from oracle import attn64
from gpu_common import LSE_TOL, O_TOL, default_scale, lib, max_abs, record

pytestmark = pytest.mark.gpu

# (B, Hq, Hkv, max_len, lens or None (uniform in [1, max_len]), mods, new tokens per sequence[, d])
CASES = [
    (3, 16, 2, 1500, None, dict(alibi=True), 1, 64),              # d = 64, general layout
    (4, 16, 8, 700, [700, 1, 300, 129], dict(window=200), 3, 64),  # d = 64, compact layout, 3 tokens
    (4, 32, 8, 700, None, {}, 1),                                  # many chunks per sequence
    (3, 32, 2, 1024, [1000, 1, 333], dict(window=300, softcap=20.0, alibi=True), 1),
    (2, 4, 4, 256, [129, 256], {}, 1),                             # G = 1, exact tile multiple
    (1, 64, 1, 520, [517], dict(alibi=True), 1),                  # G = 64: two softmax warps
    (3, 16, 2, 96, [0, 50, 96], dict(window=7), 1),               # an empty sequence
    (5, 24, 8, 2048, None, dict(softcap=30.0), 1),                 # G = 3
    (4, 32, 8, 900, None, {}, 4),                                  # 4 tokens: 16 rows per item
    (3, 16, 8, 600, [600, 2, 130], dict(window=50, alibi=True), 3),  # 6 rows; a token before the cache start
    (2, 32, 2, 300, [300, 257], dict(softcap=20.0), 8),           # 128 rows: all four softmax warps
    (2, 16, 2, 800, None, {}, 2, 64),                              # d = 64, 16 rows: four-group tiles
    (3, 32, 4, 1000, [1000, 5, 640], dict(window=300), 4),         # 32 rows: four-group tiles, full
]


def _ids(c):
    B, Hq, Hkv, n, lens, m, T = c[:7]
    d = c[7] if len(c) > 7 else 128
    return f"B{B}_H{Hq}x{Hkv}_L{n}_T{T}_d{d}_" + ("-".join(m) or "none")


def _run(ea, x, mods, scale):
    dev = {k: (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).cuda() for k, v in x.items()}
    o, lse = ea.decode_paged(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"], dev["seqlens"],
                             scale, mods)
    ea.attn_status()
    return o, lse


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_decode_matches_oracle(case):
    ea = lib()
    B, Hq, Hkv, n, lens, mk, T = case[:7]
    d = case[7] if len(case) > 7 else 128
    x = gen.paged_decode_inputs(B, Hq, Hkv, n, d, seed=900 + n, lens=lens, q_len=T)
    s = default_scale(d)
    o, lse = _run(ea, x, ea.make_mods(causal=True, **mk), s)
    O, L = attn64.decode_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["seqlens"], s,
                               attn64.Mods(causal=True, **mk))
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    empty = np.isneginf(L)  # tokens without any key
    assert np.all(og[empty] == 0.0) and np.all(np.isneginf(lg[empty]))
    eo, el = max_abs(og[~empty], O[~empty]), max_abs(lg[~empty], L[~empty])
    record("decode_cases", "O_max_abs", eo)
    record("decode_cases", "LSE_max_abs", el)
    assert eo <= O_TOL and el <= LSE_TOL, (eo, el)


def test_decode_deterministic_and_placement_free():
    """Two runs agree bit for bit, and so does a cache with the blocks moved
    to other physical slots (the table moved with them)."""
    ea = lib()
    B, Hq, Hkv, n = 6, 32, 4, 3000
    x = gen.paged_decode_inputs(B, Hq, Hkv, n, 128, seed=41)
    s = default_scale(128)
    m = ea.make_mods(alibi=True)
    o1, l1 = _run(ea, x, m, s)
    o2, l2 = _run(ea, x, m, s)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    perm = np.random.default_rng(2).permutation(x["k_cache"].shape[0])
    moved = dict(x)
    for name in ("k_cache", "v_cache"):
        c = torch.empty_like(x[name])
        c[torch.from_numpy(perm)] = x[name]
        moved[name] = c
    t = x["block_table"]
    moved["block_table"] = np.where(t >= 0, perm[np.maximum(t, 0)], -1).astype(np.int32)
    o3, l3 = _run(ea, moved, m, s)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_decode_full_workload_sampled():
    """The benchmarked decode workload, checked on sampled sequences."""
    ea = lib()
    cfg = dict(gen.WORKLOADS["paged_decode_8k"])
    x = gen.paged_decode_inputs(**cfg)
    s = default_scale(cfg["d"])
    o, lse = _run(ea, x, None, s)
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(og).all() and np.isfinite(lg).all()
    for b in (0, 17, cfg["B"] - 1):
        sub = dict(q=x["q"][b:b + 1], block_table=x["block_table"][b:b + 1], seqlens=x["seqlens"][b:b + 1])
        O, L = attn64.decode_paged(sub["q"], x["k_cache"], x["v_cache"], sub["block_table"], sub["seqlens"], s)
        eo, el = max_abs(og[b], O[0]), max_abs(lg[b], L[0])
        record("paged_decode_8k", "O_max_abs", eo)
        record("paged_decode_8k", "LSE_max_abs", el)
        assert eo <= O_TOL and el <= LSE_TOL, (b, eo, el)


def test_decode_bad_table_entry_reports_bounds():
    """A table entry outside [0, num_blocks) is caught by the kernel's own
    check and reported through attn_status; the library stays usable."""
    ea = lib()
    B, Hq, Hkv, n = 2, 8, 2, 200
    x = gen.paged_decode_inputs(B, Hq, Hkv, n, 128, seed=5, lens=[200, 100])
    bad = dict(x)
    bad["block_table"] = x["block_table"].copy()
    bad["block_table"][1, 3] = x["k_cache"].shape[0]  # one past the last block
    dev = {k: (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).cuda() for k, v in bad.items()}
    ea.decode_paged(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"], dev["seqlens"], 0.1)
    with pytest.raises(ea.AttnError) as err:
        ea.attn_status()
    assert err.value.status == 7  # ATTN_ERR_BOUNDS
    o, lse = _run(ea, x, None, 0.1)  # clean call afterwards
    O, L = attn64.decode_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["seqlens"], 0.1)
    assert max_abs(o.float().cpu().numpy(), O) <= O_TOL


def _random_case(i):
    rng = np.random.default_rng(5000 + i)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 8, 16]))
    T = int(rng.choice([1, 1, 2, 3, 4]))
    while G * T > 128:
        T -= 1
    B = int(rng.integers(1, 6))
    n = int(rng.choice([16, 100, 128, 129, 640, 1500]))
    lens = rng.integers(0, n + 1, size=B)
    lens[0] = n  # one sequence fills its table row exactly
    mk = {}
    if rng.random() < 0.5:
        mk["window"] = int(rng.choice([1, 37, 128, 4000]))
    if rng.random() < 0.4:
        mk["softcap"] = float(rng.choice([5.0, 30.0]))
    if rng.random() < 0.4:
        mk["alibi"] = True
    return B, G * Hkv, Hkv, n, [int(x) for x in lens], mk, T


@pytest.mark.parametrize("i", range(16))
def test_decode_random_shapes(i):
    """Seeded random shapes: GQA groups x tokens on both sides of the compact
    layout (8 rows), lengths 0 .. a full table row, every mod combination."""
    ea = lib()
    B, Hq, Hkv, n, lens, mk, T = _random_case(i)
    x = gen.paged_decode_inputs(B, Hq, Hkv, n, 128, seed=7000 + i, lens=lens, q_len=T)
    s = default_scale(128)
    o, lse = _run(ea, x, ea.make_mods(**mk), s)
    O, L = attn64.decode_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["seqlens"], s,
                               attn64.Mods(**mk))
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    empty = np.isneginf(L)
    assert np.all(og[empty] == 0.0) and np.all(np.isneginf(lg[empty]))
    eo, el = max_abs(og[~empty], O[~empty]), max_abs(lg[~empty], L[~empty])
    record("decode_cases", "O_max_abs", eo)
    record("decode_cases", "LSE_max_abs", el)
    assert eo <= O_TOL and el <= LSE_TOL, (B, Hq, Hkv, n, lens, mk, T, eo, el)
