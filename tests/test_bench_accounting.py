"""The benchmark's FLOP accounting (allowed query/key pairs, per row and in
total) against the oracle's mask, on small seeded cases of every mask kind."""
import numpy as np
import pytest

import attn_inputs as gen
import bench
from oracle import attn64

CASES = [
    dict(B=1, Hq=1, Hkv=1, N=300, d=64, causal=False, seed=1),
    dict(B=2, Hq=1, Hkv=1, N=257, d=64, causal=True, seed=2),
    dict(B=2, Hq=1, Hkv=1, N=700, d=64, causal=True, window=129, seed=3),
    dict(B=3, Hq=1, Hkv=1, N=900, d=64, causal=True, window=200, doc=True, seed=4),
    dict(B=2, Hq=1, Hkv=1, N=1000, d=64, causal=True, doc=True, seed=5),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: "-".join(k for k in ("causal", "window", "doc") if c.get(k)) or "none")
def test_pair_counts_match_the_oracle_mask(cfg):
    x = gen.make_inputs(**cfg)
    docs = x.get("doc_ids")
    m = attn64.Mods(causal=cfg.get("causal", False), window=cfg.get("window"), doc_ids=docs)
    assert bench.allowed_pairs(cfg, docs) == attn64.flop_pairs(m, cfg["B"], cfg["N"])
    rows = np.arange(0, cfg["N"], 7)
    for b in range(cfg["B"]):
        want = attn64.allowed(m, b, rows, np.arange(cfg["N"])).sum(axis=1)
        assert np.array_equal(bench.row_pairs(cfg, docs, b, rows), want)


def test_gqa_8k_flops():
    fwd, bwd = bench.flops(gen.WORKLOADS["gqa_causal_8k"])
    assert fwd == 4 * 64 * 128 * 8192 * 8193 // 2
    assert bwd == 2.5 * fwd


def test_peak_follows_the_clock_record():
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
    at_max = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    p, why = bench.bf16_peak(peaks, "measured", at_max)
    assert p == 1900.0 and "burst" in why
    slow = {"sm_mhz": 1485.0, "sm_max_mhz": 2070.0, "reasons": []}
    p, why = bench.bf16_peak(peaks, "measured", slow)
    assert abs(p - 1900.0 * 1485.0 / 2070.0) < 1e-9 and "1485" in why
    capped = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    p, why = bench.bf16_peak(peaks, "measured", capped)
    assert p == 1900.0 and "sw_power_cap" in why
    p, _ = bench.bf16_peak(peaks, "measured", {"sm_mhz": None, "sm_max_mhz": None, "reasons": []})
    assert p == 1900.0


def test_computed_pairs_of_analytic_masks():
    # causal: the nT (nT + 1) / 2 non-skipped tiles of every batch entry
    cfg = dict(B=2, N=1000, causal=True)
    assert bench.computed_pairs(None, cfg, None, None) == 2 * 8 * 9 // 2 * 128 * 128
    assert bench.computed_pairs(None, dict(B=1, N=300), None, None) == 9 * 128 * 128
    # the computed area always covers the allowed pairs
    full = dict(B=1, Hq=1, Hkv=1, N=8192, d=128, causal=True)
    assert bench.allowed_pairs(full) <= bench.computed_pairs(None, full, None, None)
