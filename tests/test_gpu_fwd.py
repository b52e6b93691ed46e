"""Forward parity on the GPU: the CUDA path through the C ABI against the fp64
oracle, element by element, on seeded inputs spanning several tiles, ragged
tails and every mod."""
import numpy as np
import pytest
import torch

import attn_inputs as gen
from oracle import attn64
from gpu_common import (LSE_TOL, O_TOL, default_scale, inputs, lib, max_abs, mods_pair, to_dev)

pytestmark = pytest.mark.gpu

# (B, Hq, Hkv, N, d, mods)
CASES = [
    (1, 2, 2, 128, 64, {}),                                   # the tiny MHA workload
    (1, 2, 2, 256, 128, dict(causal=True)),
    (2, 4, 2, 384, 128, dict(causal=True)),                   # GQA 2:1
    (1, 8, 1, 1000, 128, dict(causal=True)),                  # GQA 8:1, ragged tail
    (1, 2, 2, 200, 64, {}),                                   # ragged, non-causal, d=64
    (1, 3, 3, 1, 128, dict(causal=True)),                     # N = 1
    (1, 2, 2, 129, 64, dict(causal=True)),
    (1, 2, 2, 127, 128, {}),
    (2, 2, 2, 640, 128, dict(causal=True, window=300)),
    (1, 2, 2, 700, 128, dict(window=200)),                    # window without causal
    (2, 2, 1, 1024, 128, dict(causal=True, doc=True)),
    (1, 2, 2, 900, 64, dict(doc=True)),
    (1, 2, 2, 500, 128, dict(softcap=30.0)),
    (1, 4, 4, 520, 128, dict(causal=True, alibi=True)),
    (2, 4, 2, 1000, 128, dict(causal=True, window=257, doc=True, softcap=30.0, alibi=True)),
    (1, 2, 2, 777, 64, dict(causal=True, window=129, doc=True, softcap=5.0, alibi=True)),
    # document ids that are not one run per document (id = run index mod 3): the
    # kernels test ids element by element instead of using run intervals
    (2, 2, 2, 900, 128, dict(causal=True, doc="mod3")),
    (1, 2, 2, 600, 64, dict(doc="mod3", softcap=20.0, alibi=True)),
]


def _ids(c):
    B, Hq, Hkv, N, d, m = c
    return f"B{B}_H{Hq}x{Hkv}_N{N}_d{d}_" + ("-".join(m) or "none")


def _docs(B, N, seed):
    return gen.doc_ids(B, N, seed, lo=60, hi=400)


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_forward_parity(case):
    ea = lib()
    B, Hq, Hkv, N, d, mk = case
    x = inputs(B, Hq, Hkv, N, d, seed=100 + N + d + Hq)
    if mk.get("doc"):
        x["doc_ids_np"] = _docs(B, N, N)
        if mk["doc"] == "mod3":
            x["doc_ids_np"] = (x["doc_ids_np"] % 3).astype(np.int32)
    dev = to_dev(x)
    m, om = mods_pair(x, **dict(mk, doc=bool(mk.get("doc"))))
    s = default_scale(d)
    o, lse = ea.forward(dev["q"], dev["k"], dev["v"], s, m)
    ea.attn_status()
    O, L = attn64.forward(x["q"], x["k"], x["v"], s, om)
    eo = max_abs(o.float().cpu().numpy(), O)
    el = max_abs(lse.cpu().numpy(), L)
    assert eo <= O_TOL, eo
    assert el <= LSE_TOL, el


def test_forward_is_deterministic():
    ea = lib()
    x = to_dev(inputs(2, 4, 2, 1000, 128, seed=5))
    m = ea.make_mods(causal=True)
    o1, l1 = ea.forward(x["q"], x["k"], x["v"], 0.088, m)
    o2, l2 = ea.forward(x["q"], x["k"], x["v"], 0.088, m)
    ea.attn_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_forward_writes_only_its_outputs():
    """Guard bands: bytes around O and LSE stay untouched; NaN pre-fill of O is overwritten."""
    ea = lib()
    B, H, N, d = 1, 2, 300, 128
    x = to_dev(inputs(B, H, H, N, d, seed=6))
    pad = 4096
    obuf = torch.full((B * H * N * d + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((B * H * N + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    o = obuf[pad:pad + B * H * N * d].view(B, H, N, d)
    l = lbuf[pad:pad + B * H * N].view(B, H, N)
    ea.forward(x["q"], x["k"], x["v"], 0.1, ea.make_mods(causal=True), out=o, lse=l)
    ea.attn_status()
    assert torch.isnan(obuf[:pad]).all() and torch.isnan(obuf[-pad:]).all()
    assert (lbuf[:pad] == 7.0).all() and (lbuf[-pad:] == 7.0).all()
    assert not torch.isnan(o).any() and torch.isfinite(l).all()
