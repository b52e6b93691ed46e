"""Backward parity on the GPU against the fp64 oracle (relative Frobenius
error of dQ, dK, dV) and bitwise reproducibility."""
import numpy as np
import pytest
import torch

import attn_inputs as gen
from oracle import attn64
from gpu_common import GRAD_TOL, default_scale, inputs, lib, mods_pair, rel_fro, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    (1, 2, 2, 256, 128, dict(causal=True)),
    (2, 4, 2, 384, 128, dict(causal=True)),
    (1, 8, 1, 1000, 128, dict(causal=True)),
    (1, 2, 2, 200, 64, {}),
    (1, 4, 2, 600, 128, {}),   # no mask, odd tile count
    (1, 2, 2, 1, 128, dict(causal=True)),
    (1, 2, 2, 129, 64, dict(causal=True)),
    (2, 2, 2, 640, 128, dict(causal=True, window=300)),
    (1, 2, 2, 700, 128, dict(window=200)),
    (2, 2, 1, 1024, 128, dict(causal=True, doc=True)),
    (1, 2, 2, 500, 128, dict(softcap=30.0)),
    (1, 4, 4, 520, 128, dict(causal=True, alibi=True)),
    (2, 4, 2, 1000, 128, dict(causal=True, window=257, doc=True, softcap=30.0, alibi=True)),
    (1, 2, 2, 777, 64, dict(causal=True, window=129, doc=True, softcap=5.0, alibi=True)),
    # document ids that are not one run per document (id = run index mod 3)
    (2, 2, 2, 900, 128, dict(causal=True, doc="mod3")),
    (1, 2, 2, 600, 64, dict(doc="mod3", softcap=20.0, alibi=True)),
]


# More work items (batch x KV head x KV tile) than SMs: each CTA of the
# persistent causal backward takes several items in turn.
MANY = [
    (2, 16, 16, 2048, 128, dict(causal=True)),
    (4, 8, 2, 1536, 64, dict(causal=True, window=700)),
    (3, 8, 4, 1300, 128, dict(causal=True, doc=True, softcap=30.0, alibi=True)),
]


def _ids(c):
    B, Hq, Hkv, N, d, m = c
    return f"B{B}_H{Hq}x{Hkv}_N{N}_d{d}_" + ("-".join(m) or "none")


def _run(case, seed):
    ea = lib()
    B, Hq, Hkv, N, d, mk = case
    x = inputs(B, Hq, Hkv, N, d, seed=seed)
    if mk.get("doc"):
        x["doc_ids_np"] = gen.doc_ids(B, N, N, lo=60, hi=400)
        if mk["doc"] == "mod3":
            x["doc_ids_np"] = (x["doc_ids_np"] % 3).astype(np.int32)
    dev = to_dev(x)
    m, om = mods_pair(x, **dict(mk, doc=bool(mk.get("doc"))))
    s = default_scale(d)
    o, lse = ea.forward(dev["q"], dev["k"], dev["v"], s, m)
    dq, dk, dv = ea.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], s, m)
    ea.attn_status()
    return x, om, s, (dq, dk, dv), (o, lse, dev, m)


@pytest.mark.parametrize("case", CASES + MANY, ids=_ids)
def test_backward_parity(case):
    x, om, s, (dq, dk, dv), _ = _run(case, seed=300 + case[3] + case[4])
    dQ, dK, dV = attn64.backward(x["q"], x["k"], x["v"], x["do"], s, om)
    for name, a, b in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV)):
        e = rel_fro(a.float().cpu().numpy(), b)
        assert e <= GRAD_TOL, (name, e)


# MHA with many short work items per CTA (item boundaries in every CTA), plain
# causal (two-kernel backward) and with a window (one-kernel backward)
REPRO = [CASES[2], CASES[11], MANY[0], (8, 16, 16, 1024, 128, dict(causal=True)),
         (8, 16, 16, 1024, 128, dict(causal=True, window=300))]


@pytest.mark.parametrize("case", REPRO, ids=_ids)
def test_backward_is_bitwise_reproducible(case):
    ea = lib()
    x, om, s, g1, (o, lse, dev, m) = _run(case, seed=9)
    for _ in range(6):
        g2 = ea.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], s, m)
        ea.attn_status()
        for a, b in zip(g1, g2):
            assert torch.equal(a, b)
