"""Packed variable-length sequences on the GPU (attn_fwd_varlen /
attn_bwd_varlen) against the fp64 oracle's document mask over the packed
rows, and against the document-mask entry points on the same rows."""
import numpy as np
import pytest
import torch

from oracle import attn64
from gpu_common import (GRAD_TOL, LSE_TOL, O_TOL, default_scale, inputs, lib, max_abs, rel_fro, to_dev)

pytestmark = pytest.mark.gpu

# (Hq, Hkv, sequence lengths, d, mods)
CASES = [
    (4, 2, [300, 1, 129, 640, 77], 128, dict(causal=True)),
    (2, 2, [1000, 24], 64, dict(causal=True, window=200)),
    (2, 1, [513, 255, 256], 128, dict(softcap=20.0, alibi=True)),
    (8, 1, [2048, 1, 1, 700], 128, dict(causal=True, alibi=True)),
]


def _ids(c):
    Hq, Hkv, lens, d, m = c
    return f"H{Hq}x{Hkv}_n{len(lens)}_T{sum(lens)}_d{d}_" + ("-".join(m) or "none")


def _seq_ids(cu, total):
    ids = np.zeros(total, dtype=np.int32)
    for s in range(len(cu) - 1):
        ids[cu[s]:cu[s + 1]] = s
    return ids


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_varlen_parity(case):
    ea = lib()
    Hq, Hkv, lens, d, mk = case
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(cu[-1])
    x = inputs(1, Hq, Hkv, total, d, seed=500 + total)
    dev = to_dev(x)
    dcu = torch.from_numpy(cu).cuda()
    m = ea.make_mods(**mk)
    s = default_scale(d)
    o, lse = ea.forward_varlen(dev["q"], dev["k"], dev["v"], dcu, s, m)
    dq, dk, dv = ea.backward_varlen(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], dcu, s, m)
    ea.attn_status()
    ids = _seq_ids(cu, total)
    om = attn64.Mods(doc_ids=ids[None, :], **mk)
    O, L = attn64.forward(x["q"], x["k"], x["v"], s, om)
    assert max_abs(o.float().cpu().numpy(), O) <= O_TOL
    assert max_abs(lse.cpu().numpy(), L) <= LSE_TOL
    G = attn64.backward(x["q"], x["k"], x["v"], x["do"], s, om)
    for name, a, b in (("dQ", dq, G[0]), ("dK", dk, G[1]), ("dV", dv, G[2])):
        e = rel_fro(a.float().cpu().numpy(), b)
        assert e <= GRAD_TOL, (name, e)
    # the same rows through the document-mask entry points: identical results
    md = ea.make_mods(doc_ids=torch.from_numpy(ids[None, :]).cuda(), **mk)
    o2, lse2 = ea.forward(dev["q"], dev["k"], dev["v"], s, md)
    g2 = ea.backward(dev["q"], dev["k"], dev["v"], o2, lse2, dev["do"], s, md)
    ea.attn_status()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    for a, b in zip((dq, dk, dv), g2):
        assert torch.equal(a, b)
