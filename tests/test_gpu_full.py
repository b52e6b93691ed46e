"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times: the GPU computes everything, the oracle checks sampled query
rows, KV rows and heads (each computed from the definition on its own)."""
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
from oracle import attn64
from gpu_common import GRAD_TOL, LSE_TOL, O_TOL, lib, max_abs, record, rel_fro

pytestmark = pytest.mark.gpu


def _sample_rows(N, seed, n_mid=128):
    rng = np.random.default_rng(seed)
    edge = min(128, N)
    mid = rng.choice(np.arange(edge, max(edge + 1, N - edge)), size=min(n_mid, max(0, N - 2 * edge)),
                     replace=False) if N > 2 * edge else np.array([], dtype=np.int64)
    return np.unique(np.concatenate([np.arange(edge), np.sort(mid), np.arange(N - edge, N)]))


def _run_full(name):
    ea = lib()
    cfg = dict(gen.WORKLOADS[name])
    x = gen.make_inputs(**cfg)
    B, Hq, Hkv, N, d = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["N"], cfg["d"]
    dev = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    docs = x.get("doc_ids")
    ddocs = torch.from_numpy(docs).cuda() if docs is not None else None
    m = ea.make_mods(causal=cfg.get("causal", False), window=cfg.get("window"), doc_ids=ddocs,
                     softcap=cfg.get("softcap"), alibi=cfg.get("alibi", False))
    om = attn64.Mods(causal=cfg.get("causal", False), window=cfg.get("window"), doc_ids=docs,
                     softcap=cfg.get("softcap"), alibi=cfg.get("alibi", False))
    s = 1.0 / math.sqrt(d)
    o, lse = ea.forward(dev["q"], dev["k"], dev["v"], s, m)
    dq, dk, dv = ea.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], s, m)
    ea.attn_status()
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    return cfg, x, om, s, [t.float().cpu().numpy() for t in (o, lse, dq, dk, dv)]


# (workload, [(b, hk) groups to check], sample everything in a group?)
FULL = [
    ("tiny_mha", [(0, 0), (0, 1)]),
    ("causal_mha_2k", [(0, 0), (7, 9), (15, 15)]),
    ("flex_mods_4k", [(0, 0), (3, 15)]),
    ("gqa_causal_8k", [(0, 0), (0, 7)]),
]


@pytest.mark.parametrize("name,groups", FULL, ids=[f[0] for f in FULL])
def test_full_size_sampled_parity(name, groups):
    cfg, x, om, s, (o, lse, dq, dk, dv) = _run_full(name)
    N, Hq, Hkv = cfg["N"], cfg["Hq"], cfg["Hkv"]
    G = Hq // Hkv
    rows = _sample_rows(N, 1) if N > 4096 else np.arange(N)
    for b, hk in groups:
        heads = range(hk * G, (hk + 1) * G)
        for hq in list(heads)[:2] + [hk * G + G - 1]:
            O, L = attn64.head_forward(x["q"], x["k"], x["v"], s, om, b, hq, rows=rows)
            eo, el = max_abs(o[b, hq, rows], O), max_abs(lse[b, hq, rows], L)
            record(name, "O_max_abs", eo)
            record(name, "LSE_max_abs", el)
            assert eo <= O_TOL
            assert el <= LSE_TOL
        gq, gk, gv = attn64.sampled_backward(x["q"], x["k"], x["v"], x["do"], s, om, b, hk,
                                             q_rows=rows, kv_rows=rows)
        errs = {"dQ_rel_fro": rel_fro(dq[b, hk * G:(hk + 1) * G][:, rows], gq),
                "dK_rel_fro": rel_fro(dk[b, hk, rows], gk),
                "dV_rel_fro": rel_fro(dv[b, hk, rows], gv)}
        for key, e in errs.items():
            record(name, key, e)
            assert e <= GRAD_TOL, (key, e)
