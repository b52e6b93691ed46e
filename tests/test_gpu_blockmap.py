"""Block-sparsity map on the GPU: bit-exact against the oracle's element-by-
element classification."""
import numpy as np
import pytest
import torch

import attn_inputs as gen
from oracle import attn64
from gpu_common import lib

pytestmark = pytest.mark.gpu

MASKS = [
    dict(causal=True), dict(), dict(window=300), dict(causal=True, window=1024),
    dict(doc=True), dict(causal=True, doc=True), dict(causal=True, window=1024, doc=True),
    dict(causal=True, window=129, doc=True),
]


@pytest.mark.parametrize("N", [1, 128, 1000, 4096])
@pytest.mark.parametrize("mk", MASKS, ids=lambda m: "-".join(m) or "none")
def test_block_map_bit_exact(N, mk):
    ea = lib()
    B = 3
    docs = gen.doc_ids(B, N, 40 + N, lo=100, hi=1500) if mk.get("doc") else None
    dev_docs = torch.from_numpy(docs).cuda() if docs is not None else None
    m = ea.make_mods(causal=mk.get("causal", False), window=mk.get("window"), doc_ids=dev_docs)
    got = ea.block_map(B, N, m).cpu().numpy()
    ea.attn_status()
    ref = attn64.block_map(attn64.Mods(causal=mk.get("causal", False), window=mk.get("window"),
                                       doc_ids=docs), B, N)
    np.testing.assert_array_equal(got, ref)


def test_flex_workload_map_and_skip_fraction():
    """The flex-mods workload: map bit-exact and most tiles skipped."""
    ea = lib()
    cfg = gen.WORKLOADS["flex_mods_4k"]
    B, N = cfg["B"], cfg["N"]
    docs = gen.doc_ids(B, N, cfg["seed"] + 10)
    m = ea.make_mods(causal=True, window=cfg["window"], doc_ids=torch.from_numpy(docs).cuda())
    got = ea.block_map(B, N, m).cpu().numpy()
    ea.attn_status()
    ref = attn64.block_map(attn64.Mods(causal=True, window=cfg["window"], doc_ids=docs), B, N)
    np.testing.assert_array_equal(got, ref)
    assert (got == 0).mean() > 0.5


INTERNAL = [
    dict(causal=True, doc=True), dict(causal=True, window=1024, doc=True), dict(doc=True),
    dict(window=129, doc=True), dict(causal=True, window=300),
]


@pytest.mark.parametrize("ids", ["runs", "repeated"])
@pytest.mark.parametrize("mk", INTERNAL, ids=lambda m: "-".join(m))
def test_map_built_by_forward_bit_exact(ids, mk):
    """The map an attention call builds in its workspace (at offset 0), where
    non-decreasing document ids are classified from their runs and other ids
    pair by pair, equals the oracle's element-by-element map.  "repeated"
    gives every other document the same id, so equal ids sit in separate runs."""
    ea = lib()
    B, Hq, Hkv, N, d = 2, 2, 1, 1000, 64
    docs = gen.doc_ids(B, N, 321, lo=60, hi=400) if mk.get("doc") else None
    if docs is not None and ids == "repeated":
        docs = (docs % 2).astype(np.int32)
    dev_docs = torch.from_numpy(docs).cuda() if docs is not None else None
    m = ea.make_mods(causal=mk.get("causal", False), window=mk.get("window"), doc_ids=dev_docs)
    x = {k: v.cuda() for k, v in gen.make_inputs(B, Hq, Hkv, N, d, seed=55).items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    nws = ea.attn_workspace_size(ea.OP_FWD, B, Hq, Hkv, N, d, m)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    ea.attn_fwd(x["q"], x["k"], x["v"], o, lse, B, Hq, Hkv, N, d, 0.125, m, ws, nws)
    ea.attn_status()
    nT = (N + 127) // 128
    got = ws[:B * nT * nT].cpu().numpy().reshape(B, nT, nT)
    ref = attn64.block_map(attn64.Mods(causal=mk.get("causal", False), window=mk.get("window"),
                                       doc_ids=docs), B, N)
    np.testing.assert_array_equal(got, ref)
