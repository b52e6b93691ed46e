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
