"""attn_bwd_noalloc against attn_bwd, through the C ABI.

attn_bwd_noalloc is for callers that cannot allocate device memory: their
memory belongs to a framework allocator or a fixed arena, or they must not
call cudaMalloc/cudaFree because those synchronise the device.  It takes no
workspace and uses the library's fixed scratch array instead.  Both entry
points run the same deterministic kernels, so the results must be bitwise
equal on every call -- including consecutive calls of different shapes and
mods, where whatever one call left in the shared array must not leak into
the next.  This file is collected last, so a run that stops at the first
failure has already run every other test.
"""
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
from gpu_common import inputs, lib, mods_pair, to_dev

pytestmark = pytest.mark.gpu

# (B, Hq, Hkv, N, d, mods); "mod3" = document ids that are not one run per document
CASES = {
    "doc_unsorted": (2, 2, 2, 900, 128, dict(causal=True, doc="mod3")),
    "causal_gqa": (1, 8, 1, 1000, 128, dict(causal=True)),
    "all_mods": (2, 4, 2, 1000, 128, dict(causal=True, window=257, doc=True, softcap=30.0, alibi=True)),
    "plain_d64": (1, 2, 2, 333, 64, {}),
}
ORDER = ["doc_unsorted", "causal_gqa", "doc_unsorted", "all_mods", "plain_d64", "causal_gqa", "all_mods"]


def _prepare(name, seed):
    ea = lib()
    B, Hq, Hkv, N, d, mk = CASES[name]
    x = inputs(B, Hq, Hkv, N, d, seed=seed)
    if mk.get("doc"):
        x["doc_ids_np"] = gen.doc_ids(B, N, N, lo=60, hi=400)
        if mk["doc"] == "mod3":
            x["doc_ids_np"] = (x["doc_ids_np"] % 3).astype(np.int32)
    dev = to_dev(x)
    m, _ = mods_pair(x, **dict(mk, doc=bool(mk.get("doc"))))
    s = 1.0 / math.sqrt(d)
    o, lse = ea.forward(dev["q"], dev["k"], dev["v"], s, m)
    ref = ea.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], s, m)
    ea.attn_status()
    return dict(shape=(B, Hq, Hkv, N, d), dev=dev, m=m, s=s, o=o, lse=lse, ref=ref)


def test_noalloc_equals_attn_bwd_across_alternating_calls():
    ea = lib()
    prepared = {name: _prepare(name, seed=31 + i) for i, name in enumerate(CASES)}
    for name in ORDER:
        c = prepared[name]
        B, Hq, Hkv, N, d = c["shape"]
        dev = c["dev"]
        out = [torch.full_like(t, float("nan")) for t in c["ref"]]
        ea.attn_bwd_noalloc(dev["q"], dev["k"], dev["v"], c["o"], dev["do"], c["lse"], *out,
                            B, Hq, Hkv, N, d, c["s"], c["m"])
        ea.attn_status()
        for which, a, r in zip(("dQ", "dK", "dV"), out, c["ref"]):
            assert torch.equal(a, r), (name, which)


def test_noalloc_rejects_work_beyond_its_scratch():
    ea = lib()
    A = 0x10000  # aligned placeholder address, never dereferenced: the size check comes first
    B, Hq, Hkv, N, d = 1, 64, 8, 65536, 128  # far more workspace than the 8 MiB of scratch
    assert ea.attn_workspace_size(ea.OP_BWD, B, Hq, Hkv, N, d, None) > ea.NOALLOC_SCRATCH_BYTES
    st = ea.lib().attn_bwd_noalloc(A, A, A, A, A, A, A, A, A, B, Hq, Hkv, N, d, 0.1, None, None)
    assert st == 3  # ATTN_ERR_WORKSPACE
