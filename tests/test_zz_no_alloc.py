"""attn_bwd_noalloc against attn_bwd, through the C ABI.

attn_bwd_noalloc is for callers that cannot allocate device memory: their
memory belongs to a framework allocator or a fixed arena, or they must not
call cudaMalloc/cudaFree because those synchronise the device.  It takes no
workspace and uses the library's fixed scratch array instead, so its results
must match attn_bwd's on every call, including consecutive calls that reuse
the array.  This file is collected last, so a run that stops at the first
failure has already run every other test.
"""
import math

import pytest
import torch

import attn_inputs as gen
from gpu_common import GRAD_TOL, inputs, lib, mods_pair, rel_fro, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    (1, 8, 1, 1000, 128, dict(causal=True)),
    (2, 4, 2, 1000, 128, dict(causal=True, window=257, doc=True, softcap=30.0, alibi=True)),
]


@pytest.mark.parametrize("case", CASES, ids=["causal_gqa", "all_mods"])
def test_noalloc_matches_attn_bwd_on_consecutive_calls(case):
    ea = lib()
    B, Hq, Hkv, N, d, mk = case
    x = inputs(B, Hq, Hkv, N, d, seed=31)
    if mk.get("doc"):
        x["doc_ids_np"] = gen.doc_ids(B, N, N, lo=60, hi=400)
    dev = to_dev(x)
    m, _ = mods_pair(x, **mk)
    s = 1.0 / math.sqrt(d)
    o, lse = ea.forward(dev["q"], dev["k"], dev["v"], s, m)
    ref = ea.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], s, m)
    ea.attn_status()
    for _ in range(2):  # two calls in a row share the scratch array
        out = [torch.full_like(t, float("nan")) for t in ref]
        ea.attn_bwd_noalloc(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, *out,
                            B, Hq, Hkv, N, d, s, m)
        ea.attn_status()
        for a, r in zip(out, ref):
            assert rel_fro(a.float().cpu().numpy(), r.float().cpu().numpy()) <= GRAD_TOL


def test_noalloc_rejects_work_beyond_its_scratch():
    ea = lib()
    A = 0x10000  # aligned placeholder address, never dereferenced: the size check comes first
    B, Hq, Hkv, N, d = 1, 64, 8, 65536, 128  # 32 MiB of row statistics > 8 MiB of scratch
    assert ea.attn_workspace_size(ea.OP_BWD, B, Hq, Hkv, N, d, None) > ea.NOALLOC_SCRATCH_BYTES
    st = ea.lib().attn_bwd_noalloc(A, A, A, A, A, A, A, A, A, B, Hq, Hkv, N, d, 0.1, None, None)
    assert st == 3  # ATTN_ERR_WORKSPACE
