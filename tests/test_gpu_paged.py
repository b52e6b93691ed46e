"""Forward over a paged K/V cache (attn_fwd_paged): K/V rows scattered into
shuffled 16-row blocks must give the same O and LSE as the contiguous
forward -- bit for bit, the loads are the only difference -- and match the
fp64 oracle on the contiguous inputs."""
import numpy as np
import pytest
import torch

from oracle import attn64
from gpu_common import LSE_TOL, O_TOL, default_scale, inputs, lib, max_abs, mods_pair, to_dev

pytestmark = pytest.mark.gpu

# (B, Hq, Hkv, N, mods, d)
CASES = [
    (2, 8, 2, 1024, dict(causal=True), 128),
    (1, 4, 4, 400, {}, 128),                                       # ragged last tile: blocks past N are zeros
    (2, 4, 1, 640, dict(causal=True, window=200, softcap=20.0, alibi=True), 128),
    (2, 8, 2, 1024, dict(causal=True), 64),
    (1, 4, 1, 400, dict(window=100, alibi=True), 64),
]


def _ids(c):
    B, Hq, Hkv, N, m, d = c
    return f"B{B}_H{Hq}x{Hkv}_N{N}_d{d}_" + ("-".join(m) or "none")


def _page(x, B, Hkv, N, rng, spare=7):
    """Scatter [B, Hkv, N, d] rows into a shuffled [num_blocks, Hkv, 16, d] cache."""
    nb = N // 16
    num_blocks = B * nb + spare
    perm = rng.permutation(num_blocks)[:B * nb].reshape(B, nb).astype(np.int32)
    cache = torch.randn(num_blocks, Hkv, 16, x.shape[-1]).to(torch.bfloat16)  # unused blocks: noise
    for b in range(B):
        for t in range(nb):
            cache[perm[b, t]] = x[b, :, 16 * t:16 * t + 16]
    return cache, perm, num_blocks


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_paged_forward(case):
    ea = lib()
    B, Hq, Hkv, N, mk, d = case
    x = inputs(B, Hq, Hkv, N, d, seed=700 + N + d)
    rng = np.random.default_rng(N)
    kc, table, num_blocks = _page(x["k"], B, Hkv, N, rng)
    vc, _, _ = _page(x["v"], B, Hkv, N, np.random.default_rng(N))  # same permutation
    dev = to_dev(x)
    m, om = mods_pair(x, **mk)
    s = default_scale(d)
    o, lse = ea.forward_paged(dev["q"], kc.cuda(), vc.cuda(), torch.from_numpy(table).cuda(), s, m)
    o_ref, lse_ref = ea.forward(dev["q"], dev["k"], dev["v"], s, m)
    ea.attn_status()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    O, L = attn64.forward(x["q"], x["k"], x["v"], s, om)
    assert max_abs(o.float().cpu().numpy(), O) <= O_TOL
    assert max_abs(lse.cpu().numpy(), L) <= LSE_TOL
