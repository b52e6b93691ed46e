"""The bounded-wait failure path on the GPU.

Every pipeline wait in the kernels has a time limit.  Here a test hook makes
one consumer warpgroup of every CTA wait on an mbarrier that nothing
completes, with the limit cut to 1 ms: the wait must run out, the status word
must report ATTN_ERR_TIMEOUT, the grid must drain and return within a small
multiple of the limit, and the context must stay usable -- the next clean
calls in the same process match the oracle.  No fault, trap or unbounded
wait is involved: the stalled wait ends by its own limit."""
import time

import numpy as np
import pytest
import torch

from oracle import attn64
from gpu_common import GRAD_TOL, LSE_TOL, O_TOL, default_scale, inputs, lib, max_abs, mods_pair, rel_fro, to_dev

pytestmark = pytest.mark.gpu

LIMIT_NS = 1_000_000  # 1 ms


def _clean_step_matches_oracle(ea, x, dev, m, om, s):
    o, lse = ea.forward(dev["q"], dev["k"], dev["v"], s, m)
    dq, dk, dv = ea.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], s, m)
    ea.attn_status()
    O, L = attn64.forward(x["q"], x["k"], x["v"], s, om)
    assert max_abs(o.float().cpu().numpy(), O) <= O_TOL
    assert max_abs(lse.cpu().numpy(), L) <= LSE_TOL
    G = attn64.backward(x["q"], x["k"], x["v"], x["do"], s, om)
    for a, b in zip((dq, dk, dv), G):
        assert rel_fro(a.float().cpu().numpy(), b) <= GRAD_TOL


@pytest.mark.parametrize("which", ["fwd", "bwd"])
@pytest.mark.parametrize("mk", [dict(causal=True), dict(causal=True, window=200)], ids=["causal", "window"])
def test_stalled_wait_times_out_and_the_context_survives(which, mk):
    ea = lib()
    B, Hq, Hkv, N, d = 1, 8, 2, 1000, 128
    x = inputs(B, Hq, Hkv, N, d, seed=41)
    dev = to_dev(x)
    m, om = mods_pair(x, **mk)
    s = default_scale(d)
    o, lse = ea.forward(dev["q"], dev["k"], dev["v"], s, m)
    ea.attn_status()
    torch.cuda.synchronize()
    ea.attn_test_hooks(LIMIT_NS, ea.STALL_FWD if which == "fwd" else ea.STALL_BWD)
    try:
        t0 = time.perf_counter()
        if which == "fwd":
            ea.forward(dev["q"], dev["k"], dev["v"], s, m)
        else:
            ea.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], s, m)
        st = ea.lib().attn_status(None)
        elapsed = time.perf_counter() - t0
    finally:
        ea.attn_test_hooks(0, 0)
    assert st == 6, ea.status_string(st)  # ATTN_ERR_TIMEOUT
    assert elapsed < 2.0, elapsed  # drained by the 1 ms limit, not by the 1 s default
    assert ea.lib().attn_status(None) == 0  # the status word was cleared
    _clean_step_matches_oracle(ea, x, dev, m, om, s)
