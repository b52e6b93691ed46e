"""The C ABI under CUDA graph capture: a training step (forward + backward)
and a paged decode step are captured once and replayed on new inputs copied
into the captured buffers; every replay must give bit-for-bit the results
of the same calls made eagerly.  The library allocates nothing and calls no
synchronising API inside the entry points, so their kernels (and the decode
path's programmatic dependent launches) record into a graph as they are."""
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
from gpu_common import lib

pytestmark = pytest.mark.gpu


def _capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def test_training_step_graph_replay_matches_eager():
    ea = lib()
    B, Hq, Hkv, N, d = 1, 8, 2, 1000, 128
    s = 1.0 / math.sqrt(d)
    mods = ea.make_mods(causal=True, window=300, softcap=20.0)
    dev = torch.device("cuda")
    bufs = {k: v.to(dev) for k, v in gen.make_inputs(B, Hq, Hkv, N, d, seed=31).items()}
    q, k, v, do = (bufs[n] for n in ("q", "k", "v", "do"))
    o, lse = torch.empty_like(q), torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nf = ea.attn_workspace_size(ea.OP_FWD, B, Hq, Hkv, N, d, mods)
    nb = ea.attn_workspace_size(ea.OP_BWD, B, Hq, Hkv, N, d, mods)
    wf = torch.empty(max(nf, 1), dtype=torch.uint8, device=dev)
    wb = torch.empty(nb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()

    def step():
        ea.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, s, mods, wf, nf, stream)
        ea.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, s, mods, wb, nb, stream)

    with torch.cuda.stream(stream):
        step()  # first eager call: device state and descriptors set up outside capture
    stream.synchronize()
    g = _capture(step, stream)
    for seed in (41, 42):
        new = gen.make_inputs(B, Hq, Hkv, N, d, seed=seed)
        for n in ("q", "k", "v", "do"):
            bufs[n].copy_(new[n].to(dev))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
        ea.attn_status(stream)
        eager = [t.clone() for t in (o, lse, dq, dk, dv)]
        for t in (o, lse, dq, dk, dv):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        ea.attn_status()
        for a, b_ in zip(eager, (o, lse, dq, dk, dv)):
            assert torch.equal(a, b_)


def test_decode_step_graph_replay_matches_eager():
    ea = lib()
    B, Hq, Hkv, n, T = 6, 32, 4, 2000, 2
    x = gen.paged_decode_inputs(B, Hq, Hkv, n, 128, seed=77, q_len=T)
    dev = torch.device("cuda")
    q = x["q"].to(dev)
    kc, vc = x["k_cache"].to(dev), x["v_cache"].to(dev)
    table = torch.from_numpy(x["block_table"]).to(dev)
    lens = torch.from_numpy(x["seqlens"]).to(dev)
    nblk, mb = kc.shape[0], table.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=dev)
    nws = ea.attn_decode_workspace_size(B, Hq, Hkv, T, mb, 128)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    mods = ea.make_mods(alibi=True)
    stream = torch.cuda.Stream()

    def step():
        ea.attn_decode_paged(q, kc, vc, table, mb, lens, nblk, o, lse, B, Hq, Hkv, T, 128, 0.09, mods, ws, nws,
                             stream)

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    g = _capture(step, stream)
    rng = np.random.default_rng(3)
    for _ in range(2):
        q.copy_(torch.randn(q.shape, generator=torch.Generator().manual_seed(int(rng.integers(1 << 30)))).to(q))
        # new lengths too, within the blocks each sequence owns
        lens.copy_(torch.from_numpy((rng.random(B) * (x["seqlens"] + 1)).astype(np.int32)))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
        ea.attn_status(stream)
        eager = (o.clone(), lse.clone())
        o.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        ea.attn_status()
        assert torch.equal(eager[0], o) and torch.equal(eager[1], lse)
