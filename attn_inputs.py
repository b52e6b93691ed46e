"""Seeded synthetic inputs for exact tiled attention.

This module is shared by the oracle (``oracle/``) and the CUDA path's tests
and benchmark.  It holds only workload shapes and random-number draws; none of
the attention arithmetic lives here, so neither side can leak into the other
through it.

Workloads (all synthetic; the pages name no dataset):

* ``tiny_mha``        B=1 H=2 N=128 d=64, non-causal forward.
* ``causal_mha_2k``   B=16 H=16 N=2048 d=128, causal forward + backward.
* ``gqa_causal_8k``   B=1 Hq=64 Hkv=8 N=8192 d=128, causal forward + backward
                      (the Llama-3-70B attention shape named on the
                      FlexAttention/FA4 page, "Performance et Validation").
* ``flex_mods_4k``    B=4 H=16 N=4096 d=128: causal AND sliding window 1024
                      AND document mask, tanh soft-cap 30 plus ALiBi.
* ``fp8_outliers_16k`` B=2 H=16 N=16384 d=128 non-causal FP8 forward, inputs
                      N(0,1) with 0.1 % of entries scaled by 50 (the outlier
                      experiment of the FlashAttention-3 digest, "Basse
                      précision FP8 et incoherent processing").
* ``varlen_packed_16k`` packed sequences (lengths drawn like the documents).
* ``paged_prefill_8k`` causal prefill with K/V in a shuffled 16-row block cache.
* ``paged_decode_8k`` B=32 Hq=64 Hkv=8 d=128: one decode token per sequence
                      over a shuffled paged cache, context lengths uniform in
                      [4096, 8192] (the kernel fusion page's paged KV cache,
                      block_size 16).

Recipe: Q/K/V/dO are ``torch.randn`` fp32 draws from a CPU generator seeded
per tensor, rounded to bf16.  Document lengths are integers uniform in
[128, 2048] drawn sequentially from ``numpy.random.default_rng(seed + b)``
until their sum reaches N; the last one is cut so the sum is exactly N.
Outlier positions are drawn without replacement per tensor.  Hadamard sign
vectors are +-1 per KV head.
"""
from __future__ import annotations

import numpy as np
import torch

WORKLOADS = {
    "tiny_mha": dict(B=1, Hq=2, Hkv=2, N=128, d=64, causal=False, seed=1000),
    "causal_mha_2k": dict(B=16, Hq=16, Hkv=16, N=2048, d=128, causal=True, seed=2000),
    "gqa_causal_8k": dict(B=1, Hq=64, Hkv=8, N=8192, d=128, causal=True, seed=3000),
    "flex_mods_4k": dict(B=4, Hq=16, Hkv=16, N=4096, d=128, causal=True, window=1024,
                         doc=True, softcap=30.0, alibi=True, seed=4000),
    "fp8_outliers_16k": dict(B=2, Hq=16, Hkv=16, N=16384, d=128, causal=False,
                             outlier_frac=1e-3, outlier_scale=50.0, seed=5000),
    # packed variable-length sequences (lengths drawn like the documents), causal
    "varlen_packed_16k": dict(B=1, Hq=16, Hkv=4, N=16384, d=128, causal=True, doc=True,
                              varlen=True, seed=6000),
    # causal prefill with K/V in a shuffled paged cache of 16-row blocks
    "paged_prefill_8k": dict(B=2, Hq=32, Hkv=8, N=8192, d=128, causal=True, paged=True, seed=7000),
    # one decode step per sequence over a shuffled paged cache; N is the longest
    # context, lengths uniform in [min_len, N]
    "paged_decode_8k": dict(B=32, Hq=64, Hkv=8, N=8192, d=128, min_len=4096, decode=True, seed=8000),
    # the same with 4 new tokens per sequence (drafts to verify)
    "paged_decode_4tok_8k": dict(B=32, Hq=64, Hkv=8, N=8192, d=128, min_len=4096, decode=True, q_len=4,
                                 seed=8100),
}

DOC_LEN_MIN = 128
DOC_LEN_MAX = 2048


def randn_bf16(shape, seed: int) -> torch.Tensor:
    """iid N(0,1) drawn in fp32 from a seeded CPU generator, rounded to bf16."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32).to(torch.bfloat16)


def randn_f32(shape, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32)


def doc_lengths(N: int, seed: int, lo: int = DOC_LEN_MIN, hi: int = DOC_LEN_MAX) -> list[int]:
    """Sequential uniform integer lengths in [lo, hi], the last cut so they sum to N."""
    rng = np.random.default_rng(int(seed))
    lens: list[int] = []
    total = 0
    while total < N:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, N - total)
        lens.append(n)
        total += n
    return lens


def doc_ids(B: int, N: int, seed: int, lo: int = DOC_LEN_MIN, hi: int = DOC_LEN_MAX) -> np.ndarray:
    """int32 [B, N]: document index (0, 1, 2, ...) of every position, per batch row."""
    out = np.empty((B, N), dtype=np.int32)
    for b in range(B):
        lens = doc_lengths(N, seed + b, lo, hi)
        out[b] = np.repeat(np.arange(len(lens), dtype=np.int32), lens)
    return out


def with_outliers(x: torch.Tensor, frac: float, factor: float, seed: int) -> torch.Tensor:
    """Scale round(frac * numel) entries, chosen without replacement, by ``factor``."""
    flat = x.reshape(-1).clone()
    k = int(round(frac * flat.numel()))
    rng = np.random.default_rng(int(seed))
    pos = rng.choice(flat.numel(), size=k, replace=False)
    flat[torch.from_numpy(pos.astype(np.int64))] *= factor
    return flat.reshape(x.shape)


def hadamard_signs(Hkv: int, d: int, seed: int) -> np.ndarray:
    """int8 [Hkv, d] of +-1, one random sign vector per KV head."""
    rng = np.random.default_rng(int(seed))
    return (rng.integers(0, 2, size=(Hkv, d)) * 2 - 1).astype(np.int8)


def make_inputs(B, Hq, Hkv, N, d, seed, *, need_do=True, outlier_frac=0.0,
                outlier_scale=1.0, doc=False, **_):
    """Q, K, V (and dO) as CPU bf16 [B, H, N, d], plus doc ids when asked.

    Seeds: Q=seed, K=seed+1, V=seed+2, dO=seed+3, documents seed+10+b,
    outlier positions seed+30+{0,1,2}.
    """
    shapes = [(B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d)]
    if outlier_frac > 0.0:
        qkv = [randn_f32(s, seed + t) for t, s in enumerate(shapes)]
        qkv = [with_outliers(x, outlier_frac, outlier_scale, seed + 30 + t).to(torch.bfloat16)
               for t, x in enumerate(qkv)]
    else:
        qkv = [randn_bf16(s, seed + t) for t, s in enumerate(shapes)]
    out = dict(q=qkv[0], k=qkv[1], v=qkv[2])
    if need_do:
        out["do"] = randn_bf16((B, Hq, N, d), seed + 3)
    if doc:
        out["doc_ids"] = doc_ids(B, N, seed + 10)
    return out


def paged_decode_inputs(B, Hq, Hkv, N, d, seed, *, min_len=1, lens=None, spare=8, block=16, q_len=1, **_):
    """One decode step over a paged K/V cache.

    Returns q [B, Hq, d] ([B, Hq, q_len, d] when q_len > 1: the newest q_len
    tokens) and the caches [num_blocks, Hkv, block, d] (CPU bf16),
    the block table int32 [B, ceil(N / block)] and the lengths int32 [B].
    Lengths are uniform integers in [min_len, N] (seed + 10) unless given;
    sequence b owns ceil(L_b / block) blocks at shuffled physical slots
    (seed + 11), a few spare slots stay unused, and table entries past a
    sequence's last block are -1.  Seeds: q = seed, K cache = seed + 1,
    V cache = seed + 2.
    """
    if lens is None:
        lens = np.random.default_rng(int(seed) + 10).integers(min_len, N + 1, size=B)
    lens = np.asarray(lens, dtype=np.int32)
    width = -(-N // block)
    nbs = [-(-int(L) // block) for L in lens]
    num_blocks = sum(nbs) + spare
    perm = np.random.default_rng(int(seed) + 11).permutation(num_blocks).astype(np.int32)
    table = np.full((B, width), -1, dtype=np.int32)
    used = 0
    for b, nb in enumerate(nbs):
        table[b, :nb] = perm[used:used + nb]
        used += nb
    return dict(q=randn_bf16((B, Hq, d) if q_len == 1 else (B, Hq, q_len, d), seed),
                k_cache=randn_bf16((num_blocks, Hkv, block, d), seed + 1),
                v_cache=randn_bf16((num_blocks, Hkv, block, d), seed + 2),
                block_table=table, seqlens=lens)


def workload_inputs(name: str, **overrides):
    """Inputs of a named workload (shapes/mods from WORKLOADS, optionally overridden)."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    return cfg, make_inputs(**cfg)
