"""Scalar-loop attention for tiny shapes, used only to pin ``attn64``.

TEST INFRASTRUCTURE ONLY.  Written independently of ``attn64`` (no shared
helpers): every score, mask test and sum is an explicit Python loop over
scalars, so a slip in attn64's vectorised indexing (a transposed operand, a
wrong GQA head, a mask applied to the wrong axis) shows up as a mismatch.
The arithmetic follows the same readings of the pages as attn64 (plain
softmax attention with the FlexAttention mods: causal, sliding window i-j<W,
document ids, c*tanh(s/c) soft-cap, ALiBi -slope_h*(i-j)).
"""
from __future__ import annotations

import math


def _val(t, *idx):
    x = t
    for i in idx:
        x = x[i]
    return float(x)


def forward(q, k, v, scale, causal=False, window=None, doc=None, softcap=None,
            slopes=None):
    """Nested lists O[b][h][i][c], LSE[b][h][i] from explicit loops.

    ``q`` [B][Hq][N][d], ``k``/``v`` [B][Hkv][N][d] (anything indexable),
    ``doc`` [B][N] or None, ``slopes`` a list of Hq floats or None (no ALiBi).
    """
    B, Hq, N, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv = len(k[0])
    O = [[[[0.0] * d for _ in range(N)] for _ in range(Hq)] for _ in range(B)]
    L = [[[0.0] * N for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            hk = h * Hkv // Hq
            for i in range(N):
                xs = []
                js = []
                for j in range(N):
                    ok = True
                    if causal and j > i:
                        ok = False
                    if window is not None and not (i - j < window):
                        ok = False
                    if doc is not None and int(doc[b][i]) != int(doc[b][j]):
                        ok = False
                    if not ok:
                        continue
                    s = 0.0
                    for c in range(d):
                        s += _val(q, b, h, i, c) * _val(k, b, hk, j, c)
                    s *= scale
                    if softcap is not None:
                        s = softcap * math.tanh(s / softcap)
                    if slopes is not None:
                        s -= slopes[h] * (i - j)
                    xs.append(s)
                    js.append(j)
                if not xs:
                    L[b][h][i] = -math.inf
                    continue
                mx = max(xs)
                tot = 0.0
                for s in xs:
                    tot += math.exp(s - mx)
                L[b][h][i] = mx + math.log(tot)
                for s, j in zip(xs, js):
                    p = math.exp(s - mx) / tot
                    for c in range(d):
                        O[b][h][i][c] += p * _val(v, b, hk, j, c)
    return O, L


def tile_class(B, N, tile, causal=False, window=None, doc=None):
    """Nested list [b][I][J] of 0 (skip) / 1 (partial) / 2 (full), element by element."""
    nT = (N + tile - 1) // tile
    out = []
    for b in range(B):
        rowsI = []
        for I in range(nT):
            rowJ = []
            for J in range(nT):
                any_ok = False
                all_ok = True
                for i in range(I * tile, min(I * tile + tile, N)):
                    for j in range(J * tile, J * tile + tile):
                        ok = j < N
                        if ok and causal and j > i:
                            ok = False
                        if ok and window is not None and not (i - j < window):
                            ok = False
                        if ok and doc is not None and int(doc[b][i]) != int(doc[b][j]):
                            ok = False
                        any_ok = any_ok or ok
                        all_ok = all_ok and ok
                rowJ.append(2 if all_ok else (1 if any_ok else 0))
            rowsI.append(rowJ)
        out.append(rowsI)
    return out


def fwht(x):
    """Unnormalised Walsh-Hadamard transform (natural order) by butterflies."""
    y = [float(t) for t in x]
    n = len(y)
    h = 1
    while h < n:
        for start in range(0, n, 2 * h):
            for t in range(start, start + h):
                a, b = y[t], y[t + h]
                y[t], y[t + h] = a + b, a - b
        h *= 2
    return y
