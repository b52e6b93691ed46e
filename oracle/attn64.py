"""Plain fp64 definition of exact (masked, modded) softmax attention.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): product code never
imports this module.

What the method computes
------------------------
The pages describe tiled attention as reaching *exactly* the standard
attention result, only without storing the score matrix: "FlashAttention-2
(FR)", section "Contexte" (tiles processed in SRAM, full matrix never
materialised) and opening paragraph (identical computation, no loss of
precision); "FlashAttention-3 : une attention plus rapide ...", section
"Rappel du fonctionnement de FlashAttention" (tiling plus softmax rescaling
gives the correct output without approximation, backward by recomputation);
"Les kernels d'attention rapide ...", section "Attention de type
FlashAttention et attention paginée" (the naive method builds a T^2 score
matrix per head).  So the oracle *is* the naive definition, in fp64, with the
full score matrix per (batch, head).

The pages give no formulas; the readings taken here are:

* layout [B, H, N, d]; GQA maps query head hq to KV head hq // (Hq // Hkv);
* scores z = scale * q.k; soft-cap x = c * tanh(z / c) (when enabled); then
  ALiBi x -= slope_h * (i - j) with slope_h = 2^(-8 (h + 1) / Hq), h the
  0-based query head (the soft-cap does not touch the bias);
* the mask is the AND of the enabled parts: causal j <= i, sliding window
  i - j < W, documents doc[i] == doc[j];
* LSE is natural-log; a row with no allowed key gets O = 0, LSE = -inf and
  zero gradients;
* backward is the textbook calculus of the above (the pages only say it
  recomputes): D_i = sum_j P_ij dP_ij, dX = P (dP - D), dZ = dX * (1 -
  tanh^2(z / c)) with the soft-cap, dQ = scale dZ K, dK = scale dZ^T Q,
  dV = P^T dO, with dK and dV summed over the query heads of a KV group.

The feature list (ALiBi, sliding window, document masking, soft-capping) is
from "FlexAttention de PyTorch avec FlashAttention-4 change la donne",
opening paragraphs; GQA from the Hacker News thread of the FlashAttention-3
digest.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

TILE = 128  # block-sparsity granularity (FlexAttention/FA4 page, "Limitations actuelles")

MAP_SKIP, MAP_PARTIAL, MAP_FULL = 0, 1, 2


@dataclass
class Mods:
    causal: bool = False
    window: Optional[int] = None          # allowed iff i - j < window
    doc_ids: Optional[np.ndarray] = None  # int [B, N]
    softcap: Optional[float] = None       # x = c * tanh(x / c)
    alibi: bool = False
    alibi_slopes: Optional[np.ndarray] = None  # [Hq]; None -> 2^(-8(h+1)/Hq)


def alibi_slopes(Hq: int) -> np.ndarray:
    """Default ALiBi slopes 2^(-8 (h + 1) / Hq), h = 0 .. Hq-1."""
    return 2.0 ** (-8.0 * (np.arange(Hq, dtype=np.float64) + 1.0) / Hq)


def _f64(x) -> np.ndarray:
    """Exact upcast of a bf16/fp32 torch tensor or numpy array to fp64 numpy."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def allowed(mods: Mods, b: int, rows: np.ndarray, cols: np.ndarray) -> np.ndarray:
    """Boolean [len(rows), len(cols)]: which (i, j) pairs may attend."""
    i = rows[:, None]
    j = cols[None, :]
    m = np.ones((rows.size, cols.size), dtype=bool)
    if mods.causal:
        m &= j <= i
    if mods.window is not None:
        m &= (i - j) < mods.window
    if mods.doc_ids is not None:
        doc = np.asarray(mods.doc_ids)[b]
        m &= doc[rows][:, None] == doc[cols][None, :]
    return m


def logits(qh: np.ndarray, kh: np.ndarray, scale: float, mods: Mods, hq: int, Hq: int,
           rows: np.ndarray, cols: np.ndarray):
    """z = scale q k^T and x = mods(z) for the given rows/cols (fp64).

    Returns (z, x); masking is not applied here.
    """
    z = scale * (qh[rows] @ kh[cols].T)
    x = z
    if mods.softcap is not None:
        c = float(mods.softcap)
        x = c * np.tanh(z / c)
    if mods.alibi:
        slopes = alibi_slopes(Hq) if mods.alibi_slopes is None else np.asarray(
            mods.alibi_slopes, dtype=np.float64)
        x = x - slopes[hq] * (rows[:, None] - cols[None, :]).astype(np.float64)
    return z, x


def _softmax_rows(x: np.ndarray, m: np.ndarray):
    """P and LSE of rows of x restricted to the mask m (natural log)."""
    xm = np.where(m, x, -np.inf)
    mx = xm.max(axis=1)
    has = np.isfinite(mx)
    mx_safe = np.where(has, mx, 0.0)
    e = np.where(m, np.exp(xm - mx_safe[:, None]), 0.0)
    s = e.sum(axis=1)
    lse = np.where(has, mx_safe + np.log(np.where(has, s, 1.0)), -np.inf)
    P = np.where(has[:, None], e / np.where(has, s, 1.0)[:, None], 0.0)
    return P, lse


def head_forward(q, k, v, scale: float, mods: Mods, b: int, hq: int, rows=None,
                 return_p: bool = False):
    """Forward for one (b, hq): O rows and LSE rows (fp64), full score rows.

    ``q`` is [B, Hq, N, d], ``k``/``v`` [B, Hkv, N, d] (torch or numpy).
    """
    Q = _f64(q[b, hq])
    Hq = q.shape[1]
    Hkv = k.shape[1]
    hk = hq // (Hq // Hkv)
    K = _f64(k[b, hk])
    V = _f64(v[b, hk])
    N = K.shape[0]
    rows = np.arange(Q.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(N)
    _, x = logits(Q, K, scale, mods, hq, Hq, rows, cols)
    m = allowed(mods, b, rows, cols)
    P, lse = _softmax_rows(x, m)
    O = P @ V
    if return_p:
        return O, lse, P
    return O, lse


def forward(q, k, v, scale: float, mods: Mods = None):
    """O [B, Hq, N, d] and LSE [B, Hq, N] in fp64."""
    mods = mods or Mods()
    B, Hq, N, d = q.shape
    O = np.zeros((B, Hq, N, d))
    L = np.zeros((B, Hq, N))
    for b in range(B):
        for h in range(Hq):
            O[b, h], L[b, h] = head_forward(q, k, v, scale, mods, b, h)
    return O, L


def decode_paged(q, k_cache, v_cache, block_table, seqlens, scale: float, mods: Mods = None):
    """Decode step over a paged K/V cache, in fp64.

    "Les kernels d'attention rapide et la fusion d'opérateurs accélèrent les
    modèles d'IA", section "Attention de type FlashAttention et attention
    paginée": the K/V cache grows by one token per step and is stored in
    fixed-size blocks (16 tokens in the page's example) that a block table maps
    from logical to physical positions; the attention kernel translates every
    position through that table.

    Reading taken here: ``q`` is [B, Hq, d] (one new token per sequence) or
    [B, Hq, T, d] (T new tokens, e.g. drafts to verify); token t of sequence b
    sits at position i_t = L_b - T + t, L_b = ``seqlens[b]`` counting the new
    tokens, and attends to the cached keys j = 0 .. L_b - 1 that the mods allow
    for i_t (causal j <= i_t always applies; the window keeps i_t - j < W;
    ALiBi subtracts slope * (i_t - j)).  Row j of sequence b, KV head hk is row
    j % 16 of physical block ``block_table[b, j // 16]`` of the cache
    [num_blocks, Hkv, 16, d].  A token with no allowed key (L_b = 0, or
    i_t < 0) gets O = 0, LSE = -inf.  Document masks do not apply.  Returns
    O with q's shape and LSE [B, Hq] or [B, Hq, T].
    """
    mods = mods or Mods()
    if mods.doc_ids is not None:
        raise ValueError("document masks do not apply to a decode step")
    Q = _f64(q)
    one = Q.ndim == 3
    if one:
        Q = Q[:, :, None, :]
    KC = _f64(k_cache)
    VC = _f64(v_cache)
    table = np.asarray(block_table)
    lens = np.asarray(seqlens)
    B, Hq, T, d = Q.shape
    Hkv, blk = KC.shape[1], KC.shape[2]
    G = Hq // Hkv
    causal = Mods(causal=True, window=mods.window, softcap=mods.softcap, alibi=mods.alibi,
                  alibi_slopes=mods.alibi_slopes)
    O = np.zeros((B, Hq, T, d))
    LSE = np.full((B, Hq, T), -np.inf)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        blocks = table[b, :-(-L // blk)]
        ts = [t for t in range(T) if L - T + t >= 0]  # tokens with a position
        if not ts:
            continue
        rows = np.array([L - T + t for t in ts])
        cols = np.arange(L)
        m = allowed(causal, b, rows, cols)
        for hk in range(Hkv):
            K = KC[blocks, hk].reshape(-1, d)[:L]
            V = VC[blocks, hk].reshape(-1, d)[:L]
            for hq in range(hk * G, (hk + 1) * G):
                qh = np.zeros((L, d))
                qh[rows] = Q[b, hq, ts]
                _, x = logits(qh, K, scale, causal, hq, Hq, rows, cols)
                P, lse = _softmax_rows(x, m)
                O[b, hq, ts] = P @ V
                LSE[b, hq, ts] = lse
    if one:
        return O[:, :, 0], LSE[:, :, 0]
    return O, LSE


def group_backward(q, k, v, do, scale: float, mods: Mods, b: int, hk: int):
    """dQ for the query heads of KV head ``hk`` and dK, dV of that KV head.

    Returns (heads, dQ [G, N, d], dK [N, d], dV [N, d]) in fp64.
    """
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    K = _f64(k[b, hk])
    V = _f64(v[b, hk])
    N, d = K.shape
    idx = np.arange(N)
    m = allowed(mods, b, idx, idx)
    heads = list(range(hk * G, (hk + 1) * G))
    dQ = np.zeros((G, N, d))
    dK = np.zeros((N, d))
    dV = np.zeros((N, d))
    for g, hq in enumerate(heads):
        Q = _f64(q[b, hq])
        dO = _f64(do[b, hq])
        z, x = logits(Q, K, scale, mods, hq, Hq, idx, idx)
        P, _ = _softmax_rows(x, m)
        dV += P.T @ dO
        dP = dO @ V.T
        D = (P * dP).sum(axis=1)
        dX = P * (dP - D[:, None])
        if mods.softcap is not None:
            c = float(mods.softcap)
            dZ = dX * (1.0 - np.tanh(z / c) ** 2)
        else:
            dZ = dX
        dQ[g] = scale * (dZ @ K)
        dK += scale * (dZ.T @ Q)
    return heads, dQ, dK, dV


def sampled_backward(q, k, v, do, scale: float, mods: Mods, b: int, hk: int,
                     q_rows=None, kv_rows=None):
    """Selected outputs of the backward for KV head ``hk`` of batch row ``b``.

    Returns (dQ [G, len(q_rows), d], dK [len(kv_rows), d], dV [len(kv_rows), d])
    for the query heads of the group, computed from the same definitions as
    ``group_backward``: each query head's full score matrix gives P and D, and
    only the requested rows of dQ and columns of P / dS are reduced.
    """
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    K = _f64(k[b, hk])
    V = _f64(v[b, hk])
    N, d = K.shape
    idx = np.arange(N)
    qr = idx if q_rows is None else np.asarray(q_rows)
    kr = idx if kv_rows is None else np.asarray(kv_rows)
    m = allowed(mods, b, idx, idx)
    dQ = np.zeros((G, qr.size, d))
    dK = np.zeros((kr.size, d))
    dV = np.zeros((kr.size, d))
    for g in range(G):
        hq = hk * G + g
        Q = _f64(q[b, hq])
        dO = _f64(do[b, hq])
        z, x = logits(Q, K, scale, mods, hq, Hq, idx, idx)
        P, _ = _softmax_rows(x, m)
        dP = dO @ V.T
        D = (P * dP).sum(axis=1)
        dX = P * (dP - D[:, None])
        if mods.softcap is not None:
            c = float(mods.softcap)
            dZ = dX * (1.0 - np.tanh(z / c) ** 2)
        else:
            dZ = dX
        dQ[g] = scale * (dZ[qr] @ K)
        dK += scale * (dZ[:, kr].T @ Q)
        dV += P[:, kr].T @ dO
    return dQ, dK, dV


def head_rows_backward(q, k, v, do, scale: float, mods: Mods, b: int, hq: int, rows):
    """What query rows ``rows`` of head ``hq`` contribute to the backward.

    Returns (dQ[rows] [R, d], dK part [N, d], dV part [N, d]); the full dK/dV
    of a KV head are the sums of these parts over all rows of every query head
    of its group (the sums over i in dK = scale dZ^T Q and dV = P^T dO split
    by rows).  Used to time the oracle on a bounded slice of a workload.
    """
    Hq, Hkv = q.shape[1], k.shape[1]
    hk = hq // (Hq // Hkv)
    K = _f64(k[b, hk])
    V = _f64(v[b, hk])
    N = K.shape[0]
    rows = np.asarray(rows)
    idx = np.arange(N)
    Q = _f64(q[b, hq])[rows]
    dO = _f64(do[b, hq])[rows]
    z, x = logits(_f64(q[b, hq]), K, scale, mods, hq, Hq, rows, idx)
    P, _ = _softmax_rows(x, allowed(mods, b, rows, idx))
    dP = dO @ V.T
    D = (P * dP).sum(axis=1)
    dX = P * (dP - D[:, None])
    if mods.softcap is not None:
        c = float(mods.softcap)
        dZ = dX * (1.0 - np.tanh(z / c) ** 2)
    else:
        dZ = dX
    return scale * (dZ @ K), scale * (dZ.T @ Q), P.T @ dO


def backward(q, k, v, do, scale: float, mods: Mods = None):
    """dQ [B, Hq, N, d], dK and dV [B, Hkv, N, d] in fp64."""
    mods = mods or Mods()
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    dQ = np.zeros((B, Hq, N, d))
    dK = np.zeros((B, Hkv, N, d))
    dV = np.zeros((B, Hkv, N, d))
    for b in range(B):
        for hk in range(Hkv):
            heads, gq, gk, gv = group_backward(q, k, v, do, scale, mods, b, hk)
            dQ[b, heads] = gq
            dK[b, hk] = gk
            dV[b, hk] = gv
    return dQ, dK, dV


def flop_pairs(mods: Mods, B: int, N: int) -> int:
    """Number of allowed (b, i, j) pairs summed over the batch (per head)."""
    total = 0
    idx = np.arange(N)
    for b in range(B):
        total += int(allowed(mods, b, idx, idx).sum())
    return total


def block_map(mods: Mods, B: int, N: int, tile: int = TILE) -> np.ndarray:
    """uint8 [B, nT, nT] tile classes by brute force over every element.

    Tile (I, J) covers rows [I*tile, I*tile+tile) and cols [J*tile, J*tile+tile).
    Only rows i < N matter.  SKIP (0): no pair with i < N, j < N is allowed.
    FULL (2): the column range lies inside [0, N) and every pair with i < N is
    allowed.  PARTIAL (1): otherwise.  Block-sparse skipping is named on the
    FlexAttention/FA4 page, "Limitations actuelles"; the tile size 128 is the
    one named there.
    """
    nT = (N + tile - 1) // tile
    out = np.zeros((B, nT, nT), dtype=np.uint8)
    for b in range(B):
        for I in range(nT):
            rows = np.arange(I * tile, min((I + 1) * tile, N))
            for J in range(nT):
                cols = np.arange(J * tile, min((J + 1) * tile, N))
                m = allowed(mods, b, rows, cols)
                if not m.any():
                    out[b, I, J] = MAP_SKIP
                elif m.all() and (J + 1) * tile <= N:
                    out[b, I, J] = MAP_FULL
                else:
                    out[b, I, J] = MAP_PARTIAL
    return out


# --------------------------------------------------------------------------
# FP8 path: signed Hadamard rotation and e4m3 quantisation.
# "FlashAttention-3 : une attention plus rapide ...", section "Basse précision
# FP8 et incoherent processing": Q and K are multiplied by a random orthogonal
# matrix, a Hadamard transform with random signs, per head, before FP8
# quantisation, to spread outliers.
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


def sylvester_hadamard(n: int) -> np.ndarray:
    """Natural-order Sylvester Hadamard matrix of order n (a power of two)."""
    H = np.ones((1, 1))
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    if H.shape[0] != n:
        raise ValueError("n must be a power of two")
    return H


def rotation(signs: np.ndarray) -> np.ndarray:
    """M = diag(s) H / sqrt(d): rows are rotated as x -> x M (orthogonal)."""
    s = np.asarray(signs, dtype=np.float64)
    d = s.size
    return (s[:, None] * sylvester_hadamard(d)) / np.sqrt(d)


def rotate_heads(x, signs: np.ndarray, Hkv: int) -> np.ndarray:
    """Apply each head's rotation to every row: x [B, H, N, d] -> fp64.

    Query head h uses the sign vector of its KV head h // (H // Hkv).
    """
    X = _f64(x)
    H = X.shape[1]
    G = H // Hkv
    out = np.empty_like(X)
    for h in range(H):
        out[:, h] = X[:, h] @ rotation(signs[h // G])
    return out


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even), saturating at +-448.

    e4m3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, smallest normal
    2^-6, subnormal step 2^-9, largest finite 448.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)
    q = 2.0 ** (e - 3)
    r = np.round(a / q) * q  # numpy rounds half to even
    r = np.minimum(r, E4M3_MAX)
    return np.sign(x) * r


def head_amax_scales(x: np.ndarray) -> np.ndarray:
    """Per-(b, h) scale amax / 448 of an fp64 [B, H, N, d] array (1 when all zero)."""
    amax = np.abs(x).max(axis=(2, 3))
    return np.where(amax > 0, amax / E4M3_MAX, 1.0)


def quantize_e4m3(x: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """e4m3 values of x / scale per (b, h) (returned as fp64 numbers)."""
    return e4m3_round(x / scales[:, :, None, None])


def rope(x, base: float) -> np.ndarray:
    """Rotary position embedding of every row, fp64, rotate-half pairing:
    element c < d/2 of the row at position n (its index along N) pairs with
    element c + d/2 and the pair turns by the angle n * base^(-2c/d):
    (a, b) -> (a cos - b sin, b cos + a sin).  The FA3 digest ("Basse
    précision FP8 et incoherent processing") names RoPE only as the step the
    Hadamard rotation can be fused with; this is its usual definition."""
    X = _f64(x)
    d = X.shape[-1]
    h = d // 2
    inv = base ** (-2.0 * np.arange(h) / d)
    ang = np.arange(X.shape[2], dtype=np.float64)[:, None] * inv[None, :]
    c, sn = np.cos(ang), np.sin(ang)
    a, b = X[..., :h], X[..., h:]
    return np.concatenate([a * c - b * sn, b * c + a * sn], axis=-1)


def fp8_prologue(q, k, v, signs: Optional[np.ndarray], Hkv: int, rope_base: Optional[float] = None):
    """Rotated-and-quantised Q, K (rotation skipped when signs is None; RoPE
    first when rope_base is given) and V.

    Returns (q8, k8, v8) as fp64 e4m3 values and scales [3, B, H].
    """
    if rope_base is not None:
        q, k = rope(q, rope_base), rope(k, rope_base)
    Q = rotate_heads(q, signs, Hkv) if signs is not None else _f64(q)
    K = rotate_heads(k, signs, Hkv) if signs is not None else _f64(k)
    V = _f64(v)
    sq, sk, sv = head_amax_scales(Q), head_amax_scales(K), head_amax_scales(V)
    return (quantize_e4m3(Q, sq), quantize_e4m3(K, sk), quantize_e4m3(V, sv),
            np.stack([sq, sk, sv]))
