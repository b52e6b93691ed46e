"""Pins for the fp64 oracle: each check ties it to something other than itself.

Closed forms, library special cases (torch CPU float64 SDPA and autograd,
scipy's Hadamard, torch's e4m3 cast), an independent scalar-loop
implementation, and central finite differences.  CPU only.
"""
import itertools
import math

import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import attn64 as A
from oracle import brute
import attn_inputs as gen


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _docs(B, N, seed):
    rng = np.random.default_rng(seed)
    out = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        cuts = np.sort(rng.choice(np.arange(1, N), size=2, replace=False))
        out[b] = np.searchsorted(cuts, np.arange(N), side="right")
    return out


MOD_CASES = {
    "none": dict(),
    "causal": dict(causal=True),
    "window": dict(window=3),
    "causal_window": dict(causal=True, window=3),
    "doc": dict(doc=True),
    "causal_doc": dict(causal=True, doc=True),
    "softcap": dict(softcap=2.0),
    "alibi": dict(alibi=True),
    "all": dict(causal=True, window=4, doc=True, softcap=2.0, alibi=True),
}


def _mods(case, B, N, seed=7):
    c = MOD_CASES[case]
    return A.Mods(causal=c.get("causal", False), window=c.get("window"),
                  doc_ids=_docs(B, N, seed) if c.get("doc") else None,
                  softcap=c.get("softcap"), alibi=c.get("alibi", False))


# ---------------------------------------------------------------- forward pins

@pytest.mark.parametrize("case", list(MOD_CASES))
def test_forward_matches_scalar_loops(case):
    B, Hq, Hkv, N, d = 2, 4, 2, 9, 4
    q, k, v = _rand((B, Hq, N, d), 1), _rand((B, Hkv, N, d), 2), _rand((B, Hkv, N, d), 3)
    mods = _mods(case, B, N)
    scale = 0.7
    O, L = A.forward(q, k, v, scale, mods)
    slopes = list(A.alibi_slopes(Hq)) if mods.alibi else None
    Ob, Lb = brute.forward(q, k, v, scale, causal=mods.causal, window=mods.window,
                           doc=mods.doc_ids, softcap=mods.softcap, slopes=slopes)
    np.testing.assert_allclose(O, np.array(Ob), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(L, np.array(Lb), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", list(MOD_CASES))
def test_softmax_rows_sum_to_one(case):
    B, Hq, Hkv, N, d = 1, 2, 1, 11, 5
    q, k, v = _rand((B, Hq, N, d), 4), _rand((B, Hkv, N, d), 5), _rand((B, Hkv, N, d), 6)
    mods = _mods(case, B, N)
    for h in range(Hq):
        _, lse, P = A.head_forward(q, k, v, 0.5, mods, 0, h, return_p=True)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert (P >= 0).all()
        m = A.allowed(mods, 0, np.arange(N), np.arange(N))
        assert (P[~m] == 0).all()


@pytest.mark.parametrize("case", list(MOD_CASES))
def test_constant_v_returns_v(case):
    B, Hq, Hkv, N, d = 1, 2, 2, 10, 3
    q, k = _rand((B, Hq, N, d), 7), _rand((B, Hkv, N, d), 8)
    row = np.array([0.25, -1.5, 3.0])
    v = np.broadcast_to(row, (B, Hkv, N, d)).copy()
    O, _ = A.forward(q, k, v, 0.9, _mods(case, B, N))
    np.testing.assert_allclose(O, np.broadcast_to(row, O.shape), rtol=0, atol=1e-13)


def test_causal_row_zero_and_single_key():
    B, Hq, N, d = 1, 3, 6, 4
    q, k, v = _rand((B, Hq, N, d), 9), _rand((B, Hq, N, d), 10), _rand((B, Hq, N, d), 11)
    scale = 0.3
    O, L = A.forward(q, k, v, scale, A.Mods(causal=True))
    for h in range(Hq):
        np.testing.assert_allclose(O[0, h, 0], v[0, h, 0], rtol=0, atol=1e-15)
        assert L[0, h, 0] == pytest.approx(scale * float(q[0, h, 0] @ k[0, h, 0]), abs=1e-14)
    # N = 1: the only key is attended with weight 1.
    q1, k1, v1 = q[:, :, :1], k[:, :, :1], v[:, :, :1]
    O1, L1 = A.forward(q1, k1, v1, scale)
    np.testing.assert_allclose(O1, v1, rtol=0, atol=1e-15)
    np.testing.assert_allclose(L1[..., 0], scale * np.einsum("bhd,bhd->bh", q1[:, :, 0], k1[:, :, 0]),
                               atol=1e-14)


def _sdpa64(q, k, v, scale, mask=None, bias=None, causal=False):
    Hq, Hkv = q.shape[1], k.shape[1]
    rep = Hq // Hkv
    Q = torch.from_numpy(np.ascontiguousarray(q))
    K = torch.from_numpy(np.repeat(k, rep, axis=1))
    V = torch.from_numpy(np.repeat(v, rep, axis=1))
    am = None
    if mask is not None or bias is not None:
        am = torch.zeros(q.shape[0], Hq, q.shape[2], k.shape[2], dtype=torch.float64)
        if bias is not None:
            am = am + torch.from_numpy(bias)
        if mask is not None:
            am = am.masked_fill(~torch.from_numpy(mask), float("-inf"))
    return torch.nn.functional.scaled_dot_product_attention(
        Q, K, V, attn_mask=am, is_causal=causal, scale=scale).numpy()


def test_matches_torch_sdpa_float64():
    B, Hq, Hkv, N, d = 2, 4, 2, 33, 8
    q, k, v = _rand((B, Hq, N, d), 12), _rand((B, Hkv, N, d), 13), _rand((B, Hkv, N, d), 14)
    s = 1 / math.sqrt(d)
    O, _ = A.forward(q, k, v, s)
    np.testing.assert_allclose(O, _sdpa64(q, k, v, s), rtol=1e-12, atol=1e-12)
    O, _ = A.forward(q, k, v, s, A.Mods(causal=True))
    np.testing.assert_allclose(O, _sdpa64(q, k, v, s, causal=True), rtol=1e-12, atol=1e-12)
    # ALiBi as an additive bias and window/doc as a boolean mask, built by hand here.
    docs = _docs(B, N, 3)
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    slopes = 2.0 ** (-8.0 * (np.arange(Hq) + 1) / Hq)
    bias = -slopes[None, :, None, None] * (i - j)[None, None]
    bias = np.broadcast_to(bias, (B, Hq, N, N)).copy()
    mask = np.broadcast_to(((j <= i) & (i - j < 7))[None, None], (B, Hq, N, N)).copy()
    mask &= (docs[:, None, :, None] == docs[:, None, None, :])
    O, _ = A.forward(q, k, v, s, A.Mods(causal=True, window=7, doc_ids=docs, alibi=True))
    np.testing.assert_allclose(O, _sdpa64(q, k, v, s, mask=mask, bias=bias), rtol=1e-12, atol=1e-12)


def test_mod_reductions():
    B, Hq, Hkv, N, d = 2, 2, 1, 12, 4
    q, k, v = _rand((B, Hq, N, d), 15), _rand((B, Hkv, N, d), 16), _rand((B, Hkv, N, d), 17)
    causal = A.forward(q, k, v, 0.8, A.Mods(causal=True))
    plain = A.forward(q, k, v, 0.8)
    # A window at least N wide changes nothing.
    for ref, mods in [(causal, A.Mods(causal=True, window=N)), (plain, A.Mods(window=N + 5))]:
        got = A.forward(q, k, v, 0.8, mods)
        np.testing.assert_array_equal(got[0], ref[0])
    # One document is no mask.
    got = A.forward(q, k, v, 0.8, A.Mods(causal=True, doc_ids=np.zeros((B, N), np.int32)))
    np.testing.assert_array_equal(got[0], causal[0])
    # A huge soft-cap is the identity.
    got = A.forward(q, k, v, 0.8, A.Mods(softcap=1e12))
    np.testing.assert_allclose(got[0], plain[0], rtol=1e-12, atol=1e-12)
    # ALiBi with zero slopes is no bias.
    got = A.forward(q, k, v, 0.8, A.Mods(alibi=True, alibi_slopes=np.zeros(Hq)))
    np.testing.assert_array_equal(got[0], plain[0])


def test_gqa_equals_repeated_kv():
    B, Hq, Hkv, N, d = 1, 6, 2, 8, 4
    q, k, v, do = (_rand((B, Hq, N, d), 18), _rand((B, Hkv, N, d), 19),
                   _rand((B, Hkv, N, d), 20), _rand((B, Hq, N, d), 21))
    mods = A.Mods(causal=True, softcap=3.0)
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    O, L = A.forward(q, k, v, 0.6, mods)
    Or, Lr = A.forward(q, kr, vr, 0.6, mods)
    np.testing.assert_allclose(O, Or, atol=1e-14)
    np.testing.assert_allclose(L, Lr, atol=1e-14)
    dq, dk, dv = A.backward(q, k, v, do, 0.6, mods)
    dqr, dkr, dvr = A.backward(q, kr, vr, do, 0.6, mods)
    np.testing.assert_allclose(dq, dqr, atol=1e-13)
    np.testing.assert_allclose(dk, dkr.reshape(B, Hkv, 3, N, d).sum(axis=2), atol=1e-13)
    np.testing.assert_allclose(dv, dvr.reshape(B, Hkv, 3, N, d).sum(axis=2), atol=1e-13)


# --------------------------------------------------------------- backward pins

@pytest.mark.parametrize("case", ["none", "causal", "causal_window", "doc", "softcap",
                                  "alibi", "all"])
def test_backward_finite_differences(case):
    B, Hq, Hkv, N, d = 1, 2, 1, 6, 3
    q, k, v, do = (_rand((B, Hq, N, d), 22), _rand((B, Hkv, N, d), 23),
                   _rand((B, Hkv, N, d), 24), _rand((B, Hq, N, d), 25))
    mods = _mods(case, B, N)
    scale = 1.3

    def loss(qq, kk, vv):
        return float((A.forward(qq, kk, vv, scale, mods)[0] * do).sum())

    dq, dk, dv = A.backward(q, k, v, do, scale, mods)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in itertools.product(*[range(s) for s in x.shape]):
            old = x[idx]
            x[idx] = old + h
            lp = loss(q, k, v)
            x[idx] = old - h
            lm = loss(q, k, v)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_backward_matches_torch_autograd_sdpa():
    B, Hq, Hkv, N, d = 2, 4, 2, 17, 8
    q, k, v, do = (_rand((B, Hq, N, d), 26), _rand((B, Hkv, N, d), 27),
                   _rand((B, Hkv, N, d), 28), _rand((B, Hq, N, d), 29))
    s = 1 / math.sqrt(d)
    Q = torch.from_numpy(q.copy()).requires_grad_()
    K = torch.from_numpy(k.copy()).requires_grad_()
    V = torch.from_numpy(v.copy()).requires_grad_()
    O = torch.nn.functional.scaled_dot_product_attention(
        Q, K.repeat_interleave(2, dim=1), V.repeat_interleave(2, dim=1), is_causal=True, scale=s)
    O.backward(torch.from_numpy(do))
    dq, dk, dv = A.backward(q, k, v, do, s, A.Mods(causal=True))
    np.testing.assert_allclose(dq, Q.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, K.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, V.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_sampled_backward_matches_full():
    B, Hq, Hkv, N, d = 2, 4, 2, 12, 4
    q, k, v, do = (_rand((B, Hq, N, d), 60), _rand((B, Hkv, N, d), 61),
                   _rand((B, Hkv, N, d), 62), _rand((B, Hq, N, d), 63))
    mods = _mods("all", B, N)
    dq, dk, dv = A.backward(q, k, v, do, 0.9, mods)
    rows, cols = np.array([0, 5, 11]), np.array([1, 2, 10])
    gq, gk, gv = A.sampled_backward(q, k, v, do, 0.9, mods, 1, 1, rows, cols)
    np.testing.assert_allclose(gq, dq[1, 2:4][:, rows], atol=1e-13)
    np.testing.assert_allclose(gk, dk[1, 1, cols], atol=1e-13)
    np.testing.assert_allclose(gv, dv[1, 1, cols], atol=1e-13)


def test_row_slices_sum_to_full_backward():
    B, Hq, Hkv, N, d = 1, 4, 2, 11, 3
    q, k, v, do = (_rand((B, Hq, N, d), 64), _rand((B, Hkv, N, d), 65),
                   _rand((B, Hkv, N, d), 66), _rand((B, Hq, N, d), 67))
    mods = _mods("all", B, N)
    dq, dk, dv = A.backward(q, k, v, do, 0.8, mods)
    for hk in range(Hkv):
        gk = np.zeros((N, d))
        gv = np.zeros((N, d))
        for hq in (2 * hk, 2 * hk + 1):
            for rows in (np.arange(0, 4), np.arange(4, 11)):
                a, b_, c = A.head_rows_backward(q, k, v, do, 0.8, mods, 0, hq, rows)
                np.testing.assert_allclose(a, dq[0, hq, rows], atol=1e-13)
                gk += b_
                gv += c
        np.testing.assert_allclose(gk, dk[0, hk], atol=1e-13)
        np.testing.assert_allclose(gv, dv[0, hk], atol=1e-13)


def test_delta_identity():
    """rowsum(dO * O) equals rowsum(P * dP): the preprocessing shortcut is exact."""
    B, Hq, N, d = 1, 1, 9, 5
    q, k, v, do = (_rand((B, Hq, N, d), s) for s in (30, 31, 32, 33))
    mods = A.Mods(causal=True, softcap=2.5, alibi=True)
    O, lse, P = A.head_forward(q, k, v, 0.7, mods, 0, 0, return_p=True)
    dP = do[0, 0] @ v[0, 0].T
    np.testing.assert_allclose((do[0, 0] * O).sum(1), (P * dP).sum(1), rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------- block map pins

@pytest.mark.parametrize("case", ["none", "causal", "window", "causal_window", "doc", "all"])
@pytest.mark.parametrize("N", [8, 13, 16])
def test_block_map_brute_force(case, N):
    B = 2
    mods = _mods(case, B, N, seed=N)
    got = A.block_map(mods, B, N, tile=4)
    ref = brute.tile_class(B, N, 4, causal=mods.causal, window=mods.window, doc=mods.doc_ids)
    np.testing.assert_array_equal(got, np.array(ref, dtype=np.uint8))


def test_block_map_closed_forms():
    N, T = 1000, 128
    nT = 8
    causal = A.block_map(A.Mods(causal=True), 1, N, T)[0]
    I, J = np.meshgrid(np.arange(nT), np.arange(nT), indexing="ij")
    expect = np.where(J < I, 2, np.where(J == I, 1, 0))
    np.testing.assert_array_equal(causal, expect)
    plain = A.block_map(A.Mods(), 1, N, T)[0]
    np.testing.assert_array_equal(plain, np.where(J == nT - 1, 1, 2))  # ragged last column
    full = A.block_map(A.Mods(), 1, 1024, T)[0]
    assert (full == 2).all()


def test_flop_pairs_causal():
    assert A.flop_pairs(A.Mods(causal=True), 3, 50) == 3 * 50 * 51 // 2
    assert A.flop_pairs(A.Mods(), 1, 50) == 2500


# ------------------------------------------------------------------- FP8 pins

def test_hadamard_is_scipy_and_rotation_orthogonal():
    np.testing.assert_array_equal(A.sylvester_hadamard(128), scipy.linalg.hadamard(128))
    s = gen.hadamard_signs(1, 128, 3)[0]
    M = A.rotation(s)
    np.testing.assert_allclose(M @ M.T, np.eye(128), atol=1e-13)
    x = _rand(128, 5)
    fw = np.array(brute.fwht(x * s)) / math.sqrt(128)
    np.testing.assert_allclose(x @ M, fw, atol=1e-12)


def test_rotation_leaves_attention_unchanged():
    B, Hq, Hkv, N, d = 1, 4, 2, 20, 128
    q, k, v = _rand((B, Hq, N, d), 40), _rand((B, Hkv, N, d), 41), _rand((B, Hkv, N, d), 42)
    signs = gen.hadamard_signs(Hkv, d, 43)
    qr, kr = A.rotate_heads(q, signs, Hkv), A.rotate_heads(k, signs, Hkv)
    for mods in (A.Mods(), A.Mods(causal=True)):
        O, L = A.forward(q, k, v, 0.1, mods)
        Or, Lr = A.forward(qr, kr, v, 0.1, mods)
        np.testing.assert_allclose(Or, O, atol=1e-12)
        np.testing.assert_allclose(Lr, L, atol=1e-12)


def test_e4m3_round_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 30, rng.standard_normal(5000) * 1e-2,
                        np.linspace(-448, 448, 4001)])
    ref = torch.from_numpy(x).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    # torch's fp32 round trip could differ from fp64 only at exact fp32 ties; x is fp64 here,
    # so compare on values exactly representable in fp32.
    x32 = x.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x32).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(A.e4m3_round(x32), ref)
    # saturation and ties to even
    assert A.e4m3_round(np.array([500.0, -1e9]))[0] == 448.0
    assert A.e4m3_round(np.array([-1e9]))[0] == -448.0
    assert A.e4m3_round(np.array([1.0625]))[0] == 1.0     # tie between 1.0 and 1.125 -> even
    assert A.e4m3_round(np.array([1.1875]))[0] == 1.25    # tie between 1.125 and 1.25 -> even
    assert A.e4m3_round(np.array([2.0 ** -10]))[0] == 0.0  # half of the smallest subnormal


def test_fp8_prologue_scales_and_range():
    B, H, N, d = 1, 2, 64, 128
    q, k, v = _rand((B, H, N, d), 50), _rand((B, H, N, d), 51), _rand((B, H, N, d), 52)
    signs = gen.hadamard_signs(H, d, 53)
    q8, k8, v8, sc = A.fp8_prologue(q, k, v, signs, H)
    qr = A.rotate_heads(q, signs, H)
    np.testing.assert_allclose(sc[0], np.abs(qr).max(axis=(2, 3)) / 448.0)
    assert np.abs(q8).max() == 448.0 and np.abs(k8).max() == 448.0 and np.abs(v8).max() == 448.0
    # dequantised values sit within half an e4m3 step of the rotated inputs
    deq = q8 * sc[0][:, :, None, None]
    rel = np.abs(deq - qr) / np.maximum(np.abs(qr), 2.0 ** -6 * sc[0].max())
    assert rel.max() <= 2.0 ** -4 + 1e-12


# ---------------------------------------------------------- input recipe pins

def test_doc_lengths_recipe():
    for seed in range(20):
        lens = gen.doc_lengths(4096, seed)
        assert sum(lens) == 4096
        assert all(128 <= n <= 2048 for n in lens[:-1])
        assert 1 <= lens[-1] <= 2048
    ids = gen.doc_ids(3, 4096, 10)
    assert ids.shape == (3, 4096) and (np.diff(ids, axis=1) >= 0).all()


def test_outlier_recipe():
    x = torch.ones(1000, 100)
    y = gen.with_outliers(x, 1e-3, 50.0, 1)
    assert int((y == 50.0).sum()) == 100 and int((y == 1.0).sum()) == 100000 - 100


def _seq_ids(cu, total):
    ids = np.zeros(total, dtype=np.int32)
    for s_ in range(len(cu) - 1):
        ids[cu[s_]:cu[s_ + 1]] = s_
    return ids


@pytest.mark.parametrize("mk", [dict(causal=True), dict(causal=True, window=5),
                                dict(softcap=3.0, alibi=True), dict()])
def test_packed_sequences_equal_separate_runs(mk):
    """Packed variable-length sequences (document mask from the sequence
    offsets) give, row for row, the attention of each sequence run alone --
    forward and backward."""
    lens = [7, 1, 13, 4]
    cu = np.concatenate([[0], np.cumsum(lens)])
    total, d, Hq, Hkv = int(cu[-1]), 16, 4, 2
    x = gen.make_inputs(1, Hq, Hkv, total, d, 41)
    s = 0.3
    packed = A.Mods(doc_ids=_seq_ids(cu, total)[None, :], **mk)
    O, L = A.forward(x["q"], x["k"], x["v"], s, packed)
    gq, gk, gv = A.backward(x["q"], x["k"], x["v"], x["do"], s, packed)
    for a, b in zip(cu[:-1], cu[1:]):
        sl = {n: x[n][:, :, a:b] for n in ("q", "k", "v", "do")}
        m1 = A.Mods(**mk)
        O1, L1 = A.forward(sl["q"], sl["k"], sl["v"], s, m1)
        g1 = A.backward(sl["q"], sl["k"], sl["v"], sl["do"], s, m1)
        np.testing.assert_allclose(O[:, :, a:b], O1, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L[:, :, a:b], L1, rtol=0, atol=1e-12)
        for full, part in zip((gq, gk, gv), g1):
            np.testing.assert_allclose(full[:, :, a:b], part, rtol=0, atol=1e-12)


def test_rope_closed_forms():
    """RoPE: identity at position 0; a d = 2 row turns by exactly n radians at
    position n (its only frequency is base^0 = 1); row norms are kept."""
    x = np.zeros((1, 1, 5, 2))
    x[..., 0] = 1.0
    r = A.rope(x, 10000.0)
    n = np.arange(5)
    np.testing.assert_allclose(r[0, 0, :, 0], np.cos(n), atol=1e-15)
    np.testing.assert_allclose(r[0, 0, :, 1], np.sin(n), atol=1e-15)
    y = np.random.default_rng(3).standard_normal((2, 3, 17, 8))
    ry = A.rope(y, 500.0)
    np.testing.assert_allclose(ry[:, :, 0], y[:, :, 0], atol=0)
    np.testing.assert_allclose(np.linalg.norm(ry, axis=-1), np.linalg.norm(y, axis=-1), rtol=1e-13)


def test_rope_scores_depend_on_relative_position_only():
    """<rope(q)[n], rope(k)[m]> is a function of n - m: the same q and k
    vectors placed at every position give a Toeplitz score matrix."""
    rng = np.random.default_rng(5)
    qv, kv = rng.standard_normal(16), rng.standard_normal(16)
    N = 12
    q = np.broadcast_to(qv, (1, 1, N, 16)).copy()
    k = np.broadcast_to(kv, (1, 1, N, 16)).copy()
    S = A.rope(q, 100.0)[0, 0] @ A.rope(k, 100.0)[0, 0].T
    for t in range(-N + 1, N):
        diag = np.diagonal(S, offset=t)
        np.testing.assert_allclose(diag, diag[0], rtol=1e-12, atol=1e-12)
    assert not np.allclose(S[0, 0], S[0, 1])  # and does depend on it


# ---------------------------------------------------------------------------
# Decode over a paged K/V cache ("Les kernels d'attention rapide ...", section
# "Attention de type FlashAttention et attention paginée": block table from
# logical to physical blocks of 16 tokens).

def _paged_case(B, Hq, Hkv, lens, d, seed, spare=3, blk=16):
    rng = np.random.default_rng(seed)
    nbs = [-(-L // blk) for L in lens]
    width = max(max(nbs), 1)
    num_blocks = sum(nbs) + spare
    perm = rng.permutation(num_blocks)
    table = np.full((B, width), -1, dtype=np.int32)  # unused entries: never read
    used = 0
    for b, nb in enumerate(nbs):
        table[b, :nb] = perm[used:used + nb]
        used += nb
    q = rng.standard_normal((B, Hq, d))
    kc = rng.standard_normal((num_blocks, Hkv, blk, d))
    vc = rng.standard_normal((num_blocks, Hkv, blk, d))
    return q, kc, vc, table, np.asarray(lens)


DECODE_MODS = {
    "none": dict(),
    "window": dict(window=5),
    "softcap_alibi": dict(softcap=2.0, alibi=True),
    "all": dict(window=9, softcap=3.0, alibi=True),
}


@pytest.mark.parametrize("T", [1, 3], ids=["one_token", "three_tokens"])
@pytest.mark.parametrize("mk", list(DECODE_MODS), ids=list(DECODE_MODS))
def test_decode_matches_brute_force_last_rows(mk, T):
    """The decode step equals the last T rows of the causal brute-force forward
    run on the sequence's rows, gathered here by an explicit loop over
    positions, with the new tokens' queries in those rows."""
    B, Hq, Hkv, d = 2, 4, 2, 8
    lens = [37, 17]
    q, kc, vc, table, sl = _paged_case(B, Hq, Hkv, lens, d, seed=11)
    if T > 1:
        q = np.random.default_rng(12).standard_normal((B, Hq, T, d))
    cfg = DECODE_MODS[mk]
    slopes = list(A.alibi_slopes(Hq)) if cfg.get("alibi") else None
    O, L = A.decode_paged(q, kc, vc, table, sl, 0.4, A.Mods(causal=True, **cfg))
    if T == 1:
        O, L = O[:, :, None], L[:, :, None]
        q = q[:, :, None]
    for b, n in enumerate(lens):
        K = [[[float(x) for x in kc[table[b, j // 16], hk, j % 16]] for j in range(n)] for hk in range(Hkv)]
        V = [[[float(x) for x in vc[table[b, j // 16], hk, j % 16]] for j in range(n)] for hk in range(Hkv)]
        Qrows = [[[0.0] * d for _ in range(n - T)] + [list(q[b, h, t]) for t in range(T)] for h in range(Hq)]
        Ob, Lb = brute.forward([Qrows], [K], [V], 0.4, causal=True, window=cfg.get("window"),
                               softcap=cfg.get("softcap"), slopes=slopes)
        for h in range(Hq):
            for t in range(T):
                np.testing.assert_allclose(O[b, h, t], Ob[0][h][n - T + t], rtol=1e-12, atol=1e-12)
                np.testing.assert_allclose(L[b, h, t], Lb[0][h][n - T + t], rtol=1e-12, atol=1e-12)


def test_decode_tokens_before_the_cache_start_are_empty():
    """With more new tokens than cached positions, the tokens at negative
    positions have no key: O = 0, LSE = -inf; the others are unaffected."""
    B, Hq, Hkv, d, T = 1, 2, 1, 8, 4
    q, kc, vc, table, sl = _paged_case(B, Hq, Hkv, [2], d, seed=3)
    q4 = np.random.default_rng(4).standard_normal((B, Hq, T, d))
    O, L = A.decode_paged(q4, kc, vc, table, sl, 0.5)
    assert np.all(O[:, :, :2] == 0.0) and np.all(np.isneginf(L[:, :, :2]))
    O2, L2 = A.decode_paged(q4[:, :, 2:], kc, vc, table, sl, 0.5)
    np.testing.assert_array_equal(O[:, :, 2:], O2)
    np.testing.assert_array_equal(L[:, :, 2:], L2)


def test_decode_closed_forms():
    B, Hq, Hkv, d = 3, 2, 1, 8
    q, kc, vc, table, sl = _paged_case(B, Hq, Hkv, [1, 0, 21], d, seed=5)
    O, L = A.decode_paged(q, kc, vc, table, sl, 0.5, A.Mods(causal=True))
    # one cached token: O is its value row, LSE its score
    v0, k0 = vc[table[0, 0], 0, 0], kc[table[0, 0], 0, 0]
    for h in range(Hq):
        np.testing.assert_allclose(O[0, h], v0, rtol=1e-14)
        np.testing.assert_allclose(L[0, h], 0.5 * q[0, h] @ k0, rtol=1e-14)
    # empty sequence: O = 0, LSE = -inf
    assert np.all(O[1] == 0.0) and np.all(np.isneginf(L[1]))
    # window 1: only the newest token itself
    Ow, _ = A.decode_paged(q, kc, vc, table, sl, 0.5, A.Mods(causal=True, window=1))
    np.testing.assert_allclose(Ow[2, 0], vc[table[2, 20 // 16], 0, 20 % 16], rtol=1e-14)
    # constant values: O is that constant
    vconst = np.full_like(vc, 0.75)
    Oc, _ = A.decode_paged(q, kc, vconst, table, sl, 0.5)
    np.testing.assert_allclose(Oc[[0, 2]], 0.75, rtol=1e-14)


def test_decode_block_placement_is_invisible():
    """Moving the physical blocks (and the table with them) changes nothing."""
    B, Hq, Hkv, d = 2, 4, 2, 8
    q, kc, vc, table, sl = _paged_case(B, Hq, Hkv, [40, 33], d, seed=9)
    O, L = A.decode_paged(q, kc, vc, table, sl, 0.3, A.Mods(alibi=True))
    perm = np.random.default_rng(1).permutation(kc.shape[0])  # new slot of each block
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1)
    O2, L2 = A.decode_paged(q, kc2, vc2, table2, sl, 0.3, A.Mods(alibi=True))
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
