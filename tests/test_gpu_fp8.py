"""FP8 path on the GPU: Hadamard + e4m3 prologue against the oracle's
quantiser, the e4m3 forward against the oracle run on the dequantised
inputs, and the error of the whole FP8 path against the fp64 oracle on the
original inputs, with and without the Hadamard rotation (the outlier
experiment of the FlashAttention-3 digest, "Basse précision FP8 et incoherent
processing")."""
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
from oracle import attn64
from gpu_common import LSE_TOL, lib, max_abs, record

pytestmark = pytest.mark.gpu

# The e4m3 forward rounds P to e4m3: each weight carries a relative error of
# at most 2^-4 (half of e4m3's 3-bit mantissa step), so O's relative
# Frobenius error against attention on the same dequantised inputs stays
# below 2^-4.  LSE is accumulated from the unrounded weights (LSE_TOL).
FP8_O_REL = 2.0 ** -4


def _dec(codes: torch.Tensor) -> np.ndarray:
    return codes.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _quantum(x):
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return 2.0 ** (np.clip(e, -6, 8) - 3)


def _prologue(B, Hq, Hkv, N, seed, rotate):
    ea = lib()
    x = gen.make_inputs(B, Hq, Hkv, N, 128, seed, need_do=False, outlier_frac=1e-3, outlier_scale=50.0)
    signs = gen.hadamard_signs(Hkv, 128, seed + 20)
    dev = {k: v.cuda() for k, v in x.items()}
    dsig = torch.from_numpy(signs).cuda() if rotate else None
    q8, k8, v8, sc = ea.hadamard_quant_fp8(dev["q"], dev["k"], dev["v"], dsig)
    ea.attn_status()
    return x, signs, (q8, k8, v8, sc)


@pytest.mark.parametrize("rotate", [True, False], ids=["hadamard", "plain"])
# N < 256 and N = 1: one 256-row stage holds rows of many heads (per-row
# sign heads and amax atomics); N = 300, 1000: stages straddle two heads.
@pytest.mark.parametrize("shape", [(1, 4, 2, 300), (2, 2, 2, 1000), (1, 6, 3, 100), (2, 6, 3, 1)], ids=str)
def test_prologue_matches_oracle(rotate, shape):
    B, Hq, Hkv, N = shape
    x, signs, (q8, k8, v8, sc) = _prologue(B, Hq, Hkv, N, 7 + N, rotate)
    sc = sc.cpu().numpy().astype(np.float64)
    parts = [(q8, x["q"], Hq, 0, True), (k8, x["k"], Hkv, B * Hq, True),
             (v8, x["v"], Hkv, B * Hq + B * Hkv, False)]
    for codes, src, H, off, rot in parts:
        ref = attn64.rotate_heads(src, signs, Hkv) if (rotate and rot) else attn64._f64(src)
        s_ref = attn64.head_amax_scales(ref)
        s_gpu = sc[off:off + B * H].reshape(B, H)
        np.testing.assert_allclose(s_gpu, s_ref, rtol=2e-6)
        exact = ref / s_ref[:, :, None, None]
        dec = _dec(codes)
        # within one e4m3 step of the exact value; almost always the same code
        assert (np.abs(dec - exact) <= _quantum(exact) + 1e-12).all()
        same = (dec == attn64.e4m3_round(exact)).mean()
        assert same > 0.999, same


# RoPE angles are formed in fp32 on the GPU (position x an fp32 inverse
# frequency): at position n they are off by up to about 3 n 2^-24 radians
# (~4e-4 at n = 2100), which moves each rotated element by at most that
# fraction of its row's largest element.
ROPE_REL = 1e-3


@pytest.mark.parametrize("rotate", [True, False], ids=["hadamard", "plain"])
@pytest.mark.parametrize("shape", [(1, 4, 2, 300), (2, 2, 1, 2100), (1, 6, 3, 100)], ids=str)
def test_rope_prologue_matches_oracle(rotate, shape):
    """RoPE fused in front of the Hadamard rotation and the quantiser."""
    ea = lib()
    B, Hq, Hkv, N = shape
    base = 10000.0
    x = gen.make_inputs(B, Hq, Hkv, N, 128, 17 + N, need_do=False, outlier_frac=1e-3, outlier_scale=50.0)
    signs = gen.hadamard_signs(Hkv, 128, 37 + N)
    dev = {k: v.cuda() for k, v in x.items()}
    dsig = torch.from_numpy(signs).cuda() if rotate else None
    q8, k8, v8, sc = ea.hadamard_quant_fp8(dev["q"], dev["k"], dev["v"], dsig, rope_base=base)
    ea.attn_status()
    sc = sc.cpu().numpy().astype(np.float64)
    parts = [(q8, x["q"], Hq, 0, True), (k8, x["k"], Hkv, B * Hq, True),
             (v8, x["v"], Hkv, B * Hq + B * Hkv, False)]
    for codes, src, H, off, rot in parts:
        ref = attn64.rope(src, base) if rot else attn64._f64(src)
        if rotate and rot:
            ref = attn64.rotate_heads(ref, signs, Hkv)
        s_ref = attn64.head_amax_scales(ref)
        s_gpu = sc[off:off + B * H].reshape(B, H)
        np.testing.assert_allclose(s_gpu, s_ref, rtol=ROPE_REL if rot else 2e-6)
        exact = ref / s_ref[:, :, None, None]
        dec = _dec(codes)
        slack = ROPE_REL * np.abs(exact).max(axis=-1, keepdims=True) + 1e-12 if rot else 1e-12
        assert (np.abs(dec - exact) <= _quantum(exact) + slack).all()
        same = (dec == attn64.e4m3_round(exact)).mean()
        assert same > 0.995, same


def test_fp8_forward_matches_attention_on_dequantised_inputs():
    ea = lib()
    B, Hq, Hkv, N = 1, 4, 2, 700
    x, signs, (q8, k8, v8, sc) = _prologue(B, Hq, Hkv, N, 11, True)
    s = 1.0 / math.sqrt(128)
    for mods, om in [(None, attn64.Mods()), (ea.make_mods(causal=True), attn64.Mods(causal=True))]:
        o, lse = ea.forward_fp8(q8, k8, v8, sc, s, mods)
        ea.attn_status()
        scn = sc.cpu().numpy().astype(np.float64)
        qd = _dec(q8) * scn[:B * Hq].reshape(B, Hq)[:, :, None, None]
        kd = _dec(k8) * scn[B * Hq:B * Hq + B * Hkv].reshape(B, Hkv)[:, :, None, None]
        vd = _dec(v8) * scn[B * Hq + B * Hkv:].reshape(B, Hkv)[:, :, None, None]
        O, L = attn64.forward(qd, kd, vd, s, om)
        og = o.float().cpu().numpy()
        rel = np.linalg.norm(og - O) / np.linalg.norm(O)
        assert rel <= FP8_O_REL, rel
        assert max_abs(lse.cpu().numpy(), L) <= LSE_TOL


def test_fp8_outlier_workload_hadamard_lowers_error():
    """Full-size outlier workload: RMSE of O against the fp64 oracle on the
    original bf16 inputs, FP8 with vs without the rotation (sampled rows)."""
    ea = lib()
    cfg = gen.WORKLOADS["fp8_outliers_16k"]
    B, Hq, Hkv, N = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["N"]
    x = gen.make_inputs(**cfg, need_do=False)
    signs = torch.from_numpy(gen.hadamard_signs(Hkv, 128, cfg["seed"] + 20)).cuda()
    dev = {k: v.cuda() for k, v in x.items()}
    s = 1.0 / math.sqrt(128)
    outs = {}
    for name, sg in (("hadamard", signs), ("plain", None)):
        q8, k8, v8, sc = ea.hadamard_quant_fp8(dev["q"], dev["k"], dev["v"], sg)
        o, lse = ea.forward_fp8(q8, k8, v8, sc, s)
        ea.attn_status()
        outs[name] = o.float().cpu().numpy()
        assert np.isfinite(outs[name]).all()
    rng = np.random.default_rng(3)
    err = {"hadamard": [], "plain": []}
    for b, h in ((0, 0), (1, 9)):
        rows = np.sort(rng.choice(N, size=256, replace=False))
        O, _ = attn64.head_forward(x["q"], x["k"], x["v"], s, attn64.Mods(), b, h, rows=rows)
        for name in err:
            err[name].append((outs[name][b, h, rows] - O).ravel())
    rmse = {k: float(np.sqrt(np.mean(np.concatenate(v) ** 2))) for k, v in err.items()}
    print(f"fp8 outlier workload RMSE(O): {rmse} ratio {rmse['plain'] / rmse['hadamard']:.2f}")
    record("fp8_outliers_16k", "RMSE_O_hadamard", rmse["hadamard"])
    record("fp8_outliers_16k", "RMSE_O_plain", rmse["plain"])
    assert rmse["hadamard"] < rmse["plain"]
