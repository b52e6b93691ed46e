"""C ABI checks that need no GPU: the library loads, exports every function
include/attn.h declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from exact_attention_66_gb300 import _lib
    return _lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attn_fwd", "attn_bwd", "attn_fwd_fp8", "attn_hadamard_quant_fp8", "attn_block_map",
              "attn_workspace_size", "attn_status", "attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    so = ctypes.CDLL(L.LIB_PATH)
    for n in declared_functions():
        assert hasattr(so, n), n
    assert set(L.EXPORTS) <= set(declared_functions())


A = 0x10000  # an aligned, never-dereferenced address


def fwd(L, q=A, k=A, v=A, o=A, lse=A, B=1, Hq=2, Hkv=2, N=128, d=128, scale=0.1, mods=None,
        ws=None, nws=0):
    return L.lib().attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, scale,
                            ctypes.byref(mods) if mods else None, ws, nws, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(N=0), 1), (dict(Hq=0), 1), (dict(q=None), 1), (dict(lse=None), 1),
    (dict(d=96), 2), (dict(d=256), 2), (dict(Hq=3, Hkv=2), 2), (dict(q=A + 8), 2),
    (dict(lse=A + 2), 2), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(scale=0.0), 1), (dict(scale=-0.1), 1),
])
def test_fwd_argument_errors(L, kw, code):
    assert fwd(L, **kw) == code


def test_mod_argument_errors(L):
    m = L.make_mods(window=0)
    assert fwd(L, mods=m) == 1
    m = L.make_mods(causal=True)
    m.flags |= 1 << 7
    assert fwd(L, mods=m) == 1
    m = L.make_mods(softcap=-1.0)
    assert fwd(L, mods=m) == 1
    m = L.Mods()
    m.flags = L.MOD_DOC
    assert fwd(L, mods=m) == 1  # document mask without ids
    # window/doc masks need the block-map workspace
    m = L.make_mods(causal=True, window=64)
    assert fwd(L, mods=m) == 3
    need = L.attn_workspace_size(L.OP_FWD, 1, 2, 2, 128, 128, m)
    assert fwd(L, mods=m, ws=A + 16, nws=need) == 3  # misaligned workspace


def test_other_entry_points_validate(L):
    so = L.lib()
    # backward: null dq
    assert so.attn_bwd(A, A, A, A, A, A, None, A, A, 1, 2, 2, 64, 128, 0.1, None, A, 1 << 20, None) == 1
    # backward: workspace too small
    assert so.attn_bwd(A, A, A, A, A, A, A, A, A, 1, 2, 2, 64, 128, 0.1, None, A, 16, None) == 3
    # FP8 needs d = 128
    assert so.attn_fwd_fp8(A, A, A, A, A, A, 1, 2, 2, 64, 64, 0.1, None, None, 0, None) == 2
    assert so.attn_hadamard_quant_fp8(A, A, A, A, A, A, A, None, 1, 2, 2, 64, 64, A, 4096, None) == 2
    assert so.attn_hadamard_quant_fp8(A, A, A, A, A, A, None, None, 1, 2, 2, 64, 128, A, 4096, None) == 1
    # signs are read in 16-byte words
    assert so.attn_hadamard_quant_fp8(A, A, A, A, A, A, A, A + 8, 1, 2, 2, 64, 128, A, 1 << 20, None) == 2
    assert so.attn_block_map(None, 1, 100, None, None) == 1


def test_workspace_sizes(L):
    ws = L.attn_workspace_size
    assert ws(L.OP_FWD, 1, 2, 2, 1000, 128, L.make_mods(causal=True)) == 0
    m = L.make_mods(causal=True, window=64)
    # block map (B*nT*nT bytes) + per-Q-tile and per-KV-tile ranges (2 x B*nT int2), each 256-aligned
    assert ws(L.OP_FWD, 4, 16, 16, 4096, 128, m) == 4 * 32 * 32 + 2 * 1024
    # one {LSE, D} float pair per query row, rows padded to whole 128-row tiles ...
    assert ws(L.OP_BWD, 1, 64, 8, 8192, 128, None) == 64 * 8192 * 8
    assert ws(L.OP_BWD, 1, 64, 8, 8192, 128, L.make_mods(causal=True)) == 64 * 8192 * 8
    # ... and, for the one-kernel backward (causal with window / document parts,
    # d = 128), a dQ quantum per padded query row, the K/V bounds (8 bytes per
    # KV head, 256-aligned), the work-item counter (256 bytes) and the int32 dQ
    # accumulator, after the mods region
    mw = L.make_mods(causal=True, window=1024)
    mods_region = 64 * 64 + 2 * 512  # block map, tile ranges (1 x 64 int2 each, 256-aligned)
    fused = 64 * 8192 * 4 + 256 + 256 + 64 * 8192 * 128 * 4
    assert ws(L.OP_BWD, 1, 64, 8, 8192, 128, mw) == 64 * 8192 * 8 + mods_region + fused
    # d = 64 runs the two-kernel backward: no extra workspace
    assert ws(L.OP_BWD, 2, 2, 2, 1000, 64, m) == 2 * 2 * 1024 * 8 + 256 + 2 * 256
    assert ws(L.OP_QUANT_FP8, 2, 16, 16, 16384, 128, None) == 512  # 96 fp32 amax words
    assert ws(L.OP_FWD, 1, 3, 2, 128, 128, None) == 0  # invalid shape -> 0


def test_fp8_backward_workspace_and_limits(L):
    ws = L.attn_workspace_size
    m = L.make_mods(causal=True, bwd_fp8=True)
    # row statistics, then e4m3 dO and V (d bytes per row), then the dO / V scales and the
    # quantisation's amax words (2 * B * Hkv 4-byte entries each, 256-aligned)
    assert ws(L.OP_BWD, 1, 64, 8, 8192, 128, m) == 64 * 8192 * 8 + 64 * 8192 * 128 + 8 * 8192 * 128 + 2 * 256
    so = L.lib()
    rejected = [L.make_mods(causal=True, window=64, bwd_fp8=True), L.make_mods(softcap=30.0, bwd_fp8=True),
                L.make_mods(alibi=True, bwd_fp8=True)]
    for mm in rejected:  # ATTN_ERR_UNSUPPORTED before any other check of the workspace
        assert so.attn_bwd(A, A, A, A, A, A, A, A, A, 1, 2, 2, 256, 128, 0.1, ctypes.byref(mm), A, 16, None) == 2
    assert so.attn_bwd(A, A, A, A, A, A, A, A, A, 1, 2, 2, 256, 64, 0.1, ctypes.byref(m), A, 16, None) == 2


def test_status_strings(L):
    for c in range(8):
        assert L.status_string(c)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_valid_call_without_gpu_reports_cuda_error(L):
    assert fwd(L) == 4  # ATTN_ERR_CUDA: no silent CPU path


def test_varlen_entry_points_validate(L):
    so = L.lib()
    need = L.attn_workspace_size(L.OP_FWD_VARLEN, 1, 2, 2, 500, 128, None)
    # sequence ids (500 int32, rounded to 256 B) + the document mask's workspace
    assert need == 2048 + L.attn_workspace_size(L.OP_FWD, 1, 2, 2, 500, 128, L.make_mods(doc_ids=torch.zeros(1)))
    assert L.attn_workspace_size(L.OP_FWD_VARLEN, 2, 2, 2, 500, 128, None) == 0  # B must be 1
    assert L.attn_workspace_size(L.OP_BWD_VARLEN, 1, 2, 2, 500, 128, None) == \
        2048 + L.attn_workspace_size(L.OP_BWD, 1, 2, 2, 500, 128, L.make_mods(doc_ids=torch.zeros(1)))

    def fv(cu=A, n=3, mods=None, ws=A, nws=1 << 24, q=A):
        return so.attn_fwd_varlen(q, A, A, A, A, cu, n, 2, 2, 500, 128, 0.1,
                                  ctypes.byref(mods) if mods else None, ws, nws, None)
    assert fv(cu=None) == 1          # no sequence offsets
    assert fv(n=0) == 1              # no sequences
    assert fv(cu=A + 2) == 1         # misaligned offsets
    assert fv(q=None) == 1
    assert fv(mods=L.make_mods(doc_ids=torch.zeros(1))) == 1  # the sequences are the documents
    assert fv(ws=None, nws=0) == 3   # the workspace is always needed
    assert so.attn_bwd_varlen(A, A, A, A, A, A, A, A, None, A, 3, 2, 2, 500, 128, 0.1, None, A,
                              1 << 24, None) == 1  # null dv



def test_rope_prologue_validates(L):
    so = L.lib()
    for base in (0.0, 1.0, -5.0, float("nan"), float("inf")):
        assert so.attn_rope_hadamard_quant_fp8(A, A, A, A, A, A, A, None, 1, 2, 2, 64, 128, base, A, 4096,
                                               None) == 1
    assert so.attn_rope_hadamard_quant_fp8(A, A, A, A, A, A, A, None, 1, 2, 2, 64, 64, 1e4, A, 4096,
                                           None) == 2  # d must be 128


def test_paged_forward_validates(L):
    so = L.lib()

    def fp(table=A, nb=8, N=128, d=128, q=A):
        return so.attn_fwd_paged(q, A, A, table, nb, A, A, 1, 2, 2, N, d, 0.1, None, None, 0, None)
    assert fp(table=None) == 1
    assert fp(nb=0) == 1
    assert fp(q=None) == 1
    assert fp(N=120) == 2      # N must be a multiple of 16
    assert fp(d=96) == 2       # d = 64 or 128
    assert fp(d=64) in (4, 5)  # valid: stops at the device check (no GPU here)
    assert fp(table=A + 2) == 2


def test_decode_validates(L):
    so = L.lib()

    def dc(q=A, table=A, mb=8, sl=A, nb=8, lse=A, B=2, Hq=8, Hkv=2, T=1, d=128, scale=0.1, mods=None,
           ws=A, nws=1 << 30):
        return so.attn_decode_paged(q, A, A, table, mb, sl, nb, A, lse, B, Hq, Hkv, T, d, scale,
                                    ctypes.byref(mods) if mods else None, ws, nws, None)
    for kw in (dict(table=None), dict(sl=None), dict(lse=None), dict(q=None), dict(mb=0), dict(nb=0),
               dict(B=0), dict(Hq=0), dict(T=0), dict(scale=float("nan")), dict(scale=0.0)):
        assert dc(**kw) == 1, kw
    for kw in (dict(d=96), dict(Hq=3, Hkv=2), dict(Hq=129 * 2, Hkv=2), dict(Hq=32, Hkv=1, T=5),
               dict(sl=A + 2), dict(table=A + 2), dict(q=A + 8), dict(lse=A + 2)):
        assert dc(**kw) == 2, kw
    assert dc(mods=L.Mods(L.MOD_DOC, 0, 0.0, A, None)) == 2    # documents do not apply
    assert dc(mods=L.Mods(L.MOD_WINDOW, 0, 0.0, None, None)) == 1  # window must be >= 1
    assert dc(ws=None, nws=0) == 3
    assert dc(nws=1000) == 3
    assert dc() in (4, 5)  # valid: stops at the device check (no GPU here)


def test_decode_workspace_size(L):
    so = L.lib()

    def expect(B, Hq, Hkv, N):
        tiles = -(-N // 128)
        ct = min(max(1, -(-(B * Hkv * tiles) // 2432)), tiles)
        rows = B * Hq * (-(-tiles // ct))
        r256 = lambda x: -(-x // 256) * 256
        return r256(16 * B) + 256 + r256(rows * 512) + r256(rows * 4)
    for B, Hq, Hkv, N in ((32, 64, 8, 8192), (1, 8, 8, 16), (3, 12, 4, 4000), (128, 32, 8, 32768)):
        assert so.attn_workspace_size(6, B, Hq, Hkv, N, 128, None) == expect(B, Hq, Hkv, N)
    assert so.attn_workspace_size(6, 2, 8, 2, 100, 128, None) == 0     # N not a multiple of 16
    so.attn_decode_workspace_size.restype = ctypes.c_size_t
    for B, Hq, Hkv, T, mb, d in ((32, 64, 8, 1, 512, 128), (4, 32, 8, 4, 40, 128), (3, 8, 1, 16, 7, 64)):
        tiles = -(-16 * mb // 128)
        ct = min(max(1, -(-(B * Hkv * tiles) // 2432)), tiles)
        rows = B * Hq * T * (-(-tiles // ct))
        r256 = lambda x: -(-x // 256) * 256
        assert so.attn_decode_workspace_size(B, Hq, Hkv, T, mb, d, None) == \
            r256(16 * B) + 256 + r256(rows * 4 * d) + r256(rows * 4)
    assert so.attn_decode_workspace_size(2, 64, 1, 3, 8, 128, None) == 0  # 64 heads x 3 tokens > 128 rows
    assert so.attn_workspace_size(6, 2, 8, 2, 128, 96, None) == 0      # d = 64 or 128
    docm = L.Mods(L.MOD_DOC, 0, 0.0, A, None)
    assert so.attn_workspace_size(6, 2, 8, 2, 128, 128, ctypes.byref(docm)) == 0


def test_test_hooks_validate_and_reset(L):
    so = L.lib()
    assert so.attn_test_hooks(0, 4) == 1  # unknown stall bit
    assert so.attn_test_hooks(5_000_000, L.STALL_FWD | L.STALL_BWD) == 0
    assert so.attn_test_hooks(0, 0) == 0  # defaults back
