"""ctypes binding of ``libattn.so`` (declared in ``include/attn.h``).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  The functions below carry the C names and take
torch tensors (device memory, owned by the caller) in place of raw pointers.
There is no fallback: if the library is missing, importing this module
raises, and every non-OK status raises ``AttnError``.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn.so")

ATTN_OK = 0
STATUS_NAMES = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_WORKSPACE",
    4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_DEVICE", 6: "ATTN_ERR_TIMEOUT", 7: "ATTN_ERR_BOUNDS",
}

MOD_CAUSAL, MOD_WINDOW, MOD_DOC, MOD_SOFTCAP, MOD_ALIBI, MOD_BWD_FP8 = 1, 2, 4, 8, 16, 32
OP_FWD, OP_BWD, OP_FWD_FP8, OP_QUANT_FP8, OP_FWD_VARLEN, OP_BWD_VARLEN, OP_DECODE_PAGED = 0, 1, 2, 3, 4, 5, 6
TILE_SKIP, TILE_PARTIAL, TILE_FULL = 0, 1, 2

# Exported symbols, in the order include/attn.h declares them.
EXPORTS = ("attn_workspace_size", "attn_fwd", "attn_bwd", "attn_bwd_profiled", "attn_bwd_noalloc",
           "attn_fwd_paged", "attn_decode_paged", "attn_decode_workspace_size", "attn_fwd_varlen", "attn_bwd_varlen", "attn_hadamard_quant_fp8", "attn_rope_hadamard_quant_fp8",
           "attn_fwd_fp8", "attn_block_map", "attn_test_hooks", "attn_status", "attn_status_string")


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


class Mods(ctypes.Structure):
    """attn_mods_t: mod flags plus runtime scalars (pointers are device addresses)."""
    _fields_ = [("flags", ctypes.c_uint32), ("window", ctypes.c_int32), ("softcap", ctypes.c_float),
                ("doc_ids", ctypes.c_void_p), ("alibi_slopes", ctypes.c_void_p)]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first (python exact_attention_66_gb300/build.py)")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    mp = ctypes.POINTER(Mods)
    lib.attn_workspace_size.argtypes = [i, i, i, i, i, i, mp]
    lib.attn_workspace_size.restype = sz
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, mp, vp, sz, vp]
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, mp, vp, sz, vp]
    lib.attn_bwd_profiled.argtypes = lib.attn_bwd.argtypes + [ctypes.POINTER(ctypes.c_void_p)]
    lib.attn_bwd_noalloc.argtypes = lib.attn_bwd.argtypes[:16] + [vp]  # no ws, ws_bytes
    lib.attn_fwd_paged.argtypes = [vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, f, mp, vp, sz, vp]
    lib.attn_decode_paged.argtypes = [vp, vp, vp, vp, i, vp, i, vp, vp, i, i, i, i, i, f, mp, vp, sz, vp]
    lib.attn_decode_workspace_size.argtypes = [i, i, i, i, i, i, mp]
    lib.attn_decode_workspace_size.restype = sz
    lib.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, mp, vp, sz, vp]
    lib.attn_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, mp, vp, sz, vp]
    lib.attn_hadamard_quant_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp, sz, vp]
    lib.attn_rope_hadamard_quant_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, mp, vp, sz, vp]
    lib.attn_block_map.argtypes = [mp, i, i, vp, vp]
    lib.attn_test_hooks.argtypes = [ctypes.c_ulonglong, i]
    lib.attn_status.argtypes = [vp]
    lib.attn_status_string.argtypes = [i]
    lib.attn_status_string.restype = ctypes.c_char_p
    for name in ("attn_fwd", "attn_bwd", "attn_bwd_profiled", "attn_bwd_noalloc", "attn_hadamard_quant_fp8", "attn_fwd_fp8",
                 "attn_block_map", "attn_test_hooks", "attn_status"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


_lib = load_library()


def lib() -> ctypes.CDLL:
    return _lib


def status_string(status: int) -> str:
    return _lib.attn_status_string(int(status)).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str) -> None:
    if st != ATTN_OK:
        raise AttnError(st, where)


def make_mods(causal=False, window=None, doc_ids=None, softcap=None, alibi=False,
              alibi_slopes=None, bwd_fp8=False) -> Mods:
    """attn_mods_t from Python values (doc_ids / alibi_slopes: device tensors;
    bwd_fp8: the mixed e4m3 backward)."""
    m = Mods()
    m.flags = ((MOD_CAUSAL if causal else 0) | (MOD_WINDOW if window is not None else 0)
               | (MOD_DOC if doc_ids is not None else 0) | (MOD_SOFTCAP if softcap is not None else 0)
               | (MOD_ALIBI if alibi else 0) | (MOD_BWD_FP8 if bwd_fp8 else 0))
    m.window = int(window) if window is not None else 0
    m.softcap = float(softcap) if softcap is not None else 0.0
    m.doc_ids = _ptr(doc_ids)
    m.alibi_slopes = _ptr(alibi_slopes)
    m._refs = (doc_ids, alibi_slopes)  # the struct holds raw pointers: keep the tensors alive
    return m


def _mods_ref(mods):
    return ctypes.byref(mods) if mods is not None else None


def attn_workspace_size(op, B, Hq, Hkv, N, d, mods=None) -> int:
    return int(_lib.attn_workspace_size(op, B, Hq, Hkv, N, d, _mods_ref(mods)))


def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, mods=None, ws=None, ws_bytes=0, stream=None):
    _check(_lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                         float(scale), _mods_ref(mods), _ptr(ws), int(ws_bytes), _stream(stream)),
           "attn_fwd")


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, mods=None, ws=None,
             ws_bytes=0, stream=None):
    _check(_lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                         _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, float(scale), _mods_ref(mods),
                         _ptr(ws), int(ws_bytes), _stream(stream)), "attn_bwd")


def attn_bwd_profiled(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, mods, ws,
                      ws_bytes, stream, events):
    """attn_bwd recording four torch.cuda.Event objects around its kernels (see attn.h)."""
    arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
    _check(_lib.attn_bwd_profiled(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                  _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, float(scale),
                                  _mods_ref(mods), _ptr(ws), int(ws_bytes), _stream(stream), arr),
           "attn_bwd_profiled")


NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024  # ATTN_NOALLOC_SCRATCH_BYTES


def attn_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, mods=None,
                     stream=None):
    """attn_bwd without a workspace, for callers that cannot allocate device
    memory (memory owned by a framework allocator or a fixed arena, or no
    cudaMalloc/cudaFree allowed because they synchronise the device).  The
    library's fixed scratch array stands in for the workspace: the work must
    fit in NOALLOC_SCRATCH_BYTES, and calls that overlap on the GPU race."""
    _check(_lib.attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, float(scale),
                                 _mods_ref(mods), _stream(stream)), "attn_bwd_noalloc")


def attn_fwd_paged(q, k_cache, v_cache, block_table, num_blocks, o, lse, B, Hq, Hkv, N, d, scale,
                   mods=None, ws=None, ws_bytes=0, stream=None):
    _check(_lib.attn_fwd_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), num_blocks,
                               _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, float(scale), _mods_ref(mods),
                               _ptr(ws), int(ws_bytes), _stream(stream)), "attn_fwd_paged")


def attn_decode_paged(q, k_cache, v_cache, block_table, max_blocks, seqlens, num_blocks, o, lse, B, Hq,
                      Hkv, q_len, d, scale, mods=None, ws=None, ws_bytes=0, stream=None):
    _check(_lib.attn_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), max_blocks,
                                  _ptr(seqlens), num_blocks, _ptr(o), _ptr(lse), B, Hq, Hkv, q_len, d,
                                  float(scale), _mods_ref(mods), _ptr(ws), int(ws_bytes), _stream(stream)),
           "attn_decode_paged")


def attn_decode_workspace_size(B, Hq, Hkv, q_len, max_blocks, d, mods=None) -> int:
    return int(_lib.attn_decode_workspace_size(B, Hq, Hkv, q_len, max_blocks, d, _mods_ref(mods)))


def attn_fwd_varlen(q, k, v, o, lse, cu_seqlens, n_seqs, Hq, Hkv, total, d, scale, mods=None,
                    ws=None, ws_bytes=0, stream=None):
    _check(_lib.attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens),
                                n_seqs, Hq, Hkv, total, d, float(scale), _mods_ref(mods), _ptr(ws),
                                int(ws_bytes), _stream(stream)), "attn_fwd_varlen")


def attn_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens, n_seqs, Hq, Hkv, total, d, scale,
                    mods=None, ws=None, ws_bytes=0, stream=None):
    _check(_lib.attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                                _ptr(dk), _ptr(dv), _ptr(cu_seqlens), n_seqs, Hq, Hkv, total, d,
                                float(scale), _mods_ref(mods), _ptr(ws), int(ws_bytes),
                                _stream(stream)), "attn_bwd_varlen")


def attn_hadamard_quant_fp8(q, k, v, q8, k8, v8, scales, signs, B, Hq, Hkv, N, d, ws=None,
                            ws_bytes=0, stream=None):
    _check(_lib.attn_hadamard_quant_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(q8), _ptr(k8), _ptr(v8),
                                        _ptr(scales), _ptr(signs), B, Hq, Hkv, N, d, _ptr(ws),
                                        int(ws_bytes), _stream(stream)), "attn_hadamard_quant_fp8")


def attn_rope_hadamard_quant_fp8(q, k, v, q8, k8, v8, scales, signs, B, Hq, Hkv, N, d, rope_base,
                                 ws=None, ws_bytes=0, stream=None):
    _check(_lib.attn_rope_hadamard_quant_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(q8), _ptr(k8), _ptr(v8),
                                             _ptr(scales), _ptr(signs), B, Hq, Hkv, N, d, float(rope_base),
                                             _ptr(ws), int(ws_bytes), _stream(stream)),
           "attn_rope_hadamard_quant_fp8")


def attn_fwd_fp8(q8, k8, v8, scales, o, lse, B, Hq, Hkv, N, d, scale, mods=None, ws=None,
                 ws_bytes=0, stream=None):
    _check(_lib.attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(scales), _ptr(o), _ptr(lse), B, Hq,
                             Hkv, N, d, float(scale), _mods_ref(mods), _ptr(ws), int(ws_bytes),
                             _stream(stream)), "attn_fwd_fp8")


def attn_block_map(mods, B, N, out, stream=None):
    _check(_lib.attn_block_map(_mods_ref(mods), B, N, _ptr(out), _stream(stream)), "attn_block_map")


STALL_FWD, STALL_BWD = 1, 2  # ATTN_STALL_FWD, ATTN_STALL_BWD


def attn_test_hooks(wait_limit_ns=0, stall=0):
    """Pipeline-wait limit (ns; 0 = the default 1 s) and stall bits for the
    kernels launched after this call (see include/attn.h)."""
    _check(_lib.attn_test_hooks(int(wait_limit_ns), int(stall)), "attn_test_hooks")


def attn_status(stream=None):
    _check(_lib.attn_status(_stream(stream)), "attn_status")
