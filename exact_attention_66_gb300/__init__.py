"""Exact tiled attention for GB300 (sm_103a): Python front end.

The compute lives in ``libattn.so`` (hand-written CUDA kernels behind the C
ABI of ``include/attn.h``).  This package only marshals arguments: the
same-name functions of ``_lib`` take torch tensors in place of pointers, and
the helpers below allocate outputs and workspaces with torch (device memory
and streams are the only things PyTorch provides here).  Importing the
package fails if the library has not been built; there is no other path.
"""
from __future__ import annotations

import math

from ._lib import (  # noqa: F401
    AttnError, Mods, EXPORTS, MOD_ALIBI, MOD_BWD_FP8, MOD_CAUSAL, MOD_DOC, MOD_SOFTCAP, MOD_WINDOW, OP_BWD,
    OP_BWD_VARLEN, OP_DECODE_PAGED, OP_FWD, OP_FWD_FP8, OP_FWD_VARLEN, OP_QUANT_FP8, TILE_FULL, TILE_PARTIAL,
    TILE_SKIP, attn_block_map, attn_bwd, attn_bwd_profiled, attn_bwd_noalloc, attn_bwd_varlen,
    NOALLOC_SCRATCH_BYTES, attn_fwd, attn_fwd_fp8, attn_fwd_varlen, attn_hadamard_quant_fp8,
    attn_rope_hadamard_quant_fp8, attn_fwd_paged, attn_decode_paged, attn_decode_workspace_size,
    attn_status, attn_test_hooks, attn_workspace_size, lib, STALL_BWD, STALL_FWD,
    make_mods, status_string,
)

__all__ = [
    "forward", "backward", "forward_paged", "decode_paged", "forward_varlen", "backward_varlen", "hadamard_quant_fp8",
    "forward_fp8", "attn_fwd_paged", "attn_decode_paged", "attn_decode_workspace_size",
    "block_map", "make_mods", "attn_fwd", "attn_bwd", "attn_bwd_profiled", "attn_bwd_noalloc",
    "attn_fwd_varlen", "attn_bwd_varlen", "attn_hadamard_quant_fp8", "attn_rope_hadamard_quant_fp8",
    "attn_fwd_fp8", "attn_block_map",
    "attn_status", "attn_workspace_size", "AttnError",
]


def _torch():
    import torch
    return torch


def _shape(q, k):
    B, Hq, N, d = q.shape
    return B, Hq, k.shape[1], N, d


def _workspace(op, B, Hq, Hkv, N, d, mods, device):
    torch = _torch()
    n = attn_workspace_size(op, B, Hq, Hkv, N, d, mods)
    if n == 0:
        return None, 0
    return torch.empty(n, dtype=torch.uint8, device=device), n


def forward(q, k, v, scale=None, mods=None, out=None, lse=None, stream=None):
    """(O, LSE) of attention over bf16 [B, H, N, d] device tensors."""
    torch = _torch()
    B, Hq, Hkv, N, d = _shape(q, k)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if lse is None else lse
    ws, nws = _workspace(OP_FWD, B, Hq, Hkv, N, d, mods, q.device)
    attn_fwd(q, k, v, o, l, B, Hq, Hkv, N, d, scale, mods, ws, nws, stream)
    return o, l


def backward(q, k, v, o, lse, do, scale=None, mods=None, stream=None):
    """(dQ, dK, dV) for the forward that produced (o, lse)."""
    torch = _torch()
    B, Hq, Hkv, N, d = _shape(q, k)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws, nws = _workspace(OP_BWD, B, Hq, Hkv, N, d, mods, q.device)
    attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, mods, ws, nws, stream)
    return dq, dk, dv


def forward_paged(q, k_cache, v_cache, block_table, scale=None, mods=None, stream=None):
    """(O, LSE) with K/V read from a paged cache: q [B, Hq, N, d], caches
    [num_blocks, Hkv, 16, d], block_table a device int32 [B, N / 16]."""
    torch = _torch()
    B, Hq, N, d = q.shape
    num_blocks, Hkv = k_cache.shape[0], k_cache.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    l = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    ws, nws = _workspace(OP_FWD, B, Hq, Hkv, N, d, mods, q.device)
    attn_fwd_paged(q, k_cache, v_cache, block_table, num_blocks, o, l, B, Hq, Hkv, N, d, scale, mods, ws,
                   nws, stream)
    return o, l


def decode_paged(q, k_cache, v_cache, block_table, seqlens, scale=None, mods=None, stream=None):
    """(O, LSE) of one decode step: q [B, Hq, d] (the newest token of each
    sequence) or [B, Hq, T, d] (its T newest tokens), caches
    [num_blocks, Hkv, 16, d], block_table a device int32 [B, max_blocks],
    seqlens a device int32 [B] of cached tokens per sequence (the new ones
    included).  O has q's shape; LSE is [B, Hq] or [B, Hq, T]."""
    torch = _torch()
    one = q.dim() == 3
    q4 = q.unsqueeze(2) if one else q
    B, Hq, T, d = q4.shape
    num_blocks, Hkv = k_cache.shape[0], k_cache.shape[1]
    max_blocks = block_table.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q4)
    l = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    nws = attn_decode_workspace_size(B, Hq, Hkv, T, max_blocks, d, mods)
    ws = torch.empty(nws, dtype=torch.uint8, device=q.device) if nws else None
    attn_decode_paged(q4, k_cache, v_cache, block_table, max_blocks, seqlens, num_blocks, o, l, B, Hq, Hkv, T, d,
                      scale, mods, ws, nws, stream)
    return (o.squeeze(2), l.squeeze(2)) if one else (o, l)


def forward_varlen(q, k, v, cu_seqlens, scale=None, mods=None, stream=None):
    """(O, LSE) over packed sequences: q [1, Hq, total, d], k/v [1, Hkv, total, d],
    cu_seqlens a device int32 tensor of the n_seqs + 1 sequence offsets."""
    torch = _torch()
    B, Hq, Hkv, total, d = _shape(q, k)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    n_seqs = cu_seqlens.numel() - 1
    o = torch.empty_like(q)
    l = torch.empty((1, Hq, total), dtype=torch.float32, device=q.device)
    ws, nws = _workspace(OP_FWD_VARLEN, 1, Hq, Hkv, total, d, mods, q.device)
    attn_fwd_varlen(q, k, v, o, l, cu_seqlens, n_seqs, Hq, Hkv, total, d, scale, mods, ws, nws, stream)
    return o, l


def backward_varlen(q, k, v, o, lse, do, cu_seqlens, scale=None, mods=None, stream=None):
    """(dQ, dK, dV) for the forward_varlen that produced (o, lse)."""
    torch = _torch()
    B, Hq, Hkv, total, d = _shape(q, k)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    n_seqs = cu_seqlens.numel() - 1
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws, nws = _workspace(OP_BWD_VARLEN, 1, Hq, Hkv, total, d, mods, q.device)
    attn_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, cu_seqlens, n_seqs, Hq, Hkv, total, d, scale, mods,
                    ws, nws, stream)
    return dq, dk, dv


def hadamard_quant_fp8(q, k, v, signs=None, stream=None, rope_base=None):
    """(q8, k8, v8, scales): e4m3 tensors (as uint8) and fp32 dequantisation scales
    (with rope_base, RoPE is applied to Q and K first, in the same pass)."""
    torch = _torch()
    B, Hq, Hkv, N, d = _shape(q, k)
    q8 = torch.empty(q.shape, dtype=torch.uint8, device=q.device)
    k8 = torch.empty(k.shape, dtype=torch.uint8, device=q.device)
    v8 = torch.empty(v.shape, dtype=torch.uint8, device=q.device)
    scales = torch.empty(B * Hq + 2 * B * Hkv, dtype=torch.float32, device=q.device)
    ws, nws = _workspace(OP_QUANT_FP8, B, Hq, Hkv, N, d, None, q.device)
    if rope_base is None:
        attn_hadamard_quant_fp8(q, k, v, q8, k8, v8, scales, signs, B, Hq, Hkv, N, d, ws, nws, stream)
    else:
        attn_rope_hadamard_quant_fp8(q, k, v, q8, k8, v8, scales, signs, B, Hq, Hkv, N, d, rope_base,
                                     ws, nws, stream)
    return q8, k8, v8, scales


def forward_fp8(q8, k8, v8, scales, scale=None, mods=None, stream=None):
    """(O bf16, LSE fp32) from the e4m3 tensors of hadamard_quant_fp8."""
    torch = _torch()
    B, Hq, Hkv, N, d = _shape(q8, k8)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty(q8.shape, dtype=torch.bfloat16, device=q8.device)
    l = torch.empty((B, Hq, N), dtype=torch.float32, device=q8.device)
    ws, nws = _workspace(OP_FWD_FP8, B, Hq, Hkv, N, d, mods, q8.device)
    attn_fwd_fp8(q8, k8, v8, scales, o, l, B, Hq, Hkv, N, d, scale, mods, ws, nws, stream)
    return o, l


def block_map(B, N, mods, device="cuda", stream=None):
    """uint8 [B, nT, nT] tile classes (0 skip, 1 partial, 2 full)."""
    torch = _torch()
    nT = (N + 127) // 128
    out = torch.empty((B, nT, nT), dtype=torch.uint8, device=device)
    attn_block_map(mods, B, N, out, stream)
    return out
