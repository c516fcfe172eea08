"""Decode attention over an INT2/INT4 group-quantized KV cache on GB300.

Thin PyTorch-facing wrappers over the C-ABI of ``libkvq.so`` (include/kvq.h):
they check tensor dtypes, devices and shapes, pass raw device pointers and the
current CUDA stream, and raise on a non-OK status.  Every step of the
computation runs in the library's CUDA kernels; there is no other code path.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import (CHANNELWISE, DEV_BAD_PAGE, DEV_BAD_SEQ_LEN, DEV_NONFINITE, DEV_TIMEOUT, FLAG_E2M1_V, FLAG_TEST_STALL,
                   FLAG_TEST_STALL_MMA, OPERANDS_BF16, OPERANDS_FP8, TOKENWISE, AttnDesc, CacheDesc, KvqError)

BLOCK_TOKENS = 128
HEAD_DIM = 128
GROUP_Q = 4

__all__ = ["CacheDesc", "AttnDesc", "KvqError", "TOKENWISE", "CHANNELWISE", "OPERANDS_FP8", "OPERANDS_BF16",
           "DEV_BAD_SEQ_LEN", "DEV_BAD_PAGE", "DEV_NONFINITE", "DEV_TIMEOUT", "FLAG_TEST_STALL", "FLAG_TEST_STALL_MMA",
           "FLAG_E2M1_V", "cache_desc", "attn_desc", "cache_bytes", "block_bytes", "sz_per_block", "alloc_cache", "pack",
           "append", "dequant", "workspace_size", "decode_attn", "decode_attn_static", "merge", "library"]


def library() -> ctypes.CDLL:
    return _lib.load()


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, numel=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")


def cache_desc(bits: int, k_scheme: int, v_scheme: int, num_kv_heads: int, num_pages: int,
               head_dim: int = HEAD_DIM, group: int = 128) -> CacheDesc:
    return CacheDesc(bits, k_scheme, v_scheme, head_dim, num_kv_heads, num_pages, group)


def attn_desc(cache: CacheDesc, batch: int, max_blocks: int, mode: int = OPERANDS_FP8, sm_scale: float = 0.0,
              num_ctas: int = 0, flags: int = 0, num_q_heads: Optional[int] = None) -> AttnDesc:
    hq = GROUP_Q * cache.num_kv_heads if num_q_heads is None else num_q_heads
    return AttnDesc(cache, batch, hq, max_blocks, mode, sm_scale, num_ctas, flags)


def block_bytes(bits: int, head_dim: int = HEAD_DIM) -> int:
    return BLOCK_TOKENS * head_dim * bits // 8


def sz_per_block(desc: CacheDesc) -> int:
    """s (or z) values per page and KV head: 128 * head_dim / group."""
    return BLOCK_TOKENS * desc.head_dim // (desc.group_size or 128)


def cache_bytes(desc: CacheDesc) -> Tuple[int, int]:
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _lib.check(library().kvq_cache_bytes(ctypes.byref(desc), ctypes.byref(cb), ctypes.byref(sb)), "kvq_cache_bytes")
    return cb.value, sb.value


def alloc_cache(desc: CacheDesc, device="cuda"):
    """Zeroed (codes, scale, zero) arrays for one K or V cache."""
    P, H = desc.num_pages, desc.num_kv_heads
    codes = torch.zeros(P, H, block_bytes(desc.bits, desc.head_dim), dtype=torch.uint8, device=device)
    scale = torch.zeros(P, H, sz_per_block(desc), dtype=torch.float16, device=device)
    zero = torch.zeros(P, H, sz_per_block(desc), dtype=torch.float16, device=device)
    return codes, scale, zero


def _geometry(batch, max_seq_len, seq_lens, page_table, max_blocks):
    need = (max_seq_len + BLOCK_TOKENS - 1) // BLOCK_TOKENS
    if page_table is not None:
        _need(page_table, "page_table", torch.int32)
        if page_table.dim() != 2 or page_table.shape[0] != batch:
            raise ValueError("page_table must be int32 [batch, max_blocks]")
        mb = page_table.shape[1]
    else:
        mb = max_blocks if max_blocks is not None else need
    if seq_lens is not None:
        _need(seq_lens, "seq_lens", torch.int32, batch)
    return mb


def pack(desc: CacheDesc, which: int, x: torch.Tensor, seq_lens: Optional[torch.Tensor] = None,
         page_table: Optional[torch.Tensor] = None, max_blocks: Optional[int] = None, cache=None,
         dev_status: Optional[torch.Tensor] = None):
    """Quantize + pack fp32 x [B, Hkv, L, head_dim] into a K (which=0) or V
    (which=1) cache; returns (codes, scale, zero)."""
    _need(x, "x", torch.float32)
    if x.dim() != 4 or x.shape[1] != desc.num_kv_heads or x.shape[3] != desc.head_dim:
        raise ValueError("x must be fp32 [batch, num_kv_heads, max_seq_len, head_dim]")
    B, _, L, _ = x.shape
    mb = _geometry(B, L, seq_lens, page_table, max_blocks)
    codes, scale, zero = cache if cache is not None else alloc_cache(desc, x.device)
    _need(codes, "codes", torch.uint8)
    _need(scale, "scale", (torch.float16, torch.int16, torch.uint16))
    _need(zero, "zero", (torch.float16, torch.int16, torch.uint16))
    if dev_status is not None:
        _need(dev_status, "dev_status", (torch.int32, torch.uint32), 1)
    st = library().kvq_pack(ctypes.byref(desc), which, _p(x), B, L, _p(seq_lens), _p(page_table), mb, _p(codes),
                            _p(scale), _p(zero), _p(dev_status), _stream())
    _lib.check(st, "kvq_pack")
    return codes, scale, zero


def append(desc: CacheDesc, which: int, x_new: torch.Tensor, seq_lens: torch.Tensor, cache, window: torch.Tensor,
           page_table: Optional[torch.Tensor] = None, max_blocks: Optional[int] = None,
           dev_status: Optional[torch.Tensor] = None):
    """Append fp32 x_new [B, Hkv, 128] at positions seq_lens (tokens already
    cached) to a packed K (which=0) or V (which=1) cache, through the caller's
    fp32 window [B, Hkv, 128, 128] of each current block; returns the cache.
    The caller advances seq_lens afterwards."""
    _need(x_new, "x_new", torch.float32)
    _need(window, "window", torch.float32)
    _need(seq_lens, "seq_lens", torch.int32)
    if x_new.dim() != 3 or x_new.shape[1] != desc.num_kv_heads or x_new.shape[2] != desc.head_dim:
        raise ValueError("x_new must be fp32 [batch, num_kv_heads, head_dim]")
    B = x_new.shape[0]
    if tuple(window.shape) != (B, desc.num_kv_heads, BLOCK_TOKENS, desc.head_dim):
        raise ValueError("window must be fp32 [batch, num_kv_heads, 128, head_dim]")
    if seq_lens.numel() != B:
        raise ValueError("seq_lens must hold one int32 per sequence")
    if page_table is not None:
        _need(page_table, "page_table", torch.int32)
        mb = page_table.shape[1]
    elif max_blocks is not None:
        mb = int(max_blocks)
    else:
        raise ValueError("append needs page_table or max_blocks")
    codes, scale, zero = cache
    if dev_status is not None:
        _need(dev_status, "dev_status", (torch.int32, torch.uint32), 1)
    st = library().kvq_append(ctypes.byref(desc), which, _p(x_new), B, _p(seq_lens), _p(page_table), mb,
                              _p(window), _p(codes), _p(scale), _p(zero), _p(dev_status), _stream())
    _lib.check(st, "kvq_append")
    return cache


def dequant(desc: CacheDesc, which: int, cache, batch: int, max_seq_len: int,
            seq_lens: Optional[torch.Tensor] = None, page_table: Optional[torch.Tensor] = None,
            max_blocks: Optional[int] = None, dev_status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """x_hat fp32 [B, Hkv, L, 128] read back from a packed cache."""
    codes, scale, zero = cache
    mb = _geometry(batch, max_seq_len, seq_lens, page_table, max_blocks)
    out = torch.empty(batch, desc.num_kv_heads, max_seq_len, desc.head_dim, dtype=torch.float32, device=codes.device)
    st = library().kvq_dequant(ctypes.byref(desc), which, _p(codes), _p(scale), _p(zero), batch, max_seq_len,
                               _p(seq_lens), _p(page_table), mb, _p(out), _p(dev_status), _stream())
    _lib.check(st, "kvq_dequant")
    return out


def workspace_size(desc: AttnDesc) -> int:
    n = ctypes.c_size_t()
    _lib.check(library().kvq_decode_workspace_size(ctypes.byref(desc), ctypes.byref(n)), "kvq_decode_workspace_size")
    return n.value


def decode_path(desc: AttnDesc) -> int:
    """The decode kernel a call with this descriptor runs: _lib.PATH_SPECIALISED
    or _lib.PATH_GENERAL (kvq_decode_path)."""
    n = ctypes.c_int32()
    _lib.check(library().kvq_decode_path(ctypes.byref(desc), ctypes.byref(n)), "kvq_decode_path")
    return n.value


def decode_attn(desc: CacheDesc, q: torch.Tensor, k_cache, v_cache, seq_lens: torch.Tensor,
                page_table: Optional[torch.Tensor] = None, max_blocks: Optional[int] = None,
                mode: int = OPERANDS_FP8, sm_scale: float = 0.0, num_ctas: int = 0,
                out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
                flags: int = 0):
    """out fp32 [B, Hq, 128] and lse fp32 [B, Hq] for bf16 q [B, Hq, 128]."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3 or q.shape[2] != desc.head_dim:
        raise ValueError("q must be bf16 [batch, num_q_heads, head_dim]")
    B, Hq, _ = q.shape
    if page_table is not None:
        mb = _geometry(B, 1, seq_lens, page_table, None)
    else:
        if max_blocks is None:
            raise ValueError("max_blocks is required for a contiguous cache")
        mb = max_blocks
        _need(seq_lens, "seq_lens", torch.int32, B)
    ad = AttnDesc(desc, B, Hq, mb, mode, sm_scale, num_ctas, flags)
    if out is None:
        out = torch.empty(B, Hq, desc.head_dim, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, B * Hq * desc.head_dim)
    _need(lse, "lse", torch.float32, B * Hq)
    if workspace is None:
        workspace = torch.empty(workspace_size(ad), dtype=torch.uint8, device=q.device)
    kc, ks, kz = k_cache
    vc, vs, vz = v_cache
    st = library().kvq_decode_attn(ctypes.byref(ad), _p(q), _p(kc), _p(ks), _p(kz), _p(vc), _p(vs), _p(vz),
                                   _p(seq_lens), _p(page_table), _p(out), _p(lse), _p(workspace),
                                   workspace.numel(), _p(dev_status), _stream())
    _lib.check(st, "kvq_decode_attn")
    return out, lse


def decode_attn_static(desc: CacheDesc, q: torch.Tensor, k_cache, v_cache, seq_lens: torch.Tensor,
                       page_table: Optional[torch.Tensor] = None, max_blocks: Optional[int] = None,
                       mode: int = OPERANDS_FP8, sm_scale: float = 0.0, num_ctas: int = 0,
                       out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                       dev_status: Optional[torch.Tensor] = None):
    """decode_attn for callers that cannot allocate device memory: the C entry
    point keeps its scratch in a fixed device array owned by the library (see
    kvq_decode_attn_static in include/kvq.h).  `out` and `lse` are still
    caller buffers; pass them preallocated to avoid any allocation here."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3 or q.shape[2] != desc.head_dim:
        raise ValueError("q must be bf16 [batch, num_q_heads, head_dim]")
    B, Hq, _ = q.shape
    if page_table is not None:
        mb = _geometry(B, 1, seq_lens, page_table, None)
    else:
        if max_blocks is None:
            raise ValueError("max_blocks is required for a contiguous cache")
        mb = max_blocks
        _need(seq_lens, "seq_lens", torch.int32, B)
    ad = AttnDesc(desc, B, Hq, mb, mode, sm_scale, num_ctas, 0)
    if out is None:
        out = torch.empty(B, Hq, desc.head_dim, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, B * Hq * desc.head_dim)
    _need(lse, "lse", torch.float32, B * Hq)
    kc, ks, kz = k_cache
    vc, vs, vz = v_cache
    st = library().kvq_decode_attn_static(ctypes.byref(ad), _p(q), _p(kc), _p(ks), _p(kz), _p(vc), _p(vs), _p(vz),
                                          _p(seq_lens), _p(page_table), _p(out), _p(lse), _p(dev_status),
                                          _stream())
    _lib.check(st, "kvq_decode_attn_static")
    return out, lse


def merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, out: Optional[torch.Tensor] = None,
          lse: Optional[torch.Tensor] = None):
    """Log-sum-exp merge of fp32 o_parts [R, S, D] / lse_parts [R, S]."""
    _need(o_parts, "o_parts", torch.float32)
    _need(lse_parts, "lse_parts", torch.float32)
    R, S, D = o_parts.shape
    if out is None:
        out = torch.empty(R, D, dtype=torch.float32, device=o_parts.device)
    if lse is None:
        lse = torch.empty(R, dtype=torch.float32, device=o_parts.device)
    st = library().kvq_merge(_p(o_parts), _p(lse_parts), R, S, D, _p(out), _p(lse), _stream())
    _lib.check(st, "kvq_merge")
    return out, lse
