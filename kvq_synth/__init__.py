"""Seeded synthetic inputs for quantized-KV decode attention.

This module only draws random numbers; it holds none of the method's
arithmetic.  Both the CUDA library's tests/benchmark and the CPU oracle take
their inputs from here.

Value recipe (the same for every workload):
  * q ~ N(0, 1), stored as bf16 [B, Hq, D];
  * pre-quantization V ~ N(0, 1) fp32 [B, Hkv, L, D];
  * pre-quantization K ~ N(0, 1) fp32, with channel d of KV head h multiplied
    by c[h, d] = 1 + 4 |N(0, 1)| (outlier channels); one vector per KV head,
    shared across the batch;
  * sequence lengths: fixed, or log-uniform floor(exp(U(ln lo, ln hi)));
  * paged caches: a seeded random permutation of all pages forms the page
    table (128-token pages).

Everything is drawn with torch generators so the same code serves CPU and GPU
tensors; the CPU draw is the one the oracle tests use.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

BLOCK_TOKENS = 128
TOKENWISE = 0
CHANNELWISE = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    max_seq_len: int
    bits: int
    k_scheme: int
    v_scheme: int
    paged: bool = False
    ragged: Optional[tuple] = None  # (lo, hi) log-uniform lengths
    description: str = ""
    group: int = 128  # elements per quantization group (channels of a token, or tokens of a channel)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 4, 128, 256, 4, TOKENWISE, TOKENWISE,
                     description="B=1, Hkv=1, Hq=4, D=128, L=256; INT4 K/V token-wise"),
    "b8_l4k_int2": Workload("b8_l4k_int2", 8, 8, 32, 128, 4096, 2, CHANNELWISE, TOKENWISE,
                            description="B=8, Hkv=8, Hq=32, D=128, L=4096 contiguous; "
                                        "INT2 K channel-wise, V token-wise"),
    "b128_l32k_int4": Workload("b128_l32k_int4", 128, 8, 32, 128, 32768, 4, CHANNELWISE, TOKENWISE,
                               description="B=128, Hkv=8, Hq=32, D=128, L=32768; "
                                           "INT4 K channel-wise, V token-wise"),
    "b128_l32k_int2": Workload("b128_l32k_int2", 128, 8, 32, 128, 32768, 2, CHANNELWISE, TOKENWISE,
                               description="B=128, Hkv=8, Hq=32, D=128, L=32768; INT2 "
                                           "(all four K/V scheme pairs are swept)"),
    "paged_ragged_int2": Workload("paged_ragged_int2", 64, 8, 32, 128, 131072, 2, CHANNELWISE,
                                  TOKENWISE, paged=True, ragged=(1024, 131072),
                                  description="64 sequences, lengths log-uniform in [1K, 128K], "
                                              "128-token pages in a shuffled page table; INT2 "
                                              "K channel-wise, V token-wise"),
    # cache geometries beyond head dim 128 / groups of 128
    "b32_l32k_d256_g64_int4": Workload("b32_l32k_d256_g64_int4", 32, 8, 32, 256, 32768, 4, CHANNELWISE,
                                       TOKENWISE, group=64,
                                       description="B=32, Hkv=8, Hq=32, D=256, L=32768; INT4 K channel-wise, "
                                                   "V token-wise; groups of 64 (channels of a token, tokens of "
                                                   "a channel)"),
    "b32_l32k_d64_g32_int2": Workload("b32_l32k_d64_g32_int2", 32, 8, 32, 64, 32768, 2, CHANNELWISE,
                                      TOKENWISE, group=32,
                                      description="B=32, Hkv=8, Hq=32, D=64, L=32768; INT2 K channel-wise, "
                                                  "V token-wise; groups of 32"),
    "b32_l32k_d128_g32_int2": Workload("b32_l32k_d128_g32_int2", 32, 8, 32, 128, 32768, 2, CHANNELWISE,
                                       TOKENWISE, group=32,
                                       description="B=32, Hkv=8, Hq=32, D=128, L=32768; INT2 K channel-wise, "
                                                   "V token-wise; groups of 32"),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def seq_lens_for(w: Workload, seed: int) -> torch.Tensor:
    """int32 [B] sequence lengths (CPU)."""
    if w.ragged is None:
        return torch.full((w.batch,), w.max_seq_len, dtype=torch.int32)
    lo, hi = w.ragged
    g = _gen(seed * 7919 + 17, "cpu")
    u = torch.rand(w.batch, generator=g, dtype=torch.float64)
    lens = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    return lens.clamp(lo, hi).to(torch.int32)


def page_table_for(seq_lens: torch.Tensor, seed: int, max_blocks: Optional[int] = None):
    """Shuffled page table int32 [B, max_blocks] (CPU) and the page count.

    Pages are numbered 0..P-1 with P = total blocks over the batch; entries
    past a sequence's last block are -1."""
    nblk = [(int(n) + BLOCK_TOKENS - 1) // BLOCK_TOKENS for n in seq_lens.tolist()]
    if max_blocks is None:
        max_blocks = max(nblk) if nblk else 0
    total = sum(nblk)
    g = _gen(seed * 104729 + 3, "cpu")
    perm = torch.randperm(total, generator=g).to(torch.int32)
    table = torch.full((len(nblk), max(max_blocks, 1)), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    return table, total


def query(w: Workload, seed: int, device="cpu") -> torch.Tensor:
    """q ~ N(0,1) as bf16 [B, Hq, D]."""
    g = _gen(seed * 31 + 1, device)
    return torch.randn(w.batch, w.num_q_heads, w.head_dim, generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def outlier_channels(w: Workload, seed: int, device="cpu") -> torch.Tensor:
    """c[h, d] = 1 + 4 |N(0,1)|, fp32 [Hkv, D]."""
    g = _gen(seed * 131 + 5, device)
    return 1.0 + 4.0 * torch.randn(w.num_kv_heads, w.head_dim, generator=g, device=device,
                                   dtype=torch.float32).abs()


def kv_unit(w: Workload, seed: int, which: int, b: int, h: int, n_tokens: int,
            device="cpu", channel_scale: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Pre-quantization K (which=0) or V (which=1) for one (sequence, KV head):
    fp32 [n_tokens, D].  Each unit has its own generator, so any unit can be
    drawn alone."""
    g = _gen(((seed * 1000003 + which) * 65537 + b) * 257 + h, device)
    x = torch.randn(n_tokens, w.head_dim, generator=g, device=device, dtype=torch.float32)
    if which == 0:
        if channel_scale is None:
            channel_scale = outlier_channels(w, seed, device)[h]
        x = x * channel_scale.to(device)[None, :]
    return x


def kv_full(w: Workload, seed: int, which: int, seq_lens: torch.Tensor, device="cpu",
            batch_range=None) -> torch.Tensor:
    """Pre-quantization K or V, fp32 [B', Hkv, Lcap, D] with Lcap = the longest
    sequence; positions past a sequence's length are 0."""
    b0, b1 = batch_range if batch_range is not None else (0, w.batch)
    lens = seq_lens.tolist()
    lcap = max(lens[b0:b1]) if b1 > b0 else 0
    out = torch.zeros(b1 - b0, w.num_kv_heads, lcap, w.head_dim, device=device)
    cs = outlier_channels(w, seed, device) if which == 0 else None
    for b in range(b0, b1):
        for h in range(w.num_kv_heads):
            n = lens[b]
            out[b - b0, h, :n] = kv_unit(w, seed, which, b, h, n, device,
                                         None if cs is None else cs[h])
    return out


def shrink(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (for scaled-down tests)."""
    return dataclasses.replace(w, **kw)
