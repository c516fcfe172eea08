"""Shared helpers for the GPU parity tests: seeded problems, oracle results and
the product path (GPU pack + decode through the C-ABI)."""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

import kvq_synth as synth
from oracle import kvq_oracle as orc

TOL = {0: 3e-2, 1: 2e-3}       # max|out - oracle| / rms(oracle): FP8 path, BF16 mode
LSE_TOL = {0: 1e-2, 1: 1e-3}   # max|lse - oracle| (natural log units) at the default scale 1/sqrt(D)


def lse_tolerance(pb, mode: int) -> float:
    """The lse tolerance for a problem: LSE_TOL at the default softmax scale;
    an explicit scale sm_scale multiplies every score, and so the scores'
    (and the lse's) rounding error, by sm_scale * sqrt(D)."""
    s = getattr(pb, "sm_scale", 0.0)
    return LSE_TOL[mode] * (max(1.0, s * pb.w.head_dim ** 0.5) if s > 0 else 1.0)


@dataclasses.dataclass
class Problem:
    w: synth.Workload
    seed: int
    lens: torch.Tensor                  # int32 [B] (CPU)
    q: torch.Tensor                     # bf16 [B, Hq, D] (CPU)
    k: torch.Tensor                     # fp32 [B, Hkv, L, D] (CPU)
    v: torch.Tensor
    page_table: Optional[torch.Tensor]  # int32 [B, max_blocks] (CPU) or None
    num_pages: int
    max_blocks: int
    ref: dict                           # oracle results


def make_problem(w: synth.Workload, seed: int, lens=None, paged: Optional[bool] = None, q=None, k=None, v=None,
                 sm_scale: Optional[float] = None) -> Problem:
    """A seeded problem of workload w and the oracle's results for it.  q, k
    and v replace the synthetic values when given (bf16 [B, Hq, D] and fp32
    [B, Hkv, L, D] CPU tensors); sm_scale=None is the default 1/sqrt(D)."""
    lens_t = torch.tensor(lens, dtype=torch.int32) if lens is not None else synth.seq_lens_for(w, seed)
    L = max(1, int(lens_t.max()))
    max_blocks = (L + 127) // 128
    paged = w.paged if paged is None else paged
    if paged:
        pt, num_pages = synth.page_table_for(lens_t, seed, max_blocks)
        num_pages = max(num_pages, 1)
    else:
        pt, num_pages = None, w.batch * max_blocks
    q = synth.query(w, seed) if q is None else q
    k = synth.kv_full(w, seed, 0, lens_t) if k is None else k
    v = synth.kv_full(w, seed, 1, lens_t) if v is None else v
    if k.shape[2] < L:  # all-empty batch
        k = torch.zeros(w.batch, w.num_kv_heads, L, w.head_dim)
        v = torch.zeros_like(k)
    qb = q.view(torch.int16).numpy().view(np.uint16)
    ref = orc.reference_decode(qb, k.numpy(), v.numpy(), lens_t.numpy(), w.bits, w.k_scheme, w.v_scheme,
                               None if pt is None else pt.numpy(), num_pages, sm_scale=sm_scale, group=w.group)
    pb = Problem(w, seed, lens_t, q, k, v, pt, num_pages, max_blocks, ref)
    pb.sm_scale = 0.0 if sm_scale is None else float(sm_scale)
    return pb


def run_gpu(pb: Problem, mode: int = 0, num_ctas: int = 0, flags: int = 0):
    import bit_quantized_kv_decode_gb300 as kvq
    dev = torch.device("cuda")
    w = pb.w
    desc = kvq.cache_desc(w.bits, w.k_scheme, w.v_scheme, w.num_kv_heads, pb.num_pages, head_dim=w.head_dim,
                          group=w.group)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lens = pb.lens.to(dev)
    pt = None if pb.page_table is None else pb.page_table.to(dev)
    kc = kvq.pack(desc, 0, pb.k.to(dev), lens, pt, pb.max_blocks, dev_status=status)
    vc = kvq.pack(desc, 1, pb.v.to(dev), lens, pt, pb.max_blocks, dev_status=status)
    out, lse = kvq.decode_attn(desc, pb.q.to(dev), kc, vc, lens, pt, pb.max_blocks, mode=mode,
                               sm_scale=getattr(pb, "sm_scale", 0.0), num_ctas=num_ctas, dev_status=status,
                               flags=flags)
    torch.cuda.synchronize()
    return dict(out=out.cpu().double().numpy(), lse=lse.cpu().double().numpy(), k_cache=kc, v_cache=vc,
                status=int(status.item()), desc=desc)


def attn_errors(pb: Problem, res: dict):
    ref_o, ref_l = pb.ref["out"], pb.ref["lse"]
    rms = float(np.sqrt((ref_o ** 2).mean())) or 1.0
    err = float(np.abs(res["out"] - ref_o).max()) / rms
    fin = np.isfinite(ref_l)
    assert np.array_equal(fin, np.isfinite(res["lse"])), "empty-sequence lse mismatch"
    lerr = float(np.abs(res["lse"][fin] - ref_l[fin]).max()) if fin.any() else 0.0
    return err, lerr


def assert_attention_close(pb: Problem, res: dict, mode: int):
    err, lerr = attn_errors(pb, res)
    print(f"[parity] {pb.w.name} B={pb.w.batch} bits={pb.w.bits} k={pb.w.k_scheme} v={pb.w.v_scheme} "
          f"mode={mode}: max|out-oracle|/rms={err:.3e} max|lse-oracle|={lerr:.3e}")
    assert err <= TOL[mode], f"max|out-oracle|/rms = {err:.3e} > {TOL[mode]}"
    ltol = lse_tolerance(pb, mode)
    assert lerr <= ltol, f"max|lse-oracle| = {lerr:.3e} > {ltol:.3e}"
    return err, lerr


def written_pages(pb: Problem):
    """Page ids the batch covers (only those are compared bit for bit)."""
    pages = []
    for b, n in enumerate(pb.lens.tolist()):
        for j in range((n + 127) // 128):
            pages.append(int(pb.page_table[b, j]) if pb.page_table is not None else b * pb.max_blocks + j)
    return np.array(sorted(pages), dtype=np.int64)
