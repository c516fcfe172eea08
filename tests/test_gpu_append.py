"""kvq_append: growing a packed cache token by token gives the same bytes as
packing the whole sequence at once (the oracle's pack), for every bit width,
scheme pair and cache layout."""
import numpy as np
import pytest
import torch

import kvq_synth as synth
from oracle import kvq_oracle as orc

pytestmark = pytest.mark.gpu

L0 = [170, 0, 127]   # prefix lengths packed with kvq_pack (mid-block, empty, one short of a block)
STEPS = 140          # appended tokens per sequence (each crosses a block boundary)


def _written_pages(lens, pt, max_blocks):
    pages = []
    for b, n in enumerate(lens):
        for j in range((n + 127) // 128):
            pages.append(int(pt[b, j]) if pt is not None else b * max_blocks + j)
    return np.array(sorted(pages), dtype=np.int64)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kcw,vcw", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("paged", [False, True])
def test_append_equals_pack_of_whole_sequence(bits, kcw, vcw, paged):
    import bit_quantized_kv_decode_gb300 as kvq
    dev = torch.device("cuda")
    B, Hkv = len(L0), 2
    w = synth.shrink(synth.WORKLOADS["tiny"], batch=B, num_kv_heads=Hkv, num_q_heads=4 * Hkv, bits=bits,
                     k_scheme=kcw, v_scheme=vcw)
    seed = 31 + bits + 2 * kcw + vcw
    final = [n + STEPS for n in L0]
    lens_final = torch.tensor(final, dtype=torch.int32)
    max_blocks = (max(final) + 127) // 128
    if paged:
        pt, num_pages = synth.page_table_for(lens_final, seed, max_blocks)
        pt_dev = pt.to(dev)
    else:
        pt, num_pages, pt_dev = None, B * max_blocks, None
    desc = kvq.cache_desc(bits, kcw, vcw, Hkv, num_pages)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for which in (0, 1):
        x = synth.kv_full(w, seed, which, lens_final)  # fp32 [B, Hkv, Lmax, 128] (CPU)
        cache = kvq.alloc_cache(desc, dev)
        # prefix, packed whole
        lmax0 = max(max(L0), 1)
        kvq.pack(desc, which, x[:, :, :lmax0].contiguous().to(dev), torch.tensor(L0, dtype=torch.int32, device=dev),
                 pt_dev, max_blocks, cache=cache, dev_status=status)
        # the caller's window holds the raw rows of each prefix's partial last block
        window = torch.zeros(B, Hkv, 128, 128, dtype=torch.float32, device=dev)
        for b, n in enumerate(L0):
            r, j = n % 128, n // 128
            if r:
                window[b, :, :r] = x[b, :, j * 128:j * 128 + r].to(dev)
        cur = torch.tensor(L0, dtype=torch.int32, device=dev)
        for _ in range(STEPS):
            idx = cur.long().cpu()
            x_new = torch.stack([x[b, :, int(idx[b])] for b in range(B)]).contiguous().to(dev)
            kvq.append(desc, which, x_new, cur, cache, window, page_table=pt_dev, max_blocks=max_blocks,
                       dev_status=status)
            cur += 1
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref = orc.pack_cache(x.numpy(), final, bits, kcw if which == 0 else vcw, which,
                             None if pt is None else pt.numpy(), num_pages)
        pages = _written_pages(final, None if pt is None else pt.numpy(), max_blocks)
        codes, scale, zero = (t.cpu() for t in cache)
        assert np.array_equal(codes.numpy()[pages], ref[0][pages]), ("codes", which)
        assert np.array_equal(scale.view(torch.int16).numpy()[pages], ref[1].view(np.int16)[pages]), ("scale", which)
        assert np.array_equal(zero.view(torch.int16).numpy()[pages], ref[2].view(np.int16)[pages]), ("zero", which)


def test_append_bad_length_flagged():
    import bit_quantized_kv_decode_gb300 as kvq
    dev = torch.device("cuda")
    desc = kvq.cache_desc(4, 0, 0, 1, 2)
    cache = kvq.alloc_cache(desc, dev)
    window = torch.zeros(1, 1, 128, 128, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    full = torch.tensor([256], dtype=torch.int32, device=dev)  # no room left in 2 blocks
    kvq.append(desc, 0, torch.randn(1, 1, 128, device=dev), full, cache, window, max_blocks=2, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.DEV_BAD_SEQ_LEN
