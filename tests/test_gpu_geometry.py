"""Head dims 64 / 256 and groups of 32 / 64 elements on the GPU: quantize +
pack, dequantize and quantize-on-append bit-exact against the oracle, for
both bit widths and both group schemes (groups of G consecutive channels of
a token, or G consecutive tokens of a channel; rag-lover.com summary of arXiv
2611.09722, section "使える条件")."""
import numpy as np
import pytest
import torch

import kvq_synth as synth
from oracle import kvq_oracle as orc

pytestmark = pytest.mark.gpu

GEOMETRIES = [(64, 32), (64, 64), (128, 32), (128, 64), (256, 64), (256, 128)]


def _inputs(D, seed, B=3, Hkv=2, L=300):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, Hkv, L, D, generator=g) * (1 + 4 * torch.randn(D, generator=g).abs())
    lens = torch.tensor([300, 129, 1], dtype=torch.int32)
    for b in range(B):
        x[b, :, int(lens[b]):] = 0
    return x, lens


@pytest.mark.parametrize("D,G", GEOMETRIES)
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("scheme", [0, 1])
def test_pack_dequant_geometry_bitexact(D, G, bits, scheme):
    import bit_quantized_kv_decode_gb300 as kvq
    dev = torch.device("cuda")
    x, lens = _inputs(D, 100 + D + G + bits + scheme)
    B, Hkv, L, _ = x.shape
    max_blocks = 3
    pt, num_pages = synth.page_table_for(lens, 9, max_blocks)
    desc = kvq.cache_desc(bits, scheme, scheme, Hkv, num_pages, head_dim=D, group=G)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for which in (0, 1):
        cache = kvq.pack(desc, which, x.to(dev), lens.to(dev), pt.to(dev), dev_status=st)
        xh = kvq.dequant(desc, which, cache, B, L, lens.to(dev), pt.to(dev), dev_status=st).cpu().numpy()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        rc, rs, rz = orc.pack_cache(x.numpy(), lens.numpy(), bits, scheme, which, pt.numpy(), num_pages, group=G)
        codes, scale, zero = (t.cpu().numpy() for t in cache)
        pages = sorted({int(pt[b, j]) for b in range(B) for j in range((int(lens[b]) + 127) // 128)})
        assert np.array_equal(codes[pages], rc[pages])
        assert np.array_equal(scale.view(np.uint16)[pages], rs.view(np.uint16)[pages])
        assert np.array_equal(zero.view(np.uint16)[pages], rz.view(np.uint16)[pages])
        lc, ls, lz = orc.unpack_cache(rc, rs, rz, lens.numpy(), bits, which, L, pt.numpy())
        ref = orc.dequantize(lc, ls, lz, lens.numpy(), scheme).astype(np.float32)
        assert np.array_equal(xh, ref)


@pytest.mark.parametrize("D,G", [(64, 32), (256, 64)])
@pytest.mark.parametrize("scheme", [0, 1])
def test_append_geometry_bitexact(D, G, scheme):
    """Token by token across a block boundary: the cache equals the oracle's
    pack of the whole sequence."""
    import bit_quantized_kv_decode_gb300 as kvq
    dev = torch.device("cuda")
    B, Hkv, L = 2, 1, 140
    x, _ = _inputs(D, 7 + D + scheme, B=B, Hkv=Hkv, L=L)
    lens0 = torch.zeros(B, dtype=torch.int32, device=dev)
    max_blocks = 2
    desc = kvq.cache_desc(4, scheme, scheme, Hkv, B * max_blocks, head_dim=D, group=G)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cache = kvq.alloc_cache(desc, dev)
    window = torch.zeros(B, Hkv, 128, D, device=dev)
    xd = x.to(dev)
    for t in range(L):
        kvq.append(desc, 1, xd[:, :, t].contiguous(), lens0, cache, window, max_blocks=max_blocks, dev_status=st)
        lens0 += 1
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    final = np.full(B, L)
    rc, rs, rz = orc.pack_cache(x.numpy(), final, 4, scheme, 1, None, B * max_blocks, group=G)
    codes, scale, zero = (t.cpu().numpy() for t in cache)
    assert np.array_equal(codes, rc)
    assert np.array_equal(scale.view(np.uint16), rs.view(np.uint16))
    assert np.array_equal(zero.view(np.uint16), rz.view(np.uint16))
