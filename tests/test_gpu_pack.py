"""GPU quantize/pack and dequantize against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import kvq_synth as synth
from tests.kvq_testlib import make_problem, written_pages

pytestmark = pytest.mark.gpu


def _w(bits, kcw, vcw, B=3, Hkv=2):
    return synth.shrink(synth.WORKLOADS["tiny"], batch=B, num_kv_heads=Hkv, num_q_heads=4 * Hkv, bits=bits,
                        k_scheme=kcw, v_scheme=vcw)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kcw,vcw", [(0, 0), (1, 1), (1, 0), (0, 1)])
@pytest.mark.parametrize("paged", [False, True])
def test_pack_bitexact(bits, kcw, vcw, paged):
    from tests.kvq_testlib import run_gpu
    pb = make_problem(_w(bits, kcw, vcw), seed=11 + bits, lens=[300, 129, 1], paged=paged)
    res = run_gpu(pb)
    assert res["status"] == 0
    pages = written_pages(pb)
    for which, key in ((0, "k"), (1, "v")):
        codes, scale, zero = (t.cpu() for t in res[f"{key}_cache"])
        assert np.array_equal(codes.numpy()[pages], pb.ref[f"{key}_codes"][pages]), which
        assert np.array_equal(scale.view(torch.int16).numpy()[pages],
                              pb.ref[f"{key}_scale"].view(np.int16)[pages]), which
        assert np.array_equal(zero.view(torch.int16).numpy()[pages],
                              pb.ref[f"{key}_zero"].view(np.int16)[pages]), which


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("scheme", [0, 1])
def test_dequant_bitexact(bits, scheme):
    import bit_quantized_kv_decode_gb300 as kvq
    pb = make_problem(_w(bits, scheme, scheme), seed=5, lens=[300, 129, 1], paged=True)
    dev = torch.device("cuda")
    desc = kvq.cache_desc(bits, scheme, scheme, 2, pb.num_pages)
    lens = pb.lens.to(dev)
    pt = pb.page_table.to(dev)
    for which, key in ((0, "k"), (1, "v")):
        cache = (torch.tensor(pb.ref[f"{key}_codes"]).to(dev), torch.tensor(pb.ref[f"{key}_scale"]).to(dev),
                 torch.tensor(pb.ref[f"{key}_zero"]).to(dev))
        xh = kvq.dequant(desc, which, cache, 3, 300, lens, pt).cpu().numpy()
        ref = pb.ref["khat" if which == 0 else "vhat"].astype(np.float32)
        assert np.array_equal(xh, ref)


def test_pack_nonfinite_and_bad_page_flags():
    import bit_quantized_kv_decode_gb300 as kvq
    dev = torch.device("cuda")
    desc = kvq.cache_desc(4, 0, 1, 1, 4)
    x = torch.randn(1, 1, 256, 128, device=dev)
    x[0, 0, 5, 7] = float("nan")
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kvq.pack(desc, 0, x, max_blocks=2, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.DEV_NONFINITE
    st.zero_()
    pt = torch.tensor([[0, 9]], dtype=torch.int32, device=dev)  # page 9 >= num_pages
    kvq.pack(desc, 1, torch.randn(1, 1, 256, 128, device=dev), page_table=pt, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.DEV_BAD_PAGE
    st.zero_()
    lens = torch.tensor([300], dtype=torch.int32, device=dev)  # > max_seq_len
    kvq.pack(desc, 1, torch.randn(1, 1, 256, 128, device=dev), lens, max_blocks=2, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.DEV_BAD_SEQ_LEN
