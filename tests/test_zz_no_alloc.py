"""The allocation-free decode entry point (kvq_decode_attn_static).

It serves callers that cannot allocate device memory -- a runtime whose
memory plan is frozen, a plugin interface that passes only input and output
buffers -- by keeping the decode's split-merge scratch in a fixed device array
owned by the library.  This file is collected last on purpose, and it passes
both on its own in a fresh process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import kvq_synth as synth
from tests.kvq_testlib import LSE_TOL, TOL, assert_attention_close, make_problem, run_gpu

pytestmark = pytest.mark.gpu


def _problem():
    w = synth.shrink(synth.WORKLOADS["tiny"], batch=3, num_kv_heads=2, num_q_heads=8, bits=4,
                     k_scheme=1, v_scheme=0, max_seq_len=1500)
    return make_problem(w, seed=77, lens=[1500, 700, 129])


def test_static_scratch_matches_workspace_entry_point_twice():
    import bit_quantized_kv_decode_gb300 as kvq
    pb = _problem()
    dev = torch.device("cuda")
    res = run_gpu(pb, num_ctas=7)  # existing entry point, caller workspace; splits units across CTAs
    assert res["status"] == 0
    q = pb.q.to(dev)
    lens = pb.lens.to(dev)
    ref_o = torch.tensor(res["out"])
    ref_l = torch.tensor(res["lse"])
    rms = float(ref_o.pow(2).mean().sqrt())
    out = torch.empty(3, 8, 128, dtype=torch.float32, device=dev)
    lse = torch.empty(3, 8, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(2):  # the second call finds the first call's scratch contents
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        kvq.decode_attn_static(res["desc"], q, res["k_cache"], res["v_cache"], lens, max_blocks=pb.max_blocks,
                               num_ctas=7, out=out, lse=lse, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        o = out.cpu().double()
        l_ = lse.cpu().double()
        # against the workspace entry point ...
        assert float((o - ref_o).abs().max()) <= TOL[0] * rms
        assert float((l_ - ref_l).abs().max()) <= LSE_TOL[0]
        # ... and against the oracle, element by element
        assert_attention_close(pb, {"out": o.numpy(), "lse": l_.numpy()}, 0)


def test_static_scratch_general_geometry_twice():
    """Head dim 256 with groups of 32 (the block-range kernel, whose scratch
    holds per-range partial results): two calls in a row match the
    workspace entry point and the oracle."""
    import bit_quantized_kv_decode_gb300 as kvq
    w = synth.Workload("geom_d256_g32", 2, 2, 8, 256, 300, 4, 1, 1, group=32)
    pb = make_problem(w, seed=8, lens=[300, 77])
    dev = torch.device("cuda")
    res = run_gpu(pb)
    assert res["status"] == 0
    ref_o = torch.tensor(res["out"])
    rms = float(ref_o.pow(2).mean().sqrt())
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(2):
        out, lse = kvq.decode_attn_static(res["desc"], pb.q.to(dev), res["k_cache"], res["v_cache"],
                                          pb.lens.to(dev), None, pb.max_blocks, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        o = out.cpu().double()
        assert float((o - ref_o).abs().max()) <= 1e-5 * rms
        assert_attention_close(pb, {"out": o.numpy(), "lse": lse.cpu().double().numpy()}, 0)


def test_static_scratch_rejects_oversized_calls():
    import bit_quantized_kv_decode_gb300 as kvq
    from bit_quantized_kv_decode_gb300 import _lib
    lib = kvq.library()
    desc = kvq.cache_desc(4, 1, 0, 8, 1024 * 8)
    # 2000 CTAs need 2000 * 4 KiB of partial results: more than the fixed 4 MiB
    ad = _lib.AttnDesc(desc, 1024, 32, 8, 0, 0.0, 2000, 0)
    fake = ctypes.c_void_p(0x10000)
    st = lib.kvq_decode_attn_static(ctypes.byref(ad), *([fake] * 7), fake, None, fake, fake, None, None)
    assert st == 3  # KVQ_ERR_WORKSPACE, before any launch


def test_static_scratch_falls_back_to_specialised_kernel():
    """A call kvq_decode_attn runs in the general kernel (2-bit codes, K and V
    token-wise, B=64, L=16K: 65,536 (sequence, kv head, block) triples) whose
    general-kernel scratch exceeds the fixed array runs in the specialised
    kernel instead: the static output matches the workspace entry point's
    (general kernel) within the two kernels' tolerances, and the oracle on
    sampled units."""
    import bench
    import bit_quantized_kv_decode_gb300 as kvq
    from bit_quantized_kv_decode_gb300 import _lib
    from tests.test_gpu_fullsize import SEED, _oracle_unit, _sample_units
    dev = torch.device("cuda")
    w = synth.shrink(synth.WORKLOADS["b128_l32k_int2"], batch=64, max_seq_len=16384, k_scheme=0, v_scheme=0,
                     name="b64_l16k_int2_tt")
    c = bench.build_cache(w, SEED, dev, 0, 0)
    ad = kvq.attn_desc(c["desc"], w.batch, c["max_blocks"], num_q_heads=w.num_q_heads)
    assert kvq.decode_path(ad) == _lib.PATH_GENERAL
    assert kvq.workspace_size(ad) > 4 << 20
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out_g, lse_g = kvq.decode_attn(c["desc"], c["q"], c["k"], c["v"], c["lens"], c["pt"], c["max_blocks"],
                                   dev_status=st)
    out = torch.empty_like(out_g)
    lse = torch.empty_like(lse_g)
    for _ in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        kvq.decode_attn_static(c["desc"], c["q"], c["k"], c["v"], c["lens"], max_blocks=c["max_blocks"], out=out,
                               lse=lse, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        rms = float(out_g.double().pow(2).mean().sqrt())
        assert float((out.double() - out_g.double()).abs().max()) <= 2 * TOL[0] * rms
        assert float((lse.double() - lse_g.double()).abs().max()) <= 2 * LSE_TOL[0]
    got_o, ref_o, got_l, ref_l = [], [], [], []
    for b, h in _sample_units(w, c["lens_cpu"], SEED + 5)[:8]:
        ro, rl = _oracle_unit(w, c, b, h, 0, 0, dev)
        ref_o.append(ro)
        ref_l.append(rl)
        got_o.append(out[b, 4 * h:4 * h + 4].double().cpu().numpy())
        got_l.append(lse[b, 4 * h:4 * h + 4].double().cpu().numpy())
    ref_o, ref_l, got_o, got_l = map(np.stack, (ref_o, ref_l, got_o, got_l))
    rms = float(np.sqrt((ref_o ** 2).mean()))
    assert float(np.abs(got_o - ref_o).max()) <= TOL[0] * rms
    assert float(np.abs(got_l - ref_l).max()) <= LSE_TOL[0]
    del c
    torch.cuda.empty_cache()
