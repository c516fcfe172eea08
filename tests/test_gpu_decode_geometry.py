"""Decode attention on the general cache geometry (head dims 64 / 256, groups
of 32 / 64 elements, and groups of 32 / 64 with head dim 128) against the
oracle: every bit width and K/V scheme pair in both operand modes, query heads per KV head 1 / 2 /
4 / 8, ragged and empty sequences, paged caches, block ranges split one way
and many ways, an explicit softmax scale and the stall hook (the static
entry point on this geometry: tests/test_zz_no_alloc.py).  Accumulator folds per quantization group follow the
rag-lover.com summary of arXiv 2611.09722, section "限界と未検証の範囲"."""
import numpy as np
import pytest
import kvq_synth as synth
from kvq_testlib import assert_attention_close, make_problem, run_gpu

pytestmark = pytest.mark.gpu

GEOMETRIES = [(64, 32), (64, 64), (128, 32), (128, 64), (256, 32), (256, 64), (256, 128)]
PAIRS = [(0, 0), (0, 1), (1, 0), (1, 1)]


def _w(D, G, bits, ks, vs, B=3, Hkv=2, Hq=8, L=300, paged=False):
    return synth.Workload(f"geom_d{D}_g{G}", B, Hkv, Hq, D, L, bits, ks, vs, paged=paged, group=G)


@pytest.mark.parametrize("D,G", GEOMETRIES)
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("ks,vs", PAIRS)
def test_decode_geometry_parity(D, G, bits, ks, vs):
    w = _w(D, G, bits, ks, vs, paged=(D + G + bits) % 2 == 0)
    pb = make_problem(w, 300 + D + G + bits + 2 * ks + vs, lens=[300, 129, 1])
    res = run_gpu(pb)
    assert res["status"] == 0
    assert_attention_close(pb, res, 0)


@pytest.mark.parametrize("D,G", GEOMETRIES)
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("ks,vs", PAIRS)
def test_decode_geometry_parity_bf16(D, G, bits, ks, vs):
    """The BF16-operand mode (exact BF16 codes, two-part BF16 Q' and P'):
    the tighter tolerance."""
    w = _w(D, G, bits, ks, vs, paged=(D + G + bits) % 2 == 1)
    pb = make_problem(w, 700 + D + G + bits + 2 * ks + vs, lens=[300, 129, 1])
    res = run_gpu(pb, mode=1)
    assert res["status"] == 0
    assert_attention_close(pb, res, 1)


@pytest.mark.parametrize("D,G", [(64, 32), (256, 64)])
@pytest.mark.parametrize("heads", [1, 2, 8])
def test_decode_geometry_gqa(D, G, heads):
    w = _w(D, G, 4, 1, 0, B=2, Hkv=2, Hq=2 * heads)
    pb = make_problem(w, 40 + heads, lens=[257, 90])
    res = run_gpu(pb)
    assert res["status"] == 0
    assert_attention_close(pb, res, 0)


@pytest.mark.parametrize("D,G,ks,vs", [(256, 32, 0, 0), (64, 64, 1, 1), (128, 32, 1, 0)])
def test_decode_geometry_splits(D, G, ks, vs):
    """One range per unit, the default split and one block per range give the
    oracle's result.  The merge is exact up to rounding, but each range
    prescales P' from its own running maximum, so the E4M3 roundings -- not
    the results -- differ between splits: they agree to the operand error."""
    w = _w(D, G, 2, ks, vs, B=2, Hkv=1, Hq=4, L=5000, paged=True)
    pb = make_problem(w, 77, lens=[5000, 1700])
    outs = []
    for n in (1, 0, 100000):
        res = run_gpu(pb, num_ctas=n)
        assert res["status"] == 0
        assert_attention_close(pb, res, 0)
        outs.append(res["out"])
    rms = float(np.sqrt((outs[0] ** 2).mean()))
    assert np.abs(outs[0] - outs[2]).max() <= 3e-3 * rms


@pytest.mark.parametrize("lens", [[0, 0], [0, 5], [128, 0, 256]])
def test_decode_geometry_empty_and_exact_blocks(lens):
    w = _w(64, 32, 4, 0, 1, B=len(lens), Hkv=1, Hq=4, L=max(lens) or 1)
    pb = make_problem(w, 5, lens=lens)
    res = run_gpu(pb)
    assert res["status"] == 0
    for b, n in enumerate(lens):
        if n == 0:
            assert np.all(res["out"][b] == 0) and np.all(np.isneginf(res["lse"][b]))
    assert_attention_close(pb, res, 0)


@pytest.mark.parametrize("D,G", [(256, 64), (64, 32)])
@pytest.mark.parametrize("mult", [0.57, 3.4])
def test_decode_geometry_sm_scale(D, G, mult):
    """An explicit softmax scale: the same multiples of the default 1/sqrt(D)
    as the head-dim-128 cases (0.05 and 0.3 there); score and lse errors grow
    in proportion to the scale."""
    w = _w(D, G, 2, 1, 0, B=2, Hkv=1, Hq=4)
    pb = make_problem(w, 11, lens=[300, 40], sm_scale=mult / D ** 0.5)
    res = run_gpu(pb)
    assert res["status"] == 0
    assert_attention_close(pb, res, 0)


def test_decode_geometry_stall_reports_timeout():
    """The stall hook withholds one block from one CTA: its wait runs out, the
    call returns, and the timeout bit is set (nothing hangs)."""
    import bit_quantized_kv_decode_gb300 as kvq
    w = _w(64, 32, 4, 0, 0, B=1, Hkv=1, Hq=4)
    pb = make_problem(w, 3, lens=[300])
    res = run_gpu(pb, flags=kvq.FLAG_TEST_STALL)
    assert res["status"] & kvq.DEV_TIMEOUT
    res = run_gpu(pb)  # the context is still usable
    assert res["status"] == 0
    assert_attention_close(pb, res, 0)


@pytest.mark.parametrize("D,G,bits,ks,vs", [(256, 64, 4, 0, 1), (128, 32, 2, 0, 0), (64, 32, 4, 1, 0)])
def test_decode_geometry_mma_stall_reports_timeout(D, G, bits, ks, vs):
    """The MMA stall hook: the first CTA's MMA barrier waits for two signals a
    phase, so its first QK^T wait runs out (per warp with token-wise K, the
    failure read at the next CTA barrier; CTA-wide with channel-wise K): the
    call returns with the timeout bit set, nothing hangs, and the next call
    is correct."""
    import bit_quantized_kv_decode_gb300 as kvq
    w = _w(D, G, bits, ks, vs, B=2, Hkv=1, Hq=4, L=700)
    pb = make_problem(w, 5 + D + G, lens=[700, 300])
    res = run_gpu(pb, flags=kvq.FLAG_TEST_STALL_MMA)
    assert res["status"] & kvq.DEV_TIMEOUT
    res = run_gpu(pb)
    assert res["status"] == 0
    assert_attention_close(pb, res, 0)


def test_decode_geometry_e2m1_unsupported():
    """The E2M1 V placement is built for head dim 128 with groups of 128 only."""
    import bit_quantized_kv_decode_gb300 as kvq
    from bit_quantized_kv_decode_gb300 import _lib
    w = _w(64, 32, 2, 0, 0, B=1, Hkv=1, Hq=4)
    pb = make_problem(w, 3, lens=[100])
    with pytest.raises(_lib.KvqError) as e:
        run_gpu(pb, flags=kvq.FLAG_E2M1_V)
    assert e.value.status == 2



@pytest.mark.parametrize("D,G,bits,ks,vs", [(64, 32, 2, 1, 0), (256, 64, 4, 0, 1)])
def test_decode_geometry_maximum_batch(D, G, bits, ks, vs):
    """1024 sequences (the most a call takes), ragged 0..300 tokens with
    empty ones: every sequence against the oracle."""
    B = 1024
    lens = np.random.default_rng(900 + D).integers(0, 301, size=B)
    lens[::97] = 0
    w = _w(D, G, bits, ks, vs, B=B, Hkv=1, Hq=4, L=300)
    pb = make_problem(w, 910 + D, lens=lens.tolist())
    res = run_gpu(pb)
    assert res["status"] == 0
    empty = np.flatnonzero(lens == 0)
    assert np.all(res["out"][empty] == 0) and np.all(np.isneginf(res["lse"][empty]))
    assert_attention_close(pb, res, 0)


# (q scale, K scale, V scale): the prescale clamps of Q' and the group scales
MAGNITUDES = {
    "large_q_small_k": (1e3, 1e-3, 1.0),
    "q_below_2^-120": (1e-37, 1.0, 1.0),
    "zero_q": (0.0, 1.0, 1.0),
    "fp16_subnormal_scales": (1e4, 1e-5, 1e-5),
    "scales_near_fp16_max": (1e-4, 8e3, 8e3),
}


@pytest.mark.parametrize("case", sorted(MAGNITUDES))
@pytest.mark.parametrize("D,G,bits,ks,vs", [(256, 64, 4, 1, 0), (64, 32, 2, 0, 1), (128, 32, 2, 1, 1)])
def test_decode_geometry_extreme_magnitudes(case, D, G, bits, ks, vs):
    import torch
    qs, kscale, vscale = MAGNITUDES[case]
    w = _w(D, G, bits, ks, vs, B=2, Hkv=2, Hq=8, L=600)
    g = torch.Generator().manual_seed(1400 + D + G)
    q = (torch.randn(2, 8, D, generator=g) * qs).to(torch.bfloat16)
    k = torch.randn(2, 2, 600, D, generator=g) * kscale
    v = torch.randn(2, 2, 600, D, generator=g) * vscale
    k[1, :, 333:] = 0.0
    v[1, :, 333:] = 0.0
    pb = make_problem(w, 1400 + D, lens=[600, 333], q=q, k=k, v=v)
    res = run_gpu(pb)
    assert res["status"] == 0
    assert np.all(np.isfinite(res["out"]))
    assert_attention_close(pb, res, 0)


@pytest.mark.parametrize("D,G,bits,ks,vs", [(256, 32, 4, 1, 0), (64, 64, 2, 0, 0)])
def test_decode_geometry_blocks_far_below_running_max(D, G, bits, ks, vs):
    """Later blocks' scores sit 120-400 natural-log units below block 0's
    (the P' exponent clamp)."""
    import torch
    w = _w(D, G, bits, ks, vs, B=1, Hkv=1, Hq=4, L=700)
    g = torch.Generator().manual_seed(88 + D)
    q = torch.randn(1, 4, D, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 1, 700, D, generator=g)
    v = torch.randn(1, 1, 700, D, generator=g)
    qsum = q[0].float().sum(0)
    u = qsum / qsum.norm()
    gain = float((q[0].float() @ u).min()) / np.sqrt(float(D))
    for j, sh in enumerate([0.0, -300.0, -150.0, -220.0, -120.0, -400.0]):
        if sh != 0.0:
            k[0, 0, 128 * j:128 * (j + 1)] += (sh / gain) * u
    pb = make_problem(w, 89 + D, lens=[700], q=q, k=k, v=v)
    res = run_gpu(pb)
    assert res["status"] == 0
    assert np.all(np.isfinite(res["out"]))
    assert_attention_close(pb, res, 0)


def test_decode_geometry_repeat_calls_identical():
    """Same inputs, same launch shape -> the same bits (the kernel reduces in a
    fixed order; no stale workspace state)."""
    import torch
    import bit_quantized_kv_decode_gb300 as kvq
    w = _w(256, 64, 4, 1, 0, B=2, Hkv=2, Hq=8, L=2048)
    pb = make_problem(w, 19, lens=[2048, 700])
    dev = torch.device("cuda")
    res = run_gpu(pb, num_ctas=7)
    q, lens = pb.q.to(dev), pb.lens.to(dev)
    ws = torch.empty(4 << 20, dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(3):
        o, l = kvq.decode_attn(res["desc"], q, res["k_cache"], res["v_cache"], lens, max_blocks=pb.max_blocks,
                               num_ctas=7, workspace=ws)
        outs.append((o.clone(), l.clone()))
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    assert np.array_equal(outs[0][0].cpu().double().numpy(), res["out"])


def test_decode_geometry_bad_lengths_and_pages_flagged():
    import torch
    import bit_quantized_kv_decode_gb300 as kvq
    w = _w(64, 32, 4, 0, 0, B=2, Hkv=1, Hq=4, L=256, paged=True)
    pb = make_problem(w, 4, lens=[256, 200])
    dev = torch.device("cuda")
    res = run_gpu(pb)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pt = pb.page_table.to(dev)
    bad_lens = torch.tensor([256, 999], dtype=torch.int32, device=dev)
    o, l = kvq.decode_attn(res["desc"], pb.q.to(dev), res["k_cache"], res["v_cache"], bad_lens, pt, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kvq.DEV_BAD_SEQ_LEN
    assert np.all(o[1].cpu().numpy() == 0) and np.all(np.isneginf(l[1].cpu().numpy()))
    st.zero_()
    pt2 = pt.clone()
    pt2[0, 1] = 10 ** 6
    kvq.decode_attn(res["desc"], pb.q.to(dev), res["k_cache"], res["v_cache"], pb.lens.to(dev), pt2, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kvq.DEV_BAD_PAGE
