"""GPU decode attention against the oracle, element by element.

Tolerances (from the build target): max|out - oracle| <= 3e-2 * rms(oracle)
on the FP8-operand path and <= 2e-3 * rms in the BF16-operand correctness
mode; lse within 1e-2 / 1e-3 (natural log).
"""
import numpy as np
import pytest
import torch

import kvq_synth as synth
from tests.kvq_testlib import assert_attention_close, make_problem, run_gpu

pytestmark = pytest.mark.gpu


def _w(bits, kcw, vcw, B=3, Hkv=2, L=1024):
    return synth.shrink(synth.WORKLOADS["tiny"], batch=B, num_kv_heads=Hkv, num_q_heads=4 * Hkv, bits=bits,
                        k_scheme=kcw, v_scheme=vcw, max_seq_len=L)


@pytest.mark.parametrize("mode", [0, 1])
def test_tiny_workload(mode):
    """B=1, Hkv=1, Hq=4, L=256, INT4 K/V token-wise."""
    pb = make_problem(synth.WORKLOADS["tiny"], seed=1)
    res = run_gpu(pb, mode=mode)
    assert res["status"] == 0
    assert_attention_close(pb, res, mode)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kcw,vcw", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("mode", [0, 1])
def test_schemes_ragged(bits, kcw, vcw, mode):
    """Every bit width x K/V scheme pair x operand mode on a ragged batch that
    spans several tiles, a ragged tail and a one-token sequence."""
    pb = make_problem(_w(bits, kcw, vcw), seed=100 + 8 * bits + 2 * kcw + vcw, lens=[1000, 129, 1])
    res = run_gpu(pb, mode=mode)
    assert res["status"] == 0
    assert_attention_close(pb, res, mode)


@pytest.mark.parametrize("kcw,vcw", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_e2m1_v_placement(kcw, vcw):
    """2-bit V codes fed as E2M1 values from shared memory (KVQ_FLAG_E2M1_V)
    on a ragged batch, whole units and units split over CTAs."""
    import bit_quantized_kv_decode_gb300 as kvq
    pb = make_problem(_w(2, kcw, vcw), seed=700 + 2 * kcw + vcw, lens=[1000, 129, 1])
    for num_ctas in (0, 5):
        res = run_gpu(pb, mode=0, num_ctas=num_ctas, flags=kvq.FLAG_E2M1_V)
        assert res["status"] == 0
        assert_attention_close(pb, res, 0)


@pytest.mark.parametrize("gq", [1, 2, 8])
@pytest.mark.parametrize("kcw,vcw", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_query_heads_per_kv_head(gq, kcw, vcw):
    """1, 2 and 8 query heads per KV head (8 = two work units per KV head) on
    a ragged batch, both operand modes."""
    bits = 4 if kcw != vcw else 2
    w = synth.shrink(synth.WORKLOADS["tiny"], batch=3, num_kv_heads=2, num_q_heads=gq * 2, bits=bits,
                     k_scheme=kcw, v_scheme=vcw, max_seq_len=1024)
    pb = make_problem(w, seed=300 + 4 * gq + 2 * kcw + vcw, lens=[1000, 129, 1])
    for mode in (0, 1):
        res = run_gpu(pb, mode=mode)
        assert res["status"] == 0
        assert_attention_close(pb, res, mode)


@pytest.mark.parametrize("gq", [1, 8])
def test_query_heads_split_merge(gq):
    """Units cut by CTA ranges merge correctly with 1 and 8 query heads per KV head."""
    w = synth.shrink(synth.WORKLOADS["tiny"], batch=2, num_kv_heads=2, num_q_heads=gq * 2, bits=4, k_scheme=1,
                     v_scheme=0, max_seq_len=2048)
    pb = make_problem(w, seed=400 + gq, lens=[2048, 1500])
    for num_ctas in (3, 7):
        res = run_gpu(pb, mode=1, num_ctas=num_ctas)
        assert res["status"] == 0
        assert_attention_close(pb, res, 1)


@pytest.mark.parametrize("bits,kcw,vcw", [(4, 1, 0), (2, 0, 1)])
def test_maximum_batch(bits, kcw, vcw):
    """The largest batch a call takes (1024 sequences), ragged 0..300 tokens
    with empty ones: every sequence checked against the oracle."""
    B = 1024
    lens = np.random.default_rng(500 + bits).integers(0, 301, size=B)
    lens[::97] = 0
    w = synth.shrink(synth.WORKLOADS["tiny"], batch=B, num_kv_heads=1, num_q_heads=4, bits=bits, k_scheme=kcw,
                     v_scheme=vcw, max_seq_len=300)
    pb = make_problem(w, seed=600 + bits, lens=lens.tolist())
    for mode in (0, 1):
        res = run_gpu(pb, mode=mode)
        assert res["status"] == 0
        empty = np.flatnonzero(lens == 0)
        assert np.all(res["out"][empty] == 0) and np.all(np.isneginf(res["lse"][empty]))
        assert_attention_close(pb, res, mode)


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 5, 8, 17])
def test_split_ranges_merge(num_ctas):
    """Tile ranges cut (sequence, head) units in many places; merges must agree."""
    pb = make_problem(_w(4, 1, 0, B=2, Hkv=2, L=2048), seed=7, lens=[2048, 1500])
    res = run_gpu(pb, mode=1, num_ctas=num_ctas)
    assert res["status"] == 0
    assert_attention_close(pb, res, 1)


def test_edge_lengths_and_empty():
    """Empty sequences (out 0, lse -inf), exactly one block, one past a block."""
    pb = make_problem(_w(2, 1, 1, B=6, Hkv=1, L=512), seed=3, lens=[0, 128, 129, 1, 0, 512])
    for mode in (0, 1):
        res = run_gpu(pb, mode=mode)
        assert res["status"] == 0
        assert np.all(res["out"][[0, 4]] == 0) and np.all(np.isneginf(res["lse"][[0, 4]]))
        assert_attention_close(pb, res, mode)


def test_all_empty():
    pb = make_problem(_w(4, 0, 0, B=2, Hkv=1, L=128), seed=3, lens=[0, 0])
    res = run_gpu(pb)
    assert res["status"] == 0
    assert np.all(res["out"] == 0) and np.all(np.isneginf(res["lse"]))


def test_paged_ragged_scaled_down():
    """The paged ragged workload's structure at a size the oracle finishes fast:
    8 sequences, log-uniform lengths, shuffled 128-token pages."""
    w = synth.shrink(synth.WORKLOADS["paged_ragged_int2"], batch=8, num_kv_heads=2, num_q_heads=8,
                     max_seq_len=3000, ragged=(100, 3000))
    pb = make_problem(w, seed=21)
    assert pb.page_table is not None
    for mode in (0, 1):
        res = run_gpu(pb, mode=mode)
        assert res["status"] == 0
        assert_attention_close(pb, res, mode)


def test_b8_l4k_int2_full_size():
    """B=8, Hkv=8, Hq=32, L=4096, INT2 K channel-wise / V token-wise, in full."""
    pb = make_problem(synth.WORKLOADS["b8_l4k_int2"], seed=2)
    res = run_gpu(pb, mode=0)
    assert res["status"] == 0
    assert_attention_close(pb, res, 0)


def test_repeat_calls_identical():
    """Same inputs, same launch shape -> the same bits (no stale workspace state)."""
    import bit_quantized_kv_decode_gb300 as kvq
    pb = make_problem(_w(4, 1, 0, B=2, Hkv=2, L=2048), seed=9, lens=[2048, 700])
    dev = torch.device("cuda")
    res = run_gpu(pb, num_ctas=5)
    q = pb.q.to(dev)
    lens = pb.lens.to(dev)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(3):
        o, l = kvq.decode_attn(res["desc"], q, res["k_cache"], res["v_cache"], lens, max_blocks=pb.max_blocks,
                               num_ctas=5, workspace=ws)
        outs.append((o.clone(), l.clone()))
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    assert np.array_equal(outs[0][0].cpu().double().numpy(), res["out"])


def test_bad_lengths_and_pages_flagged():
    import bit_quantized_kv_decode_gb300 as kvq
    pb = make_problem(_w(4, 0, 0, B=2, Hkv=1, L=256), seed=4, lens=[256, 200], paged=True)
    dev = torch.device("cuda")
    res = run_gpu(pb)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    bad_lens = torch.tensor([256, 999], dtype=torch.int32, device=dev)
    pt = pb.page_table.to(dev)
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


def test_stalled_pipeline_times_out_cleanly():
    """A withheld tile makes every waiting stage run into its time limit; the
    call reports KVQ_DEV_TIMEOUT, the context stays usable, and the next call
    is correct."""
    import bit_quantized_kv_decode_gb300 as kvq
    pb = make_problem(_w(4, 0, 1, B=1, Hkv=1, L=1024), seed=12, lens=[1024])
    dev = torch.device("cuda")
    res = run_gpu(pb)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kvq.decode_attn(res["desc"], pb.q.to(dev), res["k_cache"], res["v_cache"], pb.lens.to(dev),
                    max_blocks=pb.max_blocks, num_ctas=1, dev_status=st, flags=kvq.FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert int(st.item()) & kvq.DEV_TIMEOUT
    again = run_gpu(pb, num_ctas=1)
    assert again["status"] == 0
    assert_attention_close(pb, again, 0)


def test_merge_kernel_matches_oracle():
    import bit_quantized_kv_decode_gb300 as kvq
    from oracle import kvq_oracle as orc
    g = torch.Generator().manual_seed(5)
    R, S, D = 37, 5, 128
    o = torch.randn(R, S, D, generator=g)
    l = torch.randn(R, S, generator=g) * 3
    l[3, :] = -float("inf")
    l[4, 1:] = -float("inf")
    out, lse = kvq.merge(o.cuda(), l.cuda())
    ro, rl = orc.merge(o.double().numpy(), l.double().numpy())
    assert np.allclose(out.cpu().double().numpy(), ro, rtol=1e-5, atol=1e-6)
    fin = np.isfinite(rl)
    assert np.allclose(lse.cpu().double().numpy()[fin], rl[fin], rtol=1e-6, atol=1e-5)
    assert np.isneginf(lse[3].item()) and np.all(out[3].cpu().numpy() == 0)
