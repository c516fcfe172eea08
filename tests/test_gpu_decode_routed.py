"""Parity of the general (block-range) kernel on the specialised kernel's
geometry: head dim 128, groups of 128, E4M3 operands.  kvq_decode_attn sends
such a call there once it holds at least 8,192 (sequence, unit, block)
triples of max_blocks per unit; here one long sequence sets max_blocks and
the others are short and ragged (with an empty one), so the oracle still
sees every element -- every bit width, scheme pair and query-head count, and
forced range counts."""
import pytest
import torch

import kvq_synth as synth
from tests.kvq_testlib import assert_attention_close, make_problem, run_gpu

pytestmark = pytest.mark.gpu

LENS = [16384, 300, 129, 1, 0, 1000, 128, 257, 2048, 77, 640, 3, 1500, 256, 900, 130]  # max_blocks = 128


def _workload(bits, kcw, vcw, gq):
    return synth.shrink(synth.WORKLOADS["tiny"], batch=len(LENS), num_kv_heads=4, num_q_heads=4 * gq, bits=bits,
                        k_scheme=kcw, v_scheme=vcw, max_seq_len=max(LENS))


def _path(pb):
    import bit_quantized_kv_decode_gb300 as kvq
    w = pb.w
    desc = kvq.cache_desc(w.bits, w.k_scheme, w.v_scheme, w.num_kv_heads, pb.num_pages, head_dim=w.head_dim,
                          group=w.group)
    return kvq.decode_path(kvq.attn_desc(desc, w.batch, pb.max_blocks, num_q_heads=w.num_q_heads))


@pytest.mark.parametrize("gq", [1, 4, 8])
@pytest.mark.parametrize("kcw,vcw", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("bits", [2, 4])
def test_general_kernel_default_geometry(bits, kcw, vcw, gq):
    from bit_quantized_kv_decode_gb300 import _lib
    pb = make_problem(_workload(bits, kcw, vcw, gq), seed=900 + 16 * bits + 8 * kcw + 4 * vcw + gq, lens=LENS)
    assert _path(pb) == _lib.PATH_GENERAL
    res = run_gpu(pb)
    assert res["status"] == 0
    assert_attention_close(pb, res, 0)


@pytest.mark.parametrize("num_ctas", [16, 100, 5000])
def test_general_kernel_default_geometry_ranges(num_ctas):
    """Forced range counts: one range per unit, a few, and more ranges than
    most sequences have blocks (every part merged by log-sum-exp)."""
    pb = make_problem(_workload(4, 1, 0, 4), seed=950 + num_ctas, lens=LENS)
    res = run_gpu(pb, num_ctas=num_ctas)
    assert res["status"] == 0
    assert_attention_close(pb, res, 0)


@pytest.mark.parametrize("bits,kcw,vcw", [(4, 1, 0), (2, 0, 0)])
def test_general_kernel_default_geometry_stall_reports_timeout(bits, kcw, vcw):
    """A withheld copy (test hook: the first CTA skips its first block) makes
    that CTA's bounded wait run out: the call returns with KVQ_DEV_TIMEOUT set,
    nothing hangs, and the next call is correct (a 4-bit and a 2-bit instance,
    whose copy rings refill at different points of a block)."""
    import bit_quantized_kv_decode_gb300 as kvq
    pb = make_problem(_workload(bits, kcw, vcw, 4), seed=970 + bits, lens=LENS)
    res = run_gpu(pb, flags=kvq.FLAG_TEST_STALL)
    assert res["status"] & kvq.DEV_TIMEOUT
    again = run_gpu(pb)
    assert again["status"] == 0
    assert_attention_close(pb, again, 0)


@pytest.mark.parametrize("bits,kcw,vcw,gq", [(2, 0, 0, 4), (4, 0, 1, 4), (4, 0, 0, 8), (4, 1, 0, 4)])
def test_general_kernel_default_geometry_mma_stall_reports_timeout(bits, kcw, vcw, gq):
    """A QK^T completion that never signals (test hook: the first CTA's MMA
    barrier waits for two signals a phase) makes the waits for it run out --
    per warp with token-wise K, the failure kept in shared memory and read at
    the next CTA barrier; CTA-wide with channel-wise K: the call returns with
    KVQ_DEV_TIMEOUT set, nothing hangs, and the next call is correct."""
    import bit_quantized_kv_decode_gb300 as kvq
    pb = make_problem(_workload(bits, kcw, vcw, gq), seed=980 + bits + 2 * vcw + gq, lens=LENS)
    res = run_gpu(pb, flags=kvq.FLAG_TEST_STALL_MMA)
    assert res["status"] & kvq.DEV_TIMEOUT
    again = run_gpu(pb)
    assert again["status"] == 0
    assert_attention_close(pb, again, 0)
