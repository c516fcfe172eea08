"""GPU parity where rounding, scaling and clamping decide the result.

Quantize + pack (bit-exact against the oracle) on crafted groups: exact grids
z + k*s, exact ties z + (k + 1/2)*s (round-half-even decides the code),
constant groups, ranges that put s at the bottom (fp16 subnormal) and near
the top of the fp16 range, offsets near the fp16 limit, and groups whose
offset or scale overflows fp16 (flagged, written as zeros).  The group rule
follows the reading of rag-lover.com's summary of arXiv 2611.09722, section
"使える条件" (asymmetric s and z per group).

Decode attention against the oracle with a non-default softmax scale, with
query and cache magnitudes that reach the kernel's power-of-two prescale
clamps (|q| < 2^-120, bf16-subnormal and zero queries, fp16-subnormal scales,
scales near the fp16 maximum), and with blocks whose scores lie far below the
running maximum (the probability-operand exponent clamp).  Tolerances as in
the other parity tests: 3e-2 * rms (FP8 operands), 2e-3 * rms (BF16 mode).
"""
import numpy as np
import pytest
import torch

import kvq_synth as synth
from oracle import kvq_oracle as orc
from tests.kvq_testlib import assert_attention_close, make_problem, run_gpu

pytestmark = pytest.mark.gpu


def _f16(v):
    return float(np.float16(v))


# ---------------------------------------------------------------------------
# Quantize + pack on crafted groups
# ---------------------------------------------------------------------------

# (s, z) pairs for which z + k*s and z + (k + 1/2)*s are exact in fp32
_GRID_SZ = [(0.0625, -1.5), (0.5, 3.0), (3.0, -100.0), (_f16(1 / 3), -100.0), (2.0 ** -10, 0.0),
            (1024.0, -30000.0), (_f16(0.1), 2.0 ** -14)]


def crafted_groups(bits, n, seed):
    """n groups of 128 fp32 values, cycling through the crafted kinds; returns
    the groups and the number of exact-tie elements they hold."""
    r = np.random.default_rng(seed)
    qmax = (1 << bits) - 1
    out = np.zeros((n, 128), np.float32)
    ties = 0
    for i in range(n):
        kind = i % 10
        s, z = _GRID_SZ[r.integers(len(_GRID_SZ))]
        if kind == 0:    # exact grid, every code present
            k = r.integers(0, qmax + 1, 128).astype(np.float64)
            k[:2] = [0, qmax]
            g = z + r.permutation(k) * s
        elif kind == 1:  # exact ties between codes, grid endpoints pinned
            k = r.integers(0, qmax, 128) + 0.5
            k[:2] = [0, qmax]
            k = r.permutation(k)
            g = z + k * s
            x32 = g.astype(np.float32).astype(np.float64)
            t = (x32 - z) / s
            ties += int(np.sum((t == k) & (k != np.round(k))))
        elif kind == 2:  # constant, fp16-exact: s = 0, every code 0
            g = np.full(128, _f16(r.standard_normal()))
        elif kind == 3:  # constant, not fp16-exact: tiny range above z
            g = np.full(128, 0.1)
        elif kind == 4:  # range near the fp16 limit of both ends
            g = r.uniform(-65000.0, 65000.0, 128)
            g[:2] = [-65000.0, 65000.0]
        elif kind == 5:  # tiny range: s an fp16 subnormal
            g = r.standard_normal() + r.uniform(0.0, 1e-6, 128)
        elif kind == 6:  # values at fp16-subnormal magnitude
            g = r.standard_normal(128) * 1e-6
        elif kind == 7:  # offset near the fp16 limit, small range
            g = -65000.0 + r.uniform(0.0, 10.0, 128)
        elif kind == 8:  # large scale: range / (2^b - 1) in the top fp16 binades
            g = r.uniform(0.0, 60000.0, 128)
        else:
            g = r.standard_normal(128)
        out[i] = g.astype(np.float32)
    return out, ties


def crafted_cache_input(bits, scheme, B, Hkv, L, seed):
    """fp32 [B, Hkv, L, 128] whose quantization groups are crafted groups:
    token rows (token-wise) or one channel over a 128-token block (channel-wise)."""
    nblk = (L + 127) // 128
    n = B * Hkv * (L if scheme == 0 else nblk * 128)
    groups, ties = crafted_groups(bits, n, seed)
    if scheme == 0:
        x = groups.reshape(B, Hkv, L, 128)
    else:  # group (b, h, j, c) -> x[b, h, 128 j : 128 j + 128, c]
        x = groups.reshape(B, Hkv, nblk, 128, 128).transpose(0, 1, 2, 4, 3).reshape(B, Hkv, nblk * 128, 128)[:, :, :L]
    return np.ascontiguousarray(x), ties


def _gpu_pack(bits, scheme, which, x, lens, page_table, num_pages, max_blocks):
    import bit_quantized_kv_decode_gb300 as kvq
    dev = torch.device("cuda")
    desc = kvq.cache_desc(bits, scheme, scheme, x.shape[1], num_pages)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pt = None if page_table is None else torch.from_numpy(page_table).to(dev)
    cache = kvq.pack(desc, which, torch.from_numpy(x).to(dev), torch.from_numpy(lens).to(dev), pt, max_blocks,
                     dev_status=st)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in cache], int(st.item())


def _pages_of(lens, page_table, max_blocks):
    pages = []
    for b, n in enumerate(lens.tolist()):
        for j in range((n + 127) // 128):
            pages.append(int(page_table[b, j]) if page_table is not None else b * max_blocks + j)
    return np.array(sorted(pages))


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("scheme", [0, 1])
@pytest.mark.parametrize("which", [0, 1])
def test_pack_crafted_groups_bitexact(bits, scheme, which):
    B, Hkv, L = 3, 2, 384
    lens = np.array([384, 300, 129], np.int32)
    x, ties = crafted_cache_input(bits, scheme, B, Hkv, L, seed=1000 + 4 * bits + 2 * scheme + which)
    assert ties > 100  # the tie groups really hold exact ties
    max_blocks = 3
    pt, num_pages = synth.page_table_for(torch.from_numpy(lens), 5, max_blocks)
    pt = pt.numpy()
    (codes, scale, zero), st = _gpu_pack(bits, scheme, which, x, lens, pt, num_pages, max_blocks)
    assert st == 0
    rc, rs, rz = orc.pack_cache(x, lens, bits, scheme, which, pt, num_pages)
    pages = _pages_of(lens, pt, max_blocks)
    assert np.array_equal(codes[pages], rc[pages])
    assert np.array_equal(scale.view(np.uint16)[pages], rs.view(np.uint16)[pages])
    assert np.array_equal(zero.view(np.uint16)[pages], rz.view(np.uint16)[pages])


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("scheme", [0, 1])
def test_pack_fp16_overflow_flagged_and_zeroed(bits, scheme):
    """A group whose offset (minimum below -65504) or scale ((max - z) / (2^b - 1)
    above 65504) overflows fp16 is flagged KVQ_DEV_NONFINITE and written as
    zeros; every other group stays bit-exact with the oracle."""
    import bit_quantized_kv_decode_gb300 as kvq
    B, Hkv, L = 1, 1, 256
    lens = np.array([L], np.int32)
    r = np.random.default_rng(7 + bits + 2 * scheme)
    x = r.standard_normal((B, Hkv, L, 128)).astype(np.float32)
    x_ref = x.copy()
    bad = []
    for g, (lo, hi) in enumerate([(-70000.0, 0.0), (0.0, 1e6)]):  # offset overflow, scale overflow
        if scheme == 0:
            t = 5 + 100 * g
            x[0, 0, t, :] = np.linspace(lo, hi, 128, dtype=np.float32)
            x_ref[0, 0, t, :] = 0.0
            bad.append(("tok", t))
        else:
            c = 3 + 50 * g
            x[0, 0, 128 * g:128 * g + 128, c] = np.linspace(lo, hi, 128, dtype=np.float32)
            x_ref[0, 0, 128 * g:128 * g + 128, c] = 0.0
    (codes, scale, zero), st = _gpu_pack(bits, scheme, 0, x, lens, None, 2, 2)
    assert st == kvq.DEV_NONFINITE
    rc, rs, rz = orc.pack_cache(x_ref, lens, bits, scheme, 0, None, 2)
    assert np.array_equal(codes, rc)  # the flagged groups: zeros, exactly like an all-zero group
    assert np.array_equal(scale.view(np.uint16), rs.view(np.uint16))
    assert np.array_equal(zero.view(np.uint16), rz.view(np.uint16))
    with pytest.raises(orc.OracleError):
        orc.pack_cache(x, lens, bits, scheme, 0, None, 2)


# ---------------------------------------------------------------------------
# Decode attention: softmax scale and extreme magnitudes
# ---------------------------------------------------------------------------

def _w(bits, kcw, vcw, B=2, Hkv=2, L=600):
    return synth.shrink(synth.WORKLOADS["tiny"], batch=B, num_kv_heads=Hkv, num_q_heads=4 * Hkv, bits=bits,
                        k_scheme=kcw, v_scheme=vcw, max_seq_len=L)


@pytest.mark.parametrize("sm_scale", [0.05, 0.3])
@pytest.mark.parametrize("bits,kcw,vcw", [(4, 1, 0), (2, 0, 1), (4, 0, 0), (2, 1, 1)])
def test_softmax_scale(sm_scale, bits, kcw, vcw):
    pb = make_problem(_w(bits, kcw, vcw), seed=900 + 4 * bits + 2 * kcw + vcw, lens=[600, 200], sm_scale=sm_scale)
    for mode in (0, 1):
        res = run_gpu(pb, mode=mode)
        assert res["status"] == 0
        assert_attention_close(pb, res, mode)


# (q scale, K scale, V scale); K and V are N(0, 1) times the scale (no
# outlier channels, so that the largest value stays inside fp16's range)
MAGNITUDES = {
    "large_q_small_k": (1e3, 1e-3, 1.0),     # big Q' prescale step, scores of ordinary size
    "q_below_2^-120": (1e-37, 1.0, 1.0),     # prescale clamp (factor 1)
    "bf16_subnormal_q": (1e-39, 1.0, 1.0),
    "zero_q": (0.0, 1.0, 1.0),
    "fp16_subnormal_scales": (1e4, 1e-5, 1e-5),  # largest s of a block below 2^-14
    "scales_near_fp16_max": (1e-4, 8e3, 8e3),    # s within the top fp16 binades
}


def _magnitude_problem(bits, kcw, vcw, case, seed):
    qs, ks, vs = MAGNITUDES[case]
    w = _w(bits, kcw, vcw)
    g = torch.Generator().manual_seed(seed)
    lens = [600, 333]
    q = (torch.randn(w.batch, w.num_q_heads, 128, generator=g) * qs).to(torch.bfloat16)
    k = torch.randn(w.batch, w.num_kv_heads, 600, 128, generator=g) * ks
    v = torch.randn(w.batch, w.num_kv_heads, 600, 128, generator=g) * vs
    k[1, :, 333:] = 0.0
    v[1, :, 333:] = 0.0
    return make_problem(w, seed, lens=lens, q=q, k=k, v=v)


@pytest.mark.parametrize("case", sorted(MAGNITUDES))
@pytest.mark.parametrize("bits,kcw,vcw", [(4, 0, 0), (4, 1, 1), (2, 1, 0), (2, 0, 1)])
def test_extreme_magnitudes(case, bits, kcw, vcw):
    pb = _magnitude_problem(bits, kcw, vcw, case, seed=1300 + 4 * bits + 2 * kcw + vcw)
    for mode in (0, 1):
        res = run_gpu(pb, mode=mode)
        assert res["status"] == 0
        assert np.all(np.isfinite(res["out"]))
        assert_attention_close(pb, res, mode)


@pytest.mark.parametrize("v_scale", [1.0, 1e-7])
@pytest.mark.parametrize("bits,kcw,vcw", [(4, 1, 0), (4, 0, 1), (2, 0, 0), (2, 1, 1)])
def test_blocks_far_below_running_max(v_scale, bits, kcw, vcw):
    """Blocks 1.. have scores hundreds of natural-log units below block 0's,
    so their tile pairs sit far below the running maximum (the P' exponent
    clamp); with V scaled by 1e-7 the V scales are fp16 subnormals as well."""
    w = _w(bits, kcw, vcw, B=2, Hkv=1, L=700)
    g = torch.Generator().manual_seed(77 + bits + 2 * kcw + vcw)
    q = torch.randn(w.batch, w.num_q_heads, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(w.batch, 1, 700, 128, generator=g)
    v = torch.randn(w.batch, 1, 700, 128, generator=g) * v_scale
    shifts = [0.0, -300.0, -150.0, -220.0, -120.0, -400.0]  # per block, natural-log score units
    for b in range(w.batch):
        qsum = q[b].float().sum(0)
        u = qsum / qsum.norm()
        # score shift of head h: sm_scale * (q_h . u) * beta, with q_h . u ~ |q_h|^2 / |qsum|
        gain = float((q[b].float() @ u).min()) / np.sqrt(128.0)
        for j, sh in enumerate(shifts):
            if sh != 0.0:
                k[b, 0, 128 * j:128 * (j + 1)] += (sh / gain) * u
    lens = [700, 650]
    k[1, :, 650:] = 0.0
    v[1, :, 650:] = 0.0
    pb = make_problem(w, 88, lens=lens, q=q, k=k, v=v)
    for mode in (0, 1):
        res = run_gpu(pb, mode=mode)
        assert res["status"] == 0
        assert np.all(np.isfinite(res["out"]))
        assert_attention_close(pb, res, mode)
