"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- hand-worked fixtures, closed forms, invariants, a library
attention routine, brute force on tiny inputs -- and the mutation tests at the
end plant plausible mistakes in the oracle and check that a pin catches each.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import kvq_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_bits(x):
    t = torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# fp16 directed rounding: largest fp16 <= x and smallest fp16 >= x
# ---------------------------------------------------------------------------

def test_fp16_directed_rounding_brackets():
    x = np.concatenate([_rng(0).standard_normal(20000).astype(np.float32) * 10,
                        np.float32([0.0, -0.0, 1.0, -1.0, 0.1, -0.1, 65504.0, -65504.0, 6e-8, -6e-8])])
    dn = o.fp16_round_down(x).astype(np.float64)
    up = o.fp16_round_up(x).astype(np.float64)
    xd = x.astype(np.float64)
    assert np.all(dn <= xd) and np.all(up >= xd)
    # no fp16 strictly between: the neighbours cross x
    with np.errstate(over="ignore"):
        nxt = np.nextafter(o.fp16_round_down(x), np.float16(np.inf)).astype(np.float64)
        prv = np.nextafter(o.fp16_round_up(x), np.float16(-np.inf)).astype(np.float64)
    assert np.all((nxt > xd) | (dn == xd))
    assert np.all((prv < xd) | (up == xd))


# ---------------------------------------------------------------------------
# Quantizer
# ---------------------------------------------------------------------------

def check_quant_bound(quantize_groups, bits, X):
    """|x - (s q + z)| <= s/2 + 2^-22 |x - z| for every element (IEEE fp32
    subtract and divide each add at most 2^-24 relative error); degenerate
    groups (s = 0) reproduce x exactly; codes lie in [0, 2^b - 1]; z <= min."""
    q, s, z = quantize_groups(X, bits)
    s64 = s.astype(np.float64)[:, None]
    z64 = z.astype(np.float64)[:, None]
    xh = s64 * q.astype(np.float64) + z64
    X64 = X.astype(np.float64)
    err = np.abs(X64 - xh)
    bound = s64 / 2 + 2.0 ** -22 * np.abs(X64 - z64)
    assert np.all(q <= (1 << bits) - 1)
    assert np.all(z64[:, 0] <= X64.min(axis=1))
    assert np.all(err <= bound), float((err - bound).max())
    # s is the tightest fp16 that covers the range: one fp16 step smaller would not
    rng = (X.max(axis=1) - z.astype(np.float32)).astype(np.float32)
    need = (rng / np.float32((1 << bits) - 1)).astype(np.float32).astype(np.float64)
    prev = np.nextafter(s, np.float16(-np.inf)).astype(np.float64)
    nz = s > 0
    assert np.all(prev[nz] < need[nz])


@pytest.mark.parametrize("bits", [2, 4])
def test_quant_error_bound(bits):
    r = _rng(bits)
    X = r.standard_normal((4000, 128)).astype(np.float32)
    X[::7] *= 13.0  # outlier groups
    X[::11] += 40.0  # offset groups
    X[5, :] = 0.25   # constant, fp16-representable
    X[6, :] = 0.1    # constant, not fp16-representable
    check_quant_bound(o.quantize_groups, bits, X)


@pytest.mark.parametrize("bits", [2, 4])
def test_quant_exact_grid(bits):
    """x = z + k*s with fp16 s, z and every code present: quantization returns
    exactly (k, s, z) and the reconstruction is exact."""
    qmax = (1 << bits) - 1
    r = _rng(10 + bits)
    for s_val, z_val in [(0.0625, -1.5), (0.5, 3.0), (2.0 ** -10, 0.0), (3.0, -100.0)]:
        k = r.integers(0, qmax + 1, size=128)
        k[0], k[1] = 0, qmax
        x = (np.float64(z_val) + k * np.float64(s_val)).astype(np.float32)
        q, s, z = o.quantize_group(x, bits)
        assert float(s) == s_val and float(z) == z_val
        assert np.array_equal(q, k.astype(np.uint8))
        assert np.array_equal(o.dequantize_value(q, s, z), x.astype(np.float64))


def test_quant_degenerate_groups():
    q, s, z = o.quantize_group(np.full(128, 0.25, np.float32), 4)
    assert float(s) == 0.0 and float(z) == 0.25 and not q.any()
    q, s, z = o.quantize_group(np.full(128, 0.1, np.float32), 2)
    assert float(z) <= 0.1 and float(s) > 0
    err = np.abs(o.dequantize_value(q, s, z) - np.float64(np.float32(0.1)))
    assert err.max() <= float(s) / 2 + 1e-12


def test_quant_rejects_nonfinite():
    x = np.zeros(128, np.float32)
    x[3] = np.nan
    with pytest.raises(o.OracleError):
        o.quantize_group(x, 4)
    x[3] = 1e6  # range overflows fp16 scale for INT2? (1e6/3 > 65504)
    with pytest.raises(o.OracleError):
        o.quantize_group(x, 2)


# ---------------------------------------------------------------------------
# Packed layout
# ---------------------------------------------------------------------------

def _pack_fixture():
    rows = []
    for line in open(os.path.join(GOLDEN, "pack_layout.txt")):
        if line.startswith("#") or not line.strip():
            continue
        b, r, c, code, off, byte = line.split()
        rows.append((int(b), int(r), int(c), int(code), int(off), int(byte, 16)))
    return rows


def check_pack_golden(pack_rows):
    for bits, r, c, code, off, byte in _pack_fixture():
        m = np.zeros((128, 128), np.uint8)
        m[r, c] = code
        blob = pack_rows(m, bits)
        assert blob.size == 128 * 128 * bits // 8
        nz = np.nonzero(blob)[0]
        assert list(nz) == [off], (bits, r, c, list(nz))
        assert blob[off] == byte


def test_pack_golden():
    check_pack_golden(o.pack_rows)


@pytest.mark.parametrize("bits", [2, 4])
def test_pack_roundtrip(bits):
    m = _rng(bits).integers(0, 1 << bits, size=(128, 128)).astype(np.uint8)
    blob = o.pack_rows(m, bits)
    assert np.array_equal(o.unpack_rows(blob, bits), m)


def test_cache_orientation_and_pages():
    """A K code (token t, channel d) is row t col d; a V code is row d col t;
    contiguous block j of sequence b is page b*max_blocks + j; a page table
    redirects it."""
    B, Hkv, L = 2, 2, 300
    x = np.zeros((B, Hkv, L, 128), np.float32)
    x[1, 1, 130, 7] = 1.0   # block 1, token 2 within the block
    lens = np.array([L, L])
    for which in (o.K_CACHE, o.V_CACHE):
        codes, s, z = o.pack_cache(x, lens, 4, o.CHANNELWISE, which)
        page = 1 * 3 + 1
        rows = o.unpack_rows(codes[page, 1], 4)
        r, c = (2, 7) if which == o.K_CACHE else (7, 2)
        assert rows[r, c] == 15 and rows.sum() == 15
        assert np.count_nonzero(codes) == 1
        pt = np.array([[5, 0, 3], [4, 2, 1]])
        codes2, _, _ = o.pack_cache(x, lens, 4, o.CHANNELWISE, which, page_table=pt, num_pages=6)
        assert np.array_equal(codes2[2], codes[page])


# ---------------------------------------------------------------------------
# Operand bit placement (format facts the pages state; checked from the
# format definitions and against torch's float8_e4m3fn decoder)
# ---------------------------------------------------------------------------

def _decode_e2m1(n):
    sgn = -1.0 if n & 8 else 1.0
    e = (n >> 1) & 3
    m = n & 1
    return sgn * (m / 2.0 if e == 0 else (1 + m / 2.0) * 2.0 ** (e - 1))


def _decode_e4m3(byte):
    sgn = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 7
    return sgn * (m / 8.0 * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7))


def test_operand_bit_placement():
    for line in open(os.path.join(GOLDEN, "operand_bit_placement.txt")):
        if line.startswith("#") or not line.strip():
            continue
        fmt, bits_hex, val = line.split()
        n = int(bits_hex, 16)
        dec = _decode_e2m1(n) if fmt == "e2m1" else _decode_e4m3(n)
        assert dec == float(val)
    for q in range(4):
        assert _decode_e2m1(q) == q / 2.0
    lib = torch.arange(16, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for q in range(16):
        assert _decode_e4m3(q) == q * 2.0 ** -9 == float(lib[q])


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def _random_problem(seed, B=2, Hkv=2, G=4, L=300, lens=None):
    r = _rng(seed)
    q = o.bf16_bits_to_f64(_bf16_bits(r.standard_normal((B, Hkv * G, 128))))
    kh = r.standard_normal((B, Hkv, L, 128)) * (1 + 4 * np.abs(r.standard_normal(128)))
    vh = r.standard_normal((B, Hkv, L, 128))
    lens = np.array(lens if lens is not None else [L] * B)
    for b in range(B):
        kh[b, :, lens[b]:] = 0
        vh[b, :, lens[b]:] = 0
    return q, kh, vh, lens


def check_attend_vs_sdpa(attend):
    """Against torch's scaled_dot_product_attention (fp64, CPU) with KV heads
    expanded for GQA and a key-padding mask for ragged lengths."""
    q, kh, vh, lens = _random_problem(1, lens=[300, 77])
    out, lse = attend(q, kh, vh, lens)
    G = q.shape[1] // kh.shape[1]
    K = torch.tensor(kh).repeat_interleave(G, dim=1)
    V = torch.tensor(vh).repeat_interleave(G, dim=1)
    Q = torch.tensor(q)[:, :, None, :]
    mask = torch.arange(kh.shape[2])[None, :] < torch.tensor(lens)[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q, K, V, attn_mask=mask[:, None, None, :])[:, :, 0].numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12), np.abs(out - ref).max()


def test_attend_vs_library_sdpa():
    check_attend_vs_sdpa(o.attend)


def test_attend_brute_force_tiny():
    """Pure-Python loops with math.exp on a tiny GQA problem."""
    r = _rng(2)
    B, Hkv, G, L, D = 1, 2, 2, 3, 128
    q = r.standard_normal((B, Hkv * G, D))
    kh = r.standard_normal((B, Hkv, L, D))
    vh = r.standard_normal((B, Hkv, L, D))
    out, lse = o.attend(q, kh, vh, [L], sm_scale=0.3)
    for h in range(Hkv * G):
        kv = h // G
        sc = [0.3 * sum(q[0, h, d] * kh[0, kv, l, d] for d in range(D)) for l in range(L)]
        w = [math.exp(x) for x in sc]
        tot = sum(w)
        assert abs(lse[0, h] - math.log(tot)) < 1e-12
        for d in range(D):
            ref = sum(w[l] * vh[0, kv, l, d] for l in range(L)) / tot
            assert abs(out[0, h, d] - ref) < 1e-12


def test_attend_closed_forms():
    q, kh, vh, _ = _random_problem(3, B=1, Hkv=1, L=64)
    sc = 1 / math.sqrt(128)
    # one token: out = v0, lse = S0
    out, lse = o.attend(q, kh, vh, [1])
    assert np.allclose(out[0], vh[0, 0, 0][None], rtol=0, atol=1e-13)
    assert np.allclose(lse[0], sc * (q[0] @ kh[0, 0, 0]), rtol=1e-13)
    # identical keys: uniform weights, lse = S + ln L
    kh2 = np.broadcast_to(kh[:, :, :1], kh.shape).copy()
    out, lse = o.attend(q, kh2, vh, [64])
    assert np.allclose(out[0], vh[0, 0].mean(axis=0)[None], atol=1e-13)
    assert np.allclose(lse[0], sc * (q[0] @ kh[0, 0, 0]) + math.log(64), rtol=1e-13)
    # empty sequence
    out, lse = o.attend(q, kh, vh, [0])
    assert not out.any() and np.all(lse == -np.inf)
    # one dominant key picks its value
    kh3 = kh.copy()
    kh3[0, 0, 5] = 400 * q[0, 0] / np.linalg.norm(q[0, 0])
    out, _ = o.attend(q, kh3, vh, [64])
    assert np.allclose(out[0, 0], vh[0, 0, 5], atol=1e-6)


# ---------------------------------------------------------------------------
# Affine folding equals dequantize-then-attend (exact-arithmetic claim)
# ---------------------------------------------------------------------------

def _packed_problem(seed, bits, kcw, vcw, lens, Hkv=2, G=4):
    r = _rng(seed)
    B, L = len(lens), max(lens)
    k = (r.standard_normal((B, Hkv, L, 128)) * (1 + 4 * np.abs(r.standard_normal(128)))).astype(np.float32)
    v = r.standard_normal((B, Hkv, L, 128)).astype(np.float32)
    qb = _bf16_bits(r.standard_normal((B, Hkv * G, 128)))
    res = o.reference_decode(qb, k, v, np.array(lens), bits, kcw, vcw)
    kc = o.unpack_cache(res["k_codes"], res["k_scale"], res["k_zero"], lens, bits, o.K_CACHE, L)
    vc = o.unpack_cache(res["v_codes"], res["v_scale"], res["v_zero"], lens, bits, o.V_CACHE, L)
    return res, kc, vc


def check_folded(attend_folded, bits, kcw, vcw):
    lens = [300, 129, 1]
    res, kc, vc = _packed_problem(7 + bits, bits, kcw, vcw, lens)
    out, lse = attend_folded(res["q"], *kc, *vc, np.array(lens), kcw, vcw)
    scale = np.abs(res["out"]).max()
    assert np.abs(out - res["out"]).max() <= 1e-12 * scale
    assert np.abs(lse - res["lse"]).max() <= 1e-12 * np.abs(res["lse"]).max()


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kcw", [0, 1])
@pytest.mark.parametrize("vcw", [0, 1])
def test_folded_equals_dequantized(bits, kcw, vcw):
    check_folded(o.attend_folded, bits, kcw, vcw)


def test_dequantized_cache_within_bound():
    """The packed-and-read-back cache reproduces every valid input within the
    quantizer bound, for all schemes (pins pack_cache/unpack_cache/dequantize
    as a chain)."""
    lens = [300, 129]
    r = _rng(5)
    x = (r.standard_normal((2, 2, 300, 128)) * 3).astype(np.float32)
    for bits in (2, 4):
        for scheme in (0, 1):
            for which in (0, 1):
                codes, s, z = o.pack_cache(x, lens, bits, scheme, which)
                c, ss, zz = o.unpack_cache(codes, s, z, lens, bits, which, 300)
                xh = o.dequantize(c, ss, zz, lens, scheme)
                for b, n in enumerate(lens):
                    err = np.abs(xh[b, :, :n] - x[b, :, :n])
                    # largest fp16 scale over the valid groups bounds the error
                    assert err.max() <= float(np.abs(s).max()) / 2 * (1 + 1e-6) + 1e-6


# ---------------------------------------------------------------------------
# Split-KV merge
# ---------------------------------------------------------------------------

def check_merge(merge, attend):
    q, kh, vh, _ = _random_problem(9, B=1, Hkv=2, L=500)
    full_o, full_l = attend(q, kh, vh, [500])
    cuts = [0, 37, 128, 129, 400, 500]
    parts_o, parts_l = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        po, pl = attend(q, kh[:, :, a:b], vh[:, :, a:b], [b - a])
        parts_o.append(po[0])
        parts_l.append(pl[0])
    parts_o.append(np.zeros_like(parts_o[0]))          # an empty split
    parts_l.append(np.full_like(parts_l[0], -np.inf))
    O = np.stack(parts_o, axis=1)
    Lp = np.stack(parts_l, axis=1)
    mo, ml = merge(O, Lp)
    assert np.allclose(mo, full_o[0], rtol=1e-12, atol=1e-13)
    assert np.allclose(ml, full_l[0], rtol=1e-12, atol=0)


def test_merge_split_invariance():
    check_merge(o.merge, o.attend)


def test_merge_all_empty():
    mo, ml = o.merge(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf))
    assert not mo.any() and np.all(ml == -np.inf)


# ---------------------------------------------------------------------------
# Mutation tests: a plausible mistake in the oracle must trip a pin
# ---------------------------------------------------------------------------

def test_mutation_gqa_mapping_caught():
    def attend_wrong(q, kh, vh, lens, sm_scale=None):
        Hkv = kh.shape[1]
        G = q.shape[1] // Hkv
        perm = np.array([(h % Hkv) * G + h // Hkv for h in range(q.shape[1])])
        return o.attend(q[:, perm], kh, vh, lens, sm_scale)
    with pytest.raises(AssertionError):
        check_attend_vs_sdpa(attend_wrong)


def test_mutation_missing_scale_caught():
    def attend_wrong(q, kh, vh, lens, sm_scale=None):
        return o.attend(q, kh, vh, lens, 1.0)
    with pytest.raises(AssertionError):
        check_attend_vs_sdpa(attend_wrong)


def test_mutation_transposed_v_caught():
    def attend_wrong(q, kh, vh, lens, sm_scale=None):
        return o.attend(q, kh, vh[:, :, ::-1], lens, sm_scale)
    with pytest.raises(AssertionError):
        check_attend_vs_sdpa(attend_wrong)


def test_mutation_dropped_offset_caught():
    def quant_wrong(X, bits):
        q, s, z = o.quantize_groups(X, bits)
        return q, s, np.zeros_like(z)
    X = _rng(0).standard_normal((64, 128)).astype(np.float32) + 3
    with pytest.raises(AssertionError):
        check_quant_bound(quant_wrong, 4, X)


def test_mutation_rounding_direction_caught():
    def quant_wrong(X, bits):  # floor instead of round-to-nearest
        q, s, z = o.quantize_groups(X, bits)
        t = (X - z.astype(np.float32)[:, None]) / np.where(s > 0, s, 1).astype(np.float32)[:, None]
        return np.clip(np.floor(t), 0, (1 << bits) - 1).astype(np.uint8), s, z
    X = _rng(1).standard_normal((64, 128)).astype(np.float32)
    with pytest.raises(AssertionError):
        check_quant_bound(quant_wrong, 4, X)


def test_mutation_nibble_order_caught():
    def pack_wrong(rows, bits):
        blob = o.pack_rows(rows, bits)
        if bits == 4:
            return ((blob >> 4) | (blob << 4)).astype(np.uint8)
        return blob
    with pytest.raises(AssertionError):
        check_pack_golden(pack_wrong)


def test_mutation_folded_vtok_offset_dropped_caught():
    def folded_wrong(q, kc, ks, kz, vc, vs, vz, lens, kcw, vcw, sm_scale=None):
        return o.attend_folded(q, kc, ks, kz, vc, vs, np.zeros_like(vz), lens, kcw, vcw, sm_scale)
    with pytest.raises(AssertionError):
        check_folded(folded_wrong, 4, 0, 0)


def test_mutation_folded_kchan_group_index_caught():
    def folded_wrong(q, kc, ks, kz, vc, vs, vz, lens, kcw, vcw, sm_scale=None):
        ks2 = ks.copy()
        ks2[:, :, 1:] = ks[:, :, :-1]   # group g uses the scales of group g-1
        return o.attend_folded(q, kc, ks2, kz, vc, vs, vz, lens, kcw, vcw, sm_scale)
    with pytest.raises(AssertionError):
        check_folded(folded_wrong, 2, 1, 0)


def test_mutation_merge_weights_caught():
    def merge_wrong(O, Lp):
        return o.merge(O, np.where(np.isfinite(Lp), 0.0, Lp))  # equal weights
    with pytest.raises(AssertionError):
        check_merge(merge_wrong, o.attend)
