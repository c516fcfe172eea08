"""Pins for the oracle's group geometry beyond the default (head dim 64 / 256,
groups of 32 / 64 elements), each against something other than the oracle:

  * the group of each element, written out here from the definition
    (token-wise: G consecutive channels of a token; channel-wise: G
    consecutive tokens of a channel, aligned to token 0): a cache whose groups
    are each constant at a distinct fp16 value must round-trip exactly, and
    any other grouping mixes values and cannot;
  * a brute-force, element-by-element dequantization (pure Python loops over
    the stored s / z layout) against ``dequantize``;
  * the folded formulation equals dequantize-then-attend to 1e-12 for every
    geometry and scheme pair ([ABS]: the folding is exact; [SUM]
    限界と未検証の範囲: accumulator folds per quantization group);
  * the s/2 quantization bound per element with its own group's scale;
  * hand-worked packed layouts for D = 64 and 256 (tests/golden).

Mutation tests plant a wrong group axis and a wrong group index and check
that a pin catches each.
"""
import math
import os

import numpy as np
import pytest

from oracle import kvq_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GEOMETRIES = [(64, 32), (64, 64), (128, 32), (128, 64), (256, 64), (256, 128)]


def _rng(seed):
    return np.random.default_rng(seed)


def group_id(scheme, t, c, group):
    """Group of element (token t of the sequence, channel c), by definition."""
    return (t, c // group) if scheme == o.TOKENWISE else (t // group, c)


def check_constant_groups(quantize_sequence, scheme, D, G, n=300):
    ids = {}
    x = np.zeros((n, D), np.float32)
    for t in range(n):
        for c in range(D):
            gid = group_id(scheme, t, c, G)
            if gid not in ids:
                ids[gid] = len(ids)
            x[t, c] = np.float32(np.float16(1.0 + 0.25 * (ids[gid] % 4000)))  # distinct fp16 values
    codes, s, z = quantize_sequence(x, 2, scheme, G)
    nblk = o.num_blocks(n)
    xh = np.zeros((nblk * 128, D))
    for j in range(nblk):
        sv = o.expand_sz(s[None, j], scheme, D, 128)[0]
        zv = o.expand_sz(z[None, j], scheme, D, 128)[0]
        xh[j * 128:(j + 1) * 128] = sv * codes[j] + zv
    assert np.array_equal(xh[:n], x.astype(np.float64))
    assert not np.any(s.astype(np.float64))  # every group constant: s = 0


@pytest.mark.parametrize("D,G", GEOMETRIES)
@pytest.mark.parametrize("scheme", [o.TOKENWISE, o.CHANNELWISE])
def test_group_membership_from_definition(D, G, scheme):
    check_constant_groups(o.quantize_sequence, scheme, D, G)


def test_mutation_group_axis_caught():
    def wrong(x, bits, scheme, group):  # channel-wise groups taken along channels
        return o.quantize_sequence(x, bits, o.TOKENWISE if scheme == o.CHANNELWISE else o.CHANNELWISE, group)
    with pytest.raises(AssertionError):
        check_constant_groups(wrong, o.CHANNELWISE, 64, 32)


def test_mutation_group_size_caught():
    def wrong(x, bits, scheme, group):
        c, s, z = o.quantize_sequence(x, bits, scheme, group * 2 if group < 128 else 64)
        return c, s, z
    with pytest.raises(Exception):
        check_constant_groups(wrong, o.TOKENWISE, 128, 32)


@pytest.mark.parametrize("D,G", GEOMETRIES + [(128, 128)])
@pytest.mark.parametrize("scheme", [o.TOKENWISE, o.CHANNELWISE])
def test_empty_sequence_shapes(D, G, scheme):
    codes, s, z = o.quantize_sequence(np.zeros((0, D), np.float32), 2, scheme, G)
    assert codes.shape == (0, 128, D) and s.shape == (0, 128 * D // G) and z.shape == s.shape
    c, s, z = o.pack_cache(np.zeros((2, 1, 128, D), np.float32), [0, 5], 4, scheme, o.V_CACHE, group=G)
    assert c.shape == (2, 1, o.block_bytes(4, D)) and s.shape == (2, 1, 128 * D // G)
    assert not c[0].any() and not s[0].any()


def _sequence(seed, D, n=260):
    r = _rng(seed)
    return (r.standard_normal((n, D)) * (1 + 4 * np.abs(r.standard_normal(D)))).astype(np.float32)


@pytest.mark.parametrize("D,G", GEOMETRIES)
@pytest.mark.parametrize("scheme", [o.TOKENWISE, o.CHANNELWISE])
def test_dequantize_brute_force(D, G, scheme):
    x = _sequence(3, D, 200)
    codes, s, z = o.quantize_sequence(x, 4, scheme, G)
    xh = o.dequantize(codes.reshape(1, 1, -1, D)[:, :, :200], s[None, None], z[None, None], [200], scheme)[0, 0]
    for t in range(0, 200, 7):
        j, tl = divmod(t, 128)
        for c in range(0, D, 5):
            if scheme == o.TOKENWISE:
                k = tl * (D // G) + c // G
            else:
                k = (tl // G) * D + c
            ref = float(s[j, k]) * int(codes[j, tl, c]) + float(z[j, k])
            assert xh[t, c] == ref


@pytest.mark.parametrize("D,G", GEOMETRIES)
@pytest.mark.parametrize("scheme", [o.TOKENWISE, o.CHANNELWISE])
def test_quant_bound_per_group(D, G, scheme):
    x = _sequence(4, D)
    x[:, 3] += 40.0
    codes, s, z = o.quantize_sequence(x, 2, scheme, G)
    n = x.shape[0]
    nblk = o.num_blocks(n)
    for j in range(nblk):
        nv = min(128, n - 128 * j)
        sv = o.expand_sz(s[None, j], scheme, D, nv)[0]
        zv = o.expand_sz(z[None, j], scheme, D, nv)[0]
        xj = x[128 * j:128 * j + nv].astype(np.float64)
        err = np.abs(xj - (sv * codes[j, :nv] + zv))
        assert np.all(err <= sv / 2 + 2.0 ** -22 * np.abs(xj - zv))
        assert np.all(zv <= xj)


def _geometry_problem(seed, D, G, bits, kcw, vcw):
    r = _rng(seed)
    B, Hkv, Gq, L = 2, 2, 4, 300
    lens = np.array([300, 150])
    k = (r.standard_normal((B, Hkv, L, D)) * (1 + 4 * np.abs(r.standard_normal(D)))).astype(np.float32)
    v = r.standard_normal((B, Hkv, L, D)).astype(np.float32)
    qb = (r.standard_normal((B, Hkv * Gq, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q = o.bf16_bits_to_f64(qb)
    kc, ks, kz = o.pack_cache(k, lens, bits, kcw, o.K_CACHE, group=G)
    vc, vs, vz = o.pack_cache(v, lens, bits, vcw, o.V_CACHE, group=G)
    K = o.unpack_cache(kc, ks, kz, lens, bits, o.K_CACHE, L)
    V = o.unpack_cache(vc, vs, vz, lens, bits, o.V_CACHE, L)
    return q, K, V, lens


def check_folded_geometry(folded, D, G, bits, kcw, vcw):
    q, K, V, lens = _geometry_problem(10 + D + G + bits + 2 * kcw + vcw, D, G, bits, kcw, vcw)
    ref_o, ref_l = o.attend(q, o.dequantize(*K, lens, kcw), o.dequantize(*V, lens, vcw), lens)
    out, lse = folded(q, *K, *V, lens, kcw, vcw)
    assert np.abs(out - ref_o).max() <= 1e-12 * max(1.0, np.abs(ref_o).max())
    assert np.abs(lse - ref_l).max() <= 1e-12 * max(1.0, np.abs(ref_l).max())


@pytest.mark.parametrize("D,G", GEOMETRIES)
@pytest.mark.parametrize("kcw,vcw", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_folded_equals_dequantized_geometry(D, G, kcw, vcw):
    check_folded_geometry(o.attend_folded, D, G, 2 if (D + G) % 3 else 4, kcw, vcw)


def test_mutation_folded_channel_group_caught():
    def wrong(q, kc, ks, kz, vc, vs, vz, lens, kcw, vcw):
        # token-wise V: every channel group uses the scales of group 0
        vs2 = vs.copy()
        B, H, nb, m = vs.shape
        per = vs2.reshape(B, H, nb, 128, -1)
        per[..., :] = per[..., :1]
        return o.attend_folded(q, kc, ks, kz, vc, vs2, vz, lens, kcw, vcw)
    with pytest.raises(AssertionError):
        check_folded_geometry(wrong, 128, 32, 2, 0, 0)


def test_mutation_folded_token_group_caught():
    def wrong(q, kc, ks, kz, vc, vs, vz, lens, kcw, vcw):
        # channel-wise K: token group g uses the scales of group g - 1
        ks2 = ks.copy()
        B, H, nb, m = ks.shape
        per = ks2.reshape(B, H, nb, -1, q.shape[2])
        per[:, :, :, 1:] = per[:, :, :, :-1].copy()
        return o.attend_folded(q, kc, ks2, kz, vc, vs, vz, lens, kcw, vcw)
    with pytest.raises(AssertionError):
        check_folded_geometry(wrong, 64, 32, 2, 1, 0)


def _geometry_fixture():
    rows = []
    for line in open(os.path.join(GOLDEN, "pack_layout_geometry.txt")):
        if line.startswith("#") or not line.strip():
            continue
        b, w, D, r, c, code, off, byte = line.split()
        rows.append((int(b), int(w), int(D), int(r), int(c), int(code), int(off), int(byte, 16)))
    return rows


def test_pack_layout_geometry_golden():
    for bits, which, D, r, c, code, off, byte in _geometry_fixture():
        nrows, ncols = (128, D) if which == 0 else (D, 128)
        m = np.zeros((nrows, ncols), np.uint8)
        m[r, c] = code
        blob = o.pack_rows(m, bits)
        assert blob.size == o.block_bytes(bits, D)
        nz = np.nonzero(blob)[0]
        assert list(nz) == [off], (bits, which, D, r, c, list(nz))
        assert blob[off] == byte
        assert np.array_equal(o.unpack_rows(blob, bits, nrows, ncols), m)


def test_cache_orientation_geometry():
    """K code (token t, channel d) is row t col d of a D-column block; V code is
    row d col t of a D-row block; s / z entries sit where the group layout
    says."""
    D, G = 256, 64
    x = np.zeros((1, 1, 200, D), np.float32)
    x[0, 0, 130, 200] = 1.0   # block 1, token 2
    for which in (o.K_CACHE, o.V_CACHE):
        for scheme in (o.TOKENWISE, o.CHANNELWISE):
            codes, s, z = o.pack_cache(x, [200], 4, scheme, which, group=G)
            rows = o.unpack_rows(codes[1, 0], 4, 128 if which == o.K_CACHE else D, D if which == o.K_CACHE else 128)
            r, c = (2, 200) if which == o.K_CACHE else (200, 2)
            assert rows[r, c] == 15 and rows.sum() == 15
            k = 2 * (D // G) + 200 // G if scheme == o.TOKENWISE else (2 // G) * D + 200
            nz = np.nonzero(s[1, 0])[0]
            assert list(nz) == [k]
