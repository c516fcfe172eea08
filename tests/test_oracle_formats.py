"""Pins for the oracle's number-format helpers and its operand-rounding
emulation, each against something other than the oracle itself:

  * ``kvq_oracle.bf16_bits_to_f64`` (turns every query bit pattern into the
    fp64 q the oracle attends with) -- all 65,536 patterns against PyTorch's
    own bfloat16 decoder, plus hand-decoded patterns from the bfloat16 format
    definition (1 sign, 8 exponent bits with bias 127, 7 fraction bits);
  * ``emulate.round_e4m3`` / ``emulate.round_bf16`` -- against PyTorch's
    float8_e4m3fn and bfloat16 casts (round to nearest, ties to even) on
    every representable value, every exact midpoint between neighbours,
    the subnormal range, zero and random values; saturation at +-448 from the
    E4M3 format definition (the largest finite E4M3 value);
  * ``emulate.split`` / ``emulate.pow2_scale`` -- closed cases: a value with
    at most 12 significant bits is the exact sum of its three E4M3 parts (16
    bits: two BF16 parts); the power-of-two scale brackets [128, 256);
  * ``emulate.attend_emulated`` -- with enough BF16 parts the rounded operands
    become exact, so it must reproduce the oracle's direct attention.

The mutation tests plant a plausible mistake in each helper and check that a
pin catches it.
"""
import numpy as np
import pytest
import torch

from oracle import emulate as em
from oracle import kvq_oracle as o


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# bf16 bit patterns -> fp64
# ---------------------------------------------------------------------------

def check_bf16_decoder(fn):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):  # NaN patterns
        got = np.asarray(fn(bits), np.float64)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))  # -0.0 stays negative
    # hand-decoded from the format definition
    hand = {0x3F80: 1.0, 0xC000: -2.0, 0x4049: 3.140625, 0x0000: 0.0, 0x0001: 2.0 ** -133,
            0x007F: 127 * 2.0 ** -133, 0x0080: 2.0 ** -126, 0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127,
            0x7F80: np.inf, 0xFF80: -np.inf, 0x3C00: 2.0 ** -7, 0xBE80: -0.25}
    for b, v in hand.items():
        assert float(fn(np.array([b], np.uint16))[0]) == v, hex(b)
    assert np.isnan(fn(np.array([0x7FC0], np.uint16))[0])


def test_bf16_bits_to_f64_exhaustive():
    check_bf16_decoder(o.bf16_bits_to_f64)


def test_mutation_bf16_wrong_shift_caught():
    def wrong(bits):
        b = np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(15)
        with np.errstate(invalid="ignore"):
            return b.view(np.float32).astype(np.float64)
    with pytest.raises(AssertionError):
        check_bf16_decoder(wrong)


def test_mutation_bf16_dropped_sign_caught():
    def wrong(bits):
        return np.abs(o.bf16_bits_to_f64(bits))
    with pytest.raises(AssertionError):
        check_bf16_decoder(wrong)


# ---------------------------------------------------------------------------
# E4M3 and BF16 rounding against PyTorch's casts
# ---------------------------------------------------------------------------

def _e4m3_values():
    """Every finite E4M3 value, decoded by PyTorch (sorted, unique, >= 0)."""
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    b = b[np.isfinite(b)]
    return np.unique(np.abs(b))


def _e4m3_probe_points():
    v = _e4m3_values()                        # 0, 2^-9 ... 448
    mids = (v[:-1] + v[1:]) / 2               # exact ties (5 significant bits: exact in fp32)
    quarter = v[:-1] + (v[1:] - v[:-1]) / 4   # off-tie points on either side
    three_q = v[:-1] + 3 * (v[1:] - v[:-1]) / 4
    r = _rng(3)
    rnd = np.exp(r.uniform(np.log(2.0 ** -12), np.log(448.0), 20000))
    pos = np.concatenate([v, mids, quarter, three_q, rnd, [2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11]])
    pos = pos.astype(np.float32).astype(np.float64)  # torch casts from fp32
    return np.concatenate([pos, -pos])


def check_round_e4m3(fn):
    x = _e4m3_probe_points()
    got = np.asarray(fn(x), np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(got, ref), float(np.abs(got - ref).max())
    # saturation (the largest finite E4M3 value is 448 = 1.75 * 2^8)
    big = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e6, -449.0, -1e9])
    assert np.array_equal(np.asarray(fn(big)), np.sign(big) * 448.0)
    assert float(fn(np.array([0.0]))[0]) == 0.0


def test_round_e4m3_matches_torch_and_saturates():
    check_round_e4m3(em.round_e4m3)


def test_mutation_e4m3_round_half_up_caught():
    def wrong(x):
        x = np.asarray(x, np.float64)
        a = np.abs(x)
        _, e = np.frexp(a)
        q = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
        return np.sign(x) * np.minimum(np.floor(a / q + 0.5) * q, 448.0)
    with pytest.raises(AssertionError):
        check_round_e4m3(wrong)


def test_mutation_e4m3_no_subnormals_caught():
    def wrong(x):  # flushes below the smallest normal (2^-6) to zero
        r = em.round_e4m3(x)
        return np.where(np.abs(r) < 2.0 ** -6, 0.0, r)
    with pytest.raises(AssertionError):
        check_round_e4m3(wrong)


def check_round_bf16(fn):
    r = _rng(4)
    v = torch.arange(0, 0x7F80, 7, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double().numpy()
    nxt = v + np.abs(v) * 2.0 ** -8 * 1.0  # roughly next neighbour (exact midpoints below)
    bits = torch.arange(0, 0x7F7F, 5, dtype=torch.int32)
    lo = bits.to(torch.int16).view(torch.bfloat16).double().numpy()
    hi = (bits + 1).to(torch.int16).view(torch.bfloat16).double().numpy()
    mids = (lo + hi) / 2                                   # exact ties, representable in fp32
    rnd = np.concatenate([r.standard_normal(20000) * 10.0 ** r.integers(-30, 30, 20000),
                          np.exp(r.uniform(np.log(1e-40), np.log(1e-36), 2000))])  # bf16 subnormals
    x = np.concatenate([v, nxt, mids, rnd, [0.0]]).astype(np.float32).astype(np.float64)
    x = np.concatenate([x, -x])
    got = np.asarray(fn(x), np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, ref), float(np.abs(got - ref).max())


def test_round_bf16_matches_torch():
    check_round_bf16(em.round_bf16)


def test_mutation_bf16_truncation_caught():
    def wrong(x):  # round toward zero
        x = np.asarray(x, np.float64)
        a = np.abs(x)
        _, e = np.frexp(a)
        q = np.ldexp(1.0, np.maximum(e - 1, -126) - 7)
        return np.sign(x) * np.floor(a / q) * q
    with pytest.raises(AssertionError):
        check_round_bf16(wrong)


# ---------------------------------------------------------------------------
# Operand splits and the power-of-two prescale
# ---------------------------------------------------------------------------

def check_split(fn):
    r = _rng(5)
    # 12 significant bits in [128, 256): exact as three E4M3 parts
    x12 = (r.integers(2048, 4096, 5000) * 2.0 ** -4) * r.choice([-1.0, 1.0], 5000)
    assert np.array_equal(fn(x12, 3, "e4m3"), x12)
    # 16 significant bits at any exponent: exact as two BF16 parts
    x16 = r.integers(1 << 15, 1 << 16, 5000) * 2.0 ** r.integers(-60, 60, 5000).astype(np.float64)
    assert np.array_equal(fn(x16, 2, "bf16"), x16)
    # arbitrary values: each E4M3 part gains at least 4 bits (the first part
    # is within 2^-4 relative of x, the residual of the next within 2^-4 of it)
    x = r.uniform(128.0, 256.0, 5000)
    for parts, bound in ((1, 2.0 ** -4), (2, 2.0 ** -8), (3, 2.0 ** -12)):
        err = np.abs(fn(x, parts, "e4m3") - x) / np.abs(x)
        assert err.max() <= bound, (parts, err.max())
    assert not np.array_equal(fn(x, 2, "e4m3"), x)


def test_split_closed_cases():
    check_split(em.split)


def test_mutation_split_drops_last_part_caught():
    def wrong(x, parts, fmt):
        return em.split(x, max(1, parts - 1), fmt)
    with pytest.raises(AssertionError):
        check_split(wrong)


def check_pow2_scale(fn):
    r = _rng(6)
    m = np.concatenate([np.exp(r.uniform(np.log(1e-30), np.log(1e30), 20000)),
                        2.0 ** np.arange(-60, 61).astype(np.float64), [128.0, 255.999, 256.0, 1.0]])
    s = np.asarray(fn(m), np.float64)
    k = np.log2(s)
    assert np.array_equal(k, np.round(k))          # exact powers of two
    y = m * s
    assert np.all((y >= 128.0) & (y < 256.0)), (y.min(), y.max())
    assert float(fn(np.array([0.0]))[0]) == 1.0


def test_pow2_scale_brackets():
    check_pow2_scale(em.pow2_scale)


def test_mutation_pow2_scale_off_by_one_caught():
    def wrong(m):
        return em.pow2_scale(m) * 2.0
    with pytest.raises(AssertionError):
        check_pow2_scale(wrong)


# ---------------------------------------------------------------------------
# The emulated folded attention: exact when the operands are
# ---------------------------------------------------------------------------

def _logical_problem(bits, kcw, vcw, seed):
    r = _rng(seed)
    B, Hkv, G, L = 2, 2, 4, 300
    lens = np.array([300, 129])
    k = (r.standard_normal((B, Hkv, L, 128)) * (1 + 4 * np.abs(r.standard_normal(128)))).astype(np.float32)
    v = r.standard_normal((B, Hkv, L, 128)).astype(np.float32)
    q = o.bf16_bits_to_f64(torch.from_numpy(r.standard_normal((B, Hkv * G, 128)).astype(np.float32))
                           .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    kc, ks, kz = o.pack_cache(k, lens, bits, kcw, o.K_CACHE)
    vc, vs, vz = o.pack_cache(v, lens, bits, vcw, o.V_CACHE)
    K = o.unpack_cache(kc, ks, kz, lens, bits, o.K_CACHE, L)
    V = o.unpack_cache(vc, vs, vz, lens, bits, o.V_CACHE, L)
    ref = o.attend(q, o.dequantize(*K, lens, kcw), o.dequantize(*V, lens, vcw), lens)
    return q, K, V, lens, ref


def check_emulated(fn, bits, kcw, vcw):
    q, K, V, lens, (ro, rl) = _logical_problem(bits, kcw, vcw, 40 + 4 * bits + 2 * kcw + vcw)
    out, lse = fn(q, *K, *V, lens, kcw, vcw, fmt="bf16", q_splits=7, p_splits=7)
    rms = np.sqrt((ro ** 2).mean())
    assert np.abs(out - ro).max() <= 1e-11 * rms
    assert np.abs(lse - rl).max() <= 1e-11
    # the production operand splits stay within the build's FP8 tolerance
    out8, _ = fn(q, *K, *V, lens, kcw, vcw, fmt="e4m3", q_splits=3, p_splits=3)
    assert np.abs(out8 - ro).max() <= 3e-2 * rms


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kcw,vcw", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_emulated_attention_reduces_to_oracle(bits, kcw, vcw):
    check_emulated(em.attend_emulated, bits, kcw, vcw)


def test_mutation_emulated_dropped_k_offset_caught():
    def wrong(q, kc, ks, kz, vc, vs, vz, lens, kcw, vcw, **kw):
        return em.attend_emulated(q, kc, ks, np.zeros_like(kz), vc, vs, vz, lens, kcw, vcw, **kw)
    with pytest.raises(AssertionError):
        check_emulated(wrong, 4, 0, 0)


def test_mutation_emulated_v_scheme_swapped_caught():
    def wrong(q, kc, ks, kz, vc, vs, vz, lens, kcw, vcw, **kw):
        return em.attend_emulated(q, kc, ks, kz, vc, vs, vz, lens, kcw, 1 - vcw, **kw)
    with pytest.raises(AssertionError):
        check_emulated(wrong, 2, 1, 0)
