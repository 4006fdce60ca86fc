"""Pins for the oracle's number encodings (BF16, FP16, half-ULP).

Each encoding is compared, exhaustively or densely, with an independent
library routine (torch's BF16 cast, numpy's FP16 cast) or with a closed form
computed here another way (binade exponents via math.frexp).
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore:overflow encountered in cast")


def _dense_f32(exponents, prefixes, low_bits, signs=(0, 1)):
    """FP32 bit patterns: for each biased exponent and mantissa prefix, every
    pattern of the low ``low_bits`` mantissa bits (covers all rounding cases)."""
    low = np.arange(1 << low_bits, dtype=np.uint32)
    out = []
    for s in signs:
        for e in exponents:
            for p in prefixes:
                out.append((np.uint32(s << 31) | np.uint32(e << 23) | np.uint32(p << low_bits)) | low)
    return np.concatenate(out).view(np.float32)


def test_bf16_rne_matches_torch_cast_dense(orc):
    # every low-16-bit pattern (ties, odd/even) under several prefixes and binades,
    # including FP32 subnormals (exponent 0) and the overflow edge (254)
    x = _dense_f32([0, 1, 2, 100, 126, 127, 128, 200, 253, 254], [0, 1, 0x3F, 0x7F], 16)
    ours = orc.bf16_rne_n(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_rne_matches_torch_cast_random(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ours = orc.bf16_rne_n(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_fp16_rne_matches_numpy_cast_dense(orc):
    # biased FP32 exponents 100..142 span 2^-27 .. 2^15 (FP16 subnormals, normals,
    # overflow); every low-13-bit pattern is enumerated under several prefixes
    x = _dense_f32(range(100, 143), [0, 1, 0x1FF, 0x3FF], 13)
    ours = orc.fp16_rne_n(x)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_fp16_rne_matches_numpy_cast_random(orc):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(1_000_000) * np.exp(rng.uniform(-25, 12, 1_000_000))).astype(np.float32)
    assert np.array_equal(orc.fp16_rne_n(x), x.astype(np.float16).view(np.uint16))
    edge = np.float32([65504.0, 65519.99, 65520.0, 70000.0, 2.0 ** -24, 2.0 ** -25,
                       2.0 ** -25 * 1.0001, 2.0 ** -26, 0.0, -0.0, 6.1e-5, -6.1e-5])
    assert np.array_equal(orc.fp16_rne_n(edge), edge.astype(np.float16).view(np.uint16))


def test_fp16_decode_all_patterns(orc):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.fp16_to_f32_n(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _gap_closed_form(b: int, direction: int) -> float:
    """BF16 gap next to pattern b on side direction, from the binade exponent."""
    x = np.array([b << 16], dtype=np.uint32).view(np.float32)[0]
    a = abs(float(x))
    if a < 2.0 ** -126:                      # zero or subnormal: fixed spacing
        return 2.0 ** -133
    _, e2 = math.frexp(a)
    E = e2 - 1                               # a in [2^E, 2^(E+1))
    away = (direction > 0) == (x > 0) or (x == 0)
    if away:
        return 2.0 ** (E - 7)
    is_pow2 = a == 2.0 ** E
    if is_pow2 and E > -126:
        return 2.0 ** (E - 8)                # below a power of two the gap halves
    return 2.0 ** (E - 7)


def test_half_ulp_all_finite_bf16(orc):
    pats = [b for b in range(65536) if (b & 0x7F80) != 0x7F80]   # finite patterns
    arr = np.array(pats, dtype=np.uint16)
    up = orc.half_ulp_n(arr, +1).astype(np.float64)
    dn = orc.half_ulp_n(arr, -1).astype(np.float64)
    for i, b in enumerate(pats):
        # past the largest finite BF16 the gap is that of its binade (IEEE's
        # unbounded-exponent rounding), 2^(127-7)
        assert up[i] == _gap_closed_form(b, +1) / 2, hex(b)
        assert dn[i] == _gap_closed_form(b, -1) / 2, hex(b)


def test_half_ulp_bound_examples(orc):
    # 1.0 = 0x3F80: gap above 2^-7, gap below 2^-8
    assert orc.half_ulp(0x3F80, +1) == 2.0 ** -8
    assert orc.half_ulp(0x3F80, -1) == 2.0 ** -9
    # zero: the smallest BF16 subnormal is 2^-133
    assert orc.half_ulp(0x0000, +1) == 2.0 ** -134
    assert orc.half_ulp(0x8000, -1) == 2.0 ** -134
    # smallest normal 2^-126: the subnormals below are spaced like the binade above
    assert orc.half_ulp(0x0080, -1) == 2.0 ** -134
    # largest finite BF16: the gap above is its binade's, not infinite
    assert orc.half_ulp(0x7F7F, +1) == 2.0 ** 119
    assert orc.half_ulp(0xFF7F, -1) == 2.0 ** 119
