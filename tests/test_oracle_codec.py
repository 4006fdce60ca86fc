"""Pins for the oracle's companding and group quantization.

What the FlashOptim page fixes (section "带压缩扩展的优化器状态量化",
companded optimizer-state quantization; Algorithms 2-3, Fig. 4):
  * phi_m(x) = 2x/(1+|x|), phi_m^-1(z) = z/(2-|z|); phi_v(x) = sqrt(x), phi_v^-1(z) = z^2;
  * groups of G = 32, one FP16 scale per group; momentum INT8, variance UINT8;
  * companding lowers the quantization error, a little for m and a lot for v
    (Fig. 4, against plain group-wise linear quantization: the linear kinds).
"""
import numpy as np
import pytest

M, V, ML, VL = 0, 1, 2, 3   # companded m, v; linear (no companding) m, v
ULP = 2.0 ** -23


def test_phi_closed_forms(orc):
    assert orc.phi_m(0.0) == 0.0
    assert orc.phi_m(1.0) == 1.0 and orc.phi_m(-1.0) == -1.0
    assert orc.phi_m(3.0) == 1.5 and orc.phi_m_inv(1.5) == 3.0
    assert orc.phi_m_inv(1.0) == 1.0 and orc.phi_m_inv(-1.0) == -1.0
    assert orc.phi_m(1e30) == 2.0          # |phi_m| < 2, reached only in the limit
    assert orc.phi_v(4.0) == 2.0 and orc.phi_v_inv(3.0) == 9.0
    assert orc.phi_v(0.0) == 0.0 and orc.phi_v_inv(0.0) == 0.0


def test_phi_m_odd_and_monotone(orc):
    x = np.sort(np.concatenate([np.geomspace(1e-30, 1e6, 20001), [0.0]])).astype(np.float32)
    z = orc.phi_n(x, "phi_m")
    assert np.array_equal(orc.phi_n(-x, "phi_m"), -z)
    assert np.all(np.diff(z.astype(np.float64)) >= 0)
    assert np.all(np.abs(z) <= 2.0)


def test_round_trips(orc):
    x = np.geomspace(1e-30, 1e3, 200001).astype(np.float32)
    x = np.concatenate([x, -x])
    back = orc.phi_n(orc.phi_n(x, "phi_m"), "phi_m_inv").astype(np.float64)
    # d phi_m^-1 / dz relative condition number at z = phi_m(x) is 1 + |x|: the
    # two roundings of phi_m and two of phi_m^-1 grow by at most that factor
    rel = np.abs(back - x) / np.abs(x)
    assert np.all(rel <= 4 * ULP * (1 + np.abs(x)))
    assert np.all(rel[np.abs(x) <= 1] <= 8 * ULP)
    xv = np.geomspace(1e-30, 1e30, 200001).astype(np.float32)
    backv = orc.phi_n(orc.phi_n(xv, "phi_v"), "phi_v_inv").astype(np.float64)
    assert np.all(np.abs(backv - xv) / xv <= 3 * ULP)


def test_zero_group(orc):
    for kind in (M, V):
        q, s = orc.quant_state(np.zeros(70, np.float32), kind)
        assert not q.any() and not s.any() and s.size == 3
        assert not orc.dequant_state(q, s, kind).any()


def test_constant_group_uses_full_range(orc):
    for c in (1e-3, 0.5, 7.0):
        q, s = orc.quant_state(np.full(32, c, np.float32), M)
        assert np.all(q == 127)
        q, s = orc.quant_state(np.full(32, -c, np.float32), M)
        assert np.all(q == -127)
        q, s = orc.quant_state(np.full(32, c, np.float32), V)
        assert np.all(q == 255)


def test_scale_is_fp16_of_group_absmax(orc):
    rng = np.random.default_rng(5)
    x = (rng.standard_t(3, 32 * 500) * 1e-3).astype(np.float32)
    q, s = orc.quant_state(x, M)
    z = orc.phi_n(x, "phi_m").reshape(-1, 32)
    assert np.array_equal(s, np.abs(z).max(1).astype(np.float16).view(np.uint16))
    v = (x * x).astype(np.float32)
    q, s = orc.quant_state(v, V)
    r = orc.phi_n(v, "phi_v").reshape(-1, 32)
    assert np.array_equal(s, r.max(1).astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("kind", [M, V])
def test_group_error_bound(orc, kind):
    """In the companded domain each code is within half a level (s/254 for m,
    s/510 for v) of the value, plus the rounding of the FP16 scale and of FP32."""
    rng = np.random.default_rng(9)
    n = 32 * 4000
    x = (rng.standard_t(3, n) * np.exp(rng.uniform(-12, 0, n))).astype(np.float32)
    if kind == V:
        x = (x * x).astype(np.float32)
    q, s = orc.quant_state(x, kind)
    levels = 127 if kind == M else 255
    sf = s.view(np.float16).astype(np.float64).repeat(32)[:n]
    c = orc.phi_n(x, "phi_m" if kind == M else "phi_v").astype(np.float64)
    chat = q.astype(np.float64) * (sf / levels)
    a = np.abs(c).reshape(-1, 32).max(1).repeat(32)
    # clamping costs at most |a - s| when the FP16 scale rounded below the absmax
    bound = sf / (2 * levels) * (1 + 1e-6) + np.maximum(a - sf, 0) + 4 * ULP * np.maximum(a, sf)
    assert np.all(np.abs(chat - c) <= bound)


@pytest.mark.parametrize("kind", [M, V])
def test_requantizing_decoded_codes_is_exact(orc, kind):
    """For many scales s and every code q: quant(dequant(q, s)) == q when the
    group also holds the top code, so that its recomputed scale is s again."""
    levels = 127 if kind == M else 255
    codes = np.arange(-127, 128) if kind == M else np.arange(0, 256)
    scales = np.float16([2.0 ** -20, 3e-6, 6.1e-5, 1e-3, 0.0371, 0.5, 1.0, 1.5]).view(np.uint16)
    for s in scales:
        groups = []
        for start in range(0, codes.size, 31):
            chunk = codes[start:start + 31]
            groups.append(np.concatenate([[levels], chunk, np.full(31 - chunk.size, levels)]))
        qin = np.concatenate(groups).astype(np.int8 if kind == M else np.uint8)
        sin = np.full(qin.size // 32, s, np.uint16)
        x = orc.dequant_state(qin, sin, kind)
        q2, s2 = orc.quant_state(x, kind)
        assert np.array_equal(s2, sin), hex(s)
        assert np.array_equal(q2, qin), hex(s)


def test_tail_group_and_group_independence(orc):
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(1000) * 1e-2).astype(np.float32)   # 31 full groups + 8
    for kind, xx in ((M, x), (V, x * x)):
        q, s = orc.quant_state(xx, kind)
        assert s.size == 32
        qa, sa = orc.quant_state(xx[:992], kind)
        qb, sb = orc.quant_state(xx[992:], kind)
        assert np.array_equal(q, np.concatenate([qa, qb])) and np.array_equal(s, np.concatenate([sa, sb]))
        # the tail scale covers only the 8 real elements
        assert s[-1] == sb[0]


def _nmse(a, b):
    return float(np.sum((a - b) ** 2) / np.sum(a ** 2))


def test_companding_reduces_error_more_for_variance(orc):
    """Fig. 4 (qualitative): against plain linear group quantization with the
    same code budget, companding helps m a little and v a lot."""
    rng = np.random.default_rng(4)
    n = 32 * 20000
    g = rng.standard_t(3, n) * 1e-4
    m = (0.1 * g).astype(np.float32)
    v = (1e-3 * g * g).astype(np.float32)

    def linear(x, levels, signed):
        # the same storage format: one FP16 scale per group of 32
        xg = x.astype(np.float64).reshape(-1, 32)
        s = _fp16_values(np.minimum(np.abs(xg).max(1, keepdims=True), 65504.0))
        with np.errstate(divide="ignore", invalid="ignore"):
            q = np.where(s > 0, np.clip(np.rint(xg / s * levels), -levels if signed else 0, levels), 0)
        return (q * s / levels).ravel()

    qm, sm = orc.quant_state(m, M)
    qv, sv = orc.quant_state(v, V)
    e_m_comp = _nmse(m.astype(np.float64), orc.dequant_state(qm, sm, M).astype(np.float64))
    e_v_comp = _nmse(v.astype(np.float64), orc.dequant_state(qv, sv, V).astype(np.float64))
    e_m_lin = _nmse(m.astype(np.float64), linear(m, 127, True))
    e_v_lin = _nmse(v.astype(np.float64), linear(v, 255, False))
    assert e_m_comp <= e_m_lin * 1.05
    assert e_v_comp < e_v_lin / 4
    # the oracle's linear kinds are the same quantizer (FP16 scales, FP32 steps)
    for x, kind, ref in ((m, ML, e_m_lin), (v, VL, e_v_lin)):
        q, s = orc.quant_state(x, kind)
        e = _nmse(x.astype(np.float64), orc.dequant_state(q, s, kind).astype(np.float64))
        assert abs(e - ref) <= 0.01 * ref


def _fp16_values(x):
    return np.asarray(x, np.float64).astype(np.float16).astype(np.float64)


@pytest.mark.parametrize("kind,levels", [(ML, 127), (VL, 255)])
def test_linear_codes_on_an_exact_grid(orc, kind, levels):
    """Values k*s/L with s an FP16 value and the group maximum equal to s:
    the linear codec returns k itself, and decodes to k * RN(s/L)."""
    s = 0.375
    ks = np.arange(-127, 128) if levels == 127 else np.arange(0, 256)
    ks = np.concatenate([ks, np.full((-len(ks)) % 32, ks[-1])])   # whole groups, max = s
    x = (ks * (s / levels)).astype(np.float32)
    x[31::32] = np.float32(s)
    q, sc = orc.quant_state(x, kind)
    assert np.all(orc.fp16_to_f32_n(sc) == s)
    want = ks.copy()
    want[31::32] = levels
    assert np.array_equal(q.astype(np.int64), want)
    d = orc.dequant_state(q, sc, kind)
    assert np.array_equal(d, (q.astype(np.float32) * np.float32(np.float32(s) / np.float32(levels))))


@pytest.mark.parametrize("kind,levels,signed", [(ML, 127, True), (VL, 255, False)])
def test_linear_codec_matches_its_float64_definition(orc, kind, levels, signed):
    """scale = FP16(max |x|); code = clamp(rint(x * L / scale)); the FP32 steps of
    the oracle differ from the float64 definition only at rounding ties."""
    rng = np.random.default_rng(31)
    g = rng.standard_t(3, 32 * 4096) * 10.0 ** rng.uniform(-8, 2, 32 * 4096).repeat(1)
    x = (g if signed else g * g).astype(np.float32)
    q, sc = orc.quant_state(x, kind)
    xg = x.astype(np.float64).reshape(-1, 32)
    s64 = _fp16_values(np.minimum(np.abs(xg).max(1), 65504.0))   # the scale is capped at FP16's max
    assert np.array_equal(orc.fp16_to_f32_n(sc).astype(np.float64), s64)
    with np.errstate(divide="ignore", invalid="ignore"):
        c64 = np.where(s64[:, None] > 0, np.rint(xg * (levels / s64[:, None])), 0)
    c64 = np.clip(c64, -levels if signed else 0, levels).ravel()
    d = q.astype(np.int64) - c64.astype(np.int64)
    assert np.abs(d).max() <= 1 and np.count_nonzero(d) <= 1e-4 * x.size
    # and where the scale is a normal FP16 value below the cap, every element
    # lies within half a step of its decoded value (capped groups saturate,
    # subnormal scales may fall below the group maximum)
    xh = orc.dequant_state(q, sc, kind).astype(np.float64).reshape(-1, 32)
    step = s64[:, None] / levels
    honest = (s64 >= 2.0 ** -14) & (np.abs(xg).max(1) <= 65504.0)
    assert honest.mean() > 0.5
    ok = np.abs(xh - xg) <= 0.5 * step * (1 + 2.0 ** -10) + np.abs(xg) * 2.0 ** -22
    assert np.all(ok[honest])


VNZ = 5   # companded v with the opt-in rule: no code 0 in a group with a non-zero scale


def test_nonzero_variance_codec_differs_only_at_zero_codes(orc):
    """The opt-in rule moves exactly the codes 0 of groups with a non-zero
    scale up to 1 (every decoded v there is then at least (s/255)^2); scales,
    all other codes and groups with a zero scale are the plain codec's."""
    rng = np.random.default_rng(51)
    g = rng.standard_t(2, 32 * 8192)
    v = (g * g).astype(np.float32)
    v[::97] = 0.0
    v[:32] = 0.0                                  # a group with scale 0
    v[32:64] = 1e-40                              # its scale rounds to 0 in FP16
    q0, s0 = orc.quant_state(v, V)
    q1, s1 = orc.quant_state(v, VNZ)
    assert np.array_equal(s0, s1)
    live = np.repeat(s0 != 0, 32)
    moved = q0 != q1
    assert moved.sum() > 100                     # heavy tails put many elements below s/510
    assert np.array_equal(moved, live & (q0 == 0))
    assert np.all(q1[moved] == 1) and np.all(q1[~live] == 0)
    d = orc.dequant_state(q1, s1, VNZ)
    sv = orc.fp16_to_f32_n(s1).astype(np.float64)
    floor = np.repeat((sv / 255) ** 2, 32)
    assert np.all(d[live] >= floor[live] * (1 - 2.0 ** -20)) and np.all(d[~live] == 0)
    # decoding is the plain codec's
    assert np.array_equal(d, orc.dequant_state(q1, s1, V))
