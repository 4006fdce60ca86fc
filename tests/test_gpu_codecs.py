"""GPU parity of the stand-alone codecs (fo_split, fo_merge, fo_quant_state,
fo_dequant_state) against the CPU oracle, through the C ABI.

Weight splitting: page section "权重复分裂" (Eq. 1-2). State quantization:
section "带压缩扩展的优化器状态量化" (Algorithms 2-3).
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import fo
from tests.gpu_helpers import assert_codes, assert_exact, assert_scales, to_dev, to_host

pytestmark = pytest.mark.gpu

RAGGED = [1, 15, 16, 17, 31, 32, 33, 1000, 4095, 4097, (1 << 20) + 7]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


def _bits_range(lo, count, stride=1):
    return (np.arange(count, dtype=np.uint64) * stride + lo).astype(np.uint32).view(np.float32)


def _finite_random_f32(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.integers(0, 2 ** 32, size=2 * n, dtype=np.uint64).astype(np.uint32).view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 3.3e38)]       # BF16 rounding stays finite
    return x[:n].copy()


SPLIT_INPUTS = {
    "binade [1,2)": lambda: _bits_range(0x3F800000, 1 << 23),
    "binade [-2^-3,-2^-2)": lambda: _bits_range(0xBE000000, 1 << 23),
    "fp32 subnormals": lambda: _bits_range(0x00000001, (1 << 23) - 1),
    "smallest normals": lambda: _bits_range(0x80800000, 1 << 22, 3),
    "random patterns": lambda: _finite_random_f32(1 << 22, 1),
    "signed zeros": lambda: np.float32([0.0, -0.0] * 40),
}


def _split_gpu(theta, bits):
    x = to_dev(theta)
    tp = torch.empty(theta.size, dtype=torch.int16, device="cuda")
    rho = torch.empty(theta.size, dtype=torch.int16 if bits == 16 else torch.int8, device="cuda")
    fo.fo_split(x, tp, rho, bits)
    return to_host(tp), to_host(rho, np.int16 if bits == 16 else np.int8)


@pytest.mark.parametrize("bits", [8, 16])
@pytest.mark.parametrize("name", list(SPLIT_INPUTS))
def test_split_matches_oracle(bits, name):
    theta = SPLIT_INPUTS[name]()
    tp, rho = _split_gpu(theta, bits)
    tp_ref, rho_ref = oracle.split(theta, bits)
    assert_exact(tp, tp_ref, "theta'")
    assert_exact(rho, rho_ref, "rho")


@pytest.mark.parametrize("bits", [8, 16])
@pytest.mark.parametrize("n", RAGGED)
def test_split_merge_ragged_sizes(bits, n):
    rng = np.random.default_rng(n)
    theta = (rng.standard_normal(n) * np.exp(rng.uniform(-20, 5, n))).astype(np.float32)
    tp, rho = _split_gpu(theta, bits)
    tp_ref, rho_ref = oracle.split(theta, bits)
    assert_exact(tp, tp_ref, "theta'")
    assert_exact(rho, rho_ref, "rho")
    out = torch.full((n,), float("nan"), device="cuda")
    fo.fo_merge(to_dev(tp), to_dev(rho), out, bits)
    assert_exact(to_host(out), oracle.merge(tp_ref, rho_ref, bits), "theta^")


@pytest.mark.parametrize("bits", [8, 16])
def test_merge_all_bf16_patterns(bits):
    """Every finite BF16 theta' against a spread of corrections, including pairs
    split never produces (a zero theta' with a negative correction and so on)."""
    pats = np.array([b for b in range(65536) if (b & 0x7F80) != 0x7F80], dtype=np.uint16)
    q = 127 if bits == 8 else 32767
    rng = np.random.default_rng(bits)
    rhos = np.unique(np.concatenate([[-q, -q + 1, -64, -1, 0, 1, 2, 63, q - 1, q],
                                     rng.integers(-q, q + 1, 22)]))
    tp = np.repeat(pats, rhos.size)
    rho = np.tile(rhos, pats.size).astype(np.int16 if bits == 16 else np.int8)
    out = torch.empty(tp.size, device="cuda")
    fo.fo_merge(to_dev(tp), to_dev(rho), out, bits)
    assert_exact(to_host(out), oracle.merge(tp, rho, bits), "theta^")


def _state_inputs(kind, n, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_t(3, n) * np.exp(rng.uniform(-30, 3, n))).astype(np.float32)
    groups = n // 32
    if groups >= 8:
        x[:32] = 0.0                                           # all-zero group
        x[32:64] = 0.37                                        # constant group
        x[64:96] = (rng.standard_normal(32) * 1e-9).astype(np.float32)  # subnormal-FP16 scale
        x[96:128] = (rng.standard_normal(32) * 1e3).astype(np.float32)  # large values
        x[128:160] = -1e-30                                    # scale rounds to 0
    if kind in (fo.FO_STATE_VARIANCE, fo.FO_STATE_VARIANCE_LINEAR, fo.FO_STATE_VARIANCE_NONZERO):
        x = np.abs(x) * np.abs(x)
        x = x.astype(np.float32)
    return x


KINDS = [fo.FO_STATE_MOMENTUM, fo.FO_STATE_VARIANCE, fo.FO_STATE_MOMENTUM_LINEAR, fo.FO_STATE_VARIANCE_LINEAR,
         fo.FO_STATE_VARIANCE_NONZERO]


def _signed(kind):
    return kind in (fo.FO_STATE_MOMENTUM, fo.FO_STATE_MOMENTUM_LINEAR)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n", RAGGED + [1 << 22])
def test_quant_matches_oracle(kind, n):
    x = _state_inputs(kind, n, n + kind)
    q = torch.empty(n, dtype=torch.int8 if _signed(kind) else torch.uint8, device="cuda")
    s = torch.empty((n + 31) // 32, dtype=torch.int16, device="cuda")
    fo.fo_quant_state(to_dev(x), q, s, kind)
    q_ref, s_ref = oracle.quant_state(x, kind)
    assert_codes(to_host(q, q_ref.dtype), q_ref, "codes")
    assert_scales(to_host(s), s_ref, "scales")


@pytest.mark.parametrize("kind", KINDS)
def test_quant_input_alignments(kind):
    """The quant kernel reads 32-byte-aligned input with 256-bit loads and
    16-byte-aligned input with 128-bit ones: both give the oracle's codes."""
    n = (1 << 16) + 45
    x = _state_inputs(kind, n, 7 * kind + 3)
    buf = torch.zeros(n + 8, device="cuda")
    for off in (4, 8):                  # 16 and 32 bytes past a 512-byte boundary
        view = buf[off:off + n]
        view.copy_(to_dev(x))
        assert view.data_ptr() % 32 == (16 if off == 4 else 0)
        q = torch.empty(n, dtype=torch.int8 if _signed(kind) else torch.uint8, device="cuda")
        s = torch.empty((n + 31) // 32, dtype=torch.int16, device="cuda")
        fo.fo_quant_state(view, q, s, kind)
        q_ref, s_ref = oracle.quant_state(x, kind)
        assert_codes(to_host(q, q_ref.dtype), q_ref, f"codes, offset {4 * off} bytes")
        assert_scales(to_host(s), s_ref, f"scales, offset {4 * off} bytes")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n", [1, 33, 1000, (1 << 20) + 7])
def test_dequant_matches_oracle(kind, n):
    rng = np.random.default_rng(n)
    if _signed(kind):
        q = rng.integers(-127, 128, n).astype(np.int8)
    else:
        q = rng.integers(0, 256, n).astype(np.uint8)
    ng = (n + 31) // 32
    # every finite non-negative FP16 scale below 2 for companded m (|z| < 2);
    # any finite scale otherwise
    top = 0x4000 if kind == fo.FO_STATE_MOMENTUM else 0x7BFF
    s = rng.integers(0, top + 1, ng).astype(np.uint16)
    out = torch.empty(n, device="cuda")
    fo.fo_dequant_state(to_dev(q), to_dev(s), out, kind)
    assert_exact(to_host(out), oracle.dequant_state(q, s, kind), "decoded state")


def test_dequant_momentum_at_the_fast_path_boundary():
    """Codes including -128 (never written by the codec, but any byte may be
    passed) with scales on both sides of FP16 1.984375, where decoding switches
    between the fast division and the IEEE one: identical to the oracle."""
    rng = np.random.default_rng(77)
    n = 32 * 4096
    q = rng.integers(-128, 128, n).astype(np.int8)
    q[::7] = -128
    s = rng.integers(0x3F00, 0x4001, n // 32).astype(np.uint16)
    out = torch.empty(n, device="cuda")
    fo.fo_dequant_state(to_dev(q), to_dev(s), out, fo.FO_STATE_MOMENTUM)
    assert_exact(to_host(out), oracle.dequant_state(q, s, fo.FO_STATE_MOMENTUM), "decoded momentum")


def test_dequant_momentum_keeps_the_sign_of_zero():
    """A zero scale (and a negative-zero scale) decode codes to signed zeros
    exactly as IEEE division does: -0 for negative codes."""
    q = np.tile(np.arange(-127, 128, 8, dtype=np.int8), 4)[:32 * 4]
    s = np.array([0x0000, 0x8000, 0x0001, 0x3C00], np.uint16)
    out = torch.empty(q.size, device="cuda")
    fo.fo_dequant_state(to_dev(q), to_dev(s), out, fo.FO_STATE_MOMENTUM)
    assert_exact(to_host(out), oracle.dequant_state(q, s, fo.FO_STATE_MOMENTUM), "signed zeros")


def test_binding_rejects_strided_views():
    """A strided view would be read as dense memory: the binding refuses it
    before calling the library."""
    x = torch.zeros(128, device="cuda")
    tp = torch.empty(64, dtype=torch.int16, device="cuda")
    rho = torch.empty(64, dtype=torch.int8, device="cuda")
    with pytest.raises(ValueError, match="contiguous"):
        fo.fo_split(x[::2], tp, rho)
    fo.fo_split(x[:64], tp, rho)        # a contiguous slice is fine
    torch.cuda.synchronize()
