"""GPU parity on inputs that leave the fast path's validated operand ranges.

The fused step computes element pairs with packed FP32 arithmetic and
FMA-based division and square root that are exact inside validated operand
ranges; a thread whose operands leave them recomputes its 16 elements with the
IEEE operations. Each case below plants one such operand in a group of an
otherwise ordinary tensor and checks the whole state bit for bit against the
oracle (page section "融合优化器步骤": the result must not depend on the path).
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import fo
from quantized_optimizer_state_gb300 import workloads as wl
from tests.gpu_helpers import assert_state_matches, device_state_from_oracle, oracle_state_from_device, to_dev

pytestmark = pytest.mark.gpu

N = 4096 + 64 + 7   # several full chunks, a partial tile and a ragged tail


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


def _base(seed, with_v=True, rho_bits=8):
    rng = np.random.default_rng(seed)
    theta = (rng.standard_normal(N) * 0.02).astype(np.float32)
    st = oracle.State.from_fp32(theta, rho_bits, with_v, 0.01)
    g = (rng.standard_normal(N) * 1e-3).astype(np.float32)
    return rng, st, g


def _step_and_compare(opt, st, g32, steps=2, hp=None):
    hp = hp or {}
    dev = device_state_from_oracle(st)
    gb = wl.to_bf16_bits(g32)
    for t in range(1, steps + 1):
        ref = oracle_state_from_device(dev)
        gdev = to_dev(gb)                    # held until the step has run
        table = fo.table_of([dev], [gdev])
        if opt == "adamw":
            oracle.adamw_step([ref], [gb], 1e-3, 0.9, 0.999, 1e-8, t)
            fo.fo_adamw_step(table, 1e-3, 0.9, 0.999, 1e-8, t)
        elif opt == "sgd":
            oracle.sgd_step([ref], [gb], 0.1, 0.9)
            fo.fo_sgd_step(table, 0.1, 0.9)
        else:
            oracle.lion_step([ref], [gb], 1e-4, 0.9, 0.99)
            fo.fo_lion_step(table, 1e-4, 0.9, 0.99)
        torch.cuda.synchronize()
        assert_state_matches(oracle_state_from_device(dev), ref, f"{opt} step {t}", N)


@pytest.mark.parametrize("opt", ["adamw", "sgd", "lion"])
def test_huge_gradients(opt):
    rng, st, g = _base(1, opt == "adamw")
    g[100] = 3e25          # |g| > 2^24: v and m leave the validated ranges
    g[2000] = -1e30
    g[4100] = 2.5e38       # near the BF16 maximum (v overflows to inf)
    # one step: the momentum of these elements companded to z = 2 gives an FP16
    # scale of 2.0, whose top code decodes to an infinite m at the next step
    _step_and_compare(opt, st, g, steps=1)


@pytest.mark.parametrize("opt", ["adamw", "sgd", "lion"])
@pytest.mark.parametrize("rho_bits", [8, 16])
def test_zero_theta_with_both_correction_signs(opt, rho_bits):
    rng, st, g = _base(2, opt == "adamw", rho_bits)
    q = 127 if rho_bits == 8 else 32767
    for i, r in ((5, 3), (6, -3), (40, q), (41, -q), (70, 0)):
        st.theta_p[i] = 0x0000
        st.rho[i] = r
    for i, r in ((300, 5), (301, -5), (302, 0)):
        st.theta_p[i] = 0x8000          # negative zero
        st.rho[i] = r
    _step_and_compare(opt, st, g)


def test_momentum_scale_two_decodes_to_infinity():
    rng, st, g = _base(3)
    # a group whose FP16 momentum scale is exactly 2.0 (2 - |z| can reach 0,
    # outside the fast division's range: the thread takes the exact path); its
    # codes stay below 127 so that every decoded momentum is finite
    st.m_scale[3] = np.float16(2.0).view(np.uint16)
    st.m_q[96:128] = np.arange(-16, 16, dtype=np.int8) * 7
    st.m_q[100] = 126
    st.m_scale[5] = np.float16(1.999).view(np.uint16)   # largest scale kept on the fast path
    st.m_q[160:192] = 127
    _step_and_compare("adamw", st, g, steps=1)


@pytest.mark.parametrize("opt", ["adamw", "sgd", "lion"])
def test_momentum_code_minus_128_near_scale_two(opt):
    """A momentum byte of -128 (never written by the quantizer, but any byte
    may be passed) under FP16 scales from 1.984375 = 127/64 up: there
    |z| = 128 s/127 reaches 2, and at 127/64 exactly z = -2 and
    phi_m^-1(z) = -2/0 = -inf. Scales just below stay on the fast path."""
    rng, st, g = _base(8, opt == "adamw")
    for grp, s in ((1, 0x3FF0), (2, 0x3FF1), (3, 0x3FFF), (4, 0x3FEF), (128, 0x3FF0)):
        st.m_scale[grp] = s
        st.m_q[32 * grp + 5] = -128
        st.m_q[32 * grp + 6] = 127
    _step_and_compare(opt, st, g, steps=1)


def test_tiny_second_moment_and_tiny_quotients():
    rng, st, g = _base(4)
    g[200:232] = 0.0                     # v = 0 at step 1: exact path
    g[500] = 1e-30                       # BF16-representable tiny gradients
    g[501] = -3e-38
    g[900:932] = 1e-20                   # tiny m/den
    st.v_scale[40] = np.float16(6e-8).view(np.uint16)   # FP16-subnormal v scale
    st.v_q[1280:1312] = 1
    _step_and_compare("adamw", st, g)


def test_sgd_momentum_above_fast_range():
    rng, st, g = _base(5, with_v=False)
    theta = (rng.standard_normal(N) * 0.02).astype(np.float32)
    theta[1000:1040] = 1e30                      # wd * theta = 1e34: |m| > 2^100
    st2 = oracle.State.from_fp32(theta, 8, False, 1e4)
    _step_and_compare("sgd", st2, g, steps=1)


@pytest.mark.parametrize("opt", ["sgd", "lion"])
def test_tiny_momenta(opt):
    """Gradients around 1e-33 (momenta below 2^-100, BF16 subnormals among
    them): companding divides by RN(1 + |m|)/2 = 1/2 exactly, where the fast
    division is exact for any dividend. Half the tensor tiny, half ordinary."""
    rng, st, g = _base(9, False)
    g[: N // 2] = (rng.standard_normal(N // 2) * 1e-33).astype(np.float32)
    g[N // 2: N // 2 + 64] = (rng.standard_normal(64) * 1e-39).astype(np.float32)   # subnormal in BF16
    _step_and_compare(opt, st, g, steps=3)
