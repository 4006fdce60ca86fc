"""GPU parity of the fused step on state that holds exact zeros and tiny values.

Page section "融合优化器步骤" (Algorithm 4). Real tables hold rows whose
gradients are exactly zero (an embedding row no token touched), whose
momentum has decayed to exactly zero while the second moment has not, and
gradients far below the usual scale. The step must give the oracle's result
bit for bit on all of them, whichever internal path computes it. Every case
runs per step: the oracle starts from the state the GPU produced before.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import fo
from quantized_optimizer_state_gb300 import workloads as wl
from tests.test_gpu_step import run_parity

pytestmark = pytest.mark.gpu

ADAMW = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)
SGD = dict(lr=0.1, momentum=0.9)
LION = dict(lr=1e-4, beta1=0.9, beta2=0.99)
SIZES = [4096, 4096 + 17, 8192, 5000, 4096, 33, 12288]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


def _thetas(seed):
    rng = np.random.default_rng(seed)
    th = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in SIZES]
    th[4][:] = 0.0                                   # a zero-initialised row (theta' = 0 at step 1)
    th[4][1::2] = -0.0
    th[6][::7] = 0.0
    return th


def _grads_fp32(seed, t):
    """Row 0: zero every step. Row 1: gradients for three steps, then zero (the
    momentum decays to zero while the second moment does not). Row 2: 1 %
    exact zeros and 1 % outliers x1e3. Row 3: tiny magnitudes from 2^-140
    (BF16 subnormals) to 2^-20, with zeros. Row 4: ordinary. Row 5: a short
    ragged row with zeros. Row 6: a third of the groups all zero."""
    r = np.random.default_rng(seed * 1000 + t)
    g = [(r.standard_t(3, n) * 1e-3).astype(np.float32) for n in SIZES]
    g[0][:] = 0.0
    if t > 3:
        g[1][:] = 0.0
    n2 = SIZES[2]
    g[2][r.random(n2) < 0.01] = 0.0
    out = r.random(n2) < 0.01
    g[2][out] *= 1e3
    n3 = SIZES[3]
    mag = np.exp2(r.uniform(-140, -20, n3)).astype(np.float32)
    g[3] = (mag * np.where(r.random(n3) < 0.5, -1, 1)).astype(np.float32)
    g[3][r.random(n3) < 0.05] = 0.0
    g[5][::3] = 0.0
    g6 = g[6].reshape(-1, 32)
    g6[::3] = 0.0
    return g


def _grads(seed, fp32):
    if fp32:
        return lambda t: _grads_fp32(seed, t)
    return lambda t: [wl.to_bf16_bits(x) for x in _grads_fp32(seed, t)]


@pytest.mark.parametrize("rho_bits", [8, 16])
@pytest.mark.parametrize("fp32", [False, True])
@pytest.mark.parametrize("v_nonzero", [False, True])
def test_adamw_zero_and_tiny_state(rho_bits, fp32, v_nonzero):
    hp = dict(ADAMW, v_nonzero=v_nonzero)
    run_parity("adamw", _thetas(1), _grads(1, fp32), 30, hp, rho_bits, 0.01,
               f"adamw zeros rho{rho_bits} fp32={fp32} vnz={v_nonzero}")


@pytest.mark.parametrize("rho_bits", [8, 16])
@pytest.mark.parametrize("wd", [0.0, 1e-4])
def test_sgd_zero_and_tiny_state(rho_bits, wd):
    run_parity("sgd", _thetas(2), _grads(2, False), 30, SGD, rho_bits, wd, f"sgd zeros rho{rho_bits} wd={wd}")


@pytest.mark.parametrize("rho_bits", [8, 16])
def test_lion_zero_and_tiny_state(rho_bits):
    run_parity("lion", _thetas(3), _grads(3, False), 30, LION, rho_bits, 0.01, f"lion zeros rho{rho_bits}")


@pytest.mark.parametrize("hp", [
    dict(ADAMW, beta1=0.0),                 # no momentum: b1*m is a signed zero
    dict(ADAMW, beta2=0.0),
    dict(ADAMW, beta1=2.0 ** -20),          # below the fast path's momentum bound
    dict(ADAMW, beta2=1.0 - 2.0 ** -30),    # 1 - b2 below 2^-24
    dict(ADAMW, lr=0.0),
    dict(ADAMW, lr=1e-30),
    dict(ADAMW, eps=2.0 ** -40),
    dict(ADAMW, eps=2.0 ** -41),
])
def test_adamw_hyper_parameter_edges(hp):
    run_parity("adamw", _thetas(4), _grads(4, False), 6, hp, 8, 0.01, f"adamw {hp}")


def test_adamw_decay_factor_near_zero():
    """1 - lr*wd of 0 and of a tiny value: a decayed theta can be zero."""
    for wd in (1.0 / ADAMW["lr"], (1.0 - 2.0 ** -12) / ADAMW["lr"]):
        run_parity("adamw", _thetas(5), _grads(5, False), 4, ADAMW, 8, wd, f"adamw wd={wd}")


@pytest.mark.parametrize("hp", [dict(SGD, momentum=0.0), dict(SGD, lr=0.0)])
def test_sgd_hyper_parameter_edges(hp):
    run_parity("sgd", _thetas(6), _grads(6, False), 6, hp, 8, 1e-4, f"sgd {hp}")


@pytest.mark.parametrize("hp", [dict(LION, beta1=0.0), dict(LION, beta2=0.0)])
def test_lion_hyper_parameter_edges(hp):
    run_parity("lion", _thetas(7), _grads(7, False), 6, hp, 8, 0.01, f"lion {hp}")
