"""Pins for the oracle's fused step with FP32 gradients.

The FlashOptim page's fused step reads BF16 gradients ("融合优化器步骤"); for
callers whose gradients are FP32 the plainest reading is that the FP32 value
enters the FP32 update unrounded. The pins:
  * a gradient whose FP32 values are exactly BF16 values gives the same state,
    bit for bit, as the same gradient given as BF16 (all three optimizers);
  * closed forms at t = 1 from zero state (SGD: theta - lr*g; AdamW:
    theta - lr*g/(|g| + eps)) hold to FP32 rounding with the FP32 gradient,
    with a 16-bit rho so that the stored master weight resolves them; and
    they do NOT hold with the gradient rounded to BF16 first (the negative
    control that shows the pin sees the gradient's low bits).
"""
import numpy as np
import pytest

from quantized_optimizer_state_gb300 import workloads as wl

F32_ULP = 2.0 ** -23


def _bf16_values(x):
    """x rounded to BF16, as FP32 values, and their bit patterns."""
    bits = wl.to_bf16_bits(np.asarray(x, np.float32))
    return (bits.astype(np.uint32) << 16).view(np.float32), bits


def _state(orc, theta0, rho_bits, with_v, wd=0.0):
    return orc.State.from_fp32(theta0, rho_bits, with_v, weight_decay=wd)


def _fields(st):
    return [st.theta_p, st.rho, st.m_q, st.m_scale] + ([st.v_q, st.v_scale] if st.v_q is not None else [])


@pytest.mark.parametrize("opt", ["adamw", "sgd", "lion"])
@pytest.mark.parametrize("rho_bits", [8, 16])
def test_bf16_valued_fp32_grad_equals_bf16_grad(orc, opt, rho_bits):
    rng = np.random.default_rng(40)
    n = 32 * 40 + 13
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    with_v = opt == "adamw"
    a = _state(orc, theta0, rho_bits, with_v, 0.01)
    b = a.copy()
    for t in (1, 2, 3):
        gf, gb = _bf16_values(rng.standard_normal(n) * 1e-2)
        if opt == "adamw":
            orc.adamw_step([a], [gb], 1e-3, 0.9, 0.999, 1e-8, t)
            orc.adamw_step([b], [gf], 1e-3, 0.9, 0.999, 1e-8, t)
        elif opt == "sgd":
            orc.sgd_step([a], [gb], 0.1, 0.9)
            orc.sgd_step([b], [gf], 0.1, 0.9)
        else:
            orc.lion_step([a], [gb], 1e-4, 0.9, 0.99)
            orc.lion_step([b], [gf], 1e-4, 0.9, 0.99)
    for fa, fb in zip(_fields(a), _fields(b)):
        assert np.array_equal(fa, fb)


def _theta1(orc, st):
    return orc.merge(st.theta_p, st.rho, st.rho_bits).astype(np.float64)


def test_sgd_first_step_uses_the_fp32_gradient(orc):
    """SGD at t = 1 from m = 0, wd = 0: m = g and theta1 = theta0 - lr*g."""
    rng = np.random.default_rng(41)
    n = 32 * 64
    theta0, _ = _bf16_values(0.02 + 0.01 * rng.random(n))   # rho = 0: theta^0 = theta0 exactly
    g = (1e-2 * (1 + rng.random(n)) * rng.choice([-1, 1], n)).astype(np.float32)
    lr = np.float32(0.1)
    st = _state(orc, theta0, 16, False)
    orc.sgd_step([st], [g], float(lr), 0.9)
    got = _theta1(orc, st)
    expect = theta0.astype(np.float64) - np.float64(lr) * g.astype(np.float64)
    # RN of the FP32 fma plus the 16-bit split/merge: a few FP32 ulps of theta1
    tol = 3 * F32_ULP * np.abs(expect)
    assert np.all(np.abs(got - expect) <= tol)
    # negative control: with the gradient rounded to BF16 the closed form misses
    gr, _ = _bf16_values(g)
    wrong = theta0.astype(np.float64) - np.float64(lr) * gr.astype(np.float64)
    assert np.mean(np.abs(got - wrong) > tol) > 0.9


def test_adamw_first_step_uses_the_fp32_gradient(orc):
    """AdamW at t = 1 from zero state, wd = 0: theta1 = theta0 - lr*g/(|g| + eps).
    eps of the size of |g| makes the step depend on the gradient's low bits."""
    rng = np.random.default_rng(42)
    n = 32 * 64
    theta0, _ = _bf16_values(0.02 + 0.01 * rng.random(n))
    g = (1e-3 * (0.5 + 1.5 * rng.random(n)) * rng.choice([-1, 1], n)).astype(np.float32)
    lr, eps = 1e-3, 1e-3
    st = _state(orc, theta0, 16, True)
    orc.adamw_step([st], [g], lr, 0.9, 0.999, eps, 1)
    got = _theta1(orc, st)
    g64 = g.astype(np.float64)
    upd = lr * g64 / (np.abs(g64) + eps)
    expect = theta0.astype(np.float64) - upd
    # the FP32 update chain (products, sqrt, two divisions) rounds a few
    # times on a step of size ~lr, the new theta once and the split once
    tol = 3 * F32_ULP * np.abs(expect) + 16 * F32_ULP * np.abs(upd)
    assert np.all(np.abs(got - expect) <= tol)
    gr, _ = _bf16_values(g)
    g64r = gr.astype(np.float64)
    wrong = theta0.astype(np.float64) - lr * g64r / (np.abs(g64r) + eps)
    assert np.mean(np.abs(got - wrong) > tol) > 0.9


def test_fp32_and_bf16_grads_mix_in_one_table(orc):
    """Rows of both gradient types in one call step as they would alone."""
    rng = np.random.default_rng(43)
    sizes = [100, 64, 33]
    thetas = [(rng.standard_normal(k) * 0.02).astype(np.float32) for k in sizes]
    grads = [(rng.standard_normal(k) * 1e-2).astype(np.float32) for k in sizes]
    grads[1] = wl.to_bf16_bits(grads[1])
    together = [_state(orc, t, 8, True) for t in thetas]
    orc.adamw_step(together, grads, 1e-3, 0.9, 0.999, 1e-8, 1)
    for i in range(len(sizes)):
        alone = _state(orc, thetas[i], 8, True)
        orc.adamw_step([alone], [grads[i]], 1e-3, 0.9, 0.999, 1e-8, 1)
        for fa, fb in zip(_fields(together[i]), _fields(alone)):
            assert np.array_equal(fa, fb)
