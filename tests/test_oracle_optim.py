"""Pins for the oracle's optimizer updates and the fused compressed step.

The FlashOptim page says the optimizers keep "standard" semantics and are
drop-in replacements (sections "融合优化器步骤" and "实践建议"):
  * with the codecs bypassed (FP32 state) the AdamW and SGD element updates are
    checked against torch.optim.AdamW / torch.optim.SGD on CPU;
  * Lion is checked against a hand-computed worked example and its invariants;
  * the fused compressed step is checked against uncompressed FP32 AdamW within
    the quantization error, and for table/group independence.
"""
import math

import numpy as np
import pytest
import torch

from tests.conftest import load_golden
from quantized_optimizer_state_gb300 import workloads as wl

F32_ULP = 2.0 ** -23


def _close_ulps(a, b, ulps):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = np.maximum(np.abs(a), np.abs(b))
    return np.all(np.abs(a - b) <= ulps * F32_ULP * scale + 1e-45)


def _close_signed(a, b, ulps):
    """|a - b| within ulps of |a| plus the rms of a: for quantities that change
    sign, near zero the rounding error is that of the operands, not of the result."""
    a = np.asarray(a, np.float64)
    d = np.abs(a - np.asarray(b, np.float64))
    return np.all(d <= ulps * F32_ULP * (np.abs(a) + np.sqrt(np.mean(a ** 2))))


def test_adamw_fp32_update_matches_torch(orc):
    rng = np.random.default_rng(0)
    n, steps = 4096, 12
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)
    wd = 0.01
    theta = (rng.standard_normal(n) * 0.02).astype(np.float32)
    p = torch.nn.Parameter(torch.from_numpy(theta.copy()))
    opt = torch.optim.AdamW([p], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                            weight_decay=wd, foreach=False, fused=False)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    for t in range(1, steps + 1):
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        orc.adamw_update_fp32(theta, m, v, g, step=t, weight_decay=wd, **hp)
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        st = opt.state[p]
        # torch uses lerp for m and divides by sqrt(bc2); the order of roundings
        # differs by a few ulp per step, contracted by the moving averages. m
        # changes sign, so near zero its error is that of its operands (~ its rms)
        assert _close_signed(m, st["exp_avg"].numpy(), 16)
        assert _close_ulps(v, st["exp_avg_sq"].numpy(), 16)
        # theta: each step may differ by about one rounding of theta and of the
        # update (size ~lr), so the gap grows at most linearly with t
        d = np.abs(theta.astype(np.float64) - p.detach().numpy())
        assert np.all(d <= (t + 2) * F32_ULP * (np.abs(theta) + hp["lr"]))


def test_adamw_bias_correction_first_step(orc):
    """At t = 1 from zero state: m = (1-b1) g and v = (1-b2) g^2; after bias
    correction m/bc1 = g and sqrt(v/bc2) = |g|, so the step is lr * g / (|g| + eps)."""
    g = np.float32([1e-3, -2e-2, 5e-1])
    theta = np.float32([0.5, -0.25, 0.0])
    m = np.zeros(3, np.float32)
    v = np.zeros(3, np.float32)
    orc.adamw_update_fp32(theta, m, v, g, 1e-3, 0.9, 0.999, 1e-8, 1, 0.0)
    expect = np.float64([0.5, -0.25, 0.0]) - 1e-3 * np.sign(g) / (1 + 1e-8 / np.abs(g))
    assert np.all(np.abs(theta - expect) <= 2 * F32_ULP * np.maximum(np.abs(expect), 1e-3))


def test_sgd_fp32_update_matches_torch(orc):
    rng = np.random.default_rng(1)
    n, steps = 4096, 12
    theta = (rng.standard_normal(n) * 0.05).astype(np.float32)
    p = torch.nn.Parameter(torch.from_numpy(theta.copy()))
    opt = torch.optim.SGD([p], lr=0.1, momentum=0.9, weight_decay=1e-4, foreach=False)
    m = np.zeros(n, np.float32)
    for _ in range(steps):
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        orc.sgd_update_fp32(theta, m, g, lr=0.1, momentum=0.9, weight_decay=1e-4)
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        assert _close_signed(m, opt.state[p]["momentum_buffer"].numpy(), 16)
        assert _close_signed(theta, p.detach().numpy(), 16)


def test_lion_worked_example(orc):
    ex = load_golden("lion_worked_example.txt")
    theta = np.float32([ex[f"theta0_{i}"] for i in range(5)])
    m = np.float32([ex[f"m0_{i}"] for i in range(5)])
    g = np.float32([ex[f"g_{i}"] for i in range(5)])
    orc.lion_update_fp32(theta, m, g, ex["lr"], ex["beta1"], ex["beta2"], ex["weight_decay"])
    assert np.allclose(theta, [ex[f"theta1_{i}"] for i in range(5)], rtol=1e-6, atol=0)
    assert np.allclose(m, [ex[f"m1_{i}"] for i in range(5)], rtol=1e-6, atol=1e-9)


def test_lion_invariants(orc):
    rng = np.random.default_rng(6)
    n = 10000
    lr, wd = 1e-4, 0.01
    theta = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g[:10] = 0
    m[:10] = 0
    th0, m0 = theta.copy(), m.copy()
    orc.lion_update_fp32(theta, m, g, lr, 0.9, 0.99, wd)
    decayed = th0.astype(np.float64) * (1 - lr * wd)
    step = theta - decayed
    c = 0.9 * m0.astype(np.float64) + 0.1 * g
    # every element moves by exactly lr against sign(c) (up to FP32 rounding)
    assert np.allclose(step, -lr * np.sign(c), rtol=0, atol=2 * F32_ULP * 0.1)
    assert np.all(theta[:10] == th0[:10] * np.float32(1 - lr * wd))
    # the momentum update does not depend on theta
    m2 = m0.copy()
    orc.lion_update_fp32(np.zeros(n, np.float32), m2, g, lr, 0.9, 0.99, wd)
    assert np.array_equal(m2, m)
    # beta1 = beta2 = 0 is signSGD with decoupled decay
    t3 = th0.copy()
    orc.lion_update_fp32(t3, np.zeros(n, np.float32), g, lr, 0.0, 0.0, 0.0)
    assert np.allclose(t3, th0 - lr * np.sign(g), rtol=0, atol=F32_ULP * 0.1)


def _fresh_states(orc, thetas, rho_bits, with_v):
    return [orc.State.from_fp32(t, rho_bits, with_v, weight_decay=0.01) for t in thetas]


@pytest.mark.parametrize("rho_bits", [8, 16])
def test_compressed_adamw_tracks_fp32_adamw(orc, rho_bits):
    """The fused compressed step stays within the quantization error of
    uncompressed FP32 AdamW on a small problem (Fig. 2's "no drift", in small)."""
    rng = np.random.default_rng(12)
    n, steps, lr = 32 * 256, 10, 1e-3
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    st = orc.State.from_fp32(theta0, rho_bits, True, weight_decay=0.01)
    ref = theta0.copy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    for t in range(1, steps + 1):
        g32 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        gb = wl.to_bf16_bits(g32)
        g = (gb.astype(np.uint32) << 16).view(np.float32)
        orc.adamw_step([st], [gb], lr, 0.9, 0.999, 1e-8, t)
        orc.adamw_update_fp32(ref, m, v, g, lr, 0.9, 0.999, 1e-8, t, 0.01)
    got = orc.merge(st.theta_p, st.rho, rho_bits).astype(np.float64)
    diff = np.abs(got - ref)
    # each Adam update is at most about lr in size; the state codecs perturb it by
    # well under a per cent for typical elements (half a code level of m and of
    # sqrt(v)), more for elements far below their group's maximum: bound the
    # median and the maximum of the accumulated difference
    assert np.median(diff) < 0.005 * lr * steps
    assert diff.max() < 0.2 * lr * steps
    # and the trajectory did move, by far more than the difference
    assert np.median(np.abs(ref - theta0)) > 0.1 * lr * steps


def test_step_is_independent_per_tensor_and_group(orc):
    rng = np.random.default_rng(13)
    sizes = [1000, 32, 33, 4096 + 7]
    thetas = [(rng.standard_normal(k) * 0.02).astype(np.float32) for k in sizes]
    grads = [wl.to_bf16_bits((rng.standard_normal(k) * 1e-3).astype(np.float32)) for k in sizes]
    a = _fresh_states(orc, thetas, 8, True)
    for t in (1, 2, 3):
        orc.adamw_step(a, grads, 1e-3, 0.9, 0.999, 1e-8, t)
    for i in range(len(sizes)):
        b = _fresh_states(orc, [thetas[i]], 8, True)
        for t in (1, 2, 3):
            orc.adamw_step(b, [grads[i]], 1e-3, 0.9, 0.999, 1e-8, t)
        for f in ("theta_p", "rho", "m_q", "m_scale", "v_q", "v_scale"):
            assert np.array_equal(getattr(a[i], f), getattr(b[0], f)), (i, f)
    # a tensor split at a group boundary steps the same as the whole
    x = thetas[3]
    whole = _fresh_states(orc, [x], 8, True)
    parts = _fresh_states(orc, [x[:2048], x[2048:]], 8, True)
    orc.adamw_step(whole, [grads[3]], 1e-3, 0.9, 0.999, 1e-8, 1)
    orc.adamw_step(parts, [grads[3][:2048].copy(), grads[3][2048:].copy()], 1e-3, 0.9, 0.999, 1e-8, 1)
    assert np.array_equal(whole[0].theta_p, np.concatenate([parts[0].theta_p, parts[1].theta_p]))
    assert np.array_equal(whole[0].m_scale, np.concatenate([parts[0].m_scale, parts[1].m_scale]))


def test_compressed_sgd_and_lion_track_fp32(orc):
    rng = np.random.default_rng(14)
    n = 32 * 128
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    for opt in ("sgd", "lion"):
        st = orc.State.from_fp32(theta0, 8, False, weight_decay=1e-4 if opt == "sgd" else 0.01)
        ref = theta0.copy()
        m = np.zeros(n, np.float32)
        for t in range(1, 6):
            gb = wl.to_bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
            g = (gb.astype(np.uint32) << 16).view(np.float32)
            if opt == "sgd":
                orc.sgd_step([st], [gb], 0.1, 0.9)
                orc.sgd_update_fp32(ref, m, g, 0.1, 0.9, 1e-4)
                tol = 0.1 * 5 * 1e-3 * 0.05
            else:
                orc.lion_step([st], [gb], 1e-4, 0.9, 0.99)
                orc.lion_update_fp32(ref, m, g, 1e-4, 0.9, 0.99, 0.01)
                tol = 1e-4 * 5 * 0.5
        got = orc.merge(st.theta_p, st.rho, 8)
        assert np.median(np.abs(got - ref)) < tol, opt


def test_bad_arguments_are_rejected(orc):
    st = orc.State.from_fp32(np.zeros(64, np.float32), 8, True)
    gb = np.zeros(64, np.uint16)
    with pytest.raises(ValueError):
        orc.adamw_step([st], [gb], 1e-3, 0.9, 0.999, 1e-8, 0)     # step must be >= 1
    st.rho_bits = 12
    with pytest.raises(ValueError):
        orc.adamw_step([st], [gb], 1e-3, 0.9, 0.999, 1e-8, 1)


def _spiky_state(orc, n, seed):
    """A state after a few AdamW steps of heavy-tailed gradients, so that many
    groups hold a v far below their group's scale."""
    rng = np.random.default_rng(seed)
    st = orc.State.from_fp32((rng.standard_normal(n) * 0.02).astype(np.float32), 8, True, 0.01)
    for t in range(1, 4):
        g = wl.to_bf16_bits((rng.standard_t(1.5, n) * 1e-3).astype(np.float32))
        orc.adamw_step([st], [g], 1e-3, 0.9, 0.999, 1e-8, t)
    return st, rng


def test_v_nonzero_step_changes_only_zero_v_codes(orc):
    """With the opt-in rule, one step from the same state writes the same
    theta', rho, m codes and scales; v codes differ only where the plain step
    writes 0 in a group with a non-zero scale, and there they are 1."""
    n = 32 * 4096
    st, rng = _spiky_state(orc, n, 61)
    g = wl.to_bf16_bits((rng.standard_t(1.5, n) * 1e-3).astype(np.float32))
    a, b = st.copy(), st.copy()
    orc.adamw_step([a], [g], 1e-3, 0.9, 0.999, 1e-8, 4)
    orc.adamw_step([b], [g], 1e-3, 0.9, 0.999, 1e-8, 4, v_nonzero=True)
    for f in ("theta_p", "rho", "m_q", "m_scale", "v_scale"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    moved = a.v_q != b.v_q
    assert moved.sum() > 10
    assert np.all((a.v_q[moved] == 0) & (b.v_q[moved] == 1))
    live = np.repeat(a.v_scale != 0, 32)
    assert np.array_equal(moved, live & (a.v_q == 0))
    vdec = orc.dequant_state(b.v_q, b.v_scale, 1)
    assert np.all(vdec[live] > 0)


def test_zero_decoded_v_moves_theta_by_m_over_eps(orc):
    """The hazard the opt-in rule avoids, as a closed form: an element whose v
    decodes to 0 while its momentum does not, with a zero gradient, moves by
    lr/bc1 * (beta1 * m) / eps."""
    lr, b1, b2, eps, t = 1e-3, 0.9, 0.999, 1e-8, 5
    st = orc.State.from_fp32(np.full(32, 0.5, np.float32), 8, True, 0.0)
    st.m_q[:] = 64
    st.m_scale[:] = orc.fp16_rne(0.01)
    st.v_q[:] = 0
    st.v_q[0] = 255
    st.v_scale[:] = orc.fp16_rne(1e-3)
    mhat = orc.dequant_state(st.m_q, st.m_scale, 0).astype(np.float64)
    g = np.zeros(32, np.uint16)
    orc.adamw_step([st], [g], lr, b1, b2, eps, t)
    got = orc.merge(st.theta_p, st.rho, 8).astype(np.float64)
    bc1 = 1 - b1 ** t
    expect = 0.5 - lr / bc1 * (b1 * mhat[1:]) / eps
    # to the resolution of the stored weight (8-bit rho: 2^-8/254 relative)
    assert np.allclose(got[1:], expect, rtol=2.0 ** -8 / 254 * 1.05 + 1e-6)
    assert np.all(np.abs(got[1:] - 0.5) > 1e5 * lr)   # five orders of magnitude above lr
