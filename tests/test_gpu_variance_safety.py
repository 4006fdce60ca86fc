"""The opt-in second-moment rule (FO_ADAMW_V_NONZERO, FO_STATE_VARIANCE_NONZERO):
GPU parity with the oracle's rule, and its effect measured on the fused step.

The page leaves the numerical-stability step of its variance quantizer
(section "带压缩扩展的优化器状态量化", Algorithm 3) unprinted. Under the plain
reading, a v below 1/510 of its group's scale decodes to 0. With the rule, a
non-zero v keeps at least code 1."""
import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import codec_study as cs
from quantized_optimizer_state_gb300 import fo
from quantized_optimizer_state_gb300 import workloads as wl
from tests.gpu_helpers import assert_state_matches, oracle_state_from_device, to_dev
from tests.test_gpu_step import RAGGED, _make_states

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


def _spiky(n, rng):
    g = rng.standard_t(3, n) * 1e-3
    spike = rng.random(n) < 0.01
    return wl.to_bf16_bits(np.where(spike, g * 1e3, g).astype(np.float32))


def _parity(thetas, rho_bits, steps, seed, what):
    dev = _make_states(thetas, "adamw", rho_bits, 0.01)
    total = sum(t.size for t in thetas)
    rng = np.random.default_rng(seed)
    moved = 0
    for t in range(1, steps + 1):
        grads = [_spiky(th.size, rng) for th in thetas]
        ref = [oracle_state_from_device(d) for d in dev]
        plain = [r.copy() for r in ref]
        oracle.adamw_step(ref, grads, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], t, v_nonzero=True)
        oracle.adamw_step(plain, grads, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], t)
        moved += sum(int(np.count_nonzero(a.v_q != b.v_q)) for a, b in zip(ref, plain))
        gdev = [to_dev(g) for g in grads]    # held until the step has run
        fo.fo_adamw_step(fo.table_of(dev, gdev), HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], t,
                         v_nonzero=True)
        torch.cuda.synchronize()
        for i, d in enumerate(dev):
            assert_state_matches(oracle_state_from_device(d), ref[i], f"{what} step {t} tensor {i}", total)
    return moved


@pytest.mark.parametrize("rho_bits", [8, 16])
def test_v_nonzero_step_matches_oracle_ragged(rho_bits):
    rng = np.random.default_rng(70 + rho_bits)
    thetas = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in RAGGED]
    moved = _parity(thetas, rho_bits, 6, 80 + rho_bits, f"v_nonzero rho{rho_bits}")
    assert moved > 0          # the rule changed some codes: the comparison is not vacuous


def test_v_nonzero_step_matches_oracle_gpt2_small():
    w = wl.workload("gpt2_small")
    thetas = [wl.init_weight(p, i) for i, p in enumerate(w.params)]
    _parity(thetas, 8, 2, 90, "v_nonzero gpt2_small")


def test_rule_removes_zero_decodes_and_bounds_updates():
    """Same spiky gradients, both modes: the plain reading leaves elements whose
    v decodes to 0 under a non-zero momentum, and their updates grow far
    beyond lr; with the rule there are none and the largest update shrinks."""
    r = cs.variance_safety_study(1 << 18, 60, 1, "cuda", spike_prob=1e-3)
    assert r["plain"]["events_total"] > 0
    assert r["v_nonzero"]["events_total"] == 0
    assert r["v_nonzero"]["max_update_lr"] < r["plain"]["max_update_lr"]
