"""GPU parity of the fused step over the full length of each workload's run.

Page sections "融合优化器步骤" (Algorithm 4) and "实验结果分析" (Fig. 2: the
compressed optimizers track their references over whole training runs).
State that only forms after many steps -- scales decayed toward FP16's
subnormal range or zero, codes held at 0 under a large group scale, momenta
that reached zero -- is compared here. Every listed step runs on the GPU; at
each checked step the oracle starts from the GPU's state before that step
(group-aligned chunks of the oracle run on all host cores).
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import fo
from quantized_optimizer_state_gb300 import workloads as wl
from tests.gpu_helpers import assert_state_matches, oracle_state_from_device, oracle_step_parallel, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


def _step(opt, dev, grads, t, hp):
    table = fo.table_of(dev, grads)
    if opt == "adamw":
        fo.fo_adamw_step(table, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], t)
    elif opt == "sgd":
        fo.fo_sgd_step(table, hp["lr"], hp["momentum"])
    else:
        fo.fo_lion_step(table, hp["lr"], hp["beta1"], hp["beta2"])


def _mismatches(got, ref):
    """Bytes that differ between two states, over every array."""
    n = 0
    for k in ("theta_p", "rho", "m_q", "m_scale", "v_q", "v_scale"):
        a, b = getattr(got, k), getattr(ref, k)
        if a is not None:
            n += int(np.count_nonzero(a.view(np.uint8) != b.view(np.uint8)))
    return n


def run_depth(name, steps, check_at, rho_bits=8, trajectory=False):
    """Run `steps` steps of workload `name` on the GPU; compare with the oracle
    at every step in `check_at`. With trajectory=True the oracle also runs its
    own trajectory from the initial state, never reseeded from the GPU, and
    the GPU's final state must equal it byte for byte (the step is exact, so
    the two trajectories do not drift apart). Returns the number of steps
    checked."""
    w = wl.workload(name, rho_bits)
    hp = {k: v for k, v in w.hparams.items() if k != "weight_decay"}
    dev = []
    for i, p in enumerate(w.params):
        d = fo.CompressedTensor(p.numel, "cuda", rho_bits, w.optimizer == "adamw", w.hparams["weight_decay"])
        theta = wl.init_weight_device(p, i, "cuda")
        d.init_from(theta)
        del theta
        dev.append(d)
    total = w.numel
    checked = 0
    torch.cuda.synchronize()
    traj = [oracle_state_from_device(d) for d in dev] if trajectory else None
    for t in range(1, steps + 1):
        grads = [wl.workload_grad_device(w, i, t, "cuda") for i in range(len(w.params))]
        check = t in check_at
        gh = [to_host(g.view(torch.int16)) for g in grads] if (check or trajectory) else None
        if trajectory:
            oracle_step_parallel(w.optimizer, traj, gh, t, hp)
        if check:
            ref = [oracle_state_from_device(d) for d in dev]
            oracle_step_parallel(w.optimizer, ref, gh, t, hp)
        _step(w.optimizer, dev, grads, t, hp)
        torch.cuda.synchronize()
        if check:
            for i, d in enumerate(dev):
                assert_state_matches(oracle_state_from_device(d), ref[i], f"{name} step {t} tensor {i}", total)
            checked += 1
        del grads
    if trajectory:
        drift = sum(_mismatches(oracle_state_from_device(d), r) for d, r in zip(dev, traj))
        assert drift == 0, f"{name}: the GPU trajectory differs from the oracle's own in {drift} bytes"
    del dev
    torch.cuda.empty_cache()
    return checked


@pytest.mark.parametrize("rho_bits", [8, 16])
def test_stress_64m_all_20_steps(rho_bits):
    assert run_depth("stress_64m", 20, set(range(1, 21)), rho_bits, trajectory=True) == 20


def test_resnet50_sgd_all_50_steps():
    assert run_depth("resnet50", 50, set(range(1, 51)), trajectory=True) == 50


def test_flat_1m_trajectory():
    assert run_depth("flat_1m", 10, {10}, trajectory=True) == 1


def test_gpt2_small_100_steps():
    assert run_depth("gpt2_small", 100, {1, 2, 25, 50, 99, 100}) == 6


def test_gpt2_small_sparse_embedding_200_steps():
    """90 % of the token-embedding rows get a zero gradient at every step: their
    momenta and second moments stay exactly zero, beside live rows."""
    assert run_depth("gpt2_small_sparse_wte", 200, {1, 2, 3, 50, 100, 199, 200}) == 7
