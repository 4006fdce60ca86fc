"""The fused step captured in a CUDA graph.

The C ABI allocates nothing and never synchronizes, and the parameter table
travels in the kernel parameters, so a step call can be captured into a CUDA
graph and replayed. FlashSGD and FlashLion carry no step counter in their
per-step scalars, so replaying one captured step N times is N steps of the
page's fused step (section "融合优化器步骤"), checked here against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import fo
from quantized_optimizer_state_gb300 import workloads as wl
from tests.gpu_helpers import assert_state_matches, device_state_from_oracle, oracle_state_from_device, to_dev

pytestmark = pytest.mark.gpu

SIZES = [1000, 4097, 33, 65536 + 5]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


def _call(opt, table):
    if opt == "sgd":
        fo.fo_sgd_step(table, 0.1, 0.9)
    else:
        fo.fo_lion_step(table, 1e-4, 0.9, 0.99)


@pytest.mark.parametrize("opt", ["sgd", "lion"])
def test_step_replays_from_a_cuda_graph(opt):
    rng = np.random.default_rng(21)
    thetas = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in SIZES]
    host = [oracle.State.from_fp32(t, 8, False, 0.01) for t in thetas]
    dev = [device_state_from_oracle(h) for h in host]
    grads = [wl.to_bf16_bits((rng.standard_t(3, n) * 1e-3).astype(np.float32)) for n in SIZES]
    gdev = [to_dev(g) for g in grads]
    table = fo.table_of(dev, gdev)

    # one ordinary call on throwaway state first, so that the library's
    # per-kernel launch configuration is settled outside the capture
    spare = [device_state_from_oracle(h) for h in host]
    _call(opt, fo.table_of(spare, gdev))
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _call(opt, table)
    torch.cuda.synchronize()
    # capturing records the launch without running it
    for d, h in zip(dev, host):
        assert np.array_equal(oracle_state_from_device(d).theta_p, h.theta_p)

    ref = [h.copy() for h in host]
    for t in range(1, 4):
        graph.replay()
        if opt == "sgd":
            oracle.sgd_step(ref, grads, 0.1, 0.9)
        else:
            oracle.lion_step(ref, grads, 1e-4, 0.9, 0.99)
        torch.cuda.synchronize()
        for i, d in enumerate(dev):
            assert_state_matches(oracle_state_from_device(d), ref[i], f"{opt} graph replay {t} tensor {i}")
