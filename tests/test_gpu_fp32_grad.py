"""GPU parity of the fused step with FP32 gradients (fo_tensor_t.grad_dtype =
FO_GRAD_F32) against the CPU oracle, through the C ABI.

The fused step of "FlashOptim: Optimizers for Memory Efficient Training"
(section "融合优化器步骤") reads BF16 gradients; the FP32-gradient kernels take
the FP32 value into the FP32 update unrounded, at 2 more bytes of reads per
parameter. Same bar as the BF16 path: theta' and scales bit-exact, codes
within +-1 on at most 1e-6 of the elements.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import fo
from quantized_optimizer_state_gb300 import workloads as wl
from tests.gpu_helpers import to_dev
from tests.test_gpu_step import (ADAMW, RAGGED, _device_workload, _hp, _make_states, _sampled_parity,
                                 _samples_of, run_parity)

pytestmark = pytest.mark.gpu

HP = {"adamw": ADAMW, "sgd": dict(lr=0.1, momentum=0.9), "lion": dict(lr=1e-4, beta1=0.9, beta2=0.99)}
WD = {"adamw": 0.01, "sgd": 1e-4, "lion": 0.01}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


def _ragged(seed, scale=0.02, bf16_rows=()):
    rng = np.random.default_rng(seed)
    thetas = [(rng.standard_normal(n) * scale).astype(np.float32) for n in RAGGED]

    def grads(t):
        r = np.random.default_rng(seed * 1000 + t)
        out = [(r.standard_t(3, n) * 1e-3).astype(np.float32) for n in RAGGED]
        return [wl.to_bf16_bits(g) if i in bf16_rows else g for i, g in enumerate(out)]
    return thetas, grads


@pytest.mark.parametrize("opt", ["adamw", "sgd", "lion"])
@pytest.mark.parametrize("rho_bits", [8, 16])
def test_ragged_table_fp32_grads(opt, rho_bits):
    thetas, grads = _ragged(20 + rho_bits, 0.05 if opt == "sgd" else 0.02)
    run_parity(opt, thetas, grads, 4, HP[opt], rho_bits, WD[opt], f"{opt} fp32-grad rho{rho_bits}")


def test_grad_types_and_widths_mixed_in_one_call():
    """Rows of both gradient types and both rho widths in one table: one launch
    per combination, each row as the oracle steps it."""
    n = len(RAGGED)
    thetas, grads = _ragged(30, bf16_rows={i for i in range(n) if i % 2})
    bits = [8 if (i // 2) % 2 == 0 else 16 for i in range(n)]
    run_parity("adamw", thetas, grads, 2, ADAMW, bits, 0.01, "mixed")
    dev = _make_states(thetas, "adamw", bits, 0.01)
    gd = [to_dev(g) for g in grads(3)]
    c0 = fo.fo_kernel_launch_count()
    fo.fo_adamw_step(fo.table_of(dev, gd), 1e-3, 0.9, 0.999, 1e-8, 1)
    torch.cuda.synchronize()
    assert fo.fo_kernel_launch_count() - c0 == 4


def test_gpt2_small_adamw_fp32_grads():
    w = wl.workload("gpt2_small")
    thetas = [wl.init_weight(p, i) for i, p in enumerate(w.params)]

    def grads(t):
        return [wl.grad_fp32(w.grad, w.grad_scale, p.numel, i, t) for i, p in enumerate(w.params)]
    hp, wd = _hp(w)
    run_parity("adamw", thetas, grads, 2, hp, w.rho_bits, wd, "gpt2_small fp32-grad")


@pytest.mark.parametrize("opt", ["adamw", "lion"])
def test_stress_64m_fp32_grads(opt):
    """Weights over 18 decades with zeros and subnormals, gradients with 1 %
    outliers x1e3 and exact zeros: the exact-path fallback with FP32 gradients."""
    w = wl.workload("stress_64m", 8)
    thetas = [wl.init_weight(p, i) for i, p in enumerate(w.params)]

    def grads(t):
        return [wl.grad_fp32(w.grad, w.grad_scale, p.numel, i, t) for i, p in enumerate(w.params)]
    run_parity(opt, thetas, grads, 2, HP[opt], 8, WD[opt], f"stress_64m {opt} fp32-grad")


def test_llama31_8b_fp32_grads_full_size_sampled():
    """The full 8.03e9-parameter AdamW table with FP32 gradients in one call,
    every eighth row sampled at head, middle and tail."""
    w = wl.workload("llama31_8b")
    dev, grads = _device_workload(w, grad_fp32=True)
    assert grads[0].dtype == torch.float32
    hp, _ = _hp(w)
    rows = set(range(0, len(w.params), 8)) | {len(w.params) - 1}
    samples = _samples_of([p.numel for p in w.params], rows=rows)
    for t in (1, 2):
        _sampled_parity(w.optimizer, dev, grads, samples, t, hp)
    del dev, grads
    torch.cuda.empty_cache()
