"""Pins for the compressed state layout, from the FlashOptim page's memory figures.

Per parameter the fused step keeps theta' (BF16, 2 B), rho (INT8, 1 B), m
(INT8, 1 B), v (UINT8, 1 B) and one FP16 scale per 32 elements for each of m
and v. The page's Table 4 (Llama-3.1-8B) and its byte counts follow from
exactly this layout.
"""
import pytest

from quantized_optimizer_state_gb300 import workloads as wl

GIB = 2.0 ** 30


def _state_bytes_per_param(rho_bits=8, with_v=True, scale_bytes=2, group=32):
    """rho + m (+ v) codes and their FP16 group scales; theta' excluded."""
    state = rho_bits // 8 + 1 + (1 if with_v else 0)
    scales = scale_bytes * (2 if with_v else 1) / group
    return state + scales


def test_parameter_counts_of_the_workloads():
    assert wl.workload("flat_1m").numel == 1_048_576
    assert wl.workload("gpt2_small").numel == 124_439_808
    assert len(wl.workload("gpt2_small").params) == 148
    assert wl.workload("resnet50").numel == 25_557_032
    assert len(wl.workload("resnet50").params) == 161
    assert wl.workload("llama31_8b").numel == 8_030_261_248
    assert len(wl.workload("llama31_8b").params) == 291
    assert wl.workload("stress_64m").numel == 1 << 26


def test_table4_memory_figures(golden):
    n = wl.workload("llama31_8b").numel
    assert round(n * 4 / GIB, 1) == golden["table4_param_gib_reference"]     # FP32 weights
    assert round(n * 2 / GIB, 1) == golden["table4_param_gib_flash"]         # BF16 theta'
    assert round(n * 8 / GIB, 1) == golden["table4_state_gib_reference"]     # FP32 m, v
    # rho + m + v + two FP16 scales per 32 = 3.125 B: one scale per group for
    # each of m and v, none for rho
    state = _state_bytes_per_param()
    assert state == 3.125
    assert round(n * state / GIB, 1) == golden["table4_state_gib_flash"]
    # quantizing m and v alone: 8 B -> 2 + 4/32 B, "about 73 %"
    assert round(100 * (1 - 2.125 / 8)) == golden["state_compression_percent"]
    assert golden["group_size"] == 32


def test_bytes_per_parameter(golden):
    grad = 2
    flash = 2 + 1 + 1 + 1 + grad               # theta', rho, m, v, BF16 grad
    assert flash == golden["flash_bytes_per_param"]
    assert flash - grad == golden["flash_bytes_per_param_grad_release"]
    assert grad == golden["grad_release_saving_bytes"]
    assert 4 + 4 + 4 + 4 == golden["adamw_bytes_per_param"]   # FP32 weight, grad, m, v
    assert 7e9 * 16 / 1e9 == golden["seven_b_reference_gb"]
    # checkpoints: FP32 weight + m + v vs theta' + rho + m + v
    assert 4 + 4 + 4 == golden["checkpoint_bytes_reference"]
    assert 2 + 1 + 1 + 1 == golden["checkpoint_bytes_flash"]
    assert 70e9 * 12 / 1e9 == golden["checkpoint_70b_gb_reference"]
    assert 70e9 * 5 / 1e9 == golden["checkpoint_70b_gb_flash"]


@pytest.mark.parametrize("opt,rho_bits,expect", [("adamw", 8, 12.25), ("adamw", 16, 14.25),
                                                  ("sgd", 8, 10.125), ("lion", 8, 10.125)])
def test_algorithmic_bytes_per_step(opt, rho_bits, expect):
    """Bytes one fused step must move per parameter if each crosses HBM once:
    read grad + theta' + rho + codes + scales, write all but grad back."""
    with_v = opt == "adamw"
    state = 2 + _state_bytes_per_param(rho_bits, with_v)   # theta' + rho + codes + scales
    assert state + 2 + state == expect
