"""Host-side checks of the drop-in optimizers (no GPU needed)."""
import pytest
import torch

from quantized_optimizer_state_gb300 import optim


def test_cpu_parameters_are_rejected():
    p = torch.nn.Parameter(torch.zeros(10))
    with pytest.raises(RuntimeError, match="CUDA"):
        optim.FlashAdamW([p])


def test_bad_rho_bits_rejected():
    p = torch.nn.Parameter(torch.zeros(10))
    with pytest.raises((ValueError, RuntimeError)):
        optim.FlashSGD([p], rho_bits=12)
