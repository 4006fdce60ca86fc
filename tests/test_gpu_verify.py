"""The fast path's hardware-dependent arithmetic, enumerated on this GPU.

The fused step (page section "融合优化器步骤") must give exactly the IEEE
results of the arithmetic contract. Its packed fast path builds division and
square root from the GPU's reciprocal and reciprocal-square-root
approximations, whose exact outputs the instruction set leaves open: each
sequence is exact on one-variable or finite operand domains given the
approximation's behaviour, and fo_verify_fast_arithmetic enumerates every one
of them on the device with the step's own device functions (about 7e9
operands). Every count must be 0.
"""
import pytest
import torch

from quantized_optimizer_state_gb300 import fo

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()


def test_every_enumerated_domain_is_exact():
    counts = fo.fo_verify_fast_arithmetic()
    assert set(counts) == set(fo.VERIFY_CHECKS)
    assert all(c == 0 for c in counts.values()), counts


def test_counts_are_overwritten():
    """The call zeroes the caller's buffer before counting."""
    buf = torch.full((fo.FO_VERIFY_COUNTS,), 12345, dtype=torch.int64, device="cuda")
    counts = fo.fo_verify_fast_arithmetic(buf)
    assert all(c == 0 for c in counts.values()), counts
