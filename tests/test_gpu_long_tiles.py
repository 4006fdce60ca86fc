"""Parity of every step kernel built for long tiles (8 chunks of 4096
elements), which the library launches for tables large enough to give each
resident CTA at least 8 such tiles (about 120M elements). Each case is one
row of 2^27 elements, checked against the oracle on chunks at its head,
middle and tail over two steps (groups are independent, so a chunk's oracle
step needs only that chunk's state)."""
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import fo
from tests.test_gpu_step import ADAMW, _sampled_parity, _samples_of

pytestmark = pytest.mark.gpu

N = 1 << 27
HP = {"adamw": ADAMW, "sgd": dict(lr=0.1, momentum=0.9), "lion": dict(lr=1e-4, beta1=0.9, beta2=0.99)}

CASES = ([("adamw", rb, gf, vnz) for rb in (8, 16) for gf in (False, True) for vnz in (False, True)]
         + [(o, rb, gf, False) for o in ("sgd", "lion") for rb in (8, 16) for gf in (False, True)])


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


@pytest.mark.parametrize("opt,rho_bits,fp32_grad,v_nonzero", CASES)
def test_long_tile_kernel(opt, rho_bits, fp32_grad, v_nonzero):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(rho_bits * 7 + fp32_grad * 3 + v_nonzero)
    d = fo.CompressedTensor(N, "cuda", rho_bits, opt == "adamw", 0.01)
    d.init_from(torch.randn(N, device="cuda", generator=gen) * 0.02)
    hp = dict(HP[opt], v_nonzero=v_nonzero) if opt == "adamw" else HP[opt]
    samples = _samples_of([N])
    for t in (1, 2):
        g = torch.randn(N, device="cuda", generator=gen) * 1e-3
        g = g if fp32_grad else g.to(torch.bfloat16)
        _sampled_parity(opt, [d], [g], samples, t, hp)
    del d
    torch.cuda.empty_cache()
