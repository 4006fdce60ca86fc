"""Parity of every step kernel, for the three tile lengths the library launches.

Long tiles (8 chunks of 4096 elements) are used for tables large enough to
give each resident CTA at least 6 of them (up to about 120M elements, at 4
resident CTAs per SM). Each long
case is one row of 2^27 elements, checked against the oracle on chunks at its
head, middle and tail over two steps (groups are independent, so a chunk's
oracle step needs only that chunk's state). Short tiles (2 chunks) serve
tables that still give every CTA a tile (a few million elements up); each
short case is a ragged table of about 6M elements, sampled the same way.
One-chunk tiles serve smaller tables; each tiny case is a small ragged table,
checked in full."""
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import fo
from quantized_optimizer_state_gb300 import workloads as wl
import numpy as np

from tests.test_gpu_step import ADAMW, RAGGED, _sampled_parity, _samples_of, run_parity

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


MID = [4 * 1024 * 1024 + 4097, 999, 1024 * 1024 + 33, 65536, 777777]


@pytest.mark.parametrize("opt,rho_bits,fp32_grad,v_nonzero", CASES)
def test_short_tile_kernel(opt, rho_bits, fp32_grad, v_nonzero):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(rho_bits * 5 + fp32_grad * 3 + v_nonzero + 7)
    dev = []
    for n in MID:
        d = fo.CompressedTensor(n, "cuda", rho_bits, opt == "adamw", 0.01)
        d.init_from(torch.randn(n, device="cuda", generator=gen) * 0.02)
        dev.append(d)
    hp = dict(HP[opt], v_nonzero=v_nonzero) if opt == "adamw" else HP[opt]
    samples = _samples_of(MID, per_row=1 << 15)
    launches = fo.fo_kernel_launch_count()
    for t in (1, 2):
        g = [torch.randn(n, device="cuda", generator=gen) * 1e-3 for n in MID]
        g = g if fp32_grad else [x.to(torch.bfloat16) for x in g]
        _sampled_parity(opt, dev, g, samples, t, hp)
    assert fo.fo_kernel_launch_count() - launches == 2
    del dev
    torch.cuda.empty_cache()


@pytest.mark.parametrize("opt,rho_bits,fp32_grad,v_nonzero", CASES)
def test_tiny_tile_kernel(opt, rho_bits, fp32_grad, v_nonzero):
    rng = np.random.default_rng(rho_bits * 7 + fp32_grad * 3 + v_nonzero + 100)
    thetas = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in RAGGED]

    def grads(t):
        r = np.random.default_rng(1000 * t + rho_bits)
        g = [(r.standard_t(3, n) * 1e-3).astype(np.float32) for n in RAGGED]
        return g if fp32_grad else [wl.to_bf16_bits(x) for x in g]
    hp = dict(HP[opt], v_nonzero=v_nonzero) if opt == "adamw" else HP[opt]
    run_parity(opt, thetas, grads, 3, hp, rho_bits, 0.01,
               f"{opt} rho{rho_bits}{' fp32' if fp32_grad else ''}{' vnz' if v_nonzero else ''}")
