"""Out-of-bounds write detection without a sanitizer.

Every array a call writes is a view into a larger buffer filled with the byte
0xA5, with guard regions before and after it. After the call, the view must
hold the oracle's result and every guard byte must still be 0xA5: a kernel
that wrote one element too many (or too few) fails here. Covered: the codecs
on ragged sizes, and the fused step on ragged tables with short tiles and on
one long row with long tiles.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import fo
from quantized_optimizer_state_gb300 import workloads as wl
from tests.gpu_helpers import assert_state_matches, to_dev, to_host

pytestmark = pytest.mark.gpu

POISON = 0xA5
PRE = 256      # guard bytes before each view (a multiple of 16: views stay aligned)
POST = 256     # guard bytes after it
RAGGED = [1, 31, 33, 1000, 4097, 65539]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


class Guarded:
    """A device view of n elements of dtype inside a poisoned byte buffer."""

    def __init__(self, n, dtype, init=None):
        esize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = n * esize
        self.raw = torch.full((PRE + self.nbytes + POST,), POISON, dtype=torch.uint8, device="cuda")
        self.view = self.raw[PRE:PRE + self.nbytes].view(dtype)
        if init is not None:
            self.view.copy_(init)

    def guards_intact(self):
        g = torch.cat([self.raw[:PRE], self.raw[PRE + self.nbytes:]])
        return bool((g == POISON).all().item())


def _host(view, np_dtype):
    return to_host(view).view(np_dtype) if view.dtype != torch.float32 else to_host(view)


@pytest.mark.parametrize("rho_bits", [8, 16])
@pytest.mark.parametrize("n", RAGGED)
def test_split_and_merge_stay_in_bounds(n, rho_bits):
    rng = np.random.default_rng(n + rho_bits)
    theta = (rng.standard_normal(n) * 0.02).astype(np.float32)
    rdt = torch.int16 if rho_bits == 16 else torch.int8
    tp, rho = Guarded(n, torch.int16), Guarded(n, rdt)
    fo.fo_split(to_dev(theta), tp.view, rho.view, rho_bits)
    back = Guarded(n, torch.float32)
    fo.fo_merge(tp.view, rho.view, back.view, rho_bits)
    torch.cuda.synchronize()
    tp_ref, rho_ref = oracle.split(theta, rho_bits)
    assert np.array_equal(_host(tp.view, np.uint16), tp_ref)
    assert np.array_equal(_host(rho.view, rho_ref.dtype), rho_ref)
    assert np.array_equal(to_host(back.view), oracle.merge(tp_ref, rho_ref, rho_bits))
    assert tp.guards_intact() and rho.guards_intact() and back.guards_intact()


@pytest.mark.parametrize("kind", [fo.FO_STATE_MOMENTUM, fo.FO_STATE_VARIANCE, fo.FO_STATE_MOMENTUM_LINEAR,
                                  fo.FO_STATE_VARIANCE_LINEAR, fo.FO_STATE_VARIANCE_NONZERO])
@pytest.mark.parametrize("n", RAGGED)
def test_quant_and_dequant_stay_in_bounds(n, kind):
    rng = np.random.default_rng(n * 7 + kind)
    x = (rng.standard_t(3, n) * 1e-3).astype(np.float32)
    if kind in (fo.FO_STATE_VARIANCE, fo.FO_STATE_VARIANCE_LINEAR, fo.FO_STATE_VARIANCE_NONZERO):
        x = (x * x).astype(np.float32)
    signed = kind in (fo.FO_STATE_MOMENTUM, fo.FO_STATE_MOMENTUM_LINEAR)
    q = Guarded(n, torch.int8 if signed else torch.uint8)
    s = Guarded((n + 31) // 32, torch.int16)
    fo.fo_quant_state(to_dev(x), q.view, s.view, kind)
    out = Guarded(n, torch.float32)
    fo.fo_dequant_state(q.view, s.view, out.view, kind)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_state(x, kind)
    assert np.array_equal(_host(q.view, q_ref.dtype), q_ref)
    assert np.array_equal(_host(s.view, np.uint16), s_ref)
    assert np.array_equal(to_host(out.view), oracle.dequant_state(q_ref, s_ref, kind))
    assert q.guards_intact() and s.guards_intact() and out.guards_intact()


class GuardedState:
    """A row's compressed state, every array a guarded view, filled from an
    oracle state."""

    def __init__(self, st):
        n, ng = st.numel, (st.numel + 31) // 32
        rdt = torch.int16 if st.rho_bits == 16 else torch.int8
        self.st = st
        self.theta = Guarded(n, torch.int16, to_dev(st.theta_p))
        self.rho = Guarded(n, rdt, to_dev(st.rho))
        self.m_q = Guarded(n, torch.int8, to_dev(st.m_q))
        self.m_scale = Guarded(ng, torch.int16, to_dev(st.m_scale))
        self.with_v = st.v_q is not None
        if self.with_v:
            self.v_q = Guarded(n, torch.uint8, to_dev(st.v_q))
            self.v_scale = Guarded(ng, torch.int16, to_dev(st.v_scale))

    def arrays(self):
        a = [self.theta, self.rho, self.m_q, self.m_scale]
        return a + ([self.v_q, self.v_scale] if self.with_v else [])

    def row(self, grad):
        return fo.row(self.theta.view, self.rho.view, self.m_q.view, self.m_scale.view, grad,
                      self.v_q.view if self.with_v else None, self.v_scale.view if self.with_v else None,
                      self.st.weight_decay, self.st.rho_bits, self.st.numel)

    def as_oracle(self):
        st = self.st
        return oracle.State(_host(self.theta.view, np.uint16), _host(self.rho.view, st.rho.dtype),
                            _host(self.m_q.view, np.int8), _host(self.m_scale.view, np.uint16),
                            _host(self.v_q.view, np.uint8) if self.with_v else None,
                            _host(self.v_scale.view, np.uint16) if self.with_v else None,
                            st.weight_decay, st.rho_bits)


def _step(opt, table, t):
    if opt == "adamw":
        fo.fo_adamw_step(table, 1e-3, 0.9, 0.999, 1e-8, t)
    elif opt == "sgd":
        fo.fo_sgd_step(table, 0.1, 0.9)
    else:
        fo.fo_lion_step(table, 1e-4, 0.9, 0.99)


def _oracle_step(opt, states, grads, t):
    if opt == "adamw":
        oracle.adamw_step(states, grads, 1e-3, 0.9, 0.999, 1e-8, t)
    elif opt == "sgd":
        oracle.sgd_step(states, grads, 0.1, 0.9)
    else:
        oracle.lion_step(states, grads, 1e-4, 0.9, 0.99)


@pytest.mark.parametrize("opt", ["adamw", "sgd", "lion"])
@pytest.mark.parametrize("rho_bits", [8, 16])
def test_fused_step_stays_in_bounds(opt, rho_bits):
    """A ragged table (short tiles): two steps, every row's arrays guarded."""
    rng = np.random.default_rng(rho_bits * 3 + len(opt))
    thetas = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in RAGGED]
    ref = [oracle.State.from_fp32(t, rho_bits, opt == "adamw", 0.01) for t in thetas]
    dev = [GuardedState(r.copy()) for r in ref]
    for t in (1, 2):
        grads = [wl.to_bf16_bits((rng.standard_t(3, n) * 1e-3).astype(np.float32)) for n in RAGGED]
        gdev = [to_dev(g) for g in grads]     # held until the step has run
        _step(opt, fo.Table([d.row(gd) for d, gd in zip(dev, gdev)]), t)
        _oracle_step(opt, ref, grads, t)
        torch.cuda.synchronize()
        for i, (d, r) in enumerate(zip(dev, ref)):
            assert_state_matches(d.as_oracle(), r, f"{opt} rho{rho_bits} step {t} row {i}")
            assert all(a.guards_intact() for a in d.arrays()), (opt, rho_bits, t, i)


LONG_N = 5 * (1 << 25) + 37   # long tiles for every optimizer on 152 SMs; a ragged last tile


@pytest.mark.parametrize("opt", ["adamw", "lion"])
def test_long_tile_step_stays_in_bounds(opt):
    """One row long enough for the long-tile launch: guards intact after a
    step, and the last 4133 elements (whole groups up to a ragged end) equal
    the oracle's step of those groups alone."""
    n = LONG_N
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    with_v = opt == "adamw"
    tp = torch.empty(n, dtype=torch.int16, device="cuda")
    rho = torch.empty(n, dtype=torch.int8, device="cuda")
    fo.fo_split(torch.randn(n, device="cuda", generator=gen) * 0.02, tp, rho, 8)
    zeros_g = np.zeros(((n + 31) // 32,), np.uint16)
    st = oracle.State(to_host(tp), to_host(rho, np.int8), np.zeros(n, np.int8), zeros_g,
                      np.zeros(n, np.uint8) if with_v else None, zeros_g.copy() if with_v else None, 0.01, 8)
    del tp, rho
    d = GuardedState(st)
    g = (torch.randn(n, device="cuda", generator=gen) * 1e-3).to(torch.bfloat16)
    tail = n - 4096 - 37          # a group boundary
    cut = lambda a, k=1: None if a is None else a[tail // k:].copy()
    ref = oracle.State(cut(st.theta_p), cut(st.rho), cut(st.m_q), cut(st.m_scale, 32), cut(st.v_q),
                       cut(st.v_scale, 32), 0.01, 8)
    _step(opt, fo.Table([d.row(g)]), 1)
    _oracle_step(opt, [ref], [to_host(g[tail:].view(torch.int16))], 1)
    torch.cuda.synchronize()
    got = d.as_oracle()
    got_tail = oracle.State(cut(got.theta_p), cut(got.rho), cut(got.m_q), cut(got.m_scale, 32),
                            cut(got.v_q), cut(got.v_scale, 32), 0.01, 8)
    assert_state_matches(got_tail, ref, f"{opt} long row tail")
    assert all(a.guards_intact() for a in d.arrays())
