"""GPU parity of the fused compressed step (fo_adamw_step, fo_sgd_step,
fo_lion_step) against the CPU oracle, through the C ABI.

Page section "融合优化器步骤" (Algorithm 4). Parity is checked per step: the
oracle starts every step from the state the GPU produced at the previous one,
so a permitted +-1 code difference cannot compound. Inputs are the seeded
synthetic workloads of quantized_optimizer_state_gb300.workloads.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import fo
from quantized_optimizer_state_gb300 import workloads as wl
from tests.gpu_helpers import (assert_state_matches, device_state_from_oracle,
                               oracle_state_from_device, to_dev, to_host)

pytestmark = pytest.mark.gpu

ADAMW = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


def _make_states(thetas, opt, rho_bits, weight_decay):
    with_v = opt == "adamw"
    bits = rho_bits if isinstance(rho_bits, (list, tuple)) else [rho_bits] * len(thetas)
    host = [oracle.State.from_fp32(t, b, with_v, weight_decay) for t, b in zip(thetas, bits)]
    return [device_state_from_oracle(h) for h in host]


def _gpu_step(opt, dev_states, dev_grads, t, hp):
    table = fo.table_of(dev_states, dev_grads)
    if opt == "adamw":
        fo.fo_adamw_step(table, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], t,
                         v_nonzero=hp.get("v_nonzero", False))
    elif opt == "sgd":
        fo.fo_sgd_step(table, hp["lr"], hp["momentum"])
    else:
        fo.fo_lion_step(table, hp["lr"], hp["beta1"], hp["beta2"])
    torch.cuda.synchronize()


def _oracle_step(opt, states, grads, t, hp):
    if opt == "adamw":
        oracle.adamw_step(states, grads, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], t,
                          v_nonzero=hp.get("v_nonzero", False))
    elif opt == "sgd":
        oracle.sgd_step(states, grads, hp["lr"], hp["momentum"])
    else:
        oracle.lion_step(states, grads, hp["lr"], hp["beta1"], hp["beta2"])


def run_parity(opt, thetas, grads_of_step, steps, hp, rho_bits=8, weight_decay=0.01, what=""):
    """Per-step parity over `steps` steps; grads_of_step(t) -> list of BF16 arrays."""
    dev = _make_states(thetas, opt, rho_bits, weight_decay)
    total = sum(t.size for t in thetas)
    for t in range(1, steps + 1):
        grads = grads_of_step(t)
        ref = [oracle_state_from_device(d) for d in dev]
        _oracle_step(opt, ref, grads, t, hp)
        _gpu_step(opt, dev, [to_dev(g) for g in grads], t, hp)
        for i, d in enumerate(dev):
            assert_state_matches(oracle_state_from_device(d), ref[i], f"{what} step {t} tensor {i}", total)
    return dev


RAGGED = [1, 15, 16, 17, 31, 32, 33, 1000, 4095, 4096, 4097, 12345, 65539]


def _ragged_inputs(seed, scale=0.02):
    rng = np.random.default_rng(seed)
    thetas = [(rng.standard_normal(n) * scale).astype(np.float32) for n in RAGGED]

    def grads(t):
        r = np.random.default_rng(seed * 1000 + t)
        return [wl.to_bf16_bits((r.standard_t(3, n) * 1e-3).astype(np.float32)) for n in RAGGED]
    return thetas, grads


@pytest.mark.parametrize("rho_bits", [8, 16, (8, 16)])
def test_adamw_ragged_table(rho_bits):
    thetas, grads = _ragged_inputs(1)
    bits = rho_bits if isinstance(rho_bits, int) else [rho_bits[i % 2] for i in range(len(thetas))]
    run_parity("adamw", thetas, grads, 5, ADAMW, bits, 0.01, "adamw ragged")


def test_sgd_ragged_table():
    thetas, grads = _ragged_inputs(2, 0.05)
    run_parity("sgd", thetas, grads, 5, dict(lr=0.1, momentum=0.9), 8, 1e-4, "sgd ragged")


def test_lion_ragged_table():
    thetas, grads = _ragged_inputs(3)
    run_parity("lion", thetas, grads, 5, dict(lr=1e-4, beta1=0.9, beta2=0.99), 8, 0.01, "lion ragged")


def _workload_inputs(w):
    thetas = [wl.init_weight(p, i) for i, p in enumerate(w.params)]

    def grads(t):
        return [wl.grad_bf16(w.grad, w.grad_scale, p.numel, i, t) for i, p in enumerate(w.params)]
    return thetas, grads


def _hp(w):
    hp = dict(w.hparams)
    wd = hp.pop("weight_decay")
    return hp, wd


def test_flat_1m_adamw_all_steps():
    w = wl.workload("flat_1m")
    thetas, grads = _workload_inputs(w)
    hp, wd = _hp(w)
    run_parity("adamw", thetas, grads, w.steps, hp, w.rho_bits, wd, "flat_1m")


def test_gpt2_small_adamw():
    w = wl.workload("gpt2_small")
    thetas, grads = _workload_inputs(w)
    hp, wd = _hp(w)
    run_parity("adamw", thetas, grads, 2, hp, w.rho_bits, wd, "gpt2_small")


def test_resnet50_sgd():
    w = wl.workload("resnet50")
    thetas, grads = _workload_inputs(w)
    hp, wd = _hp(w)
    run_parity("sgd", thetas, grads, 3, hp, w.rho_bits, wd, "resnet50")


@pytest.mark.parametrize("rho_bits", [8, 16])
def test_stress_64m_adamw(rho_bits):
    w = wl.workload("stress_64m", rho_bits)
    thetas, grads = _workload_inputs(w)
    hp, wd = _hp(w)
    run_parity("adamw", thetas, grads, 2, hp, rho_bits, wd, f"stress_64m rho{rho_bits}")


def test_many_rows_span_several_launches():
    """More rows than one launch's parameter space holds (and empty rows)."""
    rng = np.random.default_rng(5)
    sizes = [int(s) for s in rng.integers(1, 3000, 900)]
    sizes[10] = 0
    sizes[500] = 0
    thetas = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]

    def grads(t):
        r = np.random.default_rng(100 + t)
        return [wl.to_bf16_bits((r.standard_normal(n) * 1e-3).astype(np.float32)) for n in sizes]
    before = fo.fo_kernel_launch_count()
    run_parity("adamw", thetas, grads, 2, ADAMW, 8, 0.01, "900 rows")
    assert fo.fo_kernel_launch_count() - before == 2 * 3      # ceil(898 / 384) launches per step


def test_empty_table_is_a_no_op():
    before = fo.fo_kernel_launch_count()
    fo.fo_adamw_step(fo.Table([]), 1e-3, 0.9, 0.999, 1e-8, 1)
    assert fo.fo_kernel_launch_count() == before


def test_misaligned_slice_is_rejected():
    d = fo.CompressedTensor(1024, "cuda", 8, True, 0.0)
    g = torch.zeros(1024 + 8, dtype=torch.bfloat16, device="cuda")
    bad = fo.row(d.theta, d.rho, d.m_q, d.m_scale, g[1:1025], d.v_q, d.v_scale, 0.0, 8, 1024)
    with pytest.raises(fo.FoError) as e:
        fo.fo_adamw_step(fo.Table([bad]), 1e-3, 0.9, 0.999, 1e-8, 1)
    assert e.value.status == 2


def test_resume_from_buffers_is_bit_identical():
    """A checkpoint is the compressed buffers plus the step counter."""
    thetas, grads = _ragged_inputs(7)
    a = _make_states(thetas, "adamw", 8, 0.01)
    for t in (1, 2, 3):
        _gpu_step("adamw", a, [to_dev(g) for g in grads(t)], t, ADAMW)
    saved = [[b.clone().cpu() for b in d.buffers()] for d in a]
    for t in (4, 5):
        _gpu_step("adamw", a, [to_dev(g) for g in grads(t)], t, ADAMW)
    b = _make_states(thetas, "adamw", 8, 0.01)
    for d, bufs in zip(b, saved):
        for dst, src in zip(d.buffers(), bufs):
            dst.copy_(src.cuda())
    for t in (4, 5):
        _gpu_step("adamw", b, [to_dev(g) for g in grads(t)], t, ADAMW)
    for x, y in zip(a, b):
        for p, q in zip(x.buffers(), y.buffers()):
            assert torch.equal(p, q)


def _chunk_state(d: fo.CompressedTensor, lo: int, hi: int) -> oracle.State:
    """Host copy of elements [lo, hi) (lo, hi multiples of 32, or hi = numel)."""
    g0, g1 = lo // 32, (hi + 31) // 32
    sl = slice(lo, hi)
    rho = to_host(d.rho[sl], np.int16 if d.rho_bits == 16 else np.int8)
    return oracle.State(to_host(d.theta[sl]), rho, to_host(d.m_q[sl], np.int8),
                        to_host(d.m_scale[g0:g1]),
                        None if d.v_q is None else to_host(d.v_q[sl], np.uint8),
                        None if d.v_scale is None else to_host(d.v_scale[g0:g1]),
                        d.weight_decay, d.rho_bits)


def _grad_host(g: torch.Tensor) -> np.ndarray:
    """A device gradient slice as the oracle takes it: BF16 patterns or float32."""
    return to_host(g) if g.dtype == torch.float32 else to_host(g.view(torch.int16))


def _sampled_parity(opt, dev, grads_dev, samples, t, hp):
    """Run one GPU step over all rows; check sampled chunks against the oracle
    run on the same chunks' pre-step state (groups are independent)."""
    pre = [(i, lo, hi, _chunk_state(dev[i], lo, hi), _grad_host(grads_dev[i][lo:hi]))
           for i, lo, hi in samples]
    _gpu_step(opt, dev, grads_dev, t, hp)
    for i, lo, hi, st, g in pre:
        _oracle_step(opt, [st], [g], t, hp)
        assert_state_matches(_chunk_state(dev[i], lo, hi), st, f"row {i} [{lo},{hi}) step {t}")


def _samples_of(sizes, per_row=1 << 16, rows=None):
    out = []
    for i, n in enumerate(sizes):
        if rows is not None and i not in rows:
            continue
        if n <= 3 * per_row:
            out.append((i, 0, n))
        else:
            mid = (n // 2) // 32 * 32
            tail = max(0, (n - per_row) // 32 * 32)
            out += [(i, 0, per_row), (i, mid, mid + per_row), (i, tail, n)]
    return out


def _device_workload(w, grad_fp32=False):
    dev, grads = [], []
    gen = wl.grad_fp32_device if grad_fp32 else wl.grad_bf16_device
    for i, p in enumerate(w.params):
        d = fo.CompressedTensor(p.numel, "cuda", w.rho_bits, w.optimizer == "adamw",
                                w.hparams["weight_decay"])
        theta = wl.init_weight_device(p, i, "cuda")
        d.init_from(theta)
        del theta
        dev.append(d)
        grads.append(gen(w.grad, w.grad_scale, p.numel, i, 1, "cuda"))
    torch.cuda.synchronize()
    return dev, grads


@pytest.mark.parametrize("name", ["llama31_8b", "llama31_8b_lion"])
def test_llama31_8b_full_size_sampled(name):
    """The full 8.03e9-parameter table in one call (the benchmarked launch), for
    all five steps of the run, with every eighth row (and the first and last
    ones) sampled at its head, middle and tail and checked against the oracle."""
    w = wl.workload(name)
    dev, grads = _device_workload(w)
    hp, _ = _hp(w)
    rows = set(range(0, len(w.params), 8)) | {0, 1, 2, 3, 4, 5, 6, 7, len(w.params) - 2, len(w.params) - 1}
    samples = _samples_of([p.numel for p in w.params], rows=rows)
    for t in range(1, w.steps + 1):                # all 5 steps, a fresh gradient each
        if t > 1:
            for i in range(len(grads)):
                grads[i] = None
                grads[i] = wl.workload_grad_device(w, i, t, "cuda")
        _sampled_parity(w.optimizer, dev, grads, samples, t, hp)
    del dev, grads
    torch.cuda.empty_cache()


def test_tensor_larger_than_2_to_31_elements():
    n = (1 << 31) + 33
    d = fo.CompressedTensor(n, "cuda", 8, True, 0.01)
    theta = torch.randn(n, device="cuda") * 0.02
    d.init_from(theta)
    del theta
    g = (torch.randn(n, device="cuda") * 1e-3).to(torch.bfloat16)
    samples = [(0, 0, 1 << 16), (0, (1 << 31) - (1 << 15), (1 << 31) + (1 << 15)), (0, n - 4096 - 1, n)]
    samples = [(i, lo // 32 * 32, hi) for i, lo, hi in samples]
    _sampled_parity("adamw", [d], [g], samples, 1, ADAMW)
    del d, g
    torch.cuda.empty_cache()


def test_rows_may_share_a_gradient():
    """Gradients are only read: two rows stepped from one gradient tensor are
    accepted and each matches the oracle."""
    rng = np.random.default_rng(31)
    thetas = [(rng.standard_normal(5000) * 0.02).astype(np.float32) for _ in range(2)]
    dev = _make_states(thetas, "adamw", 8, 0.01)
    for t in (1, 2, 3):
        g = wl.to_bf16_bits((rng.standard_normal(5000) * 1e-3).astype(np.float32))
        gd = to_dev(g)
        ref = [oracle_state_from_device(d) for d in dev]
        _oracle_step("adamw", ref, [g, g], t, ADAMW)
        _gpu_step("adamw", dev, [gd, gd], t, ADAMW)          # one device tensor in both rows
        for i, d in enumerate(dev):
            assert_state_matches(oracle_state_from_device(d), ref[i], f"shared gradient step {t} row {i}")


def test_device_check_on_a_real_tensor(monkeypatch):
    d = fo.CompressedTensor(64, "cuda:0", 8, True, 0.0)
    g = torch.zeros(64, dtype=torch.bfloat16, device="cuda:0")
    with torch.cuda.device(0):
        assert fo.row(d.theta, d.rho, d.m_q, d.m_scale, g, d.v_q, d.v_scale).numel == 64
    monkeypatch.setattr(fo, "_current_device", lambda: 1)
    with pytest.raises(ValueError, match="current device"):
        fo.row(d.theta, d.rho, d.m_q, d.m_scale, g, d.v_q, d.v_scale)
