"""AdamW with the step counter in device memory (fo_adamw_step_dev) and the
drop-in FlashAdamW(capturable=True) built on it.

The bias corrections depend on the step count t (page section
"融合优化器步骤": the standard AdamW update). fo_adamw_step takes t from the
host, so a step captured in a CUDA graph would replay its captured t; the
device-counter variant reads t when the kernel runs. It must give exactly
the host-counter result for every t, and replays must advance t.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import fo
from quantized_optimizer_state_gb300 import optim
from quantized_optimizer_state_gb300 import workloads as wl
from tests.gpu_helpers import assert_state_matches, device_state_from_oracle, oracle_state_from_device, to_dev

pytestmark = pytest.mark.gpu

ADAMW = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)
SIZES = [1, 33, 1000, 4097, 65539, 300000]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fo.lib()
    oracle.build()


def _states(seed, rho_bits=8):
    rng = np.random.default_rng(seed)
    host = [oracle.State.from_fp32((rng.standard_normal(n) * 0.02).astype(np.float32), rho_bits, True, 0.01)
            for n in SIZES]
    return host


def _grads(seed, t, fp32=False):
    r = np.random.default_rng(seed * 1000 + t)
    g = [(r.standard_t(3, n) * 1e-3).astype(np.float32) for n in SIZES]
    return g if fp32 else [wl.to_bf16_bits(x) for x in g]


@pytest.mark.parametrize("hp,rho_bits,fp32,v_nonzero", [
    (ADAMW, 8, False, False),
    (ADAMW, 16, True, True),
    (dict(ADAMW, beta2=0.99999), 8, False, False),    # 1/sqrt(bc2) > 2^8 at small t: the IEEE path
    (dict(ADAMW, beta1=0.0, lr=0.0), 8, False, False),
])
def test_device_counter_equals_host_counter(hp, rho_bits, fp32, v_nonzero):
    """For every t (small, large, beyond the point where b^t underflows), the
    device-counter call leaves exactly the state the host-counter call does."""
    host = _states(1, rho_bits)
    # warm both copies up with a few ordinary steps so that the state is not zero
    a = [device_state_from_oracle(h) for h in host]
    for t in (1, 2, 3):
        g = [to_dev(x) for x in _grads(1, t, fp32)]
        fo.fo_adamw_step(fo.table_of(a, g), hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], t, v_nonzero=v_nonzero)
    counter = torch.zeros((), dtype=torch.int64, device="cuda")
    for t in (1, 2, 4, 5, 17, 1000, 123457, 1 << 40):
        snap = [oracle_state_from_device(d) for d in a]
        b = [device_state_from_oracle(h) for h in snap]
        g = [to_dev(x) for x in _grads(2, t % 1000, fp32)]
        fo.fo_adamw_step(fo.table_of(a, g), hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], t, v_nonzero=v_nonzero)
        counter.fill_(t)
        fo.fo_adamw_step_dev(fo.table_of(b, g), hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], counter,
                             v_nonzero=v_nonzero)
        torch.cuda.synchronize()
        for x, y in zip(a, b):
            for p, q in zip(x.buffers(), y.buffers()):
                assert torch.equal(p, q), f"t={t}"


def test_counter_below_one_updates_nothing():
    host = _states(3)
    d = [device_state_from_oracle(h) for h in host]
    before = [[x.clone() for x in s.buffers()] for s in d]
    g = [to_dev(x) for x in _grads(3, 1)]
    for t in (0, -5):
        counter = torch.full((), t, dtype=torch.int64, device="cuda")
        fo.fo_adamw_step_dev(fo.table_of(d, g), 1e-3, 0.9, 0.999, 1e-8, counter)
    torch.cuda.synchronize()
    for s, b in zip(d, before):
        for x, y in zip(s.buffers(), b):
            assert torch.equal(x, y)


def test_graph_replay_advances_the_counter():
    """[counter += 1; fo_adamw_step_dev] captured once, replayed three times
    with new gradients copied into the captured gradient buffers: the same as
    three oracle steps with t = 1, 2, 3."""
    host = _states(4)
    dev = [device_state_from_oracle(h) for h in host]
    gbuf = [torch.zeros(n, dtype=torch.int16, device="cuda") for n in SIZES]
    counter = torch.zeros((), dtype=torch.int64, device="cuda")
    table = fo.table_of(dev, gbuf)
    # warm-up outside the capture (loads the kernel): a counter of 0 updates nothing
    fo.fo_adamw_step_dev(table, 1e-3, 0.9, 0.999, 1e-8, counter)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            counter.add_(1)
            fo.fo_adamw_step_dev(table, 1e-3, 0.9, 0.999, 1e-8, counter, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    assert int(counter.item()) == 0            # capture ran nothing
    ref = [h.copy() for h in host]
    for t in (1, 2, 3):
        g = _grads(4, t)
        for buf, x in zip(gbuf, g):
            buf.copy_(to_dev(x))
        graph.replay()
        oracle.adamw_step(ref, g, 1e-3, 0.9, 0.999, 1e-8, t)
        torch.cuda.synchronize()
        for d, r in zip(dev, ref):
            assert_state_matches(oracle_state_from_device(d), r, f"replay {t}")
    assert int(counter.item()) == 3


def _params(seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.nn.Parameter((torch.randn(s, generator=g) * 0.02).cuda()) for s in [(64, 33), (1000,), (7,)]]


def test_capturable_flash_adamw_matches_and_replays():
    """FlashAdamW(capturable=True) steps exactly like FlashAdamW(); its step()
    captured in a CUDA graph and replayed continues the same trajectory."""
    pa, pb, pc = _params(5), _params(5), _params(5)
    oa = optim.FlashAdamW(pa, lr=1e-3)
    ob = optim.FlashAdamW(pb, lr=1e-3, capturable=True)
    oc = optim.FlashAdamW(pc, lr=1e-3, capturable=True)
    rng = np.random.default_rng(6)
    grads = [[torch.from_numpy(wl.to_bf16_bits((rng.standard_normal(p.numel()) * 1e-3).astype(np.float32))
                               .view(np.int16)).cuda().view(torch.bfloat16).view(p.shape) for p in pa]
             for _ in range(5)]
    for ps in (pa, pb, pc):
        for p, g in zip(ps, grads[0]):
            p.grad = g.clone()
    for step in range(2):                     # eager steps on all three
        for ps in (pa, pb, pc):
            for p, g in zip(ps, grads[step]):
                p.grad.copy_(g)
        oa.step()
        ob.step()
        oc.step()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            oc.step()
    torch.cuda.current_stream().wait_stream(side)
    for step in range(2, 5):
        for ps in (pa, pb, pc):
            for p, g in zip(ps, grads[step]):
                p.grad.copy_(g)
        oa.step()
        ob.step()
        graph.replay()
    torch.cuda.synchronize()
    for x, y, z in zip(pa, pb, pc):
        assert torch.equal(x.data, y.data) and torch.equal(x.data, z.data)
        for k in ("rho", "m_q", "m_scale", "v_q", "v_scale"):
            assert torch.equal(oa.state[x][k], ob.state[y][k])
            assert torch.equal(oa.state[x][k], oc.state[z][k])
    assert int(ob.state[pb[0]]["step"].item()) == 5 and int(oc.state[pc[0]]["step"].item()) == 5


@pytest.mark.parametrize("n", [6 * 1024 * 1024 + 77, 1 << 27])
def test_device_counter_on_long_and_short_tiles(n):
    """The device-counter kernels of the other two tile lengths (a table of a
    few million elements takes 2-chunk tiles, one of 2^27 8-chunk tiles):
    identical to the host-counter call."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(n % 1000)
    a = fo.CompressedTensor(n, "cuda", 8, True, 0.01)
    a.init_from(torch.randn(n, device="cuda", generator=gen) * 0.02)
    b = fo.CompressedTensor(n, "cuda", 8, True, 0.01)
    for x, y in zip(b.buffers(), a.buffers()):
        x.copy_(y)
    counter = torch.zeros((), dtype=torch.int64, device="cuda")
    for t in (1, 2, 3):
        g = (torch.randn(n, device="cuda", generator=gen) * 1e-3).to(torch.bfloat16)
        fo.fo_adamw_step(fo.table_of([a], [g]), 1e-3, 0.9, 0.999, 1e-8, t)
        counter.fill_(t)
        fo.fo_adamw_step_dev(fo.table_of([b], [g]), 1e-3, 0.9, 0.999, 1e-8, counter)
    torch.cuda.synchronize()
    for x, y in zip(a.buffers(), b.buffers()):
        assert torch.equal(x, y)
    del a, b
    torch.cuda.empty_cache()
