"""Drop-in optimizers (FlashAdamW, FlashSGD, FlashLion) over the C ABI.

They must produce exactly the oracle's compressed step (page sections
"融合优化器步骤" and "实践建议": drop-in, per-layer opt-out, gradient
release, compact checkpoints).
"""
import copy

import numpy as np
import pytest
import torch

import oracle
from quantized_optimizer_state_gb300 import optim
from quantized_optimizer_state_gb300 import workloads as wl
from tests.gpu_helpers import assert_state_matches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oracle.build()


SHAPES = [(64, 33), (33,), (128, 256), (1000,)]


def _params(seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.nn.Parameter((torch.randn(s, generator=g) * 0.02).cuda()) for s in SHAPES]


def _oracle_states(params_fp32, rho_bits, with_v, wd):
    return [oracle.State.from_fp32(p.detach().cpu().numpy().reshape(-1), rho_bits, with_v, wd)
            for p in params_fp32]


def _device_view(opt, p):
    st = opt.state[p]
    rho = st["rho"].cpu().numpy()
    return oracle.State(p.data.view(torch.int16).cpu().numpy().reshape(-1).view(np.uint16), rho,
                        st["m_q"].cpu().numpy(), st["m_scale"].cpu().numpy().view(np.uint16),
                        None if "v_q" not in st else st["v_q"].cpu().numpy(),
                        None if "v_scale" not in st else st["v_scale"].cpu().numpy().view(np.uint16),
                        0.0, 16 if rho.dtype == np.int16 else 8)


@pytest.mark.parametrize("kind,rho_bits", [("adamw", 8), ("adamw", 16), ("sgd", 8), ("lion", 8)])
def test_optimizer_matches_oracle(kind, rho_bits):
    params = _params(1)
    master0 = [p.detach().clone() for p in params]
    if kind == "adamw":
        opt = optim.FlashAdamW(params, lr=1e-3, weight_decay=0.01, rho_bits=rho_bits)
    elif kind == "sgd":
        opt = optim.FlashSGD(params, lr=0.1, momentum=0.9, weight_decay=1e-4, rho_bits=rho_bits)
    else:
        opt = optim.FlashLion(params, lr=1e-4, weight_decay=0.01, rho_bits=rho_bits)
    wd = {"adamw": 0.01, "sgd": 1e-4, "lion": 0.01}[kind]
    ref = _oracle_states(master0, rho_bits, kind == "adamw", wd)
    for p, r in zip(params, ref):           # split at construction
        assert p.dtype == torch.bfloat16
        assert np.array_equal(p.data.view(torch.int16).cpu().numpy().reshape(-1).view(np.uint16), r.theta_p)
    rng = np.random.default_rng(2)
    for t in range(1, 4):
        grads = [wl.to_bf16_bits((rng.standard_normal(p.numel()) * 1e-3).astype(np.float32)) for p in params]
        for p, gb in zip(params, grads):
            p.grad = torch.from_numpy(gb.view(np.int16)).cuda().view(torch.bfloat16).view(p.shape)
        opt.step()
        if kind == "adamw":
            oracle.adamw_step(ref, grads, 1e-3, 0.9, 0.999, 1e-8, t)
        elif kind == "sgd":
            oracle.sgd_step(ref, grads, 0.1, 0.9)
        else:
            oracle.lion_step(ref, grads, 1e-4, 0.9, 0.99)
        torch.cuda.synchronize()
        for p, r in zip(params, ref):
            assert_state_matches(_device_view(opt, p), r, f"{kind} step {t}")
    mw = opt.master_weights()
    for p, r in zip(params, ref):
        assert np.array_equal(mw[p].cpu().numpy().reshape(-1), oracle.merge(r.theta_p, r.rho, rho_bits))


def _model(seed):
    torch.manual_seed(seed)
    return torch.nn.Sequential(torch.nn.Linear(48, 96), torch.nn.GELU(), torch.nn.Linear(96, 7)).cuda()


def _train(model, opt, steps, release):
    g = torch.Generator(device="cuda").manual_seed(5)
    if release:
        opt.attach_grad_release()
    for _ in range(steps):
        x = torch.randn(64, 48, device="cuda", generator=g).to(torch.bfloat16)
        loss = model(x).float().square().mean()
        loss.backward()
        if not release:
            opt.step()
            opt.zero_grad(set_to_none=True)
    torch.cuda.synchronize()


def test_gradient_release_matches_plain_step():
    a, b = _model(3), _model(3)
    oa = optim.FlashAdamW(a.parameters(), lr=1e-3)
    ob = optim.FlashAdamW(b.parameters(), lr=1e-3)
    _train(a, oa, 4, release=False)
    _train(b, ob, 4, release=True)
    for pa, pb in zip(a.parameters(), b.parameters()):
        assert torch.equal(pa.data, pb.data)
        assert pb.grad is None
        for k in ("rho", "m_q", "m_scale", "v_q", "v_scale"):
            assert torch.equal(oa.state[pa][k], ob.state[pb][k])


def test_checkpoint_resume_is_bit_identical():
    a = _model(4)
    oa = optim.FlashAdamW(a.parameters(), lr=1e-3)
    _train(a, oa, 2, release=False)
    ckpt = {"model": {k: v.clone() for k, v in a.state_dict().items()},
            "opt": copy.deepcopy(oa.state_dict())}
    # compact: theta' (BF16) + rho + codes + scales, about 5 B per parameter
    n = sum(p.numel() for p in a.parameters())
    model_bytes = sum(v.numel() * v.element_size() for v in ckpt["model"].values())
    assert model_bytes == 2 * n
    assert oa.state_bytes() <= 3.125 * n + 64 * 6
    _train(a, oa, 3, release=False)
    b = _model(99)
    b.load_state_dict(ckpt["model"])
    ob = optim.FlashAdamW(b.parameters(), lr=1e-3)
    ob.load_state_dict(ckpt["opt"])
    _train(b, ob, 3, release=False)
    for pa, pb in zip(a.parameters(), b.parameters()):
        assert torch.equal(pa.data, pb.data)


def test_uncompressed_group_is_standard_adamw():
    torch.manual_seed(7)
    w1 = torch.nn.Parameter(torch.randn(300, device="cuda") * 0.02)
    w2 = torch.nn.Parameter(torch.randn(300, device="cuda") * 0.02)
    ref = torch.nn.Parameter(w2.detach().clone())
    opt = optim.FlashAdamW([{"params": [w1]}, {"params": [w2], "compress": False}], lr=1e-3)
    topt = torch.optim.AdamW([ref], lr=1e-3, weight_decay=0.01)
    for _ in range(3):
        g = torch.randn(300, device="cuda") * 1e-3
        w1.grad = g.to(torch.bfloat16)
        w2.grad = g.clone()
        ref.grad = g.clone()
        opt.step()
        topt.step()
    assert w2.dtype == torch.float32 and torch.equal(w2.data, ref.data)
    assert w1.dtype == torch.bfloat16


def test_cached_table_with_in_place_grads_and_changed_weight_decay():
    """Gradients written in place keep every pointer, so the step reuses its
    table; changing a group's weight decay between steps must still take
    effect. The second-moment floor is on. Checked against the oracle at
    every step."""
    params = _params(7)
    master0 = [p.detach().clone() for p in params]
    opt = optim.FlashAdamW(params, lr=1e-3, weight_decay=0.01, v_nonzero=True)
    ref = _oracle_states(master0, 8, True, 0.01)
    for p in params:
        p.grad = torch.zeros(p.shape, dtype=torch.bfloat16, device="cuda")
    rng = np.random.default_rng(8)
    for t in range(1, 5):
        if t == 3:
            opt.param_groups[0]["weight_decay"] = 0.1
            for r in ref:
                r.weight_decay = 0.1
        grads = [wl.to_bf16_bits((rng.standard_t(3, p.numel()) * 1e-3).astype(np.float32)) for p in params]
        for p, gb in zip(params, grads):
            p.grad.view(torch.int16).view(-1).copy_(torch.from_numpy(gb.view(np.int16)))
        opt.step()
        oracle.adamw_step(ref, grads, 1e-3, 0.9, 0.999, 1e-8, t, v_nonzero=True)
        torch.cuda.synchronize()
        for p, r in zip(params, ref):
            assert_state_matches(_device_view(opt, p), r, f"cached table step {t}")
    assert len(opt._tables) == 1


# Tensor.grad_dtype exists only in newer PyTorch; where it is missing that
# route does not exist, and the "step_params" route covers the FP32 path
FP32_ROUTES = ["step_params"] + (["grad_dtype"] if hasattr(torch.Tensor, "grad_dtype") else [])


@pytest.mark.parametrize("route", FP32_ROUTES)
@pytest.mark.parametrize("kind", ["adamw", "lion"])
def test_fp32_gradients_reach_the_step_unrounded(kind, route):
    """FP32 gradients of BF16 parameters must reach the step as FP32 (the
    oracle's FP32-gradient path), not rounded to BF16. Route "grad_dtype":
    autograd accumulates them with Tensor.grad_dtype = float32 (PyTorch
    versions that have it). Route "step_params": the same gradients handed to
    the optimizer's stepping code directly, so the FP32 path runs on any
    PyTorch. Negative control: the oracle fed the same gradients rounded to
    BF16 ends in another state."""
    params = _params(11)
    master0 = [p.detach().clone() for p in params]
    if kind == "adamw":
        opt = optim.FlashAdamW(params, lr=1e-3, weight_decay=0.01)
    else:
        opt = optim.FlashLion(params, lr=1e-4, weight_decay=0.01)
    ref = _oracle_states(master0, 8, kind == "adamw", 0.01)
    rounded = [r.copy() for r in ref]
    fp32_grads = {}
    if route == "grad_dtype":
        for p in params:
            p.grad_dtype = torch.float32
    else:
        opt._grad_of = lambda p: fp32_grads[id(p)]
    rng = np.random.default_rng(12)

    def oracle_step(states, grads, t):
        if kind == "adamw":
            oracle.adamw_step(states, grads, 1e-3, 0.9, 0.999, 1e-8, t)
        else:
            oracle.lion_step(states, grads, 1e-4, 0.9, 0.99)

    for t in range(1, 4):
        grads = [(rng.standard_t(3, p.numel()) * 1e-3).astype(np.float32) for p in params]
        for p, g in zip(params, grads):
            if route == "grad_dtype":
                p.grad = torch.from_numpy(g).cuda().view(p.shape)
                assert p.grad.dtype == torch.float32
            else:
                fp32_grads[id(p)] = torch.from_numpy(g).cuda()
        if route == "grad_dtype":
            opt.step()
        else:
            opt._step_params(params, opt.param_groups[0])
        oracle_step(ref, grads, t)
        oracle_step(rounded, [wl.to_bf16_bits(g) for g in grads], t)
        torch.cuda.synchronize()
        for p, r in zip(params, ref):
            assert_state_matches(_device_view(opt, p), r, f"{kind} fp32 grad step {t}")
    assert any(not np.array_equal(_device_view(opt, p).m_q, r.m_q) for p, r in zip(params, rounded))


@pytest.mark.parametrize("bucket", [0, 3000, 1 << 30])
def test_gradient_release_buckets_match_plain_step(bucket):
    """Release with every parameter stepped on its own (bucket 0), in buckets
    that fill during backward (3000 elements) and in one bucket stepped when
    backward ends: all equal the plain step bit for bit, and every gradient
    is freed."""
    a, b = _model(13), _model(13)
    oa = optim.FlashAdamW(a.parameters(), lr=1e-3)
    ob = optim.FlashAdamW(b.parameters(), lr=1e-3)
    _train(a, oa, 3, release=False)
    ob.attach_grad_release(bucket_numel=bucket)
    g = torch.Generator(device="cuda").manual_seed(5)
    for _ in range(3):
        x = torch.randn(64, 48, device="cuda", generator=g).to(torch.bfloat16)
        b(x).float().square().mean().backward()
        assert all(p.grad is None for p in b.parameters())
    torch.cuda.synchronize()
    for pa, pb in zip(a.parameters(), b.parameters()):
        assert torch.equal(pa.data, pb.data)
        assert ob.state[pb]["step"] == 3
        for k in ("rho", "m_q", "m_scale", "v_q", "v_scale"):
            assert torch.equal(oa.state[pa][k], ob.state[pb][k])


def test_failed_call_leaves_step_counters_unchanged():
    from quantized_optimizer_state_gb300 import fo
    params = _params(21)
    opt = optim.FlashAdamW(params, lr=1e-3)
    for p in params:
        p.grad = torch.zeros(p.shape, dtype=torch.bfloat16, device="cuda")

    def refuse(table, group, t):
        raise fo.FoError("fo_adamw_step", 4, "refused")

    opt._launch = refuse
    with pytest.raises(fo.FoError):
        opt.step()
    assert all(opt.state[p]["step"] == 0 for p in params)
    del opt._launch
    opt.step()
    assert all(opt.state[p]["step"] == 1 for p in params)


def test_cached_table_does_not_keep_gradients_alive():
    """The optimizer reuses its tables across steps, but a table must not hold
    the step's gradients: freeing them after the step frees their memory."""
    import gc
    import weakref
    params = _params(22)
    opt = optim.FlashAdamW(params, lr=1e-3)
    for p in params:
        p.grad = torch.zeros(p.shape, dtype=torch.bfloat16, device="cuda")
    refs = [weakref.ref(p.grad) for p in params]
    opt.step()
    opt.zero_grad(set_to_none=True)
    gc.collect()
    assert all(r() is None for r in refs)
