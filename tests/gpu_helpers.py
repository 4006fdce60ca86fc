"""Shared helpers of the GPU parity tests: device state <-> oracle state and the
comparison rules.

Comparison rules (the parity bar of the fused step):
  * theta' (BF16 patterns): bit-exact;
  * integer codes (rho, m, v): bit-exact, except at most +-1 LSB on at most
    1e-6 of the elements, where FP32 rounding can land on a code boundary;
  * FP16 scales: within 1e-6 relative (two distinct FP16 values differ by far
    more, so in practice bit-exact);
  * reconstructed FP32 weights: within 1e-6 relative.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from quantized_optimizer_state_gb300 import fo

DEV = "cuda"

_NP_OF_TORCH = {torch.int16: np.uint16, torch.int8: np.int8, torch.uint8: np.uint8,
                torch.float32: np.float32}


def to_dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    """Host numpy array -> device tensor with the same bytes."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    else:
        t = torch.from_numpy(a)
    return t.to(DEV)


def to_host(t: torch.Tensor, np_dtype=None) -> np.ndarray:
    a = t.detach().cpu().numpy()
    if np_dtype is not None:
        a = a.view(np_dtype)
    elif t.dtype == torch.int16:
        a = a.view(np.uint16)
    return a


def device_state_from_oracle(st: "oracle.State") -> fo.CompressedTensor:
    d = fo.CompressedTensor(st.numel, DEV, st.rho_bits, st.v_q is not None, st.weight_decay)
    d.theta.copy_(to_dev(st.theta_p))
    d.rho.copy_(to_dev(st.rho))
    d.m_q.copy_(to_dev(st.m_q))
    d.m_scale.copy_(to_dev(st.m_scale))
    if st.v_q is not None:
        d.v_q.copy_(to_dev(st.v_q))
        d.v_scale.copy_(to_dev(st.v_scale))
    return d


def oracle_state_from_device(d: fo.CompressedTensor) -> "oracle.State":
    rho = to_host(d.rho, np.int16 if d.rho_bits == 16 else np.int8)
    return oracle.State(to_host(d.theta), rho, to_host(d.m_q, np.int8), to_host(d.m_scale),
                        None if d.v_q is None else to_host(d.v_q, np.uint8),
                        None if d.v_scale is None else to_host(d.v_scale),
                        d.weight_decay, d.rho_bits)


def assert_codes(got: np.ndarray, ref: np.ndarray, what: str, n_total: int | None = None):
    got = got.astype(np.int64)
    ref = ref.astype(np.int64)
    d = got - ref
    nbad = int(np.count_nonzero(d))
    if nbad == 0:
        return 0
    n_total = n_total or got.size
    allowed = math.floor(1e-6 * n_total)
    idx = np.nonzero(d)[0][:8]
    assert np.abs(d).max() <= 1 and nbad <= allowed, (
        f"{what}: {nbad} mismatches (allowed {allowed} of +-1), first at {idx.tolist()}: "
        f"got {got[idx].tolist()} want {ref[idx].tolist()}")
    return nbad


def assert_exact(got: np.ndarray, ref: np.ndarray, what: str):
    if np.array_equal(got.view(np.uint8), ref.view(np.uint8)):
        return
    g = got.reshape(-1)
    r = ref.reshape(-1)
    idx = np.nonzero(g != r)[0][:8]
    raise AssertionError(f"{what}: {np.count_nonzero(g != r)} mismatches, first at {idx.tolist()}: "
                         f"got {g[idx].tolist()} want {r[idx].tolist()}")


def assert_scales(got: np.ndarray, ref: np.ndarray, what: str):
    g = got.view(np.float16).astype(np.float64)
    r = ref.view(np.float16).astype(np.float64)
    bad = np.abs(g - r) > 1e-6 * np.abs(r)
    assert not bad.any(), f"{what}: {int(bad.sum())} scales differ, first at {np.nonzero(bad)[0][:8].tolist()}"


def assert_state_matches(d: "oracle.State", ref: "oracle.State", what: str, n_total=None):
    """Compare a state read back from the device with the oracle's."""
    assert_exact(d.theta_p, ref.theta_p, what + " theta'")
    assert_codes(d.rho, ref.rho, what + " rho", n_total)
    assert_codes(d.m_q, ref.m_q, what + " m codes", n_total)
    assert_scales(d.m_scale, ref.m_scale, what + " m scales")
    if ref.v_q is not None:
        assert_codes(d.v_q, ref.v_q, what + " v codes", n_total)
        assert_scales(d.v_scale, ref.v_scale, what + " v scales")


def _chunks_of(st: "oracle.State", g: np.ndarray, chunk: int):
    """Group-aligned pieces of one state (views: the oracle updates them in place)."""
    n = st.numel
    out = []
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        g0, g1 = lo // 32, (hi + 31) // 32
        sub = oracle.State(st.theta_p[lo:hi], st.rho[lo:hi], st.m_q[lo:hi], st.m_scale[g0:g1],
                           None if st.v_q is None else st.v_q[lo:hi],
                           None if st.v_scale is None else st.v_scale[g0:g1],
                           st.weight_decay, st.rho_bits)
        out.append((sub, np.ascontiguousarray(g[lo:hi])))
    return out


_POOL = None


def oracle_step_parallel(opt: str, states, grads, t: int, hp: dict, chunk: int = 1 << 20):
    """One oracle step over large states, cut into group-aligned chunks that
    run on a thread per host core (groups are independent, so this equals one
    call over the whole table; the oracle itself is unchanged)."""
    import concurrent.futures as cf
    import os
    global _POOL
    if _POOL is None:
        _POOL = cf.ThreadPoolExecutor(max(1, len(os.sched_getaffinity(0))))
    pieces = [p for st, g in zip(states, grads) for p in _chunks_of(st, g, chunk)]
    if opt == "adamw":
        f = lambda p: oracle.adamw_step([p[0]], [p[1]], hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], t,
                                        v_nonzero=hp.get("v_nonzero", False))
    elif opt == "sgd":
        f = lambda p: oracle.sgd_step([p[0]], [p[1]], hp["lr"], hp["momentum"])
    else:
        f = lambda p: oracle.lion_step([p[0]], [p[1]], hp["lr"], hp["beta1"], hp["beta2"])
    list(_POOL.map(f, pieces))
