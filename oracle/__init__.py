"""CPU oracle for the FlashOptim compressed optimizer step (test infrastructure).

This package wraps ``oracle.c`` -- a plain, slow, scalar FP32 restatement of
"FlashOptim: Optimizers for Memory Efficient Training" (weight splitting,
companded group quantization, the fused AdamW / SGD / Lion step) -- with
ctypes over numpy arrays. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it; the product library never does.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MOMENTUM = 0
VARIANCE = 1
MOMENTUM_LINEAR = 2   # group quantization without companding (Fig. 4's comparison)
VARIANCE_LINEAR = 3
VARIANCE_NONZERO = 5  # companded v, no code 0 where the group scale is non-zero (opt-in rule)
GROUP = 32

# -ffp-contract=off: no implicit fused multiply-add (gcc contracts by default on
# targets with FMA, e.g. aarch64); no -ffast-math: IEEE semantics throughout.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc if it is missing or older than its sources."""
    with _lock:
        stale = force or not os.path.exists(_LIB) or any(
            os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
        if stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
            os.replace(tmp, _LIB)
    return _LIB


class Tensor(ctypes.Structure):
    """Mirror of ``oracle_tensor_t`` (one row of the parameter table)."""
    _fields_ = [
        ("theta", ctypes.c_void_p),
        ("rho", ctypes.c_void_p),
        ("m_q", ctypes.c_void_p),
        ("m_scale", ctypes.c_void_p),
        ("v_q", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
        ("grad", ctypes.c_void_p),
        ("numel", ctypes.c_int64),
        ("weight_decay", ctypes.c_double),
        ("rho_bits", ctypes.c_int32),
        ("grad_is_f32", ctypes.c_int32),
    ]


class AdamWHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("v_nonzero", ctypes.c_int32), ("pad", ctypes.c_int32)]


class SGDHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("momentum", ctypes.c_double)]


class LionHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double)]


def lib() -> ctypes.CDLL:
    """The oracle library: ``liboracle.so``, or the build of a modified
    oracle.c that the environment variable ORACLE_LIB names (the mutation
    test points the pins at such builds)."""
    global _lib
    if _lib is None:
        l = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        f64 = ctypes.c_double
        u16 = ctypes.c_uint16
        sig = {
            "oracle_bf16_to_f32": (f32, [u16]),
            "oracle_bf16_rne": (u16, [f32]),
            "oracle_fp16_rne": (u16, [f32]),
            "oracle_fp16_to_f32": (f32, [u16]),
            "oracle_half_ulp": (f32, [u16, i32]),
            "oracle_phi_m": (f32, [f32]),
            "oracle_phi_m_inv": (f32, [f32]),
            "oracle_phi_v": (f32, [f32]),
            "oracle_phi_v_inv": (f32, [f32]),
            "oracle_bf16_rne_n": (None, [vp, vp, i64]),
            "oracle_fp16_rne_n": (None, [vp, vp, i64]),
            "oracle_fp16_to_f32_n": (None, [vp, vp, i64]),
            "oracle_half_ulp_n": (None, [vp, i32, vp, i64]),
            "oracle_phi_n": (None, [vp, vp, i64, i32]),
            "oracle_split": (None, [vp, vp, vp, i64, i32]),
            "oracle_merge": (None, [vp, vp, vp, i64, i32]),
            "oracle_quant_state": (None, [vp, vp, vp, i64, i32]),
            "oracle_dequant_state": (None, [vp, vp, vp, i64, i32]),
            "oracle_adamw_step": (i32, [vp, ctypes.c_int32, vp, i64]),
            "oracle_sgd_step": (i32, [vp, ctypes.c_int32, vp]),
            "oracle_lion_step": (i32, [vp, ctypes.c_int32, vp]),
            "oracle_adamw_update_fp32": (None, [vp, vp, vp, vp, i64, vp, i64, f64]),
            "oracle_sgd_update_fp32": (None, [vp, vp, vp, i64, vp, f64]),
            "oracle_lion_update_fp32": (None, [vp, vp, vp, i64, vp, f64]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _ptr(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    assert a.flags.c_contiguous, "oracle buffers must be C-contiguous"
    return a.ctypes.data


def _rho_dtype(rho_bits: int):
    return np.int16 if rho_bits == 16 else np.int8


# --- scalar encodings -------------------------------------------------------

def bf16_rne(x: float) -> int:
    return lib().oracle_bf16_rne(x)


def fp16_rne(x: float) -> int:
    return lib().oracle_fp16_rne(x)


def fp16_to_f32(h: int) -> float:
    return lib().oracle_fp16_to_f32(h)


def half_ulp(theta_p_bits: int, direction: int) -> float:
    return lib().oracle_half_ulp(theta_p_bits, direction)


def phi_m(x: float) -> float:
    return lib().oracle_phi_m(x)


def phi_m_inv(z: float) -> float:
    return lib().oracle_phi_m_inv(z)


def phi_v(x: float) -> float:
    return lib().oracle_phi_v(x)


def phi_v_inv(z: float) -> float:
    return lib().oracle_phi_v_inv(z)


# --- array forms of the encodings --------------------------------------------

def bf16_rne_n(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_bf16_rne_n(_ptr(x), _ptr(out), x.size)
    return out


def fp16_rne_n(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_fp16_rne_n(_ptr(x), _ptr(out), x.size)
    return out


def fp16_to_f32_n(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().oracle_fp16_to_f32_n(_ptr(h), _ptr(out), h.size)
    return out


def half_ulp_n(theta_p: np.ndarray, direction: int) -> np.ndarray:
    theta_p = np.ascontiguousarray(theta_p, dtype=np.uint16)
    out = np.empty(theta_p.shape, np.float32)
    lib().oracle_half_ulp_n(_ptr(theta_p), direction, _ptr(out), theta_p.size)
    return out


_PHI = {"phi_m": 0, "phi_m_inv": 1, "phi_v": 2, "phi_v_inv": 3}


def phi_n(x: np.ndarray, which: str) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.float32)
    lib().oracle_phi_n(_ptr(x), _ptr(out), x.size, _PHI[which])
    return out


# --- array codecs -----------------------------------------------------------

def split(theta: np.ndarray, rho_bits: int = 8):
    theta = np.ascontiguousarray(theta, dtype=np.float32)
    tp = np.empty(theta.shape, np.uint16)
    rho = np.empty(theta.shape, _rho_dtype(rho_bits))
    lib().oracle_split(_ptr(theta), _ptr(tp), _ptr(rho), theta.size, rho_bits)
    return tp, rho


def merge(theta_p: np.ndarray, rho: np.ndarray, rho_bits: int = 8) -> np.ndarray:
    theta_p = np.ascontiguousarray(theta_p, dtype=np.uint16)
    rho = np.ascontiguousarray(rho, dtype=_rho_dtype(rho_bits))
    out = np.empty(theta_p.shape, np.float32)
    lib().oracle_merge(_ptr(theta_p), _ptr(rho), _ptr(out), theta_p.size, rho_bits)
    return out


def _code_dtype(kind: int):
    if kind not in (MOMENTUM, VARIANCE, MOMENTUM_LINEAR, VARIANCE_LINEAR, VARIANCE_NONZERO):
        raise ValueError(f"unknown state kind {kind}")
    return np.int8 if kind in (MOMENTUM, MOMENTUM_LINEAR) else np.uint8


def quant_state(x: np.ndarray, kind: int):
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.empty(x.shape, _code_dtype(kind))
    scales = np.empty((x.size + GROUP - 1) // GROUP, np.uint16)
    lib().oracle_quant_state(_ptr(x), _ptr(q), _ptr(scales), x.size, kind)
    return q, scales


def dequant_state(q: np.ndarray, scales: np.ndarray, kind: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=_code_dtype(kind))
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    out = np.empty(q.shape, np.float32)
    lib().oracle_dequant_state(_ptr(q), _ptr(scales), _ptr(out), q.size, kind)
    return out


# --- compressed state and fused steps ----------------------------------------

class State:
    """Compressed per-tensor state held in numpy arrays (host memory)."""

    def __init__(self, theta_p, rho, m_q, m_scale, v_q=None, v_scale=None,
                 weight_decay=0.0, rho_bits=8):
        self.theta_p = np.ascontiguousarray(theta_p, dtype=np.uint16)
        self.rho = np.ascontiguousarray(rho, dtype=_rho_dtype(rho_bits))
        self.m_q = np.ascontiguousarray(m_q, dtype=np.int8)
        self.m_scale = np.ascontiguousarray(m_scale, dtype=np.uint16)
        self.v_q = None if v_q is None else np.ascontiguousarray(v_q, dtype=np.uint8)
        self.v_scale = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.uint16)
        self.weight_decay = float(weight_decay)
        self.rho_bits = int(rho_bits)

    @property
    def numel(self) -> int:
        return self.theta_p.size

    @classmethod
    def from_fp32(cls, theta: np.ndarray, rho_bits=8, with_v=True, weight_decay=0.0):
        """Initial state: theta', rho = split(theta0); zero codes and zero scales."""
        tp, rho = split(theta, rho_bits)
        n = tp.size
        ng = (n + GROUP - 1) // GROUP
        return cls(tp, rho, np.zeros(n, np.int8), np.zeros(ng, np.uint16),
                   np.zeros(n, np.uint8) if with_v else None,
                   np.zeros(ng, np.uint16) if with_v else None,
                   weight_decay, rho_bits)

    def copy(self) -> "State":
        c = lambda a: None if a is None else a.copy()
        return State(c(self.theta_p), c(self.rho), c(self.m_q), c(self.m_scale), c(self.v_q),
                     c(self.v_scale), self.weight_decay, self.rho_bits)

    def row(self, grad: np.ndarray) -> Tensor:
        """A table row over this state; grad is BF16 bit patterns (uint16) or float32."""
        assert grad.dtype in (np.uint16, np.float32), grad.dtype
        assert grad.size == self.numel and grad.flags.c_contiguous
        return Tensor(_ptr(self.theta_p), _ptr(self.rho), _ptr(self.m_q), _ptr(self.m_scale),
                      _ptr(self.v_q), _ptr(self.v_scale), _ptr(grad), self.numel,
                      self.weight_decay, self.rho_bits, int(grad.dtype == np.float32))


def _table(states, grads):
    rows = (Tensor * max(1, len(states)))()
    for i, (s, g) in enumerate(zip(states, grads)):
        rows[i] = s.row(g)
    return rows


def adamw_step(states, grads, lr, beta1, beta2, eps, step: int, v_nonzero: bool = False):
    """One fused FlashAdamW step over the list of states (updated in place);
    v_nonzero selects the opt-in rule that keeps a non-zero v off code 0."""
    hp = AdamWHparams(lr, beta1, beta2, eps, int(v_nonzero), 0)
    rc = lib().oracle_adamw_step(_table(states, grads), len(states), ctypes.byref(hp), step)
    if rc != 0:
        raise ValueError("oracle_adamw_step: bad argument")


def sgd_step(states, grads, lr, momentum):
    hp = SGDHparams(lr, momentum)
    rc = lib().oracle_sgd_step(_table(states, grads), len(states), ctypes.byref(hp))
    if rc != 0:
        raise ValueError("oracle_sgd_step: bad argument")


def lion_step(states, grads, lr, beta1, beta2):
    hp = LionHparams(lr, beta1, beta2)
    rc = lib().oracle_lion_step(_table(states, grads), len(states), ctypes.byref(hp))
    if rc != 0:
        raise ValueError("oracle_lion_step: bad argument")


def adamw_update_fp32(theta, m, v, g, lr, beta1, beta2, eps, step, weight_decay):
    """The AdamW element update on uncompressed FP32 arrays (in place)."""
    hp = AdamWHparams(lr, beta1, beta2, eps, 0, 0)
    g = np.ascontiguousarray(g, dtype=np.float32)
    lib().oracle_adamw_update_fp32(_ptr(theta), _ptr(m), _ptr(v), _ptr(g), theta.size,
                                   ctypes.byref(hp), step, weight_decay)


def sgd_update_fp32(theta, m, g, lr, momentum, weight_decay):
    hp = SGDHparams(lr, momentum)
    g = np.ascontiguousarray(g, dtype=np.float32)
    lib().oracle_sgd_update_fp32(_ptr(theta), _ptr(m), _ptr(g), theta.size, ctypes.byref(hp),
                                 weight_decay)


def lion_update_fp32(theta, m, g, lr, beta1, beta2, weight_decay):
    hp = LionHparams(lr, beta1, beta2)
    g = np.ascontiguousarray(g, dtype=np.float32)
    lib().oracle_lion_update_fp32(_ptr(theta), _ptr(m), _ptr(g), theta.size, ctypes.byref(hp),
                                  weight_decay)
