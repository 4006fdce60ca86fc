"""Thin ctypes binding of ``libfo.so`` (declared in ``include/fo.h``).

The functions keep the C names and only marshal arguments: torch tensors (or
raw integer device addresses) become pointers, a torch stream becomes its
``cudaStream_t``. Every computation runs in the library's CUDA kernels; if
the library cannot be loaded the call raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import threading
from typing import Iterable, List, Optional, Sequence

from . import build as _build

GROUP = 32
GRAD_BF16 = 0   # fo_grad_dtype_t
GRAD_F32 = 1
FO_STATE_MOMENTUM = 0
FO_STATE_VARIANCE = 1
FO_STATE_MOMENTUM_LINEAR = 2   # group quantization without companding (quality studies)
FO_STATE_VARIANCE_LINEAR = 3
FO_STATE_VARIANCE_NONZERO = 5  # companded v; no code 0 where the group scale is non-zero (opt-in rule)
FO_ADAMW_V_NONZERO = 1         # fo_adamw_hparams_t.flags: requantize v with that rule
FO_MAX_TENSORS = 1 << 20

STATUS = {0: "FO_OK", 1: "FO_ERR_NULL", 2: "FO_ERR_MISALIGNED", 3: "FO_ERR_SIZE",
          4: "FO_ERR_BAD_ARG", 5: "FO_ERR_TOO_MANY_TENSORS", 6: "FO_ERR_CUDA", 7: "FO_ERR_ALIAS"}


class FoError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {message} (status {status})")
        self.status = status


class FoTensor(ctypes.Structure):
    """Mirror of ``fo_tensor_t``."""
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
        ("grad_dtype", ctypes.c_int32),
    ]


class AdamWHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class SGDHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("momentum", ctypes.c_double)]


class LionHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double)]


assert ctypes.sizeof(FoTensor) == 80

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

# symbol -> (restype, argtypes), exactly the functions include/fo.h declares
_VP, _I64, _I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
SIGNATURES = {
    "fo_split": (ctypes.c_int, [_VP, _VP, _VP, _I64, _I32, _VP]),
    "fo_merge": (ctypes.c_int, [_VP, _VP, _VP, _I64, _I32, _VP]),
    "fo_quant_state": (ctypes.c_int, [_VP, _VP, _VP, _I64, ctypes.c_int, _VP]),
    "fo_dequant_state": (ctypes.c_int, [_VP, _VP, _VP, _I64, ctypes.c_int, _VP]),
    "fo_adamw_step": (ctypes.c_int, [_VP, _I32, _VP, _I64, _VP]),
    "fo_sgd_step": (ctypes.c_int, [_VP, _I32, _VP, _VP]),
    "fo_lion_step": (ctypes.c_int, [_VP, _I32, _VP, _VP]),
    "fo_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fo_last_cuda_error": (ctypes.c_int, []),
    "fo_kernel_launch_count": (ctypes.c_uint64, []),
}


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the CUDA library; raise if impossible."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                try:
                    path = _build.build()
                    l = ctypes.CDLL(path)
                except Exception as e:  # no silent fallback: the caller sees why
                    raise RuntimeError(f"libfo.so (the CUDA library) is unavailable: {e}") from e
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(l, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = l
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        msg = lib().fo_status_string(status).decode()
        if status == 6:
            msg += f" (cudaError {lib().fo_last_cuda_error()})"
        raise FoError(fn, status, msg)


def _ptr(x) -> Optional[int]:
    """A device address: None, an int taken as is, or a contiguous CUDA
    tensor's data pointer (a host tensor's address would send the kernels to
    host memory, and a strided view would be read as if it were dense)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("the library reads and writes device memory: pass CUDA tensors")
    if not x.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return None
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _numel(x, n):
    if n is not None:
        return int(n)
    return int(x.numel())


# --- codecs ----------------------------------------------------------------

def fo_split(theta_f32, theta_bf16, rho, rho_bits: int = 8, n: Optional[int] = None, stream=None):
    _check("fo_split", lib().fo_split(_ptr(theta_f32), _ptr(theta_bf16), _ptr(rho),
                                      _numel(theta_f32, n), rho_bits, _stream(stream)))


def fo_merge(theta_bf16, rho, theta_f32, rho_bits: int = 8, n: Optional[int] = None, stream=None):
    _check("fo_merge", lib().fo_merge(_ptr(theta_bf16), _ptr(rho), _ptr(theta_f32),
                                      _numel(theta_bf16, n), rho_bits, _stream(stream)))


def fo_quant_state(x, q, scales, kind: int, n: Optional[int] = None, stream=None):
    _check("fo_quant_state", lib().fo_quant_state(_ptr(x), _ptr(q), _ptr(scales), _numel(x, n),
                                                  kind, _stream(stream)))


def fo_dequant_state(q, scales, x, kind: int, n: Optional[int] = None, stream=None):
    _check("fo_dequant_state", lib().fo_dequant_state(_ptr(q), _ptr(scales), _ptr(x), _numel(q, n),
                                                      kind, _stream(stream)))


# --- tables and fused steps ----------------------------------------------------

class Table:
    """A host array of ``fo_tensor_t`` rows, built once and reused across steps."""

    def __init__(self, rows: Sequence[FoTensor]):
        self.n = len(rows)
        self.rows = (FoTensor * max(1, self.n))(*rows)

    @property
    def ptr(self) -> int:
        return ctypes.addressof(self.rows)


def _grad_dtype(grad, grad_dtype: Optional[int]) -> int:
    """FP32 for a float32 tensor, else BF16 (bfloat16 or int16 bit patterns);
    an explicit grad_dtype wins (needed for raw pointers)."""
    if grad_dtype is not None:
        return int(grad_dtype)
    dt = getattr(grad, "dtype", None)
    return GRAD_F32 if dt is not None and str(dt) == "torch.float32" else GRAD_BF16


def row(theta, rho, m_q, m_scale, grad, v_q=None, v_scale=None, weight_decay: float = 0.0,
        rho_bits: int = 8, numel: Optional[int] = None, grad_dtype: Optional[int] = None) -> FoTensor:
    return FoTensor(_ptr(theta), _ptr(rho), _ptr(m_q), _ptr(m_scale), _ptr(v_q), _ptr(v_scale),
                    _ptr(grad), _numel(theta, numel), float(weight_decay), int(rho_bits),
                    _grad_dtype(grad, grad_dtype))


def fo_adamw_step(table: Table, lr: float, beta1: float, beta2: float, eps: float, step: int,
                  stream=None, v_nonzero: bool = False):
    """v_nonzero: the opt-in rule that keeps a non-zero v off code 0 (FO_ADAMW_V_NONZERO)."""
    hp = AdamWHparams(lr, beta1, beta2, eps, FO_ADAMW_V_NONZERO if v_nonzero else 0, 0)
    _check("fo_adamw_step", lib().fo_adamw_step(table.ptr, table.n, ctypes.addressof(hp), int(step),
                                                _stream(stream)))


def fo_sgd_step(table: Table, lr: float, momentum: float, stream=None):
    hp = SGDHparams(lr, momentum)
    _check("fo_sgd_step", lib().fo_sgd_step(table.ptr, table.n, ctypes.addressof(hp), _stream(stream)))


def fo_lion_step(table: Table, lr: float, beta1: float, beta2: float, stream=None):
    hp = LionHparams(lr, beta1, beta2)
    _check("fo_lion_step", lib().fo_lion_step(table.ptr, table.n, ctypes.addressof(hp), _stream(stream)))


def fo_status_string(status: int) -> str:
    return lib().fo_status_string(status).decode()


def fo_kernel_launch_count() -> int:
    return int(lib().fo_kernel_launch_count())


# --- device-resident compressed state (torch tensors as memory) ---------------

class CompressedTensor:
    """The compressed state of one parameter tensor, in device memory.

    theta' (BF16 patterns), rho (int8 or int16), momentum codes and scales and,
    for AdamW, second-moment codes and scales. Memory comes from torch; every
    value is written by the library's kernels.
    """

    def __init__(self, numel: int, device, rho_bits: int = 8, with_v: bool = True,
                 weight_decay: float = 0.0, theta=None):
        """theta: optional int16 device tensor of numel elements to hold theta'
        (for example a view into one buffer shared by all rows); it must start on
        a 16-byte boundary."""
        import torch
        self.numel = int(numel)
        self.rho_bits = int(rho_bits)
        self.weight_decay = float(weight_decay)
        ng = (self.numel + GROUP - 1) // GROUP
        e = lambda dt: torch.empty(self.numel, dtype=dt, device=device)
        if theta is not None:
            if theta.dtype != torch.int16 or theta.numel() != self.numel or theta.data_ptr() % 16:
                raise ValueError("theta must be a 16-byte aligned int16 tensor of numel elements")
            self.theta = theta
        else:
            self.theta = e(torch.int16)
        self.rho = e(torch.int16 if rho_bits == 16 else torch.int8)
        self.m_q = torch.zeros(self.numel, dtype=torch.int8, device=device)
        self.m_scale = torch.zeros(ng, dtype=torch.int16, device=device)
        self.v_q = torch.zeros(self.numel, dtype=torch.uint8, device=device) if with_v else None
        self.v_scale = torch.zeros(ng, dtype=torch.int16, device=device) if with_v else None

    def init_from(self, theta_f32, stream=None):
        """theta', rho = split(theta_f32); momentum and variance start at zero."""
        fo_split(theta_f32, self.theta, self.rho, self.rho_bits, stream=stream)

    def row(self, grad) -> FoTensor:
        return row(self.theta, self.rho, self.m_q, self.m_scale, grad, self.v_q, self.v_scale,
                   self.weight_decay, self.rho_bits, self.numel)

    def buffers(self) -> List:
        return [b for b in (self.theta, self.rho, self.m_q, self.m_scale, self.v_q, self.v_scale)
                if b is not None]


def table_of(states: Iterable[CompressedTensor], grads: Iterable) -> Table:
    return Table([s.row(g) for s, g in zip(states, grads)])
