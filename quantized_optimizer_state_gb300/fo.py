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
    "fo_adamw_step_dev": (ctypes.c_int, [_VP, _I32, _VP, _VP, _VP]),
    "fo_sgd_step": (ctypes.c_int, [_VP, _I32, _VP, _VP]),
    "fo_lion_step": (ctypes.c_int, [_VP, _I32, _VP, _VP]),
    "fo_verify_fast_arithmetic": (ctypes.c_int, [_VP, _VP]),
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


def _current_device() -> int:
    import torch
    return torch.cuda.current_device()


def _dtype_names(dtypes) -> str:
    return " or ".join(str(d).replace("torch.", "") for d in dtypes)


def _ptr(x, name: str = "tensor", dtypes=None, min_numel: Optional[int] = None) -> Optional[int]:
    """A device address: None, an int taken as is, or the data pointer of a
    contiguous CUDA tensor on the current device, of one of ``dtypes`` and with
    at least ``min_numel`` elements. Every call launches on the current device,
    so a host tensor, a strided view, a tensor of another device, a tensor of
    the wrong element type or one too short for the call would make the
    kernels read or write the wrong memory: each is refused here."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError(f"{name}: the library reads and writes device memory: pass CUDA tensors")
    if not x.is_contiguous():
        raise ValueError(f"{name}: tensors passed to the library must be contiguous")
    if dtypes is not None and x.dtype not in dtypes:
        raise TypeError(f"{name} must be {_dtype_names(dtypes)}, not {str(x.dtype).replace('torch.', '')}")
    if min_numel is not None and x.numel() < min_numel:
        raise ValueError(f"{name} holds {x.numel()} elements; the call needs {min_numel}")
    cur = _current_device()
    if x.device.index != cur:
        raise ValueError(f"{name} is on cuda:{x.device.index} but the current device is cuda:{cur}; "
                         "the library launches on the current device (use torch.cuda.device)")
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return None
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    dev = getattr(stream, "device", None)
    if dev is not None and getattr(dev, "index", None) is not None and dev.index != _current_device():
        raise ValueError(f"the stream belongs to cuda:{dev.index} but the current device is "
                         f"cuda:{_current_device()}; the library launches on the current device")
    return stream.cuda_stream


def _numel(x, n):
    if n is not None:
        return int(n)
    return int(x.numel())


def _groups(n: int) -> int:
    return (int(n) + GROUP - 1) // GROUP


class _Dtypes:
    """Element types the C ABI accepts for each kind of array (torch dtypes,
    resolved on first use so that importing this module does not import torch)."""
    _cache = None

    @classmethod
    def get(cls):
        if cls._cache is None:
            import torch
            half_bits = (torch.int16, torch.bfloat16)          # BF16 bit patterns
            scales = (torch.int16, torch.float16)              # FP16 bit patterns
            if hasattr(torch, "uint16"):
                half_bits += (torch.uint16,)
                scales += (torch.uint16,)
            cls._cache = {
                "f32": (torch.float32,),
                "bf16": half_bits,
                "scale": scales,
                "rho8": (torch.int8,),
                "rho16": (torch.int16,),
                "m_q": (torch.int8,),
                "v_q": (torch.uint8,),
            }
        return cls._cache


def _rho_dtypes(rho_bits: int):
    return _Dtypes.get()["rho16" if int(rho_bits) == 16 else "rho8"]


def _code_dtypes(kind: int):
    variance = int(kind) in (FO_STATE_VARIANCE, FO_STATE_VARIANCE_LINEAR, FO_STATE_VARIANCE_NONZERO)
    return _Dtypes.get()["v_q" if variance else "m_q"]


# --- codecs ----------------------------------------------------------------

def fo_split(theta_f32, theta_bf16, rho, rho_bits: int = 8, n: Optional[int] = None, stream=None):
    n = _numel(theta_f32, n)
    d = _Dtypes.get()
    _check("fo_split", lib().fo_split(_ptr(theta_f32, "theta_f32", d["f32"], n),
                                      _ptr(theta_bf16, "theta_bf16", d["bf16"], n),
                                      _ptr(rho, "rho", _rho_dtypes(rho_bits), n),
                                      n, rho_bits, _stream(stream)))


def fo_merge(theta_bf16, rho, theta_f32, rho_bits: int = 8, n: Optional[int] = None, stream=None):
    n = _numel(theta_bf16, n)
    d = _Dtypes.get()
    _check("fo_merge", lib().fo_merge(_ptr(theta_bf16, "theta_bf16", d["bf16"], n),
                                      _ptr(rho, "rho", _rho_dtypes(rho_bits), n),
                                      _ptr(theta_f32, "theta_f32", d["f32"], n),
                                      n, rho_bits, _stream(stream)))


def fo_quant_state(x, q, scales, kind: int, n: Optional[int] = None, stream=None):
    n = _numel(x, n)
    d = _Dtypes.get()
    _check("fo_quant_state", lib().fo_quant_state(_ptr(x, "x", d["f32"], n), _ptr(q, "q", _code_dtypes(kind), n),
                                                  _ptr(scales, "scales", d["scale"], _groups(n)), n,
                                                  kind, _stream(stream)))


def fo_dequant_state(q, scales, x, kind: int, n: Optional[int] = None, stream=None):
    n = _numel(q, n)
    d = _Dtypes.get()
    _check("fo_dequant_state", lib().fo_dequant_state(_ptr(q, "q", _code_dtypes(kind), n),
                                                      _ptr(scales, "scales", d["scale"], _groups(n)),
                                                      _ptr(x, "x", d["f32"], n), n, kind, _stream(stream)))


# --- tables and fused steps ----------------------------------------------------

class Table:
    """A host array of ``fo_tensor_t`` rows, built once and reused across steps.

    The table holds a reference to every tensor its rows point into, so that
    none of them can be freed (and its memory handed to another tensor by the
    caching allocator) while the table is alive."""

    def __init__(self, rows: Sequence[FoTensor]):
        self.n = len(rows)
        self.keep = [getattr(r, "keep", ()) for r in rows]
        self.rows = (FoTensor * max(1, self.n))(*rows)

    @property
    def ptr(self) -> int:
        return ctypes.addressof(self.rows)

    def release(self) -> None:
        """Drop the table's references to its tensors (the caller then keeps
        them alive for as long as it uses the table). Work already enqueued is
        unaffected: torch's allocator reuses freed memory in stream order."""
        self.keep = []


def _grad_dtype(grad, grad_dtype: Optional[int]) -> int:
    """fo_grad_dtype_t of a gradient: FP32 for a float32 tensor, BF16 for
    bfloat16 (or int16 bit patterns); any other element type is refused rather
    than read as BF16 words. For a raw address, grad_dtype says which
    (BF16 when omitted)."""
    dt = getattr(grad, "dtype", None)
    if dt is None:
        return GRAD_BF16 if grad_dtype is None else int(grad_dtype)
    d = _Dtypes.get()
    if dt in d["f32"]:
        found = GRAD_F32
    elif dt in d["bf16"]:
        found = GRAD_BF16
    else:
        raise TypeError(f"grad must be bfloat16 (or int16 BF16 patterns) or float32, not "
                        f"{str(dt).replace('torch.', '')}")
    if grad_dtype is not None and int(grad_dtype) != found:
        raise TypeError("grad_dtype does not match the gradient tensor's element type")
    return found


def row(theta, rho, m_q, m_scale, grad, v_q=None, v_scale=None, weight_decay: float = 0.0,
        rho_bits: int = 8, numel: Optional[int] = None, grad_dtype: Optional[int] = None) -> FoTensor:
    """One ``fo_tensor_t``. Tensors are checked (device, contiguity, element
    type, length) and kept alive by the row (and by any Table built from it)."""
    n = _numel(theta, numel)
    ng = _groups(n)
    d = _Dtypes.get()
    gdt = _grad_dtype(grad, grad_dtype)
    r = FoTensor(_ptr(theta, "theta", d["bf16"], n), _ptr(rho, "rho", _rho_dtypes(rho_bits), n),
                 _ptr(m_q, "m_q", d["m_q"], n), _ptr(m_scale, "m_scale", d["scale"], ng),
                 _ptr(v_q, "v_q", d["v_q"], n), _ptr(v_scale, "v_scale", d["scale"], ng),
                 _ptr(grad, "grad", d["f32"] if gdt == GRAD_F32 else d["bf16"], n), n,
                 float(weight_decay), int(rho_bits), gdt)
    r.keep = tuple(x for x in (theta, rho, m_q, m_scale, v_q, v_scale, grad) if x is not None and not isinstance(x, int))
    return r


def fo_adamw_step(table: Table, lr: float, beta1: float, beta2: float, eps: float, step: int,
                  stream=None, v_nonzero: bool = False):
    """v_nonzero: the opt-in rule that keeps a non-zero v off code 0 (FO_ADAMW_V_NONZERO)."""
    hp = AdamWHparams(lr, beta1, beta2, eps, FO_ADAMW_V_NONZERO if v_nonzero else 0, 0)
    _check("fo_adamw_step", lib().fo_adamw_step(table.ptr, table.n, ctypes.addressof(hp), int(step),
                                                _stream(stream)))


def fo_adamw_step_dev(table: Table, lr: float, beta1: float, beta2: float, eps: float, step,
                      stream=None, v_nonzero: bool = False):
    """AdamW with the step counter read on the device when the kernel runs:
    ``step`` is a one-element int64 CUDA tensor (or a raw device address). For
    steps captured in a CUDA graph; the caller advances the counter."""
    hp = AdamWHparams(lr, beta1, beta2, eps, FO_ADAMW_V_NONZERO if v_nonzero else 0, 0)
    import torch
    ptr = _ptr(step, "step", (torch.int64,), 1)
    _check("fo_adamw_step_dev", lib().fo_adamw_step_dev(table.ptr, table.n, ctypes.addressof(hp), ptr,
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


FO_VERIFY_COUNTS = 6
VERIFY_CHECKS = ("reciprocal", "square_root", "phi_m_adamw", "phi_m_sgd_lion", "momentum_decode",
                 "scale_divisions")


def fo_verify_fast_arithmetic(counts=None, stream=None) -> dict:
    """Enumerate, on the current device, every operand domain on which the
    fast path's division and square root depend on the GPU's approximations,
    and return the mismatch count of each against the IEEE operation (all 0
    where the fast path is exact). ``counts``: an optional int64 CUDA tensor of
    FO_VERIFY_COUNTS elements to write into; the call waits for the result."""
    import torch
    if counts is None:
        counts = torch.zeros(FO_VERIFY_COUNTS, dtype=torch.int64, device="cuda")
    ptr = _ptr(counts, "counts", (torch.int64,), FO_VERIFY_COUNTS)
    s = _stream(stream)
    _check("fo_verify_fast_arithmetic", lib().fo_verify_fast_arithmetic(ptr, s))
    torch.cuda.synchronize()
    return dict(zip(VERIFY_CHECKS, (int(c) for c in counts.cpu().tolist())))


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
