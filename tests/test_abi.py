"""The C-ABI library builds, loads and exports what include/fo.h declares.

No compute call is made here: every call below is rejected by the host-side
argument checks before anything touches CUDA, so these run without a GPU.
"""
import ctypes
import os
import re

import pytest

from quantized_optimizer_state_gb300 import fo

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "fo.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fo_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    lib = fo.lib()
    names = _declared_functions()
    assert "fo_adamw_step" in names and "fo_split" in names and len(names) >= 10
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(fo.SIGNATURES)


def test_struct_layout_matches_header():
    # 7 pointers, int64 numel, double weight_decay, int32 rho_bits, int32 grad_dtype
    assert ctypes.sizeof(fo.FoTensor) == 80
    assert fo.FoTensor.numel.offset == 56 and fo.FoTensor.weight_decay.offset == 64
    assert ctypes.sizeof(fo.AdamWHparams) == 40     # 4 doubles, uint32 flags, uint32 reserved


def test_status_strings():
    for code, name in fo.STATUS.items():
        assert fo.fo_status_string(code).startswith(name)
    assert "unknown" in fo.fo_status_string(99)


def _call(fn, *args):
    return getattr(fo.lib(), fn)(*args)


def test_codec_argument_errors():
    A = 1 << 20          # a 16-byte aligned fake address: never dereferenced
    assert _call("fo_split", A, A, A, 0, 8, None) == 0                  # n = 0 is a no-op
    assert _call("fo_split", A, A, A, -1, 8, None) == 3                 # FO_ERR_SIZE
    assert _call("fo_split", None, A, A, 10, 8, None) == 1              # FO_ERR_NULL
    assert _call("fo_split", A, A, A, 10, 12, None) == 4                # rho_bits
    assert _call("fo_split", A + 2, A, A, 10, 8, None) == 2             # misaligned
    assert _call("fo_merge", A, A + 8, A, 10, 16, None) == 2
    assert _call("fo_quant_state", A, A, A, 10, 7, None) == 4           # bad kind
    assert _call("fo_quant_state", A, A, A, 10, 4, None) == 4           # 4 is not a kind
    assert _call("fo_dequant_state", A, A, A, 10, 6, None) == 4
    assert _call("fo_quant_state", A, A, A + 1, 10, 0, None) == 2       # odd scale address
    assert _call("fo_dequant_state", A, None, A, 10, 1, None) == 1


def _table(**over):
    A = 1 << 24
    base = dict(theta=A, rho=A + (1 << 20), m_q=A + (2 << 20), m_scale=A + (3 << 20),
                v_q=A + (4 << 20), v_scale=A + (5 << 20), grad=A + (6 << 20), numel=100,
                weight_decay=0.01, rho_bits=8, grad_dtype=0)
    base.update(over)
    return fo.FoTensor(**base)


def _adamw(rows, step=1, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, flags=0, reserved=0):
    arr = (fo.FoTensor * max(1, len(rows)))(*rows)
    hp = fo.AdamWHparams(lr, beta1, beta2, eps, flags, reserved)
    return _call("fo_adamw_step", ctypes.addressof(arr), len(rows), ctypes.addressof(hp), step, None)


def test_step_argument_errors():
    assert _adamw([]) == 0                                         # empty table: no-op
    assert _adamw([_table(numel=0)]) == 0                          # empty rows are skipped
    assert _adamw([_table()], step=0) == 3
    assert _adamw([_table(numel=-5)]) == 3
    assert _adamw([_table(theta=None)]) == 1
    assert _adamw([_table(v_q=None)]) == 1                         # AdamW needs v
    assert _adamw([_table(rho_bits=4)]) == 4
    assert _adamw([_table(grad_dtype=2)]) == 4                     # not BF16 (0) or FP32 (1)
    assert _adamw([_table(grad_dtype=-1)]) == 4
    assert _adamw([_table(weight_decay=float("nan"))]) == 4
    assert _adamw([_table(grad=(1 << 24) + (6 << 20) + 8)]) == 2   # misaligned grad
    assert _adamw([_table(m_scale=(1 << 24) + (3 << 20) + 1)]) == 2
    assert _adamw([_table(grad=(1 << 24) + 64)]) == 7              # grad overlaps theta'
    # an FP32 gradient spans 4 bytes an element: 100 of them from 304 bytes
    # below rho reach into it (100 BF16 ones would not)
    assert _adamw([_table(grad=(1 << 24) + (1 << 20) - 304, grad_dtype=1)]) == 7
    # state buffers of one row overlapping each other
    assert _adamw([_table(m_q=(1 << 24) + 96)]) == 7               # m codes inside theta'
    assert _adamw([_table(v_scale=(1 << 24) + (3 << 20) + 6)]) == 7  # v scales inside m scales
    assert _adamw([_table(rho=(1 << 24) + (2 << 20) - 96)]) == 7   # rho's 100 bytes reach m codes
    assert _adamw([_table(rho=(1 << 24) + (2 << 20) - 96, rho_bits=16)]) == 7
    # 100 bytes of rho ending 12 bytes short of the m codes: no overlap, so the
    # next row's error is the one reported (nothing launches)
    assert _adamw([_table(rho=(1 << 24) + (2 << 20) - 112), _table(numel=-1)]) == 3
    assert _adamw([_table()], lr=float("inf")) == 4
    assert _adamw([_table()], beta1=1.0) == 4
    assert _adamw([_table()], eps=0.0) == 4
    assert _adamw([_table()], flags=2) == 4                        # unknown flag bit
    assert _adamw([_table()], reserved=1) == 4
    assert _adamw([_table(numel=0)], flags=fo.FO_ADAMW_V_NONZERO) == 0
    assert _adamw([_table(), _table(numel=-1)]) == 3               # checked before any launch
    hp = fo.AdamWHparams(1e-3, 0.9, 0.999, 1e-8)
    assert _call("fo_adamw_step", None, 3, ctypes.addressof(hp), 1, None) == 1
    assert _call("fo_adamw_step", None, -1, ctypes.addressof(hp), 1, None) == 3
    assert _call("fo_adamw_step", None, fo.FO_MAX_TENSORS + 1, ctypes.addressof(hp), 1, None) == 5
    arr = (fo.FoTensor * 1)(_table())
    assert _call("fo_adamw_step", ctypes.addressof(arr), 1, None, 1, None) == 1


def test_sgd_and_lion_need_no_v():
    arr = (fo.FoTensor * 1)(_table(v_q=None, v_scale=None, numel=-1))
    sgd = fo.SGDHparams(0.1, 0.9)
    lion = fo.LionHparams(1e-4, 0.9, 0.99)
    # the v pointers are not required; the bad numel is what is reported
    assert _call("fo_sgd_step", ctypes.addressof(arr), 1, ctypes.addressof(sgd), None) == 3
    assert _call("fo_lion_step", ctypes.addressof(arr), 1, ctypes.addressof(lion), None) == 3
    # SGD and Lion ignore the v buffers, so theirs may coincide with theta'
    two = (fo.FoTensor * 2)(_table(v_q=1 << 24, v_scale=1 << 24), _table(numel=-1))
    assert _call("fo_sgd_step", ctypes.addressof(two), 2, ctypes.addressof(sgd), None) == 3
    assert _adamw([_table(v_q=1 << 24, v_scale=1 << 24)]) == 7
    bad = fo.SGDHparams(-0.1, 0.9)
    assert _call("fo_sgd_step", ctypes.addressof(arr), 1, ctypes.addressof(bad), None) == 4
    badl = fo.LionHparams(1e-4, 0.9, 1.5)
    assert _call("fo_lion_step", ctypes.addressof(arr), 1, ctypes.addressof(badl), None) == 4


def test_rejected_calls_launch_nothing():
    before = fo.fo_kernel_launch_count()
    assert _adamw([_table(rho_bits=3)]) == 4
    assert _call("fo_split", 16, 16, 16, -1, 8, None) == 3
    assert fo.fo_kernel_launch_count() == before


def test_binding_rejects_host_and_strided_tensors():
    """The binding refuses tensors the kernels would misread, before any call."""
    import torch
    x = torch.zeros(64)
    with pytest.raises(ValueError, match="CUDA"):
        fo.fo_split(x, torch.zeros(64, dtype=torch.int16), torch.zeros(64, dtype=torch.int8))
    with pytest.raises(ValueError, match="CUDA"):
        fo.row(x, None, None, None, None)
    assert fo._ptr(None) is None and fo._ptr(1 << 20) == 1 << 20


def test_rows_of_one_table_may_not_share_written_memory():
    """Every array a step writes must be disjoint from every other array of the
    table, in its own row or another (one launch would race; two launches
    would step the same state twice)."""
    MB = 1 << 20
    second = dict(theta=(1 << 26), rho=(1 << 26) + MB, m_q=(1 << 26) + 2 * MB, m_scale=(1 << 26) + 3 * MB,
                  v_q=(1 << 26) + 4 * MB, v_scale=(1 << 26) + 5 * MB, grad=(1 << 26) + 6 * MB)
    assert _adamw([_table(), _table()]) == 7                                   # the same row twice
    assert _adamw([_table(), _table(**dict(second, theta=(1 << 24) + 64))]) == 7   # theta' inside theta'
    assert _adamw([_table(), _table(**dict(second, grad=(1 << 24) + (2 << 20)))]) == 7  # grad over m codes
    assert _adamw([_table(), _table(**dict(second, v_scale=(1 << 24) + (5 << 20) + 6))]) == 7   # last 2 bytes
    assert _adamw([_table(numel=0), _table(numel=0)]) == 0                     # empty rows hold nothing
    # rows of different launches (correction widths) are checked too
    assert _adamw([_table(), _table(**dict(second, rho_bits=16, m_q=(1 << 24) + 32))]) == 7
    sgd = fo.SGDHparams(0.1, 0.9)
    two = (fo.FoTensor * 2)(_table(v_q=None, v_scale=None),
                            _table(**dict(second, v_q=None, v_scale=None, m_scale=(1 << 24) + (3 << 20) + 2)))
    assert _call("fo_sgd_step", ctypes.addressof(two), 2, ctypes.addressof(sgd), None) == 7


def test_codec_outputs_may_not_overlap_their_inputs():
    A = 1 << 20
    assert _call("fo_split", A, A + 16, A + 4096, 10, 8, None) == 7           # theta' inside the FP32 input
    assert _call("fo_split", A, A + 4096, A + 4096 + 16, 10, 8, None) == 7    # rho inside theta'
    assert _call("fo_merge", A, A + 4096, A + 16, 10, 8, None) == 7           # output over theta'
    assert _call("fo_quant_state", A, A + 4096, A + 4096 + 4, 64, 0, None) == 7  # scales inside the codes
    assert _call("fo_dequant_state", A, A + 4096, A + 32, 64, 1, None) == 7   # output over the codes
    assert _call("fo_split", A, A, A, (1 << 46) + 1, 8, None) == 3            # size bound


class _FakeCuda:
    """Stands in for a CUDA tensor in binding checks that run before any call."""

    def __init__(self, dtype, n, dev=0, addr=1 << 20):
        import types
        self.dtype, self._n, self._addr = dtype, n, addr
        self.device = types.SimpleNamespace(index=dev)
        self.is_cuda = True

    def is_contiguous(self):
        return True

    def numel(self):
        return self._n

    def data_ptr(self):
        return self._addr


def test_binding_rejects_wrong_device_dtype_and_length(monkeypatch):
    import types
    import torch
    monkeypatch.setattr(fo, "_current_device", lambda: 0)
    F = _FakeCuda
    n = 100
    ok = dict(theta=F(torch.int16, n), rho=F(torch.int8, n), m_q=F(torch.int8, n), m_scale=F(torch.int16, 4),
              grad=F(torch.bfloat16, n), v_q=F(torch.uint8, n), v_scale=F(torch.float16, 4))
    r = fo.row(**ok)
    assert r.numel == n and r.grad_dtype == fo.GRAD_BF16 and len(r.keep) == 7
    assert fo.row(**dict(ok, grad=F(torch.float32, n))).grad_dtype == fo.GRAD_F32
    with pytest.raises(ValueError, match="cuda:1"):
        fo.row(**dict(ok, m_q=F(torch.int8, n, dev=1)))                 # another device's tensor
    for name, bad in [("theta", F(torch.float32, n)), ("rho", F(torch.int16, n)), ("m_q", F(torch.uint8, n)),
                      ("v_q", F(torch.int8, n)), ("m_scale", F(torch.float32, 4)),
                      ("grad", F(torch.float16, n)), ("grad", F(torch.float64, n)), ("grad", F(torch.int8, n))]:
        with pytest.raises(TypeError, match=name):
            fo.row(**dict(ok, **{name: bad}))
    with pytest.raises(TypeError):
        fo.row(**ok, grad_dtype=fo.GRAD_F32)                            # contradicts the tensor's type
    with pytest.raises(TypeError, match="rho"):
        fo.row(**dict(ok, rho=F(torch.int8, n)), rho_bits=16)
    with pytest.raises(ValueError, match="needs 4"):
        fo.row(**dict(ok, v_scale=F(torch.int16, 3)))                   # too few scales
    with pytest.raises(ValueError, match="needs 100"):
        fo.row(**dict(ok, grad=F(torch.bfloat16, 99)))
    with pytest.raises(TypeError, match="q"):
        fo.fo_quant_state(F(torch.float32, n), F(torch.int8, n), F(torch.int16, 4), fo.FO_STATE_VARIANCE)
    with pytest.raises(TypeError, match="x"):
        fo.fo_dequant_state(F(torch.int8, n), F(torch.int16, 4), F(torch.float16, n), fo.FO_STATE_MOMENTUM)
    with pytest.raises(ValueError, match="needs"):
        fo.fo_split(F(torch.float32, n), F(torch.int16, n - 1), F(torch.int8, n))
    stream = types.SimpleNamespace(device=types.SimpleNamespace(index=2), cuda_stream=0)
    with pytest.raises(ValueError, match="stream"):
        fo._stream(stream)


def test_table_keeps_its_tensors_alive(monkeypatch):
    import gc
    import weakref
    import torch
    monkeypatch.setattr(fo, "_current_device", lambda: 0)
    F = _FakeCuda
    g = F(torch.bfloat16, 64)
    ref = weakref.ref(g)
    t = fo.Table([fo.row(F(torch.int16, 64), F(torch.int8, 64), F(torch.int8, 64), F(torch.int16, 2), g)])
    del g
    gc.collect()
    assert ref() is not None                # the table holds the gradient it points into
    t.release()
    gc.collect()
    assert ref() is None


def test_adamw_step_dev_argument_errors():
    """The device-counter AdamW call checks its hyper-parameters, the counter's
    address and the table on the host, before anything is launched."""
    hp = fo.AdamWHparams(1e-3, 0.9, 0.999, 1e-8)
    bad_hp = fo.AdamWHparams(1e-3, 1.0, 0.999, 1e-8)
    rows = (fo.FoTensor * 1)(_table(rho_bits=3))          # an invalid row: never launches
    A = 1 << 20
    assert _call("fo_adamw_step_dev", ctypes.addressof(rows), 1, ctypes.addressof(hp), None, None) == 1
    assert _call("fo_adamw_step_dev", ctypes.addressof(rows), 1, ctypes.addressof(hp), A + 4, None) == 2
    assert _call("fo_adamw_step_dev", ctypes.addressof(rows), 1, ctypes.addressof(bad_hp), A, None) == 4
    assert _call("fo_adamw_step_dev", ctypes.addressof(rows), 1, None, A, None) == 1
    assert _call("fo_adamw_step_dev", ctypes.addressof(rows), 1, ctypes.addressof(hp), A, None) == 4   # the row
    assert _call("fo_adamw_step_dev", None, 0, ctypes.addressof(hp), A, None) == 0                      # empty table


def test_verify_fast_arithmetic_argument_errors():
    A = 1 << 20
    assert _call("fo_verify_fast_arithmetic", None, None) == 1          # FO_ERR_NULL
    assert _call("fo_verify_fast_arithmetic", A + 4, None) == 2         # not 8-byte aligned


def test_verify_binding_rejects_wrong_counts(monkeypatch):
    """The counts buffer must be an int64 CUDA tensor of FO_VERIFY_COUNTS
    entries on the current device: refused before any call otherwise."""
    import torch
    monkeypatch.setattr(fo, "_current_device", lambda: 0)
    F = _FakeCuda
    with pytest.raises(TypeError, match="counts"):
        fo.fo_verify_fast_arithmetic(F(torch.int32, fo.FO_VERIFY_COUNTS))
    with pytest.raises(ValueError, match="needs"):
        fo.fo_verify_fast_arithmetic(F(torch.int64, fo.FO_VERIFY_COUNTS - 1))
    with pytest.raises(ValueError, match="CUDA"):
        fo.fo_verify_fast_arithmetic(torch.zeros(fo.FO_VERIFY_COUNTS, dtype=torch.int64))
    assert len(fo.VERIFY_CHECKS) == fo.FO_VERIFY_COUNTS
    hdr = open(os.path.join(ROOT, "include", "fo.h")).read()
    assert re.search(r"#define FO_VERIFY_COUNTS (\d+)", hdr).group(1) == str(fo.FO_VERIFY_COUNTS)
