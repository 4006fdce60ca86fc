"""Drop-in PyTorch optimizers over the fused compressed step: FlashAdamW,
FlashSGD and FlashLion.

"FlashOptim: Optimizers for Memory Efficient Training" presents its
optimizers as drop-in replacements for the standard ones with unchanged
hyper-parameters (page sections "创新点和贡献" and "实践建议"). Here each
parameter's BF16 data *is* theta'; the optimizer keeps the correction rho and
the companded INT8 momentum (and UINT8 second moment) with their FP16 group
scales, and one call of the C ABI updates every parameter of a group in one
kernel launch. Features from the page's practical advice:

* per-group opt-out: ``rho_bits=16`` for a finer master weight, or
  ``compress=False`` to keep an FP32 master weight and FP32 moments updated by
  the standard PyTorch optimizer for that group;
* gradient release: :meth:`attach_grad_release` steps parameters during
  backward as their gradients become ready (in buckets of a bounded size, one
  fused call each) and frees each gradient once its step is enqueued;
* compact checkpoints: :meth:`state_dict` holds theta' (through the model's
  parameters), rho, codes, scales and the step counters -- about 5 bytes per
  parameter for AdamW instead of 12;
* :meth:`master_weights` rebuilds the FP32 master weights.

Parameters must live on a CUDA device: there is no CPU path.
"""
from __future__ import annotations

from typing import Callable, Dict, Iterable, List, Optional

import torch

from . import fo

_GROUP = fo.GROUP


def _bits16(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16)


class _FlashOptimizer(torch.optim.Optimizer):
    _kind = ""          # "adamw", "sgd", "lion"
    _with_v = False
    _reference = None   # torch optimizer class for compress=False groups

    def __init__(self, params, defaults: Dict):
        defaults.setdefault("rho_bits", 8)
        defaults.setdefault("compress", True)
        super().__init__(params, defaults)
        self._fallback: Dict[int, torch.optim.Optimizer] = {}
        # built tables, reused while every pointer in them is unchanged
        self._tables: Dict[tuple, tuple] = {}
        for gi, group in enumerate(self.param_groups):
            if group["rho_bits"] not in (8, 16):
                raise ValueError("rho_bits must be 8 or 16")
            for p in group["params"]:
                if not p.is_cuda:
                    raise RuntimeError(f"{type(self).__name__} needs CUDA parameters (no CPU path)")
                if group["compress"]:
                    self._init_compressed(p, group)
            if not group["compress"]:
                self._fallback[gi] = self._make_reference(group)

    # -- state ------------------------------------------------------------

    def _init_compressed(self, p: torch.Tensor, group: Dict) -> None:
        """theta', rho = split(FP32 weights) (rho = 0 for weights that are BF16
        already); moments start at zero codes with zero scales."""
        if not p.is_contiguous():
            raise ValueError("parameters must be contiguous")
        n = p.numel()
        rb = group["rho_bits"]
        rho = torch.zeros(n, dtype=torch.int16 if rb == 16 else torch.int8, device=p.device)
        if p.dtype == torch.float32:
            master = p.detach().reshape(-1).contiguous()
            tp = torch.empty(n, dtype=torch.bfloat16, device=p.device)
            with torch.cuda.device(p.device):
                fo.fo_split(master, _bits16(tp), rho, rb)
            p.data = tp.view(p.shape)
        elif p.dtype != torch.bfloat16:
            raise TypeError("parameters must be float32 (split on first use) or bfloat16")
        ng = (n + _GROUP - 1) // _GROUP
        st = self.state[p]
        if group.get("capturable"):
            st["step"] = self._group_counter(group, p.device)   # shared int64 device tensor
        else:
            st["step"] = 0      # a Python int: the step counter t of this parameter
        st["rho"] = rho
        st["m_q"] = torch.zeros(n, dtype=torch.int8, device=p.device)
        st["m_scale"] = torch.zeros(ng, dtype=torch.int16, device=p.device)
        if self._with_v:
            st["v_q"] = torch.zeros(n, dtype=torch.uint8, device=p.device)
            st["v_scale"] = torch.zeros(ng, dtype=torch.int16, device=p.device)

    def _group_counter(self, group: Dict, device) -> torch.Tensor:
        """The device step counter of a capturable group's parameters on `device`."""
        counters = self.__dict__.setdefault("_counters", {})
        key = (id(group), torch.device(device).index)
        if key not in counters:
            counters[key] = torch.zeros((), dtype=torch.int64, device=device)
        return counters[key]

    def _make_reference(self, group: Dict) -> torch.optim.Optimizer:
        hp = {k: v for k, v in group.items() if k not in ("params", "rho_bits", "compress", "v_nonzero")}
        for p in group["params"]:
            if p.dtype != torch.float32:
                raise TypeError("compress=False groups keep FP32 parameters")
        return self._reference(group["params"], **self._reference_args(hp))

    @staticmethod
    def _grad_of(p: torch.Tensor) -> torch.Tensor:
        """The gradient as the step reads it: BF16 as it is, FP32 as it is
        (for example with ``Tensor.grad_dtype`` set to float32, which
        accumulates FP32 gradients for BF16 parameters; the step then uses
        them unrounded), any other type widened or rounded to FP32."""
        g = p.grad
        if g.dtype != torch.bfloat16 and g.dtype != torch.float32:
            g = g.float()
        if not g.is_contiguous():
            g = g.contiguous()
        return g

    def _row(self, p: torch.Tensor, g: torch.Tensor, group: Dict) -> fo.FoTensor:
        st = self.state[p]
        grad = _bits16(g) if g.dtype == torch.bfloat16 else g   # float32: fo.GRAD_F32
        return fo.row(_bits16(p.data), st["rho"], st["m_q"], st["m_scale"], grad,
                      st.get("v_q"), st.get("v_scale"), self._weight_decay(group),
                      group["rho_bits"], p.numel())

    def _table(self, ps: List[torch.Tensor], grads: List[torch.Tensor], group: Dict) -> fo.Table:
        """The table of these parameters, rebuilt only when a pointer, the
        weight decay or the correction width changed since the last call."""
        key = (id(group), tuple(id(p) for p in ps))
        ptrs = (self._weight_decay(group), group["rho_bits"],
                tuple(p.data_ptr() for p in ps), tuple((g.data_ptr(), g.dtype) for g in grads),
                tuple(self.state[p]["m_q"].data_ptr() for p in ps))
        hit = self._tables.get(key)
        if hit is not None and hit[0] == ptrs:
            return hit[1]
        table = fo.Table([self._row(p, g, group) for p, g in zip(ps, grads)])
        self._tables[key] = (ptrs, table)
        return table

    def _weight_decay(self, group: Dict) -> float:
        return float(group.get("weight_decay", 0.0))

    # -- stepping ---------------------------------------------------------

    @torch.no_grad()
    def step(self, closure: Optional[Callable] = None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        for gi, group in enumerate(self.param_groups):
            if not group["compress"]:
                self._fallback[gi].step()
                continue
            params = [p for p in group["params"] if p.grad is not None]
            self._step_params(params, group)
        return loss

    def _step_params(self, params: List[torch.Tensor], group: Dict) -> None:
        if not params:
            return
        # parameters of a group on the same device that have taken the same
        # number of steps share a call (a launch only touches its own device)
        if group.get("capturable"):
            self._step_params_capturable(params, group)
            return
        by_key: Dict[tuple, List[torch.Tensor]] = {}
        for p in params:
            by_key.setdefault((int(self.state[p]["step"]) + 1, p.device.index), []).append(p)
        for (t, dev), ps in by_key.items():
            grads = [self._grad_of(p) for p in ps]     # alive until the launch is enqueued
            with torch.cuda.device(dev):
                table = self._table(ps, grads, group)
                try:
                    self._launch(table, group, t)
                finally:
                    # the cached table must not keep this step's gradients alive
                    table.release()
            # the step counters advance only once the call has succeeded, so a
            # refused call (fo.FoError) leaves them as they were
            for p in ps:
                self.state[p]["step"] = t

    def _step_params_capturable(self, params: List[torch.Tensor], group: Dict) -> None:
        """Capturable groups (FlashAdamW): the step counter is a device tensor
        shared by the group's parameters on one device, advanced on the device
        and read by the kernel, so the step can be captured in a CUDA graph and
        replayed with the bias corrections moving on."""
        by_dev: Dict[int, List[torch.Tensor]] = {}
        for p in params:
            by_dev.setdefault(p.device.index, []).append(p)
        for dev, ps in by_dev.items():
            counter = self.state[ps[0]]["step"]
            grads = [self._grad_of(p) for p in ps]
            with torch.cuda.device(dev):
                table = self._table(ps, grads, group)
                counter.add_(1)
                try:
                    self._launch_dev(table, group, counter)
                except fo.FoError:
                    counter.sub_(1)       # a refused call leaves the counter as it was
                    raise
                finally:
                    table.release()

    def _launch(self, table: fo.Table, group: Dict, t: int) -> None:
        raise NotImplementedError

    def _launch_dev(self, table: fo.Table, group: Dict, counter: torch.Tensor) -> None:
        raise NotImplementedError

    # -- gradient release ---------------------------------------------------

    def attach_grad_release(self, params: Optional[Iterable[torch.Tensor]] = None,
                            bucket_numel: int = 1 << 24) -> List:
        """Step compressed parameters during backward, as their gradients
        become ready, and free each gradient once its step is enqueued (no
        gradient accumulation across backward passes).

        Parameters whose gradients are ready wait in a bucket per parameter
        group; the bucket is stepped in one fused call once it holds
        ``bucket_numel`` elements, and whatever is left is stepped at the end
        of the backward pass. At most about ``bucket_numel`` elements of
        gradient per group are therefore alive beyond the one autograd is
        producing; ``bucket_numel=0`` steps each parameter on its own. Returns
        the hook handles."""
        handles = []
        wanted = None if params is None else {id(p) for p in params}
        queued = [False]

        class Bucket:
            __slots__ = ("group", "params", "numel")

            def __init__(self, group):
                self.group, self.params, self.numel = group, [], 0

        buckets: List[Bucket] = []

        def flush(b: Bucket) -> None:
            ps, b.params, b.numel = b.params, [], 0
            with torch.no_grad():
                self._step_params(ps, b.group)
            for q in ps:
                q.grad = None

        def flush_all() -> None:
            queued[0] = False
            for b in buckets:
                if b.params:
                    flush(b)

        self._release_flush = flush_all
        seen = set()
        for group in self.param_groups:
            if not group["compress"]:
                continue
            bucket = Bucket(group)
            buckets.append(bucket)
            for p in group["params"]:
                if id(p) in seen or (wanted is not None and id(p) not in wanted):
                    continue
                seen.add(id(p))

                # per call: two attribute updates and a compare; the bucket
                # and the element count are bound when the hook is made
                def hook(param, b=bucket, n=p.numel()):
                    b.params.append(param)
                    b.numel += n
                    if b.numel >= bucket_numel:
                        flush(b)
                    elif not queued[0]:
                        # the rest of the bucket is stepped when this backward pass ends
                        torch.autograd.Variable._execution_engine.queue_callback(flush_all)
                        queued[0] = True

                handles.append(p.register_post_accumulate_grad_hook(hook))
        return handles

    def flush_grad_release(self) -> None:
        """Step the parameters still waiting in a gradient-release bucket (for
        a backward pass that ended early, for example through an exception)."""
        f = getattr(self, "_release_flush", None)
        if f is not None:
            f()

    # -- checkpoints ----------------------------------------------------------

    _COMPRESSED = ("rho", "m_q", "m_scale", "v_q", "v_scale")

    def load_state_dict(self, state_dict: Dict) -> None:
        """Load a state_dict written by state_dict(). The compressed buffers keep
        their integer dtypes (torch's loader would cast every state tensor of a
        floating-point parameter to the parameter's dtype)."""
        saved = state_dict["state"]
        kept = {}
        plain = {}
        for k, st in saved.items():
            kept[k] = {n: v for n, v in st.items() if n in self._COMPRESSED}
            plain[k] = {n: v for n, v in st.items() if n not in self._COMPRESSED}
        super().load_state_dict({"state": plain, "param_groups": state_dict["param_groups"]})
        saved_ids = [i for g in state_dict["param_groups"] for i in g["params"]]
        params = [p for g in self.param_groups for p in g["params"]]
        for sid, p in zip(saved_ids, params):
            for n, v in kept.get(sid, {}).items():
                cur = self.state[p].get(n)
                if cur is not None and (cur.dtype != v.dtype or cur.shape != v.shape):
                    raise ValueError(f"state '{n}' does not match the parameter's layout")
                self.state[p][n] = v.to(device=p.device).clone()
        self.__dict__.pop("_counters", None)
        for group in self.param_groups:
            for p in group["params"]:
                st = self.state.get(p)
                if not st or "step" not in st:
                    continue
                if group.get("capturable"):
                    # one counter per group and device again, holding the saved count
                    c = self._group_counter(group, p.device)
                    c.fill_(int(st["step"]))
                    st["step"] = c
                else:
                    st["step"] = int(st["step"])    # checkpoints may hold it as a tensor
        self._tables.clear()

    # -- export ---------------------------------------------------------------

    @torch.no_grad()
    def master_weights(self) -> Dict[torch.Tensor, torch.Tensor]:
        """FP32 master weights theta^ = merge(theta', rho) of every compressed parameter."""
        out = {}
        for group in self.param_groups:
            if not group["compress"]:
                continue
            for p in group["params"]:
                w = torch.empty(p.numel(), dtype=torch.float32, device=p.device)
                with torch.cuda.device(p.device):
                    fo.fo_merge(_bits16(p.data.reshape(-1)), self.state[p]["rho"], w, group["rho_bits"])
                out[p] = w.view(p.shape)
        return out

    def state_bytes(self) -> int:
        """Bytes held by the compressed optimizer state (rho, codes, scales)."""
        n = 0
        for st in self.state.values():
            for k, v in st.items():
                if isinstance(v, torch.Tensor) and k != "step":
                    n += v.numel() * v.element_size()
        return n


class FlashAdamW(_FlashOptimizer):
    """AdamW (decoupled weight decay) with compressed master weight and state.

    v_nonzero=True opts into a rule the page does not have: a non-zero second
    moment is never stored as code 0, which would decode it to 0 and let the
    momentum drive an update of about lr*m/eps.

    capturable=True keeps each group's step counter in device memory (one
    int64 tensor shared by the group's parameters on a device, advanced on the
    device by every step()), so that step() can be captured in a CUDA graph:
    each replay advances the counter and the kernel derives the bias
    corrections from it. Every parameter of such a group with a gradient is
    stepped with the group's count (a parameter without a gradient at some
    step is skipped, but the count moves on)."""
    _kind = "adamw"
    _with_v = True
    _reference = torch.optim.AdamW

    def __init__(self, params, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01,
                 rho_bits=8, compress=True, v_nonzero=False, capturable=False):
        super().__init__(params, dict(lr=lr, betas=betas, eps=eps, weight_decay=weight_decay,
                                      rho_bits=rho_bits, compress=compress, v_nonzero=v_nonzero,
                                      capturable=capturable))

    @staticmethod
    def _reference_args(hp):
        return dict(lr=hp["lr"], betas=hp["betas"], eps=hp["eps"], weight_decay=hp["weight_decay"])

    def _launch(self, table, group, t):
        b1, b2 = group["betas"]
        fo.fo_adamw_step(table, group["lr"], b1, b2, group["eps"], t,
                         v_nonzero=bool(group.get("v_nonzero", False)))

    def _launch_dev(self, table, group, counter):
        b1, b2 = group["betas"]
        fo.fo_adamw_step_dev(table, group["lr"], b1, b2, group["eps"], counter,
                             v_nonzero=bool(group.get("v_nonzero", False)))


class FlashSGD(_FlashOptimizer):
    """SGD with momentum (dampening 0, no Nesterov, L2 weight decay)."""
    _kind = "sgd"
    _reference = torch.optim.SGD

    def __init__(self, params, lr=0.1, momentum=0.9, weight_decay=0.0, rho_bits=8, compress=True):
        super().__init__(params, dict(lr=lr, momentum=momentum, weight_decay=weight_decay,
                                      rho_bits=rho_bits, compress=compress))

    @staticmethod
    def _reference_args(hp):
        return dict(lr=hp["lr"], momentum=hp["momentum"], weight_decay=hp["weight_decay"])

    def _launch(self, table, group, t):
        fo.fo_sgd_step(table, group["lr"], group["momentum"])


class _ReferenceLion(torch.optim.Optimizer):
    """Uncompressed Lion (FP32 state) for compress=False groups."""

    def __init__(self, params, lr=1e-4, betas=(0.9, 0.99), weight_decay=0.0):
        super().__init__(params, dict(lr=lr, betas=betas, weight_decay=weight_decay))

    @torch.no_grad()
    def step(self):
        for group in self.param_groups:
            b1, b2 = group["betas"]
            for p in group["params"]:
                if p.grad is None:
                    continue
                st = self.state[p]
                if "m" not in st:
                    st["m"] = torch.zeros_like(p)
                m = st["m"]
                c = m.mul(b1).add_(p.grad, alpha=1 - b1)
                p.mul_(1 - group["lr"] * group["weight_decay"]).add_(torch.sign(c), alpha=-group["lr"])
                m.mul_(b2).add_(p.grad, alpha=1 - b2)


class FlashLion(_FlashOptimizer):
    """Lion (Chen et al. 2023) with decoupled weight decay."""
    _kind = "lion"
    _reference = _ReferenceLion

    def __init__(self, params, lr=1e-4, betas=(0.9, 0.99), weight_decay=0.0, rho_bits=8, compress=True):
        super().__init__(params, dict(lr=lr, betas=betas, weight_decay=weight_decay,
                                      rho_bits=rho_bits, compress=compress))

    @staticmethod
    def _reference_args(hp):
        return dict(lr=hp["lr"], betas=hp["betas"], weight_decay=hp["weight_decay"])

    def _launch(self, table, group, t):
        b1, b2 = group["betas"]
        fo.fo_lion_step(table, group["lr"], b1, b2)
