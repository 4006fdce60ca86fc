"""Codec-quality study: the two quality figures of "FlashOptim: Optimizers for
Memory Efficient Training", reproduced on synthetic inputs with this
library's kernels, and a measurement of the opt-in second-moment rule.

* Fig. 3 (section "实验结果分析", weight reconstruction): every FP32 value of
  each binade [2^e, 2^(e+1)) is split into theta' + rho and merged back
  (``fo_split`` / ``fo_merge``, 8- and 16-bit rho). Reported per binade: the
  share reconstructed bit-exactly and the mean and largest relative error.
  The page's comparison scheme, BF16 + BF16 (the rounding error itself stored
  as BF16), is evaluated beside it with torch casts: it is a reference point
  for the figure, not part of the library.
* Fig. 4 (same section, state quantization): Adam-like momentum and second
  moment built from heavy-tailed (Student-t, nu = 3) gradients with per-group
  magnitudes spread over several decades, quantized and decoded with the
  companded codecs and with the plain linear ones (``fo_quant_state`` /
  ``fo_dequant_state``, ``FO_STATE_*`` and ``FO_STATE_*_LINEAR``). Reported:
  quantiles of the per-group normalised squared error
  sum (x - x^)^2 / sum x^2 and the share of groups decoded to all zeros.

* Second-moment safety: the fused AdamW step with and without
  ``FO_ADAMW_V_NONZERO`` on identical spiky gradients, counting the elements
  whose v decodes to 0 while their momentum does not, and the largest update.

The codec kernels' throughput is measured on the way (CUDA events, bytes each
kernel must move). ``python -m quantized_optimizer_state_gb300.codec_study``
prints one JSON document.
"""
from __future__ import annotations

import argparse
import json
from typing import Dict, Iterable, List, Sequence

import torch

from . import fo

BINADE = 1 << 23   # FP32 values per binade


def binade_values(e: int, device, stride: int = 1) -> torch.Tensor:
    """All (or every stride-th) positive FP32 values in [2^e, 2^(e+1)), e in [-126, 127]."""
    lo = (e + 127) << 23
    bits = torch.arange(0, BINADE, stride, dtype=torch.int64, device=device) + lo
    return bits.to(torch.int32).view(torch.float32)


def _stats(theta: torch.Tensor, rec: torch.Tensor) -> Dict[str, float]:
    exact = (rec.view(torch.int32) == theta.view(torch.int32)).double().mean().item()
    t64 = theta.double()
    rel = (rec.double() - t64).abs() / t64
    return {"exact_percent": 100.0 * exact, "mean_rel": rel.mean().item(), "max_rel": rel.max().item()}


def split_merge(theta: torch.Tensor, rho_bits: int) -> torch.Tensor:
    """theta^ = merge(split(theta)) through the library."""
    n = theta.numel()
    tp = torch.empty(n, dtype=torch.int16, device=theta.device)
    rho = torch.empty(n, dtype=torch.int16 if rho_bits == 16 else torch.int8, device=theta.device)
    rec = torch.empty_like(theta)
    fo.fo_split(theta, tp, rho, rho_bits)
    fo.fo_merge(tp, rho, rec, rho_bits)
    return rec


def bf16_pair(theta: torch.Tensor) -> torch.Tensor:
    """The page's comparison scheme: theta' = BF16(theta), e = BF16(theta - theta'),
    rebuilt as theta' + e in FP32."""
    tb = theta.to(torch.bfloat16).float()
    e = (theta - tb).to(torch.bfloat16).float()
    return tb + e


def reconstruction_sweep(exponents: Iterable[int], device="cuda", stride: int = 1,
                         rho_bits: Sequence[int] = (8, 16)) -> List[Dict]:
    """Fig. 3: one row per binade with the statistics of each scheme."""
    rows = []
    for e in exponents:
        theta = binade_values(e, device, stride)
        row = {"binade": e, "values": theta.numel()}
        for rb in rho_bits:
            row[f"rho{rb}"] = _stats(theta, split_merge(theta, rb))
        row["bf16_bf16"] = _stats(theta, bf16_pair(theta))
        rows.append(row)
    return rows


def _summary(rows: List[Dict], key: str) -> Dict[str, float]:
    n = sum(r["values"] for r in rows)
    return {
        "exact_percent": sum(r[key]["exact_percent"] * r["values"] for r in rows) / n,
        "mean_rel": sum(r[key]["mean_rel"] * r["values"] for r in rows) / n,
        "max_rel": max(r[key]["max_rel"] for r in rows),
    }


def adam_like_state(n_groups: int, seed: int, device="cuda", steps: int = 20, beta1: float = 0.9,
                    beta2: float = 0.999, decades=(-6.0, -1.0)):
    """Momentum and second moment after `steps` EMA updates of Student-t(3)
    gradients whose per-group scale is log-uniform over `decades` (base 10)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    n = n_groups * 32
    scale = torch.pow(10.0, torch.empty(n_groups, device=device).uniform_(*decades, generator=gen))
    scale = scale.repeat_interleave(32)
    m = torch.zeros(n, device=device)
    v = torch.zeros(n, device=device)
    for _ in range(steps):
        z = torch.randn(n, device=device, generator=gen)
        c = torch.randn(3, n, device=device, generator=gen).square().sum(0)
        g = z / torch.sqrt(c / 3.0) * scale
        m.mul_(beta1).add_(g, alpha=1 - beta1)
        v.mul_(beta2).addcmul_(g, g, value=1 - beta2)
    return m, v


def quantize_roundtrip(x: torch.Tensor, kind: int) -> torch.Tensor:
    n = x.numel()
    signed = kind in (fo.FO_STATE_MOMENTUM, fo.FO_STATE_MOMENTUM_LINEAR)
    q = torch.empty(n, dtype=torch.int8 if signed else torch.uint8, device=x.device)
    s = torch.empty((n + 31) // 32, dtype=torch.int16, device=x.device)
    out = torch.empty_like(x)
    fo.fo_quant_state(x, q, s, kind)
    fo.fo_dequant_state(q, s, out, kind)
    return out


def group_nmse(x: torch.Tensor, xh: torch.Tensor) -> torch.Tensor:
    """Per-group sum (x - x^)^2 / sum x^2 (groups of 32; all-zero groups dropped)."""
    xg = x.double().view(-1, 32)
    d = (xh.double().view(-1, 32) - xg).square().sum(1)
    p = xg.square().sum(1)
    keep = p > 0
    return d[keep] / p[keep]


QUANTILES = (0.5, 0.9, 0.99, 0.999)


def _nmse_summary(x: torch.Tensor, xh: torch.Tensor) -> Dict[str, float]:
    e = group_nmse(x, xh)
    qs = torch.quantile(e.float().cpu(), torch.tensor(QUANTILES)).tolist()
    lost = ((xh.view(-1, 32) == 0).all(1) & (x.view(-1, 32) != 0).any(1)).double().mean().item()
    out = {f"p{q * 100:g}": v for q, v in zip(QUANTILES, qs)}
    out.update({"mean": e.mean().item(), "max": e.max().item(), "all_zero_groups_percent": 100.0 * lost})
    return out


def nmse_study(n_groups: int = 1 << 20, seed: int = 0, device="cuda", decades=(-6.0, -1.0)) -> Dict:
    """Fig. 4: per-group NMSE of the companded and the linear codecs."""
    m, v = adam_like_state(n_groups, seed, device, decades=decades)
    return {
        "groups": n_groups,
        "grad_scale_decades": list(decades),
        "momentum": {"companded": _nmse_summary(m, quantize_roundtrip(m, fo.FO_STATE_MOMENTUM)),
                     "linear": _nmse_summary(m, quantize_roundtrip(m, fo.FO_STATE_MOMENTUM_LINEAR))},
        "variance": {"companded": _nmse_summary(v, quantize_roundtrip(v, fo.FO_STATE_VARIANCE)),
                     "linear": _nmse_summary(v, quantize_roundtrip(v, fo.FO_STATE_VARIANCE_LINEAR))},
    }


def zero_v_events(st: "fo.CompressedTensor") -> int:
    """Elements whose second moment decodes to 0 while their momentum does not
    (v code 0 in a group with a non-zero scale, m code non-zero): the next step
    divides a non-zero momentum by sqrt(0) + eps there."""
    vq = st.v_q.view(-1, 32) if st.numel % 32 == 0 else None
    if vq is None:
        raise ValueError("whole groups only")
    live = (st.v_scale != 0).view(-1, 1)
    return int(((vq == 0) & live & (st.m_q.view(-1, 32) != 0)).sum().item())


def variance_safety_study(n: int = 1 << 22, steps: int = 200, seed: int = 0, device="cuda",
                          lr: float = 1e-3, spike_prob: float = 1e-4, spike: float = 1e3) -> Dict:
    """Run the fused AdamW step with and without FO_ADAMW_V_NONZERO on the same
    gradients: Student-t(3) noise of scale 1e-3 with rare spikes (probability
    spike_prob, size x spike) that pin a group's v scale for thousands of steps.
    Reports per mode the zero-decode events per step and the largest update
    |theta_t - theta_{t-1}| in units of lr."""
    fo.lib()
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    theta0 = torch.randn(n, device=device, generator=gen) * 0.02
    modes = {}
    for name, flag in (("plain", False), ("v_nonzero", True)):
        st = fo.CompressedTensor(n, device, 8, True, 0.01)
        st.init_from(theta0)
        modes[name] = (st, flag, {"events": [], "max_update_lr": [], "p999_update_lr": []})
    prev = {k: theta0.clone() for k in modes}
    cur = torch.empty(n, device=device)
    for t in range(1, steps + 1):
        z = torch.randn(n, device=device, generator=gen)
        c = torch.randn(3, n, device=device, generator=gen).square().sum(0)
        g = z / torch.sqrt(c / 3.0) * 1e-3
        spikes = torch.rand(n, device=device, generator=gen) < spike_prob
        g = torch.where(spikes, g * spike, g).to(torch.bfloat16)
        for name, (st, flag, rec) in modes.items():
            fo.fo_adamw_step(fo.table_of([st], [g]), lr, 0.9, 0.999, 1e-8, t, v_nonzero=flag)
            fo.fo_merge(st.theta, st.rho, cur, 8)
            upd = (cur - prev[name]).abs() / lr
            rec["events"].append(zero_v_events(st))
            rec["max_update_lr"].append(upd.max().item())
            rec["p999_update_lr"].append(torch.quantile(upd[:1 << 20], 0.999).item())
            prev[name].copy_(cur)
    out = {"params": n, "steps": steps, "spike_prob": spike_prob, "spike": spike}
    for name, (_, _, rec) in modes.items():
        ev = rec["events"]
        out[name] = {
            "events_total": int(sum(ev)), "events_last_step": ev[-1],
            "steps_with_events": int(sum(1 for e in ev if e)),
            "max_update_lr": max(rec["max_update_lr"]),
            "p999_update_lr_last": rec["p999_update_lr"][-1],
        }
    return out


def _time(fn, reps: int) -> float:
    """Mean milliseconds of fn() over reps launches on the current stream."""
    fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def codec_throughput(n: int = 1 << 28, device="cuda", reps: int = 10) -> Dict[str, Dict[str, float]]:
    """GB/s of each codec kernel over n elements (inputs larger than L2),
    counting the bytes it must move (each once)."""
    x = torch.randn(n, device=device) * 0.02
    tp = torch.empty(n, dtype=torch.int16, device=device)
    r8 = torch.empty(n, dtype=torch.int8, device=device)
    q = torch.empty(n, dtype=torch.int8, device=device)
    s = torch.empty((n + 31) // 32, dtype=torch.int16, device=device)
    out = torch.empty_like(x)
    sb = 2 * ((n + 31) // 32)
    cases = {
        "split_rho8": (lambda: fo.fo_split(x, tp, r8, 8), 4 * n + 2 * n + n),
        "merge_rho8": (lambda: fo.fo_merge(tp, r8, out, 8), 2 * n + n + 4 * n),
        "quant_momentum": (lambda: fo.fo_quant_state(x, q, s, fo.FO_STATE_MOMENTUM), 4 * n + n + sb),
        "dequant_momentum": (lambda: fo.fo_dequant_state(q, s, out, fo.FO_STATE_MOMENTUM), n + sb + 4 * n),
    }
    res = {}
    for name, (fn, nbytes) in cases.items():
        ms = _time(fn, reps)
        res[name] = {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9}
    return res


def run(quick: bool = False, device="cuda") -> Dict:
    fo.lib()
    # FP16's normal range is [2^-14, 65504]; BF16 spans FP32's normal
    # exponents, up to the binade below 2^127 (above the largest BF16, theta'
    # would round to infinity, outside the splitting's domain)
    fp16_range = range(-14, 16)
    bf16_range = range(-126, 127, 1 if not quick else 23)
    stride = 1 if not quick else 257
    sweep_fp16 = reconstruction_sweep(fp16_range, device, stride)
    sweep_bf16 = reconstruction_sweep(bf16_range, device, stride)
    out = {
        "figure3": {
            "fp16_range": {k: _summary(sweep_fp16, k) for k in ("rho8", "rho16", "bf16_bf16")},
            "bf16_range": {k: _summary(sweep_bf16, k) for k in ("rho8", "rho16", "bf16_bf16")},
            "stride": stride,
            "binades_fp16": [sweep_fp16[0]["binade"], sweep_fp16[-1]["binade"]],
            "per_binade_bf16": sweep_bf16,
        },
        # gradient scales over five decades (v reaches below FP16's range),
        # and over two (every group's v has an FP16 scale)
        "figure4": nmse_study(1 << (14 if quick else 20), 0, device, decades=(-6.0, -1.0)),
        "figure4_fp16_scales": nmse_study(1 << (14 if quick else 20), 1, device, decades=(-2.0, 0.0)),
        "variance_safety": variance_safety_study(1 << (18 if quick else 22), 50 if quick else 300, 0, device),
        "throughput": codec_throughput(1 << (24 if quick else 28), device),
    }
    return out


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--quick", action="store_true", help="strided sweep and small NMSE sample")
    p.add_argument("--per-binade", action="store_true", help="keep the per-binade rows in the output")
    args = p.parse_args(argv)
    res = run(args.quick)
    if not args.per_binade:
        res["figure3"].pop("per_binade_bf16")
    print(json.dumps(res, indent=1))
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
