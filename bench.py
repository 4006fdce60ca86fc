"""Benchmark of the fused compressed optimizer step (FlashAdamW) on GB300.

Default workload: the Llama-3.1-8B parameter table (291 tensors, 8.03e9
parameters, BF16 theta' + INT8 rho + INT8 m + UINT8 v, FP16 group scales),
one fused FlashAdamW step per iteration over the whole table -- one kernel
launch of the library per step. Inputs are seeded synthetic tensors drawn on
the device; nothing is skipped inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
("replicas only": the step has no exchange), the timed region is bracketed by
barriers, the time is the maximum over ranks and rank 0 prints one JSON line.
``--impl reference`` times the CPU oracle (plain scalar C) on the host cores
over a bounded sample of the same workload and prints the same line.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The end-to-end leg runs copy-in, step and copy-out on three streams. With
# CUDA's default of 8 hardware work queues per device, streams can share a
# queue, and a copy-out waiting on its step then holds back a copy-in queued
# behind it (the two link directions stop overlapping). One queue per stream
# avoids that (198.7-201.6 against 127.2-138.4 ms per step on one box); it
# must be set before CUDA is initialised.
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")

METRIC = "FlashAdamW step params/s and achieved HBM GB/s vs ~8 TB/s (1xGB300)"
UNIT = "params/s"
# bytes one FlashAdamW step must move per parameter (each byte once):
# read grad 2 + theta' 2 + rho 1 + m 1 + v 1 + 2 FP16 scales / 32, write all but
# grad: 12.25 (8-bit rho), 14.25 (16-bit); an FP32 gradient reads 2 more
GRAD_BYTES = {"bf16": 2, "f32": 4}
FALLBACK_HBM_GBS = 6800.0
CPU_SAMPLE_ROWS = ("layers.0.input_layernorm.weight", "layers.0.post_attention_layernorm.weight",
                   "layers.0.self_attn.q_proj.weight", "layers.0.self_attn.k_proj.weight",
                   "layers.0.self_attn.v_proj.weight", "layers.0.self_attn.o_proj.weight")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="llama31_8b")
    p.add_argument("--rho-bits", type=int, default=8, choices=(8, 16))
    p.add_argument("--grad-dtype", default="bf16", choices=tuple(GRAD_BYTES),
                   help="gradient element type the fused step reads")
    p.add_argument("--v-nonzero", action="store_true",
                   help="AdamW: requantize v with no code 0 in groups with a non-zero scale (opt-in rule)")
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="time budget of the CPU oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--record-traffic", metavar="CSV:WORKLOAD[,CSV:WORKLOAD]",
                   help="store the DRAM bytes per parameter of ncu --csv captures of one step-kernel launch each "
                        "(two sizes: the slope between them) for --rho-bits, --grad-dtype, and exit")
    p.add_argument("--traffic-command", default=None, help="the ncu command line, recorded with --record-traffic")
    p.add_argument("--grad-release", action="store_true",
                   help="time gradient release against a plain step() on --workload (GPT-2 small by default) and exit")
    p.add_argument("--grad-release-gemm-tokens", type=int, default=0,
                   help="--grad-release with a GEMM backward over this many tokens per matrix parameter")
    p.add_argument("--oracle-full-step", action="store_true",
                   help="time the oracle over one step of the whole table (one-off measurement; prints one JSON line)")
    p.add_argument("--no-per-config", action="store_true",
                   help="skip timing the other workloads (flat 1M, GPT-2 small, ResNet-50, Lion 8B, stress set)")
    return p.parse_args(argv)


def _workload(args):
    """The named workload; --v-nonzero adds the opt-in v rule to AdamW's hyper-parameters."""
    import dataclasses
    from quantized_optimizer_state_gb300 import workloads as wl
    w = wl.workload(args.workload, args.rho_bits)
    if getattr(args, "v_nonzero", False):
        if w.optimizer != "adamw":
            raise SystemExit("--v-nonzero applies to AdamW workloads only")
        w = dataclasses.replace(w, hparams=dict(w.hparams, v_nonzero=True))
    return w


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _config(w, rho_bits, n_gpus, grad_dtype="bf16"):
    gname = grad_dtype.upper().replace("F32", "FP32")
    return {
        "workload": f"{w.name}: {len(w.params)} tensors, {w.numel} params, Flash{w.optimizer}"
                    f" step (BF16 theta' + INT{rho_bits} rho + INT8 m"
                    f"{' + UINT8 v' if w.optimizer == 'adamw' else ''}, G=32 FP16 scales,"
                    f" {gname} grads)",
        "params": w.numel,
        "tensors": len(w.params),
        "optimizer": w.optimizer,
        "rho_bits": rho_bits,
        "grad_dtype": grad_dtype,
        "hparams": w.hparams,
        "algorithmic_bytes_per_param": _algo_bytes(w, rho_bits, grad_dtype),
        "l2": "inputs larger than L2 (each step streams ~%.0f GB)"
              % (w.numel * _algo_bytes(w, rho_bits, grad_dtype) / 1e9),
        "grads": f"one seeded synthetic {gname} gradient set, reused every step",
        "parallelism": "replicas" if n_gpus > 1 else "single GPU",
    }


def _algo_bytes(w, rho_bits, grad_dtype="bf16"):
    """Read and write theta' (2), rho (1 or 2), m (1), v (1, AdamW) and their FP16
    group scales (2/32 each); read the gradient."""
    state = 2 + rho_bits // 8 + 1 + 2 / 32
    if w.optimizer == "adamw":
        state += 1 + 2 / 32
    return 2 * state + GRAD_BYTES[grad_dtype]


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (the cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def _cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleSample:
    """Host state of a few rows of the workload (or, with whole_table, of all of
    them), cut into group-aligned chunks that the oracle steps on parallel
    threads (the oracle itself is untouched). The sample's inputs come from the
    host generators; the whole table's from the seeded device generators,
    copied to the host (8e9 values would take minutes on the host)."""

    def __init__(self, w, rho_bits, grad_dtype="bf16", chunk=1 << 20, whole_table=False):
        import numpy as np
        import oracle
        from quantized_optimizer_state_gb300 import workloads as wl
        self.w = w
        names = {p.name: i for i, p in enumerate(w.params)}
        rows = list(range(len(w.params))) if whole_table else \
            ([names[n] for n in CPU_SAMPLE_ROWS if n in names] or [0])
        self.states, self.grads, self.chunks = [], [], []
        with_v = w.optimizer == "adamw"
        self.threads = _cpu_threads()

        def host_inputs(i):
            p = w.params[i]
            g = (wl.workload_grad_fp32 if grad_dtype == "f32" else wl.workload_grad_bf16)(w, i, 1)
            return wl.init_weight(p, i), g

        def device_inputs(i):
            import torch
            dev = torch.device("cuda", torch.cuda.current_device())
            theta = wl.init_weight_device(w.params[i], i, dev).cpu().numpy()
            g = wl.workload_grad_device(w, i, 1, dev, fp32=grad_dtype == "f32").cpu()
            g = g.numpy() if grad_dtype == "f32" else g.view(torch.int16).numpy().view(np.uint16)
            return theta, g

        def prepare(i):
            theta, g = (device_inputs if whole_table else host_inputs)(i)
            return oracle.State.from_fp32(theta, rho_bits, with_v, w.hparams["weight_decay"]), g

        t0 = time.perf_counter()
        with cf.ThreadPoolExecutor(self.threads) as pool:
            prepared = list(pool.map(prepare, rows))
        self.setup_seconds = time.perf_counter() - t0
        for i, (st, g) in zip(rows, prepared):
            p = w.params[i]
            self.states.append(st)
            self.grads.append(g)
            for lo in range(0, p.numel, chunk):
                hi = min(p.numel, lo + chunk)
                g0, g1 = lo // 32, (hi + 31) // 32
                sub = oracle.State(st.theta_p[lo:hi], st.rho[lo:hi], st.m_q[lo:hi], st.m_scale[g0:g1],
                                   None if st.v_q is None else st.v_q[lo:hi],
                                   None if st.v_scale is None else st.v_scale[g0:g1],
                                   st.weight_decay, rho_bits)
                self.chunks.append((sub, np.ascontiguousarray(g[lo:hi])))
        self.params = sum(s.numel for s in self.states)
        self.pool = cf.ThreadPoolExecutor(self.threads)
        if whole_table:
            self.desc = (f"the whole table ({len(rows)} rows, {self.params} params), {len(self.chunks)} chunks "
                         f"on {self.threads} threads")
        else:
            self.desc = (f"{len(rows)} rows of layer 0 ({self.params} params: "
                         + ", ".join(w.params[i].name.split('.')[-2] for i in rows)
                         + f"), {len(self.chunks)} chunks on {self.threads} threads")

    def step(self, t):
        import oracle
        hp = self.w.hparams
        if self.w.optimizer == "adamw":
            vnz = bool(hp.get("v_nonzero", False))
            f = lambda c: oracle.adamw_step([c[0]], [c[1]], hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], t,
                                            v_nonzero=vnz)
        elif self.w.optimizer == "sgd":
            f = lambda c: oracle.sgd_step([c[0]], [c[1]], hp["lr"], hp["momentum"])
        else:
            f = lambda c: oracle.lion_step([c[0]], [c[1]], hp["lr"], hp["beta1"], hp["beta2"])
        list(self.pool.map(f, self.chunks))

    def close(self):
        self.pool.shutdown()


def cpu_baseline(w, rho_bits, seconds, grad_dtype="bf16"):
    s = OracleSample(w, rho_bits, grad_dtype)
    s.step(1)                                   # warm-up
    t0 = time.perf_counter()
    steps = 0
    while True:
        s.step(2 + steps)
        steps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    s.close()
    return {"value": s.params * steps / dt, "unit": UNIT, "cores": s.threads, "kind": "oracle",
            "sample": f"{s.desc}; {steps} steps in {dt:.1f} s"}


def oracle_full_step(args):
    """The cpu_baseline leg with the whole table as its sample: the oracle over
    one step of every parameter of the workload (all of Llama-3.1-8B by
    default) on the host cores. A one-off measurement beside the bounded
    sample that the default line reports."""
    w = _workload(args)
    s = OracleSample(w, args.rho_bits, args.grad_dtype, whole_table=True)
    t0 = time.perf_counter()
    s.step(1)
    dt = time.perf_counter() - t0
    s.close()
    out = {"oracle_full_step": {"workload": w.name, "params": s.params, "tensors": len(s.states),
                                "optimizer": w.optimizer, "step_seconds": dt, "params_per_s": s.params / dt,
                                "threads": s.threads, "chunks": len(s.chunks), "setup_seconds": s.setup_seconds,
                                "sample": s.desc}}
    print(json.dumps(out), flush=True)
    return 0


def run_reference(args):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return 0
    from quantized_optimizer_state_gb300 import workloads as wl
    w = _workload(args)
    s = OracleSample(w, args.rho_bits, args.grad_dtype)
    for t in range(1, args.warmup + 1):
        s.step(t)
    t0 = time.perf_counter()
    for k in range(args.steps):
        s.step(args.warmup + 1 + k)
    dt = time.perf_counter() - t0
    s.close()
    value = s.params * args.steps / dt
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": _config(w, args.rho_bits, ws, args.grad_dtype),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": s.threads, "kind": "oracle",
                         "sample": f"each step: {s.desc}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_start, t_end):
        rows = [l for (t, l) in self.lines if t_start - 0.1 <= t <= t_end + 0.3]
        mhz, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in rows:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


def _gpu_id_for_smi(device_index: int) -> str:
    import torch
    try:
        p = torch.cuda.get_device_properties(device_index)
        return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[device_index] if vis else str(device_index)


# ---------------------------------------------------------------------------
# The GPU arm
# ---------------------------------------------------------------------------

# DRAM traffic of the step kernel, captured with ncu on a small case and
# stored per parameter (see record_traffic); valid while the sources hash to
# the captured version.
TRAFFIC = os.path.join(ROOT, "profiles", "fo_fused_step_kernel_traffic.json")
STEP_SOURCES = ("fo_api.cu", "fo_device.cuh", "fo_internal.h", "fo_pair.cuh", "fo_step.cu", "fo_step.cuh",
                "fo_step_adamw.cu", "fo_step_adamw_dev.cu", "fo_step_sgd.cu", "fo_step_lion.cu")


def _kernel_source_hash() -> str:
    """sha256 (first 16 hex digits) of the sources that build and launch the
    fused step kernel (the codec kernels' file is not among them) and the C
    header."""
    import hashlib
    csrc = os.path.join(ROOT, "quantized_optimizer_state_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in STEP_SOURCES]
    files.append(os.path.join(ROOT, "include", "fo.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_key(optimizer: str, rho_bits: int, grad_dtype: str) -> str:
    return f"{optimizer}_rho{rho_bits}_{grad_dtype}"


def _profiled_traffic(optimizer: str, rho_bits: int, grad_dtype: str, params: int):
    """DRAM bytes per launch for a table of `params` parameters: the captured
    bytes per parameter of this kernel variant times the parameters, or None
    when no capture matches the current sources."""
    try:
        with open(TRAFFIC) as f:
            rec = json.load(f).get(_traffic_key(optimizer, rho_bits, grad_dtype))
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_sha256_16") != _kernel_source_hash():
        return None
    return float(rec["dram_bytes_per_param"]) * params


def _ncu_bytes(csv_path: str) -> float:
    """dram__bytes_read.sum + dram__bytes_write.sum of the one fused-step launch
    in an ncu --csv log."""
    import csv
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}
    with open(csv_path) as f:
        lines = f.read().splitlines()
    start = next(i for i, l in enumerate(lines) if l.startswith('"ID"'))
    rows = list(csv.reader(lines[start:]))
    h = rows[0]
    k, m, u, v = (h.index(x) for x in ("Kernel Name", "Metric Name", "Metric Unit", "Metric Value"))
    got = {}
    for r in rows[1:]:
        if len(r) > v and "fo_fused_step_kernel" in r[k] and r[m] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            got.setdefault(r[m], []).append(float(r[v].replace(",", "")) * scale[r[u]])
    if set(got) != {"dram__bytes_read.sum", "dram__bytes_write.sum"} or len(got["dram__bytes_read.sum"]) != 1:
        raise SystemExit(f"{csv_path}: expected one fused-step launch with both DRAM byte counters")
    return got["dram__bytes_read.sum"][0] + got["dram__bytes_write.sum"][0]


def record_traffic(args):
    """Store the DRAM bytes per parameter of the step kernel in TRAFFIC, keyed by
    kernel variant and stamped with the current source hash. args.record_traffic
    lists ncu --csv captures (one launch each, counters dram__bytes_read.sum and
    dram__bytes_write.sum) as CSV:WORKLOAD items separated by commas. With two
    captures of different sizes the figure is the slope between them: at the end
    of a launch up to an L2's worth of written lines can still sit in L2 (written
    back later), a constant that the difference cancels. With one capture it is
    that capture's bytes over its parameters."""
    from quantized_optimizer_state_gb300 import workloads as wl
    caps = []
    for item in args.record_traffic.split(","):
        path, _, name = item.partition(":")
        w = wl.workload(name or args.workload, args.rho_bits)
        caps.append((w, _ncu_bytes(path)))
    caps.sort(key=lambda c: c[0].numel)
    w = caps[-1][0]
    if len(caps) >= 2:
        (w0, b0), (w1, b1) = caps[0], caps[-1]
        per_param = (b1 - b0) / (w1.numel - w0.numel)
        how = f"slope between {w0.name} ({b0:.0f} B) and {w1.name} ({b1:.0f} B)"
    else:
        per_param = caps[0][1] / w.numel
        how = f"{w.name}: {caps[0][1]:.0f} B over its parameters"
    try:
        with open(TRAFFIC) as f:
            data = json.load(f)
    except (OSError, ValueError):
        data = {}
    key = _traffic_key(w.optimizer, args.rho_bits, args.grad_dtype)
    data[key] = {
        "source_sha256_16": _kernel_source_hash(), "captures": [[c[0].name, c[0].numel, c[1]] for c in caps],
        "dram_bytes_per_param": per_param, "derivation": how,
        "algorithmic_bytes_per_param": _algo_bytes(w, args.rho_bits, args.grad_dtype),
        "command": args.traffic_command or "",
    }
    with open(TRAFFIC, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps(data[key]))
    return 0


def _measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def flat_offsets(sizes, align=64):
    """Start offsets (in elements) of consecutive tensors in one flat buffer,
    each rounded up to a multiple of `align` elements (16-byte aligned for any
    element size), and the buffer's total length."""
    offs, at = [], 0
    for n in sizes:
        offs.append(at)
        at += (n + align - 1) // align * align
    return offs, at


def _build_states(w, rho_bits, device, grad_dtype="bf16"):
    """Compressed state and one gradient per tensor. theta' and the gradients of
    all rows are views into two flat buffers, so the end-to-end leg copies
    contiguous ranges."""
    import torch
    from quantized_optimizer_state_gb300 import fo
    from quantized_optimizer_state_gb300 import workloads as wl
    offs, total = flat_offsets([p.numel for p in w.params])
    gdt = torch.float32 if grad_dtype == "f32" else torch.bfloat16
    flat_theta = torch.empty(total, dtype=torch.int16, device=device)
    flat_grad = torch.empty(total, dtype=gdt, device=device)
    states, grads = [], []
    for i, p in enumerate(w.params):
        o = offs[i]
        d = fo.CompressedTensor(p.numel, device, rho_bits, w.optimizer == "adamw",
                                w.hparams["weight_decay"], theta=flat_theta[o:o + p.numel])
        theta = wl.init_weight_device(p, i, device)
        d.init_from(theta)
        del theta
        states.append(d)
        g = flat_grad[o:o + p.numel]
        g.copy_(wl.workload_grad_device(w, i, 1, device, fp32=grad_dtype == "f32"))
        grads.append(g)
    torch.cuda.synchronize(device)
    return states, grads, {"theta": flat_theta, "grad": flat_grad, "offs": offs}


def _stepper(w, table):
    return _stepper_of(w)(table)


def _stepper_of(w):
    """table -> step(t, stream) for the workload's optimizer."""
    hp = w.hparams
    return lambda table: _make_step(w.optimizer, hp, table)


def _make_step(opt, hp, table):
    from quantized_optimizer_state_gb300 import fo
    if opt == "adamw":
        vnz = bool(hp.get("v_nonzero", False))
        return lambda t, s: fo.fo_adamw_step(table, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], t, s,
                                             v_nonzero=vnz)
    if opt == "sgd":
        return lambda t, s: fo.fo_sgd_step(table, hp["lr"], hp["momentum"], s)
    return lambda t, s: fo.fo_lion_step(table, hp["lr"], hp["beta1"], hp["beta2"], s)


def reduce_scalar(x, op, ws, device=None):
    """x reduced over the ranks with op ("max" or "sum"); x itself when ws == 1."""
    if ws == 1 or op is None:
        return x
    import torch
    import torch.distributed as dist
    rop = {"max": dist.ReduceOp.MAX, "sum": dist.ReduceOp.SUM}.get(op, op)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=rop)
    return float(t.item())


def job_throughput(ws, params_per_rank, steps, elapsed_ms_max):
    """Whole-job params/s: all ranks' parameters over the slowest rank's time."""
    return ws * params_per_rank * steps / (elapsed_ms_max * 1e-3)


def run_ours(args):
    import torch
    import torch.distributed as dist
    from quantized_optimizer_state_gb300 import fo
    from quantized_optimizer_state_gb300 import workloads as wl

    ws, rank, local = _dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        if ws > 1:
            dist.barrier()

    def reduce(x, op):
        return reduce_scalar(x, op, ws, device)

    fo.lib()
    w = _workload(args)
    states, grads, flat = _build_states(w, args.rho_bits, device, args.grad_dtype)
    table = fo.table_of(states, grads)
    step = _stepper(w, table)
    stream = torch.cuda.current_stream(device)

    t = 0
    for _ in range(args.warmup):
        t += 1
        step(t, stream)
    torch.cuda.synchronize(device)

    sampler = ClockSampler(_gpu_id_for_smi(local))
    time.sleep(0.6)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_all0, t_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = fo.fo_kernel_launch_count()
    barrier()
    torch.cuda.synchronize(device)
    wall0 = time.time()
    t_all0.record(stream)
    for k in range(args.steps):
        t += 1
        ev[k][0].record(stream)
        step(t, stream)
        ev[k][1].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize(device)
    barrier()
    wall1 = time.time()
    launches = fo.fo_kernel_launch_count() - launches0
    time.sleep(0.3)
    sampler.stop()
    clocks = sampler.summary(wall0, wall1)

    elapsed_ms = t_all0.elapsed_time(t_all1)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    elapsed_ms = reduce(elapsed_ms, "max")
    launches_total = int(reduce(float(launches), "sum"))
    kernel_ms = statistics.mean(step_ms)     # one library kernel per step on this stream
    kernel_ms = reduce(kernel_ms, "max")

    # end to end through the public API with host buffers: per step, the BF16
    # gradients go host -> device from pinned memory and the updated BF16
    # theta' comes back device -> host; the step runs in between.
    e2e = None
    if not args.no_e2e:
        e2e = _e2e(w, states, grads, flat, _stepper_of(w), stream, device, args.e2e_steps, t, barrier, reduce, ws)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.rho_bits, args.cpu_seconds, args.grad_dtype)

    # the other configurations, one at a time after the headline's state is freed
    per_config = None
    if ws == 1 and not args.no_per_config:
        del table, step, states, grads, flat
        torch.cuda.empty_cache()
        per_config = {key: measure_config(name, rb, steps, 5, flush, device, stream)
                      for key, name, rb, steps, flush in PER_CONFIG}

    if rank == 0:
        peak, peak_kind = _measured_peak()
        algo = _algo_bytes(w, args.rho_bits, args.grad_dtype) * w.numel
        achieved = algo / (kernel_ms * 1e-3) / 1e9
        out = {
            "metric": METRIC, "value": job_throughput(ws, w.numel, args.steps, elapsed_ms), "unit": UNIT,
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": _config(w, args.rho_bits, ws, args.grad_dtype),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": _profiled_traffic(w.optimizer, args.rho_bits, args.grad_dtype, w.numel),
                         "kernel": f"fo_fused_step_kernel<{w.optimizer}>",
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s",
                         "algorithmic_bytes_per_launch": algo,
                         "kernel_ms_mean": kernel_ms, "kernel_ms_min": min(step_ms)},
            "gpu_launches": launches_total,
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "per_config": per_config,
        }
        print(json.dumps(out), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# Per-configuration figures (each of the other workloads, timed the same way)
# ---------------------------------------------------------------------------

# (key, workload, rho_bits, timed steps, flush L2 between steps). The 2^20-
# parameter step moves 12.8 MB, which fits in L2: it is timed as latency with
# a 512 MB write between steps, so every step starts from DRAM. The others
# stream far more than L2 holds per step.
PER_CONFIG = (
    ("flat_1m", "flat_1m", 8, 200, True),
    ("gpt2_small", "gpt2_small", 8, 300, False),
    ("gpt2_small_sparse_wte", "gpt2_small_sparse_wte", 8, 300, False),
    ("resnet50", "resnet50", 8, 500, False),
    ("llama31_8b_lion", "llama31_8b_lion", 8, 40, False),
    ("stress_64m_rho8", "stress_64m", 8, 100, False),
    ("stress_64m_rho16", "stress_64m", 16, 100, False),
)
L2_FLUSH_BYTES = 512 << 20


def measure_config(name, rho_bits, steps, warmup, flush, device, stream):
    """Time `steps` fused steps of workload `name` (one seeded gradient set),
    each bracketed by CUDA events on the launching stream; returns the
    per-configuration record."""
    import torch
    from quantized_optimizer_state_gb300 import fo
    from quantized_optimizer_state_gb300 import workloads as wl
    w = wl.workload(name, rho_bits)
    states, grads, flat = _build_states(w, rho_bits, device)
    step = _stepper(w, fo.table_of(states, grads))
    scratch = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device) if flush else None
    t = 0
    for _ in range(warmup):
        t += 1
        step(t, stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize(device)
    w0 = time.perf_counter()
    for k in range(steps):
        t += 1
        if scratch is not None:
            scratch.fill_(k & 0xFF)
        ev[k][0].record(stream)
        step(t, stream)
        ev[k][1].record(stream)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - w0
    ms = [a.elapsed_time(b) for a, b in ev]
    del states, grads, flat, scratch
    torch.cuda.empty_cache()
    peak, _ = _measured_peak()
    algo = _algo_bytes(w, rho_bits) * w.numel
    mean = statistics.mean(ms)
    return {"workload": name, "optimizer": w.optimizer, "rho_bits": rho_bits, "params": w.numel,
            "tensors": len(w.params), "steps": steps, "kernel_ms": mean, "kernel_ms_median": statistics.median(ms),
            "kernel_ms_min": min(ms), "ms_per_step": None if flush else 1e3 * wall / steps,
            "params_per_s": w.numel / (mean * 1e-3), "gbs": algo / (mean * 1e-3) / 1e9,
            "frac": algo / (mean * 1e-3) / 1e9 / peak, "algorithmic_bytes_per_step": algo,
            "timing": ("latency: CUDA events around each step, 512 MB written between steps (L2 flushed)"
                       if flush else "CUDA events around each step; each step streams more than L2 holds")}


def _chunks(sizes, n_chunks):
    """Consecutive tensor index ranges of roughly equal element counts."""
    total = sum(sizes)
    out, cur, acc = [], [], 0
    for i, n in enumerate(sizes):
        cur.append(i)
        acc += n
        if acc >= total * (len(out) + 1) / n_chunks and len(out) < n_chunks - 1:
            out.append(cur)
            cur = []
    if cur:
        out.append(cur)
    return out


def _async_engine_count(device_index: int):
    """cudaDevAttrAsyncEngineCount of the device (copy engines that can run
    concurrently with kernels and each other), read through the CUDA runtime;
    None if the runtime library cannot be found."""
    import ctypes
    import glob
    cands = ["libcudart.so", "libcudart.so.13", "libcudart.so.12"]
    cands += sorted(glob.glob("/usr/local/cuda/lib64/libcudart.so*"))
    for name in cands:
        try:
            rt = ctypes.CDLL(name)
        except OSError:
            continue
        v = ctypes.c_int(0)
        if rt.cudaDeviceGetAttribute(ctypes.byref(v), 40, device_index) == 0:   # cudaDevAttrAsyncEngineCount
            return int(v.value)
    return None


def _link_rates(h_src, d_dst, d_src, h_dst, nbytes, stream_a, stream_b, device):
    """Host-link rates (GB/s) with pinned buffers: host -> device alone, device
    -> host alone, and both at once on two streams (best of three each)."""
    import torch
    n_in = nbytes // h_src.element_size()
    n_out = nbytes // h_dst.element_size()

    def timed(fn):
        best = float("inf")
        for _ in range(3):
            torch.cuda.synchronize(device)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(device)
            best = min(best, time.perf_counter() - t0)
        return best

    def h2d():
        with torch.cuda.stream(stream_a):
            d_dst[:n_in].copy_(h_src[:n_in], non_blocking=True)

    def d2h():
        with torch.cuda.stream(stream_b):
            h_dst[:n_out].copy_(d_src[:n_out], non_blocking=True)

    def both():
        h2d()
        d2h()
    return {"h2d_gbs": nbytes / timed(h2d) / 1e9, "d2h_gbs": nbytes / timed(d2h) / 1e9,
            "both_directions_gbs": 2 * nbytes / timed(both) / 1e9, "probe_bytes": nbytes}


def _both_full_ms(h_src, d_dst, d_src, h_dst, piece, stream_a, stream_b, device):
    """Milliseconds to copy the whole of h_src to d_dst and of d_src to h_dst at
    once (two streams, pieces of `piece` elements interleaved): the end-to-end
    leg's own copies with no compute, the floor of one end-to-end step."""
    import torch
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    n_in, n_out = h_src.numel(), h_dst.numel()
    for a in range(0, max(n_in, n_out), piece):
        if a < n_in:
            with torch.cuda.stream(stream_a):
                d_dst[a:min(n_in, a + piece)].copy_(h_src[a:min(n_in, a + piece)], non_blocking=True)
        if a < n_out:
            with torch.cuda.stream(stream_b):
                h_dst[a:min(n_out, a + piece)].copy_(d_src[a:min(n_out, a + piece)], non_blocking=True)
    torch.cuda.synchronize(device)
    return (time.perf_counter() - t0) * 1e3


def _e2e(w, states, grads, flat, step_fn_of, stream, device, steps, t, barrier, reduce, ws, n_chunks=16,
         piece_bytes=128 << 20):
    """End to end through the C ABI with host buffers: every step copies all
    gradients host -> device from pinned memory and the updated BF16 theta'
    device -> host. The table is cut into chunks of consecutive tensors so that
    the copy-in of one chunk, the fused step of the previous one and the
    copy-out of the one before overlap on three streams (the step is independent
    per tensor). theta' and the gradients live in flat buffers, so each chunk's
    copies are contiguous ranges, issued in pieces of piece_bytes. On the GB300
    box that keeps both link directions busy at once, where whole-tensor copies
    of up to 1 GB did not overlap."""
    import torch
    from quantized_optimizer_state_gb300 import fo
    sizes = [p.numel for p in w.params]
    offs = flat["offs"]
    f_grad, f_theta = flat["grad"], flat["theta"]
    h_grad = torch.empty(f_grad.numel(), dtype=f_grad.dtype, pin_memory=True)
    h_out = torch.empty(f_theta.numel(), dtype=torch.int16, pin_memory=True)
    h_grad.copy_(f_grad)
    chunks = _chunks(sizes, n_chunks)
    ranges = [(offs[c[0]], offs[c[-1]] + sizes[c[-1]]) for c in chunks]
    steppers = [step_fn_of(fo.table_of([states[i] for i in c], [grads[i] for i in c])) for c in chunks]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    # what the host link and the copy engines allow on this machine, measured
    # before the timed region (the end-to-end time is bound by them)
    link = _link_rates(h_grad, f_grad, f_theta, h_out, min(1 << 30, h_out.numel() * 2), s_in, s_out, device)
    link["copy_engines"] = _async_engine_count(device.index if device.index is not None else 0)
    ev_in = [torch.cuda.Event() for _ in chunks]
    ev_done = [torch.cuda.Event() for _ in chunks]
    g_piece = max(1, piece_bytes // f_grad.element_size())
    t_piece = max(1, piece_bytes // 2)
    h2d = sum(hi - lo for lo, hi in ranges) * f_grad.element_size()
    d2h = sum(hi - lo for lo, hi in ranges) * 2

    def one(t):
        for c, (lo, hi) in enumerate(ranges):
            with torch.cuda.stream(s_in):
                for a in range(lo, hi, g_piece):
                    b = min(hi, a + g_piece)
                    f_grad[a:b].copy_(h_grad[a:b], non_blocking=True)
                ev_in[c].record(s_in)
            stream.wait_event(ev_in[c])
            steppers[c](t, stream)
            ev_done[c].record(stream)
            s_out.wait_event(ev_done[c])
            with torch.cuda.stream(s_out):
                for a in range(lo, hi, t_piece):
                    b = min(hi, a + t_piece)
                    h_out[a:b].copy_(f_theta[a:b], non_blocking=True)
        # the next step's copy-in overwrites gradients the step has read: order it
        s_in.wait_stream(stream)
        stream.wait_stream(s_out)

    t += 1
    one(t)                                   # warm-up
    torch.cuda.synchronize(device)
    # the same copies with no compute, just before and just after the timed
    # steps: the shared host link's concurrent rate varies over time on this
    # pool (the same 2 x 16 GB took 101-159 ms a minute apart in one process)
    piece = max(1, piece_bytes // 2)
    link["both_full_ms_before"] = _both_full_ms(h_grad.view(torch.int16), f_grad.view(torch.int16), f_theta, h_out,
                                                piece, s_in, s_out, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    s_in.wait_stream(stream)
    for _ in range(steps):
        t += 1
        one(t)
    e1.record(stream)
    torch.cuda.synchronize(device)
    link["both_full_ms_after"] = _both_full_ms(h_grad.view(torch.int16), f_grad.view(torch.int16), f_theta, h_out,
                                               piece, s_in, s_out, device)
    barrier()
    ms = reduce(e0.elapsed_time(e1), "max")
    return {"value": job_throughput(ws, w.numel, steps, ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / steps, "link": link,
            "path": f"pinned host {str(f_grad.dtype).split('.')[-1]} grads -> device, fused step,"
                    f" theta' -> pinned host; {len(chunks)} tensor chunks pipelined on copy-in/compute/"
                    f"copy-out streams, copies in {piece_bytes >> 20} MB pieces of flat buffers"}


# ---------------------------------------------------------------------------
# Gradient release against a plain optimizer step (drop-in optimizers)
# ---------------------------------------------------------------------------

def grad_release_study(name="gpt2_small", iters=20, warmup=5, gemm_tokens=0):
    """Backward + FlashAdamW step of a table's parameters three ways: a plain
    step() after backward, gradient release in buckets (the default size) and
    release of every parameter on its own. The backward pass is synthetic and
    identical in all three: the loss is sum(p * c) for a fixed random c per
    parameter (each gradient is c in BF16), or, with gemm_tokens = T > 0, for
    each matrix parameter p of shape (a, b) sum(x @ p) for a fixed random x of
    shape (T, a), so that forward and backward are GEMMs of 2abT flops each,
    as in a layer fed T tokens (a GPU-bound backward). Reported per
    iteration: the whole iteration (host wall time), the host time spent in
    the optimizer's stepping code, the GPU time of the optimizer's work (CUDA
    events around each of its calls) and its kernel launches."""
    import torch
    from quantized_optimizer_state_gb300 import fo, optim
    from quantized_optimizer_state_gb300 import workloads as wl
    w = wl.workload(name)
    dev = torch.device("cuda", torch.cuda.current_device())

    gen = torch.Generator(device=dev)
    gen.manual_seed(5)

    def make():
        ps, cs = [], []
        for i, p in enumerate(w.params):
            x = wl.init_weight_device(p, i, dev).view(p.shape)
            ps.append(torch.nn.Parameter(x))
            if gemm_tokens and len(p.shape) == 2:
                cs.append(torch.randn(gemm_tokens, p.shape[0], device=dev, generator=gen) * 0.01)
            else:
                cs.append(wl.workload_grad_device(w, i, 1, dev).view(p.shape))
        opt = optim.FlashAdamW(ps, lr=w.hparams["lr"], betas=(w.hparams["beta1"], w.hparams["beta2"]),
                               eps=w.hparams["eps"], weight_decay=w.hparams["weight_decay"])
        # the optimizer holds compressed parameters as their BF16 theta': the
        # GEMM inputs take the parameters' type
        cs = [c.to(p.dtype) if c.shape != p.shape else c for p, c in zip(ps, cs)]
        return ps, cs, opt

    def term(p, c):
        return (c @ p).float().sum() if c.shape != p.shape else (p * c).float().sum()

    out = {"study": "grad_release", "workload": name, "params": w.numel, "tensors": len(w.params),
           "iters": iters,
           "backward": f"GEMMs over {gemm_tokens} tokens per matrix" if gemm_tokens else "element-wise"}
    for mode, bucket in (("plain_step", None), ("release_bucketed", 1 << 24), ("release_per_parameter", 0)):
        ps, cs, opt = make()
        calls = []                      # (host seconds, start event, end event) per optimizer call
        inner = opt._step_params

        def timed_step_params(params, group, inner=inner, calls=calls):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            e0.record()
            inner(params, group)
            e1.record()
            calls.append((time.perf_counter() - t0, e0, e1))
        opt._step_params = timed_step_params
        if bucket is not None:
            opt.attach_grad_release(bucket_numel=bucket)

        def one():
            sum(term(p, c) for p, c in zip(ps, cs)).backward()
            if bucket is None:
                opt.step()
                opt.zero_grad(set_to_none=True)
        for _ in range(warmup):
            one()
        torch.cuda.synchronize(dev)
        calls.clear()
        l0 = fo.fo_kernel_launch_count()
        t0 = time.perf_counter()
        for _ in range(iters):
            one()
        torch.cuda.synchronize(dev)
        total = (time.perf_counter() - t0) * 1e3 / iters
        out[mode] = {"iteration_ms": total,
                     "optimizer_host_ms": 1e3 * sum(c[0] for c in calls) / iters,
                     "optimizer_gpu_ms": sum(c[1].elapsed_time(c[2]) for c in calls) / iters,
                     "optimizer_calls": len(calls) / iters,
                     "optimizer_launches": (fo.fo_kernel_launch_count() - l0) / iters,
                     "bucket_numel": bucket}
        del ps, cs, opt, calls
        torch.cuda.empty_cache()
    return out


def main(argv=None):
    args = parse_args(argv)
    if args.record_traffic:
        return record_traffic(args)
    if args.grad_release:
        print(json.dumps(grad_release_study(args.workload if args.workload != "llama31_8b" else "gpt2_small",
                                            gemm_tokens=args.grad_release_gemm_tokens)), flush=True)
        return 0
    if args.oracle_full_step:
        return oracle_full_step(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
