"""Seeded synthetic inputs for the fused optimizer step.

This module holds only parameter-list shapes and seeded random generators.
It contains none of the method's arithmetic (no splitting, companding,
quantization or optimizer update) so that the CUDA path and the CPU oracle can
both be fed from it without sharing any computation.

Workloads (parameter lists of public architectures, built from shapes only;
no weights or datasets are used or needed):

* ``flat_1m``    one flat tensor of 1,048,576 parameters, FlashAdamW.
* ``gpt2_small`` GPT-2 small, 148 tensors, 124,439,808 parameters, FlashAdamW.
* ``resnet50``   ResNet-50, 161 tensors, 25,557,032 parameters, FlashSGD.
* ``llama31_8b`` Llama-3.1-8B, 291 tensors, 8,030,261,248 parameters,
                 FlashAdamW (and FlashLion).
* ``flat_128m``, ``flat_256m`` one flat tensor of 2**27 or 2**28 parameters with the Llama-3.1-8B
                 table's distributions (weights N(0, 0.02), Student-t(3) x 1e-4
                 gradients), FlashAdamW: a small case of the same kernel for
                 DRAM-counter captures.
* ``gpt2_small_sparse_wte`` the GPT-2 small table whose token-embedding rows
                 get an exactly zero gradient at every step for a fixed 90 % of
                 the vocabulary (tokens no batch contains), FlashAdamW.
* ``stress_64m`` one flat tensor of 2**26 parameters with extreme magnitudes,
                 zeros and BF16 subnormals, FlashAdamW with 8- and 16-bit rho.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Sequence

import numpy as np

# ---------------------------------------------------------------------------
# Parameter lists
# ---------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class ParamSpec:
    """One parameter tensor: name, shape and how its initial FP32 value is drawn."""
    name: str
    shape: tuple
    init: str            # "normal", "ones", "zeros", "kaiming", "stress"
    std: float = 0.0     # for "normal"; fan-in for "kaiming" is taken from the shape

    @property
    def numel(self) -> int:
        return int(np.prod(self.shape))


def flat_params(n: int, init: str = "normal", std: float = 0.02) -> List[ParamSpec]:
    return [ParamSpec("flat", (n,), init, std)]


def gpt2_small_params() -> List[ParamSpec]:
    """GPT-2 small: 12 layers, d=768, MLP 3072, vocab 50257, ctx 1024, head tied."""
    d, f, vocab, ctx = 768, 3072, 50257, 1024
    ps = [ParamSpec("wte", (vocab, d), "normal", 0.02),
          ParamSpec("wpe", (ctx, d), "normal", 0.02)]
    for i in range(12):
        p = f"h.{i}."
        ps += [ParamSpec(p + "ln_1.weight", (d,), "ones"),
               ParamSpec(p + "ln_1.bias", (d,), "zeros"),
               ParamSpec(p + "attn.c_attn.weight", (d, 3 * d), "normal", 0.02),
               ParamSpec(p + "attn.c_attn.bias", (3 * d,), "zeros"),
               ParamSpec(p + "attn.c_proj.weight", (d, d), "normal", 0.02),
               ParamSpec(p + "attn.c_proj.bias", (d,), "zeros"),
               ParamSpec(p + "ln_2.weight", (d,), "ones"),
               ParamSpec(p + "ln_2.bias", (d,), "zeros"),
               ParamSpec(p + "mlp.c_fc.weight", (d, f), "normal", 0.02),
               ParamSpec(p + "mlp.c_fc.bias", (f,), "zeros"),
               ParamSpec(p + "mlp.c_proj.weight", (f, d), "normal", 0.02),
               ParamSpec(p + "mlp.c_proj.bias", (d,), "zeros")]
    ps += [ParamSpec("ln_f.weight", (d,), "ones"), ParamSpec("ln_f.bias", (d,), "zeros")]
    return ps


def resnet50_params() -> List[ParamSpec]:
    """ResNet-50 (bottleneck blocks 3-4-6-3, expansion 4, 1000 classes)."""
    ps = [ParamSpec("conv1.weight", (64, 3, 7, 7), "kaiming")]
    ps += _bn("bn1", 64)
    inplanes = 64
    for li, (planes, blocks) in enumerate([(64, 3), (128, 4), (256, 6), (512, 3)], start=1):
        for b in range(blocks):
            p = f"layer{li}.{b}."
            out = planes * 4
            ps += [ParamSpec(p + "conv1.weight", (planes, inplanes, 1, 1), "kaiming")]
            ps += _bn(p + "bn1", planes)
            ps += [ParamSpec(p + "conv2.weight", (planes, planes, 3, 3), "kaiming")]
            ps += _bn(p + "bn2", planes)
            ps += [ParamSpec(p + "conv3.weight", (out, planes, 1, 1), "kaiming")]
            ps += _bn(p + "bn3", out)
            if b == 0:
                ps += [ParamSpec(p + "downsample.0.weight", (out, inplanes, 1, 1), "kaiming")]
                ps += _bn(p + "downsample.1", out)
            inplanes = out
    ps += [ParamSpec("fc.weight", (1000, 2048), "normal", 0.01),
           ParamSpec("fc.bias", (1000,), "zeros")]
    return ps


def _bn(prefix: str, c: int) -> List[ParamSpec]:
    return [ParamSpec(prefix + ".weight", (c,), "ones"), ParamSpec(prefix + ".bias", (c,), "zeros")]


def llama31_8b_params(layers: int = 32) -> List[ParamSpec]:
    """Llama-3.1-8B: hidden 4096, MLP 14336, 32 q / 8 kv heads of 128, vocab 128256."""
    h, f, kv, vocab = 4096, 14336, 1024, 128256
    ps = [ParamSpec("embed_tokens.weight", (vocab, h), "normal", 0.02)]
    for i in range(layers):
        p = f"layers.{i}."
        ps += [ParamSpec(p + "self_attn.q_proj.weight", (h, h), "normal", 0.02),
               ParamSpec(p + "self_attn.k_proj.weight", (kv, h), "normal", 0.02),
               ParamSpec(p + "self_attn.v_proj.weight", (kv, h), "normal", 0.02),
               ParamSpec(p + "self_attn.o_proj.weight", (h, h), "normal", 0.02),
               ParamSpec(p + "mlp.gate_proj.weight", (f, h), "normal", 0.02),
               ParamSpec(p + "mlp.up_proj.weight", (f, h), "normal", 0.02),
               ParamSpec(p + "mlp.down_proj.weight", (h, f), "normal", 0.02),
               ParamSpec(p + "input_layernorm.weight", (h,), "ones"),
               ParamSpec(p + "post_attention_layernorm.weight", (h,), "ones")]
    ps += [ParamSpec("norm.weight", (h,), "ones"),
           ParamSpec("lm_head.weight", (vocab, h), "normal", 0.02)]
    return ps


# ---------------------------------------------------------------------------
# Workload definitions
# ---------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    params: Sequence[ParamSpec]
    optimizer: str               # "adamw", "sgd", "lion"
    hparams: dict
    steps: int
    grad: str                    # "normal", "student_t", "stress"
    grad_scale: float
    rho_bits: int = 8
    # tensor name -> fraction of its rows (first dimension) whose gradient is
    # exactly zero at every step (for example embedding rows no token touches)
    zero_rows: tuple = ()

    @property
    def numel(self) -> int:
        return sum(p.numel for p in self.params)


ADAMW_HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
SGD_HP = dict(lr=0.1, momentum=0.9, weight_decay=1e-4)
LION_HP = dict(lr=1e-4, beta1=0.9, beta2=0.99, weight_decay=0.01)


def workload(name: str, rho_bits: int = 8) -> Workload:
    if name == "flat_1m":
        return Workload(name, flat_params(1 << 20), "adamw", ADAMW_HP, 10, "normal", 1e-3, rho_bits)
    if name == "gpt2_small":
        return Workload(name, gpt2_small_params(), "adamw", ADAMW_HP, 100, "student_t", 1e-4,
                        rho_bits)
    if name == "resnet50":
        return Workload(name, resnet50_params(), "sgd", SGD_HP, 50, "normal", 1e-3, rho_bits)
    if name == "llama31_8b":
        return Workload(name, llama31_8b_params(), "adamw", ADAMW_HP, 5, "student_t", 1e-4,
                        rho_bits)
    if name == "llama31_8b_lion":
        return Workload(name, llama31_8b_params(), "lion", LION_HP, 5, "student_t", 1e-4,
                        rho_bits)
    if name == "flat_128m":
        return Workload(name, flat_params(1 << 27), "adamw", ADAMW_HP, 5, "student_t", 1e-4, rho_bits)
    if name == "flat_256m":
        return Workload(name, flat_params(1 << 28), "adamw", ADAMW_HP, 5, "student_t", 1e-4, rho_bits)
    if name == "gpt2_small_sparse_wte":
        return Workload(name, gpt2_small_params(), "adamw", ADAMW_HP, 200, "student_t", 1e-4,
                        rho_bits, zero_rows=(("wte", 0.9),))
    if name == "stress_64m":
        return Workload(name, flat_params(1 << 26, "stress"), "adamw", ADAMW_HP, 20, "stress",
                        1e-3, rho_bits)
    raise KeyError(name)


WORKLOADS = ("flat_1m", "flat_128m", "flat_256m", "gpt2_small", "gpt2_small_sparse_wte", "resnet50", "llama31_8b", "llama31_8b_lion",
             "stress_64m")

# ---------------------------------------------------------------------------
# Seeded generators (host, numpy)
# ---------------------------------------------------------------------------

WEIGHT_SEED = 0          # seed of the initial weights
GRAD_SEED_BASE = 1000    # gradients of step t use seed GRAD_SEED_BASE + t


def _rng(seed: int, tensor_index: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[seed, tensor_index]))


def init_weight(spec: ParamSpec, tensor_index: int, seed: int = WEIGHT_SEED) -> np.ndarray:
    """Initial FP32 weights of one tensor (host)."""
    n = spec.numel
    rng = _rng(seed, tensor_index)
    if spec.init == "ones":
        return np.ones(n, np.float32)
    if spec.init == "zeros":
        return np.zeros(n, np.float32)
    if spec.init == "normal":
        return (rng.standard_normal(n, dtype=np.float32) * np.float32(spec.std)).astype(np.float32)
    if spec.init == "kaiming":
        fan_in = int(np.prod(spec.shape[1:]))
        std = math.sqrt(2.0) / math.sqrt(fan_in)
        return (rng.standard_normal(n, dtype=np.float32) * np.float32(std)).astype(np.float32)
    if spec.init == "stress":
        return stress_weights(n, rng)
    raise KeyError(spec.init)


def stress_weights(n: int, rng: np.random.Generator) -> np.ndarray:
    """|theta| log-uniform over [1e-8, 1e2] with random sign; 0.1 % exact +-0 and
    0.1 % values whose BF16 rounding is subnormal (|theta| < 2^-126)."""
    mag = np.exp(rng.uniform(math.log(1e-8), math.log(1e2), n)).astype(np.float32)
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0).astype(np.float32)
    x = (mag * sign).astype(np.float32)
    k = max(1, n // 1000)
    idx = rng.choice(n, size=2 * k, replace=False)
    x[idx[:k]] = np.where(rng.random(k) < 0.5, np.float32(0.0), np.float32(-0.0))
    sub = (rng.uniform(2.0 ** -133, 2.0 ** -126, k) * np.where(rng.random(k) < 0.5, -1, 1))
    x[idx[k:]] = sub.astype(np.float32)
    return x


def grad_fp32(kind: str, scale: float, n: int, tensor_index: int, step: int) -> np.ndarray:
    """FP32 gradient of one tensor at step ``step`` (host), before BF16 rounding."""
    rng = _rng(GRAD_SEED_BASE + step, tensor_index)
    if kind == "normal":
        return (rng.standard_normal(n, dtype=np.float32) * np.float32(scale)).astype(np.float32)
    if kind == "student_t":
        return (rng.standard_t(3.0, n) * scale).astype(np.float32)
    if kind == "stress":
        g = rng.standard_normal(n, dtype=np.float32) * np.float32(scale)
        u = rng.random(n)
        g = np.where(u < 0.01, g * np.float32(1e3), g)          # 1 % outliers x1e3
        g = np.where((u >= 0.01) & (u < 0.011), np.float32(0.0), g)  # 0.1 % exact zeros
        return g.astype(np.float32)
    raise KeyError(kind)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP32 -> BF16 bit patterns (round to nearest even, via torch's CPU cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def grad_bf16(kind: str, scale: float, n: int, tensor_index: int, step: int) -> np.ndarray:
    return to_bf16_bits(grad_fp32(kind, scale, n, tensor_index, step))


# ---------------------------------------------------------------------------
# Seeded generators (device, torch) for workloads too large to build on the host
# ---------------------------------------------------------------------------


def _torch_gen(device, seed: int, tensor_index: int):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tensor_index) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def init_weight_device(spec: ParamSpec, tensor_index: int, device, seed: int = WEIGHT_SEED):
    """Initial FP32 weights drawn on the device (same distributions as the host version,
    a different random stream)."""
    import torch
    n = spec.numel
    if spec.init == "ones":
        return torch.ones(n, dtype=torch.float32, device=device)
    if spec.init == "zeros":
        return torch.zeros(n, dtype=torch.float32, device=device)
    g = _torch_gen(device, seed, tensor_index)
    if spec.init == "normal":
        return torch.randn(n, generator=g, device=device, dtype=torch.float32).mul_(spec.std)
    if spec.init == "kaiming":
        fan_in = int(np.prod(spec.shape[1:]))
        std = math.sqrt(2.0) / math.sqrt(fan_in)
        return torch.randn(n, generator=g, device=device, dtype=torch.float32).mul_(std)
    if spec.init == "stress":
        u = torch.rand(n, generator=g, device=device, dtype=torch.float64)
        mag = torch.exp(u * (math.log(1e2) - math.log(1e-8)) + math.log(1e-8))
        sgn = torch.where(torch.rand(n, generator=g, device=device) < 0.5, -1.0, 1.0)
        x = (mag * sgn).to(torch.float32)
        sel = torch.rand(n, generator=g, device=device)
        x = torch.where(sel < 0.001, torch.zeros_like(x) * sgn.to(torch.float32), x)
        sub = (torch.rand(n, generator=g, device=device, dtype=torch.float64)
               * (2.0 ** -126 - 2.0 ** -133) + 2.0 ** -133) * sgn
        x = torch.where((sel >= 0.001) & (sel < 0.002), sub.to(torch.float32), x)
        return x
    raise KeyError(spec.init)


def grad_bf16_device(kind: str, scale: float, n: int, tensor_index: int, step: int, device):
    """BF16 gradient of one tensor drawn on the device."""
    import torch
    return grad_fp32_device(kind, scale, n, tensor_index, step, device).to(torch.bfloat16)


def grad_fp32_device(kind: str, scale: float, n: int, tensor_index: int, step: int, device):
    """FP32 gradient of one tensor drawn on the device (the BF16 one before rounding)."""
    import torch
    g = _torch_gen(device, GRAD_SEED_BASE + step, tensor_index)
    if kind == "normal":
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32).mul_(scale)
    elif kind == "student_t":
        # Student-t(3) = N(0,1) / sqrt(chi2_3 / 3), chi2_3 as a sum of three squared normals.
        z = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        c = torch.randn(3, n, generator=g, device=device, dtype=torch.float32).square_().sum(0)
        x = (z / torch.sqrt(c / 3.0)).mul_(scale)
    elif kind == "stress":
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32).mul_(scale)
        u = torch.rand(n, generator=g, device=device)
        x = torch.where(u < 0.01, x * 1e3, x)
        x = torch.where((u >= 0.01) & (u < 0.011), torch.zeros_like(x), x)
    else:
        raise KeyError(kind)
    return x


# ---------------------------------------------------------------------------
# Gradients of a workload's tensor (with its all-zero rows)
# ---------------------------------------------------------------------------

ZERO_ROW_SEED = 7


def zero_row_mask(w: Workload, tensor_index: int):
    """Boolean mask over the first dimension of tensor ``tensor_index``: the rows
    whose gradient is zero at every step, or None."""
    spec = w.params[tensor_index]
    frac = dict(w.zero_rows).get(spec.name)
    if not frac:
        return None
    return _rng(ZERO_ROW_SEED, tensor_index).random(spec.shape[0]) < frac


def workload_grad_fp32(w: Workload, tensor_index: int, step: int) -> np.ndarray:
    spec = w.params[tensor_index]
    g = grad_fp32(w.grad, w.grad_scale, spec.numel, tensor_index, step)
    mask = zero_row_mask(w, tensor_index)
    if mask is not None:
        g.reshape(spec.shape[0], -1)[mask] = 0.0
    return g


def workload_grad_bf16(w: Workload, tensor_index: int, step: int) -> np.ndarray:
    return to_bf16_bits(workload_grad_fp32(w, tensor_index, step))


def workload_grad_device(w: Workload, tensor_index: int, step: int, device, fp32: bool = False):
    """The tensor's gradient drawn on the device (BF16, or FP32 with fp32=True)."""
    import torch
    spec = w.params[tensor_index]
    g = grad_fp32_device(w.grad, w.grad_scale, spec.numel, tensor_index, step, device)
    mask = zero_row_mask(w, tensor_index)
    if mask is not None:
        g.view(spec.shape[0], -1)[torch.from_numpy(mask).to(g.device)] = 0.0
    return g if fp32 else g.to(torch.bfloat16)
