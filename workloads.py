"""Seeded synthetic inputs for the fused AdamW step: shapes and value distributions.

This module holds no part of the optimizer's arithmetic. Tests, the smoke check and
bench.py draw inputs from it, and the same arrays are then handed to both the CUDA
library and the CPU oracle, so neither side needs a bit-identical random generator.

Workloads (all synthetic: shape stand-ins only, no trained weights, no dataset):
  flat_1m        one fp32 tensor of 1,048,576 params ~N(0, 0.02^2); grads ~N(0, 1e-2^2)
  flat_16m       one fp32 tensor of 16,777,216 params; grads ~N(0, 1e-3^2)
  vit_base       ViT-Base-shaped list, 148 tensors, 86,564,352 params; grads ~N(0, 1e-2^2)
  flat_1g_heavy  one tensor of 2^30 params; grads 1e-3 * Student-t(3) with 1% outliers x100
  gpt_1p3b       GPT-style list, 292 tensors, 1,315,819,520 params; bf16 grads ~N(0, 1e-3^2)
Parameters are N(0, 0.02^2) except LayerNorm weights (1) and biases (0), as at init.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

DEFAULT_SEED = 1234


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    init: str = "normal"  # "normal" | "ones" | "zeros"

    @property
    def numel(self) -> int:
        n = 1
        for d in self.shape:
            n *= d
        return n


def vit_base_specs() -> list[TensorSpec]:
    """ViT-Base/16 parameter list as the workload lists it: patch embed 768x3x16x16,
    cls 1x768, pos 197x768, 12 blocks of {qkv 768x2304+b, proj 768x768+b,
    fc1 768x3072+b, fc2 3072x768+b, two LayerNorms w/b of 768}, head 768x1000."""
    d = 768
    specs = [TensorSpec("patch_embed.weight", (d, 3, 16, 16)),
             TensorSpec("cls_token", (1, d)),
             TensorSpec("pos_embed", (197, d))]
    for i in range(12):
        b = f"blocks.{i}."
        specs += [TensorSpec(b + "norm1.weight", (d,), "ones"), TensorSpec(b + "norm1.bias", (d,), "zeros"),
                  TensorSpec(b + "attn.qkv.weight", (d, 3 * d)), TensorSpec(b + "attn.qkv.bias", (3 * d,), "zeros"),
                  TensorSpec(b + "attn.proj.weight", (d, d)), TensorSpec(b + "attn.proj.bias", (d,), "zeros"),
                  TensorSpec(b + "norm2.weight", (d,), "ones"), TensorSpec(b + "norm2.bias", (d,), "zeros"),
                  TensorSpec(b + "mlp.fc1.weight", (d, 4 * d)), TensorSpec(b + "mlp.fc1.bias", (4 * d,), "zeros"),
                  TensorSpec(b + "mlp.fc2.weight", (4 * d, d)), TensorSpec(b + "mlp.fc2.bias", (d,), "zeros")]
    specs.append(TensorSpec("head.weight", (d, 1000)))
    return specs


def gpt_1p3b_specs() -> list[TensorSpec]:
    """GPT-style 1.3B list: tied token embedding 50304x2048, learned positions 2048x2048,
    24 layers of {LN w/b, qkv 2048x6144+b, proj 2048x2048+b, LN w/b, fc1 2048x8192+b,
    fc2 8192x2048+b}, final LN w/b."""
    d, f, vocab, ctx = 2048, 8192, 50304, 2048
    specs = [TensorSpec("wte", (vocab, d)), TensorSpec("wpe", (ctx, d))]
    for i in range(24):
        b = f"h.{i}."
        specs += [TensorSpec(b + "ln_1.weight", (d,), "ones"), TensorSpec(b + "ln_1.bias", (d,), "zeros"),
                  TensorSpec(b + "attn.c_attn.weight", (d, 3 * d)), TensorSpec(b + "attn.c_attn.bias", (3 * d,), "zeros"),
                  TensorSpec(b + "attn.c_proj.weight", (d, d)), TensorSpec(b + "attn.c_proj.bias", (d,), "zeros"),
                  TensorSpec(b + "ln_2.weight", (d,), "ones"), TensorSpec(b + "ln_2.bias", (d,), "zeros"),
                  TensorSpec(b + "mlp.c_fc.weight", (d, f)), TensorSpec(b + "mlp.c_fc.bias", (f,), "zeros"),
                  TensorSpec(b + "mlp.c_proj.weight", (f, d)), TensorSpec(b + "mlp.c_proj.bias", (d,), "zeros")]
    specs += [TensorSpec("ln_f.weight", (d,), "ones"), TensorSpec("ln_f.bias", (d,), "zeros")]
    return specs


@dataclass(frozen=True)
class Workload:
    name: str
    specs: tuple
    mode: str                 # headline moment mode: "fp32" | "bf16m" | "q8"
    grad_std: float
    grad_dtype: str = "f32"   # "f32" | "bf16"
    grad_kind: str = "normal" # "normal" | "student_t_outliers"
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    steps: int = 10
    stochastic_rounding: bool = False
    percentile: float = 100.0
    seed: int = 42            # stochastic-rounding key
    description: str = field(default="", compare=False)

    @property
    def numel(self) -> int:
        return sum(s.numel for s in self.specs)

    @property
    def sizes(self) -> list[int]:
        return [s.numel for s in self.specs]


WORKLOADS = {
    "flat_1m": Workload("flat_1m", (TensorSpec("w", (1 << 20,)),), "bf16m", 1e-2, weight_decay=0.01, steps=10,
                        description="AdamW, one fp32 tensor of 1,048,576 params, bf16 moments, 10 steps"),
    "flat_16m": Workload("flat_16m", (TensorSpec("w", (1 << 24,)),), "q8", 1e-3, steps=20,
                         description="8-bit block-wise AdamW, one fp32 tensor of 16,777,216 params, "
                                     "block 2048, round to nearest, 20 steps"),
    "vit_base": Workload("vit_base", tuple(vit_base_specs()), "bf16m", 1e-2, weight_decay=0.01, steps=50,
                         description="ViT-Base-shaped list, 148 tensors, 86,564,352 params, bf16 moments, 50 steps"),
    "flat_1g_heavy": Workload("flat_1g_heavy", (TensorSpec("w", (1 << 30,)),), "q8", 1e-3,
                              grad_kind="student_t_outliers", weight_decay=0.1, steps=10,
                              stochastic_rounding=True, percentile=99.9,
                              description="8-bit AdamW with Philox stochastic rounding and 99.9th-percentile "
                                          "block scaling on a flat 2^30-param tensor, 10 steps"),
    "gpt_1p3b": Workload("gpt_1p3b", tuple(gpt_1p3b_specs()), "q8", 1e-3, grad_dtype="bf16",
                         weight_decay=0.01, steps=20,
                         description="GPT-style 1.3B list, 292 tensors, bf16 grads, fp32/bf16/8-bit moments, 20 steps"),
}


# ------------------------------------------------------------------ numpy (small, for tests)
def init_params_np(specs, seed: int = DEFAULT_SEED) -> list[np.ndarray]:
    rng = np.random.default_rng(seed)
    out = []
    for s in specs:
        if s.init == "ones":
            out.append(np.ones(s.numel, np.float32))
        elif s.init == "zeros":
            out.append(np.zeros(s.numel, np.float32))
        else:
            out.append((rng.standard_normal(s.numel) * 0.02).astype(np.float32))
    return out


def grads_np(sizes, step: int, std: float, seed: int = DEFAULT_SEED, kind: str = "normal") -> list[np.ndarray]:
    """Fresh fp32 grads for 1-based ``step`` from seed ``seed + step``."""
    rng = np.random.default_rng(seed + step)
    out = []
    for n in sizes:
        if kind == "normal":
            g = rng.standard_normal(n) * std
        elif kind == "student_t_outliers":
            z = rng.standard_normal(n)
            chi2 = rng.chisquare(3, n)
            g = std * z / np.sqrt(chi2 / 3.0)
            g = np.where(rng.random(n) < 0.01, g * 100.0, g)
        else:
            raise ValueError(kind)
        out.append(g.astype(np.float32))
    return out


def to_bf16_bits_truncate(x: np.ndarray) -> np.ndarray:
    """Input generator for bf16 grads: keeps the top 16 bits of each fp32 draw. Any bf16
    bit pattern is a valid grad; this only produces one with a realistic spread."""
    return (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def random_moments_np(n: int, seed: int, m_std: float = 1e-3, v_scale: float = 1e-6):
    """A plausible mid-training fp32 moment pair (m signed, v >= 0)."""
    rng = np.random.default_rng(seed)
    m = (rng.standard_normal(n) * m_std).astype(np.float32)
    v = (rng.exponential(1.0, n) * v_scale).astype(np.float32)
    return m, v


# ------------------------------------------------------------------ torch (device, for the bench)
def flat_views(sizes, dtype, device=None, pin: bool = False):
    """Tensors of `sizes` elements laid out back to back in one buffer (as a flat-parameter
    optimizer keeps them), each start rounded up to 16 bytes. Returns (buffer, views)."""
    import torch
    esz = torch.empty((), dtype=dtype).element_size()
    align = max(1, 16 // esz)
    offs, cur = [], 0
    for n in sizes:
        offs.append(cur)
        cur += -(-n // align) * align
    if pin:
        buf = torch.empty(max(cur, 1), dtype=dtype, pin_memory=True)
    else:
        buf = torch.empty(max(cur, 1), dtype=dtype, device=device)
    return buf, [buf[o:o + n] for o, n in zip(offs, sizes)]


def init_params_torch(specs, device, seed: int = DEFAULT_SEED, flat: bool = False):
    """Parameters on `device`; with `flat`, views of one buffer (see flat_views)."""
    import torch
    if flat:
        _, views = flat_views([s.numel for s in specs], torch.float32, device)
        for v, t in zip(views, init_params_torch(specs, device, seed)):
            v.copy_(t)
        return views
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = []
    for s in specs:
        if s.init == "ones":
            out.append(torch.ones(s.numel, dtype=torch.float32, device=device))
        elif s.init == "zeros":
            out.append(torch.zeros(s.numel, dtype=torch.float32, device=device))
        else:
            t = torch.empty(s.numel, dtype=torch.float32, device=device)
            t.normal_(0.0, 0.02, generator=gen)
            out.append(t)
    return out


def grads_torch(sizes, step: int, std: float, device, seed: int = DEFAULT_SEED, kind: str = "normal",
                dtype: str = "f32", out=None):
    """Fresh grads for 1-based ``step`` from seed ``seed + step`` (written into ``out`` if given)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + step)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    res = []
    for i, n in enumerate(sizes):
        g = torch.empty(n, dtype=torch.float32, device=device)
        g.normal_(0.0, 1.0, generator=gen)
        if kind == "student_t_outliers":
            chi = torch.empty(n, 3, dtype=torch.float32, device=device).normal_(generator=gen).square_().sum(1)
            g.div_(torch.sqrt(chi / 3.0))
            mask = torch.rand(n, device=device, generator=gen) < 0.01
            g.mul_(std)
            g[mask] *= 100.0
        else:
            g.mul_(std)
        if out is not None:
            out[i].copy_(g.to(tdt))
            res.append(out[i])
        else:
            res.append(g.to(tdt))
    return res
