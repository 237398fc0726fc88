"""Seeded synthetic inputs for the cast workloads.

Only random draws live here: nothing of the cast, the scale rule or the MX
rule.  Both the CUDA path and the CPU oracle consume these tensors (the
oracle receives the same bytes, copied to the host).

Workloads (the shapes and distributions the pages' settings call for;
N(0, s) means standard deviation s):
  current_4096   4096 fp32 ~ N(0, 1), seed 0                     (E4M3, window 0)
  spike_seq      16 steps of bf16 [4096, 4096] ~ N(0, 1), seed 1000+s; at
                 step 9 a random 0.1% of the entries x8 (before the bf16
                 rounding)                                       (E4M3)
  grad_group     64 bf16 tensors, rows/cols uniform on {1024..8192}, random
                 signs, magnitudes log-uniform on [1e-8, 1e2] times a per-tensor
                 log-uniform factor in [1e-4, 1e1]; fresh draws per step
                                                                 (E5M2, window 16)
  mx_tanh        bf16 [16384, 8192] = tanh(N(0, 2)), seed 4000   (MX E4M3)
  decoder_1b1    every weight / activation / activation-gradient tensor of
                 a 24-layer decoder (hidden 2048, FFN 8192, batch 4 x seq 4096):
                 weights ~ N(0, 0.02) -> E4M3; activations ~ N(0, 1) with
                 0.01% outliers x20 -> E4M3; gradients ~ N(0, 1) * 1e-3 -> E5M2
"""
from __future__ import annotations

import math

import torch

E4M3, E5M2 = 0, 1


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


# ---- current_4096 ----------------------------------------------------------

def current_4096(device="cpu") -> torch.Tensor:
    return torch.randn(4096, generator=_gen("cpu", 0), dtype=torch.float32).to(device)


# ---- spike_seq -------------------------------------------------------------

SPIKE_STEPS, SPIKE_STEP, SPIKE_SHAPE = 16, 9, (4096, 4096)


def spike_step(s: int, device="cpu", shape=SPIKE_SHAPE) -> torch.Tensor:
    g = _gen("cpu", 1000 + s)
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if s == SPIKE_STEP:
        n = x.numel()
        idx = torch.randperm(n, generator=g)[: n // 1000]
        x.view(-1)[idx] *= 8.0
    return x.to(torch.bfloat16).to(device)


# ---- grad_group ------------------------------------------------------------

GRAD_SIDES = (1024, 2048, 4096, 8192)


def grad_group_shapes(count: int = 64, seed: int = 3000, sides=GRAD_SIDES):
    g = _gen("cpu", seed)
    idx = torch.randint(0, len(sides), (count, 2), generator=g)
    lf = torch.empty(count).uniform_(math.log(1e-4), math.log(1e1), generator=g)
    return [(sides[int(a)], sides[int(b)]) for a, b in idx.tolist()], torch.exp(lf).tolist()


def grad_group_step(s: int, device="cuda", count: int = 64, sides=GRAD_SIDES):
    shapes, factors = grad_group_shapes(count, sides=sides)
    g = _gen(device, 3000 + s)
    out = []
    for (r, c), f in zip(shapes, factors):
        mag = torch.empty(r, c, device=device, dtype=torch.float32).uniform_(
            math.log(1e-8), math.log(1e2), generator=g).exp_()
        sign = torch.randint(0, 2, (r, c), device=device, generator=g, dtype=torch.int8)
        mag.mul_(sign.to(torch.float32).mul_(2).sub_(1)).mul_(f)
        out.append(mag.to(torch.bfloat16))
        del mag, sign
    return out


# ---- mx_tanh ---------------------------------------------------------------

MX_SHAPE = (16384, 8192)


def mx_tanh(device="cuda", sigma: float = 2.0, shape=MX_SHAPE, seed: int = 4000) -> torch.Tensor:
    x = torch.randn(*shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    return torch.tanh(x.mul_(sigma)).to(torch.bfloat16)


# ---- decoder_1b1 -----------------------------------------------------------

LAYERS, HIDDEN, FFN, TOKENS = 24, 2048, 8192, 4 * 4096

# (name, shape as (rows, cols) with T = tokens, format, kind)
def decoder_tensor_specs(layers=LAYERS, hidden=HIDDEN, ffn=FFN, tokens=TOKENS):
    H, F, T = hidden, ffn, tokens
    per_layer = [
        ("Wq", (H, H), E4M3, "w"), ("Wk", (H, H), E4M3, "w"), ("Wv", (H, H), E4M3, "w"),
        ("Wo", (H, H), E4M3, "w"), ("Wup", (H, F), E4M3, "w"), ("Wdown", (F, H), E4M3, "w"),
        ("X_ln1", (T, H), E4M3, "a"), ("X_attn", (T, H), E4M3, "a"),
        ("X_ln2", (T, H), E4M3, "a"), ("X_act", (T, F), E4M3, "a"),
        ("dY_q", (T, H), E5M2, "g"), ("dY_k", (T, H), E5M2, "g"), ("dY_v", (T, H), E5M2, "g"),
        ("dY_o", (T, H), E5M2, "g"), ("dY_up", (T, F), E5M2, "g"), ("dY_down", (T, H), E5M2, "g"),
    ]
    return [(f"L{l}.{name}", shape, fmt, kind, l, k)
            for l in range(layers) for k, (name, shape, fmt, kind) in enumerate(per_layer)]


def decoder_tensor(spec, step: int, device="cuda", out: torch.Tensor | None = None) -> torch.Tensor:
    name, (r, c), fmt, kind, layer, k = spec
    g = _gen(device, 5_000_000 + 10_000 * step + 100 * layer + k)
    x = torch.randn(r, c, generator=g, device=device, dtype=torch.float32)
    if kind == "w":
        x.mul_(0.02)
    elif kind == "a":
        n = x.numel()
        idx = torch.randint(0, n, (max(1, n // 10000),), generator=g, device=device)
        x.view(-1)[idx] *= 20.0
    else:
        x.mul_(1e-3)
    if out is None:
        return x.to(torch.bfloat16)
    out.copy_(x)
    return out


def decoder_step(step: int, device="cuda", **sizes):
    specs = decoder_tensor_specs(**sizes)
    return specs, [decoder_tensor(s, step, device) for s in specs]
