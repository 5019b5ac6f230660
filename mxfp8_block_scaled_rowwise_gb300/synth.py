"""Seeded synthetic inputs for the MoE MXFP8 hot path.

This module only draws random numbers and routing decisions; it holds none of
the method's arithmetic (no quantization, no permutation, no GEMM), so both the
CUDA path and the CPU oracle can consume the very same bytes it produces.

Workload recipes (shapes after the Kimi-2.5 dimensions quoted on the kucoin.com
page "Cursor's MoK демонстрирует повышение производительности на 2,37x на NVIDIA
GB300 NVL72", section "02": hidden 7168, expert intermediate 2048):

* ``tiny``      T=512, K=256, E=4 experts, top-1 uniform routing, W [4, 512, 256].
* ``quant``     bf16 [16384, 7168]: z * exp(2 g_row) (log-normal row magnitudes)
                with 0.1 % of the entries multiplied by 1000.
* ``ffn``       T=16384, top-8 of E=32 (131072 routed rows), hidden 7168,
                W1 [32, 4096, 7168] (fused gate/up), W2 [32, 7168, 2048], down
                input h [131072, 2048]; router logits N(0, 1).
* ``ffn_bwd``   the ``ffn`` shapes plus dY_down [131072, 7168] and dH [131072, 4096]
                ~ N(0, 1e-2).
* ``skewed``    T=4096, top-8 of E=128, hidden 4096, intermediate 1536; expert
                popularity Zipf(1.2) over a seeded rank order, 4 seeded experts
                never chosen; routing = top-8 of log p + Gumbel noise.

All tensors are drawn in fp32 from a seeded ``torch.Generator`` and rounded to
bf16 (round to nearest even).  Routing ties go to the lower expert id.
"""
from __future__ import annotations

import math

import torch

SEEDS = {"tiny": 1001, "quant": 1002, "ffn": 1003, "ffn_bwd": 1004, "skewed": 1005}


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, gen: torch.Generator, std: float = 1.0, device="cpu") -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def lognormal_rows_bf16(rows: int, cols: int, gen: torch.Generator, sigma: float = 2.0,
                        outlier_frac: float = 1e-3, outlier_mult: float = 1e3,
                        device="cpu") -> torch.Tensor:
    """z_ij * exp(sigma * g_i) with z, g ~ N(0,1); a seeded 0.1 % of entries times 1000."""
    z = torch.randn(rows, cols, generator=gen, device=device, dtype=torch.float32)
    g = torch.randn(rows, 1, generator=gen, device=device, dtype=torch.float32)
    z.mul_(torch.exp(sigma * g))
    n_out = int(round(outlier_frac * rows * cols))
    if n_out > 0:
        idx = torch.randint(0, rows * cols, (n_out,), generator=gen, device=device)
        flat = z.view(-1)
        flat[idx] = flat[idx] * outlier_mult
    return z.to(torch.bfloat16)


def topk_ids(logits: torch.Tensor, k: int) -> torch.Tensor:
    """Router top-k (input generation only): largest logits, ties -> lower expert id."""
    order = torch.sort(logits, dim=1, descending=True, stable=True).indices
    return order[:, :k].to(torch.int32).contiguous()


def uniform_ids(T: int, E: int, k: int, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """top-k of uniform random logits (k distinct experts per token)."""
    logits = torch.rand(T, E, generator=gen, device=device)
    return topk_ids(logits, k)


def zipf_ids(T: int, E: int, k: int, gen: torch.Generator, s: float = 1.2, n_zero: int = 4,
             device="cpu") -> torch.Tensor:
    """Weighted sampling without replacement: top-k of log p_e + Gumbel(0,1).

    p_e ~ rank_e^-s over a seeded random rank order; n_zero seeded experts get p = 0."""
    ranks = torch.randperm(E, generator=gen, device="cpu").to(torch.float64) + 1.0
    logp = -s * torch.log(ranks)
    zero = torch.randperm(E, generator=gen, device="cpu")[:n_zero]
    logp[zero] = -math.inf
    u = torch.rand(T, E, generator=gen, device="cpu", dtype=torch.float64).clamp_(1e-300, 1.0)
    gumbel = -torch.log(-torch.log(u))
    ids = topk_ids((logp.unsqueeze(0) + gumbel).to(torch.float64), k)
    return ids.to(device)


def tiny(device="cpu"):
    g = generator(SEEDS["tiny"], device)
    T, K, E, N = 512, 256, 4, 512
    x = randn_bf16((T, K), g, device=device)
    w = randn_bf16((E, N, K), g, device=device)
    ids = uniform_ids(T, E, 1, g, device=device)
    return dict(x=x, w=w, ids=ids, T=T, K=K, E=E, N=N, k=1)


def quant(device="cpu", rows: int = 16384, cols: int = 7168):
    g = generator(SEEDS["quant"], device)
    return dict(x=lognormal_rows_bf16(rows, cols, g, device=device), rows=rows, cols=cols)


def ffn(device="cpu", T: int = 16384, E: int = 32, k: int = 8, hidden: int = 7168, inter: int = 2048,
        with_weights: bool = True):
    g = generator(SEEDS["ffn"], device)
    x = randn_bf16((T, hidden), g, device=device)
    logits = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    ids = topk_ids(logits, k)
    out = dict(x=x, ids=ids, T=T, E=E, k=k, hidden=hidden, inter=inter, R=T * k)
    if with_weights:
        out["w1"] = randn_bf16((E, 2 * inter, hidden), g, device=device)
        out["w2"] = randn_bf16((E, hidden, inter), g, device=device)
        out["h"] = randn_bf16((T * k, inter), g, device=device)
    return out


def ffn_bwd(device="cpu", R: int = 131072, hidden: int = 7168, inter: int = 2048):
    g = generator(SEEDS["ffn_bwd"], device)
    dy = randn_bf16((R, hidden), g, std=1e-2, device=device)
    dh = randn_bf16((R, 2 * inter), g, std=1e-2, device=device)
    return dict(dy=dy, dh=dh)


def skewed(device="cpu", T: int = 4096, E: int = 128, k: int = 8, hidden: int = 4096, inter: int = 1536,
           with_weights: bool = True):
    g = generator(SEEDS["skewed"], device)
    ids = zipf_ids(T, E, k, generator(SEEDS["skewed"] + 7), device=device)
    x = randn_bf16((T, hidden), g, device=device)
    out = dict(x=x, ids=ids, T=T, E=E, k=k, hidden=hidden, inter=inter, R=T * k)
    if with_weights:
        out["w1"] = randn_bf16((E, 2 * inter, hidden), g, device=device)
        out["w2"] = randn_bf16((E, hidden, inter), g, device=device)
        out["dy"] = randn_bf16((T * k, hidden), g, std=1e-2, device=device)
    return out


def bf16_bits(t: torch.Tensor):
    """The raw bf16 bit patterns of a CPU tensor as a numpy uint16 array."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
