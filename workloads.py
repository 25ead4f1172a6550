"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds shapes, value distributions and seeds only -- none of the method's
arithmetic.  The shapes are those of the source pages' model (hidden size 7168, MoE
expert width 2048, top-8 routing over 256 experts, decode batches of at most 256 tokens
per expert; page 4, third paragraph); the distributions stand in for real activations,
weights and gradients, which need a trained model and data.

Weights use the PyTorch Linear layout ``W_lin [out_features, in_features]`` so that
``Y = X W_lin^T``; the Fprop B operand is then ``W_lin`` itself (K-major).
"""
from __future__ import annotations

import math

import torch

HIDDEN = 7168
EXPERT_WIDTH = 2048
N_EXPERTS = 256
TOP_K = 8


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=torch.device(device)).manual_seed(seed)


def normal(shape, std, g, device, dtype=torch.bfloat16):
    """N(0, std^2) draws rounded to ``dtype``; 3-D shapes are drawn one matrix at a time
    to bound the float32 temporary."""
    if len(shape) == 3:
        out = torch.empty(shape, dtype=dtype, device=device)
        for i in range(shape[0]):
            out[i] = (torch.randn(shape[1:], generator=g, device=device, dtype=torch.float32) * std).to(dtype)
        return out
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(dtype)


def with_outlier_columns(x: torch.Tensor, frac: float, factor: float, g) -> torch.Tensor:
    """Scale a fraction of the columns (channels) by ``factor``: activation outliers."""
    cols = x.shape[1]
    k = max(1, int(round(frac * cols)))
    idx = torch.randperm(cols, generator=g, device=g.device)[:k].to(x.device)
    x = x.clone()
    x[:, idx] = (x[:, idx].float() * factor).to(x.dtype)
    return x


def student_t3(shape, scale, g, device, dtype=torch.bfloat16):
    """Student-t with 3 degrees of freedom: Z / sqrt(V / 3), V a chi-square(3) draw."""
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    v = (torch.randn((3,) + tuple(shape), generator=g, device=device, dtype=torch.float32) ** 2).sum(0)
    return (z / torch.sqrt(v / 3.0) * scale).to(dtype)


# ------------------------------------------------------------------ configurations

def tiny_fprop(device="cpu"):
    """A 256x512 ~ N(0,1) with 1% of columns x50; W_lin 256x512 ~ N(0, 0.02).  Seed 0."""
    g = _gen(0, device)
    a = with_outlier_columns(normal((256, 512), 1.0, g, device), 0.01, 50.0, g)
    w = normal((256, 512), 0.02, g, device)
    return {"A": a, "W": w}


def dense_fprop(device="cuda", m=4096, k=HIDDEN, n=18432):
    """A m x k ~ N(0,1) with 0.1% outlier channels x100; W_lin n x k ~ N(0, 0.02).  Seed 1."""
    g = _gen(1, device)
    a = with_outlier_columns(normal((m, k), 1.0, g, device), 0.001, 100.0, g)
    w = normal((n, k), 0.02, g, device)
    return {"A": a, "W": w}


def backward_pair(device="cuda", t=8192, k=HIDDEN, n=EXPERT_WIDTH):
    """dY t x n = 1e-3 * Student-t(3); X t x k ~ N(0,1); W_lin n x k ~ N(0, 0.02).  Seed 2."""
    g = _gen(2, device)
    dy = student_t3((t, n), 1e-3, g, device)
    x = normal((t, k), 1.0, g, device)
    w = normal((n, k), 0.02, g, device)
    return {"dY": dy, "X": x, "W": w}


def zipf_routing_counts(tokens=16384, experts=N_EXPERTS, top_k=TOP_K, alpha=1.1, device="cpu", seed=3):
    """Per-expert token counts of top-k routing by softmax over N(0,1) logits plus a
    Zipf(alpha) expert bias ln p_e, p_e proportional to (e+1)^-alpha.  (Top-k of the
    softmax equals top-k of the logits.)"""
    g = _gen(seed, device)
    logits = torch.randn((tokens, experts), generator=g, device=device, dtype=torch.float32)
    bias = -alpha * torch.log(torch.arange(1, experts + 1, device=device, dtype=torch.float32))
    bias = bias - torch.logsumexp(bias, 0)
    top = torch.topk(logits + bias, top_k, dim=1).indices
    return torch.bincount(top.reshape(-1), minlength=experts).to(torch.int64)


def offsets_from_counts(counts: torch.Tensor) -> torch.Tensor:
    off = torch.zeros(counts.numel() + 1, dtype=torch.int64, device=counts.device)
    off[1:] = torch.cumsum(counts, 0)
    return off


def moe_prefill(device="cuda", tokens=16384, hidden=HIDDEN, width=EXPERT_WIDTH, experts=N_EXPERTS,
                with_weights=True):
    """MoE prefill: routed rows grouped by expert (dispatch itself is not modelled).

    up:   X_up [sum M, hidden] ~ N(0,1),  W_up [E, 2*width, hidden] ~ N(0, 0.02)  (gate+up)
    down: X_dn [sum M, width]  ~ N(0,1),  W_dn [E, hidden, width]   ~ N(0, 0.02)
    Seed 3."""
    counts = zipf_routing_counts(tokens, experts, device="cpu")
    off = offsets_from_counts(counts)
    rows = int(off[-1])
    g = _gen(3, device)
    out = {"counts": counts, "offsets": off, "X_up": normal((rows, hidden), 1.0, g, device),
           "X_dn": normal((rows, width), 1.0, g, device)}
    if with_weights:
        out["W_up"] = normal((experts, 2 * width, hidden), 0.02, g, device)
        out["W_dn"] = normal((experts, hidden, width), 0.02, g, device)
    return out


def moe_decode_counts(experts=N_EXPERTS, max_tokens=256, seed=4):
    g = _gen(seed, "cpu")
    return torch.randint(1, max_tokens + 1, (experts,), generator=g, dtype=torch.int64)


def moe_decode(device="cuda", hidden=HIDDEN, width=EXPERT_WIDTH, experts=N_EXPERTS, max_tokens=256,
               with_weights=True):
    """MoE decode: 1..256 tokens per expert (uniform), BF16 activations, same projections
    as the prefill case.  Seed 4."""
    counts = moe_decode_counts(experts, max_tokens)
    off = offsets_from_counts(counts)
    rows = int(off[-1])
    g = _gen(4, device)
    out = {"counts": counts, "offsets": off, "X_up": normal((rows, hidden), 1.0, g, device),
           "X_dn": normal((rows, width), 1.0, g, device)}
    if with_weights:
        out["W_up"] = normal((experts, 2 * width, hidden), 0.02, g, device)
        out["W_dn"] = normal((experts, hidden, width), 0.02, g, device)
    return out


def bf16_bits(t: torch.Tensor):
    """BF16 tensor -> numpy uint16 array of its bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("math", "torch")]
