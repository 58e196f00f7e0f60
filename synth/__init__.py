"""Seeded synthetic inputs shared by the oracle, the tests and the benchmark.

This module holds input synthesis only: random numbers, shapes and the
workload table.  None of the compression arithmetic lives here (no
quantizer, no least-squares coefficient, no residual, no attention).

Workloads stand in for the looped models the ResidualQuant pages evaluate
(Ouro-1.4B: 24 layers run 4 loops, 16 KV heads of width 128; Huginn-3.5B:
a 4-layer block run 32 loops, taken as 8 groups of 4, 55 KV heads of width
96).  Neither the weights nor the evaluation sets exist here, so the KV
cache is drawn from a generator with the property the explainer page
("ResidualQuant stores looped-Transformer KV caches as 2-bit residuals",
the paragraph on why residuals quantize well) describes: the loops of one
token are near-copies of each other, and the raw KV carries a few large
outlier channels that the residual does not.

Recipe (per (layer, group, batch row, head, token), K and V drawn
independently):
  base  ~ N(0, 1) per channel, channels 3 and 77 multiplied by 8;
  loop i of the group = alpha_i * base + 0.3 * N(0, 1), except that in the
  Ouro-shaped workloads the last loop (the anchor) is base itself.
  Ouro alphas (0.7, 0.85, 0.95) for the three earlier loops; Huginn alphas
  (0.7, 0.85, 0.95, 1.0) with noise on all four.
Queries and the current token's KV are drawn the same way (queries
~ N(0, 1)).  Everything is rounded to bfloat16, the dtype the model hands
to the cache.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "rotation", "group_alphas", "looped_kv", "looped_kv_slice", "queries",
    "to_bf16_f64", "looped_kv_torch", "queries_torch",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: model shape, batch, context and code layout."""
    name: str
    num_layers: int
    loops_per_group: int
    num_groups: int
    num_heads: int
    head_dim: int
    group_size: int
    batch: int
    context: int
    alphas: tuple
    anchor_is_base: bool  # True: the last loop equals the base vector
    outlier_channels: tuple = (3, 77)
    outlier_scale: float = 8.0
    noise: float = 0.3

    @property
    def calls_per_step(self) -> int:
        return self.num_layers * self.loops_per_group * self.num_groups

    @property
    def appends_per_step(self) -> int:
        return self.num_layers * self.num_groups


OURO_ALPHAS = (0.7, 0.85, 0.95)
HUGINN_ALPHAS = (0.7, 0.85, 0.95, 1.0)


def group_alphas(p: int) -> tuple:
    """Loop similarity to the base for groups of p loops: 0.7 rising evenly to 1.0."""
    return tuple(0.7 + 0.3 * i / (p - 1) for i in range(p)) if p > 1 else (1.0,)

WORKLOADS = {
    # one layer, 4 loops, batch 1, 2 heads, width 128, 256 tokens
    "toy": Workload("toy", 1, 4, 1, 2, 128, 32, 1, 256, OURO_ALPHAS, True),
    # Ouro-1.4B shape at 8k context, batch 4
    "ouro8k": Workload("ouro8k", 24, 4, 1, 16, 128, 32, 4, 8192, OURO_ALPHAS, True),
    # Ouro-1.4B shape at 16k context, batch 2 and batch 4
    "ouro16k_b2": Workload("ouro16k_b2", 24, 4, 1, 16, 128, 32, 2, 16384, OURO_ALPHAS, True),
    "ouro16k_b4": Workload("ouro16k_b4", 24, 4, 1, 16, 128, 32, 4, 16384, OURO_ALPHAS, True),
    # Huginn-3.5B shape: 4-layer block, 32 loops as 8 groups of 4, 55 heads of width 96
    "huginn": Workload("huginn", 4, 4, 8, 55, 96, 32, 2, 4096, HUGINN_ALPHAS, False),
    # the same 32 loops as 4 groups of 8 and as 2 groups of 16 loops per anchor (the
    # larger groups the arXiv summary mentions from the appendix)
    "huginn_g8": Workload("huginn_g8", 4, 8, 4, 55, 96, 32, 2, 4096, group_alphas(8), False),
    "huginn_g16": Workload("huginn_g16", 4, 16, 2, 55, 96, 32, 2, 4096, group_alphas(16), False),
}


def sweep_workload(batch: int, group_size: int = 32) -> Workload:
    """Batch-sweep point on the Ouro-1.4B shape at 8k context."""
    return Workload(f"ouro8k_b{batch}_g{group_size}", 24, 4, 1, 16, 128, group_size,
                    batch, 8192, OURO_ALPHAS, True)


def rotation(d: int, seed: int = 0) -> np.ndarray:
    """Seeded d x d orthogonal matrix: QR of a Gaussian, signs of diag(R) made positive.

    Stands in for the offline-calibrated rotation the pages describe (the
    ai4snews summary, closing paragraph: calibrated once, then fixed).
    Returns float64.
    """
    rng = np.random.default_rng(np.random.PCG64(seed))
    a = rng.standard_normal((d, d))
    q, r = np.linalg.qr(a)
    sgn = np.sign(np.diag(r))
    sgn[sgn == 0] = 1.0
    return q * sgn[None, :]


def _kv_f32(rng: np.random.Generator, w: Workload, batch: int, ntok: int) -> np.ndarray:
    """float32 [P, 2, B, H, n, d] for one (layer, group)."""
    P, H, d = w.loops_per_group, w.num_heads, w.head_dim
    shape = (2, batch, H, ntok, d)
    base = rng.standard_normal(shape, dtype=np.float32)
    for ch in w.outlier_channels:
        if ch < d:
            base[..., ch] *= np.float32(w.outlier_scale)
    out = np.empty((P,) + shape, dtype=np.float32)
    for i in range(P):
        if i == P - 1 and w.anchor_is_base:
            out[i] = base
        else:
            alpha = w.alphas[i]
            out[i] = np.float32(alpha) * base + np.float32(w.noise) * rng.standard_normal(shape, dtype=np.float32)
    return out


def looped_kv_slice(seed: int, w: Workload, ntok: int, layer: int, group: int, b: int, h: int):
    """KV of one (layer, group, batch row, head), drawn from its own stream (seeded by
    the tuple), so a single slice of a full-size cache can be regenerated alone.

    Returns (bf16 tensor [P, 2, ntok, d], float64 copy of the same values)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, layer, group, b, h]))
    one = dataclasses.replace(w, num_heads=1)
    t, f = to_bf16_f64(_kv_f32(rng, one, 1, ntok))
    return t[:, :, 0, 0], f[:, :, 0, 0]


def to_bf16_f64(x: np.ndarray):
    """Round float32 values to bfloat16 (torch CPU cast); return (torch bf16 tensor, float64 ndarray)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t, t.to(torch.float64).numpy()


def looped_kv(seed: int, w: Workload, batch: Optional[int] = None, ntok: Optional[int] = None):
    """KV for one (layer, group): (bf16 tensor [P,2,B,H,n,d], float64 copy of the same values)."""
    rng = np.random.default_rng(np.random.PCG64(seed))
    b = w.batch if batch is None else batch
    n = w.context if ntok is None else ntok
    return to_bf16_f64(_kv_f32(rng, w, b, n))


def queries(seed: int, batch: int, heads: int, d: int):
    """Decode queries ~ N(0,1): (bf16 tensor [B,H,d], float64 copy)."""
    rng = np.random.default_rng(np.random.PCG64(seed))
    return to_bf16_f64(rng.standard_normal((batch, heads, d), dtype=np.float32))


# ---- device-side generation for the full-size benchmark (same recipe, torch RNG) ----

def looped_kv_torch(gen, w: Workload, batch: int, ntok: int, device):
    """Same recipe on the device with a seeded torch.Generator; bf16 [P,2,B,H,n,d]."""
    import torch
    P, H, d = w.loops_per_group, w.num_heads, w.head_dim
    shape = (2, batch, H, ntok, d)
    base = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    for ch in w.outlier_channels:
        if ch < d:
            base[..., ch] *= w.outlier_scale
    out = torch.empty((P,) + shape, device=device, dtype=torch.bfloat16)
    for i in range(P):
        if i == P - 1 and w.anchor_is_base:
            out[i] = base.to(torch.bfloat16)
        else:
            noise = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
            out[i] = (w.alphas[i] * base + w.noise * noise).to(torch.bfloat16)
    return out


def queries_torch(gen, batch: int, heads: int, d: int, device):
    import torch
    return torch.randn((batch, heads, d), generator=gen, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def softmax_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
