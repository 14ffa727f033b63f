"""Seeded input generator shared by the tests, the smoke check and the bench.

Draw recipe (one layer at a time):
  * sigma_j = exp(0.75 * z), z ~ N(0, 1), one value per (seq, KV head, channel),
    drawn on the CPU in float64 and stored as float32.  With ``outlier_channels``
    set, that many channels per (seq, KV head) are chosen uniformly and their
    sigma is multiplied by ``outlier_scale``.
  * K[i, j] = bf16(z * sigma_j), z ~ N(0, 1) (float32 draw, round to nearest even).
  * V[i, j] = bf16(z), z ~ N(0, 1).
  * q[h, j] ~ N(0, 1) float32 per query head (CPU draw).
  * needles: ``n_needles`` distinct positions per (seq, KV head), uniform in
    [n_sink, n - n_recent); at each, K[i, j] = bf16(4 sigma_j sign(qbar_j)) where
    qbar is the mean of the G queries of that KV head (sign(0) = +1).
  * per-sequence budgets drawn uniformly from ``per_seq_budgets`` when given.

CPU draws (sigma, q, needles, budgets) use a CPU ``torch.Generator`` so they
are identical whatever device holds K and V.  K and V are drawn on the target
device from a generator seeded per layer.  The module does no quantisation,
scoring or selection: it only produces inputs.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from .configs import WorkloadConfig

_MASK64 = (1 << 64) - 1


def _mix(*parts: int) -> int:
    """SplitMix64-style combination of integers into a 63-bit seed."""
    z = 0x9E3779B97F4A7C15
    for p in parts:
        z = (z + (p & _MASK64) + 0x9E3779B97F4A7C15) & _MASK64
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        z ^= z >> 31
    return z & ((1 << 63) - 1)


def _cpu_gen(*parts: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(_mix(*parts))
    return g


def _dev_gen(device, *parts: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_mix(*parts))
    return g


@dataclass
class LayerInputs:
    k: torch.Tensor          # [N][H][n][D] bfloat16 on the target device
    v: torch.Tensor          # [N][H][n][D] bfloat16 on the target device
    q: torch.Tensor          # [N][H][G][D] float32 (CPU)
    sigma2: torch.Tensor     # [N][H][D] float32 (CPU)
    budgets: torch.Tensor    # [N] int32 bits/token (CPU)
    needles: Optional[torch.Tensor]  # [N][H][n_needles] int64 (CPU) or None


def unit_sigma(cfg: WorkloadConfig, layer: int) -> torch.Tensor:
    """sigma [N][H][D] float32 for one layer (CPU)."""
    g = _cpu_gen(cfg.seed, layer, 1)
    z = torch.randn((cfg.n_seq, cfg.n_kv_heads, cfg.head_dim), generator=g, dtype=torch.float64)
    sigma = torch.exp(0.75 * z)
    if cfg.outlier_channels > 0:
        for s in range(cfg.n_seq):
            for h in range(cfg.n_kv_heads):
                pick = torch.randperm(cfg.head_dim, generator=g)[: cfg.outlier_channels]
                sigma[s, h, pick] *= cfg.outlier_scale
    return sigma.to(torch.float32)


def gen_layer(cfg: WorkloadConfig, layer: int, device="cpu", n_tokens: Optional[int] = None,
              n_seq: Optional[int] = None) -> LayerInputs:
    """Inputs of one layer.  ``n_tokens``/``n_seq`` override the config's sizes
    (used to draw smaller cases with the same recipe)."""
    n = cfg.n_tokens if n_tokens is None else n_tokens
    N = cfg.n_seq if n_seq is None else n_seq
    H, G, D = cfg.n_kv_heads, cfg.group, cfg.head_dim
    sigma = unit_sigma(cfg, layer)[:N]
    gq = _cpu_gen(cfg.seed, layer, 2)
    q = torch.randn((N, H, G, D), generator=gq, dtype=torch.float32)

    gk = _dev_gen(device, cfg.seed, layer, 3)
    k32 = torch.randn((N, H, n, D), generator=gk, dtype=torch.float32, device=device)
    k32.mul_(sigma.to(device)[:, :, None, :])
    gv = _dev_gen(device, cfg.seed, layer, 4)
    v = torch.randn((N, H, n, D), generator=gv, dtype=torch.float32, device=device).to(torch.bfloat16)

    needles = None
    if cfg.n_needles > 0:
        gn = _cpu_gen(cfg.seed, layer, 5)
        lo, hi = cfg.n_sink, n - cfg.n_recent
        pos = torch.empty((N, H, cfg.n_needles), dtype=torch.int64)
        qbar = q.mean(dim=2)  # [N][H][D]
        sgn = torch.where(qbar >= 0, 1.0, -1.0).to(torch.float32)
        for s in range(N):
            for h in range(H):
                p = torch.randperm(hi - lo, generator=gn)[: cfg.n_needles] + lo
                pos[s, h] = torch.sort(p).values
                val = (4.0 * sigma[s, h] * sgn[s, h]).to(device)
                k32[s, h, pos[s, h].to(device), :] = val[None, :]
        needles = pos
    k = k32.to(torch.bfloat16)
    del k32

    if cfg.per_seq_budgets:
        gb = _cpu_gen(cfg.seed, layer, 6)
        choice = torch.randint(0, len(cfg.per_seq_budgets), (N,), generator=gb)
        budgets = torch.tensor([cfg.per_seq_budgets[c] for c in choice.tolist()], dtype=torch.int32)
    else:
        budgets = torch.full((N,), cfg.budgets[0], dtype=torch.int32)
    return LayerInputs(k=k, v=v, q=q, sigma2=(sigma * sigma), budgets=budgets, needles=needles)


def random_scores(n_rows: int, n: int, seed: int, tie_frac: float = 0.0) -> torch.Tensor:
    """float32 [n_rows][n] scores for selection tests; ``tie_frac`` of the
    entries are snapped to a coarse grid so that exact ties occur."""
    g = _cpu_gen(seed, 7)
    s = torch.randn((n_rows, n), generator=g, dtype=torch.float32)
    if tie_frac > 0:
        m = torch.rand((n_rows, n), generator=g) < tie_frac
        s = torch.where(m, torch.round(s * 4) / 4, s)
    return s
