"""The five synthetic workload shapes of the bit-plane KV scan.

Shapes follow the Qwen3-8B example used throughout the Fathom page
("Fathom: per-query read depth for sparse decoding over an offloaded KV
cache", section 1): 36 layers, 8 KV heads of 128 channels, 4 query heads
per KV head, k = 512 selected keys per query head.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class WorkloadConfig:
    name: str
    n_seq: int            # N: sequences decoded together
    n_layers: int         # L
    n_kv_heads: int       # H
    group: int            # G: query heads per KV head
    head_dim: int         # D
    n_tokens: int         # n: tokens per sequence after the decode step's append
    budgets: tuple        # bits/token per (layer, KV head); one entry per pass
    k: int                # per-query-head selection size, sinks and recent included
    seed: int
    residency: str = "hbm"          # "hbm" or "host"
    n_needles: int = 0              # planted high-|q.k| keys per (seq, KV head)
    outlier_channels: int = 0       # channels per (seq, KV head) whose sigma is scaled
    outlier_scale: float = 1.0
    per_seq_budgets: tuple = ()     # if set, budget of each sequence drawn from this set
    fixed_baselines: tuple = field(default=())  # ("sparq", r, t) / ("uniform", t) depth rules
    n_sink: int = 4
    n_recent: int = 32

    @property
    def cap_tokens(self) -> int:
        # capacity rounded up to a whole number of 512-token groups
        return ((self.n_tokens + 511) // 512) * 512


CONFIGS = {
    "tiny": WorkloadConfig(
        name="tiny", n_seq=1, n_layers=1, n_kv_heads=1, group=4, head_dim=128,
        n_tokens=4096, budgets=(68,), k=64, seed=0),
    "qwen3_8b_layer": WorkloadConfig(
        name="qwen3_8b_layer", n_seq=1, n_layers=1, n_kv_heads=8, group=4, head_dim=128,
        n_tokens=32768, budgets=(68, 92, 136), k=512, seed=1, n_needles=8),
    "full_step": WorkloadConfig(
        name="full_step", n_seq=4, n_layers=36, n_kv_heads=8, group=4, head_dim=128,
        n_tokens=131072, budgets=(32, 44, 56, 68, 80, 92, 104, 116, 128, 136), k=512, seed=2,
        fixed_baselines=(("sparq", 32, 4), ("uniform", 2))),
    "host_1m": WorkloadConfig(
        name="host_1m", n_seq=1, n_layers=8, n_kv_heads=8, group=4, head_dim=128,
        n_tokens=1048576, budgets=(68, 92, 136), k=512, seed=3, residency="host"),
    "multi_session": WorkloadConfig(
        name="multi_session", n_seq=32, n_layers=1, n_kv_heads=8, group=4, head_dim=128,
        n_tokens=65536, budgets=(82,), k=512, seed=4, outlier_channels=6, outlier_scale=8.0,
        per_seq_budgets=(32, 68, 92, 136)),
}
