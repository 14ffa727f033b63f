"""Byte counts of the scan path (cost model of the Fathom page, section 3.1, Eq. 1).

A decode step reads about W + N L H (b n / 8 + k_U R) bytes: W the weights read
once per step, N sequences of n tokens, L layers, H KV heads, b scan bits per
token per (layer, KV head), k_U distinct winner rows per KV head after the
union of its G query heads' selections, R the bytes of one full K+V row.
Bits per token of a depth vector: every read plane costs 1 bit per token and
every channel read at depth >= 1 costs its fp16 scale, 16 bits per 64-token
block, i.e. 1/4 bit per token (section 1: "4-bit coordinates plus block
scales", 136 bits for 32 channels at depth 4).
"""
from __future__ import annotations


def depth_bits(depths) -> float:
    """Scan bits per token of one depth vector (iterable of ints in 0..4)."""
    ds = [int(t) for t in depths]
    return sum(ds) + 0.25 * sum(1 for t in ds if t > 0)


def depth_quarter_bits(depths) -> int:
    ds = [int(t) for t in depths]
    return 4 * sum(ds) + sum(1 for t in ds if t > 0)


def row_bytes(head_dim: int = 128) -> int:
    """R: one K row plus one V row in bf16."""
    return 2 * 2 * head_dim


def scan_bytes(bits_per_token: float, n: int) -> float:
    """b n / 8 for one (sequence, layer, KV head)."""
    return bits_per_token * n / 8.0


def dense_kv_bytes(n_layers: int, n_kv_heads: int, head_dim: int, n: int, n_seq: int = 1) -> int:
    """Full bf16 K and V read once per step (dense attention)."""
    return n_seq * n_layers * n_kv_heads * n * row_bytes(head_dim)


def step_bytes(n_seq: int, n_layers: int, n_kv_heads: int, bits_per_token: float, n: int,
               k_union: float, head_dim: int = 128, weights: float = 0.0) -> float:
    """Eq. 1: W + N L H (b n / 8 + k_U R)."""
    per_unit = scan_bytes(bits_per_token, n) + k_union * row_bytes(head_dim)
    return weights + n_seq * n_layers * n_kv_heads * per_unit


def union_bound(group: int, k: int, n_fixed: int = 36) -> int:
    """Largest possible union: the fixed tokens once plus G disjoint top sets."""
    return n_fixed + group * (k - n_fixed)
