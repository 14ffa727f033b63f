"""GB300-native query-dependent prefix reads of a bit-plane K cache.

The compute path is libbpkv (CUDA kernels for sm_103a behind the C ABI in
``include/bpkv.h``).  This package is its thin Python binding: the functions
named ``bpkv_*`` marshal torch tensors to the C entry points of the same name;
``Cache`` holds one layer's cache buffers as torch tensors (torch is used only
to own device or pinned host memory and streams).
"""
from __future__ import annotations

import ctypes

from ._binding import (  # noqa: F401
    BpkvError, bpkv_alloc_depths, bpkv_cache, bpkv_calibrate_channels, bpkv_clear_status, bpkv_decode_step,
    bpkv_dense_attend, bpkv_encode_append, bpkv_fixed_depths, bpkv_read_status, bpkv_rotate, bpkv_row_cache_stats, bpkv_scan, bpkv_scan_topk, bpkv_scan_topk_noalloc, bpkv_selection_map, bpkv_selftest_wait, bpkv_sparse_attend, bpkv_sparse_attend_vdepth,
    bpkv_status_string, bpkv_step_args, bpkv_topk, bpkv_union, bpkv_version, bpkv_workspace_size, header_symbols, load)

HEAD_DIM = 128
WS_SCAN_TOPK, WS_ATTEND, WS_DENSE, WS_STEP = 1, 2, 4, 8
DEPTH_WATERFILL, DEPTH_FIXED, DEPTH_DENSE, DEPTH_GIVEN = 0, 1, 2, 3
DEV_OVERFLOW, DEV_SELECT, DEV_TIMEOUT = 1, 2, 4
STEP_VDEPTH = 1


class Cache:
    """One layer's bit-plane K cache and bf16 K/V rows for N sequences x H KV heads.

    residency "hbm": all buffers in device memory.  "host": planes, scales and
    rows in pinned host memory, read by the kernels in place over the host link.
    """

    def __init__(self, n_seq: int, n_kv_heads: int, group: int, cap_tokens: int, device="cuda",
                 residency: str = "hbm", values: bool = False, rc_slots: int = 0):
        import torch
        if cap_tokens % 512:
            raise ValueError("cap_tokens must be a multiple of 512")
        D, nb = HEAD_DIM, cap_tokens // 64
        self.device = torch.device(device)
        host = residency == "host"

        def buf(shape, dtype):
            if host:
                # pinned host memory from a 256-byte boundary: the kernels' reads
                # of it are not cached, so a row segment that starts inside a
                # 32-byte sector moves one more sector over the link
                n = dtype.itemsize
                for e in shape:
                    n *= e
                raw = torch.empty(n + 256, dtype=torch.uint8, pin_memory=True)
                off = (-raw.data_ptr()) % 256
                return raw[off:off + n].view(dtype).view(shape)
            return torch.empty(shape, dtype=dtype, device=self.device)

        self.planes = buf((n_seq, n_kv_heads, D, 4, nb), torch.int64)
        self.scales = buf((n_seq, n_kv_heads, D, nb), torch.int16)
        self.k_rows = buf((n_seq, n_kv_heads, cap_tokens, D), torch.bfloat16)
        self.v_rows = buf((n_seq, n_kv_heads, cap_tokens, D), torch.bfloat16)
        self.seq_len = torch.zeros(n_seq, dtype=torch.int64, device=self.device)
        self.basis = None
        # the value rows' own code (value-side read depth), when asked for
        self.vplanes = buf((n_seq, n_kv_heads, cap_tokens, 4, D // 64), torch.int64) if values else None
        self.vscales = buf((n_seq, n_kv_heads, cap_tokens), torch.int16) if values else None
        self.c = bpkv_cache(n_seq, n_kv_heads, group, D, cap_tokens, 0, 1 if host else 0, 0,
                            self.planes.data_ptr(), self.scales.data_ptr(), self.k_rows.data_ptr(),
                            self.v_rows.data_ptr(), self.seq_len.data_ptr(), None,
                            self.vplanes.data_ptr() if values else None, self.vscales.data_ptr() if values else None)
        # device row cache of recently selected rows (host-resident caches)
        self.rc_rows = self.rc_tok = None
        if rc_slots:
            self.rc_rows = torch.empty((n_seq, n_kv_heads, rc_slots, 2, D), dtype=torch.bfloat16, device=self.device)
            self.rc_tok = torch.full((n_seq, n_kv_heads, rc_slots), -1, dtype=torch.int32, device=self.device)
            self.c.rc_rows = self.rc_rows.data_ptr()
            self.c.rc_tok = self.rc_tok.data_ptr()
            self.c.rc_slots = rc_slots

    def set_basis(self, basis):
        """Code the keys in an orthogonal basis R, float [H][D][D] on the device
        (None: the raw channels); set it before the first append."""
        self.basis = None if basis is None else basis.contiguous()
        self.c.basis = None if basis is None else self.basis.data_ptr()

    @property
    def n_max(self) -> int:
        return int(self.c.n_max)

    def append(self, k_new, v_new, stream=None):
        """Append k_new/v_new [N][H][t][D] bf16 (device) to every sequence."""
        bpkv_encode_append(self.c, k_new, v_new, k_new.shape[2], stream)

    def copy_from(self, other: "Cache"):
        """Take over another cache's contents (same shapes), e.g. a host-resident
        copy of a cache built in device memory; copies run on the current stream."""
        for name in ("planes", "scales", "k_rows", "v_rows", "seq_len", "vplanes", "vscales"):
            if getattr(self, name) is not None and getattr(other, name) is not None:
                getattr(self, name).copy_(getattr(other, name), non_blocking=True)
        self.c.n_max = other.c.n_max

    def workspace(self, k: int, what: int):
        import torch
        n = bpkv_workspace_size(self.c, k, what)
        if n == 0:
            raise BpkvError("bpkv_workspace_size", -1)
        return torch.empty(n, dtype=torch.uint8, device=self.device)


def cache_array(caches):
    """ctypes array of the bpkv_cache structs of several layers (for bpkv_decode_step)."""
    arr = (bpkv_cache * len(caches))(*[c.c for c in caches])
    return arr


def sync_n_max(caches, arr):
    """Copy n_max back from a cache array after bpkv_decode_step raised it."""
    for c, s in zip(caches, arr):
        c.c.n_max = s.n_max


__all__ = [n for n in dir() if n.startswith("bpkv_")] + ["Cache", "cache_array", "sync_n_max", "BpkvError"]
_ = ctypes
