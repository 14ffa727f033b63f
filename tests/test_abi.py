"""The C ABI library without a GPU: it builds, loads, exports every entry point
that include/bpkv.h declares, and rejects invalid arguments on the host before
enqueueing anything (none of these calls reaches the GPU)."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def L():
    from bit_plane_kv_encode_gb300 import build as B
    from bit_plane_kv_encode_gb300 import _binding
    B.build()
    return _binding.load()


def test_exports_every_header_symbol(L):
    from bit_plane_kv_encode_gb300 import header_symbols
    names = header_symbols()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert L.bpkv_version() == 2


def test_binding_names_match_header():
    import bit_plane_kv_encode_gb300 as pk
    for n in pk.header_symbols():
        assert hasattr(pk, n), f"binding lacks {n}"


def _cache(**kw):
    from bit_plane_kv_encode_gb300 import bpkv_cache
    fake = 1 << 20  # aligned non-null placeholder addresses: never dereferenced on these paths
    d = dict(n_seq=1, n_kv_heads=8, group=4, head_dim=128, cap_tokens=4096, n_max=0, residency=0, reserved=0,
             planes=fake, scales=fake, k_rows=fake, v_rows=fake, seq_len=fake)
    d.update(kw)
    return bpkv_cache(**d)


def test_workspace_size_rules(L):
    from bit_plane_kv_encode_gb300 import WS_ATTEND, WS_SCAN_TOPK, WS_STEP
    c = _cache()
    ws = L.bpkv_workspace_size(ctypes.byref(c), 512, WS_SCAN_TOPK)
    # status word + N H G cap float32 scores
    assert ws >= 256 + 1 * 8 * 4 * 4096 * 4
    assert L.bpkv_workspace_size(ctypes.byref(c), 512, WS_STEP) >= ws
    assert L.bpkv_workspace_size(ctypes.byref(c), 512, WS_ATTEND) > 256
    for bad in [dict(head_dim=64), dict(group=9), dict(cap_tokens=1000), dict(n_max=5000), dict(planes=0),
                dict(k_rows=(1 << 20) + 2), dict(residency=2)]:
        assert L.bpkv_workspace_size(ctypes.byref(_cache(**bad)), 512, WS_STEP) == 0, bad
    assert L.bpkv_workspace_size(ctypes.byref(c), 0, WS_STEP) == 0


def test_invalid_arguments_rejected_on_host(L):
    EINVAL, ENOWS, EUNSUP = -1, -2, -4
    fake = ctypes.c_void_p(1 << 20)
    c = _cache()
    assert L.bpkv_encode_append(None, fake, fake, 1, None) == EINVAL
    assert L.bpkv_encode_append(ctypes.byref(c), fake, fake, 0, None) == EINVAL
    assert L.bpkv_encode_append(ctypes.byref(c), fake, fake, 4097, None) == EINVAL
    assert L.bpkv_encode_append(ctypes.byref(c), ctypes.c_void_p((1 << 20) + 8), fake, 1, None) == EINVAL
    assert L.bpkv_encode_append(ctypes.byref(_cache(head_dim=96)), fake, fake, 1, None) == EUNSUP
    assert L.bpkv_alloc_depths(ctypes.byref(c), fake, None, fake, fake, None) == EINVAL
    assert L.bpkv_fixed_depths(ctypes.byref(c), fake, 32, 5, fake, None) == EINVAL
    assert L.bpkv_scan(ctypes.byref(_cache(n_max=100)), fake, fake, fake, 50, None) == EINVAL
    # k must hold the fixed tokens
    assert L.bpkv_topk(ctypes.byref(c), fake, 4096, 30, 4, 32, fake, fake, 1 << 20, None) == EINVAL
    assert L.bpkv_topk(ctypes.byref(c), fake, 4096, 64, 4, 32, fake, None, 0, None) == ENOWS
    assert L.bpkv_scan_topk(ctypes.byref(c), fake, fake, 64, 4, 32, fake, fake, 100, None) == ENOWS
    assert L.bpkv_union(ctypes.byref(c), fake, 8192, fake, fake, fake, None) == EINVAL  # G k > 16384
    assert L.bpkv_sparse_attend(ctypes.byref(c), fake, fake, fake, fake, 2048, fake, fake, 10, None) == ENOWS
    assert L.bpkv_dense_attend(ctypes.byref(c), fake, fake, fake, 10, None) == ENOWS
    assert L.bpkv_decode_step(None, 1, None, fake, 0, None) == EINVAL
    assert L.bpkv_status_string(-1) == b"invalid argument"
    # the bounded-wait self-test: workspace and limits checked on the host
    assert L.bpkv_selftest_wait(None, 2, 100, None) == ENOWS
    assert L.bpkv_selftest_wait(ctypes.c_void_p((1 << 20) + 16), 2, 100, None) == ENOWS
    assert L.bpkv_selftest_wait(fake, 0, 100, None) == EINVAL
    assert L.bpkv_selftest_wait(fake, 2, 0, None) == EINVAL
    assert L.bpkv_selftest_wait(fake, 2, (1 << 21) + 1, None) == EINVAL
    # the step's reserved flags must be 0
    from bit_plane_kv_encode_gb300 import bpkv_step_args
    a = bpkv_step_args(fake.value, fake.value, fake.value, fake.value, fake.value, 0, 0, 0, 512, 4, 32, fake.value,
                       None, None, None, 1, None)
    arr = (type(c) * 1)(c)
    assert L.bpkv_decode_step(arr, 1, ctypes.byref(a), fake, 1 << 30, None) == EINVAL
