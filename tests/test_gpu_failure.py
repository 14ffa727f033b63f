"""Failure detection without a GPU fault: the library's bounded in-kernel wait
(the one the selection's CTAs use to wait for one another) is made to run out
by a self-test kernel whose barrier expects an arrival that never comes.  The
wait must give up within its short limit, record BPKV_DEV_TIMEOUT in the
status word and leave the context usable."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    import __graft_entry__
    __graft_entry__.build()
    import bit_plane_kv_encode_gb300 as m
    return m


def test_bounded_wait_times_out_and_reports(pk):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    # a barrier every arrival reaches completes without an error
    pk.bpkv_selftest_wait(ws, 1, 1 << 14)
    assert pk.bpkv_read_status(ws) == 0
    # one of two arrivals: the wait gives up after 2^14 rounds of ~100 ns
    t0 = time.perf_counter()
    pk.bpkv_selftest_wait(ws, 2, 1 << 14)
    status = pk.bpkv_read_status(ws)
    dt = time.perf_counter() - t0
    assert status == pk.DEV_TIMEOUT
    assert dt < 0.5, f"the wait took {dt:.3f} s"
    pk.bpkv_clear_status(ws)
    assert pk.bpkv_read_status(ws) == 0


def test_context_usable_after_timeout(pk):
    """After a wait gave up, the next kernels run and give correct results."""
    from gpu_helpers import build_cache
    ws0 = torch.zeros(256, dtype=torch.uint8, device="cuda")
    pk.bpkv_selftest_wait(ws0, 3, 1 << 12)
    assert pk.bpkv_read_status(ws0) == pk.DEV_TIMEOUT
    g = torch.Generator().manual_seed(3)
    n, H, G = 5000, 2, 4
    k = torch.randn((1, H, n, 128), generator=g).to(torch.bfloat16).cuda()
    v = torch.randn((1, H, n, 128), generator=g).to(torch.bfloat16).cuda()
    cache = build_cache(k, v, G)
    q = torch.randn((1, H, G, 128), generator=g).cuda()
    depths = torch.full((1, H, 128), 4, dtype=torch.uint8, device="cuda")
    ws = cache.workspace(64, pk.WS_SCAN_TOPK)
    idx = torch.zeros((1, H, G, 64), dtype=torch.int32, device="cuda")
    pk.bpkv_clear_status(ws)
    pk.bpkv_scan_topk(cache.c, q, depths, 64, 4, 32, idx, ws, ws.numel())
    assert pk.bpkv_read_status(ws) == 0
    # the 36 fixed tokens are always in every list
    fixed = set(range(4)) | set(range(n - 32, n))
    for h in range(H):
        for gg in range(G):
            assert fixed <= set(idx[0, h, gg].tolist())
