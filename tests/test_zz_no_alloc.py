"""bpkv_scan_topk_noalloc: the scan + top-k call for callers that cannot
allocate device memory (their own pool holds the GPU's memory, or they must
avoid the synchronisation that allocation can cause).  Its score scratch is a
fixed array inside the library instead of a caller workspace, so its results
must be exactly those of bpkv_scan_topk, call after call, and requests larger
than the array must be refused.  Kept in a file that pytest collects last."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    import __graft_entry__
    __graft_entry__.build()
    import bit_plane_kv_encode_gb300 as m
    return m


def _case(pk, n, H, seed):
    from gpu_helpers import build_cache
    g = torch.Generator(device="cpu").manual_seed(seed)
    N, G, D = 1, 4, 128
    sig = torch.exp(0.75 * torch.randn((N, H, 1, D), generator=g))
    k = (torch.randn((N, H, n, D), generator=g) * sig).to(torch.bfloat16).cuda()
    v = torch.randn((N, H, n, D), generator=g).to(torch.bfloat16).cuda()
    cache = build_cache(k, v, G, cap=max(512, (n + 511) // 512 * 512))
    return cache, g


def _compare(pk, cache, g, H, K, budgets):
    N, G = 1, 4
    ws = cache.workspace(K, pk.WS_SCAN_TOPK)
    pk.bpkv_clear_status(ws)
    for call, b in enumerate(budgets):
        q = torch.randn((N, H, G, 128), generator=g).cuda()
        s2 = torch.exp(torch.randn((N, H, 128), generator=g)).cuda()
        budget = torch.tensor([4 * b], dtype=torch.int32).cuda()
        depths = torch.zeros((N, H, 128), dtype=torch.uint8, device="cuda")
        pk.bpkv_alloc_depths(cache.c, q, s2, budget, depths)
        want = torch.full((N, H, G, K), -7, dtype=torch.int32, device="cuda")
        got = torch.full((N, H, G, K), -7, dtype=torch.int32, device="cuda")
        pk.bpkv_scan_topk(cache.c, q, depths, K, 4, 32, want, ws, ws.numel())
        pk.bpkv_scan_topk_noalloc(cache.c, q, depths, K, 4, 32, got)
        torch.cuda.synchronize()
        assert pk.bpkv_read_status(ws) == 0
        assert (want >= -1).all()
        assert torch.equal(got, want), f"call {call}: {int((got != want).sum())} indices differ"


# n = 32768: score rows as wide as the capacity; n = 70001: the array packs
# rows at round_up(n, 64) = 70016 floats, narrower than the 70144-token
# capacity the workspace call uses; n = 131073 on one KV head: long rows (the
# selection's second histogram level); n = 0: nothing to scan, every list -1
@pytest.mark.parametrize("n,H", [(32768, 8), (70001, 8), (131073, 1), (0, 8)])
def test_noalloc_matches_workspace_call_twice(pk, n, H):
    cache, g = _case(pk, n, H, seed=21 + n % 97)
    _compare(pk, cache, g, H, 512, [68, 92])


def test_noalloc_repeated_calls(pk):
    # the same array reused by many calls in a row, with budgets and queries
    # changing between calls: every call must still match the workspace call
    cache, g = _case(pk, 70001, 8, seed=5)
    _compare(pk, cache, g, 8, 512, [68, 92, 136, 32, 92, 68, 136, 44, 92, 104])


def test_noalloc_refuses_oversized_request(pk):
    # 256 + rows (4 round_up(n, 64) + 40984) bytes with rows = N H G = 64: > 16 MiB
    cache, g = _case(pk, 65600, 16, seed=22)
    q = torch.randn((1, 16, 4, 128), generator=g).cuda()
    depths = torch.full((1, 16, 128), 1, dtype=torch.uint8, device="cuda")
    idx = torch.zeros((1, 16, 4, 512), dtype=torch.int32, device="cuda")
    with pytest.raises(pk.BpkvError) as e:
        pk.bpkv_scan_topk_noalloc(cache.c, q, depths, 512, 4, 32, idx)
    assert e.value.status == -2
    assert np.all(idx.cpu().numpy() == 0)  # nothing was enqueued
