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
    cache = build_cache(k, v, G)
    return cache, g


def test_noalloc_matches_workspace_call_twice(pk):
    n, H, K = 32768, 8, 512
    cache, g = _case(pk, n, H, seed=21)
    N, G = 1, 4
    ws = cache.workspace(K, pk.WS_SCAN_TOPK)
    for call in range(2):
        q = torch.randn((N, H, G, 128), generator=g).cuda()
        s2 = torch.exp(torch.randn((N, H, 128), generator=g)).cuda()
        budget = torch.tensor([4 * (68 + 24 * call)], dtype=torch.int32).cuda()
        depths = torch.zeros((N, H, 128), dtype=torch.uint8, device="cuda")
        pk.bpkv_alloc_depths(cache.c, q, s2, budget, depths)
        want = torch.full((N, H, G, K), -7, dtype=torch.int32, device="cuda")
        got = torch.full((N, H, G, K), -7, dtype=torch.int32, device="cuda")
        pk.bpkv_scan_topk(cache.c, q, depths, K, 4, 32, want, ws, ws.numel())
        pk.bpkv_scan_topk_noalloc(cache.c, q, depths, K, 4, 32, got)
        torch.cuda.synchronize()
        assert (want >= -1).all()
        assert torch.equal(got, want), f"call {call}: {int((got != want).sum())} indices differ"


def test_noalloc_refuses_oversized_request(pk):
    # rows (4 round_up(n, 64) + 40984) bytes with rows = N H G = 64: 64 x (262400 + 40984) > 16 MiB
    cache, g = _case(pk, 65600, 16, seed=22)
    q = torch.randn((1, 16, 4, 128), generator=g).cuda()
    depths = torch.full((1, 16, 128), 1, dtype=torch.uint8, device="cuda")
    idx = torch.zeros((1, 16, 4, 512), dtype=torch.int32, device="cuda")
    with pytest.raises(pk.BpkvError) as e:
        pk.bpkv_scan_topk_noalloc(cache.c, q, depths, 512, 4, 32, idx)
    assert e.value.status == -2
    assert np.all(idx.cpu().numpy() == 0)  # nothing was enqueued
