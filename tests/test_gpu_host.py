"""Host-resident cache (Fathom page: KV cache and index in host memory, the
scan's bytes crossing the interconnect): planes, scales and rows in pinned
host memory, read in place by the same kernels over the host link."""
import numpy as np
import pytest
import torch

from gpu_helpers import bits16, bits64, build_cache, check_selection_map, check_unit, decode_one_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    import __graft_entry__
    __graft_entry__.build()
    import bit_plane_kv_encode_gb300 as m
    return m


def _decode(pk, cache, inp, cfg, flags=0):
    N, H, n, D = inp.k.shape
    G = cfg.group
    dev = torch.device("cuda")
    ws = cache.workspace(cfg.k, pk.WS_STEP)
    out = torch.zeros((1, N, H, G, D), device=dev)
    depths = torch.zeros((1, N, H, D), dtype=torch.uint8, device=dev)
    idx = torch.zeros((1, N, H, G, cfg.k), dtype=torch.int32, device=dev)
    q = inp.q.to(dev)[None].contiguous()
    s2 = inp.sigma2.to(dev)[None].contiguous()
    bq = (4 * inp.budgets).to(torch.int32).to(dev)
    kn = inp.k[:, :, n - 1].to(dev)[None].contiguous()
    vn = inp.v[:, :, n - 1].to(dev)[None].contiguous()
    a = pk.bpkv_step_args(kn.data_ptr(), vn.data_ptr(), q.data_ptr(), s2.data_ptr(), bq.data_ptr(), 0, 0, 0,
                          cfg.k, cfg.n_sink, cfg.n_recent, out.data_ptr(), depths.data_ptr(), idx.data_ptr(),
                          None, flags)
    arr = pk.cache_array([cache])
    pk.bpkv_clear_status(ws)
    pk.bpkv_decode_step(arr, 1, a, ws, ws.numel())
    pk.sync_n_max([cache], arr)
    torch.cuda.synchronize()
    assert pk.bpkv_read_status(ws) == 0
    return depths[0], idx[0], out[0]


def test_host_encode_bitexact(pk, orc):
    g = torch.Generator().manual_seed(31)
    N, H, n = 1, 2, 5000
    k = (torch.randn((N, H, n, 128), generator=g) * 3).to(torch.bfloat16).cuda()
    v = torch.randn((N, H, n, 128), generator=g).to(torch.bfloat16).cuda()
    c = build_cache(k, v, 4, residency="host", chunks=[1000, 1, 63, 64, 2000])
    torch.cuda.synchronize()
    assert c.planes.device.type == "cpu" and c.planes.is_pinned()
    nb = (n + 63) // 64
    for h in range(H):
        sc, pl = orc.encode(bits16(k[0, h]), c.c.cap_tokens // 64)
        assert np.array_equal(bits64(c.planes[0, h])[:, :, :nb], pl[:, :, :nb])
        assert np.array_equal(bits16(c.scales[0, h])[:, :nb], sc[:, :nb])
    assert torch.equal(c.k_rows[0, :, :n].cuda(), k[0])


def test_host_decode_equals_hbm(pk):
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS["host_1m"]
    inp = gen_layer(cfg, 0, device="cuda", n_tokens=65536)
    N, H, n, D = inp.k.shape
    dev_cache = build_cache(inp.k, inp.v, cfg.group, cap=((n + 511) // 512) * 512, n_prefill=n - 1)
    host_cache = pk.Cache(N, H, cfg.group, dev_cache.c.cap_tokens, residency="host")
    host_cache.copy_from(dev_cache)
    torch.cuda.synchronize()
    r_dev = _decode(pk, dev_cache, inp, cfg)
    r_host = _decode(pk, host_cache, inp, cfg)
    for a, b in zip(r_dev, r_host):
        assert torch.equal(a, b)
    nb = (n + 63) // 64
    assert torch.equal(dev_cache.planes[..., :nb].cpu(), host_cache.planes[..., :nb])


@pytest.mark.slow
def test_host_1m_layer_sampled(pk, orc):
    """One layer of the million-token host-resident workload at full size."""
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS["host_1m"]
    inp = gen_layer(cfg, 1, device="cuda")
    N, H, n, D = inp.k.shape
    dev_cache = build_cache(inp.k, inp.v, cfg.group, cap=cfg.cap_tokens, n_prefill=n - 1)
    host_cache = pk.Cache(N, H, cfg.group, cfg.cap_tokens, residency="host")
    host_cache.copy_from(dev_cache)
    torch.cuda.synchronize()
    del dev_cache
    torch.cuda.empty_cache()
    d, idx, out = _decode(pk, host_cache, inp, cfg)
    inp.k, inp.v = inp.k.cpu(), inp.v.cpu()
    for h in (0, 5):
        check_unit(orc, cfg, inp, host_cache, d, idx, out, 0, h, what=f"host1m h{h}")


def test_row_cache_identical_and_hits(pk):
    """The device row cache of recently selected rows (host-resident caches):
    over steps whose queries drift, outputs equal those of the same cache
    without it bit for bit, the first step reads every row over the link and
    later steps find most rows in the row cache."""
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS["host_1m"]
    n0, steps = 65536 - 8, 6
    inp = gen_layer(cfg, 2, device="cuda", n_tokens=n0 + steps)
    N, H, n_all, D = inp.k.shape
    G = cfg.group
    cap = (n_all + 1023) // 1024 * 1024
    dev_cache = build_cache(inp.k, inp.v, G, cap=cap, n_prefill=n0)
    plain = pk.Cache(N, H, G, cap, residency="host")
    cached = pk.Cache(N, H, G, cap, residency="host", rc_slots=4096)
    plain.copy_from(dev_cache)
    cached.copy_from(dev_cache)
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(5)
    drift = torch.randn(inp.q.shape, generator=g)
    dev = torch.device("cuda")
    outs = {}
    stats = []
    for name, cache in (("plain", plain), ("cached", cached)):
        ws = cache.workspace(cfg.k, pk.WS_STEP)
        arr = pk.cache_array([cache])
        outs[name] = []
        for t in range(steps):
            q = (inp.q + 0.05 * t * drift).to(dev)[None].contiguous()
            s2 = inp.sigma2.to(dev)[None].contiguous()
            bq = (4 * inp.budgets).to(torch.int32).to(dev)
            kn = inp.k[:, :, n0 + t][None].contiguous()
            vn = inp.v[:, :, n0 + t][None].contiguous()
            out = torch.zeros((1, N, H, G, D), device=dev)
            a = pk.bpkv_step_args(kn.data_ptr(), vn.data_ptr(), q.data_ptr(), s2.data_ptr(), bq.data_ptr(), 0, 0, 0,
                                  cfg.k, cfg.n_sink, cfg.n_recent, out.data_ptr(), None, None, None, 0)
            pk.bpkv_clear_status(ws)
            pk.bpkv_decode_step(arr, 1, a, ws, ws.numel())
            torch.cuda.synchronize()
            assert pk.bpkv_read_status(ws) == 0
            outs[name].append(out.clone())
            if name == "cached":
                stats.append(pk.bpkv_row_cache_stats(arr[0], cfg.k, ws))
        pk.sync_n_max([cache], arr)
    for t in range(steps):
        assert torch.equal(outs["plain"][t], outs["cached"][t]), f"step {t}"
    assert (stats[0][..., 0] == 0).all() and (stats[0][..., 1] > 0).all()  # first step: all misses
    later = np.stack(stats[1:])
    assert later[..., 0].sum() > 0.5 * later.sum(), later.sum(axis=(1, 2))


def test_host_selection_map_matches_lists(pk):
    """A decode step over caches in pinned host memory (the scan's host form
    and the row-cache attention): the selection map the attention reads holds
    exactly the middle tokens of the step's index lists on every row."""
    import dataclasses
    from workload import CONFIGS, gen_layer
    cfg = dataclasses.replace(CONFIGS["multi_session"], n_seq=2, n_tokens=70001, n_sink=4, n_recent=32, k=336)
    inp = gen_layer(cfg, 0, device="cuda")
    keep = {}
    cache, d, idx, out = decode_one_layer(inp, cfg, keep=keep, residency="host")
    assert check_selection_map(pk, cfg, cache, idx, keep["ws"], cfg.n_tokens)
