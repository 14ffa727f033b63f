"""CUDA path vs CPU oracle, kernel by kernel, through the C ABI.

Bars: planes, scales, depths, indices and unions bit-exact; scores within
1e-5 max(|oracle|, sum_j |q_j khat_j|); top-k sets equal except keys within
1e-4 max|score| of the k-th score; attention within 2e-3 max-abs.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import (ATTN_ATOL, abs_score_scale, bits16, bits64, build_cache, check_scores,
                         check_topk_sets)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    import __graft_entry__
    __graft_entry__.build()
    import bit_plane_kv_encode_gb300 as m
    return m


def _rand_kv(N, H, n, seed, scale=None, dev="cuda"):
    g = torch.Generator(device="cpu").manual_seed(seed)
    D = 128
    sig = torch.exp(0.75 * torch.randn((N, H, 1, D), generator=g)) if scale is None else scale
    k = (torch.randn((N, H, n, D), generator=g) * sig).to(torch.bfloat16)
    v = torch.randn((N, H, n, D), generator=g).to(torch.bfloat16)
    return k.to(dev), v.to(dev)


# ------------------------------------------------------------------ encode

@pytest.mark.parametrize("n,chunks", [(4096, None), (64 * 3 + 17, [1] * 70 + [63, 1, 64, 65]),
                                      (1000, [500, 1, 1, 1, 200]), (64, [64]), (1, [1])])
def test_encode_bitexact(pk, orc, n, chunks):
    N, H = 2, 3
    k, v = _rand_kv(N, H, n, seed=n)
    k[0, 1, :, 5] = 0                                      # an all-zero channel
    k[1, 2, : min(n, 40), 7] = torch.tensor(3.0e38).to(torch.bfloat16)  # scale saturates
    c = build_cache(k, v, group=4, chunks=chunks)
    torch.cuda.synchronize()
    assert c.n_max == n and c.seq_len.tolist() == [n] * N
    nb_cap = c.c.cap_tokens // 64
    for s in range(N):
        for h in range(H):
            sc, pl = orc.encode(bits16(k[s, h]), nb_cap)
            nb = (n + 63) // 64
            assert np.array_equal(bits64(c.planes[s, h])[:, :, :nb], pl[:, :, :nb]), (s, h)
            assert np.array_equal(bits16(c.scales[s, h])[:, :nb], sc[:, :nb]), (s, h)
            assert torch.equal(c.k_rows[s, h, :n], k[s, h]) and torch.equal(c.v_rows[s, h, :n], v[s, h])


def test_encode_token_by_token_equals_bulk(pk):
    k, v = _rand_kv(1, 2, 300, seed=5)
    bulk = build_cache(k, v, 4)
    inc = build_cache(k, v, 4, chunks=[1] * 300)
    torch.cuda.synchronize()
    nb = (300 + 63) // 64
    assert torch.equal(bulk.planes[..., :nb], inc.planes[..., :nb])
    assert torch.equal(bulk.scales[..., :nb], inc.scales[..., :nb])


def test_encode_rejects_overflow(pk):
    k, v = _rand_kv(1, 1, 512, seed=6)
    c = build_cache(k, v, 4, cap=512)
    with pytest.raises(pk.BpkvError):
        c.append(k[:, :, :1].contiguous(), v[:, :, :1].contiguous())


# ------------------------------------------------------------------ depths

def _depth_inputs(N, H, G, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn((N, H, G, 128), generator=g)
    s2 = torch.exp(torch.randn((N, H, 128), generator=g) * 1.5)
    q[0, 0] = 1.0          # equal g everywhere: all ties
    s2[0, 0] = 1.0
    q[0, 1, :, 10:20] = 0  # worthless channels
    s2[1 % N, 1, 3] = 0
    q[0, 2, :, 64:] = q[0, 2, :, :64]  # pairwise ties
    s2[0, 2, 64:] = s2[0, 2, :64]
    return q, s2


@pytest.mark.parametrize("budget", [0, 1, 4, 5, 32, 44, 68, 92, 136, 200, 288, 544, 10000])
def test_alloc_depths_bitexact(pk, orc, budget):
    N, H, G = 3, 4, 4
    q, s2 = _depth_inputs(N, H, G, seed=budget)
    k, v = _rand_kv(N, H, 64, seed=1)
    c = build_cache(k, v, G)
    bq = torch.tensor([budget * 4, budget * 4 + 3, max(budget * 4 - 1, 0)], dtype=torch.int32)
    d = torch.zeros((N, H, 128), dtype=torch.uint8, device="cuda")
    pk.bpkv_alloc_depths(c.c, q.cuda(), s2.cuda(), bq.cuda(), d)
    got = d.cpu().numpy()
    for s in range(N):
        for h in range(H):
            want = orc.alloc_depths(q[s, h].numpy(), s2[s, h].numpy(), int(bq[s]))
            assert np.array_equal(got[s, h], want), (s, h, budget)


@pytest.mark.parametrize("r,t", [(32, 4), (16, 4), (128, 2), (0, 4), (200, 1), (7, 3)])
def test_fixed_depths_bitexact(pk, orc, r, t):
    N, H, G = 2, 3, 4
    q, _ = _depth_inputs(N, H, G, seed=r * 10 + t)
    k, v = _rand_kv(N, H, 64, seed=2)
    c = build_cache(k, v, G)
    d = torch.zeros((N, H, 128), dtype=torch.uint8, device="cuda")
    pk.bpkv_fixed_depths(c.c, q.cuda(), r, t, d)
    got = d.cpu().numpy()
    for s in range(N):
        for h in range(H):
            assert np.array_equal(got[s, h], orc.fixed_depths(q[s, h].numpy(), r, t)), (s, h)


# ------------------------------------------------------------------ scan

@pytest.mark.parametrize("n,G,depth_kind", [(4096, 4, "water68"), (5000 + 17, 4, "random"), (777, 8, "full"),
                                            (2048, 1, "thumb"), (130, 4, "water136"), (3, 2, "random"),
                                            (3000 + 5, 4, "above4")])
def test_scan_scores(pk, orc, n, G, depth_kind):
    N, H = 2, 2
    k, v = _rand_kv(N, H, n, seed=n + G)
    c = build_cache(k, v, G)
    g = torch.Generator(device="cpu").manual_seed(7)
    q = torch.randn((N, H, G, 128), generator=g)
    if depth_kind == "random":
        d = torch.randint(0, 5, (N, H, 128), generator=g, dtype=torch.uint8)
    elif depth_kind == "full":
        d = torch.full((N, H, 128), 4, dtype=torch.uint8)
    elif depth_kind == "thumb":
        d = torch.full((N, H, 128), 2, dtype=torch.uint8)
    elif depth_kind == "above4":
        # depth values above 4 read the whole 4-plane code (never the next channel's planes)
        d = torch.randint(0, 5, (N, H, 128), generator=g, dtype=torch.uint8)
        for val, lo in ((5, 0), (17, 40), (255, 80)):
            d[..., lo:lo + 12] = val
    else:
        b = int(depth_kind[5:])
        s2 = torch.exp(torch.randn((N, H, 128), generator=g))
        d = torch.stack([torch.stack([torch.from_numpy(orc.alloc_depths(q[s, h].numpy(), s2[s, h].numpy(), 4 * b))
                                      for h in range(H)]) for s in range(N)])
    scores = torch.full((N, H, G, c.c.cap_tokens), float("nan"), device="cuda")
    pk.bpkv_scan(c.c, q.cuda(), d.cuda(), scores, c.c.cap_tokens)
    got = scores.cpu().numpy()
    nb_cap = c.c.cap_tokens // 64
    for s in range(N):
        for h in range(H):
            kb = bits16(k[s, h])
            sc, pl = orc.encode(kb, nb_cap)
            ref = orc.scores(n, sc, pl, d[s, h].numpy(), q[s, h].numpy())
            scale = abs_score_scale(q[s, h].numpy(), kb, np.minimum(d[s, h].numpy(), 4))
            check_scores(got[s, h, :, :n], ref, scale, what=f"{depth_kind} s{s} h{h}")
            assert np.isnan(got[s, h, :, n:]).all()  # nothing written past seq_len


# ------------------------------------------------------------------ top-k / union

@pytest.mark.parametrize("n,k,ties", [(4096, 64, 0.0), (4096, 64, 0.5), (100, 64, 0.3), (64, 64, 0.0),
                                      (37, 36, 0.0), (1000, 36, 0.2), (20000, 512, 0.9), (5, 64, 0.0),
                                      (600, 512, 0.0), (3000, 1024, 0.7)])
def test_topk_exact_on_given_scores(pk, orc, n, k, ties):
    from workload.gen import random_scores
    N, H, G = 1, 2, 4
    kk, vv = _rand_kv(N, H, n, seed=3)
    c = build_cache(kk, vv, G)
    sc = random_scores(N * H * G, n, seed=n + k, tie_frac=ties).reshape(N, H, G, n)
    ld = c.c.cap_tokens
    buf = torch.zeros((N, H, G, ld), device="cuda")
    buf[..., :n] = sc.cuda()
    idx = torch.zeros((N, H, G, k), dtype=torch.int32, device="cuda")
    ws = c.workspace(k, pk.WS_SCAN_TOPK)
    pk.bpkv_clear_status(ws)
    pk.bpkv_topk(c.c, buf, ld, k, 4, 32, idx, ws, ws.numel())
    assert pk.bpkv_read_status(ws) == 0
    got = idx.cpu().numpy()
    for h in range(H):
        for g in range(G):
            want = orc.topk(sc[0, h, g].numpy().astype(np.float64), k)
            assert np.array_equal(got[0, h, g], want), (h, g)


def test_union_exact(pk, orc):
    N, H, G, k, n = 2, 3, 4, 64, 3000
    kk, vv = _rand_kv(N, H, n, seed=4)
    c = build_cache(kk, vv, G)
    g = torch.Generator(device="cpu").manual_seed(9)
    idx = torch.full((N, H, G, k), -1, dtype=torch.int32)
    for s in range(N):
        for h in range(H):
            for q in range(G):
                m = int(torch.randint(0, k + 1, (1,), generator=g))
                pool = 200 if (s + h) % 2 else n  # heavy overlap in some units
                idx[s, h, q, :m] = torch.sort(torch.randperm(pool, generator=g)[:m].to(torch.int32)).values
    uidx = torch.zeros((N, H, G * k), dtype=torch.int32, device="cuda")
    umask = torch.zeros((N, H, G * k), dtype=torch.uint8, device="cuda")
    ucnt = torch.zeros((N, H), dtype=torch.int32, device="cuda")
    pk.bpkv_union(c.c, idx.cuda(), k, uidx, umask, ucnt)
    for s in range(N):
        for h in range(H):
            wu, wm = orc.union(idx[s, h].numpy())
            u = int(ucnt[s, h])
            assert u == len(wu)
            assert np.array_equal(uidx[s, h, :u].cpu().numpy(), wu)
            assert np.array_equal(umask[s, h, :u].cpu().numpy(), wm)
            assert (uidx[s, h, u:] == -1).all()


# ------------------------------------------------------------------ attention

@pytest.mark.parametrize("n,k", [(4096, 64), (700, 512), (40, 64), (20000, 512)])
def test_sparse_attend(pk, orc, n, k):
    N, H, G = 2, 2, 4
    kk, vv = _rand_kv(N, H, n, seed=n, scale=2.0)
    c = build_cache(kk, vv, G)
    g = torch.Generator(device="cpu").manual_seed(11)
    q = torch.randn((N, H, G, 128), generator=g)
    idx = torch.zeros((N, H, G, k), dtype=torch.int32)
    refs = {}
    for s in range(N):
        for h in range(H):
            for qh in range(G):
                score = torch.randn(n, generator=g).numpy().astype(np.float64)
                idx[s, h, qh] = torch.from_numpy(orc.topk(score, k))
            refs[s, h] = orc.attend(q[s, h].numpy(), bits16(kk[s, h]), bits16(vv[s, h]), idx[s, h].numpy())
    uidx = torch.zeros((N, H, G * k), dtype=torch.int32, device="cuda")
    umask = torch.zeros((N, H, G * k), dtype=torch.uint8, device="cuda")
    ucnt = torch.zeros((N, H), dtype=torch.int32, device="cuda")
    pk.bpkv_union(c.c, idx.cuda(), k, uidx, umask, ucnt)
    out = torch.zeros((N, H, G, 128), device="cuda")
    ws = c.workspace(k, pk.WS_ATTEND)
    pk.bpkv_sparse_attend(c.c, q.cuda(), uidx, umask, ucnt, G * k, out, ws, ws.numel())
    got = out.cpu().numpy()
    for (s, h), r in refs.items():
        assert np.max(np.abs(got[s, h] - r)) <= ATTN_ATOL, (s, h, np.max(np.abs(got[s, h] - r)))


@pytest.mark.parametrize("n", [1, 100, 4096, 5000])
def test_dense_attend(pk, orc, n):
    N, H, G = 1, 2, 4
    kk, vv = _rand_kv(N, H, n, seed=n + 1, scale=2.0)
    c = build_cache(kk, vv, G)
    q = torch.randn((N, H, G, 128), generator=torch.Generator().manual_seed(3))
    out = torch.zeros((N, H, G, 128), device="cuda")
    ws = c.workspace(1, pk.WS_DENSE)
    pk.bpkv_dense_attend(c.c, q.cuda(), out, ws, ws.numel())
    got = out.cpu().numpy()
    for h in range(H):
        ref = orc.dense_attend(q[0, h].numpy(), bits16(kk[0, h]), bits16(vv[0, h]), n)
        assert np.max(np.abs(got[0, h] - ref)) <= ATTN_ATOL


@pytest.mark.parametrize("n_ties,n_above", [(10000, 100), (5000, 475), (6000, 0)])
def test_topk_massive_ties(pk, orc, n_ties, n_above):
    """More than 4096 scores equal to the threshold score: the lowest indices win."""
    N, H, G, n, k = 1, 1, 4, 20000, 512
    kk, vv = _rand_kv(N, H, n, seed=8)
    c = build_cache(kk, vv, G)
    g = torch.Generator(device="cpu").manual_seed(n_ties + n_above)
    sc = torch.rand((N, H, G, n), generator=g) * 0.5          # below the tie value
    for q in range(G):
        perm = torch.randperm(n, generator=g)
        sc[0, 0, q, perm[:n_ties]] = 1.0
        sc[0, 0, q, perm[n_ties:n_ties + n_above]] = 2.0 + torch.rand(n_above, generator=g)
    ld = c.c.cap_tokens
    buf = torch.zeros((N, H, G, ld), device="cuda")
    buf[..., :n] = sc.cuda()
    idx = torch.zeros((N, H, G, k), dtype=torch.int32, device="cuda")
    ws = c.workspace(k, pk.WS_SCAN_TOPK)
    pk.bpkv_clear_status(ws)
    pk.bpkv_topk(c.c, buf, ld, k, 4, 32, idx, ws, ws.numel())
    assert pk.bpkv_read_status(ws) == 0
    for q in range(G):
        want = orc.topk(sc[0, 0, q].numpy().astype(np.float64), k)
        assert np.array_equal(idx[0, 0, q].cpu().numpy(), want), q


def _topk_rows(pk, c, sc, k, n_sink=4, n_recent=32):
    """bpkv_topk on given scores [N][H][G][n] (the kernel counts its own histogram)."""
    N, H, G, n = sc.shape
    ld = c.c.cap_tokens
    buf = torch.zeros((N, H, G, ld), device="cuda")
    buf[..., :n] = sc.cuda()
    idx = torch.zeros((N, H, G, k), dtype=torch.int32, device="cuda")
    ws = c.workspace(k, pk.WS_SCAN_TOPK)
    pk.bpkv_clear_status(ws)
    pk.bpkv_topk(c.c, buf, ld, k, n_sink, n_recent, idx, ws, ws.numel())
    assert pk.bpkv_read_status(ws) == 0
    return idx.cpu().numpy()


@pytest.mark.parametrize("n,k,ties", [(70000, 512, 0.3), (100003, 2048, 0.0), (32772, 512, 0.0),
                                      (32805, 100, 0.95)])
def test_topk_long_rows(pk, orc, n, k, ties):
    """Rows longer than one staged tile of 32768 keys: every pass runs tile by tile."""
    from workload.gen import random_scores
    N, H, G = 1, 1, 2
    kk, vv = _rand_kv(N, H, n, seed=11)
    c = build_cache(kk, vv, G)
    sc = random_scores(N * H * G, n, seed=n + 7 * k, tie_frac=ties).reshape(N, H, G, n)
    got = _topk_rows(pk, c, sc, k)
    for g in range(G):
        want = orc.topk(sc[0, 0, g].numpy().astype(np.float64), k)
        assert np.array_equal(got[0, 0, g], want), g


@pytest.mark.parametrize("n,spread", [(20000, 3000), (20000, 40), (70000, 0), (20000, 0), (50000, 200000)])
def test_topk_refinement_levels(pk, orc, n, spread):
    """Scores packed into a few ulps of 1.0: the first-level bucket holds most
    keys, so the second and third radix levels (and, at spread 0 or with long
    runs of equal keys, the ordered tie cut) decide the set."""
    N, H, G, k = 1, 1, 2, 512
    kk, vv = _rand_kv(N, H, n, seed=12)
    c = build_cache(kk, vv, G)
    g = torch.Generator(device="cpu").manual_seed(n + spread)
    steps = torch.randint(0, max(spread, 1), (N, H, G, n), generator=g) if spread else torch.zeros(
        (N, H, G, n), dtype=torch.int64)
    sc = (1.0 + steps.double() * 2.0 ** -23).float()
    got = _topk_rows(pk, c, sc, k)
    for q in range(G):
        want = orc.topk(sc[0, 0, q].numpy().astype(np.float64), k)
        assert np.array_equal(got[0, 0, q], want), q


@pytest.mark.parametrize("n,G,budget", [(3000, 4, 136), (40000, 2, 92), (700, 8, 68), (37, 4, 136)])
def test_scan_topk_histogram_matches_topk(pk, n, G, budget):
    """bpkv_scan_topk (histogram counted by the scan) gives the same indices as
    bpkv_scan followed by bpkv_topk (histogram counted by the top-k kernel)."""
    N, H, k = 2, 2, 256
    kk, vv = _rand_kv(N, H, n, seed=13)
    c = build_cache(kk, vv, G)
    gq = torch.Generator(device="cpu").manual_seed(n + G)
    q = torch.randn((N, H, G, 128), generator=gq).cuda()
    s2 = torch.ones((N, H, 128), device="cuda")
    bq = torch.full((N,), budget * 4, dtype=torch.int32, device="cuda")
    depths = torch.zeros((N, H, 128), dtype=torch.uint8, device="cuda")
    pk.bpkv_alloc_depths(c.c, q, s2, bq, depths)
    ws = c.workspace(k, pk.WS_SCAN_TOPK)
    idx_a = torch.zeros((N, H, G, k), dtype=torch.int32, device="cuda")
    pk.bpkv_clear_status(ws)
    pk.bpkv_scan_topk(c.c, q, depths, k, 4, 32, idx_a, ws, ws.numel())
    assert pk.bpkv_read_status(ws) == 0
    ld = c.c.cap_tokens
    scores = torch.zeros((N, H, G, ld), device="cuda")
    pk.bpkv_scan(c.c, q, depths, scores, ld)
    idx_b = torch.zeros_like(idx_a)
    pk.bpkv_topk(c.c, scores, ld, k, 4, 32, idx_b, ws, ws.numel())
    assert pk.bpkv_read_status(ws) == 0
    assert torch.equal(idx_a, idx_b)


@pytest.mark.parametrize("N,H,G,n", [(2, 8, 4, 70001), (1, 8, 8, 70001), (1, 4, 2, 300000)])
def test_scan_topk_grid_too_large_for_cut(pk, orc, N, H, G, n):
    """Grids too large for the cut to count its own histograms: the scan counts
    them (in shared memory for up to 4 query heads; k_hist for more).  Same
    indices as bpkv_scan + bpkv_topk, and sampled rows equal the oracle's top-k
    of the oracle's scores."""
    k = 512
    kk, vv = _rand_kv(N, H, n, seed=23)
    c = build_cache(kk, vv, G)
    gq = torch.Generator(device="cpu").manual_seed(n + G + 7)
    q = torch.randn((N, H, G, 128), generator=gq).cuda()
    s2 = torch.ones((N, H, 128), device="cuda")
    bq = torch.full((N,), 92 * 4, dtype=torch.int32, device="cuda")
    depths = torch.zeros((N, H, 128), dtype=torch.uint8, device="cuda")
    pk.bpkv_alloc_depths(c.c, q, s2, bq, depths)
    ws = c.workspace(k, pk.WS_SCAN_TOPK)
    idx_a = torch.zeros((N, H, G, k), dtype=torch.int32, device="cuda")
    pk.bpkv_clear_status(ws)
    pk.bpkv_scan_topk(c.c, q, depths, k, 4, 32, idx_a, ws, ws.numel())
    assert pk.bpkv_read_status(ws) == 0
    ld = c.c.cap_tokens
    scores = torch.zeros((N, H, G, ld), device="cuda")
    pk.bpkv_scan(c.c, q, depths, scores, ld)
    idx_b = torch.zeros_like(idx_a)
    pk.bpkv_topk(c.c, scores, ld, k, 4, 32, idx_b, ws, ws.numel())
    assert pk.bpkv_read_status(ws) == 0
    differ = [tuple(int(x) for x in r) for r in (idx_a != idx_b).any(dim=-1).nonzero().cpu()]
    assert not differ, f"rows (seq, head, query head) whose lists differ: {differ[:8]}"
    # one sampled unit against the oracle (scores and top-k sets within the bar)
    s, h = N - 1, H - 1
    kb = bits16(kk[s, h])
    scales, planes = orc.encode(kb, c.c.cap_tokens // 64)
    d = depths[s, h].cpu().numpy()
    qq = q[s, h].cpu().numpy()
    ref = orc.scores(n, scales, planes, d, qq)
    check_scores(scores[s, h, :, :n].cpu().numpy(), ref, abs_score_scale(qq, kb, d), "large-grid scan")
    for g in range(G):
        check_topk_sets(idx_a[s, h, g].cpu().numpy(), orc.topk(ref[g], k), ref[g], k, what=f"head {g}")


@pytest.mark.parametrize("n,ties", [(140000, 0.0), (150001, 0.9), (270000, 0.0), (300001, 0.9)])
def test_topk_long_rows_level1(pk, orc, n, ties):
    """Rows over a grid too large to run cooperatively.  Of 262144 keys or
    more: the level-1 histogram (k_hist1) narrows the level-0 bucket before
    the cut.  Shorter: a bucket of more than 1024 keys (the heavy ties) is
    refined by the row's last CTA."""
    from workload.gen import random_scores
    N, H, G, k = 1, 4, 4, 512
    kk, vv = _rand_kv(N, H, n, seed=14)
    c = build_cache(kk, vv, G)
    sc = random_scores(N * H * G, n, seed=n, tie_frac=ties).reshape(N, H, G, n)
    got = _topk_rows(pk, c, sc, k)
    for h in range(H):
        for g in range(G):
            want = orc.topk(sc[0, h, g].numpy().astype(np.float64), k)
            assert np.array_equal(got[0, h, g], want), (h, g)


@pytest.mark.parametrize("n,n_sink,n_recent,k,ties", [(140000, 5, 30, 512, 0.0), (98307, 7, 33, 300, 0.5),
                                                      (70001, 0, 0, 64, 0.0), (65537, 3, 1, 37, 0.9)])
def test_topk_streaming_cut_unaligned(pk, orc, n, n_sink, n_recent, k, ties):
    """Grids too large to run cooperatively (the row bucket kernel, then the
    streaming cut over token-aligned 8192-token chunks) with sink and recent
    counts that are not multiples of 4: the middle range starts and ends
    inside 16-byte score groups and inside chunks."""
    from workload.gen import random_scores
    N, H, G = 1, 8, 4  # 32 rows: more CTAs than fit at once for every n here
    kk, vv = _rand_kv(N, H, n, seed=15)
    c = build_cache(kk, vv, G)
    sc = random_scores(N * H * G, n, seed=n + k, tie_frac=ties).reshape(N, H, G, n)
    got = _topk_rows(pk, c, sc, k, n_sink, n_recent)
    for h in range(H):
        for g in range(G):
            want = orc.topk(sc[0, h, g].numpy().astype(np.float64), k, n_sink, n_recent)
            assert np.array_equal(got[0, h, g], want), (h, g)
