"""Value-side read depth (ReadKV page, sections 5.3-5.4) on the GPU against the
oracle: the value rows' own 4-bit code bit-exact (bulk appends and the decode
step's append), and the second read stage (row weights from the exact-key
attention, greedy value depths, output through each row's prefix).

The depths are decided by float32 row weights on the GPU and by float64
weights in the oracle, so they are held to validity, not equality: the GPU's
taken items must be a greedy choice for weights within float32 rounding of
the oracle's (every taken item worth at least every untaken one, up to a
relative 1e-4), the planes used must be min(budget, items worth > 0), and the
output must match the oracle's stage evaluated on the GPU's depths within the
attention bar (2e-3)."""
import numpy as np
import pytest
import torch

from gpu_helpers import ATTN_ATOL, bits16, bits64, build_cache, check_topk_sets

pytestmark = pytest.mark.gpu

W_RTOL = 1e-4  # row weights and the greedy order: float32 against float64


@pytest.fixture(scope="module")
def pk():
    import __graft_entry__
    __graft_entry__.build()
    import bit_plane_kv_encode_gb300 as m
    return m


def _kv(N, H, n, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    sig = torch.exp(0.75 * torch.randn((N, H, 1, 128), generator=g))
    k = (torch.randn((N, H, n, 128), generator=g) * sig).to(torch.bfloat16)
    v = (torch.randn((N, H, n, 128), generator=g) * torch.exp(torch.randn((N, H, n, 1), generator=g))).to(torch.bfloat16)
    if n > 5:
        v[0, 0, 5] = 0  # an all-zero row: scale 0, every code 8
    return k, v, g


def _values_cache(pk, k, v, group, chunks=None, cap=None):
    from bit_plane_kv_encode_gb300 import Cache
    N, H, n, _ = k.shape
    cap = cap or (n + 511) // 512 * 512
    c = Cache(N, H, group, cap, values=True)
    pos = 0
    for t in (chunks or [n]):
        t = min(t, n - pos)
        if t <= 0:
            break
        c.append(k[:, :, pos:pos + t].contiguous().cuda(), v[:, :, pos:pos + t].contiguous().cuda())
        pos += t
    if pos < n:
        c.append(k[:, :, pos:].contiguous().cuda(), v[:, :, pos:].contiguous().cuda())
    torch.cuda.synchronize()
    return c


@pytest.mark.parametrize("n,chunks", [(1000, None), (64 * 3 + 17, [1] * 40 + [63, 1, 64, 65]), (1, [1])])
def test_value_encode_bitexact(pk, orc, n, chunks):
    N, H = 2, 3
    k, v, _ = _kv(N, H, n, seed=n)
    c = _values_cache(pk, k, v, 4, chunks)
    for s in range(N):
        for h in range(H):
            vs, vp = orc.v_encode(bits16(v[s, h]))
            assert np.array_equal(bits16(c.vscales[s, h])[:n], vs), (s, h)
            assert np.array_equal(bits64(c.vplanes[s, h])[:n], vp), (s, h)


def _check_depths(w_ref, dep, budget, what=""):
    """dep (GPU) is a greedy choice for the float64 weights w_ref up to W_RTOL."""
    n_u = len(w_ref)
    val = lambda r, t: w_ref[r] * 4.0 ** (-t)  # noqa: E731
    positive = sum(1 for r in range(n_u) for t in range(4) if val(r, t) > 0)
    assert int(dep.sum()) == min(budget, positive), f"{what}: {int(dep.sum())} planes for budget {budget}"
    taken = [val(r, t) for r in range(n_u) for t in range(int(dep[r]))]
    untaken = [val(r, t) for r in range(n_u) for t in range(int(dep[r]), 4)]
    if taken and untaken:
        assert min(taken) >= max(untaken) * (1 - W_RTOL), f"{what}: taken {min(taken)} < untaken {max(untaken)}"


def _union_on_device(uidx, umask, u_cap):
    ui = torch.full((1, 1, u_cap), -1, dtype=torch.int32)
    um = torch.zeros((1, 1, u_cap), dtype=torch.uint8)
    ui[0, 0, :len(uidx)] = torch.from_numpy(uidx)
    um[0, 0, :len(umask)] = torch.from_numpy(umask)
    return ui.cuda(), um.cuda(), torch.tensor([[len(uidx)]], dtype=torch.int32).cuda()


@pytest.mark.parametrize("n,G,k", [(4096, 4, 64), (20000 + 7, 4, 512), (3000, 8, 256), (700, 1, 100)])
def test_attend_vdepth_vs_oracle(pk, orc, n, G, k):
    """One unit's stage over the oracle's union, at budgets from nothing to every plane."""
    k_, v_, g = _kv(1, 1, n, seed=n + G)
    c = _values_cache(pk, k_, v_, G)
    q = torch.randn((1, 1, G, 128), generator=g)
    kb, vb = bits16(k_[0, 0]), bits16(v_[0, 0])
    scales, planes = orc.encode(kb, c.c.cap_tokens // 64)
    depth = np.full(128, 4, np.uint8)
    sc = orc.scores(n, scales, planes, depth, q[0, 0].numpy())
    idx = np.stack([orc.topk(sc[h], k, 4, 32) for h in range(G)])
    uidx, umask = orc.union(idx)
    n_u = len(uidx)
    u_cap = G * k
    ui, um, uc = _union_on_device(uidx, umask, u_cap)
    vs, vp = orc.v_encode(vb)
    for budget in [0, n_u // 3, n_u, 2 * n_u + 1, 4 * n_u, 10 * n_u]:
        out = torch.zeros((1, 1, G, 128), device="cuda")
        dep = torch.zeros((1, 1, u_cap), dtype=torch.uint8, device="cuda")
        wt = torch.zeros((1, 1, u_cap), dtype=torch.float32, device="cuda")
        pk.bpkv_sparse_attend_vdepth(c.c, q.cuda(), ui, um, uc, u_cap, budget, out, dep, wt)
        torch.cuda.synchronize()
        d = dep[0, 0, :n_u].cpu().numpy()
        ref = orc.attend_vdepth(q[0, 0].numpy(), kb, vs, vp, uidx, umask, budget, depth_in=d)
        w = wt[0, 0, :n_u].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(w - ref["weight"])) <= W_RTOL * np.max(ref["weight"]), f"budget {budget}: weights"
        _check_depths(ref["weight"], d, budget, what=f"n{n} G{G} budget {budget}")
        err = float(np.max(np.abs(out[0, 0].cpu().numpy() - ref["out"])))
        assert err <= ATTN_ATOL, f"budget {budget}: output err {err}"
        if budget == 0:
            assert not out.any()
        if budget >= 4 * n_u:
            assert (d == 4).all()
    # the oracle's own allocation at a middle budget gives the same output up to near-ties
    ref = orc.attend_vdepth(q[0, 0].numpy(), kb, vs, vp, uidx, umask, n_u)
    out = torch.zeros((1, 1, G, 128), device="cuda")
    pk.bpkv_sparse_attend_vdepth(c.c, q.cuda(), ui, um, uc, u_cap, n_u, out)
    torch.cuda.synchronize()
    assert float(np.max(np.abs(out[0, 0].cpu().numpy() - ref["out"]))) <= 5 * ATTN_ATOL


@pytest.mark.parametrize("wl,n_tok,budget_rows", [("tiny", 4096, 1.0), ("qwen3_8b_layer", 32768, 2.0),
                                                  ("tiny", 300, 0.5)])
def test_decode_step_vdepth(pk, orc, wl, n_tok, budget_rows):
    """A whole decode step with value-side depths: the new token's value row is
    coded by the step, each head's selection follows the tie rule, and the
    output equals the oracle's second stage over the GPU's union and depths."""
    from bit_plane_kv_encode_gb300 import Cache
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS[wl]
    inp = gen_layer(cfg, 4, device="cuda", n_tokens=n_tok)
    N, H, n, D = inp.k.shape
    G, K = cfg.group, cfg.k
    c = Cache(N, H, G, (n + 511) // 512 * 512, values=True)
    c.append(inp.k[:, :, :n - 1].contiguous(), inp.v[:, :, :n - 1].contiguous())
    ws = c.workspace(K, pk.WS_STEP)
    out = torch.zeros((1, N, H, G, D), device="cuda")
    depths = torch.zeros((1, N, H, D), dtype=torch.uint8, device="cuda")
    idx = torch.zeros((1, N, H, G, K), dtype=torch.int32, device="cuda")
    vdep = torch.zeros((1, N, H, G * K), dtype=torch.uint8, device="cuda")
    q = inp.q.cuda()[None].contiguous()
    s2 = inp.sigma2.cuda()[None].contiguous()
    bq = (4 * inp.budgets).to(torch.int32).cuda()
    kn = inp.k[:, :, n - 1][None].contiguous()
    vn = inp.v[:, :, n - 1][None].contiguous()
    budget_v = int(budget_rows * min(n, G * K))
    a = pk.bpkv_step_args(kn.data_ptr(), vn.data_ptr(), q.data_ptr(), s2.data_ptr(), bq.data_ptr(), 0, 0, 0, K,
                          cfg.n_sink, cfg.n_recent, out.data_ptr(), depths.data_ptr(), idx.data_ptr(), None,
                          pk.STEP_VDEPTH, None, budget_v, vdep.data_ptr())
    arr = pk.cache_array([c])
    pk.bpkv_clear_status(ws)
    pk.bpkv_decode_step(arr, 1, a, ws, ws.numel())
    torch.cuda.synchronize()
    assert pk.bpkv_read_status(ws) == 0
    kc, vc = inp.k.cpu(), inp.v.cpu()
    for h in range(H):
        kb, vb = bits16(kc[0, h]), bits16(vc[0, h])
        vs, vp = orc.v_encode(vb)
        assert np.array_equal(bits64(c.vplanes[0, h])[:n], vp) and np.array_equal(bits16(c.vscales[0, h])[:n], vs)
        ref = orc.decode_unit(kb, vb, inp.q[0, h].numpy(), inp.sigma2[0, h].numpy(), int(inp.budgets[0]), K,
                              cfg.n_sink, cfg.n_recent, nb_cap=c.c.cap_tokens // 64)
        gi = idx[0, 0, h].cpu().numpy()
        for gg in range(G):
            check_topk_sets(gi[gg], ref["idx"][gg], ref["scores"][gg], K, cfg.n_sink, cfg.n_recent, what=f"h{h} g{gg}")
        uidx, umask = orc.union(gi)
        d = vdep[0, 0, h, :len(uidx)].cpu().numpy()
        st = orc.attend_vdepth(inp.q[0, h].numpy(), kb, vs, vp, uidx, umask, budget_v, depth_in=d)
        _check_depths(st["weight"], d, budget_v, what=f"{wl} h{h}")
        err = float(np.max(np.abs(out[0, 0, h].cpu().numpy() - st["out"])))
        assert err <= ATTN_ATOL, f"{wl} h{h}: {err}"
