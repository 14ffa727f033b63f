"""Decode steps in sequence and several layers in one call: the appended
token counts in seq_len from the end of its layer's step, and every later
step (or layer) sees the cache it left.  Checked against the oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import build_cache, check_unit

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    import __graft_entry__
    __graft_entry__.build()
    import bit_plane_kv_encode_gb300 as m
    return m


def _args(pk, cfg, k_new, v_new, q, sigma2, budget_q, out, depths, idx):
    return pk.bpkv_step_args(k_new.data_ptr(), v_new.data_ptr(), q.data_ptr(), sigma2.data_ptr(), budget_q.data_ptr(),
                             pk.DEPTH_WATERFILL, 0, 0, cfg.k, cfg.n_sink, cfg.n_recent, out.data_ptr(),
                             depths.data_ptr(), idx.data_ptr(), None, 0)


@pytest.mark.parametrize("wl,n_tok,steps", [("tiny", 4096 + 60, 6), ("qwen3_8b_layer", 3000, 3)])
def test_consecutive_steps(pk, orc, wl, n_tok, steps):
    """`steps` decode steps on one cache, a new query each step, crossing a
    64-token block boundary; each step is checked on every unit."""
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS[wl]
    inp = gen_layer(cfg, 2, device="cuda", n_tokens=n_tok)
    N, H, n, D = inp.k.shape
    G = cfg.group
    n0 = n - steps
    k_all, v_all = inp.k, inp.v
    cache = build_cache(k_all, v_all, G, cap=((n + 511) // 512) * 512, n_prefill=n0)
    ws = cache.workspace(cfg.k, pk.WS_STEP)
    arr = pk.cache_array([cache])
    gq = torch.Generator(device="cpu").manual_seed(99)
    sigma2 = inp.sigma2.cuda()[None].contiguous()
    budget_q = (4 * inp.budgets).to(torch.int32).cuda()
    for st in range(steps):
        t = n0 + st  # token appended by this step
        q_cpu = inp.q + 0.25 * st * torch.randn(inp.q.shape, generator=gq)
        q = q_cpu.cuda()[None].contiguous()
        out = torch.zeros((1, N, H, G, D), device="cuda")
        depths = torch.zeros((1, N, H, D), dtype=torch.uint8, device="cuda")
        idx = torch.zeros((1, N, H, G, cfg.k), dtype=torch.int32, device="cuda")
        k_new = k_all[:, :, t][None].contiguous()
        v_new = v_all[:, :, t][None].contiguous()
        a = _args(pk, cfg, k_new, v_new, q, sigma2, budget_q, out, depths, idx)
        pk.bpkv_clear_status(ws)
        pk.bpkv_decode_step(arr, 1, a, ws, ws.numel())
        pk.sync_n_max([cache], arr)
        torch.cuda.synchronize()
        assert pk.bpkv_read_status(ws) == 0
        assert torch.all(cache.seq_len.cpu() == t + 1), (st, cache.seq_len.cpu())
        # the oracle sees the first t + 1 tokens and this step's query
        sub = type(inp)(**{**inp.__dict__})
        sub.k, sub.v, sub.q = k_all[:, :, : t + 1].cpu(), v_all[:, :, : t + 1].cpu(), q_cpu
        for s in range(N):
            for h in range(H):
                same, _ = check_unit(orc, cfg, sub, cache, depths[0], idx[0], out[0], s, h, what=f"step {st} s{s} h{h}")
                assert same >= G - 1


def test_two_layers_one_call(pk, orc):
    """Two layers (own caches, queries and new tokens) in one bpkv_decode_step."""
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS["qwen3_8b_layer"]
    L = 2
    inps = [gen_layer(cfg, l, device="cuda", n_tokens=5000 + 7 * l) for l in range(L)]
    # layers share the cache shape: use the shorter length for both
    n = min(i.k.shape[2] for i in inps)
    N, H, _, D = inps[0].k.shape
    G = cfg.group
    caches = [build_cache(i.k[:, :, :n], i.v[:, :, :n], G, cap=((n + 511) // 512) * 512, n_prefill=n - 1)
              for i in inps]
    ws = caches[0].workspace(cfg.k, pk.WS_STEP)
    q = torch.stack([i.q for i in inps]).cuda().contiguous()
    sigma2 = torch.stack([i.sigma2 for i in inps]).cuda().contiguous()
    budget_q = (4 * inps[0].budgets).to(torch.int32).cuda()
    k_new = torch.stack([i.k[:, :, n - 1] for i in inps]).contiguous()
    v_new = torch.stack([i.v[:, :, n - 1] for i in inps]).contiguous()
    out = torch.zeros((L, N, H, G, D), device="cuda")
    depths = torch.zeros((L, N, H, D), dtype=torch.uint8, device="cuda")
    idx = torch.zeros((L, N, H, G, cfg.k), dtype=torch.int32, device="cuda")
    a = _args(pk, cfg, k_new, v_new, q, sigma2, budget_q, out, depths, idx)
    arr = pk.cache_array(caches)
    pk.bpkv_clear_status(ws)
    pk.bpkv_decode_step(arr, L, a, ws, ws.numel())
    pk.sync_n_max(caches, arr)
    torch.cuda.synchronize()
    assert pk.bpkv_read_status(ws) == 0
    for l in range(L):
        assert torch.all(caches[l].seq_len.cpu() == n)
        sub = type(inps[l])(**{**inps[l].__dict__})
        sub.k, sub.v = inps[l].k[:, :, :n].cpu(), inps[l].v[:, :, :n].cpu()
        for h in range(H):
            same, _ = check_unit(orc, cfg, sub, caches[l], depths[l], idx[l], out[l], 0, h, what=f"layer {l} h{h}")
            assert same >= G - 1
