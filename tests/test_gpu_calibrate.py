"""Offline-calibrated channel sets (Fathom page, section 2, "Double Sparsity")
and decode steps that read a caller-given depth vector: bpkv_calibrate_channels
against the oracle bit for bit, and a decode step with BPKV_DEPTH_GIVEN against
the oracle's decode of the same depths."""
import dataclasses

import numpy as np
import pytest
import torch

from gpu_helpers import bits16, check_unit, decode_one_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    import __graft_entry__
    __graft_entry__.build()
    import bit_plane_kv_encode_gb300 as m
    return m


def _calib(units, G, m_q, m_k, seed, dyadic=False):
    g = torch.Generator(device="cpu").manual_seed(seed)
    if dyadic:
        # sums exact in double: ties of the statistic stay exact ties
        q = (torch.randint(0, 33, (units, m_q, G, 128), generator=g) / 4.0).float()
        q = q * (torch.randint(0, 2, q.shape, generator=g) * 2 - 1)
        k = (torch.randint(0, 33, (units, m_k, 128), generator=g) / 8.0)
    else:
        q = torch.randn((units, m_q, G, 128), generator=g)
        k = torch.randn((units, m_k, 128), generator=g) * torch.exp(0.75 * torch.randn((units, 1, 128), generator=g))
    k = k.to(torch.bfloat16)
    # an exact tie between two channels of unit 0 (equal columns)
    q[0, :, :, 7] = q[0, :, :, 3]
    k[0, :, 7] = k[0, :, 3]
    return q.contiguous(), k.contiguous()


@pytest.mark.parametrize("units,G,m_q,m_k,c,t,dyadic", [
    (3, 4, 16, 512, 32, 4, False), (2, 8, 1, 64, 16, 2, False), (5, 1, 7, 1000, 40, 3, False),
    (2, 4, 8, 16, 32, 4, True), (1, 2, 3, 5, 128, 1, False), (2, 4, 4, 100, 0, 4, False),
    (4, 4, 64, 4096, 200, 2, False)])
def test_calibrate_matches_oracle(pk, orc, units, G, m_q, m_k, c, t, dyadic):
    q, k = _calib(units, G, m_q, m_k, seed=units * 100 + m_q, dyadic=dyadic)
    d = torch.full((units, 128), 77, dtype=torch.uint8, device="cuda")
    pk.bpkv_calibrate_channels(q.cuda(), k.cuda(), units, G, m_q, m_k, c, t, d)
    torch.cuda.synchronize()
    got = d.cpu().numpy()
    for u in range(units):
        want = orc.calibrate_channels(q[u].numpy(), bits16(k[u]), c, t)
        assert np.array_equal(got[u], want), (u, np.nonzero(got[u] != want))


def test_calibrate_rejects_bad_arguments(pk):
    q = torch.zeros((1, 1, 4, 128), device="cuda")
    k = torch.zeros((1, 1, 128), dtype=torch.bfloat16, device="cuda")
    d = torch.zeros((1, 128), dtype=torch.uint8, device="cuda")
    for args in [(0, 4, 1, 1, 32, 4), (1, 0, 1, 1, 32, 4), (1, 4, 0, 1, 32, 4), (1, 4, 1, 0, 32, 4),
                 (1, 4, 1, 1, -1, 4), (1, 4, 1, 1, 32, 5)]:
        with pytest.raises(pk.BpkvError):
            pk.bpkv_calibrate_channels(q, k, *args, d)


def test_decode_step_given_depths(pk, orc):
    """Depths calibrated from each unit's own first 2048 keys and 4 random
    queries, then one decode step that reads them (BPKV_DEPTH_GIVEN); every
    unit is compared with the oracle decoding the same depth vector."""
    from workload import CONFIGS, gen_layer
    cfg = dataclasses.replace(CONFIGS["qwen3_8b_layer"], n_tokens=6000, n_kv_heads=4)
    inp = gen_layer(cfg, 0)
    N, H, n, D = inp.k.shape
    G = cfg.group
    g = torch.Generator(device="cpu").manual_seed(3)
    q_cal = torch.randn((N * H, 4, G, D), generator=g).contiguous()
    k_cal = inp.k[:, :, :2048].reshape(N * H, 2048, D).contiguous()
    depths_in = torch.zeros((N * H, D), dtype=torch.uint8, device="cuda")
    pk.bpkv_calibrate_channels(q_cal.cuda(), k_cal.cuda(), N * H, G, 4, 2048, 32, 4, depths_in)
    depths_in = depths_in.view(1, N, H, D)
    cache, depths, idx, out = decode_one_layer(inp, cfg, depth_rule=pk.DEPTH_GIVEN, depths_in=depths_in)
    assert torch.equal(depths, depths_in[0])
    for s in range(N):
        for h in range(H):
            dv = depths_in[0, s, h].cpu().numpy()
            want = orc.calibrate_channels(q_cal[s * H + h].numpy(), bits16(k_cal[s * H + h]), 32, 4)
            assert np.array_equal(dv, want)
            check_unit(orc, cfg, inp, cache, depths, idx, out, s, h, depth=dv, what=f"unit {s},{h}")


def test_given_depths_above_four_read_as_four(pk):
    """Depth values above 4 are read as 4 by the decode step (and reported so)."""
    from workload import CONFIGS, gen_layer
    cfg = dataclasses.replace(CONFIGS["tiny"], n_tokens=700)
    inp = gen_layer(cfg, 0)
    N, H, n, D = inp.k.shape
    raw = torch.zeros((1, N, H, D), dtype=torch.uint8)
    raw[..., :10] = 9
    raw[..., 10:20] = 4
    _, d_hi, _, out_hi = decode_one_layer(inp, cfg, depth_rule=pk.DEPTH_GIVEN, depths_in=raw.cuda())
    four = raw.clamp(max=4)
    _, d_4, _, out_4 = decode_one_layer(inp, cfg, depth_rule=pk.DEPTH_GIVEN, depths_in=four.cuda())
    assert torch.equal(d_hi, four[0].cuda()) and torch.equal(d_4, four[0].cuda())
    assert torch.equal(out_hi, out_4)


def test_given_depths_above_four_vs_oracle(pk, orc):
    """A decode step given depth values 5, 17 and 255 against the oracle's
    decode of the same raw depth vector (both read them as 4)."""
    from gpu_helpers import ATTN_ATOL, check_topk_sets
    from workload import CONFIGS, gen_layer
    cfg = dataclasses.replace(CONFIGS["tiny"], n_tokens=3000)
    inp = gen_layer(cfg, 2)
    N, H, n, D = inp.k.shape
    g = torch.Generator().manual_seed(11)
    raw = torch.randint(0, 5, (1, N, H, D), generator=g).to(torch.uint8)
    raw[..., 0:8], raw[..., 30:38], raw[..., 90:98] = 5, 17, 255
    cache, depths, idx, out = decode_one_layer(inp, cfg, depth_rule=pk.DEPTH_GIVEN, depths_in=raw.cuda())
    assert torch.equal(depths.cpu(), raw[0].clamp(max=4))
    kb, vb = bits16(inp.k[0, 0]), bits16(inp.v[0, 0])
    ref = orc.decode_unit(kb, vb, inp.q[0, 0].numpy(), inp.sigma2[0, 0].numpy(), None, cfg.k, cfg.n_sink,
                          cfg.n_recent, nb_cap=cache.c.cap_tokens // 64, depth=raw[0, 0, 0].numpy())
    for gg in range(cfg.group):
        gi = idx[0, 0, gg].cpu().numpy()
        d = check_topk_sets(gi, ref["idx"][gg], ref["scores"][gg], cfg.k, cfg.n_sink, cfg.n_recent, what=f"g{gg}")
        want = ref["out"][gg] if d == 0 else orc.attend(inp.q[0, 0, gg:gg + 1].numpy(), kb, vb, gi[None])[0]
        assert float(np.max(np.abs(out[0, 0, gg].cpu().numpy() - want))) <= ATTN_ATOL
