"""Keys coded in a fixed orthogonal basis (Fathom page, contributions: KLT planes
for models without QK norm; ReadKV page, section 5.1: Hadamard-sign transform):
bpkv_rotate, the encoder and whole decode steps against the oracle, bit for bit
where the arithmetic is integer or an identical float32 chain."""
import dataclasses

import numpy as np
import pytest
import torch

from gpu_helpers import bits16, bits64, build_cache, check_unit, decode_one_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    import __graft_entry__
    __graft_entry__.build()
    import bit_plane_kv_encode_gb300 as m
    return m


def hadamard_sign(H, seed):
    """Per KV head: diag(signs) H_128 / sqrt(128) (orthogonal)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    h = torch.ones((1, 1))
    while h.shape[0] < 128:
        h = torch.cat([torch.cat([h, h], 1), torch.cat([h, -h], 1)], 0)
    out = []
    for _ in range(H):
        s = torch.randint(0, 2, (128, 1), generator=g).float() * 2 - 1
        out.append(s * h / 128 ** 0.5)
    return torch.stack(out).float().contiguous()


def klt_like(H, seed):
    """Per KV head: a random orthogonal basis (QR of a Gaussian matrix)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.stack([torch.linalg.qr(torch.randn((128, 128), generator=g, dtype=torch.float64))[0]
                        for _ in range(H)]).float().contiguous()


def test_rotate_matches_oracle(pk, orc):
    N, H, rows = 2, 3, 5
    g = torch.Generator(device="cpu").manual_seed(1)
    x = torch.randn((N, H, rows, 128), generator=g)
    R = torch.randn((H, 128, 128), generator=g)  # any matrix: the arithmetic is what is checked
    y = torch.zeros_like(x).cuda()
    pk.bpkv_rotate(R.cuda(), N, H, rows, x.cuda(), y)
    got = y.cpu().numpy()
    for s in range(N):
        for h in range(H):
            assert np.array_equal(got[s, h], orc.rotate(x[s, h].numpy(), R[h].numpy())), (s, h)


@pytest.mark.parametrize("kind,n,chunks", [("hadamard", 3000, None), ("klt", 1000, [1, 63, 1, 200, 5]),
                                           ("hadamard", 64, None)])
def test_encode_with_basis(pk, orc, kind, n, chunks):
    N, H = 2, 2
    g = torch.Generator(device="cpu").manual_seed(n)
    k = (torch.randn((N, H, n, 128), generator=g) * torch.exp(0.75 * torch.randn((N, H, 1, 128), generator=g)))
    k = k.to(torch.bfloat16).cuda()
    v = torch.randn((N, H, n, 128), generator=g).to(torch.bfloat16).cuda()
    R = (hadamard_sign(H, 5) if kind == "hadamard" else klt_like(H, 5)).cuda()
    c = build_cache(k, v, 4, chunks=chunks, basis=R)
    torch.cuda.synchronize()
    nb = (n + 63) // 64
    for s in range(N):
        for h in range(H):
            kr = orc.rotate_keys(bits16(k[s, h]), R[h].cpu().numpy())
            sc, pl = orc.encode(kr, c.c.cap_tokens // 64)
            assert np.array_equal(bits64(c.planes[s, h])[:, :, :nb], pl[:, :, :nb]), (s, h)
            assert np.array_equal(bits16(c.scales[s, h])[:, :nb], sc[:, :nb]), (s, h)
            assert np.array_equal(bits16(c.k_rows[s, h, :n]), bits16(k[s, h]))  # rows stay unrotated


@pytest.mark.parametrize("kind,rule", [("hadamard", 0), ("klt", 0), ("klt", 1)])
def test_decode_step_with_basis(pk, orc, kind, rule):
    """One decode step on every unit of a 4-head layer with the keys coded in a
    basis: planes, depths (from q R), top-k sets and attention against the
    oracle's decode of the same basis."""
    from workload import CONFIGS, gen_layer
    cfg = dataclasses.replace(CONFIGS["qwen3_8b_layer"], n_tokens=5000, n_kv_heads=4)
    inp = gen_layer(cfg, 0)
    N, H = inp.k.shape[:2]
    R = hadamard_sign(H, 9) if kind == "hadamard" else klt_like(H, 9)
    fixed = (32, 4) if rule == 1 else (0, 0)
    cache, depths, idx, out = decode_one_layer(inp, cfg, depth_rule=rule, fixed=fixed, basis=R.cuda())
    for s in range(N):
        for h in range(H):
            check_unit(orc, cfg, inp, cache, depths, idx, out, s, h, depth_rule=rule, fixed=fixed,
                       what=f"{kind} unit {s},{h}", basis=R[h].numpy())


def test_scan_with_queries_in_basis(pk, orc):
    """The stand-alone scan takes q already in the cache's basis (bpkv_rotate)."""
    N, H, G, n = 1, 2, 4, 2000
    g = torch.Generator(device="cpu").manual_seed(4)
    k = (torch.randn((N, H, n, 128), generator=g) * 2).to(torch.bfloat16).cuda()
    v = torch.randn((N, H, n, 128), generator=g).to(torch.bfloat16).cuda()
    R = klt_like(H, 3).cuda()
    c = build_cache(k, v, G, basis=R)
    q = torch.randn((N, H, G, 128), generator=g).cuda()
    qr = torch.zeros_like(q)
    pk.bpkv_rotate(R, N, H, G, q, qr)
    d = torch.randint(0, 5, (N, H, 128), generator=g, dtype=torch.uint8).cuda()
    scores = torch.full((N, H, G, c.c.cap_tokens), float("nan"), device="cuda")
    pk.bpkv_scan(c.c, qr, d, scores, c.c.cap_tokens)
    torch.cuda.synchronize()
    from gpu_helpers import abs_score_scale, check_scores
    for h in range(H):
        kr = orc.rotate_keys(bits16(k[0, h]), R[h].cpu().numpy())
        sc, pl = orc.encode(kr, c.c.cap_tokens // 64)
        qh = orc.rotate(q[0, h].cpu().numpy(), R[h].cpu().numpy())
        ref = orc.scores(n, sc, pl, d[0, h].cpu().numpy(), qh)
        check_scores(scores[0, h, :, :n].cpu().numpy(), ref, abs_score_scale(qh, kr, d[0, h].cpu().numpy()),
                     f"head {h}")
