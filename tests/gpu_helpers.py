"""Helpers shared by the GPU parity tests, the smoke check and the bench:
building caches from generated inputs, running the oracle on a unit and the
comparison rules (bit-exact, score tolerance, top-k tie rule, attention
tolerance)."""
from __future__ import annotations

import numpy as np
import torch

SCORE_RTOL = 1e-5      # |gpu - oracle| <= 1e-5 max(|oracle|, sum_j |q_j khat_j|)
TIE_REL = 1e-4         # top-k sets may differ only on keys within 1e-4 max|score| of the k-th score
ATTN_ATOL = 2e-3       # attention outputs, max abs vs the float64 oracle


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def bits64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().numpy().view(np.uint64)


def build_cache(k: torch.Tensor, v: torch.Tensor, group: int, cap: int | None = None, n_prefill: int | None = None,
                residency: str = "hbm", chunks=None, basis=None):
    """Cache holding the first n_prefill (default all) rows of k/v [N][H][n][D]
    (keys coded in `basis`, float [H][D][D] on the device, when given)."""
    from bit_plane_kv_encode_gb300 import Cache
    N, H, n, _ = k.shape
    cap = cap if cap is not None else ((n + 511) // 512) * 512
    c = Cache(N, H, group, cap, device=k.device, residency=residency)
    if basis is not None:
        c.set_basis(basis)
    n_pre = n if n_prefill is None else n_prefill
    pos = 0
    for t in (chunks or [n_pre]):
        t = min(t, n_pre - pos)
        if t <= 0:
            break
        c.append(k[:, :, pos:pos + t].contiguous(), v[:, :, pos:pos + t].contiguous())
        pos += t
    if pos < n_pre:
        c.append(k[:, :, pos:n_pre].contiguous(), v[:, :, pos:n_pre].contiguous())
    return c


def abs_score_scale(q: np.ndarray, k_bits: np.ndarray, depth: np.ndarray) -> np.ndarray:
    """sum_j |q_gj khat_xj| [G][n], keys dequantised independently of the oracle."""
    from pins import dequant_direct
    kh = dequant_direct(k_bits, depth)
    return np.abs(q.astype(np.float64)) @ np.abs(kh).T


def check_scores(gpu: np.ndarray, ref: np.ndarray, scale: np.ndarray, what: str = ""):
    bound = SCORE_RTOL * np.maximum(np.abs(ref), scale)
    err = np.abs(gpu.astype(np.float64) - ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} scores out of tolerance, worst {np.max(err / (bound + 1e-300)):.3g}x"


def check_topk_sets(gpu_idx: np.ndarray, ref_idx: np.ndarray, ref_score: np.ndarray, k: int, n_sink: int = 4,
                    n_recent: int = 32, what: str = ""):
    """Same size; any differing key has an oracle score within TIE_REL max|score| of the
    oracle's k-th candidate score."""
    g = set(int(i) for i in gpu_idx if i >= 0)
    r = set(int(i) for i in ref_idx if i >= 0)
    assert len(g) == len(r), f"{what}: sizes {len(g)} vs {len(r)}"
    assert list(gpu_idx[:len(g)]) == sorted(g), f"{what}: gpu list not ascending"
    diff = g ^ r
    if not diff:
        return 0
    n = ref_score.shape[0]
    lo, hi = min(n_sink, n), max(n - n_recent, min(n_sink, n))
    cand = ref_score[lo:hi]
    n_top = k - n_sink - n_recent
    kth = np.sort(cand)[::-1][n_top - 1]
    tol = TIE_REL * np.max(np.abs(ref_score))
    for i in diff:
        assert lo <= i < hi, f"{what}: fixed token {i} differs"
        assert abs(ref_score[i] - kth) <= tol, f"{what}: key {i} score {ref_score[i]} vs k-th {kth} (tol {tol})"
    return len(diff)


def decode_one_layer(inp, cfg, depth_rule=0, fixed=(0, 0), budgets=None, residency="hbm", dev="cuda", flags=0,
                     lists=True, depths_in=None, basis=None, keep=None):
    """Prefill n-1 tokens of a generated layer, then one bpkv_decode_step (appends
    token n-1 and runs the whole path).  Returns (cache, depths, idx, out) with
    depths [N][H][D], idx [N][H][G][k], out [N][H][G][D] on the device; with
    lists=False the step writes no index lists (idx stays zero).  keep: a dict
    that receives the step's workspace ("ws")."""
    import bit_plane_kv_encode_gb300 as pk
    N, H, n, D = inp.k.shape
    G = cfg.group
    k_all, v_all = inp.k.to(dev), inp.v.to(dev)
    cache = build_cache(k_all, v_all, G, cap=cfg.cap_tokens, n_prefill=n - 1, residency=residency, basis=basis)
    ws = cache.workspace(cfg.k, pk.WS_STEP)
    out = torch.zeros((1, N, H, G, D), dtype=torch.float32, device=dev)
    depths = torch.zeros((1, N, H, D), dtype=torch.uint8, device=dev)
    idx = torch.zeros((1, N, H, G, cfg.k), dtype=torch.int32, device=dev)
    q = inp.q.to(dev)[None].contiguous()
    sigma2 = inp.sigma2.to(dev)[None].contiguous()
    b = inp.budgets if budgets is None else budgets
    budget_q = (4 * b).to(torch.int32).to(dev)
    k_new = k_all[:, :, n - 1][None].contiguous()
    v_new = v_all[:, :, n - 1][None].contiguous()
    a = pk.bpkv_step_args(k_new.data_ptr(), v_new.data_ptr(), q.data_ptr(), sigma2.data_ptr(), budget_q.data_ptr(),
                          depth_rule, fixed[0], fixed[1], cfg.k, cfg.n_sink, cfg.n_recent, out.data_ptr(),
                          depths.data_ptr(), idx.data_ptr() if lists else None, None, flags,
                          depths_in.data_ptr() if depths_in is not None else None)
    arr = pk.cache_array([cache])
    pk.bpkv_clear_status(ws)
    pk.bpkv_decode_step(arr, 1, a, ws, ws.numel())
    pk.sync_n_max([cache], arr)
    torch.cuda.synchronize()
    assert pk.bpkv_read_status(ws) == 0
    if keep is not None:
        keep["ws"] = ws
    return cache, depths[0], idx[0], out[0]


def check_unit(orc, cfg, inp, cache, depths, idx, out, s, h, depth_rule=0, fixed=(0, 0), budget_bits=None,
               what="", depth=None, basis=None):
    """Oracle decode of unit (s, h) vs the GPU results.  Every head's output is
    checked: against the oracle's own decode where the sets match exactly, and
    otherwise (a set that differs only on near-ties, as check_topk_sets
    allows) against the oracle's attention over the GPU's selected set.
    Returns (heads whose sets matched exactly, the oracle's decode)."""
    n = inp.k.shape[2]
    kb, vb = bits16(inp.k[s, h]), bits16(inp.v[s, h])
    b = int(inp.budgets[s]) if budget_bits is None else budget_bits
    ref = orc.decode_unit(kb, vb, inp.q[s, h].numpy(), inp.sigma2[s, h].numpy(), b, cfg.k, cfg.n_sink,
                          cfg.n_recent, nb_cap=cache.c.cap_tokens // 64,
                          fixed=fixed if depth_rule == 1 else None, depth=depth, basis=basis)
    nb = (n + 63) // 64
    assert np.array_equal(bits64(cache.planes[s, h])[:, :, :nb], ref["planes"][:, :, :nb]), f"{what} planes"
    assert np.array_equal(bits16(cache.scales[s, h])[:, :nb], ref["scales"][:, :nb]), f"{what} scales"
    assert np.array_equal(depths[s, h].cpu().numpy(), ref["depth"]), f"{what} depths"
    same = 0
    for g in range(cfg.group):
        gi = idx[s, h, g].cpu().numpy()
        d = check_topk_sets(gi, ref["idx"][g], ref["scores"][g], cfg.k, cfg.n_sink, cfg.n_recent,
                            what=f"{what} g{g}")
        want = ref["out"][g] if d == 0 else orc.attend(inp.q[s, h, g:g + 1].numpy(), kb, vb, gi[None])[0]
        err = float(np.max(np.abs(out[s, h, g].cpu().numpy() - want)))
        assert err <= ATTN_ATOL, f"{what} g{g} attention err {err} ({'same set' if d == 0 else f'{d} near-ties'})"
        same += d == 0
    return same, ref


def check_selection_map(pk, cfg, cache, idx, ws, n):
    """The range attention's selection map (bpkv_selection_map) holds exactly
    the middle tokens of the step's index lists on every row, bit for bit.
    Returns False (nothing checked) when the step took the cooperative cut,
    which writes no map."""
    import numpy as np
    try:
        smap = pk.bpkv_selection_map(cache.c, cfg.k, ws)
    except pk.BpkvError:
        return False
    idx = idx.cpu().numpy() if hasattr(idx, "cpu") else idx
    lo = min(cfg.n_sink, n)
    hi = max(n - cfg.n_recent, lo)
    bits = np.unpackbits(smap.view(np.uint8), bitorder="little").reshape(*smap.shape[:3], -1)
    N, H, G = smap.shape[:3]
    for s in range(N):
        for h in range(H):
            for g in range(G):
                want = set(int(x) for x in idx[s, h, g] if lo <= x < hi)
                if len(want) == hi - lo or not want:
                    continue  # every middle token or none: the map row is not written
                got = set(int(x) for x in np.nonzero(bits[s, h, g, lo:hi])[0] + lo)
                assert got == want, f"s{s} h{h} g{g}: map has {len(got)} middle tokens, lists {len(want)}"
    return True
