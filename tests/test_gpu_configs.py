"""Whole decode steps on the five workload shapes, through bpkv_decode_step in
the launch configuration the bench times, checked against the oracle on every
unit (small shapes) or on sampled (sequence, KV head) units (full sizes)."""
import numpy as np
import pytest
import torch

from gpu_helpers import check_selection_map, check_unit, decode_one_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    import __graft_entry__
    __graft_entry__.build()
    import bit_plane_kv_encode_gb300 as m
    return m


@pytest.mark.parametrize("k", [64, 100], ids=["k64_fixed_included", "k100_literal"])
def test_tiny_all_units(pk, orc, k):
    """The tiny layer at k = 64 (the 36 sink and recent tokens counted in k)
    and at the literal "64 per query head plus 4 sinks and 32 recent", k = 100."""
    import dataclasses
    from workload import CONFIGS, gen_layer
    cfg = dataclasses.replace(CONFIGS["tiny"], k=k)
    inp = gen_layer(cfg, 0, device="cpu")
    cache, d, idx, out = decode_one_layer(inp, cfg)
    same, _ = check_unit(orc, cfg, inp, cache, d, idx, out, 0, 0, what=f"tiny k{k}")
    assert same >= 3
    # 36 fixed tokens plus k - 36 chosen ones per head
    assert all(int((idx[0, 0, g] >= 0).sum()) == k for g in range(cfg.group))


@pytest.mark.parametrize("budget", [68, 92, 136])
def test_qwen3_layer_all_units(pk, orc, budget):
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS["qwen3_8b_layer"]
    inp = gen_layer(cfg, 0, device="cuda")
    inp.k, inp.v = inp.k.cpu(), inp.v.cpu()
    b = torch.full((cfg.n_seq,), budget, dtype=torch.int32)
    cache, d, idx, out = decode_one_layer(inp, cfg, budgets=b)
    same_total, found = 0, 0
    for h in range(cfg.n_kv_heads):
        same, _ = check_unit(orc, cfg, inp, cache, d, idx, out, 0, h, budget_bits=budget, what=f"b{budget} h{h}")
        same_total += same
        sel = set(idx[0, h].flatten().tolist())
        found += sum(int(p) in sel for p in inp.needles[0, h])
    assert same_total >= cfg.n_kv_heads * cfg.group // 2
    # quality, not parity: planted high |q.k| keys are found by some head of their KV head
    assert found >= 0.9 * inp.needles.numel()


@pytest.mark.parametrize("rule,fixed", [(1, (32, 4)), (1, (128, 2))])
def test_full_step_layer_fixed_sampled(pk, orc, rule, fixed):
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS["full_step"]
    inp = gen_layer(cfg, 5, device="cuda")
    cache, d, idx, out = decode_one_layer(inp, cfg, depth_rule=rule, fixed=fixed)
    inp.k, inp.v = inp.k.cpu(), inp.v.cpu()
    for (s, h) in [(0, 0), (3, 7)]:
        check_unit(orc, cfg, inp, cache, d, idx, out, s, h, depth_rule=rule, fixed=fixed, what=f"fixed{fixed}")


def test_full_step_layer_waterfill_sampled(pk, orc):
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS["full_step"]
    inp = gen_layer(cfg, 17, device="cuda")
    b = torch.tensor([32, 68, 104, 136], dtype=torch.int32)
    cache, d, idx, out = decode_one_layer(inp, cfg, budgets=b)
    inp.k, inp.v = inp.k.cpu(), inp.v.cpu()
    for (s, h) in [(0, 3), (1, 0), (2, 5), (3, 7)]:
        check_unit(orc, cfg, inp, cache, d, idx, out, s, h, budget_bits=int(b[s]), what=f"s{s}h{h}")


def test_multi_session_sampled(pk, orc):
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS["multi_session"]
    inp = gen_layer(cfg, 0, device="cuda")
    cache, d, idx, out = decode_one_layer(inp, cfg)
    inp.k, inp.v = inp.k.cpu(), inp.v.cpu()
    for (s, h) in [(0, 0), (7, 3), (19, 6), (31, 7)]:
        check_unit(orc, cfg, inp, cache, d, idx, out, s, h, what=f"s{s}h{h}")
    # every sequence's depth vectors respect its own budget
    from workload.bytes_model import depth_quarter_bits
    dd = d.cpu().numpy()
    for s in range(cfg.n_seq):
        for h in range(cfg.n_kv_heads):
            assert depth_quarter_bits(dd[s, h]) <= 4 * int(inp.budgets[s])


@pytest.mark.parametrize("wl,n_tok,rule,fixed,budget", [("qwen3_8b_layer", 32768, 0, (0, 0), 92),
                                                        ("full_step", 131072, 1, (32, 4), None),
                                                        ("multi_session", 65536, 0, (0, 0), None),
                                                        ("qwen3_8b_layer", 20000 + 13, 1, (1, 1), None),
                                                        ("tiny", 4096, 0, (0, 0), 0),
                                                        ("tiny", 37, 0, (0, 0), 136)])
def test_step_without_lists_matches(pk, wl, n_tok, rule, fixed, budget):
    """A step that writes no index lists (the attention reads only the selection
    cuts) gives bit-identical outputs to one that writes them."""
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS[wl]
    inp = gen_layer(cfg, 5, device="cuda", n_tokens=n_tok, n_seq=min(cfg.n_seq, 4))
    b = None if budget is None else torch.full((inp.k.shape[0],), budget, dtype=torch.int32)
    r_l = decode_one_layer(inp, cfg, depth_rule=rule, fixed=fixed, budgets=b, lists=True)
    r_n = decode_one_layer(inp, cfg, depth_rule=rule, fixed=fixed, budgets=b, lists=False)
    assert torch.equal(r_l[1], r_n[1])
    assert torch.equal(r_l[3], r_n[3])
    assert (r_n[2] == 0).all()  # no lists were written


@pytest.mark.parametrize("n_tok,k,fixed", [(20000 + 3, 512, (0, 4)), (20000 + 3, 36, (32, 4)), (5000, 37, (32, 4)),
                                           (200000 + 9, 512, (8, 1))])
def test_step_selection_edges(pk, orc, n_tok, k, fixed):
    """Decode steps whose selection is decided by the scan's candidates at the
    edges: every score equal (no channel read: ties all the way, the lowest
    indices win), no middle token kept (k = 36), one kept (k = 37), and rows
    longer than one scan CTA's part with few distinct score values."""
    import dataclasses
    from workload import CONFIGS, gen_layer
    cfg = dataclasses.replace(CONFIGS["qwen3_8b_layer"], k=k, n_tokens=n_tok)
    inp = gen_layer(cfg, 9, device="cuda", n_tokens=n_tok)
    keep = {}
    cache, d, idx, out = decode_one_layer(inp, cfg, depth_rule=1, fixed=fixed, keep=keep)
    # the long rows take the streaming cut; with few distinct scores their
    # buckets overflow the candidate buffer, so the rank refines them
    mapped = check_selection_map(pk, cfg, cache, idx, keep["ws"], n_tok)
    assert mapped == (n_tok > 100000)
    inp.k, inp.v = inp.k.cpu(), inp.v.cpu()
    for h in (0, 5):
        check_unit(orc, cfg, inp, cache, d, idx, out, 0, h, depth_rule=1, fixed=fixed, what=f"n{n_tok} k{k} h{h}")


@pytest.mark.parametrize("n_sink,n_recent,n_tok", [(5, 30, 70001), (0, 1, 65536 + 1023), (7, 0, 40000 + 3)])
def test_step_unaligned_sink_recent(pk, orc, n_sink, n_recent, n_tok):
    """Decode steps through the row buckets and the streaming cut (a grid
    larger than fits at once: 2 sequences x 8 KV heads x 4 heads) with sink
    and recent counts that are not multiples of 4, so the middle range starts
    and ends inside score groups and selection windows; every head of the
    sampled units is checked against the oracle."""
    import dataclasses
    from workload import CONFIGS, gen_layer
    cfg = dataclasses.replace(CONFIGS["multi_session"], n_seq=2, n_tokens=n_tok, n_sink=n_sink, n_recent=n_recent,
                              k=n_sink + n_recent + 200)
    inp = gen_layer(cfg, 0, device="cuda")
    cache, d, idx, out = decode_one_layer(inp, cfg)
    inp.k, inp.v = inp.k.cpu(), inp.v.cpu()
    for (s, h) in [(0, 0), (1, 5)]:
        check_unit(orc, cfg, inp, cache, d, idx, out, s, h, what=f"sink{n_sink} recent{n_recent} s{s}h{h}")


@pytest.mark.parametrize("n_sink,n_recent,n_tok,residency", [(4, 32, 70001, "hbm"), (5, 30, 65536 + 1023, "hbm"),
                                                             (0, 0, 40000 + 3, "hbm")])
def test_selection_map_matches_lists(pk, n_sink, n_recent, n_tok, residency):
    """The selection map the range attention reads (written by the streaming
    cut: the tokens above each row's bucket, then the bucket's chosen ones by
    the row's rank kernel) holds exactly the middle tokens of the step's own
    index lists, bit for bit, on every row (caches in pinned host memory:
    test_gpu_host.py)."""
    import dataclasses
    from workload import CONFIGS, gen_layer
    cfg = dataclasses.replace(CONFIGS["multi_session"], n_seq=2, n_tokens=n_tok, n_sink=n_sink, n_recent=n_recent,
                              k=n_sink + n_recent + 300)
    inp = gen_layer(cfg, 0, device="cuda")
    keep = {}
    cache, d, idx, out = decode_one_layer(inp, cfg, keep=keep, residency=residency)
    assert check_selection_map(pk, cfg, cache, idx, keep["ws"], n_tok)


def test_selection_map_cooperative_cut_unsupported(pk):
    """Small problems take the cooperative cut, which writes no map."""
    from workload import CONFIGS, gen_layer
    cfg = CONFIGS["tiny"]
    inp = gen_layer(cfg, 0, device="cpu")
    keep = {}
    cache, d, idx, out = decode_one_layer(inp, cfg, keep=keep)
    with pytest.raises(pk.BpkvError):
        pk.bpkv_selection_map(cache.c, cfg.k, keep["ws"])
