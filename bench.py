#!/usr/bin/env python
"""Benchmark of the decode-time prefix-plane KV scan path on one GB300.

A step is one decode pass of one Qwen3-8B-shaped layer (8 KV heads x 4 query
heads, D = 128, batch 1, n = 32768 tokens, k = 512) at each of the budgets
68, 92 and 136 bits/token: for each budget, bpkv_decode_step appends the new
token (encode), allocates depths, scans the plane prefixes, selects top-k,
forms the GQA union and runs sparse attention.  The step is captured once in a
CUDA graph and replayed; the L2 cache is flushed (a 256 MiB write) before
every timed step, outside the timed events.

Metric: keys scored/s = (budgets x N x H x n) / step time.  The JSON line also
carries decode-step us per layer, per-stage times, the roofline of the
dominant kernel, the end-to-end number through host buffers, the CPU oracle
baseline and the clocks seen while timing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

STAGES = ["encode", "depths", "scan", "topk", "union", "attend"]
LAUNCHES_PER_PASS = {"encode": 2, "depths": 1, "scan": 1, "topk": 1, "union": 1, "attend": 2}
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="qwen3_8b_layer")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true")
    return p.parse_args()


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def all_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "of measured"
    except Exception:
        return FALLBACK_HBM_GBS, "of fallback"


class Clocks:
    """nvidia-smi samples (200 ms) taken while the timed loop runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ workload

def make_workload(cfg, steps: int, warmup: int, dev):
    import torch
    import bit_plane_kv_encode_gb300 as pk
    from workload import gen_layer

    inp = gen_layer(cfg, 0, device=dev)
    N, H, n, D = inp.k.shape
    G = cfg.group
    cap = ((n + warmup + steps + 64 + 511) // 512) * 512
    budgets = list(cfg.budgets)
    passes = []
    for b in budgets:
        c = pk.Cache(N, H, G, cap, device=dev)
        c.append(inp.k[:, :, : n - 1].contiguous(), inp.v[:, :, : n - 1].contiguous())
        passes.append(dict(budget=b, cache=c, cap=cap))
    torch.cuda.synchronize()
    ws = passes[0]["cache"].workspace(cfg.k, pk.WS_STEP)
    io = dict(
        q=inp.q.to(dev)[None].contiguous(),
        sigma2=inp.sigma2.to(dev)[None].contiguous(),
        k_new=inp.k[:, :, n - 1][None].contiguous(),
        v_new=inp.v[:, :, n - 1][None].contiguous(),
    )
    for p in passes:
        b = p["budget"]
        p["budget_q"] = torch.full((N,), 4 * b, dtype=torch.int32, device=dev)
        p["out"] = torch.zeros((1, N, H, G, D), dtype=torch.float32, device=dev)
        p["depths"] = torch.zeros((1, N, H, D), dtype=torch.uint8, device=dev)
        p["idx"] = torch.zeros((1, N, H, G, cfg.k), dtype=torch.int32, device=dev)
        p["events"] = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
        for e in p["events"]:
            e.record()  # create the event handles
        p["ev_arr"] = (__import__("ctypes").c_void_p * 7)(*[e.cuda_event for e in p["events"]])
        p["arr"] = pk.cache_array([p["cache"]])
        p["args"] = pk.bpkv_step_args(
            io["k_new"].data_ptr(), io["v_new"].data_ptr(), io["q"].data_ptr(), io["sigma2"].data_ptr(),
            p["budget_q"].data_ptr(), pk.DEPTH_WATERFILL, 0, 0, cfg.k, cfg.n_sink, cfg.n_recent,
            p["out"].data_ptr(), p["depths"].data_ptr(), p["idx"].data_ptr(),
            __import__("ctypes").cast(p["ev_arr"], __import__("ctypes").c_void_p))
    torch.cuda.synchronize()
    return inp, passes, ws, io


def run_step(passes, ws):
    import bit_plane_kv_encode_gb300 as pk
    for p in passes:
        # n_max is the launch-sizing bound: the capacity, so that graph replays stay
        # valid while the sequences grow by one token per replay
        p["arr"][0].n_max = p["cap"] - 1
        pk.bpkv_decode_step(p["arr"], 1, p["args"], ws, ws.numel())


def stage_times_ms(passes):
    out = {s: 0.0 for s in STAGES}
    for p in passes:
        ev = p["events"]
        for i, s in enumerate(STAGES):
            out[s] += ev[i].elapsed_time(ev[i + 1])
    return out


def bench_ours(args, cfg, rank, world, local):
    import torch
    import bit_plane_kv_encode_gb300 as pk
    from workload.bytes_model import depth_bits, row_bytes

    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    inp, passes, ws, io = make_workload(cfg, args.steps, args.warmup, dev)
    N, H, n, D = inp.k.shape
    G = cfg.group
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    graph = None
    stream = torch.cuda.Stream(device=dev)
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            run_step(passes, ws)

    def step():
        if graph is not None:
            graph.replay()
        else:
            run_step(passes, ws)

    pk.bpkv_clear_status(ws)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = pk.bpkv_read_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")

    clocks = Clocks(local)
    time.sleep(0.5)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ms, stage_ms = [], {s: [] for s in STAGES}
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()
        e0.record()
        step()
        e1.record()
        e1.synchronize()
        step_ms.append(e0.elapsed_time(e1))
        for s, v in stage_times_ms(passes).items():
            stage_ms[s].append(v)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    assert pk.bpkv_read_status(ws) == 0

    total_ms = all_max(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    keys_per_step = len(passes) * N * H * n
    value = world * keys_per_step / (ms_per_step / 1e3)

    # algorithmic bytes per pass (Fathom page, section 3.1 Eq. 1 terms)
    scan_bytes, rows_bytes, score_bytes = 0.0, 0.0, 0.0
    union_rows = 0
    for p in passes:
        dd = p["depths"][0].cpu().numpy()
        idx = p["idx"][0].cpu().numpy()
        for s in range(N):
            for h in range(H):
                scan_bytes += depth_bits(dd[s, h]) * n / 8
                u = len({int(i) for i in idx[s, h].ravel() if i >= 0})
                union_rows += u
                rows_bytes += u * row_bytes(D)
        score_bytes += N * H * G * n * 4
    stage_mean = {s: statistics.mean(v) for s, v in stage_ms.items()}
    stage_bytes = {"scan": scan_bytes, "topk": score_bytes, "attend": rows_bytes}
    dom = max(stage_bytes, key=lambda s: stage_mean[s])
    hbm, peak_src = peaks()
    achieved = stage_bytes[dom] / (stage_mean[dom] / 1e3) / 1e9
    traffic = load_traffic(dom)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "peak_source": peak_src,
                "traffic": traffic, "algorithmic_bytes_per_launch": round(stage_bytes[dom] / len(passes))}

    # end to end through host buffers: inputs copied in, outputs copied out, inside the timed region
    e2e = bench_e2e(args, passes, io, ws, flush, dev, keys_per_step, world)

    line = {
        "metric": "keys scored/s", "value": round(value), "unit": "keys/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; K ~ N(0, sigma_j^2), sigma_j = exp(0.75 z), 8 planted needles/head)",
        "config": {"workload": cfg.name, "n_seq": N, "n_kv_heads": H, "group": G, "head_dim": D,
                   "n_tokens": n, "budgets_bits": list(cfg.budgets), "k": cfg.k, "n_sink": cfg.n_sink,
                   "n_recent": cfg.n_recent, "residency": cfg.residency,
                   "l2": "flushed before every timed step (256 MiB write, outside the events)",
                   "cuda_graph": graph is not None, "parallelism": f"replicas x{world}"},
        "decode_step_us_per_layer": round(ms_per_step * 1e3 / len(passes), 2),
        "achieved_gbs_step": round((scan_bytes + rows_bytes) / (ms_per_step / 1e3) / 1e9, 1),
        "stages_us_per_step": {s: round(v * 1e3, 2) for s, v in stage_mean.items()},
        "bytes_per_step": {"scan": round(scan_bytes), "rows": round(rows_bytes), "scores_overhead": round(score_bytes),
                           "union_rows": union_rows},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": args.steps * len(passes) * sum(LAUNCHES_PER_PASS.values()),
        "clocks": clk,
        "wall_s_timed": round(wall, 3),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp, args.cpu_seconds)
    return line


def bench_e2e(args, passes, io, ws, flush, dev, keys_per_step, world):
    """Same step with its per-step inputs (q, new K/V row, sigma^2, budgets) copied
    from pinned host memory before it and every output copied back after it."""
    import torch
    host_in = {k: v.cpu().pin_memory() for k, v in io.items()}
    host_b = [p["budget_q"].cpu().pin_memory() for p in passes]
    host_out = [torch.empty(p["out"].shape, dtype=p["out"].dtype).pin_memory() for p in passes]
    bi = sum(t.numel() * t.element_size() for t in host_in.values()) + sum(t.numel() * 4 for t in host_b)
    bo = sum(t.numel() * t.element_size() for t in host_out)

    def step():
        for k, v in host_in.items():
            io[k].copy_(v, non_blocking=True)
        for p, hb in zip(passes, host_b):
            p["budget_q"].copy_(hb, non_blocking=True)
        run_step(passes, ws)
        for p, ho in zip(passes, host_out):
            ho.copy_(p["out"], non_blocking=True)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=torch.cuda.Stream(device=dev)):
        step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    n_e2e = max(3, min(args.steps, 50))
    for _ in range(n_e2e):
        flush.zero_()
        e0.record()
        graph.replay()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = all_max(statistics.mean(times), world)
    return {"value": round(world * keys_per_step / (ms / 1e3)), "unit": "keys/s", "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": round(ms, 5), "steps": n_e2e}


def load_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it still matches
    the kernel source it was taken from."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))[kernel]
    except Exception:
        return None
    src = os.path.join(ROOT, "bit_plane_kv_encode_gb300", "csrc", d["source"])
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return d["dram_bytes_per_launch"] if h == d.get("source_sha256_16") else None


# ------------------------------------------------------------------ CPU oracle

def _oracle_units(cfg, inp):
    """Per-unit oracle inputs (encoded once, outside any timing)."""
    import numpy as np
    import torch
    from oracle import Oracle
    o = Oracle()
    N, H, n, _ = inp.k.shape
    units = []
    kc, vc = inp.k.cpu(), inp.v.cpu()
    for s in range(N):
        for h in range(H):
            kb = kc[s, h].contiguous().view(torch.int16).numpy().view(np.uint16)
            vb = vc[s, h].contiguous().view(torch.int16).numpy().view(np.uint16)
            sc, pl = o.encode(kb, (n + 63) // 64)
            units.append((s, h, kb, vb, sc, pl))
    return o, units


def _oracle_step(o, cfg, inp, units, pool):
    """One decode step of the workload on the CPU oracle: per (budget, unit)
    re-encode of the tail block, depths, scores, top-k, union, attention."""
    import numpy as np
    n = inp.k.shape[2]

    def one(args):
        b, (s, h, kb, vb, sc, pl) = args
        tail = (n - 1) // 64 * 64
        sc_t, pl_t = o.encode(kb[tail:n], 1)
        q = inp.q[s, h].numpy()
        d = o.alloc_depths(q, inp.sigma2[s, h].numpy(), 4 * b)
        score = o.scores(n, sc, pl, d, q)
        idx = np.stack([o.topk(score[g], cfg.k, cfg.n_sink, cfg.n_recent) for g in range(q.shape[0])])
        o.union(idx)
        o.attend(q, kb, vb, idx)
        return sc_t.shape[0] + pl_t.shape[0]

    jobs = [(b, u) for b in cfg.budgets for u in units]
    list(pool.map(one, jobs))
    return len(jobs)


def cpu_baseline(cfg, inp, seconds: float) -> dict:
    import concurrent.futures as cf
    cores = os.cpu_count() or 1
    o, units = _oracle_units(cfg, inp)
    n = inp.k.shape[2]
    done, t0 = 0, time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        while True:
            done += _oracle_step(o, cfg, inp, units, pool)
            el = time.perf_counter() - t0
            if el >= seconds:
                break
    return {"value": round(done * n / el), "unit": "keys/s", "cores": cores, "kind": "oracle",
            "sample": f"{done // len(units) // len(cfg.budgets)} full steps of {cfg.name} "
                      f"({len(cfg.budgets)} budgets x {len(units)} (seq, KV head) units, n={n}), "
                      f"{el:.1f} s, threads over units"}


def bench_reference(args, cfg, rank, world):
    """The reference arm: the CPU oracle as it stands, timed on the host cores."""
    import concurrent.futures as cf
    from workload import gen_layer
    if rank != 0:
        return None
    inp = gen_layer(cfg, 0, device="cpu")
    o, units = _oracle_units(cfg, inp)
    n = inp.k.shape[2]
    cores = os.cpu_count() or 1
    times = []
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        for _ in range(args.warmup):
            _oracle_step(o, cfg, inp, units, pool)
        for _ in range(args.steps):
            t0 = time.perf_counter()
            _oracle_step(o, cfg, inp, units, pool)
            times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    keys = len(cfg.budgets) * len(units) * n
    val = round(keys / (ms / 1e3))
    return {"impl": "reference", "metric": "keys scored/s", "value": val, "unit": "keys/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "n_tokens": n, "budgets_bits": list(cfg.budgets), "k": cfg.k},
            "cpu_baseline": {"value": val, "unit": "keys/s", "cores": cores, "kind": "oracle",
                             "sample": f"every step is one full {cfg.name} step on the host cores"},
            "e2e": {"value": val, "unit": "keys/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    from workload import CONFIGS
    cfg = CONFIGS[args.workload]
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        line = bench_reference(args, cfg, rank, args.gpus)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    rank, world, local = dist_setup()
    line = bench_ours(args, cfg, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
