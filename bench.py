#!/usr/bin/env python
"""Benchmark of one DFlash2 draft + select + verify step on GB300.

`python bench.py --gpus N --steps K --warmup W` prints one JSON line.

A step = dflash2_draft_block + dflash2_select + dflash2_verify over one batch of
seeded synthetic inputs of the drafter's full geometry (default workload:
5 layers, width 5120, 32/8 heads, FFN 17408, vocab 248320, BF16 weights,
1 request, context 1024, greedy).  The timed region is one CUDA-graph launch of
exactly K steps, bracketed by a barrier and device synchronisation; inputs are
resident in HBM and far larger than L2 (6.1 GB of weights stream every step).

`value` is steps/s summed over ranks (independent replicas, weak scaling).
`e2e` is the same metric through the C ABI with host buffers: every step copies
its inputs from pinned host memory, runs as one dflash2_step call (the handle's
CUDA graph of the step) and reads its result back; the inputs go on a second
stream into one of two buffer sets, overlapping the previous step.  `roofline`
covers the LM-head + top-16 kernel, timed with CUDA events captured inside the
graph on the launching stream; `roofline.projections` covers the drafter's weight
projections (every other weight stream), each launch bracketed by events in a
separate graph.  Fractions are given against the measured copy bandwidth and
against the nominal 8 TB/s.  `cpu_baseline` times the oracle on the host.

The default line also carries the metric's other operating points, each measured
in the same process (`--no-r16` skips them): `r16`, 16 requests (configuration 5:
Q8 weights, ragged contexts 512..32768, mixed temperatures), its 100 consecutive
steps with the emitted tokens appended between steps, captured as one graph;
`q8_r1` (configuration 3: Q8, one request, context 2048, T = 1.0) and `r4`
(configuration 4: Q8, four requests, context 8192, T = 0.7), 100 steps each; and
`tree`: the draft-tree variant of the default workload (draft block + tree of 12
nodes + greedy tree verification), 100 steps.

`--impl reference` times the CPU oracle (the only reference this method has
here) on the same workload and prints the same line with "impl": "reference".
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "DFlash2 draft+verify steps/s at 1 and 16 req; achieved HBM GB/s vs peak"


# DRAM bytes (read + write) of one LM-head launch, keyed by (vocabulary, width,
# requests): dram__bytes_read.sum + dram__bytes_write.sum of lmhead_kernel in a
# one-pass ncu capture of the full-size one-request workload (the launch-list capture
# of this benchmark's own command).  Valid for the current lmhead_kernel; re-capture
# when the kernel changes.
LMHEAD_TRAFFIC = {(248320, 5120, 1): 2.54e9 + 2.87e6}
TRAFFIC_SOURCE = "ncu dram__bytes_read.sum + dram__bytes_write.sum of lmhead_kernel, full-size 1-request capture"
NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s quoted for GB300 HBM3e, beside the measured copy rate


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", type=int, default=2)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=100)
    p.add_argument("--no-r16", action="store_true",
                   help="skip the other operating points (configurations 5, 3 and 4) that ride along the default line")
    return p.parse_args(argv)


def max_over_ranks(x: float, world: int) -> float:
    """The largest of each rank's value (a time: the job takes as long as its slowest
    replica).  Works on a process group of either backend (nccl: a device tensor)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sync_ranks(world: int) -> None:
    """Barrier across the replicas (no-op for one rank)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_rate(units_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: every rank processed units_per_rank units, the job took
    the slowest rank's time (weak scaling: per-rank work fixed as ranks grow)."""
    return world * units_per_rank / (ms_max / 1e3)


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:  # noqa: BLE001
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "fallback": True}


def step_bytes(wl, n_req):
    """Algorithmic bytes of one step: every weight streamed once (codebooks: only the
    gathered rows), visible K/V read, new K/V written, taps and target rows read."""
    g = wl.geom
    H, F, V = g.hidden, g.ffn, g.vocab
    mats = (g.q_dim * H + 2 * g.kv_dim * H + H * g.q_dim + 3 * F * H + 2 * g.delta_dim * H)
    per_weight = 2.0 if wl.weight_format == "bf16" else 68.0 / 64.0
    w = (mats * g.n_layers + H * g.n_taps * H + g.rank * H) * per_weight
    w += V * H * 2                                           # LM head (BF16 in both formats)
    P = g.block - 1                                          # proposals per request
    w += (1 + (P - 1) * 16 + P * 16) * g.rank * per_weight * n_req  # codebook rows gathered
    kv_key = 2 * g.kv_dim * 2 * g.n_layers                   # K and V, BF16, all layers
    kv = sum(min(c, g.window - 1) for c in wl.ctx[:n_req]) * kv_key + g.block * n_req * kv_key
    taps = n_req * g.block * g.n_taps * H * 4
    target = n_req * g.block * V * 4
    return w + kv + taps + target


class Clocks:
    """nvidia-smi samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index):
        self.dev = dev_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"dflash2_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:  # noqa: BLE001
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        rows = [l.split(", ") for l in open(self.path).read().strip().splitlines() if l.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def cpu_baseline(wl, W, inp, kc_host, vc_host, target_np):
    """The oracle, as it stands, on one full step of request 0 (bounded: one step)."""
    import oracle
    g = wl.geom
    cores = len(os.sched_getaffinity(0))
    t0 = time.perf_counter()
    kl = [kc_host[l, 0].copy() for l in range(g.n_layers)]
    vl = [vc_host[l, 0].copy() for l in range(g.n_layers)]
    res = oracle.step(g, W, int(inp["anchors"][0]), int(inp["ctx_len"][0]), int(inp["n_new"][0]),
                      inp["taps"][0][: int(inp["n_new"][0])], kl, vl, wl.temps[0], wl.philox_seed, 0,
                      lambda lg: target_np[0].astype(np.float64))
    dt = time.perf_counter() - t0
    return {"value": 1.0 / dt, "unit": "steps/s", "cores": cores, "kind": "oracle",
            "sample": f"1 full step of request 0 of {wl.name} (FP64 NumPy, {dt:.1f} s)"}, res


def setup(wl, device_index):
    """Weights, caches, inputs and target rows of a workload on the device."""
    import torch
    import block_drafter_pos_gb300 as bd
    import workloads as wk

    g = wl.geom
    t0 = time.time()
    W = wk.make_weights(g, wl.weight_format, wl.seed)
    inp = wk.make_request_inputs(wl)
    R, cap = wl.n_req, wl.kv_capacity
    kc = np.zeros((g.n_layers, R, cap, g.n_kv_heads, g.head_dim), np.uint16)
    vc = np.zeros_like(kc)
    for l in range(g.n_layers):
        for r in range(R):
            K, V = inp["kv"][l][r]
            lo = int(inp["kv_lo"][r])
            kc[l, r, lo:lo + len(K)] = K
            vc[l, r, lo:lo + len(V)] = V
    drafter = bd.Drafter(g, wl.weight_format, W, R, cap)
    dev = torch.device("cuda", device_index)
    B, P = g.block, g.block - 1
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    S = {
        "anchors": T(inp["anchors"]), "ctx_len": T(inp["ctx_len"]), "n_new": T(inp["n_new"]),
        "taps": T(inp["taps"]), "kc": T(kc.view(np.int16)), "vc": T(vc.view(np.int16)),
        "cand_ids": torch.zeros((R, P, 16), dtype=torch.int32, device=dev),
        "cand_logits": torch.zeros((R, P, 16), dtype=torch.float32, device=dev),
        "gate": torch.zeros((R, P, g.rank), dtype=torch.float32, device=dev),
        "logits": torch.zeros((R, P, g.vocab), dtype=torch.float32, device=dev),
        "temps": T(np.array(wl.temps, np.float32)),
        "seeds": T(np.full(R, wl.philox_seed, np.uint64).view(np.int64)),
        "offsets": T(np.array(wl.philox_offsets or [0] * R, np.uint64).view(np.int64)),
        "path": torch.zeros((R, P), dtype=torch.int32, device=dev),
        "q_rows": torch.zeros((R, P, 16), dtype=torch.float32, device=dev),
        "status": torch.zeros((R,), dtype=torch.int32, device=dev),
        "n_acc": torch.zeros((R,), dtype=torch.int32, device=dev),
        "emitted": torch.zeros((R, B), dtype=torch.int32, device=dev),
        "n_emit": torch.zeros((R,), dtype=torch.int32, device=dev),
    }
    # untimed pass: drafter logits -> synthetic target rows = drafter logits + N(0, sigma)
    bd.dflash2_draft_block(drafter.handle, R, S["anchors"], S["ctx_len"], S["n_new"], S["taps"], S["kc"], S["vc"],
                           S["cand_ids"], S["cand_logits"], S["gate"], S["logits"])
    torch.cuda.synchronize()
    lg = S["logits"]
    target = torch.empty((R, B, g.vocab), dtype=torch.float32, device=dev)
    for r in range(R):
        noise = torch.from_numpy(wk.make_target_noise(wl, 0, r)).to(dev)
        target[r, :P] = lg[r] + noise[:P]
        target[r, P] = lg[r, P - 1] + noise[P]
    S["target"] = target
    setup_s = time.time() - t0
    return drafter, S, W, inp, kc, vc, setup_s


def run_step(bd, h, R, S, ev=None):
    bd.dflash2_draft_block(h, R, S["anchors"], S["ctx_len"], S["n_new"], S["taps"], S["kc"], S["vc"], S["cand_ids"],
                           S["cand_logits"], S["gate"], None)
    bd.dflash2_select(h, R, S["anchors"], S["cand_ids"], S["cand_logits"], S["gate"], S["temps"], S["seeds"],
                      S["offsets"], S["path"], S["q_rows"], None, S["status"])
    bd.dflash2_verify(h, R, S["target"], S["path"], S["cand_ids"], S["q_rows"], S["temps"], S["seeds"], S["offsets"],
                      S["n_acc"], S["emitted"], S["n_emit"], None, S["status"])


def measure_point(args, world, local_rank, cfg):
    """One more operating point of the metric, measured in the same process: a
    workload's step captured as one CUDA graph after W eager warm-up steps.  A
    workload of consecutive steps (configuration 5: 16 Q8 requests, ragged contexts,
    mixed temperatures) runs its 100 steps, each draft + select + verify followed by
    the device-side state update (dflash2_advance: the emitted tokens become the next
    step's anchor and new context rows), the initial state restored before each
    replay; the others run 100 repetitions of their step.  Max over ranks."""
    import torch
    import block_drafter_pos_gb300 as bd
    import workloads as wk

    wl = wk.workload(cfg)
    R = wl.n_req
    drafter, S, _, _, _, _, setup_s = setup(wl, local_rank)
    h = drafter.handle
    loop = wl.steps > 1
    K = wl.steps if loop else 100

    def one_step():
        run_step(bd, h, R, S)
        if loop:
            bd.dflash2_advance(h, R, S["emitted"], S["n_emit"], S["anchors"], S["ctx_len"], S["n_new"], S["offsets"])

    state0 = {k: S[k].clone() for k in ("anchors", "ctx_len", "n_new", "offsets")}

    def restore():
        for k, v in state0.items():
            S[k].copy_(v)

    for _ in range(max(3, args.warmup)):
        one_step()
    torch.cuda.synchronize()
    restore()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev:
        a.record()
        b.record()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.current_stream()
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(graph, stream=cap_stream):
            for i in range(K):
                bd.dflash2_set_lmhead_events(h, ev[i][0], ev[i][1])
                one_step()
    bd.dflash2_set_lmhead_events(h, None, None)
    stream.wait_stream(cap_stream)
    restore()
    graph.replay()
    torch.cuda.synchronize()
    restore()
    torch.cuda.synchronize()
    sync_ranks(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    graph.replay()
    t1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), world)
    st = S["status"].cpu().numpy()
    assert np.all(st == 0), st
    lm_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    pk = peaks()
    sb = step_bytes(wl, R)
    step_s = ms / 1e3 / K
    lm_bytes = bd.dflash2_lmhead_bytes(h, R)
    wide = R * wl.geom.block >= (40 if wl.weight_format == "bf16" else 32)
    out = {"workload": wl.name, "block": wl.geom.block, "requests_per_gpu": R, "context": wl.ctx[:R] if R <= 4 else "U[512, 32768]",
           "weights": wl.weight_format, "temperature": wl.temps[:R] if R <= 4 else "round-robin 0, 0.7, 1.0",
           "steps": K, "value": job_rate(K, world, ms), "unit": "steps/s", "ms_per_step": ms / K,
           "drafted_tokens_per_s": job_rate(K, world, ms) * (wl.geom.block - 1) * R,
           "step_bytes": sb, "step_gbs": sb / step_s / 1e9, "step_hbm_frac": sb / step_s / 1e9 / pk["hbm_gbs"],
           "step_frac_vs_8tbs": sb / step_s / 1e9 / NOMINAL_HBM_GBS,
           "lmhead": {"kernel": ("wide_kernel<0> (LM head, tcgen05 GEMM) + logits_topk_kernel" if wide
                                 else "lmhead_kernel (LM head GEMV + fused top-16)"), "launch_ms": lm_ms,
                      "achieved_gbs": lm_bytes / (lm_ms / 1e3) / 1e9,
                      "frac": lm_bytes / (lm_ms / 1e3) / 1e9 / pk["hbm_gbs"]},
           "setup_s": setup_s}
    if loop:
        grown = int((S["ctx_len"] - state0["ctx_len"]).sum().item())  # context rows appended over the K steps
        out["loop"] = f"{K} consecutive steps with the emitted tokens appended ({grown} context rows over all requests)"
    del graph, drafter, S
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def measure_tree(bd, h, R, S, wl, budget=12, steps=100):
    """The draft-tree variant of the step on the same workload (the pages' DDTree,
    budget 12): draft block + tree build + greedy tree verification against
    budget + 1 target rows per request (the root's and each node's), captured as one
    graph of `steps` steps.  The rows are the drafter's logits of the node's next
    block position plus N(0, sigma) noise, built once from an untimed tree."""
    import torch
    g = wl.geom
    dev = S["anchors"].device
    z = lambda shape, dt=torch.int32: torch.zeros(shape, dtype=dt, device=dev)
    T = {"token": z((R, budget)), "parent": z((R, budget)), "depth": z((R, budget)),
         "score": z((R, budget), torch.float32), "n": z((R,)), "status": z((R,)), "n_acc": z((R,)),
         "emitted": z((R, 8)), "n_emit": z((R,))}

    def build():
        bd.dflash2_draft_block(h, R, S["anchors"], S["ctx_len"], S["n_new"], S["taps"], S["kc"], S["vc"],
                               S["cand_ids"], S["cand_logits"], S["gate"], None)
        bd.dflash2_tree_build(h, R, budget, S["anchors"], S["cand_ids"], S["cand_logits"], S["gate"], T["token"],
                              T["parent"], T["depth"], T["score"], T["n"], None, T["status"])

    build()
    torch.cuda.synchronize()
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed + 7)
    rows = torch.empty((R, budget + 1, g.vocab), dtype=torch.float32, device=dev)
    dep = T["depth"].clamp(1, 7) - 1
    for r in range(R):
        rows[r, 0] = S["logits"][r, 0]
        rows[r, 1:] = S["logits"][r, torch.clamp(dep[r] + 1, max=6).long()]
        rows[r] += torch.randn((budget + 1, g.vocab), generator=gen, device=dev) * wl.sigma[r]

    def one():
        build()
        bd.dflash2_tree_verify(h, R, budget, rows, T["token"], T["parent"], T["n"], T["n_acc"], T["emitted"],
                               T["n_emit"], T["status"])

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.current_stream()
    cs = torch.cuda.Stream()
    cs.wait_stream(stream)
    with torch.cuda.stream(cs):
        with torch.cuda.graph(graph, stream=cs):
            for _ in range(steps):
                one()
    stream.wait_stream(cs)
    graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    graph.replay()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    assert int(T["status"].abs().sum().item()) == 0
    del graph
    return {"workload": wl.name, "budget": budget, "steps": steps, "value": 1e3 / ms, "unit": "steps/s",
            "ms_per_step": ms, "nodes_per_step": int(T["n"].sum().item()),
            "emitted_per_step": float(T["n_emit"].float().mean().item()),
            "timing": "draft block + tree build + greedy tree verify, one CUDA graph; target rows resident"}


def measure_projections(bd, h, one_step, restore, n_launch, proj_bytes, steps=10):
    """Roofline of the drafter's weight projections (the GEMV / tensor-core GEMM family,
    every projection launch of the step but the LM head): a separate graph of `steps`
    steps whose projection launches are each bracketed by CUDA events on the launching
    stream.  An event record between launches removes their dependent-launch overlap,
    so this is the family's rate launch by launch, not inside the timed step (whose
    graph carries no such events)."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * n_launch)] for _ in range(steps)]
    for row in evs:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.current_stream()
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(graph, stream=cap_stream):
            for i in range(steps):
                bd.dflash2_set_projection_events(h, evs[i])
                one_step()
    bd.dflash2_set_projection_events(h, None)
    stream.wait_stream(cap_stream)
    restore()
    graph.replay()
    torch.cuda.synchronize()
    restore()
    graph.replay()
    torch.cuda.synchronize()
    per_step = [sum(row[2 * j].elapsed_time(row[2 * j + 1]) for j in range(n_launch)) for row in evs]
    ms = statistics.median(per_step)
    pk = peaks()
    gbs = proj_bytes / (ms / 1e3) / 1e9
    del graph
    return {"kernels": "gemv_kernel (bulk-copy pipeline + mma.sync) / wide_kernel (tcgen05)", "launches": n_launch,
            "bytes": proj_bytes, "ms": ms, "achieved": gbs, "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
            "frac_vs_8tbs": gbs / NOMINAL_HBM_GBS,
            "timing": f"each launch bracketed by events in a separate graph of {steps} steps (median step); "
                      "launch by launch, without the dependent-launch overlap of the timed step"}


def main_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import block_drafter_pos_gb300 as bd
    import workloads as wk

    torch.cuda.set_device(local_rank)
    bd.build()
    wl = wk.workload(args.config)
    R = wl.n_req
    drafter, S, W, inp, kc_host, vc_host, setup_s = setup(wl, local_rank)
    h = drafter.handle
    K, Wm = args.steps, args.warmup
    stream = torch.cuda.current_stream()
    # a workload of consecutive steps (configuration 5) appends each step's emitted
    # tokens before the next (dflash2_advance); its initial state is restored before
    # every replay
    loop = wl.steps > 1
    if loop:
        K = min(K, wl.steps)
    state0 = {k: S[k].clone() for k in ("anchors", "ctx_len", "n_new", "offsets")}

    def restore():
        for k, v in state0.items():
            S[k].copy_(v)

    def one_step():
        run_step(bd, h, R, S)
        if loop:
            bd.dflash2_advance(h, R, S["emitted"], S["n_emit"], S["anchors"], S["ctx_len"], S["n_new"], S["offsets"])

    # warm-up (eager), then count launches of one step
    for _ in range(Wm):
        one_step()
    torch.cuda.synchronize()
    n0 = bd.dflash2_launch_count(h)
    one_step()
    launches_per_step = bd.dflash2_launch_count(h) - n0
    torch.cuda.synchronize()
    restore()
    # one CUDA graph of exactly K steps, with the LM-head kernel bracketed by events
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev:  # torch creates the CUDA events on first record; the graph re-records them
        a.record()
        b.record()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(graph, stream=cap_stream):
            for i in range(K):
                bd.dflash2_set_lmhead_events(h, ev[i][0], ev[i][1])
                one_step()
    bd.dflash2_set_lmhead_events(h, None, None)
    stream.wait_stream(cap_stream)
    restore()
    graph.replay()  # warm replay (graph upload)
    torch.cuda.synchronize()
    restore()
    torch.cuda.synchronize()
    clocks = Clocks(local_rank)
    clocks.start()
    time.sleep(0.15)
    sync_ranks(world)
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record()
    graph.replay()
    t_end.record()
    torch.cuda.synchronize()
    sync_ranks(world)
    clk = clocks.stop()
    ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    lm_ms = [a.elapsed_time(b) for a, b in ev]
    steps_per_s = job_rate(K, world, ms)
    # sanity of the timed outputs
    st = S["status"].cpu().numpy()
    ne = S["n_emit"].cpu().numpy()
    assert np.all(st == 0) and np.all(ne >= 1), (st, ne)
    restore()

    # end to end through the C ABI with host buffers
    E = args.e2e_steps
    pin = lambda t: t.cpu().pin_memory()
    host_in = {k: pin(S[k]) for k in ("anchors", "ctx_len", "n_new", "taps", "temps", "seeds", "offsets", "target")}
    host_out = {k: torch.empty_like(S[k], device="cpu").pin_memory() for k in ("emitted", "n_emit", "n_acc")}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())

    # One call per step: dflash2_step replays the handle's CUDA graph of the step's
    # argument set (captured on its first call).  A step's inputs go into one of two
    # sets of device buffers on a side stream, once the step two steps back (the last
    # to read that set) has verified, so the copies of step i overlap step i - 1; the
    # step waits for its copies.  Two buffer sets, two argument sets, two graphs.
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    dev_in = [{k: S[k] for k in host_in}, {k: torch.empty_like(S[k]) for k in host_in}]
    verified = [torch.cuda.Event(), torch.cuda.Event()]
    landed = [torch.cuda.Event(), torch.cuda.Event()]
    n_e2e = [0]

    def e2e_step():
        j = n_e2e[0] % 2
        n_e2e[0] += 1
        D = dev_in[j]
        side.wait_event(verified[j])
        with torch.cuda.stream(side):
            for k, v in host_in.items():
                D[k].copy_(v, non_blocking=True)
        landed[j].record(side)
        main.wait_event(landed[j])
        bd.dflash2_step(h, R, D["anchors"], D["ctx_len"], D["n_new"], D["taps"], S["kc"], S["vc"], S["cand_ids"],
                        S["cand_logits"], S["gate"], D["temps"], D["seeds"], D["offsets"], S["path"], S["q_rows"],
                        S["status"], D["target"], S["n_acc"], S["emitted"], S["n_emit"])
        verified[j].record(main)
        for k, v in host_out.items():
            v.copy_(S[k], non_blocking=True)

    for ev in verified:
        ev.record(main)
    for _ in range(4):  # both argument sets: first calls (capture), then replays
        e2e_step()
    torch.cuda.synchronize()
    sync_ranks(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for ev in verified:
        ev.record(main)  # no copy of the timed steps starts before the timed region
    for _ in range(E):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_val = job_rate(E, world, e2e_ms)

    proj = measure_projections(bd, h, one_step, restore, bd.dflash2_projection_launches(h),
                               bd.dflash2_projection_bytes(h))
    restore()
    tree = None
    if args.config == 2 and not args.no_r16:
        tree = measure_tree(bd, h, R, S, wl)
        restore()
    pk = peaks()
    lm_bytes = bd.dflash2_lmhead_bytes(h, R)
    lm_avg_s = statistics.mean(lm_ms) / 1e3
    achieved = lm_bytes / lm_avg_s / 1e9
    sb = step_bytes(wl, R)
    step_s = ms / 1e3 / K
    line = {
        "metric": METRIC, "value": steps_per_s, "unit": "steps/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.weight_format == "bf16" else "q8g64xf16",
        "data": "synthetic (seeded, drafter geometry; random weights, no checkpoint)",
        "config": {"workload": wl.name, "requests_per_gpu": R, "context": wl.ctx[:R], "weights": wl.weight_format,
                   "temperature": wl.temps[:R], "l2": "inputs larger than L2 (weights stream every step)",
                   "parallelism": f"{world} independent replica(s)",
                   "timing": ("one CUDA graph of K consecutive steps, emitted tokens appended between steps" if loop
                              else "one CUDA graph of K steps")},
        "drafted_tokens_per_s": steps_per_s * 7 * R,
        "step_bytes": sb, "step_gbs": sb / step_s / 1e9, "step_hbm_frac": sb / step_s / 1e9 / pk["hbm_gbs"],
        "step_frac_vs_8tbs": sb / step_s / 1e9 / NOMINAL_HBM_GBS,
        "roofline": {"kernel": ("lmhead_kernel (LM head GEMV + fused top-16)" if R < (5 if wl.weight_format == "bf16" else 4) else
                                "wide_kernel<0> (LM head, tcgen05 GEMM) + logits_topk_kernel"), "bound": "hbm",
                     "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                     "frac_vs_8tbs": achieved / NOMINAL_HBM_GBS,
                     "traffic": LMHEAD_TRAFFIC.get((wl.geom.vocab, wl.geom.hidden, R)),
                     "traffic_source": TRAFFIC_SOURCE if (wl.geom.vocab, wl.geom.hidden, R) in LMHEAD_TRAFFIC else None,
                     "launch_ms": statistics.mean(lm_ms), "share_of_step": statistics.mean(lm_ms) / (ms / K),
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)",
                     "projections": proj},
        "e2e": {"value": e2e_val, "unit": "steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        **({"tree": tree} if tree is not None else {}),
        "gpu_launches": int(launches_per_step * K),
        "clocks": clk,
        "setup_s": setup_s,
    }
    if args.config == 2 and not args.no_r16:
        # the metric's other operating points: 16 requests (configuration 5), the Q8
        # one-request and four-request workloads (configurations 3 and 4), and the
        # one-request workload with blocks of 16
        del graph
        torch.cuda.synchronize()
        line["r16"] = measure_point(args, world, local_rank, 5)
        line["q8_r1"] = measure_point(args, world, local_rank, 3)
        line["r4"] = measure_point(args, world, local_rank, 4)
        line["block16"] = measure_point(args, world, local_rank, 9)
    if rank == 0 and not args.no_cpu_baseline:
        cb, _ = cpu_baseline(wl, W, inp, kc_host, vc_host, S["target"].cpu().numpy())
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)


def main_reference(args, rank, world):
    """The oracle, as it stands, on host cores: each step one full oracle step of request 0."""
    if rank != 0:
        return
    import workloads as wk
    import oracle

    wl = wk.workload(args.config)
    g = wl.geom
    W = wk.make_weights(g, wl.weight_format, wl.seed)
    inp = wk.make_request_inputs(wl)
    cap = wl.kv_capacity
    kc = np.zeros((g.n_layers, 1, cap, g.n_kv_heads, g.head_dim), np.uint16)
    vc = np.zeros_like(kc)
    for l in range(g.n_layers):
        K, V = inp["kv"][l][0]
        lo = int(inp["kv_lo"][0])
        kc[l, 0, lo:lo + len(K)] = K
        vc[l, 0, lo:lo + len(V)] = V
    noise = wk.make_target_noise(wl, 0, 0).astype(np.float64)

    def tfn(lg):
        z = np.concatenate([lg, lg[6:7]], 0)
        return z + noise

    def one():
        kl = [kc[l, 0].copy() for l in range(g.n_layers)]
        vl = [vc[l, 0].copy() for l in range(g.n_layers)]
        oracle.step(g, W, int(inp["anchors"][0]), int(inp["ctx_len"][0]), 8, inp["taps"][0], kl, vl, wl.temps[0],
                    wl.philox_seed, 0, tfn)

    steps = max(1, min(args.steps, 3))
    warm = min(args.warmup, 1)
    for _ in range(warm):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    dt = time.perf_counter() - t0
    v = steps / dt
    cores = len(os.sched_getaffinity(0))
    sample = f"{steps} full oracle step(s) of request 0 of {wl.name} after {warm} warm-up (FP64 NumPy)"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": world, "steps": steps,
            "warmup": warm, "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "requests_per_gpu": wl.n_req, "context": wl.ctx, "weights": wl.weight_format},
            "cpu_baseline": {"value": v, "unit": "steps/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        main_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl")
    main_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
