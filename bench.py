#!/usr/bin/env python
"""Throughput of the LiLiCorr draft-time rerank on GB300: draft blocks reranked per second.

Default workload: the high-concurrency shape (batch 256 blocks of B = 16 positions,
V = 151,936, K = 16, bf16 logits, medium-entropy tier, encoder 2 x hidden 256 / 4 heads /
FFN 1024, d_e 128), synthetic seeded inputs and random-init weights.

One step = one lilicorr_rerank call over the batch (logit pass, node build, encoder,
fusion/heads/scores, greedy walk) with inputs resident in HBM.  The logits (1,167 MB per
step) are larger than L2, so no flush is needed between steps.  The headline times the
step as a CUDA graph (the entry point allocates nothing and never synchronises, so one
call captures whole) replayed once per step; a separate eager pass with per-kernel
events gives the breakdown (`kernels`) and the launch count (`--no-graph` times the
eager pass instead).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Under torchrun every rank runs its own batch (blocks are independent: weak scaling, no
collective on the data path); rank 0 prints one JSON line.
"""
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

METRIC = "draft blocks reranked/sec at 1 GB300; logit-pass HBM GB/s as % of peak"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def describe(wl):
    d = wl.dims
    return (f"{wl.name}: batch {wl.batch}, B {wl.B}, V {wl.V}, K {wl.K}, {wl.ldtype} logits; "
            f"encoder {d['layers']} layers, hidden {d['hidden']}, {d['heads']} heads, "
            f"FFN {d['ffn']}, d_e {d['d_e']}")


# ------------------------------------------------------------------ clocks during timing

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l.strip().split(",") for l in open(self.path) if l.strip()]
        os.unlink(self.path)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle timing

def oracle_timing(workload, tier, blocks, steps=1, warmup=1, procs=0, batch=None):
    """The oracle in a fresh process (oracle/time_oracle.py): one thread (procs = 0) timing
    `steps` steps of `blocks` blocks, or `procs` one-thread processes with `blocks` blocks
    each.  BLAS / OpenMP threads are pinned to one, so the cores reported are the ones
    used."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    cmd = [sys.executable, "-m", "oracle.time_oracle", "--workload", workload,
           "--blocks", str(blocks), "--steps", str(steps), "--warmup", str(warmup)]
    if procs:
        cmd += ["--procs", str(procs)]
    else:
        cmd += ["--batch", str(batch or blocks * (steps + warmup))]
    if tier:
        cmd += ["--tier", tier]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle timing failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_baseline(workload, tier, one_blocks=2, one_steps=2, all_blocks=2):
    """The oracle on this host: one thread, and every core (one process per core)."""
    n = host_cores()
    one = oracle_timing(workload, tier, one_blocks, steps=one_steps, warmup=1)
    allc = oracle_timing(workload, tier, all_blocks, steps=all_blocks, procs=n)
    return {
        "value": allc["blocks_per_s"], "unit": "blocks/s", "cores": n, "kind": "oracle",
        "sample": (f"{allc['blocks']} blocks of {workload}{'/' + tier if tier else ''} "
                   f"({all_blocks} per process after one warm-up block, {n} one-thread "
                   f"processes, float64, full rows)"),
        "one_thread": {"value": one["blocks_per_s"], "unit": "blocks/s", "cores": 1,
                       "sample": f"{one_blocks} blocks x {one_steps} timed steps, 1 thread"},
    }


# ------------------------------------------------------------------ ncu traffic record

def recorded_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, only if the
    kernel's source is unchanged since the capture (sha256 recorded beside the figure)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        if line.lstrip().startswith("#"):
            continue
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("kernel") != kernel:
            continue
        src = os.path.join(ROOT, "draft_block_candidate_gb300", "csrc", f.get("source", ""))
        if not os.path.exists(src):
            return None
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if sha != f.get("src_sha"):
            return None
        return float(f["bytes_per_launch"])
    return None


# ------------------------------------------------------------------ arms

def run_reference(a):
    """The oracle as the reference arm, on every host core: one one-thread process per core,
    each step one block per process (cycling over two distinct blocks per process)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    n = host_cores()
    res = oracle_timing(a.workload, a.tier, 2, steps=a.steps, procs=n)
    v = res["blocks_per_s"]
    wlname = a.workload + (f"/{a.tier}" if a.tier else "")
    sample = (f"{n} blocks of {wlname} per step (one per host core, {n} one-thread "
              f"processes), {a.steps} steps over {res['distinct_blocks']} distinct blocks "
              f"after one warm-up block per process; float64, full rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "blocks/s",
        "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": res["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wlname, "sample": sample},
        "cpu_baseline": {"value": v, "unit": "blocks/s", "cores": n, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "blocks/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def rank_workload(name, tier, batch, rank):
    """This rank's blocks for a weak-scaling run: the model (weights) is the one every rank
    shares; the blocks are drawn from a seed of their own, so that N ranks process N
    different batches of the same workload."""
    from synth import make_workload
    from synth.inputs import CONFIGS
    if rank == 0:
        return make_workload(name, tier=tier, batch=batch)
    shared = make_workload(name, tier=tier, batch=1).weights
    return make_workload(name, tier=tier, batch=batch,
                         seed=CONFIGS[name]["seed"] + 7919 * rank, weights=shared)


def max_over_ranks(x, device):
    """The largest x over all ranks (x itself on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(batch_per_rank, steps, world, seconds):
    """Whole-job blocks/s: every rank's blocks over the slowest rank's time."""
    return batch_per_rank * steps * world / seconds


LM_D = 4096  # drafter hidden width of the vocabulary projection (the 8B target's width)


def time_lm_head(lc, rows, V, K, dev, stream, peak_tflops, calls=5, D=LM_D):
    """The vocabulary projection fused with the top-K / log-partition pass
    (lilicorr_lm_head_topk_lse) on `rows` drafter hidden states: random bf16 operands
    made on the device, CUDA-event time per call on the launching stream."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    h = torch.randn(rows, D, device=dev, generator=g).to(torch.bfloat16)
    w = (torch.randn(V, D, device=dev, generator=g) * (1.5 / D ** 0.5)).to(torch.bfloat16)
    out = lc.lm_head_topk_lse(h, w, K, stream=stream)
    ws = torch.empty(lc.lm_head_workspace_bytes(rows, V, D, K), dtype=torch.uint8, device=dev)
    for _ in range(3):
        lc.lm_head_topk_lse(h, w, K, workspace=ws, out=out, stream=stream)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(calls):
        lc.lm_head_topk_lse(h, w, K, workspace=ws, out=out, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) / calls * 1e3
    tflops = 2.0 * rows * V * D / (us * 1e-6) / 1e12
    del h, w, ws, out
    return {"rows": rows, "V": V, "D": D, "K": K, "us_per_call": us, "bound": "tensor",
            "achieved": tflops, "peak": peak_tflops, "unit": "TFLOP/s",
            "frac": tflops / peak_tflops, "calls": calls,
            "data": "synthetic: hidden N(0,1), vocabulary matrix N(0, 1.5^2/D), bf16, on device"}


# the per-workload sub-results the line carries beside the headline: every configuration
# of the synthetic workloads at its stated size (the high-concurrency medium tier is the
# headline itself)
SUBCONFIGS = [
    ("tiny", {}, "tiny"),
    ("single", {}, "config 1 (single request)"),
    *[("sweep", dict(batch=b), f"config 2 (sweep) batch {b}") for b in (1, 4, 16, 32, 64, 128)],
    ("highconc", dict(tier="low"), "config 3 (high concurrency) low tier"),
    ("highconc", dict(tier="high"), "config 3 (high concurrency) high tier"),
    ("widepool", {}, "config 4 (wide pool)"),
]
HEADLINE_LABEL = "config 3 (high concurrency) medium tier"


def gemm_work(wl, B, K):
    """Executed tensor work per launch of each contraction (split-bf16 operands double the
    contraction dimension) and of the attention."""
    import math
    H, F, E = wl.dims["hidden"], wl.dims["ffn"], wl.dims["d_e"]
    S = (B - 1) * K
    M = wl.batch * S
    fl = {"qkv_gemm": 2 * M * 3 * H * 2 * H, "out_gemm": 2 * M * H * 2 * H,
          "ffn1_gemm": 2 * M * F * 2 * H, "ffn2_gemm": 2 * M * H * 2 * F,
          "node_gemm": 2 * M * H * 2 * H, "fuse_gemm": 2 * M * H * 4 * H,
          "heads_gemm": 2 * M * 2 * E * 2 * H}
    # attention (128-query tiles over all keys): S = Q K^T as three split products,
    # O' = P [V_hi | V_lo] as two products of width 2 dh
    nh = wl.dims["heads"]
    dh = max(H // nh, 64)  # head dim 32 runs on zero-filled 64-wide tiles
    keys = 128 * math.ceil(S / 128)
    fl["attention"] = wl.batch * nh * math.ceil(S / 128) * (
        3 * 2 * 128 * keys * dh + 2 * 2 * 128 * keys * 2 * dh)
    return fl


def algorithmic_bytes(wl):
    """Bytes one call must move at least: the logits read once (rows 1..B-1 of every
    block), the gathered embedding rows, every weight once, the target state and the
    outputs (tokens, path scores)."""
    import numpy as np
    es = 2 if wl.ldtype == "bf16" else 4
    logits = wl.batch * (wl.B - 1) * wl.V * es
    H = wl.dims["hidden"]
    M = wl.batch * (wl.B - 1) * wl.K
    emb = M * H * wl.weights["embed"].dtype.itemsize
    weights = sum(int(np.asarray(v).nbytes) for v in wl.weights.values()
                  if v is not wl.weights["embed"])
    tgt = 0 if wl.target_state is None else int(wl.target_state.nbytes)
    outs = wl.batch * wl.B * 4 + wl.batch * (wl.B - 1) * 4
    return {"logits": logits, "embedding_rows": emb, "weights": weights,
            "target_state": tgt, "outputs": outs,
            "total": logits + emb + weights + tgt + outs}


def measure_workload(lc, wl, steps, warmup, dev, stream, graph=True, world=1, barrier=None):
    """Time lilicorr_rerank on workload `wl` (inputs resident on the device): an eager pass
    with per-kernel events (breakdown, launch count), then the headline timing, one CUDA
    graph of one call replayed per step (or the eager steps themselves)."""
    import numpy as np
    import torch
    barrier = barrier or (lambda: None)
    batch, B, V, K = wl.batch, wl.B, wl.V, wl.K
    if wl.ldtype == "bf16":
        logits = torch.from_numpy(wl.logits.view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        logits = torch.from_numpy(wl.logits).to(dev)
    tgt = torch.from_numpy(wl.target_state.view(np.int16)).view(torch.bfloat16).to(dev)
    anc = torch.from_numpy(wl.anchor_ids).to(dev)
    w = lc.Weights(wl.dims, wl.weights, device=dev.index or 0)
    ws = w.workspace(batch, B, K)
    out = {"tokens": torch.empty(batch, B, dtype=torch.int32, device=dev),
           "path_score": torch.empty(batch, B - 1, dtype=torch.float32, device=dev)}

    def step(st=stream):
        lc.rerank(w, logits, K, target_state=tgt, anchor_ids=anc, workspace=ws, out=out,
                  stream=st)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    lc.stage_timing(True)
    lc.stage_times()  # clear
    barrier()
    torch.cuda.synchronize(dev)
    n0 = lc.launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    launches_per_step = (lc.launch_count() - n0) / steps
    ms_eager = e0.elapsed_time(e1)
    lc.stage_timing(False)
    st = lc.stage_times()
    ms = ms_eager
    mode = "eager (one lilicorr_rerank per step)"
    if graph:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step(cap)
        torch.cuda.synchronize(dev)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        ms = e0.elapsed_time(e1)
        mode = "CUDA graph of one lilicorr_rerank, replayed per step"
        del g
    calls = st.pop("calls")
    per_kernel = {k: {"ms_per_step": v["ms"] / max(calls, 1),
                      "avg_launch_us": 1e3 * v["ms"] / max(v["launches"], 1),
                      "launches_per_step": v["launches"] / max(calls, 1)}
                  for k, v in st.items() if v["launches"]}
    res = {"ms": ms, "ms_eager": ms_eager, "mode": mode, "per_kernel": per_kernel,
           "launches_per_step": launches_per_step,
           "logit_bytes": batch * (B - 1) * V * (2 if wl.ldtype == "bf16" else 4),
           "inputs": (logits, tgt, anc), "weights": w, "out": out}
    return res


def summarise(wl, m, pk, steps, world=1):
    """The per-workload figures of one measurement."""
    step_ms = m["ms"] / steps
    k1 = m["per_kernel"]["logit_pass"]
    gbs = m["logit_bytes"] / (k1["avg_launch_us"] * 1e-6) / 1e9
    t_roof = m["logit_bytes"] / (pk["hbm_gbs"] * 1e9)
    dominant = max(m["per_kernel"], key=lambda k: m["per_kernel"][k]["ms_per_step"])
    fl = gemm_work(wl, wl.B, wl.K)
    enc = {k: fl[k] / (v["avg_launch_us"] * 1e-6) / 1e12
           for k, v in m["per_kernel"].items() if k in fl}
    return {
        "workload": describe(wl), "batch": wl.batch, "K": wl.K,
        "blocks_per_s": job_throughput(wl.batch, steps, world, m["ms"] / 1e3),
        "ms_per_step": step_ms, "eager_ms_per_step": m["ms_eager"] / steps,
        "launch": m["mode"],
        "logit_pass": {"avg_launch_us": k1["avg_launch_us"], "achieved_gbs": gbs,
                       "frac_of_peak": gbs / pk["hbm_gbs"], "bytes_per_launch": m["logit_bytes"]},
        "e2e_fraction_of_logits_roofline": t_roof / (step_ms / 1e3),
        "logits_roofline_us": t_roof * 1e6,
        "dominant_kernel": dominant,
        "kernels_us_per_step": {k: round(1e3 * v["ms_per_step"], 2)
                                for k, v in m["per_kernel"].items()},
        "tensor_tflops_executed": {k: round(v, 1) for k, v in enc.items()},
        "algorithmic_bytes": algorithmic_bytes(wl),
        "gpu_launches_per_step": m["launches_per_step"],
    }


def run_gb300(a):
    import numpy as np
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as lc

    # CPU baseline first (fresh, thread-pinned processes), rank 0 at N = 1 only.
    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = oracle_baseline(a.workload, a.tier, one_blocks=a.cpu_blocks)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    pk, pk_kind = peaks()
    stream = torch.cuda.current_stream(dev)
    wl = rank_workload(a.workload, a.tier, a.batch, rank)
    batch, B, V, K = wl.batch, wl.B, wl.V, wl.K
    clocks = ClockSampler(local)
    time.sleep(0.3)
    m = measure_workload(lc, wl, a.steps, a.warmup, dev, stream, graph=not a.no_graph,
                         world=world, barrier=barrier)
    clk = clocks.stop()
    ms = max_over_ranks(m["ms"], dev)
    value = job_throughput(batch, a.steps, world, ms / 1e3)
    launches = int(round(m["launches_per_step"] * a.steps))
    logits, tgt, anc = m["inputs"]
    w = m["weights"]

    # e2e through the host-memory entry point: H2D copies in, D2H tokens out, per step.
    e2e = None
    if not a.no_e2e:
        logits_host = logits.cpu()
        pin_logits = logits_host.pin_memory()
        pin_tgt = tgt.cpu().pin_memory()
        pin_anc = anc.cpu().pin_memory()
        tok_h = torch.empty(batch, B, dtype=torch.int32).pin_memory()
        ps_h = torch.empty(batch, B - 1, dtype=torch.float32).pin_memory()
        wsh = lc.rerank_host_workspace(w, batch, B, K, lc.BF16)
        for _ in range(2):
            lc.rerank_host(w, pin_logits, K, target_state=pin_tgt, anchor_ids=pin_anc,
                           tokens=tok_h, path_score=ps_h, workspace=wsh, stream=stream)
        barrier()
        t0 = time.perf_counter()
        for _ in range(a.e2e_steps):
            lc.rerank_host(w, pin_logits, K, target_state=pin_tgt, anchor_ids=pin_anc,
                           tokens=tok_h, path_score=ps_h, workspace=wsh, stream=stream)
        el = time.perf_counter() - t0
        barrier()
        el = max_over_ranks(el, dev)
        # the entry point copies rows 1..B-1 of each block (row 0 is never read)
        h2d = (pin_logits.numel() // B * (B - 1) * 2 + pin_tgt.numel() * 2 + pin_anc.numel() * 4)
        d2h = tok_h.numel() * 4 + ps_h.numel() * 4
        e2e = {"value": job_throughput(batch, a.e2e_steps, world, el), "unit": "blocks/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": a.e2e_steps,
               "api": "lilicorr_rerank_host (pinned host buffers; chunked copies overlapped "
                      "with compute)"}
        del wsh, pin_logits, logits_host
    del logits, tgt, anc, m["inputs"]
    w.close()
    torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    head = summarise(wl, m, pk, a.steps, world)
    per_kernel = m["per_kernel"]
    step_ms = ms / a.steps
    dominant = head["dominant_kernel"]
    k1 = per_kernel["logit_pass"]
    logit_bytes = m["logit_bytes"]
    k1_gbs = head["logit_pass"]["achieved_gbs"]
    logit_pass = {"achieved": k1_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                  "frac": k1_gbs / pk["hbm_gbs"], "bytes_per_launch": logit_bytes,
                  "avg_launch_us": k1["avg_launch_us"], "peak_kind": pk_kind}
    fl = gemm_work(wl, B, K)
    if dominant == "logit_pass":
        roof = {"bound": "hbm", "kernel": "logit_pass", "achieved": k1_gbs, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": k1_gbs / pk["hbm_gbs"],
                "traffic": recorded_traffic("logit_pass"), "peak_kind": pk_kind}
    elif dominant in fl:
        tf = fl[dominant] / (per_kernel[dominant]["avg_launch_us"] * 1e-6) / 1e12
        peak = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
        roof = {"bound": "tensor", "kernel": dominant, "achieved": tf, "peak": peak,
                "unit": "TFLOP/s", "frac": tf / peak, "traffic": recorded_traffic(dominant),
                "peak_kind": pk_kind + " sustained bf16"}
    else:
        roof = {"bound": "latency", "kernel": dominant, "achieved": None, "peak": None,
                "unit": None, "frac": None, "traffic": None}

    # every other configuration at its stated size (same launch form as the headline)
    configs = {}
    if world == 1 and not a.no_configs:
        for name, kw, label in SUBCONFIGS:
            sw = rank_workload(name, kw.get("tier"), kw.get("batch"), 0)
            sm = measure_workload(lc, sw, a.config_steps, 3, dev, stream, graph=not a.no_graph)
            sm["weights"].close()
            del sm["inputs"]
            torch.cuda.empty_cache()
            r = summarise(sw, sm, pk, a.config_steps)
            if not a.no_cpu_baseline:
                r["oracle"] = oracle_baseline(name, kw.get("tier"), one_blocks=1, one_steps=1,
                                              all_blocks=1)
            configs[label] = r
            del sw
        head_cfg = dict(head)
        if cpu is not None:
            head_cfg["oracle"] = cpu
        configs[HEADLINE_LABEL] = head_cfg

    lm = None
    if not a.no_lm_head:
        lm = time_lm_head(lc, batch * (B - 1), V, K, dev, stream, pk["bf16_tflops"])
    line = {
        "metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": describe(wl), "batch_per_gpu": batch, "B": B, "V": V, "K": K,
                   "l2": f"inputs larger than L2 ({logit_bytes / 1e6:.0f} MB of logits per step); no flush",
                   "parallelism": f"dp{world} (independent blocks per rank)",
                   "launch": m["mode"]},
        "roofline": roof,
        "logit_pass": logit_pass,
        "e2e_fraction_of_logits_roofline": head["e2e_fraction_of_logits_roofline"],
        "gpu_launches": launches,
        "eager_ms_per_step": m["ms_eager"] / a.steps,
        "kernels": per_kernel,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clk,
        "lm_head_topk_lse": lm,
        "configs": configs,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_lm_head_only(a):
    """lilicorr_lm_head_topk_lse alone on the workload's drafted rows (a small --batch or
    --lm-v keeps an ncu capture short); CUDA-event timing on the launching stream."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as lc
    from synth.inputs import CONFIGS
    cfg = CONFIGS[a.workload]
    batch = a.batch or cfg["batch"]
    V = a.lm_v or cfg["V"]
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    pk, _ = peaks()
    r = time_lm_head(lc, batch * (cfg["B"] - 1), V, cfg["K"], dev, torch.cuda.current_stream(dev),
                     pk["bf16_tflops"], calls=a.steps)
    print(json.dumps({"kernel": "lm_head_topk", **r}), flush=True)


def run_logit_pass_only(a):
    """lilicorr_topk_lse alone on the workload's logits (a small --batch keeps an ncu
    capture short); CUDA-event timing on the launching stream."""
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as lc
    from synth import make_workload

    wl = make_workload(a.workload, tier=a.tier, batch=a.batch)
    x = torch.from_numpy(wl.logits.view(np.int16)).view(torch.bfloat16).cuda()
    ws = lc.topk_lse_workspace(wl.batch, wl.B, wl.V, wl.K, lc.BF16, x.device)
    out = lc.topk_lse(x, wl.K, workspace=ws)
    for _ in range(a.warmup):
        lc.topk_lse(x, wl.K, workspace=ws, out=out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.steps):
        lc.topk_lse(x, wl.K, workspace=ws, out=out)
    e1.record()
    torch.cuda.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / a.steps
    nbytes = wl.batch * (wl.B - 1) * wl.V * 2
    pk, kind = peaks()
    print(json.dumps({"kernel": "logit_pass", "workload": describe(wl), "avg_launch_us": us,
                      "GB/s": nbytes / us / 1e3, "frac_of_peak": nbytes / us / 1e3 / pk["hbm_gbs"],
                      "peak_kind": kind, "bytes_per_launch": nbytes}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="highconc")
    ap.add_argument("--tier", default="medium")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-blocks", type=int, default=2,
                    help="blocks per timed step of the one-thread oracle leg")
    ap.add_argument("--config-steps", type=int, default=20,
                    help="timed steps of each per-configuration sub-result")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration sub-results")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-lm-head", action="store_true",
                    help="skip the fused vocabulary projection + top-K / LSE measurement")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of a replayed CUDA graph")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch")
    ap.add_argument("--only", default=None, choices=["logit_pass", "lm_head"],
                    help="time one kernel alone (profiling driver); prints its own JSON")
    ap.add_argument("--lm-v", type=int, default=None,
                    help="vocabulary size of --only lm_head (default: the workload's V)")
    a = ap.parse_args()
    if a.workload != "highconc":
        a.tier = None
    if a.warmup < 3:
        a.warmup = 3
    if a.impl == "reference":
        run_reference(a)
    elif a.only == "logit_pass":
        run_logit_pass_only(a)
    elif a.only == "lm_head":
        run_lm_head_only(a)
    else:
        run_gb300(a)


if __name__ == "__main__":
    main()
