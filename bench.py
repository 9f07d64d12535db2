#!/usr/bin/env python3
"""Benchmark of the MoE FFN layer forward on GB300: tokens/s and fraction of roofline.

Default workload: the 2.4B+MoE-128 layer (d=3584, f=14336, E=128 experts, top-2 with
normalised gate weights, capacity factor 1.25, uniform routing) at T = 16384 tokens, fp16
weights and activations with fp32 accumulation, all expert weights (26.3 GB) resident in HBM:
the largest configured layer that one GPU holds.  A step is one moe_layer_forward call (gate,
dispatch, both expert GEMMs with fused GeLU and combine) on one of 4 seeded token batches,
cycled so routing changes from step to step; the expert weights alone exceed L2 (129 MB)
two hundred times over, so every step streams them from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (under torchrun): independent replicas, one per GPU (weak scaling); each rank times
its K steps between barriers, the slowest rank's time counts.  --impl reference times the
plain CPU oracle on the host cores on sub-batches of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/sec on 1 GB300 and % of roofline (tensor peak or HBM GB/s)"
UNIT = "tokens/s"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="moe2p4b_e128_top2")
    p.add_argument("--tokens", type=int, default=16384)
    p.add_argument("--experts", type=int, default=None,
                   help="override the workload's expert count (smaller profiling cases)")
    p.add_argument("--stack", default=None,
                   help="time a pyramid stack of layers (a name in synth.STACKS) under one CUDA "
                        "graph instead of one layer; --tokens tokens per step")
    p.add_argument("--capacity-factor", type=float, default=None,
                   help="override the workload's capacity factor; inf = dropless")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=20.0)
    p.add_argument("--no-graph", action="store_true",
                   help="launch each timed step directly instead of replaying its CUDA graph")
    return p.parse_args()


def bench_config(args):
    """The workload with the command line's overrides."""
    cfg, T = synth.workload(args.workload, args.tokens)
    if getattr(args, "experts", None):
        cfg = cfg.at(E=args.experts)
    if getattr(args, "capacity_factor", None) is not None:
        cfg = cfg.at(cf=args.capacity_factor)
    return cfg, T


MODEL_NAMES = {
    "moe350m_e128": "350M+MoE-128 layer, top-1",
    "moe1p3b_e128_zipf": "1.3B+MoE-128 layer, top-1, Zipf(1.1) routing",
    "prmoe_e64": "PR-MoE residual layer, E 64", "prmoe_e128": "PR-MoE residual layer, E 128",
    "top2_e64": "Top2-MoE at the PR-MoE shape, E 64", "top2_e128": "Top2-MoE at the PR-MoE shape, E 128",
    "moe2p4b_e128_top2": "2.4B+MoE-128 layer, top-2, uniform routing",
    "moe2p4b_e128_top2_zipf": "2.4B+MoE-128 layer, top-2, Zipf(1.2) routing",
}


def workload_name(cfg):
    """The workload as the JSON line names it: registry key and the model layer it is."""
    what = MODEL_NAMES.get(cfg.name)
    return f"{cfg.name}: {what}" if what else cfg.name


def cf_json(cf):
    """The capacity factor as a JSON value (\"inf\" for the dropless mode)."""
    return "inf" if math.isinf(cf) else cf


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------------ clocks sampler
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        inside = [s for t, s in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        if not inside:
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - (t0 + t1) / 2))[1]]
        sm = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in inside if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4)
                          if len(s) > 5 + i and s[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside)}


# ------------------------------------------------------------------------ CPU oracle timing
class OracleRunner:
    """The plain CPU oracle on contiguous sub-batches of the workload: each sub-batch is a full
    layer call of its own (gate, softmax/top-k, capacity dispatch, expert FFNs in double,
    combine).  Host weights are drawn once, outside any timing."""

    def __init__(self, cfg, T, seed):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.cfg, self.T = cfg, T
        dt = synth.F16 if cfg.dtype == "f16" else synth.F32
        self.x = synth.fill((T, cfg.d), dt, seed, synth.TID_TOKENS, cfg.tok_sigma)
        cs = synth.gate_col_scale(cfg, seed)
        self.Wg = synth.fill((cfg.d, cfg.E), synth.F32, seed, synth.TID_WG, cfg.w_sigma, col_scale=cs)
        self.w1, self.w2 = synth.expert_slices(cfg, range(cfg.E), seed)
        self.Wr1 = self.Wr2 = None
        if cfg.residual:
            self.Wr1 = synth.fill((cfg.d, cfg.f_res), dt, seed, synth.TID_WR1, cfg.w_sigma)
            self.Wr2 = synth.fill((cfg.f_res, cfg.d), dt, seed, synth.TID_WR2, cfg.w_sigma)
        self.cf = float(np.float32(cfg.cf))
        self.pos = 0

    def run(self, n):
        n = max(1, min(n, self.T))
        if self.pos + n > self.T:
            self.pos = 0
        x = self.x[self.pos:self.pos + n]
        self.pos += n
        t0 = time.perf_counter()
        self.oracle.layer_forward(x, self.Wg, self.w1, self.w2, self.cfg.k, self.cf, self.Wr1,
                                  self.Wr2)
        return time.perf_counter() - t0

    def size_for(self, seconds):
        """Sub-batch size that takes about `seconds` (calibrated on one small call)."""
        per_tok = self.run(8) / 8
        return max(1, min(self.T, int(seconds / per_tok)))

    def describe(self, n, steps):
        return (f"{steps} sub-batch(es) of {n} contiguous tokens from the T={self.T} batch, each "
                f"a full oracle layer call (own routing and capacity), host weights drawn untimed")


def cpu_model():
    """The host CPU's name as the kernel reports it (model name, else the Arm part number)."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        info = []
    for key in ("model name", "Model name", "CPU part"):
        for line in info:
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip() + ("" if key != "CPU part" else
                                                        f" (CPU part, {platform.machine()})")
    return platform.machine()


def oracle_tokens_per_s(cfg, T, seed, budget_s):
    """The oracle on all host cores (about 3/4 of the budget), then on one core (the rest)."""
    r = OracleRunner(cfg, T, seed)
    n = r.size_for(budget_s / 4)
    spent, done, steps = 0.0, 0, 0
    while spent < budget_s * 0.75 and steps < 64:
        spent += r.run(n)
        done += n
        steps += 1
    cores = r.oracle.num_threads()
    r.oracle.set_num_threads(1)
    try:
        n1 = r.size_for(budget_s / 8)
        one = r.run(n1)
    finally:
        r.oracle.set_num_threads(cores)
    extra = {"single_core_value": n1 / one, "single_core_sample": f"{n1} tokens, {one:.1f} s",
             "nproc": os.cpu_count(), "cpu_model": cpu_model()}
    return done / spent, cores, r.describe(n, steps) + f", {spent:.1f} s", extra


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg, T = bench_config(args)
    K, W = args.steps, args.warmup
    r = OracleRunner(cfg, T, args.seed)
    n = r.size_for(min(5.0, 150.0 / max(1, K + W)))
    for _ in range(W):
        r.run(n)
    t0 = time.perf_counter()
    busy = 0.0
    for _ in range(K):
        busy += r.run(n)
    elapsed = time.perf_counter() - t0
    rate = n * K / busy
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": K, "warmup": W, "ms_per_step": 1000.0 * elapsed / max(1, K),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(cfg), "T": T, "d": cfg.d, "f": cfg.f, "E": cfg.E,
                   "k": cfg.k, "capacity_factor": cf_json(cfg.cf)},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": r.oracle.num_threads(),
                         "kind": "oracle", "sample": r.describe(n, K)},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------ ranks
def max_over_ranks(values, dist, device):
    """Element-wise maximum of per-rank timings (the slowest rank defines the job's time)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tokens_per_s(world, T, K, ms):
    """Whole-job throughput: every rank processed K steps of T tokens in at most `ms`."""
    return world * T * K / (ms / 1000.0)


# ------------------------------------------------------------------------ GPU arm
def traffic_record(kernel_file):
    """Per-launch DRAM bytes from the committed ncu summary, if taken on this kernel source and
    this launch plan (the plan file chooses the kernel variant and its tiles)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    for key_file, key_sha in ((kernel_file, "kernel_sha256"),
                              (os.path.join(ROOT, rec.get("plan_file", "")), "plan_sha256")):
        if not os.path.isfile(key_file):
            return None
        if rec.get(key_sha) != hashlib.sha256(open(key_file, "rb").read()).hexdigest():
            return None
    return rec


def run_ours(args):
    import torch
    import torch.distributed as dist

    import sparse_expert_ffn_layer_gb300 as moe

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")

    cfg, T = bench_config(args)
    seed = args.seed + 1000 * rank
    f16 = cfg.dtype == "f16"
    tdt = torch.float16 if f16 else torch.float32
    n_batches = 4
    W1 = torch.empty((cfg.E, cfg.d, cfg.f), dtype=tdt, device="cuda")
    W2 = torch.empty((cfg.E, cfg.f, cfg.d), dtype=tdt, device="cuda")
    synth.fill_cuda(W1, seed, synth.TID_W1, cfg.w_sigma)
    synth.fill_cuda(W2, seed, synth.TID_W2, cfg.w_sigma)
    cs = synth.gate_col_scale(cfg, seed)
    Wg = torch.from_numpy(synth.fill((cfg.d, cfg.E), synth.F32, seed, synth.TID_WG, cfg.w_sigma,
                                     col_scale=cs)).cuda()
    Wr1 = Wr2 = None
    if cfg.residual:
        Wr1 = torch.empty((cfg.d, cfg.f_res), dtype=tdt, device="cuda")
        Wr2 = torch.empty((cfg.f_res, cfg.d), dtype=tdt, device="cuda")
        synth.fill_cuda(Wr1, seed, synth.TID_WR1, cfg.w_sigma)
        synth.fill_cuda(Wr2, seed, synth.TID_WR2, cfg.w_sigma)
    host_tok = [torch.from_numpy(synth.fill((T, cfg.d), synth.F16 if f16 else synth.F32, seed,
                                            synth.TID_TOKENS + (b << 8), cfg.tok_sigma)).pin_memory()
                for b in range(n_batches)]
    dev_tok = [h.cuda() for h in host_tok]
    out = torch.empty((T, cfg.d), dtype=tdt, device="cuda")
    host_out = torch.empty((T, cfg.d), dtype=tdt).pin_memory()
    mlp = moe.MOE_MLP_RESIDUAL if cfg.residual else moe.MOE_MLP_STANDARD
    ws = torch.empty(moe.moe_workspace_size(T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.cf, mlp, cfg.f_res,
                                            moe.MOE_F16 if f16 else moe.MOE_F32),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step(tok, idx=None, slot=None, dst=None):
        moe.moe_layer_forward(tok, Wg, W1, W2, cfg.k, cfg.cf, out if dst is None else dst, ws,
                              mlp_type=mlp, Wr1=Wr1, Wr2=Wr2, topk_idx_out=idx,
                              slot_of_out=slot)

    # routing statistics of each batch (for the algorithmic byte and FLOP counts)
    stats = []
    idx = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    slot = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    for b in range(n_batches):
        step(dev_tok[b], idx, slot)
        i_np, s_np = idx.cpu().numpy(), slot.cpu().numpy()
        kept_mask = s_np >= 0
        active = len(np.unique(i_np[kept_mask]))
        stats.append((active, int(kept_mask.sum())))
    if moe.moe_status_read(ws) != moe.MOE_OK:
        raise RuntimeError("device status not OK after the routing pass")
    A = float(np.mean([s[0] for s in stats]))
    S = float(np.mean([s[1] for s in stats]))

    for i in range(args.warmup):
        step(dev_tok[i % n_batches])
    torch.cuda.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_STAGE_EVENTS)]
           for _ in range(K)]
    for ev_step in evs:                  # torch creates the CUDA event at its first record
        for ev in ev_step:
            ev.record(stream)
    # Each timed step is one moe_layer_forward call.  By default the call is captured into a
    # CUDA graph per token batch and the graphs are replayed back to back, so the device
    # timing is not limited by host-side launch cost at small T.  The timed region carries
    # no stage events (each event record costs about a microsecond); a second pass of K
    # steps, each captured with its own stage events, times the stages and the dominant
    # kernel.
    cap_stream = torch.cuda.Stream()

    def capture(batch, events=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap_stream):
            if events is not None:
                moe.moe_set_stage_events(events)
            step(dev_tok[batch])
        moe.moe_set_stage_events(None)
        return g

    n0 = moe.moe_kernel_launches()
    plain = [] if args.no_graph else [capture(b) for b in range(n_batches)]
    # kernels per step: counted by the library at each launch while the graphs were captured
    kernels_per_step = (moe.moe_kernel_launches() - n0) // n_batches if plain else None
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(local)
    uuid = getattr(props, "uuid", None)
    gpu_id = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else uuid
    clocks = ClockSampler(gpu_id if gpu_id else str(local))
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0.record(stream)
    for i in range(K):
        if plain:
            plain[i % n_batches].replay()
        else:
            step(dev_tok[i % n_batches])
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    clocks.stop()
    status = moe.moe_status_read(ws)
    if status != moe.MOE_OK:
        raise RuntimeError(f"device status {moe.moe_status_string(status)}")
    ms = e0.elapsed_time(e1)

    # End to end through the public API with host buffers, right after the timed pass (the same
    # thermal and power state): every step copies its tokens from
    # pinned host memory to the device, runs the layer and copies its output back.  Two-deep
    # pipeline as a serving loop runs it: step i+1's tokens go in and step i's output comes out
    # on copy streams while step i+1 computes (double-buffered device input and output).
    h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dev_in = [torch.empty_like(dev_tok[0]) for _ in range(2)]
    dev_out = [torch.empty_like(out) for _ in range(2)]
    host_outs = [host_out, torch.empty_like(host_out).pin_memory()]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    # the layer call of each buffer pair, captured once (as a serving loop replays its graphs)
    e2e_graphs = []
    if not args.no_graph:
        for b in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap_stream):
                step(dev_in[b], dst=dev_out[b])
            e2e_graphs.append(g)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    h0.record(stream)
    h2d_s.wait_event(h0)
    d2h_s.wait_event(h0)
    with torch.cuda.stream(h2d_s):
        dev_in[0].copy_(host_tok[0], non_blocking=True)
        ev_in[0].record(h2d_s)
    for i in range(K):
        b, nb = i % 2, (i + 1) % 2
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])           # step i-2's output has left dev_out[b]
        if e2e_graphs:
            e2e_graphs[b].replay()
        else:
            step(dev_in[b], dst=dev_out[b])
        ev_comp[b].record(stream)
        if i + 1 < K:
            with torch.cuda.stream(h2d_s):
                if i >= 1:
                    h2d_s.wait_event(ev_comp[nb])  # step i-1 has read dev_in[nb]
                dev_in[nb].copy_(host_tok[(i + 1) % n_batches], non_blocking=True)
                ev_in[nb].record(h2d_s)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev_comp[b])
            host_outs[b].copy_(dev_out[b], non_blocking=True)
            ev_out[b].record(d2h_s)
    stream.wait_event(ev_out[(K - 1) % 2])
    if K > 1:
        stream.wait_event(ev_out[K % 2])
    h1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = h0.elapsed_time(h1)

    # decode sizes: the same steps with warm weights (one batch's graph replayed, so its
    # routed experts' weights stay in L2 from one step to the next), beside the cold number
    warm = None
    if plain and T <= 64 and world == 1:
        for _ in range(3):
            plain[0].replay()
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        for _ in range(K):
            plain[0].replay()
        w1.record(stream)
        torch.cuda.synchronize()
        wms = w0.elapsed_time(w1)
        warm = {"value": job_tokens_per_s(1, T, K, wms), "unit": UNIT, "ms_per_step": wms / K,
                "active_experts": stats[0][0],
                "mode": "one token batch replayed K times: its routed experts' weights stay in L2"}

    # stage pass: the same K steps, each with its own stage events
    if args.no_graph:
        for i in range(K):
            moe.moe_set_stage_events(evs[i])
            step(dev_tok[i % n_batches])
        moe.moe_set_stage_events(None)
        stage_source = "second pass of K direct calls with stage events"
    else:
        staged = [capture(i % n_batches, evs[i]) for i in range(K)]
        torch.cuda.synchronize()
        for g in staged:
            g.replay()
        stage_source = "second pass of K graph replays with stage events"
    torch.cuda.synchronize()
    stage_ms = np.zeros(moe.MOE_STAGE_EVENTS - 1)
    for i in range(K):
        for j in range(moe.MOE_STAGE_EVENTS - 1):
            stage_ms[j] += evs[i][j].elapsed_time(evs[i][j + 1])
    stage_ms /= K
    # spread of single steps (first to last stage event of each staged step; each includes
    # the event records, so it sits a little above the event-free mean)
    step_each = np.array([evs[i][0].elapsed_time(evs[i][-1]) for i in range(K)])
    step_pct = {f"p{q}": float(np.percentile(step_each, q)) for q in (10, 50, 90)}

    # the box's plain pinned copy rates for this step's buffers (one cudaMemcpyAsync per copy,
    # CUDA events on a copy stream), beside the end-to-end number they bound
    def copy_gbs(dst, src, reps=10):
        cs = torch.cuda.Stream()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(cs):
            dst.copy_(src, non_blocking=True)
            c0.record(cs)
            for _ in range(reps):
                dst.copy_(src, non_blocking=True)
            c1.record(cs)
        torch.cuda.synchronize()
        return reps * src.numel() * src.element_size() / (c0.elapsed_time(c1) / 1000.0) / 1e9

    h2d_gbs = copy_gbs(dev_in[0], host_tok[0])
    d2h_gbs = copy_gbs(host_outs[0], dev_out[0])

    if world > 1:
        ms, ms_e2e = max_over_ranks([ms, ms_e2e], dist, "cuda")
    if rank != 0:
        dist.destroy_process_group()
        return

    value = job_tokens_per_s(world, T, K, ms)
    value_e2e = job_tokens_per_s(world, T, K, ms_e2e)
    hbm, bf16, bf16_sus, peak_src = peaks()
    el = 2 if f16 else 4
    # algorithmic bytes per launch: the active experts' weights once, plus activations
    bytes_g1 = A * cfg.d * cfg.f * el + T * cfg.d * el
    bytes_g2 = A * cfg.f * cfg.d * el + T * cfg.d * el
    if cfg.residual:
        bytes_g1 += cfg.d * cfg.f_res * el
        bytes_g2 += cfg.f_res * cfg.d * el
    g1_ms, g2_ms = stage_ms[3], stage_ms[4]
    dom = "g1" if g1_ms >= g2_ms else "g2"
    dom_bytes, dom_ms = (bytes_g1, g1_ms) if dom == "g1" else (bytes_g2, g2_ms)
    achieved = dom_bytes / (dom_ms / 1000.0) / 1e9
    kernel_file = os.path.join(ROOT, "sparse_expert_ffn_layer_gb300", "csrc", "grouped_gemm.cu")
    trec = traffic_record(kernel_file)
    traffic = None
    if trec is not None and trec.get("workload") == f"{cfg.name}:T{T}":
        traffic = trec.get("per_launch_bytes", {}).get(dom)
    # whole-layer roofline
    layer_bytes = bytes_g1 + bytes_g2 + cfg.d * cfg.E * 4
    layer_flops = 4.0 * cfg.d * cfg.f * S + 2.0 * T * cfg.d * cfg.E + \
        (4.0 * T * cfg.d * cfg.f_res if cfg.residual else 0.0)
    t_roof = max(layer_bytes / (hbm * 1e9), layer_flops / (bf16 * 1e12))
    if kernels_per_step is None:         # direct launches: count one more step
        n0 = moe.moe_kernel_launches()
        step(dev_tok[0])
        torch.cuda.synchronize()
        kernels_per_step = moe.moe_kernel_launches() - n0
    launches_per_step = kernels_per_step

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16" if f16 else "f32",
        "data": "synthetic (seeded counter-based draws; 4 token batches cycled)",
        "config": {"workload": workload_name(cfg), "T": T, "d": cfg.d, "f": cfg.f, "E": cfg.E,
                   "k": cfg.k,
                   "capacity_factor": cf_json(cfg.cf),
                   "mlp_type": "residual" if cfg.residual else "standard",
                   "l2": f"inputs larger than L2: {2 * cfg.E * cfg.d * cfg.f * el / 1e9:.2f} GB of "
                         "expert weights per step vs 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "kernel": "grouped_gemm_kernel (expert GEMM1 + GeLU)" if dom == "g1"
                     else "grouped_gemm_kernel (expert GEMM2 + combine)",
                     "peak_source": peak_src},
        "layer_roofline": {"bound": "hbm" if layer_bytes / (hbm * 1e9) >= layer_flops / (bf16 * 1e12)
                           else "tensor", "roofline_ms": t_roof * 1000, "frac": t_roof * 1000 / (ms / K),
                           "bytes": layer_bytes, "flops": layer_flops},
        "stage_ms": {name: float(v) for name, v in zip(moe.STAGES, stage_ms)},
        "stage_ms_source": stage_source,
        "step_ms_staged": step_pct,
        "routing": {"active_experts": A, "kept_slots": S},
        "e2e": {"value": value_e2e, "unit": UNIT, "h2d_bytes_per_step": T * cfg.d * el,
                "d2h_bytes_per_step": T * cfg.d * el,
                "mode": "pinned host copies in and out every step, two-deep pipeline with compute"
                        + ("" if args.no_graph else "; the layer call of each buffer pair as a CUDA graph"),
                "copy_gbs": {"h2d": h2d_gbs, "d2h": d2h_gbs}},
        "gpu_launches": K * launches_per_step,
        "launch": "direct" if args.no_graph else "one CUDA graph per step, replayed back to back",
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    if warm is not None:
        line["warm_l2"] = warm
    if world == 1 and not args.no_cpu_baseline:
        rate, cores, desc, extra = oracle_tokens_per_s(cfg, T, seed, args.cpu_budget_s)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc, **extra}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_stack(args):
    """A pyramid stack of layers chained through device buffers, one CUDA graph per token
    batch covering every layer; value = tokens through the whole stack per second."""
    import torch

    import sparse_expert_ffn_layer_gb300 as moe

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    names = synth.STACKS[args.stack]
    cfgs = [synth.CONFIGS[n] for n in names]
    if args.capacity_factor is not None:
        cfgs = [c.at(cf=args.capacity_factor) for c in cfgs]
    T, d = args.tokens, cfgs[0].d
    assert all(c.d == d and c.dtype == "f16" for c in cfgs)
    layers = []
    for l, c in enumerate(cfgs):
        sd = synth.layer_seed(args.seed, l)
        L = {"W1": torch.empty((c.E, c.d, c.f), dtype=torch.float16, device="cuda"),
             "W2": torch.empty((c.E, c.f, c.d), dtype=torch.float16, device="cuda")}
        synth.fill_cuda(L["W1"], sd, synth.TID_W1, c.w_sigma)
        synth.fill_cuda(L["W2"], sd, synth.TID_W2, c.w_sigma)
        L["Wg"] = torch.from_numpy(synth.fill((c.d, c.E), synth.F32, sd, synth.TID_WG, c.w_sigma,
                                              col_scale=synth.gate_col_scale(c, sd))).cuda()
        L["Wr1"] = L["Wr2"] = None
        if c.residual:
            L["Wr1"] = torch.empty((c.d, c.f_res), dtype=torch.float16, device="cuda")
            L["Wr2"] = torch.empty((c.f_res, c.d), dtype=torch.float16, device="cuda")
            synth.fill_cuda(L["Wr1"], sd, synth.TID_WR1, c.w_sigma)
            synth.fill_cuda(L["Wr2"], sd, synth.TID_WR2, c.w_sigma)
        layers.append(L)
    n_batches = 4
    x = [torch.from_numpy(synth.fill((T, d), synth.F16, args.seed, synth.TID_TOKENS + (b << 8),
                                     1.0)).cuda() for b in range(n_batches)]
    bufs = [torch.empty((T, d), dtype=torch.float16, device="cuda") for _ in range(2)]
    ws = torch.empty(max(moe.moe_workspace_size(T, c.d, c.f, c.E, c.k, c.cf,
                                                1 if c.residual else 0, c.f_res, moe.MOE_F16)
                         for c in cfgs), dtype=torch.uint8, device="cuda")
    idx = [torch.empty((T, c.k), dtype=torch.int32, device="cuda") for c in cfgs]
    slot = [torch.empty((T, c.k), dtype=torch.int32, device="cuda") for c in cfgs]

    def run(b, events=None, stats=False):
        for l, c in enumerate(cfgs):
            L = layers[l]
            src = x[b] if l == 0 else bufs[(l - 1) % 2]
            if events is not None:
                moe.moe_set_stage_events(events[l])
            moe.moe_layer_forward(src, L["Wg"], L["W1"], L["W2"], c.k, c.cf, bufs[l % 2], ws,
                                  mlp_type=1 if c.residual else 0, Wr1=L["Wr1"], Wr2=L["Wr2"],
                                  topk_idx_out=idx[l] if stats else None,
                                  slot_of_out=slot[l] if stats else None)
        moe.moe_set_stage_events(None)

    # routing statistics per layer (active experts) for the algorithmic bytes
    active = np.zeros(len(cfgs))
    for b in range(n_batches):
        run(b, stats=True)
        for l in range(len(cfgs)):
            s_np, i_np = slot[l].cpu().numpy(), idx[l].cpu().numpy()
            active[l] += len(np.unique(i_np[s_np >= 0])) / n_batches
    if moe.moe_status_read(ws) != moe.MOE_OK:
        raise RuntimeError("device status not OK after the routing pass")
    cap = torch.cuda.Stream()
    n0 = moe.moe_kernel_launches()
    graphs = []
    for b in range(n_batches):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            run(b)
        graphs.append(g)
    kernels_per_step = (moe.moe_kernel_launches() - n0) // n_batches
    for i in range(max(3, args.warmup)):
        graphs[i % n_batches].replay()
    torch.cuda.synchronize()
    K = args.steps
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    uuid = getattr(props, "uuid", None)
    gpu_id = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else uuid
    clocks = ClockSampler(gpu_id if gpu_id else "0")
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0.record(stream)
    for i in range(K):
        graphs[i % n_batches].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    clocks.stop()
    if moe.moe_status_read(ws) != moe.MOE_OK:
        raise RuntimeError("device status not OK after the timed region")
    ms = e0.elapsed_time(e1) / K
    # per-layer times: replays of a graph carrying stage events around every layer
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_STAGE_EVENTS)]
           for _ in cfgs]
    for ev_l in evs:
        for ev in ev_l:
            ev.record(stream)
    torch.cuda.synchronize()
    gs = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gs, stream=cap):
        run(0, events=evs)
    reps = min(K, 20)
    layer_ms = np.zeros(len(cfgs))
    for _ in range(reps):
        gs.replay()
        torch.cuda.synchronize()
        layer_ms += [ev_l[0].elapsed_time(ev_l[-1]) for ev_l in evs]
    layer_ms /= reps
    hbm, bf16, _, peak_src = peaks()
    el = 2
    bytes_total = 0.0
    for l, c in enumerate(cfgs):
        bytes_total += active[l] * 2 * c.d * c.f * el + c.d * c.E * 4 + 2 * T * c.d * el
        if c.residual:
            bytes_total += 2 * c.d * c.f_res * el
    t_roof_ms = bytes_total / (hbm * 1e9) * 1e3
    line = {
        "metric": "PR-MoE stack tokens/sec on 1 GB300 (all layers per token) and % of HBM roofline",
        "value": T / (ms / 1000.0), "unit": UNIT, "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic (seeded counter-based draws; 4 token batches cycled)",
        "config": {"workload": args.stack, "layers": list(names), "T": T,
                   "capacity_factor": cf_json(cfgs[0].cf),
                   "l2": "inputs larger than L2: every layer's weights are distinct",
                   "parallelism": "single GPU"},
        "roofline": {"bound": "hbm", "achieved": bytes_total / (ms / 1000.0) / 1e9, "peak": hbm,
                     "unit": "GB/s", "frac": t_roof_ms / ms, "traffic": None,
                     "kernel": "whole stack (algorithmic bytes of every layer / step time)",
                     "peak_source": peak_src},
        "layer_ms": [float(v) for v in layer_ms],
        "active_experts": [float(v) for v in active],
        "gpu_launches": K * kernels_per_step,
        "launch": "one CUDA graph per step covering every layer, replayed back to back",
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.stack:
        run_stack(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
