#!/usr/bin/env python
"""Constrained decode throughput (filter + score + select) on one GB300.

One step = one full L-step constrained beam decode of one request batch,
all kernels of the CUDA library (index lookup, gather-add, selective or full
projection, masked log-softmax, cumulative add, top-K select, emit), replayed
from a CUDA graph with inputs resident in HBM and L2 flushed (a 256 MiB
write) before every timed step.  Default workload: the large catalogue
(L=4, V=8192, 100M items with Zipf(1.05) first tokens and geometric fan-out
decay, d=512, bf16 weights, batch 64, beam 256, top-K 256), the largest
configuration; its batch sweep (1, 8, 32, 64) is reported beside the line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl zerogr|reference]

Under torchrun (N > 1) every rank decodes its own request batch against a
replicated index (independent replicas, no collective on the data path);
the time is the max over ranks.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload.
"""
from __future__ import annotations

import os

# the CPU oracle is timed per process (one a core); keep numpy's BLAS single-threaded
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import dataclasses
import hashlib
import json
import math
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "constrained decode requests/s (filter+score+select)"
UNIT = "requests/s"
L2_FLUSH_BYTES = 256 << 20


def workload_desc(cfg) -> str:
    return (f"{cfg.name}: L={cfg.L}, V={cfg.V}, {cfg.n_items:,} items ({cfg.catalogue}), d={cfg.d}, "
            f"{cfg.w_dtype} W, batch {cfg.batch}, beam {cfg.beam}, top-K {cfg.topk}")


# ---------------------------------------------------------------- distributed helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def request_seed(rank: int) -> int:
    """Each replica decodes its own batch (weak scaling)."""
    return 1000 + rank


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 7]
        os.unlink(self.f.name)
        sm = [float(r[0]) for r in rows if r[0].strip().replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- roofline accounting

def step_bytes(st: dict, cfg, s: int) -> int:
    """Algorithmic bytes of step s (1-based) of the filtering-first decode,
    one unit = one (live beam, legal slot) pair plus the per-beam terms:
    the beam's index row (rowptr pair and its column entries, or its bitmap
    row), the C_{s-1} row of its gather-add (s >= 2), one W_s row per
    (beam, legal slot), and W (score, slot) survivor pairs per beam; the last
    step adds the outputs B*K*(4L+4).  Re-reads of a weight row by other beams
    are counted (most are L2 hits), so this is the work the method moves
    through the memory system, not its HBM traffic."""
    e = 4 if cfg.w_dtype == "f32" else 2
    n = st["live_beams"]
    b = st["index_bytes"]
    b += n * cfg.d * 4 if s >= 2 else 0
    b += st["legal_slots"] * cfg.d * e
    b += n * cfg.beam * 8
    if s == cfg.L:
        b += cfg.batch * cfg.topk * (4 * cfg.L + 4)
    return int(b)


def step_unique_bytes(st: dict, cfg, s: int) -> int:
    """Lower bound on the HBM bytes of step s with a cold L2: the index rows,
    each distinct legal weight row once, the C rows, survivors."""
    e = 4 if cfg.w_dtype == "f32" else 2
    n = st["live_beams"]
    b = st["index_bytes"] + st["unique_tokens"] * cfg.d * e
    b += n * cfg.d * 4 if s >= 2 else 0
    b += n * cfg.beam * 8
    return int(b)


def full_flops(st: dict, cfg, s: int) -> int:
    n = cfg.batch * (1 if s == 1 else cfg.beam)
    return 2 * n * cfg.V * cfg.d


def kernel_source_hash() -> str:
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "generative_recommendation_constrained_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def launches_per_decode(variants, s0: int, L: int, w_dtype: str) -> int:
    """Kernels one decode launches: a stand-alone selective step three (chunk
    counting, scoring, select); a full step its gather-add (steps >= 2), the
    hidden split (half-precision weights), the projection and the select; a
    naive step its gather-add (steps >= 2), four compaction kernels, the dot
    products and the select; the fused steps from s0 on one launch."""
    n = 0
    for s, v in enumerate(variants[:s0 - 1]):
        if v == 0:
            n += 3
        elif v == 1:
            n += (1 if s >= 1 else 0) + (1 if w_dtype != "f32" else 0) + 2
        else:
            n += (1 if s >= 1 else 0) + 6
    return n + (1 if s0 <= L else 0)


def ncu_entry(kernel: str, cfg_name: str):
    """The committed ncu summary of a kernel on a workload, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except ValueError:
        return None
    ent = d.get(f"{cfg_name}:{kernel}")
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent


def ncu_traffic(kernel: str, cfg_name: str):
    """DRAM bytes per launch from a committed ncu summary (None when absent or stale)."""
    ent = ncu_entry(kernel, cfg_name)
    return ent.get("dram_bytes_per_launch") if ent else None


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "src": "fallback"}


# ---------------------------------------------------------------- CPU oracle leg

_ORACLE_CTX = {}


def host_cpu_model() -> str:
    """The host CPU's model name (/proc/cpuinfo, else lscpu, else platform)."""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_requests(wid: int, n_workers: int, budget_s: float):
    """Decode requests wid, wid + n_workers, ... of the batch one at a time
    until budget_s elapses; returns (requests decoded, seconds)."""
    import oracle
    c = _ORACLE_CTX
    B = c["u"].shape[0]
    done = 0
    t0 = time.perf_counter()
    while True:
        q = (wid + done * n_workers) % B
        oracle.decode(c["trie"], c["model"], c["u"][q:q + 1], c["beam"], c["topk"])
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return done, time.perf_counter() - t0


def _oracle_batch(sel):
    """Decode the requests `sel` one at a time; returns seconds."""
    import oracle
    c = _ORACLE_CTX
    t0 = time.perf_counter()
    for q in sel:
        oracle.decode(c["trie"], c["model"], c["u"][q:q + 1], c["beam"], c["topk"])
    return time.perf_counter() - t0


def oracle_setup(cfg, sids, model, u):
    """Build the oracle's trie once (timed) and keep what the workers read.
    Worker pools are forked from this process, so this and the pools must run
    before the first CUDA call of the process."""
    import oracle
    t0 = time.perf_counter()
    trie = oracle.Trie(sids, cfg.L, cfg.V)
    _ORACLE_CTX.update(trie=trie, model=model, u=u, beam=cfg.beam, topk=cfg.topk)
    return time.perf_counter() - t0


def oracle_rates(cfg, sids, model, u, budget_s: float) -> dict:
    """Requests/s of the CPU oracle as it stands (fp64 numpy, requests decoded
    one at a time): on one host thread, then on every host core (one forked
    worker process per core, requests dealt round-robin, each worker decoding
    for budget_s).  Must run before the first CUDA call of the process."""
    import multiprocessing as mp
    t_trie = oracle_setup(cfg, sids, model, u)
    _oracle_requests(0, 1, 0.0)          # warms the trie's lookups of the first step
    done1, dt1 = _oracle_requests(0, 1, budget_s)
    cores = os.cpu_count() or 1
    with mp.get_context("fork").Pool(cores) as pool:
        res = pool.starmap(_oracle_requests, [(w, cores, budget_s) for w in range(cores)])
    rate_all = sum(d / t for d, t in res)
    done_all = sum(d for d, _ in res)
    return {"value": rate_all, "unit": UNIT, "cores": cores, "kind": "oracle",
            "cpu_model": host_cpu_model(), "one_thread": done1 / dt1,
            "sample": f"requests of the workload decoded one at a time for {budget_s:.0f} s: {done1} on 1 thread, "
                      f"{done_all} on {cores} worker processes (one a core); trie build {t_trie:.1f} s excluded; "
                      f"fp64 numpy oracle"}


def run_reference(args, cfg):
    """The oracle (this method exists only as web pages of text; there is no
    installable reference implementation) timed as it stands on every host
    core: each step decodes four requests per core (the requests of the batch
    in turn, at most the batch), handed one at a time to whichever of the
    forked worker processes (one a core) is free, so that the step measures
    the oracle's throughput rather than its slowest request."""
    import multiprocessing as mp
    rank, world, _ = dist_env()
    if rank != 0:
        return
    sids = synth.make_catalogue(cfg, 0)
    model = synth.make_model(cfg.L, cfg.V, cfg.d, cfg.w_dtype, 0)
    u = synth.make_requests(cfg.batch, cfg.d, request_seed(0))
    t_trie = oracle_setup(cfg, sids, model, u)
    _oracle_batch([0])  # warms the trie's first-step lookups once; the forked workers inherit them
    cores = os.cpu_count() or 1
    per_step = max(1, min(cfg.batch, args.ref_requests or 4 * cores))
    times = []
    with mp.get_context("fork").Pool(cores) as pool:
        def step(i):
            lo = (i * per_step) % cfg.batch
            sel = (np.arange(lo, lo + per_step) % cfg.batch).tolist()
            t0 = time.perf_counter()
            pool.map(_oracle_batch, [[q] for q in sel], chunksize=1)
            return time.perf_counter() - t0
        for i in range(args.warmup):
            step(i)
        for i in range(args.steps):
            times.append(step(i))
    ms = 1000.0 * sum(times) / len(times)
    val = per_step / (ms / 1000.0)
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "global_batch": cfg.batch, "beam": cfg.beam, "topk": cfg.topk,
                   "sample": f"each step decodes {per_step} requests of the batch (bounded CPU sample)"},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": host_cpu_model(),
                         "sample": f"{per_step} requests per step x {args.steps} steps on {cores} worker processes, "
                                   f"fp64 numpy oracle; trie build {t_trie:.1f} s excluded"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU leg

def run_gpu(args, cfg):
    import torch
    rank, world, local = dist_env()
    sids = synth.make_catalogue(cfg, 0)
    model = synth.make_model(cfg.L, cfg.V, cfg.d, cfg.w_dtype, 0)
    u = synth.make_requests(cfg.batch, cfg.d, request_seed(rank))
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # before any CUDA call: the oracle's worker pool is forked from this process
        cpu = oracle_rates(cfg, sids, model, u, args.cpu_seconds)
        _ORACLE_CTX.clear()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import generative_recommendation_constrained_gb300 as zg
    from generative_recommendation_constrained_gb300.device import Decoder, DeviceModel
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream().cuda_stream

    warm_u = synth.make_requests(cfg.batch, cfg.d, 99)
    B, beam, K = cfg.batch, cfg.beam, cfg.topk

    idx = zg.zg_index_build(sids, cfg.V, stream=stream)
    info = zg.zg_index_info_get(idx)
    dm = DeviceModel(model, dev)
    u_dev = torch.from_numpy(u).to(dev)
    if args.plan:
        plan = zg.zg_plan_force(idx, B, beam, [1 if ch == "f" else 0 for ch in args.plan])
        zg.zg_plan_set_fusion(plan, args.cluster)
    else:
        plan = zg.zg_tune(idx, dm.struct, torch.from_numpy(warm_u).to(dev), B, beam, K, 20, stream)
    zg.zg_plan_set_full_projection(plan, {"split": 0, "single": 1}[args.hidden],
                                   {"auto": 0, "written": 1, "tops": 2}[args.scores])
    variants, step_ms, cluster_ctas, fused_ms = zg.zg_plan_describe(plan)
    dec = Decoder(idx, plan, dm, B, beam, K, dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def capture(d, x=None):
        x = u_dev if x is None else x
        d(x)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                d(x)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        return g

    def timed(g, steps, warmup):
        for _ in range(warmup):
            flush.fill_(1.0)
            g.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        barrier(world)
        torch.cuda.synchronize()
        for a, b in ev:
            flush.fill_(1.0)
            a.record()
            g.replay()
            b.record()
        torch.cuda.synchronize()
        barrier(world)
        return [a.elapsed_time(b) for a, b in ev]

    graph = capture(dec)
    if args.quick:
        # short fixed sequence for profilers: warm-up replays and a few decodes
        times = timed(graph, args.steps, max(args.warmup, 3))
        zg.zg_check_device_status(stream)
        if rank == 0:
            print(json.dumps({"quick": True, "ms_per_step": statistics.fmean(times),
                              "plan": [int(v) for v in variants], "cluster_ctas": int(cluster_ctas)}))
        return
    sampler = ClockSampler(local)
    t_clock0 = time.perf_counter()
    times = timed(graph, args.steps, max(args.warmup, 3))
    # keep the GPU busy long enough for the clock samples (untimed replays)
    while time.perf_counter() - t_clock0 < 1.5:
        for _ in range(50):
            graph.replay()
        torch.cuda.synchronize()
    clocks = sampler.stop()
    zg.zg_check_device_status(stream)

    ms = statistics.fmean(times)
    ms_max = max_over_ranks(ms, world, dev)
    value = B * world / (ms_max / 1000.0)

    # unconstrained full-vocabulary decode on the same inputs (the pages' speed reference)
    udec = Decoder(None, None, dm, B, beam, K, dev)
    ugraph = capture(udec)
    utimes = timed(ugraph, max(10, args.steps // 2), 3)
    ums = max_over_ranks(statistics.fmean(utimes), world, dev)

    # score-first order on the same inputs (every token projected, log-softmax
    # over the codebook, then the mask): the conventional baseline, and the
    # top-K overlap of the two orders (a mechanism check on random weights)
    plan_sf = zg.zg_plan_force(idx, B, beam, [1] * cfg.L)
    zg.zg_plan_set_order(plan_sf, zg.ZG_ORDER_SCORE_FIRST)
    sdec = Decoder(idx, plan_sf, dm, B, beam, K, dev)
    sgraph = capture(sdec)
    stimes = timed(sgraph, max(10, args.steps // 2), 3)
    sms = max_over_ranks(statistics.fmean(stimes), world, dev)
    ff_sids = dec(u_dev)[0].cpu().numpy()
    sf_sids = sdec(u_dev)[0].cpu().numpy()
    overlap = float(np.mean([len({tuple(x) for x in ff_sids[q]} & {tuple(x) for x in sf_sids[q]}) / K
                             for q in range(B)]))

    contrast = [step_contrast(zg, idx, dm, cfg, B, u_dev, flush, Decoder)]
    if B > 1:
        contrast.append(step_contrast(zg, idx, dm, cfg, 1, u_dev[:1].contiguous(), flush, Decoder))

    # per-kernel times and work counts (traced decode, L2 flushed before each)
    traces = []
    for _ in range(max(5, min(args.steps, 30))):
        flush.fill_(1.0)
        traces.append(dec.trace(u_dev))
    L = cfg.L
    s0 = traces[-1]["fused_from"] or (L + 1)
    steps_last = traces[-1]["steps"]
    kern = []   # (avg ms, steps, kernel name, algorithmic amount, bound)
    peaks = load_peaks()
    for s in range(1, s0):
        st = steps_last[s - 1]
        avg = {k: statistics.fmean(t["steps"][s - 1][k] for t in traces)
               for k in ("ms_gather", "ms_project", "ms_select")}
        if st["variant"] == 0:
            kern.append((avg["ms_project"], [s], "k_selective", step_bytes(st, cfg, s), "hbm",
                         step_unique_bytes(st, cfg, s)))
            # the chunk counting: per live beam its state (16 B) and index row bounds (8 B)
            # read, its chunk count, first entry and fan-out (12 B) written
            kern.append((avg["ms_gather"], [s], "k_beam_items", st["live_beams"] * 36, "hbm", None))
        else:
            name = "k_full_simt" if cfg.w_dtype == "f32" else "k_full_tc"
            kern.append((avg["ms_project"], [s], name, full_flops(st, cfg, s),
                         "alu" if cfg.w_dtype == "f32" else "tensor", None))
            if s >= 2 or cfg.w_dtype != "f32":
                kern.append((avg["ms_gather"], [s], "k_gather_add", st["live_beams"] * cfg.d * 12, "hbm", None))
        kern.append((avg["ms_select"], [s], "k_select", st["legal_slots"] * 4 + st["live_beams"] * 16, "hbm",
                     None))
    if s0 <= L:
        if s0 == 1:
            # the whole decode is this one launch: its duration is the timed step itself
            fused_kernel_ms = ms
        else:
            fused_kernel_ms = statistics.fmean(t["ms_fused"] for t in traces)
        fb = sum(step_bytes(steps_last[s - 1], cfg, s) for s in range(s0, L + 1))
        fu = sum(step_unique_bytes(steps_last[s - 1], cfg, s) for s in range(s0, L + 1))
        kern.append((fused_kernel_ms, list(range(s0, L + 1)), "k_decode_cluster", fb, "hbm", fu))
    kern.sort(key=lambda x: -x[0])
    top_ms, top_steps, top_name, alg, bound, uniq = kern[0]
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": alg / (top_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
        if uniq:
            roof["achieved_distinct_rows"] = uniq / (top_ms * 1e-3) / 1e9
    elif bound == "tensor":
        roof = {"bound": "tensor", "achieved": alg / (top_ms * 1e-3) / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        sm_mhz = clocks.get("sm_mhz") or peaks["sm_max_mhz"]
        # 152 SMs x 128 fp32 FMA lanes x 2 flops per clock
        roof = {"bound": "alu", "achieved": alg / (top_ms * 1e-3) / 1e12,
                "peak": 152 * 128 * 2 * sm_mhz * 1e6 / 1e12, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if bound == "hbm" and top_name in ("k_selective", "k_decode_cluster"):
        roof["note"] = ("per-(beam, slot) bytes, weight rows counted at every gather; the step's codebook "
                        "is held in L2 (evict_last), so most are L2 hits: traffic is the DRAM bytes per launch")
    roof["traffic"] = ncu_traffic(top_name, cfg.name)
    ent = ncu_entry(top_name, cfg.name)
    if ent and ent.get("lts_throughput_pct") is not None:
        # the same launch's L2 throughput as a fraction of L2 peak (ncu, cold L2)
        roof["l2_throughput_frac_ncu"] = ent["lts_throughput_pct"] / 100.0
    if ent and ent.get("lts_bytes") is not None:
        roof["l2_bytes"] = ent["lts_bytes"]  # lts__t_bytes of the launch: next to the DRAM traffic
    roof["kernel"] = f"{top_name} (steps {top_steps[0]}-{top_steps[-1]})"
    roof["ms_per_launch"] = top_ms
    roof["algorithmic"] = alg
    roof["peak_src"] = peaks["src"]
    work = [{k: v for k, v in st.items() if not k.startswith("ms_")} for st in steps_last]

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region
    n_host = zg.zg_decode_host_workspace_size(idx, plan, dm.struct, B, beam, K)
    ws_h = torch.empty(n_host, dtype=torch.uint8, device=dev)
    u_pin = torch.from_numpy(u).pin_memory()
    o_sids = torch.empty((B, K, L), dtype=torch.int32).pin_memory()
    o_sc = torch.empty((B, K), dtype=torch.float32).pin_memory()
    for _ in range(3):
        zg.zg_decode_host(idx, plan, dm.struct, u_pin, B, beam, K, o_sids, o_sc, ws_h, n_host, stream)
    e2e_steps = max(10, args.steps)
    barrier(world)
    e2e_s = 0.0
    for _ in range(e2e_steps):
        flush.fill_(1.0)  # untimed, like the device-timed steps
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        zg.zg_decode_host(idx, plan, dm.struct, u_pin, B, beam, K, o_sids, o_sc, ws_h, n_host, stream)
        e2e_s += time.perf_counter() - t0  # the call returns once the results are in host memory
    e2e_ms = e2e_s * 1000.0 / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)

    sweep = None
    if cfg.name == "large" and not args.no_sweep:
        sweep = batch_sweep(zg, idx, dm, cfg, u, warm_u, flush, capture, timed, Decoder, dev, stream, world)

    launches_per_step = launches_per_decode([int(v) for v in variants], s0, L, cfg.w_dtype)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": cfg.w_dtype if cfg.w_dtype != "f32" else "f32",
            "data": "synthetic",
            "config": {"workload": workload_desc(cfg), "global_batch": B * world, "beam": beam, "topk": K,
                       "plan": ["full" if v else "selective" for v in variants],
                       "full_projection": {"hidden": args.hidden, "scores": args.scores},
                       "tune_ms": [[round(float(x), 4) for x in r] for r in step_ms],
                       "cluster_ctas": int(cluster_ctas),
                       "tune_fused_ms": [round(float(x), 4) for x in fused_ms],
                       "l2": "flushed by a 256 MiB write before every timed step",
                       "parallelism": f"replicas x{world}: requests sharded, index replicated, no collective",
                       "index_bytes": info["bytes"], "dense_trie_bytes": info["dense_trie_bytes"],
                       "index_gb": info["bytes"] / 1e9, "dense_trie_gb": info["dense_trie_bytes"] / 1e9},
            "p10_ms": float(np.percentile(times, 10)), "p50_ms": float(np.percentile(times, 50)),
            "p90_ms": float(np.percentile(times, 90)),
            "e2e": {"value": B * world / (e2e_ms / 1000.0), "unit": UNIT,
                    "h2d_bytes_per_step": B * cfg.d * 4, "d2h_bytes_per_step": B * K * L * 4 + B * K * 4,
                    "ms_per_step": e2e_ms},
            "gpu_launches": launches_per_step * args.steps,
            "gpu_launches_per_step": launches_per_step,
            "roofline": roof,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "unconstrained": {"ms_per_step": ums, "value": B * world / (ums / 1000.0), "unit": UNIT,
                              "constrained_speedup": ums / ms_max},
            "contrast": contrast,
            "score_first": {"ms_per_step": sms, "value": B * world / (sms / 1000.0), "unit": UNIT,
                            "filter_first_speedup": sms / ms_max, "topk_overlap": overlap},
            "kernels": [{"kernel": n, "steps": st, "ms": round(t, 5)} for t, st, n, _, _, _ in kern],
            "batch_sweep": sweep,
            "work": work,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- batch sweep

def batch_sweep(zg, idx, dm, cfg, u, warm_u, flush, capture, timed, Decoder, dev, stream, world,
                batches=(1, 8, 32, 64), steps: int = 30):
    """Constrained and unconstrained decode latency at each batch size of the
    large catalogue's sweep: requests 0..B-1 of the workload, the plan tuned
    at that batch, graph replays with L2 flushed before each (CUDA events)."""
    import torch
    out = []
    for B in batches:
        if B > u.shape[0]:
            continue
        ub = torch.from_numpy(np.ascontiguousarray(u[:B])).to(dev)
        plan = zg.zg_tune(idx, dm.struct, torch.from_numpy(np.ascontiguousarray(warm_u[:B])).to(dev), B,
                          cfg.beam, cfg.topk, 10, stream)
        variants, _, cluster_ctas, _ = zg.zg_plan_describe(plan)
        dec = Decoder(idx, plan, dm, B, cfg.beam, cfg.topk, dev)
        t = timed(capture(dec, ub), steps, 3)
        udec = Decoder(None, None, dm, B, cfg.beam, cfg.topk, dev)
        ut = timed(capture(udec, ub), steps, 3)
        ms = max_over_ranks(statistics.fmean(t), world, dev)
        ums = max_over_ranks(statistics.fmean(ut), world, dev)
        out.append({"batch": B, "ms_per_batch": ms, "requests_per_s": B * world / (ms / 1000.0),
                    "p10_ms": float(np.percentile(t, 10)), "p90_ms": float(np.percentile(t, 90)),
                    "unconstrained_ms": ums, "constrained_speedup": ums / ms,
                    "plan": "".join("f" if v else "s" for v in variants), "cluster_ctas": int(cluster_ctas)})
        del dec, udec
    return out


# ---------------------------------------------------------------- scoring-variant contrast

def step_contrast(zg, idx, dm, cfg, B, u_dev, flush, Decoder, reps: int = 5):
    """The comparison of the pages' compact-list figure at the step with the
    most legal tokens: the step's kernels (gather-add, projection, select)
    timed under an all-full, an all-naive (compact list + temporary matrix)
    and an all-padded-slots (selective, stand-alone) plan; median of `reps`
    traced decodes, L2 flushed before each."""
    out = {"batch": B}
    times = {}
    for name, v in (("full", 1), ("naive", 2), ("padded", 0)):
        plan = zg.zg_plan_force(idx, B, cfg.beam, [v] * cfg.L)
        zg.zg_plan_set_fusion(plan, 0)
        try:
            dec = Decoder(idx, plan, dm, B, cfg.beam, cfg.topk, u_dev.device)
        except zg.ZgError as e:  # the naive temporary matrix does not fit
            out[name] = str(e)
            continue
        runs = []
        for _ in range(reps):
            flush.fill_(1.0)
            runs.append(dec.trace(u_dev))
        times[name] = runs
        del dec
    if "padded" not in times:
        return out
    legal = [st["legal_slots"] for st in times["padded"][-1]["steps"]]
    s = int(np.argmax(legal))
    out["step"] = s + 1
    out["legal_slots"] = int(legal[s])
    out["scores_full"] = int(B * (1 if s == 0 else cfg.beam) * cfg.V)
    for name, runs in times.items():
        out[f"{name}_ms"] = statistics.median(
            r["steps"][s]["ms_gather"] + r["steps"][s]["ms_project"] + r["steps"][s]["ms_select"] for r in runs)
    if "naive_ms" in out:
        out["naive_over_full"] = out["naive_ms"] / out["full_ms"]
        out["naive_over_padded"] = out["naive_ms"] / out["padded_ms"]
    out["pages"] = {"naive_over_full": 5.1, "naive_over_padded": 8.5}
    return out


# ---------------------------------------------------------------- index rebuild leg

def run_index_rebuild(args, cfg):
    """Rebuild throughput of the step-sliced index (items/s of zg_index_build:
    sort + dedup and the two-pass fill on host threads, streamed to HBM
    through two pinned buffers) and whether a decode served at the same time
    on the same GPU slows down: the mid-sparse decode graph is replayed on its
    own stream before and while the index of `cfg` is rebuilt on a host
    thread, and the median replay times are compared."""
    import threading
    import torch
    import generative_recommendation_constrained_gb300 as zg
    from generative_recommendation_constrained_gb300.device import Decoder, DeviceModel
    dev = torch.device("cuda", 0)
    sids = synth.make_catalogue(cfg, 0)
    # the decode being served meanwhile: the mid-sparse workload, fused plan
    scfg = synth.CONFIGS["mid_sparse"]
    s_sids = synth.make_catalogue(scfg, 0)
    s_model = synth.make_model(scfg.L, scfg.V, scfg.d, scfg.w_dtype, 0)
    serve = torch.cuda.Stream(device=dev)
    s_idx = zg.zg_index_build(s_sids, scfg.V, stream=serve.cuda_stream)
    dm = DeviceModel(s_model, dev)
    u = torch.from_numpy(synth.make_requests(scfg.batch, scfg.d, 1000)).to(dev)
    plan = zg.zg_plan_force(s_idx, scfg.batch, scfg.beam, [0] * scfg.L)
    dec = Decoder(s_idx, plan, dm, scfg.batch, scfg.beam, scfg.topk, dev)
    with torch.cuda.stream(serve):
        dec(u, serve.cuda_stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=serve):
            dec(u, serve.cuda_stream)
    torch.cuda.synchronize()

    def replay_times(stop):
        out = []
        while not stop():
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(serve):
                a.record(serve)
                g.replay()
                b.record(serve)
            b.synchronize()
            out.append(a.elapsed_time(b))
        return out

    t_end = time.perf_counter() + 2.0
    alone = replay_times(lambda: time.perf_counter() > t_end)
    build_stream = torch.cuda.Stream(device=dev)
    res = {}

    def build():
        t0 = time.perf_counter()
        idx = zg.zg_index_build(sids, cfg.V, stream=build_stream.cuda_stream)
        build_stream.synchronize()
        res["s"] = time.perf_counter() - t0
        res["info"] = zg.zg_index_info_get(idx)
        del idx

    for _ in range(max(1, args.warmup // 10)):  # untimed: pages in the host buffers
        build()
    th = threading.Thread(target=build)
    th.start()
    during = replay_times(lambda: not th.is_alive())
    th.join()
    info = res["info"]
    n = int(info["n_input"])
    line = {
        "metric": "index rebuild items/s (sort + dedup + two-pass fill + H2D)", "value": n / res["s"],
        "unit": "items/s", "n_gpus": 1, "higher_is_better": True, "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "items": n, "unique": int(info["n_unique"]),
                   "index_bytes": int(info["bytes"]), "host_threads": os.cpu_count()},
        "seconds": res["s"],
        "phases_ms": {"sort": info["ms_sort"], "count": info["ms_count"], "fill_and_copy": info["ms_fill"],
                      "total": info["ms_total"]},
        "concurrent_decode": {"workload": "mid_sparse (fused, 8 CTAs a cluster)",
                              "ms_alone_median": statistics.median(alone),
                              "ms_during_rebuild_median": statistics.median(during) if during else None,
                              "replays_during": len(during),
                              "slowdown": (statistics.median(during) / statistics.median(alone)) if during else None},
    }
    print(json.dumps(line), flush=True)


def run_light_decoder(args, cfg):
    """The decode with a light causal decoder producing the hidden vectors
    (2 layers, width d, 4 heads, MLP 4d, 2 concept vectors a request; random
    weights): graph-replayed decode time, and from a traced decode the
    decoder's share of the step kernels' time, next to the same workload's
    decode with the synthetic gather-add model."""
    import torch
    import generative_recommendation_constrained_gb300 as zg
    from generative_recommendation_constrained_gb300.device import Decoder, DeviceModel
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream
    sids = synth.make_catalogue(cfg, 0)
    model = synth.make_model(cfg.L, cfg.V, cfg.d, cfg.w_dtype, 0)
    deco = synth.make_deco(cfg.L, cfg.V, cfg.d, M=2, heads=4, ffn=4 * cfg.d, layers=2, seed=0)
    B, beam, K = cfg.batch, cfg.beam, cfg.topk
    c = torch.from_numpy(synth.make_concepts(B, 2, cfg.d, request_seed(0))).to(dev)
    u = torch.from_numpy(synth.make_requests(B, cfg.d, request_seed(0))).to(dev)
    idx = zg.zg_index_build(sids, cfg.V, stream=stream)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = {}
    for name, dm, x in (("light_decoder", DeviceModel(model, dev, deco=deco), c),
                        ("gather_add", DeviceModel(model, dev), u)):
        plan = zg.zg_tune(idx, dm.struct, x, B, beam, K, 5, stream)
        dec = Decoder(idx, plan, dm, B, beam, K, dev)
        dec(x)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                dec(x, side.cuda_stream)
        torch.cuda.current_stream().wait_stream(side)
        times = []
        for i in range(args.warmup + args.steps):
            flush.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            if i >= args.warmup:
                times.append(a.elapsed_time(b))
        flush.fill_(1.0)
        tr = dec.trace(x)
        model_ms = sum(st["ms_model"] for st in tr["steps"])
        step_ms = sum(st["ms_model"] + st["ms_gather"] + st["ms_project"] + st["ms_select"] for st in tr["steps"])
        out[name] = {"ms_per_batch": statistics.fmean(times), "requests_per_s": B / (statistics.fmean(times) / 1e3),
                     "plan": "".join("f" if v else "s" for v in zg.zg_plan_describe(plan)[0]),
                     "traced_model_ms": model_ms, "traced_step_kernels_ms": step_ms}
    ld = out["light_decoder"]
    ld["model_share_of_step_kernels"] = ld["traced_model_ms"] / ld["traced_step_kernels_ms"]
    line = {"metric": "constrained decode with a light causal decoder producing the hidden vectors",
            "unit": "ms/batch", "value": ld["ms_per_batch"], "higher_is_better": False, "n_gpus": 1,
            "data": "synthetic", "config": {"workload": workload_desc(cfg),
                                            "decoder": "2 layers, width d, 4 heads, MLP 4d, 2 concept vectors, "
                                                       "fp32 random weights"},
            **out}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["zerogr", "reference"], default="zerogr")
    ap.add_argument("--workload", default="large", choices=sorted(synth.CONFIGS))
    ap.add_argument("--batch", type=int, default=0, help="requests per batch (0: the workload's own)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the large catalogue's batch sweep")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-requests", type=int, default=0, help="requests a reference-arm step (0: four per core, at most the batch)")
    ap.add_argument("--quick", action="store_true",
                    help="tune, capture and replay only (a short command for profilers)")
    ap.add_argument("--plan", default="", help="fixed per-step variants instead of tuning, e.g. sss or fss")
    ap.add_argument("--cluster", type=int, default=8, help="fused cluster size with --plan (0: no fusion)")
    ap.add_argument("--hidden", choices=["split", "single"], default="split",
                    help="tensor-core full steps: the hidden as hi + lo halves, or one rounding")
    ap.add_argument("--scores", choices=["auto", "written", "tops"], default="auto",
                    help="full steps: scores written out, or chunk tops handed to the select")
    ap.add_argument("--light-decoder", action="store_true",
                    help="decode with a light causal decoder producing the hidden vectors (one JSON line)")
    ap.add_argument("--index-rebuild", action="store_true",
                    help="rebuild throughput of the workload's index while a decode is served (one JSON line)")
    args = ap.parse_args(argv)
    cfg = synth.CONFIGS[args.workload]
    if args.batch:
        cfg = dataclasses.replace(cfg, batch=args.batch)
    if args.plan and len(args.plan) != cfg.L:
        ap.error(f"--plan needs {cfg.L} letters (s or f)")
    if args.impl == "reference":
        run_reference(args, cfg)
    elif args.index_rebuild:
        run_index_rebuild(args, cfg)
    elif args.light_decoder:
        run_light_decoder(args, cfg)
    else:
        run_gpu(args, cfg)


if __name__ == "__main__":
    main()
