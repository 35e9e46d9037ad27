"""Benchmark: one step = get_dispatch_layout -> dispatch -> combine (identity
experts: combine reads the dispatched rows) over one batch of seeded
synthetic routing and hidden states, on one GB300 per process.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config skewed] [--tokens-per-rank N]

Prints one JSON line (rank 0).  `value` is whole-job tokens/s with inputs
resident in HBM; `e2e` is the same metric with the step's inputs copied from
pinned host memory and the combined output copied back inside the timed
region (pipelined over token chunks on two copy streams; consecutive steps
overlap their copies, chunk by chunk).  Multi-GPU runs (torchrun) are independent replicas, one problem per
GPU (the shuffle on one GPU has no cross-GPU step): per-GPU work is fixed,
value = N * T / max-over-ranks step time.

`--impl reference` times the plain CPU oracle (the correctness reference)
on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import CONFIGS, Config, make_case  # noqa: E402

METRIC = "dispatch+combine tokens/s and HBM GB/s (% of 8 TB/s roofline) at 1 GB300"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 << 20  # GB300 L2
DEFAULT_CONFIG = "skewed"  # the largest bf16 workload (most bytes moved per phase)


# ----------------------------------------------------------------------------
# host logic shared by the replicas (tested on CPU with gloo)
# ----------------------------------------------------------------------------
def replica_config(cfg: Config, rank: int) -> Config:
    """Each replica draws its own batch: same shape, seed offset by rank."""
    if rank == 0:
        return cfg
    from dataclasses import replace
    return replace(cfg, seed=cfg.seed + 1000 * rank)


def max_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_replica: int, n_replicas: int, ms_per_step: float) -> float:
    return tokens_per_replica * n_replicas / (ms_per_step / 1e3)


def algorithmic_bytes(cfg: Config, P: int) -> dict:
    """Bytes each kernel must move at minimum (payload only; metadata apart)."""
    T, H, K, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_ranks
    if cfg.fp8:
        dispatch = T * H * 2 + P * H * 1 + P * (H // 128) * 4
    else:
        dispatch = T * H * 2 + P * H * 2
    combine = P * H * 2 + T * H * 2
    meta_dispatch = T * R * 4 + T * K * 12 + P * (4 + 12 * K)  # slot, routing, recv metadata
    meta_combine = T * R * 4 + T * K * 12
    layout = T * K * 8 + T * R * (1 + 4) + T * 8 * 2  # routing in; mask, slot out; scratch
    return dict(dispatch=dispatch, combine=combine, meta_dispatch=meta_dispatch,
                meta_combine=meta_combine, layout=layout)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_traffic(kernel: str, workload: str):
    """dram bytes per launch from a committed ncu summary, if it still
    matches the kernel source (profiles/ncu_traffic.txt)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    import hashlib
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = dict(p.split("=", 1) for p in line.split())
        if parts.get("kernel") != kernel or parts.get("workload") != workload:
            continue
        src = os.path.join(ROOT, "combine_get_dispatch_04_gb300", "csrc", parts["source"])
        if not os.path.exists(src):
            return None
        if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != parts["sha"]:
            return None
        return float(parts["dram_bytes_per_launch"])
    return None


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons; the
    summary keeps the samples whose timestamps fall inside the timed region."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.rows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        from datetime import datetime
        for ln in out.splitlines():
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                ts = datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                self.rows.append((ts, float(p[1]), float(p[2]), p[5:9]))
            except ValueError:
                continue

    def summary(self, t0: float, t1: float):
        rows = [r for r in self.rows if t0 <= r[0] <= t1]
        padded = False
        if not rows:  # a short region: take the samples next to it
            rows = [r for r in self.rows if t0 - 0.25 <= r[0] <= t1 + 0.25]
            padded = True
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({self.NAMES[i] for r in rows for i, v in enumerate(r[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": rows[0][2],
                "reasons": reasons, "samples": len(rows), "window_padded": padded}


# ----------------------------------------------------------------------------
# CPU oracle on a bounded sample: the first n tokens of every source rank
# form a smaller batch of the same workload
# ----------------------------------------------------------------------------
def sub_batch(case, n_per_rank: int):
    from workloads import Case
    cfg = case.cfg
    Tr = cfg.tokens_per_rank
    n = min(n_per_rank, Tr)
    rows = np.concatenate([np.arange(s * Tr, s * Tr + n) for s in range(cfg.num_ranks)])
    from dataclasses import replace
    sub_cfg = replace(cfg, tokens_per_rank=n)
    return Case(sub_cfg, np.ascontiguousarray(case.topk_idx[rows]),
                np.ascontiguousarray(case.topk_weights[rows]),
                np.ascontiguousarray(case.x_bits[rows]))


def oracle_step(case) -> float:
    """One pass of the oracle (layout, dispatch, combine with identity experts);
    returns seconds."""
    import oracle
    cfg = case.cfg
    t0 = time.perf_counter()
    L = oracle.layout(case.topk_idx, cfg.num_experts, cfg.num_ranks)
    d = oracle.dispatch(case.x_bits, case.topk_idx, case.topk_weights, cfg.num_experts,
                        cfg.num_ranks, L.slot, L.num_rows, use_fp8=cfg.fp8, fill=None)
    y = d.recv_x
    if cfg.fp8:  # combine is bf16 in: dequantised rows stand in for expert outputs
        y = np.zeros((L.num_rows, cfg.hidden), np.uint16)
    oracle.combine(y, case.topk_idx, case.topk_weights, cfg.num_experts, cfg.num_ranks, L.slot)
    return time.perf_counter() - t0


def calibrate_sample(case, target_s: float) -> int:
    """Tokens per source rank that make one oracle step take about target_s."""
    n = 8
    while True:
        dt = oracle_step(sub_batch(case, n))
        if dt > 0.2 or n >= case.cfg.tokens_per_rank:
            break
        n *= 4
    per_tok = dt / (n * case.cfg.num_ranks)
    return int(max(1, min(case.cfg.tokens_per_rank, target_s / per_tok / case.cfg.num_ranks)))


def cpu_baseline(case, target_s: float = 10.0) -> dict:
    n = calibrate_sample(case, target_s)
    sub = sub_batch(case, n)
    dt = oracle_step(sub)
    T = sub.cfg.num_tokens
    return {"value": T / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"first {n} tokens of each of the {case.cfg.num_ranks} source ranks "
                       f"({T} tokens, same routing/hidden rows as the workload): layout + "
                       f"dispatch + combine, single-threaded C oracle, {dt:.2f} s")}


# ----------------------------------------------------------------------------
def config_dict(cfg: Config, P: int, cap: int, x_bytes: int) -> dict:
    routing = "uniform distinct top-k" if cfg.routing == "uniform" else f"Zipf(s={cfg.zipf_s}) top-k"
    if cfg.mask_prob:
        routing += f", {int(round(cfg.mask_prob * 100))}% of slots masked"
    return {"workload": cfg.name, "num_ranks": cfg.num_ranks,
            "tokens_per_rank": cfg.tokens_per_rank, "num_tokens": cfg.num_tokens,
            "hidden": cfg.hidden, "num_experts": cfg.num_experts, "num_topk": cfg.num_topk,
            "routing": routing, "payload": "fp8_e4m3+scales" if cfg.fp8 else "bf16",
            "recv_rows": P, "recv_capacity_rows": cap, "seed": cfg.seed,
            "l2": (f"inputs larger than L2 (x {x_bytes / 1e9:.2f} GB; receive buffer "
                   f"{P * cfg.hidden * (1 if cfg.fp8 else 2) / 1e9:.2f} GB)"
                   if x_bytes * 3 + P * cfg.hidden * 4 >= 2 * L2_BYTES else
                   "L2 flushed between steps (256 MB write outside the per-step events)"),
            "experts": "identity (combine reads the dispatched rows)" if not cfg.fp8
                       else "random bf16 expert outputs"}


def run_reference(args, cfg: Config):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    case = make_case(cfg)
    import oracle
    P = oracle.layout(case.topk_idx, cfg.num_experts, cfg.num_ranks).num_rows
    budget = 150.0
    per_step = budget / max(1, args.steps + args.warmup)
    n = calibrate_sample(case, per_step)
    sub = sub_batch(case, n)
    for _ in range(args.warmup):
        oracle_step(sub)
    times = [oracle_step(sub) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    value = sub.cfg.num_tokens / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; no dataset)",
        "config": dict(config_dict(cfg, P, cfg.num_tokens * min(cfg.num_topk, cfg.num_ranks),
                                   cfg.num_tokens * cfg.hidden * 2), layout="ht"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"each step: first {n} tokens of each source rank "
                                   f"({sub.cfg.num_tokens} tokens), single-threaded C oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, cfg: Config):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import combine_get_dispatch_04_gb300 as ep
    from combine_get_dispatch_04_gb300 import build as ep_build
    if not ep_build.up_to_date():
        raise SystemExit("libep.so is missing or stale: run __graft_entry__.build() first")
    ep.load()

    rcfg = replica_config(cfg, rank)
    case = make_case(rcfg)
    T, H, K, R, E = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_ranks, cfg.num_experts
    idx = torch.from_numpy(case.topk_idx).to(dev)
    w = torch.from_numpy(case.topk_weights).to(dev)
    x = torch.from_numpy(case.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    from dataclasses import replace as _replace

    if args.layout == "ht":
        # rank-major: worst-case capacity T * min(K, R) rows, no host sync per step
        cap = ep.worst_case_rows(T, K, R)
        L = ep.alloc_layout(T, E, R, dev)
        D = ep.alloc_dispatched(cap, H, K, E, R, cfg.fp8, dev)

        def do_layout():
            ep.get_dispatch_layout(idx, E, R, err=err, out=L, path=args.layout_kernels)

        def do_dispatch(a, b):
            Lc = L if (a, b) == (0, T) else _replace(
                L, slot=L.slot[a:b], is_token_in_rank=L.is_token_in_rank[a:b])
            ep.dispatch(x[a:b], idx[a:b], w[a:b], Lc, use_fp8=cfg.fp8, err=err, out=D)

        def do_combine(a, b):
            Lc = L if (a, b) == (0, T) else _replace(
                L, slot=L.slot[a:b], is_token_in_rank=L.is_token_in_rank[a:b])
            ep.combine(Y, idx[a:b], w[a:b], Lc, err=err, out=out[a:b])

        recv_rows = cap
        recv_payload = D.recv_x
    else:
        # expert-major: T rows per expert (the worst case with distinct experts per
        # token) when the buffers stay under 32 GB, else 1.25x the largest count
        LL = ep.ll_get_dispatch_layout(idx, E, R, T)
        torch.cuda.synchronize(dev)
        max_count = int(LL.ll_count.max().item())
        cap = T if E * T * H * 2 <= (32 << 30) else ((max_count * 5 // 4 + 63) // 64) * 64
        LL = ep.alloc_ll_layout(T, K, E, R, cap, dev)
        DL = None

        def do_layout():
            ep.ll_get_dispatch_layout(idx, E, R, err=err, out=LL, path=args.layout_kernels)

        def do_dispatch(a, b):
            LLc = LL if (a, b) == (0, T) else _replace(LL, ll_slot=LL.ll_slot[a:b])
            ep.ll_dispatch(x[a:b], LLc, use_fp8=cfg.fp8, err=err, out=DL)

        def do_combine(a, b):
            LLc = LL if (a, b) == (0, T) else _replace(LL, ll_slot=LL.ll_slot[a:b])
            ep.ll_combine(Y, w[a:b], LLc, err=err, out=out[a:b])

        do_layout()
        DL = ep.ll_dispatch(x, LL, use_fp8=cfg.fp8, err=err)
        recv_rows = E * cap
        recv_payload = DL.recv_x

    if cfg.fp8:  # combine is bf16 in: random expert outputs in the receive layout
        gen = torch.Generator(device=dev)
        gen.manual_seed(rcfg.seed)
        Y = torch.randn((recv_rows, H), generator=gen, device=dev).to(torch.bfloat16)
    else:
        Y = recv_payload

    def step(ev=None, per_kernel=True):
        # ev[0] / ev[3] bracket the step; ev[1] / ev[2] (per_kernel) split it
        # into layout, dispatch and combine
        if ev is not None:
            ev[0].record(stream)
        do_layout()
        if ev is not None and per_kernel:
            ev[1].record(stream)
        do_dispatch(0, T)
        if ev is not None and per_kernel:
            ev[2].record(stream)
        do_combine(0, T)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    P = ep.total_rows(L) if args.layout == "ht" else int(LL.ll_count.sum().item())
    P_est = P
    if int(err.item()) != 0:
        raise SystemExit(f"device error word {int(err.item())} after warm-up")

    graph = None
    if args.graph:  # every one-time set-up ran in the warm-up steps
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize(dev)

    # ---------------- timed region: inputs resident in HBM ----------------
    # Pass 1 times exactly K steps as a user runs them: no event between the
    # kernels, because an event recorded between two kernels stops the second
    # one's early (programmatic) launch, which costs several microseconds per
    # kernel edge.  Pass 2 runs K more steps with an event around every
    # kernel, for the per-kernel durations (layout, dispatch, combine) that the
    # roofline uses; these include that lost overlap.
    # Workloads that move less than twice L2 per step get L2 flushed between
    # steps (a 256 MB write outside the per-step events); the others stream
    # far more than L2 holds.
    step_bytes = T * H * 2 * 3 + (P_est * H * 2 * 2)
    flush = step_bytes < 2 * L2_BYTES
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)

    def timed_pass(per_kernel):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for i in range(args.steps):
            if flush:
                scrub.fill_(i & 0xFF)
            if graph is not None and not per_kernel:
                if flush:
                    evs[i][0].record(stream)
                graph.replay()
                if flush:
                    evs[i][3].record(stream)
            else:
                step(evs[i] if (flush or per_kernel) else None, per_kernel=per_kernel)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        if flush:
            step_ms = statistics.mean(e[0].elapsed_time(e[3]) for e in evs)
        else:
            step_ms = t_start.elapsed_time(t_end) / args.steps
        return step_ms, evs

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(1.0)  # let nvidia-smi start sampling before the timed region
    wall0 = time.time()
    ms_local, _ = timed_pass(per_kernel=False)
    ms_kernels_local, evs = timed_pass(per_kernel=True)
    wall1 = time.time()
    sampler.stop()
    ms = max_over_ranks(ms_local, dev)
    ms_with_kernel_events = max_over_ranks(ms_kernels_local, dev)
    lay_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    dis_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    com_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    clocks = sampler.summary(wall0, wall1)
    clocks["timed_region_s"] = round(wall1 - wall0, 3)

    # ---------------- end to end: pinned host buffers, copies timed --------
    h_idx = torch.from_numpy(case.topk_idx).pin_memory()
    h_w = torch.from_numpy(case.topk_weights).pin_memory()
    h_x = torch.from_numpy(case.x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_out = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(1, min(args.steps, 20))
    # The step through the public API on host buffers, pipelined over token
    # chunks: routing in -> layout; then per chunk, x in (copy stream) ->
    # dispatch + combine of that chunk's tokens (compute stream) -> out back
    # (second copy stream).  Every step moves all inputs in and the whole
    # result out.
    n_chunks = max(1, min(args.e2e_chunks, T // args.e2e_min_chunk_tokens))
    bounds = [T * i // n_chunks for i in range(n_chunks + 1)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(n_chunks)]      # x chunk landed
    ev_used = [torch.cuda.Event() for _ in range(n_chunks)]    # x chunk read by dispatch
    ev_done = [torch.cuda.Event() for _ in range(n_chunks)]    # out chunk computed
    ev_back = [torch.cuda.Event() for _ in range(n_chunks)]    # out chunk copied back
    first = [True]

    def e2e_step():
        # routing in and layout on the compute stream (after the previous
        # step's kernels, which read idx and w)
        idx.copy_(h_idx, non_blocking=True)
        w.copy_(h_w, non_blocking=True)
        for c in range(n_chunks):
            a, b = bounds[c], bounds[c + 1]
            with torch.cuda.stream(s_in):
                if not first[0]:
                    s_in.wait_event(ev_used[c])  # the previous step has read this x chunk
                x[a:b].copy_(h_x[a:b], non_blocking=True)
                ev_in[c].record(s_in)
        do_layout()
        for c in range(n_chunks):
            a, b = bounds[c], bounds[c + 1]
            stream.wait_event(ev_in[c])
            do_dispatch(a, b)
            ev_used[c].record(stream)
            if not first[0]:
                stream.wait_event(ev_back[c])  # the previous step's copy of this out chunk is done
            do_combine(a, b)
            ev_done[c].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[c])
                h_out[a:b].copy_(out[a:b], non_blocking=True)
                ev_back[c].record(s_out)
        first[0] = False

    def e2e_drain():
        for c in range(n_chunks):
            stream.wait_event(ev_back[c])

    e2e_step()
    e2e_drain()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e2e_drain()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    # the pipelined steps must give the resident step's result, bit for bit
    step()
    torch.cuda.synchronize(dev)
    e2e_check = "out matches the device-resident step" if torch.equal(
        h_out.view(torch.int16), out.cpu().view(torch.int16)) else "MISMATCH"
    h2d = h_idx.numel() * 8 + h_w.numel() * 4 + h_x.numel() * 2
    d2h = h_out.numel() * 2
    if int(err.item()) != 0:
        raise SystemExit(f"device error word {int(err.item())}")

    layout_kernels = None
    if args.layout == "ll":
        if args.layout_kernels == "single" or (args.layout_kernels == "auto"
                                               and ep.ll_auto_single_launch(T, K, R, E)):
            layout_launches, layout_kernels = 1, "single"
        else:
            layout_launches, layout_kernels = 3, "multi"  # rank, expert scan, assign
    elif args.layout_kernels == "single" or (args.layout_kernels == "auto"
                                             and ep.auto_single_launch(T, R, E)):
        layout_launches, layout_kernels = 1, "single"  # one thread-block cluster
    else:  # count + assign, with the scan folded in unless R * blocks > 8192 (T > 0)
        nb = R * ((T // R + 511) // 512)
        layout_launches, layout_kernels = (2 if R * nb <= 8192 else 3), "multi"
    if rank == 0:
        peak, peak_kind = load_peaks()
        ab = algorithmic_bytes(cfg, P)
        gbs = (ab["dispatch"] + ab["combine"]) / (ms / 1e3) / 1e9
        kern = {
            "layout": {"ms": lay_ms, "bytes": ab["layout"], "launches_per_step": layout_launches},
            "dispatch": {"ms": dis_ms, "bytes": ab["dispatch"], "launches_per_step": 1,
                         "gbs": ab["dispatch"] / (dis_ms / 1e3) / 1e9},
            "combine": {"ms": com_ms, "bytes": ab["combine"], "launches_per_step": 1,
                        "gbs": ab["combine"] / (com_ms / 1e3) / 1e9},
        }
        for k in ("dispatch", "combine"):
            kern[k]["frac"] = kern[k]["gbs"] / peak
        dom = "dispatch" if dis_ms >= com_ms else "combine"
        kname = {"dispatch": "dispatch_kernel", "combine": "combine_kernel"}[dom]
        src = {"dispatch": "ep_dispatch.cu", "combine": "ep_combine.cu"}[dom]
        # expert-major runs have their own captures ("<workload>/ll")
        traffic = load_traffic(kname, cfg.name + ("/ll" if args.layout == "ll" else ""))
        cpu = None if (args.no_cpu_baseline or world > 1 or args.layout == "ll") else cpu_baseline(case)
        line = {
            "metric": METRIC, "value": whole_job_tokens_per_s(T, world, ms), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3+bf16" if cfg.fp8 else "bf16",
            "data": "synthetic (seeded routing and N(0,1) hidden states; no dataset)",
            "config": dict(config_dict(cfg, P, recv_rows, T * H * 2), layout=args.layout,
                           **({"step_launch": "cuda_graph_replay"} if graph is not None else {}),
                           **({"layout_kernels": layout_kernels} if layout_kernels else {})),
            "hbm_gbs": gbs, "hbm_frac": gbs / peak, "peak_gbs": peak, "peak_kind": peak_kind,
            "roofline": {"bound": "hbm", "kernel": kname, "source": src,
                         "achieved": kern[dom]["gbs"], "peak": peak, "unit": "GB/s",
                         "frac": kern[dom]["gbs"] / peak, "traffic": traffic,
                         "algorithmic_bytes_per_launch": ab[dom],
                         "peak_note": f"of {peak_kind} (copy bandwidth)"},
            "kernels": kern,
            "kernel_timing": {"steps": args.steps, "ms_per_step": ms_with_kernel_events,
                              "note": "per-kernel events in a second pass of K steps; an event "
                                      "between two kernels stops the early launch of the second, "
                                      "so these steps run slower than the plain ones"},
            "e2e": {"value": whole_job_tokens_per_s(T, world, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "steps": e2e_steps, "token_chunks": n_chunks,
                    "check": e2e_check},
            "gpu_launches": (layout_launches + 2) * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=list(CONFIGS))
    ap.add_argument("--seed", type=int, default=None,
                    help="draw the workload with this seed instead of its own")
    ap.add_argument("--tokens-per-rank", type=int, default=None,
                    help="scale the workload (same recipe) for profiling runs")
    ap.add_argument("--layout", choices=["ht", "ll"], default="ht",
                    help="receive layout: rank-major (ht, default) or expert-major (ll)")
    ap.add_argument("--layout-kernels", choices=["auto", "multi", "single"], default="auto",
                    help="layout kernels: one cluster launch (single, small batches), the "
                         "multi-launch form, or the library's choice (auto)")
    ap.add_argument("--graph", action="store_true",
                    help="time the plain steps as replays of one CUDA graph of the step "
                         "(no host launch cost; the per-kernel pass stays eager)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="token chunks the end-to-end step pipelines its copies over")
    ap.add_argument("--e2e-min-chunk-tokens", type=int, default=2048,
                    help="fewest tokens in one end-to-end chunk (smaller chunks add more host "
                         "work per step than they overlap)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    cfg = CONFIGS[args.config]
    if args.tokens_per_rank:
        cfg = cfg.scaled(args.tokens_per_rank)
    if args.seed is not None:
        from dataclasses import replace
        cfg = replace(cfg, seed=args.seed)
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
