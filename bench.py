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

The default run (skewed routing) also times the other four workloads, each
at its own size, and reports them under `workloads`: device step, per-kernel
times and roofline fractions, and the clock window of each.

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
FUSED_AUTO_MAX_TOKENS = 0  # largest batch the default step runs as one fused launch
E2E_PASSES = 3  # timed passes of the end-to-end step; the median pass is reported


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
        # source: the kernel's files, '+'-separated, hashed in that order
        h = hashlib.sha256()
        for name in parts["source"].split("+"):
            src = os.path.join(ROOT, "combine_get_dispatch_04_gb300", "csrc", name)
            if not os.path.exists(src):
                return None
            h.update(open(src, "rb").read())
        if h.hexdigest()[:16] != parts["sha"]:
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


def host_cpu() -> dict:
    """This host's logical cores and CPU model (lscpu, else /proc/cpuinfo)."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "model": model or platform.machine()}


def cpu_baseline(case, target_s: float = 10.0) -> dict:
    """The oracle's step on a bounded sample of the workload: the median of
    three runs of about a third of target_s each."""
    n = calibrate_sample(case, target_s / 3)
    sub = sub_batch(case, n)
    times = sorted(oracle_step(sub) for _ in range(3))
    dt = times[1]
    T = sub.cfg.num_tokens
    return {"value": T / dt, "unit": UNIT, "cores": 1, "kind": "oracle", "host": host_cpu(),
            "sample": (f"first {n} tokens of each of the {case.cfg.num_ranks} source ranks "
                       f"({T} tokens, same routing/hidden rows as the workload): layout + "
                       f"dispatch + combine, single-threaded C oracle, median of 3 runs "
                       f"({', '.join(f'{v:.2f}' for v in times)} s)")}


# ----------------------------------------------------------------------------
def config_dict(cfg: Config, P: int, cap: int, x_bytes: int, flush: bool | None = None) -> dict:
    routing = "uniform distinct top-k" if cfg.routing == "uniform" else f"Zipf(s={cfg.zipf_s}) top-k"
    if cfg.mask_prob:
        routing += f", {int(round(cfg.mask_prob * 100))}% of slots masked"
    if flush is None:
        flush = needs_l2_flush(cfg, P)
    return {"workload": cfg.name, "num_ranks": cfg.num_ranks,
            "tokens_per_rank": cfg.tokens_per_rank, "num_tokens": cfg.num_tokens,
            "hidden": cfg.hidden, "num_experts": cfg.num_experts, "num_topk": cfg.num_topk,
            "routing": routing, "payload": "fp8_e4m3+scales" if cfg.fp8 else "bf16",
            "recv_rows": P, "recv_capacity_rows": cap, "seed": cfg.seed,
            "l2": ("L2 flushed between steps (a read of twice L2, outside the per-step events; "
                   f"x is {x_bytes / 1e6:.1f} MB)" if flush else
                   f"inputs larger than L2 (x {x_bytes / 1e9:.2f} GB; receive buffer "
                   f"{P * cfg.hidden * (1 if cfg.fp8 else 2) / 1e9:.2f} GB)"),
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
                         "host": host_cpu(),
                         "sample": f"each step: first {n} tokens of each source rank "
                                   f"({sub.cfg.num_tokens} tokens), single-threaded C oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class StepRunner:
    """One workload's device buffers and its step (layout -> dispatch ->
    combine) through the public API; the token range [a, b) of dispatch and
    combine serves the end-to-end pipeline's chunks."""

    def __init__(self, ep, cfg: Config, rcfg: Config, args, dev, case):
        import torch
        self.ep, self.cfg, self.args, self.dev = ep, cfg, args, dev
        T, H, K, R, E = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_ranks, cfg.num_experts
        self.T = T
        self.idx = torch.from_numpy(case.topk_idx).to(dev)
        self.w = torch.from_numpy(case.topk_weights).to(dev)
        self.x = torch.from_numpy(case.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        self.views = {}  # (a, b) -> the layout's rows of those tokens, made once
        # layout and dispatch in one launch (small batches)
        self.fused = args.layout == "ht" and (
            args.layout_kernels == "fused" or
            (args.layout_kernels == "auto" and auto_fused(ep, cfg)))
        if args.layout_kernels == "fused" and not ep.fused_fits(T, R, E):
            raise SystemExit("--layout-kernels fused: the batch does not fit the one-launch form")
        if args.layout == "ht":
            # rank-major: worst-case capacity T * min(K, R) rows, no host sync per step
            self.cap = ep.worst_case_rows(T, K, R)
            self.L = ep.alloc_layout(T, E, R, dev)
            self.D = ep.alloc_dispatched(self.cap, H, K, E, R, cfg.fp8, dev)
            self.recv_rows = self.cap
            recv_payload = self.D.recv_x
        else:
            # expert-major: T rows per expert (the worst case with distinct experts per
            # token) when the buffers stay under 32 GB, else 1.25x the largest count
            LL = ep.ll_get_dispatch_layout(self.idx, E, R, T)
            torch.cuda.synchronize(dev)
            max_count = int(LL.ll_count.max().item())
            cap = T if E * T * H * 2 <= (32 << 30) else ((max_count * 5 // 4 + 63) // 64) * 64
            self.L = ep.alloc_ll_layout(T, K, E, R, cap, dev)
            self.do_layout()
            self.D = ep.ll_dispatch(self.x, self.L, use_fp8=cfg.fp8, err=self.err)
            self.recv_rows = E * cap
            recv_payload = self.D.recv_x
        if cfg.fp8:  # combine is bf16 in: random expert outputs in the receive layout
            gen = torch.Generator(device=dev)
            gen.manual_seed(rcfg.seed)
            self.Y = torch.randn((self.recv_rows, H), generator=gen, device=dev).to(torch.bfloat16)
        else:
            self.Y = recv_payload

    def _view(self, a, b):
        from dataclasses import replace
        if (a, b) == (0, self.T):
            return self.L
        v = self.views.get((a, b))
        if v is None:
            L = self.L
            if self.args.layout == "ht":
                v = replace(L, slot=L.slot[a:b], is_token_in_rank=L.is_token_in_rank[a:b])
            else:
                v = replace(L, ll_slot=L.ll_slot[a:b])
            self.views[(a, b)] = v
        return v

    def do_layout(self):
        ep, cfg = self.ep, self.cfg
        if self.args.layout == "ht":
            path = "auto" if self.args.layout_kernels == "fused" else self.args.layout_kernels
            ep.get_dispatch_layout(self.idx, cfg.num_experts, cfg.num_ranks, err=self.err,
                                   out=self.L, path=path)
        else:
            ep.ll_get_dispatch_layout(self.idx, cfg.num_experts, cfg.num_ranks, err=self.err,
                                      out=self.L, path=self.args.layout_kernels)

    def do_layout_dispatch(self):
        """The step's layout and dispatch: one fused launch, or the two calls."""
        if self.fused:
            self.ep.layout_dispatch(self.x, self.idx, self.w, self.cfg.num_experts,
                                    self.cfg.num_ranks, use_fp8=self.cfg.fp8, err=self.err,
                                    layout=self.L, out=self.D)
        else:
            self.do_layout()
            self.do_dispatch(0, self.T)

    def do_dispatch(self, a, b):
        Lc = self._view(a, b)
        if self.args.layout == "ht":
            self.ep.dispatch(self.x[a:b], self.idx[a:b], self.w[a:b], Lc, use_fp8=self.cfg.fp8,
                             err=self.err, out=self.D)
        else:
            self.ep.ll_dispatch(self.x[a:b], Lc, use_fp8=self.cfg.fp8, err=self.err, out=self.D)

    def do_combine(self, a, b):
        Lc = self._view(a, b)
        if self.args.layout == "ht":
            self.ep.combine(self.Y, self.idx[a:b], self.w[a:b], Lc, err=self.err,
                            out=self.out[a:b])
        else:
            self.ep.ll_combine(self.Y, self.w[a:b], Lc, err=self.err, out=self.out[a:b])

    def step(self, ev=None, per_kernel=True):
        # ev[0] / ev[3] bracket the step; ev[1] / ev[2] (per_kernel) split it
        # into layout, dispatch and combine
        s = self.stream
        if ev is not None:
            ev[0].record(s)
        if self.fused:  # layout + dispatch in one launch: the layout's share reads 0
            if ev is not None and per_kernel:
                ev[1].record(s)
            self.do_layout_dispatch()
        else:
            self.do_layout()
            if ev is not None and per_kernel:
                ev[1].record(s)
            self.do_dispatch(0, self.T)
        if ev is not None and per_kernel:
            ev[2].record(s)
        self.do_combine(0, self.T)
        if ev is not None:
            ev[3].record(s)

    def step_isolated(self, ev, flush):
        """One step with every kernel alone between its own pair of events
        (ev[0..5]), L2 flushed before each: no kernel is charged for the
        write-back of the lines the one before it left dirty, nor served
        from lines it left in L2 (ncu's cache control measures the same)."""
        s = self.stream
        flush()
        ev[0].record(s)
        if not self.fused:
            self.do_layout()
        ev[1].record(s)
        flush()
        ev[2].record(s)
        if self.fused:
            self.do_layout_dispatch()
        else:
            self.do_dispatch(0, self.T)
        ev[3].record(s)
        flush()
        ev[4].record(s)
        self.do_combine(0, self.T)
        ev[5].record(s)

    def rows(self) -> int:
        if self.args.layout == "ht":
            return self.ep.total_rows(self.L)
        return int(self.L.ll_count.sum().item())

    def layout_launches(self):
        ep, args, cfg = self.ep, self.args, self.cfg
        if self.fused:
            return 0, "fused"  # counted with the dispatch's launch
        T, K, R, E = cfg.num_tokens, cfg.num_topk, cfg.num_ranks, cfg.num_experts
        if args.layout == "ll":
            if args.layout_kernels == "single" or (args.layout_kernels == "auto"
                                                   and ep.ll_auto_single_launch(T, K, R, E)):
                return 1, "single"
            return 3, "multi"  # rank, expert scan, assign
        if args.layout_kernels == "single" or (args.layout_kernels == "auto"
                                               and ep.auto_single_launch(T, R, E)):
            return 1, "single"  # one thread-block cluster
        # count + assign, with the scan folded in unless R * blocks > 8192 (T > 0)
        nb = R * ((T // R + 511) // 512)
        return (2 if R * nb <= 8192 else 3), "multi"


def auto_fused(ep, cfg: Config) -> bool:
    """The default step fuses layout and dispatch into one launch for the
    batches where that measured faster (decode-size batches)."""
    return ep.fused_fits(cfg.num_tokens, cfg.num_ranks, cfg.num_experts) and \
        cfg.num_tokens <= FUSED_AUTO_MAX_TOKENS


def launch_bound(cfg: Config, P: int) -> bool:
    """True for a step whose algorithmic bytes fit in L2 (the small workload):
    its kernels take less time than the host needs to launch them."""
    ab = algorithmic_bytes(cfg, P)
    return ab["dispatch"] + ab["combine"] < L2_BYTES


def needs_l2_flush(cfg: Config, P: int) -> bool:
    """Flush L2 between timed steps when the step's input rows fit in L2 (they
    could stay resident from one step to the next) or the whole step moves
    less than twice L2."""
    x_bytes = cfg.num_tokens * cfg.hidden * 2
    step_bytes = x_bytes * 3 + P * cfg.hidden * 2 * 2
    return x_bytes < L2_BYTES or step_bytes < 2 * L2_BYTES


def time_device(run: StepRunner, args, world: int, graph=None, min_region_s: float = 0.5):
    """Timed passes of exactly K steps with the inputs resident in HBM.

    The plain pass times K steps as a user runs them: no event between the
    kernels, because an event recorded between two kernels stops the second
    one's early (programmatic) launch, which costs several microseconds per
    kernel edge.  It is repeated until the passes cover min_region_s (so
    that the clock sampler sees the GPU under load), and the median pass is
    reported.  With an L2 flush (a read of a buffer twice the size of L2,
    which leaves no dirty lines behind) between steps, a pair of events
    brackets each step instead and the flush stays outside them.

    Two more passes of K steps give per-kernel durations.  In the first,
    each kernel runs alone between its own events with L2 flushed before it
    (StepRunner.step_isolated): these times feed the roofline.  The second
    puts an event between the kernels of ordinary steps (in_step): there
    each kernel also pays for the write-back of the lines the one before it
    left dirty in L2, and loses its early launch."""
    import torch
    import torch.distributed as dist
    dev, stream, K = run.dev, run.stream, args.steps
    P = run.rows()
    flush = needs_l2_flush(run.cfg, P)
    scrub = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)

    def one_pass(per_kernel):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for i in range(K):
            if flush:
                scrub.sum()
            if graph is not None and not per_kernel:
                if flush:
                    evs[i][0].record(stream)
                graph.replay()
                if flush:
                    evs[i][3].record(stream)
            else:
                run.step(evs[i] if (flush or per_kernel) else None, per_kernel=per_kernel)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        if flush:
            step_ms = statistics.mean(e[0].elapsed_time(e[3]) for e in evs)
        else:
            step_ms = t_start.elapsed_time(t_end) / K
        return step_ms, evs

    wall0 = time.time()
    passes = []
    while True:
        ms, _ = one_pass(per_kernel=False)
        passes.append(ms)
        if time.time() - wall0 >= min_region_s or len(passes) >= 200:
            break
    ms_kernels, evs = one_pass(per_kernel=True)
    iso = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    torch.cuda.synchronize(dev)
    for i in range(K):
        run.step_isolated(iso[i], lambda: scrub.sum())
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    mean = lambda a, b, evl: statistics.mean(e[a].elapsed_time(e[b]) for e in evl)  # noqa: E731
    return {
        "P": P, "flush": flush, "ms": statistics.median(passes), "passes": passes,
        "window": (wall0, wall1),
        "ms_kernels": ms_kernels,
        "layout_ms": mean(0, 1, iso), "dispatch_ms": mean(2, 3, iso),
        "combine_ms": mean(4, 5, iso),
        "in_step": {"layout_ms": mean(0, 1, evs), "dispatch_ms": mean(1, 2, evs),
                    "combine_ms": mean(2, 3, evs)},
    }


def link_bandwidth(dev, nbytes: int = 256 << 20) -> dict:
    """Pinned host <-> device copy rates of this machine (GB/s), each direction
    alone and both at once on two streams: the floor under `e2e`."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h2 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d2 = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn, reps=3):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            best = min(best, time.perf_counter() - t0)
        return best

    def both():
        with torch.cuda.stream(s1):
            d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)

    t_in = timed(lambda: d.copy_(h, non_blocking=True))
    t_out = timed(lambda: h2.copy_(d2, non_blocking=True))
    t_both = timed(both)
    return {"h2d_gbs": nbytes / t_in / 1e9, "d2h_gbs": nbytes / t_out / 1e9,
            "both_gbs": 2 * nbytes / t_both / 1e9, "bytes_per_copy": nbytes}


def time_e2e(run: StepRunner, args, case, world: int) -> dict:
    """The step through the public API on host buffers, pipelined over token
    chunks: routing in -> layout; then per chunk, x in (copy stream) ->
    dispatch + combine of that chunk's tokens (compute stream) -> out back
    (second copy stream).  Every step moves all inputs in and the whole
    result out.  The device-side routing, x and out are double-buffered by
    step parity and the routing travels on the input copy stream, so that
    one step's copies wait only on the kernels of the step before the
    previous one: neither copy direction waits behind the other's step."""
    import torch
    import torch.distributed as dist
    dev, stream, T, H = run.dev, run.stream, run.T, run.cfg.hidden
    h_idx = torch.from_numpy(case.topk_idx).pin_memory()
    h_w = torch.from_numpy(case.topk_weights).pin_memory()
    h_x = torch.from_numpy(case.x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_out = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    steps = max(1, min(args.steps, 20))
    n_chunks = max(1, min(args.e2e_chunks, T // args.e2e_min_chunk_tokens))
    bounds = [T * i // n_chunks for i in range(n_chunks + 1)]
    chunks = [(bounds[c], bounds[c + 1]) for c in range(n_chunks)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # buffers of parity 0 are the runner's own; parity 1 a second set
    bufs = [(run.idx, run.w, run.x, run.out),
            (torch.empty_like(run.idx), torch.empty_like(run.w), torch.empty_like(run.x),
             torch.empty_like(run.out))]
    E = lambda: [torch.cuda.Event() for _ in range(n_chunks)]  # noqa: E731
    ev_route = [torch.cuda.Event(), torch.cuda.Event()]  # routing landed, per parity
    ev_in = [E(), E()]       # x chunk landed
    ev_used = [E(), E()]     # x chunk read by dispatch
    ev_done = [E(), E()]     # out chunk computed
    ev_back = [E(), E()]     # out chunk copied back
    ev_step = [torch.cuda.Event(), torch.cuda.Event()]  # the step's last kernel (routing free)
    used = [False, False]
    step_no = [0]

    def e2e_step():
        par = step_no[0] & 1
        idx, w, x, out = bufs[par]
        run.idx, run.w, run.x, run.out = idx, w, x, out
        with torch.cuda.stream(s_in):
            if used[par]:
                s_in.wait_event(ev_step[par])  # the routing of two steps back is no longer read
            idx.copy_(h_idx, non_blocking=True)
            w.copy_(h_w, non_blocking=True)
            ev_route[par].record(s_in)
            for c, (a, b) in enumerate(chunks):
                if used[par]:
                    s_in.wait_event(ev_used[par][c])
                x[a:b].copy_(h_x[a:b], non_blocking=True)
                ev_in[par][c].record(s_in)
        stream.wait_event(ev_route[par])
        run.do_layout()
        for c, (a, b) in enumerate(chunks):
            stream.wait_event(ev_in[par][c])
            run.do_dispatch(a, b)
            ev_used[par][c].record(stream)
            if used[par]:
                stream.wait_event(ev_back[par][c])  # this buffer's copy of two steps back is done
            run.do_combine(a, b)
            ev_done[par][c].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[par][c])
                h_out[a:b].copy_(out[a:b], non_blocking=True)
                ev_back[par][c].record(s_out)
        ev_step[par].record(stream)
        used[par] = True
        step_no[0] += 1

    def e2e_drain():
        for par in (0, 1):
            if used[par]:
                for c in range(n_chunks):
                    stream.wait_event(ev_back[par][c])

    # warm-up: one untimed pass (the first pass after only two steps often
    # read slower than the ones after it)
    for _ in range(max(2, steps)):
        e2e_step()
    e2e_drain()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    # Passes of `steps` steps each, the median pass reported (as for the
    # device time), after the untimed pass above.
    pass_ms, host_s = [], 0.0
    for _ in range(E2E_PASSES):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h0 = time.perf_counter()
        for _ in range(steps):
            e2e_step()
        e2e_drain()
        host_s += time.perf_counter() - h0  # enqueueing only: the calls return before the GPU is done
        e1.record(stream)
        torch.cuda.synchronize(dev)
        pass_ms.append(e0.elapsed_time(e1) / steps)
    e2e_ms = max_over_ranks(statistics.median(pass_ms), dev)
    # the pipelined steps must give the resident step's result, bit for bit
    run.idx, run.w, run.x, run.out = bufs[0]
    run.step()
    torch.cuda.synchronize(dev)
    same = torch.equal(h_out.view(torch.int16), run.out.cpu().view(torch.int16))
    h2d = h_idx.numel() * 8 + h_w.numel() * 4 + h_x.numel() * 2
    d2h = h_out.numel() * 2
    del bufs
    link = link_bandwidth(dev)
    floor_ms = 1e3 * max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9),
                         (h2d + d2h) / (link["both_gbs"] * 1e9))
    return {"value": whole_job_tokens_per_s(T, world, e2e_ms), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
            "steps": steps, "passes_ms": [round(v, 3) for v in pass_ms],
            "token_chunks": n_chunks,
            "host_enqueue_ms_per_step": 1e3 * host_s / (steps * E2E_PASSES),
            "link": {k: round(v, 1) for k, v in link.items()},
            "link_floor_ms": floor_ms,
            "check": "out matches the device-resident step" if same else "MISMATCH"}


def pages_convention(cfg: Config, P: int, kern: dict) -> dict:
    """The byte accounting of the pages' own benchmarks, for context only
    ("[Not ready] MSCCLPP EP implementation", the bench commits): the
    dispatch counts each rank's bench_tokens * hidden, and the combine one
    copy per dispatched row back to its owner; bandwidth is reported per rank
    (aggregate / ranks) and aggregated.  Over all ranks of one call that is
    T * H payload elements for the dispatch and P * H bf16 rows for the
    combine; the roofline counts every row read and written instead."""
    T, H, R = cfg.num_tokens, cfg.hidden, cfg.num_ranks
    out = {"note": "dispatch: bench_tokens * hidden per rank (E4M3 bytes for the FP8 dispatch, "
                   "else bf16); combine: one bf16 copy per dispatched row; per rank = "
                   "aggregate / ranks; context only, not the roofline's bytes"}
    for k, b in (("dispatch", T * H * (1 if cfg.fp8 else 2)), ("combine", P * H * 2)):
        gbs = b / (kern[k]["ms"] / 1e3) / 1e9
        out[k] = {"bytes": b, "aggregate_gbs": round(gbs, 1), "per_rank_gbs": round(gbs / R, 1)}
    return out


def kernel_report(cfg: Config, P: int, t: dict, peak: float) -> dict:
    ab = algorithmic_bytes(cfg, P)
    kern = {
        "layout": {"ms": t["layout_ms"], "bytes": ab["layout"]},
        "dispatch": {"ms": t["dispatch_ms"], "bytes": ab["dispatch"]},
        "combine": {"ms": t["combine_ms"], "bytes": ab["combine"]},
    }
    for k in ("dispatch", "combine"):
        kern[k]["gbs"] = ab[k] / (kern[k]["ms"] / 1e3) / 1e9
        kern[k]["frac"] = kern[k]["gbs"] / peak
    return kern


def other_workloads(args, ep, dev, peak: float) -> dict:
    """The remaining workloads at their own sizes, each timed as the default
    one (K steps, passes repeated to 0.3 s, median pass; one pass with
    per-kernel events): device step, per-kernel times and roofline
    fractions, and the clock window of each."""
    import torch
    out = {}
    names = args.workload_list.split(",") if args.workload_list else list(CONFIGS)
    for name in names:
        if name == args.config:
            continue
        cfg = CONFIGS[name]
        case = make_case(cfg)
        run = StepRunner(ep, cfg, cfg, args, dev, case)
        for _ in range(args.warmup):
            run.step()
        torch.cuda.synchronize(dev)
        # a step that moves less than L2 holds is bound by host launches, not
        # by the GPU: replay it as one CUDA graph, as a serving loop would
        graph = None
        if launch_bound(cfg, run.rows()):
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                run.step()
            graph.replay()
            torch.cuda.synchronize(dev)
        t = time_device(run, args, 1, graph=graph, min_region_s=0.3)
        if int(run.err.item()) != 0:
            raise SystemExit(f"{name}: device error word {int(run.err.item())}")
        P = t["P"]
        kern = kernel_report(cfg, P, t, peak)
        ab = algorithmic_bytes(cfg, P)
        launches, kinds = run.layout_launches()
        out[name] = {
            "tokens_per_s": whole_job_tokens_per_s(cfg.num_tokens, 1, t["ms"]),
            "ms_per_step": t["ms"], "steps": args.steps, "passes": len(t["passes"]),
            "hbm_gbs": (ab["dispatch"] + ab["combine"]) / (t["ms"] / 1e3) / 1e9,
            "layout_ms": kern["layout"]["ms"], "layout_kernels": kinds,
            "dispatch": dict({k: kern["dispatch"][k] for k in ("ms", "gbs", "frac")},
                             bytes=ab["dispatch"], traffic=load_traffic("dispatch_kernel", name)),
            "combine": dict({k: kern["combine"][k] for k in ("ms", "gbs", "frac")},
                            bytes=ab["combine"], traffic=load_traffic("combine_kernel", name)),
            "kernel_timing": {"in_step_ms_per_step": t["ms_kernels"],
                              "in_step": t["in_step"]},
            "recv_rows": P, "dtype": "e4m3+bf16" if cfg.fp8 else "bf16",
            "l2": "flushed between steps (read of 2x L2, outside the per-step events)"
                  if t["flush"] else "inputs larger than L2",
            "_window": t["window"], "gpu_launches": (launches + 2) * args.steps * len(t["passes"]),
            "step_launch": "cuda_graph_replay" if graph is not None else "eager",
        }
        del run, case
        torch.cuda.empty_cache()
    return out


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
    T = cfg.num_tokens
    run = StepRunner(ep, cfg, rcfg, args, dev, case)
    for _ in range(args.warmup):
        run.step()
    torch.cuda.synchronize(dev)
    if int(run.err.item()) != 0:
        raise SystemExit(f"device error word {int(run.err.item())} after warm-up")

    graph = None
    if args.graph:  # every one-time set-up ran in the warm-up steps
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run.step()
        graph.replay()
        torch.cuda.synchronize(dev)

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(1.0)  # let nvidia-smi start sampling before the timed region
    t = time_device(run, args, world, graph=graph)
    ms = max_over_ranks(t["ms"], dev)
    ms_with_kernel_events = max_over_ranks(t["ms_kernels"], dev)
    P = t["P"]

    e2e = time_e2e(run, args, case, world)
    if int(run.err.item()) != 0:
        raise SystemExit(f"device error word {int(run.err.item())}")
    layout_launches, layout_kernels = run.layout_launches()
    recv_rows = run.recv_rows
    del run
    torch.cuda.empty_cache()

    peak, peak_kind = load_peaks()
    block = None
    if rank == 0 and world == 1 and args.workloads:
        block = other_workloads(args, ep, dev, peak)
    sampler.stop()

    def clocks_of(window):
        c = sampler.summary(*window)
        c["timed_region_s"] = round(window[1] - window[0], 3)
        return c

    clocks = clocks_of(t["window"])
    if block is not None:
        for name in block:
            block[name]["clocks"] = clocks_of(block[name].pop("_window"))
    if rank == 0:
        ab = algorithmic_bytes(cfg, P)
        gbs = (ab["dispatch"] + ab["combine"]) / (ms / 1e3) / 1e9
        kern = kernel_report(cfg, P, t, peak)
        kern["layout"]["launches_per_step"] = layout_launches
        kern["dispatch"]["launches_per_step"] = 1
        kern["combine"]["launches_per_step"] = 1
        dom = "dispatch" if kern["dispatch"]["ms"] >= kern["combine"]["ms"] else "combine"
        kname = {"dispatch": "dispatch_kernel", "combine": "combine_kernel"}[dom]
        src = {"dispatch": "ep_dispatch.cu+ep_scatter.cuh", "combine": "ep_combine.cu"}[dom]
        # expert-major runs have their own captures ("<workload>/ll")
        traffic = load_traffic(kname, cfg.name + ("/ll" if args.layout == "ll" else ""))
        cpu = None if (args.no_cpu_baseline or world > 1 or args.layout == "ll") else cpu_baseline(case)
        line = {
            "metric": METRIC, "value": whole_job_tokens_per_s(T, world, ms), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3+bf16" if cfg.fp8 else "bf16",
            "data": "synthetic (seeded routing and N(0,1) hidden states; no dataset)",
            "config": dict(config_dict(cfg, P, recv_rows, T * cfg.hidden * 2, t["flush"]),
                           layout=args.layout,
                           **({"step_launch": "cuda_graph_replay"} if graph is not None else {}),
                           **({"layout_kernels": layout_kernels} if layout_kernels else {})),
            "hbm_gbs": gbs, "hbm_frac": gbs / peak, "peak_gbs": peak, "peak_kind": peak_kind,
            "roofline": {"bound": "hbm", "kernel": kname, "source": src,
                         "achieved": kern[dom]["gbs"], "peak": peak, "unit": "GB/s",
                         "frac": kern[dom]["gbs"] / peak, "traffic": traffic,
                         "algorithmic_bytes_per_launch": ab[dom],
                         "peak_note": f"of {peak_kind} (copy bandwidth)"},
            "kernels": kern,
            "pages_convention": pages_convention(cfg, P, kern),
            "passes": {"n": len(t["passes"]), "steps_each": args.steps,
                       "ms_min": min(t["passes"]), "ms_max": max(t["passes"]),
                       "note": "value and ms_per_step come from the median pass"},
            "kernel_timing": {"steps": args.steps,
                              "kernels": "each kernel alone between its own events, with L2 "
                                         "flushed (a read of twice L2) before it: no kernel pays "
                                         "for the write-back of the lines the previous one left "
                                         "dirty",
                              "in_step": t["in_step"], "in_step_ms_per_step": ms_with_kernel_events,
                              "note": "in_step: ordinary steps with an event between the kernels; "
                                      "an event stops the next kernel's early launch, and each "
                                      "kernel pays for the previous one's dirty lines"},
            "e2e": e2e,
            "gpu_launches": (layout_launches + 2) * args.steps * len(t["passes"]),
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        if block is not None:
            line["workloads"] = block
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_sharded(args, cfg: Config):
    """The sharded form under torchrun, one rank per GPU: every rank holds the
    workload's tokens_per_rank tokens, the experts are spread over the N
    ranks, and one step is shard layout -> count exchange -> dispatch ->
    all-to-all-v -> (identity experts) -> reverse all-to-all-v -> combine
    (combine_get_dispatch_04_gb300.sharded).  value = N * T_r / the slowest
    rank's step time."""
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist.init_process_group("nccl", device_id=dev)
    import combine_get_dispatch_04_gb300 as ep
    from combine_get_dispatch_04_gb300 import build as ep_build
    from combine_get_dispatch_04_gb300 import sharded
    from dataclasses import replace
    if not ep_build.up_to_date():
        raise SystemExit("libep.so is missing or stale: run __graft_entry__.build() first")
    ep.load()
    if cfg.num_experts % world:
        raise SystemExit(f"{cfg.num_experts} experts do not spread over {world} ranks")
    gcfg = replace(cfg, num_ranks=world)  # the same routing recipe over `world` ranks
    case = make_case(gcfg)
    Tr = gcfg.tokens_per_rank
    a, b = rank * Tr, (rank + 1) * Tr
    idx = torch.from_numpy(np.ascontiguousarray(case.topk_idx[a:b])).to(dev)
    w = torch.from_numpy(np.ascontiguousarray(case.topk_weights[a:b])).to(dev)
    x = torch.from_numpy(np.ascontiguousarray(case.x_bits[a:b]).view(np.int16)).view(
        torch.bfloat16).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sep = sharded.ShardedEP(sharded.DistExchange())

    def step():
        recv, handle = sep.dispatch(x, idx, w, gcfg.num_experts, use_fp8=gcfg.fp8, err=err)
        y = recv.recv_x if not gcfg.fp8 else torch.ones(
            (recv.recv_x.shape[0], gcfg.hidden), dtype=torch.bfloat16, device=dev)
        return sep.combine(y, handle, err=err)

    for _ in range(args.warmup):
        out = step()
    torch.cuda.synchronize(dev)
    if not bool(torch.isfinite(out.float()).all()):
        raise SystemExit("combine produced a non-finite value")
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    if int(err.item()) != 0:
        raise SystemExit(f"device error word {int(err.item())}")
    if rank == 0:
        line = {
            "metric": METRIC, "value": whole_job_tokens_per_s(Tr, world, ms), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3+bf16" if gcfg.fp8 else "bf16",
            "data": "synthetic (seeded routing and N(0,1) hidden states; no dataset)",
            "config": dict(workload=cfg.name, tokens_per_rank=Tr, num_ranks=world,
                           hidden=gcfg.hidden, num_experts=gcfg.num_experts,
                           num_topk=gcfg.num_topk, parallelism=f"ep{world} sharded",
                           steps_include="count exchange with a host copy, all-to-all-v both ways"),
            # per step: the shard layout (count + assign, or + scan), dispatch, combine
            "gpu_launches": (2 + (world * ((Tr + 511) // 512) > 8192) + 2) * args.steps,
        }
        print(json.dumps(line), flush=True)
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
    ap.add_argument("--layout-kernels", choices=["auto", "multi", "single", "fused"],
                    default="auto",
                    help="layout kernels: one cluster launch (single, small batches), the "
                         "multi-launch form, layout and dispatch in one launch (fused, small "
                         "batches), or the benchmark's choice (auto)")
    ap.add_argument("--graph", action="store_true",
                    help="time the plain steps as replays of one CUDA graph of the step "
                         "(no host launch cost; the per-kernel pass stays eager)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sharded", action="store_true",
                    help="under torchrun: the sharded form, one rank per GPU with the "
                         "workload's tokens per rank (the default --gpus N run is N "
                         "independent replicas of the one-GPU shuffle)")
    ap.add_argument("--workloads", dest="workloads", action="store_true", default=None,
                    help="also time the other workloads (default: on for the default run)")
    ap.add_argument("--no-workloads", dest="workloads", action="store_false")
    ap.add_argument("--workload-list", default=None,
                    help="comma-separated workloads for the `workloads` block (default: all "
                         "but --config)")
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="token chunks the end-to-end step pipelines its copies over")
    ap.add_argument("--e2e-min-chunk-tokens", type=int, default=2048,
                    help="fewest tokens in one end-to-end chunk (smaller chunks add more host "
                         "work per step than they overlap)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    cfg = CONFIGS[args.config]
    if args.workloads is None:  # the default run carries every workload in its line
        args.workloads = (args.config == DEFAULT_CONFIG and not args.tokens_per_rank
                          and args.seed is None and args.layout == "ht" and not args.graph)
    if args.tokens_per_rank:
        cfg = cfg.scaled(args.tokens_per_rank)
    if args.seed is not None:
        from dataclasses import replace
        cfg = replace(cfg, seed=args.seed)
    if args.impl == "reference":
        run_reference(args, cfg)
    elif args.sharded:
        run_sharded(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
