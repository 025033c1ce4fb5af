"""Benchmark of the MXFP4 MoE layer on one GB300 (or N replicas under torchrun).

Metric: effective HBM bandwidth of one layer call, TB/s = algorithmic bytes /
time, where the bytes are the packed weights + E8M0 scales of the distinct
experts the call touches plus the bf16 activations read and written
(3*I*H*(1/2 + 1/32) per expert + 4*T*H).  Router weights are not counted
(reported beside).  us_per_call is reported as well.

A step is one moe_layer_forward call (router -> top-k + grouping -> gate/up ->
down + combine) on the workload's inputs, already resident in HBM.  Steps
rotate over L distinct device copies of the weights (a multi-layer decode), so
that no step finds its weights in L2 (L * touched bytes > 2.5 x L2).  Steps
are replayed from a CUDA graph; W warm-up steps precede the K timed ones.

Extra JSON keys:
  roofline      the dominant kernel against the measured HBM copy bandwidth:
                for T <= 8 the layer is one kernel (algorithmic bytes of the
                whole layer / its CUDA-event duration); otherwise the gate/up
                kernel with its h finalize.  traffic: the ncu DRAM bytes per
                launch recorded for the current kernel sources, else null.
  per_config    the other configurations the metric names (GLM T = 4 and 16)
                and the 1T-class shape at T = 1 and 4, each timed the same way
                (graph replay over its own weight rotation) plus 16 L2-scrubbed
                single calls.
  kernel_us     per-kernel CUDA-event times of eagerly queued calls (for a
                single-launch call: launch-inclusive, eager);
  phase_us      for the single-launch kernel, its phases from the kernel's
                own timestamps (first CTA's view).
  l2_scrubbed_single_call  64 calls, each after writing a buffer of 4x the L2
                size (not timed) and bracketed alone by CUDA events: median,
                p10, p90.
  cpu_baseline  the FP64 oracle on this host, a bounded sample.
  e2e           the same metric through moe_layer_forward_hostio, with the
                pinned host->device copy of x and the device->host copy of y
                inside every step.
  clocks        nvidia-smi samples taken during the timed region.

--impl reference times the oracle (the only other implementation of this
layer) on the same workload and prints the same line with "impl":
"reference".

--act mxfp8 runs the MXFP8 live-activation-quantisation variant
(moe_layer_forward_mxfp8: x and h quantised to MXFP8, both projections as
block-scaled tcgen05 MMAs) on the same workload and bytes; its roofline
object is the gate/up GEMM, its e2e copies x from and y to pinned host memory
around every call, and the reference arm runs the oracle's MXFP8 mode.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from block_scaled_fp4_moe_gb300 import inputs  # noqa: E402

METRIC = "MoE layer µs/call and effective HBM TB/s (% of 8 TB/s) at T=1/4/16 tokens"
PAGES_ROOFLINE_TBS = 8.0
DEFAULT_CONFIG = "glm_t1"
def touched_bytes(cfg: inputs.MoEConfig, n_experts: int) -> dict:
    per_expert = 3 * cfg.I * cfg.H * (0.5 + 1.0 / 32)
    act = 2 * cfg.T * cfg.H * 2
    return {"per_expert": per_expert, "weights": n_experts * per_expert, "activations": act,
            "total": n_experts * per_expert + act,
            "gateup": n_experts * 2 * cfg.I * cfg.H * (0.5 + 1.0 / 32) + cfg.T * cfg.H * 2,
            "router": cfg.H * cfg.E * 4}


def read_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's `value` (the timed region's length), so that
    the job's time is that of its slowest replica."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, bytes_per_call: float, per_call_s: float) -> float:
    """Whole-job effective TB/s: every replica moves `bytes_per_call` per call."""
    return world * bytes_per_call / per_call_s / 1e12


# ---------------------------------------------------------------- reference

def oracle_call_factory(cfg: inputs.MoEConfig, act: str = "exact"):
    import oracle
    x = inputs.make_x(cfg)
    wr, bias = inputs.make_router(cfg)
    route = oracle.route(x, wr, bias, cfg.top_k)
    experts = {}
    for e in sorted(set(int(v) for v in route["ids"].ravel())):
        experts[e] = inputs.make_expert(cfg, e)

    def call(tokens):
        r = oracle.route(x, wr, bias, cfg.top_k)
        return oracle.moe_tokens(x, r["ids"], r["w"], lambda e: experts[e], tokens, act=act)
    return call, route


def time_oracle(cfg, budget_s: float, max_calls: int | None = None, act: str = "exact"):
    """Wall time of whole oracle layer calls on a bounded sample of tokens."""
    import oracle
    call, route = oracle_call_factory(cfg, act)
    n_exp = len(set(int(v) for v in route["ids"].ravel()))
    # tokens per call: all of them when the whole call fits the budget, else a prefix
    t0 = time.perf_counter()
    call(np.arange(1, dtype=np.int32))
    per_token = time.perf_counter() - t0
    n_tok = max(1, min(cfg.T, int(budget_s / max(per_token, 1e-6))))
    tokens = np.arange(n_tok, dtype=np.int32)
    times = []
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        call(tokens)
        times.append(time.perf_counter() - t0)
        if (max_calls and len(times) >= max_calls) or time.perf_counter() - t_start > budget_s:
            break
    per_call = statistics.median(times) * cfg.T / n_tok          # scaled to the whole batch
    b = touched_bytes(cfg, n_exp)
    cores = oracle.num_threads()
    return {"per_call_s": per_call, "tbs": b["total"] / per_call / 1e12, "cores": cores,
            "sample": f"{len(times)} oracle call(s) on {n_tok} of {cfg.T} token(s), scaled to T={cfg.T}",
            "n_experts": n_exp}


def run_reference(args, cfg):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        time_oracle(cfg, budget_s=0.0, max_calls=1, act=args.act)
    res = [time_oracle(cfg, budget_s=budget, max_calls=1, act=args.act) for _ in range(args.steps)]
    per_call = statistics.median(r["per_call_s"] for r in res)
    b = touched_bytes(cfg, res[0]["n_experts"])
    val = b["total"] / per_call / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_call * 1e3,
            "us_per_call": per_call * 1e6, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(cfg), "name": cfg.name, "activations": args.act},
            "cpu_baseline": {"value": val, "unit": "TB/s", "cores": res[0]["cores"], "kind": "oracle",
                             "sample": res[0]["sample"]},
            "e2e": {"value": val, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def describe(cfg):
    return (f"{cfg.name}: T={cfg.T}, H={cfg.H}, {cfg.E} routed + {cfg.has_shared} shared experts, "
            f"top-{cfg.top_k}, I={cfg.I}, MXFP4 (E2M1 + E8M0/32) weights, bf16 activations")


# ---------------------------------------------------------------- our arm

# Configurations reported beside the headline one (the metric names T = 1, 4
# and 16; the 1T-class shape at T = 1 and 4 carries the same bandwidth target).
PER_CONFIG = ("glm_verify_t4", "glm_verify_t16", "1t_t1", "1t_t4")


def kernel_source_digest() -> str:
    """Digest of the CUDA sources: a DRAM-traffic record taken on other
    sources no longer describes the kernel that runs."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_scaled_fp4_moe_gb300", "csrc")
    for path in sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh")) +
                       glob.glob(os.path.join(csrc, "*.h"))):
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """dram__bytes_read.sum + dram__bytes_write.sum per launch of `kernel` on
    `workload`, from the ncu record in profiles/dram_traffic.txt, or None when
    no record was taken on the current kernel sources."""
    digest = kernel_source_digest()
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.txt")) as f:
            for line in f:
                parts = line.split("#", 1)[0].split()
                if len(parts) >= 5 and parts[0] == workload and parts[1] == kernel and parts[2] == digest:
                    return int(parts[3]) + int(parts[4])
    except OSError:
        pass
    return None


class Workload:
    """One configuration's inputs resident in HBM, with L copies of the
    repacked weights and router (L * touched bytes > 2.5 x L2) so that steps
    rotating over them never find their weights in L2."""

    def __init__(self, cfg, dev, act="exact", base=None):
        import torch

        from block_scaled_fp4_moe_gb300 import moe
        self.cfg, self.dev, self.act = cfg, dev, act
        self.mx = act == "mxfp8"
        self.x = inputs.make_x(cfg)
        wr, bias = inputs.make_router(cfg)
        if base is None:
            bank_np = inputs.make_bank(cfg)
            base = moe.MXFP4Bank.from_host(bank_np, cfg.E, cfg.has_shared, device=dev, with_mx=self.mx)
            del bank_np
        self.xd = torch.from_numpy(self.x.view(np.int16)).to(dev).view(torch.bfloat16)
        self.wrd = torch.from_numpy(wr).to(dev)
        self.bd = None if bias is None else torch.from_numpy(bias).to(dev)
        self.ws = moe.alloc_workspace(cfg.T, base, cfg.top_k, device=dev)
        self.y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
        ids = torch.empty((cfg.T, cfg.slots), dtype=torch.int32, device=dev)
        tw = torch.empty((cfg.T, cfg.slots), dtype=torch.float32, device=dev)
        self.layer = moe.moe_layer_forward_mxfp8 if self.mx else moe.moe_layer_forward
        self.layer(self.xd, self.wrd, self.bd, cfg.top_k, base, 1.0, self.y, ids, tw, self.ws)
        st = moe.moe_check_device_status(self.ws)
        if st != 0:
            raise RuntimeError(moe.moe_status_string(st))
        self.n_exp = len(set(ids.cpu().numpy().ravel().tolist()))
        self.bytes = touched_bytes(cfg, self.n_exp)
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.n_layers = max(2, math.ceil(2.5 * self.l2 / self.bytes["total"]))
        self.base = base
        self.banks = [base] + [base.clone_packed() for _ in range(self.n_layers - 1)]
        self.routers = [self.wrd] + [self.wrd.clone() for _ in range(self.n_layers - 1)]
        launches = moe.moe_layer_launches(cfg.T, base, cfg.top_k)
        if self.mx:
            # routing (+ x quantisation) by the single-launch kernel's routing
            # phases when the layer would be one launch, else two routing
            # launches and the x quantisation; then gate/up GEMM, h finalise,
            # down GEMM, combine
            launches = 5 if launches == 1 else 7
        self.launches = launches
        # the copies above were enqueued on the current stream; the timed calls
        # run on another (non-blocking) stream, which must not start before
        # they are complete
        torch.cuda.synchronize(dev)

    def call(self, i, stream, chain=False):
        from block_scaled_fp4_moe_gb300 import moe
        cfg, L = self.cfg, self.n_layers
        if chain:
            # a chain of layers: each call names the next one, whose router and
            # shared expert it prefetches into L2 once its own streams are done
            j = (i + 1) % L
            moe.moe_layer_forward_next(self.xd, self.routers[i % L], self.bd, cfg.top_k, self.banks[i % L], 1.0,
                                       self.y, ws=self.ws, next_router_w=self.routers[j], next_bank=self.banks[j],
                                       stream=stream)
        else:
            self.layer(self.xd, self.routers[i % L], self.bd, cfg.top_k, self.banks[i % L], 1.0, self.y,
                       ws=self.ws, stream=stream)

    def graph_time(self, steps, warmup, stream, chain=False, world=1, clocks=None):
        """Seconds per call over exactly `steps` calls replayed from CUDA
        graphs of one rotation, after `warmup` untimed calls; max over ranks."""
        import torch
        import torch.distributed as dist
        L = self.n_layers
        stream.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(stream):
            for i in range(max(warmup, L)):
                self.call(i, stream, chain)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(L):
                self.call(i, torch.cuda.current_stream(), chain)
        reps, rest = divmod(steps, L)
        tail = None
        if rest:
            tail = torch.cuda.CUDAGraph()
            with torch.cuda.graph(tail, stream=stream):
                for i in range(rest):
                    self.call(i, torch.cuda.current_stream(), chain)
        for _ in range(max(1, math.ceil(warmup / L))):
            graph.replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.__enter__()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(reps):
                graph.replay()
            if tail is not None:
                tail.replay()
            ev1.record(stream)
        stream.synchronize()
        if clocks is not None:
            clocks.__exit__()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        elapsed = ev0.elapsed_time(ev1) / 1e3
        return max_over_ranks(elapsed, world, self.dev) / steps

    def scrubbed_single_calls(self, n, stream):
        """n calls, each after writing a buffer of 4x the L2 size (not timed)
        and bracketed alone by CUDA events: median, p10, p90 (us)."""
        import torch
        scrub = torch.empty(self.l2, dtype=torch.float32, device=self.dev)     # 4 bytes x L2 size
        ce = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        stream.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(stream):
            for i, (e0, e1) in enumerate(ce):
                scrub.fill_(float(i))
                e0.record(stream)
                self.call(i, stream)
                e1.record(stream)
        stream.synchronize()
        cold = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in ce)
        del scrub
        med = statistics.median(cold)
        return {"median_us": med, "p10_us": cold[len(cold) // 10], "p90_us": cold[(9 * len(cold)) // 10],
                "calls": len(cold), "median_tbs": self.bytes["total"] / (med * 1e-6) / 1e12}

    def release(self):
        import torch
        self.banks = self.routers = None
        self.base = None
        torch.cuda.empty_cache()


def per_config_line(wl, per_call, scrubbed, peak):
    tbs = wl.bytes["total"] / per_call / 1e12
    return {"workload": describe(wl.cfg), "T": wl.cfg.T, "experts_touched": wl.n_exp,
            "bytes_per_call": wl.bytes["total"], "launches_per_call": wl.launches,
            "us_per_call": per_call * 1e6, "tbs": tbs, "pct_of_8TBs": 100 * tbs / PAGES_ROOFLINE_TBS,
            "frac_of_measured_copy": tbs * 1e3 / peak if peak else None,
            "l2_scrubbed_single_call_us": scrubbed["median_us"],
            "l2_scrubbed_single_call_tbs": scrubbed["median_tbs"]}


def run_mine(args, cfg):
    import torch
    import torch.distributed as dist

    from block_scaled_fp4_moe_gb300 import _build, moe

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    moe.lib()

    mx = args.act == "mxfp8"
    wl = Workload(cfg, dev, args.act)
    b = wl.bytes
    stream = torch.cuda.Stream(device=dev)
    steps = max(1, args.steps)
    clk = ClockSampler(local)
    per_call = wl.graph_time(steps, args.warmup, stream, chain=args.chain, world=world, clocks=clk)
    st = moe.moe_check_device_status(wl.ws, stream=stream)
    if st != 0:
        raise RuntimeError(moe.moe_status_string(st))
    launches = wl.launches

    # ---- per-kernel times: the same steps launched eagerly with events between
    # the kernels, queued behind a bounded sleep kernel so that the GPU runs
    # them back to back (no host gaps inside the measured intervals).  When a
    # call is a single launch, events 1..4 all follow it and the interval
    # ev0 -> ev4 includes the launch of the kernel; its phases come from the
    # kernel's own timestamps instead.
    if mx:
        kern = {"route": [], "quant_x": [], "gateup_gemm": [], "quant_h_down_combine": []}
        profiled = moe.moe_layer_forward_mxfp8_profiled
    else:
        kern = {"router": [], "topk_group": [], "gateup_hfin": [], "down_combine": []}
        profiled = moe.moe_layer_forward_profiled
    whole = []
    n_layers = wl.n_layers
    n_prof = min(max(steps, n_layers), 400)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_prof)]
    with torch.cuda.stream(stream):
        for row in evs:            # torch creates the CUDA event on its first record
            for e in row:
                e.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(2e9 * 60e-6 * n_prof))      # ~60 us of host time per queued step
        for i in range(n_prof):
            profiled(wl.xd, wl.routers[i % n_layers], wl.bd, cfg.top_k, wl.banks[i % n_layers], 1.0, wl.y, wl.ws,
                     evs[i], stream=stream)
    stream.synchronize()
    for i in range(n_prof):
        for j, name in enumerate(kern):
            kern[name].append(evs[i][j].elapsed_time(evs[i][j + 1]) * 1e3)
        whole.append(evs[i][0].elapsed_time(evs[i][4]) * 1e3)
    phases = None
    if launches == 1:
        kern_us = {"fused_layer_kernel_launch_inclusive": statistics.median(whole)}
        kernel_source = ("cuda events around each eagerly queued single-launch call (includes the launch; the "
                         "kernel's own duration inside the timed graph replay is us_per_call)")
        samples = []
        for i in range(min(64, 4 * n_layers)):
            moe.moe_layer_forward(wl.xd, wl.routers[i % n_layers], wl.bd, cfg.top_k, wl.banks[i % n_layers], 1.0,
                                  wl.y, ws=wl.ws, stream=stream)
            samples.append(moe.moe_read_phase_times(wl.ws, stream=stream))
        phases = {k: statistics.median(s_[k] for s_ in samples) for k in moe.PHASE_NAMES}
    else:
        kernel_source = "cuda events between the kernels of eagerly queued steps"
        kern_us = {k: statistics.median(v) for k, v in kern.items()}

    scrubbed = wl.scrubbed_single_calls(64, stream)

    # ---- end to end through host buffers
    xh = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    xs = torch.empty_like(wl.xd)

    def e2e_call(i):
        if mx:
            # pinned x -> device, the layer, y -> pinned host, all on `stream`,
            # then wait for the copy back
            with torch.cuda.stream(stream):
                xs.copy_(xh, non_blocking=True)
                wl.layer(xs, wl.routers[i % n_layers], wl.bd, cfg.top_k, wl.banks[i % n_layers], 1.0, wl.y,
                         ws=wl.ws, stream=stream)
                yh.copy_(wl.y, non_blocking=True)
            stream.synchronize()
        else:
            moe.moe_layer_forward_hostio(xh, wl.routers[i % n_layers], wl.bd, cfg.top_k, wl.banks[i % n_layers],
                                         1.0, yh, wl.ws, stream=stream)
    for i in range(3):
        e2e_call(i)
    n_e2e = min(steps, 2000)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        e2e_call(i)
    e2e_per_call = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, dev)
    if not torch.equal(yh.to(dev), wl.y):
        raise RuntimeError("host-buffer entry point disagrees with the device entry point")

    peaks = read_peaks()
    peak = peaks.get("hbm_gbs")
    if mx:
        # the gate/up GEMM: its weights plus the MXFP8 codes and scales of x
        roof_kernel, traffic_key = "mx8_gemm_kernel<gate/up> (tcgen05 kind::mxf8f6f4 block-scaled)", "mx8_gemm_gateup"
        roof_bytes = wl.n_exp * 2 * cfg.I * cfg.H * (0.5 + 1.0 / 32) + cfg.T * cfg.H * (1 + 1.0 / 32)
        roof_us = kern_us["gateup_gemm"]
    elif launches == 1:
        # one launch per step: its average duration inside the timed graph
        # replay is the step time
        roof_kernel, traffic_key = "fused_layer_kernel (the whole layer)", "fused_layer_kernel"
        roof_bytes = b["total"]
        roof_us = per_call * 1e6
    else:
        roof_kernel, traffic_key = "ffn_tc_kernel<gate/up> (+ h finalisation)", "ffn_tc_gateup"
        roof_bytes = b["gateup"]
        roof_us = kern_us["gateup_hfin"]
    achieved = roof_bytes / (roof_us * 1e-6) / 1e9

    # ---- the other headline configurations, each in the same launch form:
    # graph replay over its own rotation, and L2-scrubbed single calls
    per_config = None
    if args.per_config and not mx and not args.chain and cfg.name == DEFAULT_CONFIG:
        per_config = {cfg.name: per_config_line(wl, per_call, scrubbed, peak)}
        glm_base = wl.banks[0]
        wl.banks = wl.banks[:1]
        wl.routers = wl.routers[:1]
        torch.cuda.empty_cache()
        base_1t = None
        for name in PER_CONFIG:
            c2 = inputs.CONFIGS[name]
            shared = glm_base if (c2.H, c2.E, c2.I) == (cfg.H, cfg.E, cfg.I) else base_1t
            w2 = Workload(c2, dev, "exact", base=shared)
            if shared is None:
                base_1t = w2.base
            n2 = max(4 * w2.n_layers, min(steps, 200))
            pc = w2.graph_time(n2, args.warmup, stream, world=world)
            sc = w2.scrubbed_single_calls(16, stream)
            st = moe.moe_check_device_status(w2.ws, stream=stream)
            if st != 0:
                raise RuntimeError(f"{name}: {moe.moe_status_string(st)}")
            per_config[name] = per_config_line(w2, pc, sc, peak)
            per_config[name]["steps"] = n2
            w2.release()
        del base_1t
        torch.cuda.empty_cache()

    line = None
    if rank == 0:
        cpu = time_oracle(cfg, budget_s=args.cpu_budget, act=args.act)
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": job_value(world, b["total"], per_call), "unit": "TB/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": per_call * 1e3, "us_per_call": per_call * 1e6,
            "pct_of_8TBs": 100 * b["total"] / per_call / 1e12 / PAGES_ROOFLINE_TBS,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("mxfp4 weights x mxfp8 (e4m3 + e8m0/32) activations -> f32 accumulate (tcgen05 "
                      "block-scaled), bf16 out" if mx else "mxfp4 weights x f16 activations -> f32 accumulate, bf16 out"),
            "data": "synthetic",
            "config": {"workload": describe(cfg), "name": cfg.name, "T": cfg.T, "experts_touched": wl.n_exp,
                       "activations": args.act,
                       "bytes_per_call": b["total"], "router_bytes_not_counted": b["router"],
                       "l2": f"inputs larger than L2: steps rotate over {n_layers} weight copies "
                             f"({n_layers} x {b['total'] / 1e6:.1f} MB vs L2 {wl.l2 / 1e6:.0f} MB)",
                       "launch": f"cuda graph replay, {launches} kernel launch(es) per call" +
                                 (", layers chained (moe_layer_forward_next: the next layer's router and shared "
                                  "expert prefetched into L2)" if args.chain else ""),
                       "parallelism": f"replicas x{world}"},
            "kernel_us": kern_us, "kernel_timing": kernel_source, "phase_us": phases,
            "l2_scrubbed_single_call": scrubbed,
            "per_config": per_config,
            "roofline": {"bound": "hbm", "kernel": roof_kernel, "achieved": achieved,
                         "peak": peak if peak else 6800.0, "unit": "GB/s",
                         "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak else "fallback",
                         "frac": achieved / (peak if peak else 6800.0),
                         "traffic": recorded_traffic(cfg.name, traffic_key),
                         "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, recorded "
                                           "for these kernel sources (null: not captured on them)",
                         "algorithmic_bytes": roof_bytes},
            "cpu_baseline": {"value": cpu["tbs"], "unit": "TB/s", "cores": cpu["cores"], "kind": "oracle",
                             "sample": cpu["sample"]},
            "e2e": {"value": job_value(world, b["total"], e2e_per_call), "unit": "TB/s",
                    "us_per_call": e2e_per_call * 1e6,
                    "h2d_bytes_per_step": cfg.T * cfg.H * 2, "d2h_bytes_per_step": cfg.T * cfg.H * 2},
            "gpu_launches": launches * steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_profile_case(args, cfg):
    """A short, plain sequence of layer calls for ncu: one weight copy, no
    graphs, no oracle; the command a committed profile summary names."""
    import torch

    from block_scaled_fp4_moe_gb300 import _build, moe
    _build.build()
    dev = torch.device("cuda", 0)
    x = inputs.make_x(cfg)
    wr, bias = inputs.make_router(cfg)
    mx = args.act == "mxfp8"
    bank = moe.MXFP4Bank.from_host(inputs.make_bank(cfg), cfg.E, cfg.has_shared, device=dev, with_mx=mx)
    xd = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    wrd = torch.from_numpy(wr).to(dev)
    bd = None if bias is None else torch.from_numpy(bias).to(dev)
    ws = moe.alloc_workspace(cfg.T, bank, cfg.top_k, device=dev)
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    layer = moe.moe_layer_forward_mxfp8 if mx else moe.moe_layer_forward
    for _ in range(args.profile_calls):
        layer(xd, wrd, bd, cfg.top_k, bank, 1.0, y, ws=ws)
    st = moe.moe_check_device_status(ws)
    print(json.dumps({"profile_case": cfg.name, "act": args.act, "calls": args.profile_calls, "status": st}))
    return 0 if st == 0 else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=list(inputs.CONFIGS))
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--chain", action=argparse.BooleanOptionalAction, default=False,
                    help="time the calls as a chain of layers that prefetch the next layer's router and shared "
                         "expert (moe_layer_forward_next)")
    ap.add_argument("--act", choices=["exact", "mxfp8"], default="exact",
                    help="activations: exact (bf16 x, f16 hi/lo h) or the MXFP8 live-quantisation variant")
    ap.add_argument("--per-config", action=argparse.BooleanOptionalAction, default=True,
                    help="also measure the other headline configurations (GLM T=4, 16; 1T T=1, 4) in the same run")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="profiling mode: run this many plain layer calls on one weight copy and exit")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)     # never fewer than 3 untimed warm-up steps
    cfg = inputs.CONFIGS[args.config]
    if args.chain and args.act != "exact":
        ap.error("--chain applies to the exact-activation layer only")
    if args.profile_calls:
        return run_profile_case(args, cfg)
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_mine(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
