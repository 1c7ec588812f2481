#!/usr/bin/env python3
"""Benchmark of the batched speculative-sampling verify step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 2] [--mode sample]
    python bench.py --impl reference ...   # the float64 CPU oracle on host cores

One step = one verify call over one batch of synthetic inputs (all rows read
once, acceptance, first-reject scan, residual/bonus draw).  The default
workload is config 2 (B=8, gamma=3, V=128256, bf16, T=0.8).  Inputs are
rotated over enough device copies that each step reads logits that are not
in L2.  Rank 0 prints one JSON line.  Under torchrun each rank runs its own
batch (requests are independent: no data-path collective), so scaling is
weak and the value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft tokens/sec per verify call"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="2", help="workload: 1, 2, 3, 4, 5a, 5b")
    ap.add_argument("--mode", choices=["sample", "greedy"], default="sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layout", choices=["padded", "packed"], default="padded",
                    help="padded [B][G+1][V] rows, or packed rows with a cu_draft prefix")
    ap.add_argument("--schedule", choices=["auto", "stream", "persistent"], default="auto",
                    help="auto: the resident cluster path, the streaming cluster path or the "
                         "persistent grid, the first that applies; stream: never the resident "
                         "path; persistent: always the grid")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every timed step from Python instead of one CUDA-graph replay")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of rank `rank`'s batch: rank 0 keeps the workload's own seed, so a
    1-GPU run and rank 0 of an N-GPU run verify the same requests."""
    return base_seed if rank == 0 else base_seed * 1000 + rank


def across_ranks(ms: float, units, world: int, device=None):
    """Slowest rank's time and the sum over ranks of each count in `units`
    (verified tokens, emitted tokens, bytes).  Requests are independent, so
    this is the only exchange between ranks: no collective in the data path."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    u = torch.tensor([float(x) for x in units], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), [float(x) for x in u.tolist()]


def workload_desc(w, mode):
    from speculative_decoding_verification_62_gb300 import workloads as W
    return {"workload": f"config {w.name}: {W.CONFIGS[w.name]['desc']}", "B": w.B,
            "gamma_max": w.G, "gamma_sum": w.gamma_sum(), "V": w.V, "mode": mode,
            "input_sha256": w.sha256()}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def oracle_time(w, mode, budget_s=4.0, max_calls=100000, min_calls=1):
    """Time the float64 oracle on the whole batch, repeated for ~budget_s."""
    import oracle
    from speculative_decoding_verification_62_gb300 import workloads as W
    inp = W.oracle_inputs(w)
    cores = os.cpu_count() or 1
    calls, t0 = 0, time.perf_counter()
    while True:
        if mode == "sample":
            oracle.sample(**inp, nthreads=cores)
        else:
            oracle.greedy(inp["target"], inp["draft_tokens"], inp["gamma"], nthreads=cores)
        calls += 1
        el = time.perf_counter() - t0
        if calls >= max_calls or (el >= budget_s and calls >= min_calls):
            break
    used = min(cores, w.B)  # OpenMP over requests: one thread per request at most
    return dict(value=w.gamma_sum() * calls / el, unit=UNIT, cores=used, kind="oracle",
                sample=f"{calls} call(s) of the full batch ({w.B} requests) of config {w.name}, "
                       f"float64 C oracle, OpenMP over requests ({used} of {cores} host "
                       f"threads busy), {el:.2f} s wall",
                seconds=el, calls=calls)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch  # noqa: F401  (inputs are drawn with torch's CPU generator)
    from speculative_decoding_verification_62_gb300 import workloads as W
    w = W.make(args.config, device="cpu")
    t = []
    for _ in range(args.warmup):
        oracle_time(w, args.mode, budget_s=0.0, max_calls=1)
    for _ in range(args.steps):
        t.append(oracle_time(w, args.mode, budget_s=0.0, max_calls=1)["seconds"])
    total = sum(t)
    value = w.gamma_sum() * args.steps / total
    cores = min(os.cpu_count() or 1, w.B)  # OpenMP over requests
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_desc(w, args.mode),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step is one call of the float64 C oracle on the "
                                       f"full batch of config {w.name} ({w.B} requests), "
                                       f"OpenMP over {cores} host threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_62_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(config, mode, kernel):
    """DRAM bytes per launch from the committed ncu summary, if it describes
    this kernel and the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(f"{config}/{mode}")
    if not e or e.get("source_hash") != source_hash() or e.get("kernel") != kernel:
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from speculative_decoding_verification_62_gb300 import binding
    from speculative_decoding_verification_62_gb300 import workloads as W

    # each rank draws its own batch (different seed): weak scaling by request
    base = W.make(args.config, device=dev)
    if rank:
        base = W.make(args.config, device=dev, seed=rank_seed(base.meta["seed"], rank))
    mode = args.mode
    B, G, V = base.B, base.G, base.V
    binding.spec_verify_set_schedule({"auto": binding.SCHEDULE_AUTO,
                                      "stream": binding.SCHEDULE_STREAM,
                                      "persistent": binding.SCHEDULE_PERSISTENT}[args.schedule])
    route, csize = binding.spec_verify_route(base.target.dtype, B, G, V, greedy=mode == "greedy")
    kernel = {binding.ROUTE_CLUSTER: "cluster_kernel", binding.ROUTE_STREAM: "stream_kernel",
              binding.ROUTE_CLAIMS: "stream_kernel", binding.ROUTE_PERSISTENT: "verify_kernel"}[route]
    schedule = {binding.ROUTE_CLUSTER: f"resident clusters of {csize} CTAs, one per request",
                binding.ROUTE_STREAM: f"streaming clusters of {csize} CTAs, one per request",
                binding.ROUTE_CLAIMS: "streaming CTAs claiming requests in turn, longest first",
                binding.ROUTE_PERSISTENT: "persistent grid"}[route]
    launches_per_call = 1

    packed = args.layout == "packed"
    # inputs in the chosen layout: lens is gamma (padded) or cu_draft (packed)
    if packed:
        pk = W.pack(base)
        src = dict(target=pk.target, draft=pk.draft, draft_tokens=pk.draft_tokens,
                   lens=pk.cu_draft, uniforms=pk.uniforms, temperature=pk.temperature)
    else:
        src = dict(target=base.target, draft=base.draft, draft_tokens=base.draft_tokens,
                   lens=base.gamma, uniforms=base.uniforms, temperature=base.temperature)

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 2**20)
    per_copy = src["target"].numel() * src["target"].element_size()
    if mode == "sample":
        per_copy += src["draft"].numel() * src["draft"].element_size()
    ncopy = max(2, math.ceil(4 * l2 / per_copy))
    ncopy = min(ncopy, max(2, int(0.3 * torch.cuda.mem_get_info(dev)[0] // per_copy)))
    targets = [src["target"]] + [src["target"].clone() for _ in range(ncopy - 1)]
    drafts = [src["draft"]] + [src["draft"].clone() for _ in range(ncopy - 1)] \
        if mode == "sample" else [None] * ncopy
    v = binding.Verifier(B, G, V, dev)
    stream = torch.cuda.current_stream(dev)

    def call(t, d, x, s):
        if mode == "sample" and packed:
            v.sample_packed(t, d, x["lens"], x["draft_tokens"], x["uniforms"],
                            x["temperature"], stream=s)
        elif mode == "sample":
            v.sample(t, d, x["draft_tokens"], x["lens"], x["uniforms"], x["temperature"],
                     stream=s)
        elif packed:
            v.greedy_packed(t, x["lens"], x["draft_tokens"], stream=s)
        else:
            v.greedy(t, x["draft_tokens"], x["lens"], stream=s)

    def step(i, s=None):
        j = i % ncopy
        call(targets[j], drafts[j], src, stream if s is None else s)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    # The timed steps are captured once into a CUDA graph and replayed, so the
    # device time is not bounded by the Python launch path (which the e2e
    # number below includes).
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cap = torch.cuda.current_stream(dev)
            for i in range(args.steps):
                step(i, cap)
        graph.replay()  # one untimed replay
        torch.cuda.synchronize(dev)
    status = binding.spec_verify_status(v.workspace, stream)
    if status:
        raise RuntimeError(f"device status flags: {binding.status_names(status)}")

    clocks = Clocks(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    emitted_local = int(v.num_accepted.sum().item()) + B
    ms_max, (gsum_all, emitted_all) = across_ranks(
        ms, [base.gamma_sum(), emitted_local], world, dev)
    ms_step = ms_max / args.steps
    value = gsum_all / (ms_step * 1e-3)

    bytes_min = base.bytes_min(mode)
    # roofline of one GPU: this rank's algorithmic bytes over its own step time
    achieved = bytes_min / (ms / args.steps * 1e-3) / 1e9
    peak, peak_src = measured_peak_hbm()

    # ---- end to end through the public API from pinned host memory ----
    e2e = None
    if not args.no_e2e:
        host = {k: x.cpu().pin_memory() for k, x in src.items()}
        dbuf = {k: torch.empty_like(x) for k, x in src.items()}
        out_h = torch.empty((B, G + 1), dtype=torch.int32).pin_memory()
        nacc_h = torch.empty((B,), dtype=torch.int32).pin_memory()
        keys = [k for k in host if mode == "sample" or k not in ("draft", "uniforms",
                                                                   "temperature")]
        h2d = sum(host[k].numel() * host[k].element_size() for k in keys)
        d2h = out_h.numel() * 4 + nacc_h.numel() * 4

        def e2e_step():
            for k in keys:
                dbuf[k].copy_(host[k], non_blocking=True)
            call(dbuf["target"], dbuf["draft"], dbuf, stream)
            out_h.copy_(v.out_tokens, non_blocking=True)
            nacc_h.copy_(v.num_accepted, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(dev)
        k2 = max(10, min(args.steps, 100))
        if world > 1:
            dist.barrier()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(k2):
            e2e_step()
        f1.record(stream)
        torch.cuda.synchronize(dev)
        te_max, (gsum_e2e,) = across_ranks(f0.elapsed_time(f1), [base.gamma_sum()], world, dev)
        e2e = {"value": gsum_e2e / (te_max / k2 * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": te_max / k2}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_time(W.make(args.config, device="cpu"), mode)
        cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}

    if world > 1:
        dist.barrier()
    if rank == 0:
        cfg = workload_desc(base, mode)
        cfg.update({"layout": args.layout,
                    "schedule": schedule,
                    "parallelism": f"replicas x{world} (independent requests)",
                    "launch": "one CUDA-graph replay of the timed steps" if graph is not None
                              else "one Python call per step",
                    "l2": f"rotating {ncopy} device copies of the logits "
                          f"({ncopy * per_copy / 2**20:.0f} MiB > 4x L2 {l2 / 2**20:.0f} MiB)",
                    "emitted_tokens_per_s": emitted_all / (ms_step * 1e-3),
                    "bytes_min_per_step": bytes_min})
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if base.target.dtype == torch.bfloat16 else "f32",
                "data": "synthetic", "config": cfg,
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                             "frac": achieved / peak, "peak_source": peak_src,
                             "traffic": None if packed else profiled_traffic(args.config, mode, kernel),
                             "kernel": kernel + " (one launch per step)"},
                "clocks": clk, "e2e": e2e, "gpu_launches": args.steps * launches_per_call,
                "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
