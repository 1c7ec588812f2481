#!/usr/bin/env python3
"""Benchmark of the batched speculative-sampling verify step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 5b] [--mode sample]
    python bench.py --impl reference ...   # the float64 CPU oracle on host cores

One step = one verify call over one batch of synthetic inputs (row statistics,
acceptance, first-reject scan, residual/bonus draw; on request claims a
request's rows are read only up to its first rejection).  The default
workload is config 5b (B=512, gamma=3, V=128256, bf16, T in {0.5, 1, 1.5}):
919 MB of logits per call, the largest of the standard workloads.  Inputs
are drawn once on the CPU (so both arms and the parity check see the same
bytes, named by their SHA-256) and rotated over device copies whose total
exceeds 4x the L2, so no step reads logits left in L2 by the previous one.

Timing: W untimed steps, then the K timed steps are captured into one CUDA
graph, and that graph is replayed back to back for at least --min-seconds
(each replay between CUDA events on the launching stream, with a device
synchronize before the first and after the last), so that the SM clock is
sampled under load; ms_per_step is the median replay time over K.  Rank 0
prints one JSON line.  Under torchrun each rank runs its own batch (requests
are independent: no data-path collective), so scaling is weak and the value
is the sum over ranks over the slowest rank's time.
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
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="5b", help="workload: 1, 2, 3, 4, 5a, 5b")
    ap.add_argument("--mode", choices=["sample", "greedy"], default="sample")
    ap.add_argument("--min-seconds", type=float, default=1.5,
                    help="replay the K-step graph back to back for at least this long")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layout", choices=["padded", "packed"], default="padded",
                    help="padded [B][G+1][V] rows, or packed rows with a cu_draft prefix")
    ap.add_argument("--read", choices=["lazy", "eager"], default="lazy",
                    help="request claims: read a sampled request's positions one at a time, "
                         "stopping at the first rejection (lazy, the default), or all rows first")
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


def base_seed(config: str) -> int:
    return 620 + int(config[0])


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


def workload_desc(w, mode, sha):
    from speculative_decoding_verification_62_gb300 import workloads as W
    return {"workload": f"config {w.name}: {W.CONFIGS[w.name]['desc']}", "B": w.B,
            "gamma_max": w.G, "gamma_sum": w.gamma_sum(), "V": w.V, "mode": mode,
            "input_sha256": sha}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def _oracle_call(inp, mode, nthreads):
    import oracle
    B = len(inp["gamma"])
    if mode == "sample":
        return oracle.sample(**inp, nthreads=nthreads, rows_first=B < nthreads)
    return oracle.greedy(inp["target"], inp["draft_tokens"], inp["gamma"], nthreads=nthreads)


def _subset(w, n):
    from speculative_decoding_verification_62_gb300 import workloads as W
    return W.oracle_inputs(w, list(range(n)) if n < w.B else None)


def cpu_baseline(w, mode, budget_s=8.0):
    """The float64 oracle as it stands, on the host cores: one call on the
    whole batch with every thread (OpenMP over requests, and over rows first
    when the batch has fewer requests than threads), then a bounded sample of
    the batch (its first requests) on one thread.  Returns the baseline dict
    and the full-batch oracle result (for the parity counts)."""
    cores = os.cpu_count() or 1
    full = _subset(w, w.B)
    t0 = time.perf_counter()
    ref = _oracle_call(full, mode, cores)
    t_all = time.perf_counter() - t0
    calls = 1
    while time.perf_counter() - t0 < 1.0:  # small batches: repeat to a second
        _oracle_call(full, mode, cores)
        calls += 1
    t_all = (time.perf_counter() - t0) / calls
    per_req_1t = t_all * min(cores, w.B) / w.B  # about one thread's time per request
    n1 = max(1, min(w.B, int(budget_s / max(per_req_1t, 1e-9))))
    sub = _subset(w, n1)
    t1 = time.perf_counter()
    _oracle_call(sub, mode, 1)
    t1 = time.perf_counter() - t1
    g = w.gamma.cpu().numpy()
    v_all = float(g.sum()) / t_all
    v_1 = float(g[:n1].sum()) / t1
    used = cores if mode == "sample" and w.B < cores else min(cores, w.B)
    return {"value": v_all, "unit": UNIT, "cores": used, "kind": "oracle",
            "value_1thread": v_1,
            "sample": f"float64 C oracle on the host: {calls} call(s) of the full batch of "
                      f"config {w.name} ({w.B} requests) on {used} of {cores} threads "
                      f"({t_all:.3f} s per call; OpenMP over "
                      f"{'rows, then requests' if mode == 'sample' and w.B < cores else 'requests'}); "
                      f"value_1thread: the first {n1} requests on 1 thread ({t1:.2f} s)"}, ref


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch  # noqa: F401  (inputs are drawn with torch's CPU generator)
    from speculative_decoding_verification_62_gb300 import workloads as W
    w = W.make(args.config)
    sha = w.sha256()
    cores = os.cpu_count() or 1
    # each step: the oracle on the first n requests, n sized to about a second
    t0 = time.perf_counter()
    _oracle_call(_subset(w, 1), args.mode, cores)
    per_req = max(time.perf_counter() - t0, 1e-6)
    n = max(1, min(w.B, int(1.0 * min(cores, w.B) / per_req)))
    inp = _subset(w, n)
    gsum = int(w.gamma[:n].sum())
    for _ in range(args.warmup):
        _oracle_call(inp, args.mode, cores)
    t = []
    for _ in range(args.steps):
        t1 = time.perf_counter()
        _oracle_call(inp, args.mode, cores)
        t.append(time.perf_counter() - t1)
    total = sum(t)
    value = gsum * args.steps / total
    used = cores if args.mode == "sample" and n < cores else min(cores, n)
    sample = (f"each step is one call of the float64 C oracle on the first {n} of the "
              f"{w.B} requests of config {w.name} on {used} of {cores} host threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_desc(w, args.mode, sha), requests_per_step=n),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": sample},
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
        power = [num(r[3]) or 0.0 for r in rows]
        pmax = max(power)
        # under load: samples within 70 % of the highest power seen
        load = [r for r, p in zip(rows, power) if p >= 0.7 * pmax] or rows
        sm = [num(r[1]) for r in load if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in load for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": pmax}


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

    # each rank draws its own batch (different seed): weak scaling by request.
    # The batch is drawn on the CPU and copied, so its bytes do not depend on
    # the device (the same bytes as the reference arm and the CPU baseline).
    host_w = W.make(args.config, seed=rank_seed(base_seed(args.config), rank))
    sha = host_w.sha256()
    base = host_w.to(dev)
    mode = args.mode
    B, G, V = base.B, base.G, base.V
    binding.spec_verify_set_schedule({"auto": binding.SCHEDULE_AUTO,
                                      "stream": binding.SCHEDULE_STREAM,
                                      "persistent": binding.SCHEDULE_PERSISTENT}[args.schedule])
    binding.spec_verify_set_lazy(args.read == "lazy")
    route, csize = binding.spec_verify_route(base.target.dtype, B, G, V, greedy=mode == "greedy")
    # request claims read lazily: sampling from two requests per CTA (one CTA
    # per SM; on the pipeline kernel), greedy whenever requests are claimed
    # (two CTAs per SM)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    lazy = args.read == "lazy" and (route == binding.ROUTE_PIPELINE or (
        route == binding.ROUTE_CLAIMS and (B >= 2 * sms if mode == "sample" else B > 2 * sms)))
    kernel = {binding.ROUTE_CLUSTER: "cluster_kernel", binding.ROUTE_STREAM: "stream_kernel",
              binding.ROUTE_CLAIMS: "stream_kernel", binding.ROUTE_PIPELINE: "pipe_kernel",
              binding.ROUTE_PERSISTENT: "verify_kernel"}[route]
    upto = (", positions read one at a time up to the first "
            + ("rejection" if mode == "sample" else "mismatch")) if lazy else ""
    schedule = {binding.ROUTE_CLUSTER: f"resident clusters of {csize} CTAs, one per request",
                binding.ROUTE_STREAM: f"streaming clusters of {csize} CTAs, one per request",
                binding.ROUTE_CLAIMS: "streaming CTAs claiming requests in turn, longest first"
                                      + upto,
                binding.ROUTE_PIPELINE: "one CTA per SM with two requests in flight, claimed in "
                                        "turn, longest first" + upto,
                binding.ROUTE_PERSISTENT: "persistent grid"}[route]
    # the persistent grid runs batches of more than 1536 requests as several launches
    launches_per_call = math.ceil(B / 1536) if route == binding.ROUTE_PERSISTENT else 1

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
    K = args.steps
    ncopy = max(2, math.ceil(4 * l2 / per_copy))
    ncopy = min(ncopy, max(2, int(0.3 * torch.cuda.mem_get_info(dev)[0] // per_copy)))
    if K % ncopy == 1:  # the next replay's first step must not reread the last step's copy
        ncopy += 1
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
    # The K timed steps are captured once into a CUDA graph, so the device
    # time is not bounded by the Python launch path (which the e2e number
    # below includes).
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cap = torch.cuda.current_stream(dev)
            for i in range(K):
                step(i, cap)
        graph.replay()  # one untimed replay
        torch.cuda.synchronize(dev)
    status = binding.spec_verify_status(v.workspace, stream)
    if status:
        raise RuntimeError(f"device status flags: {binding.status_names(status)}")

    def run_k():
        if graph is not None:
            graph.replay()
        else:
            for i in range(K):
                step(i)

    # replays needed for --min-seconds, from one timed replay
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    run_k()
    c1.record(stream)
    torch.cuda.synchronize(dev)
    reps = max(3, min(20000, math.ceil(args.min_seconds * 1e3 / max(c0.elapsed_time(c1), 1e-3))))
    if world > 1:  # every rank replays as often as the slowest needs
        reps = int(across_ranks(float(reps), [], world, dev)[0])
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.4)  # the sampler's first samples
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    for a, b in ev:
        a.record(stream)
        run_k()
        b.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    per_rep = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.median(per_rep)
    emitted_local = int(v.num_accepted.sum().item()) + B
    ms_max, (gsum_all, emitted_all) = across_ranks(
        ms, [base.gamma_sum(), emitted_local], world, dev)
    ms_step = ms_max / K
    value = gsum_all / (ms_step * 1e-3)

    bytes_min = base.bytes_min(mode)
    # roofline of one GPU: this rank's algorithmic bytes (one read of every
    # logit row plus the small inputs and outputs) over its own step time.
    # Read lazily, a call reads only the rows up to each request's first
    # rejection (and the bonus row after a full acceptance); the rate of those
    # bytes, the HBM bandwidth the call actually draws, is reported beside it.
    bytes_need = base.bytes_needed(mode, v.num_accepted, lazy, ctas=sms)
    achieved = bytes_min / (ms / K * 1e-3) / 1e9
    needed = bytes_need / (ms / K * 1e-3) / 1e9
    peak, peak_src = measured_peak_hbm()
    gpu_out = (v.out_tokens.cpu().numpy(), v.num_accepted.cpu().numpy())

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
        k2 = max(10, min(K, 100))
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

    # ---- CPU baseline (the oracle on the host), and parity of this batch ----
    cpu, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, ref = cpu_baseline(host_w, mode)
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        import parity as P
        if packed:
            parity = None  # the oracle runs on the padded batch; packed parity is tested
        elif mode == "sample":
            rep = P.compare_sample(ref, gpu_out[0], gpu_out[1], host_w.gamma.numpy())
            parity = rep.to_dict()
        else:
            parity = {"requests": B, "mismatches": len(P.compare_greedy(ref, *gpu_out))}

    if world > 1:
        dist.barrier()
    if rank == 0:
        cfg = workload_desc(base, mode, sha)
        cfg.update({"layout": args.layout,
                    "schedule": schedule,
                    "parallelism": f"replicas x{world} (independent requests)",
                    "launch": "CUDA-graph replays of the K timed steps" if graph is not None
                              else "one Python call per step",
                    "timing": f"median of {reps} back-to-back timed replays of {K} steps "
                              f"(min {min(per_rep) / K * 1e3:.2f} us, max "
                              f"{max(per_rep) / K * 1e3:.2f} us per step)",
                    "l2": f"inputs larger than L2: rotating {ncopy} device copies of the logits "
                          f"({ncopy * per_copy / 2**20:.0f} MiB; L2 {l2 / 2**20:.0f} MiB)",
                    "emitted_tokens_per_s": emitted_all / (ms_step * 1e-3),
                    "bytes_min_per_step": bytes_min,
                    "bytes_needed_per_step": bytes_need})
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": K, "warmup": args.warmup, "repeats": reps, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if base.target.dtype == torch.bfloat16 else "f32",
                "data": "synthetic", "config": cfg,
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                             "frac": achieved / peak, "peak_source": peak_src,
                             "bytes": "one read of every logit row plus small inputs/outputs",
                             "needed_bytes": bytes_need,
                             "needed_gbs": needed,
                             "needed_frac": needed / peak,
                             "needed_note": ("the call reads each request's rows only up to its "
                                             "first rejection (lazy positions): frac counts every "
                                             "logit, needed_frac the bytes the call reads")
                                            if lazy else "the call reads every row",
                             "traffic": None if packed else profiled_traffic(args.config, mode, kernel),
                             "kernel": kernel + " (one launch per step)"},
                "clocks": clk, "e2e": e2e, "gpu_launches": reps * K * launches_per_call,
                "cpu_baseline": cpu, "parity": parity}
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
