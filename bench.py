"""Benchmark of the DSpark Markov-head draft hot path on GB300.

One step = one draft block for one batch: the fused Markov-head draft with the
confidence head over B = 128 requests, K = 16 positions, V = 151936, r = 256
(d = 2048, survival threshold 0.3, T = 1.0), i.e. every sampled token, its
log-probability, the confidence values, survival products and verify lengths.

Printed (rank 0, one JSON line): draft tokens/s for the whole job (value),
device-timed with CUDA events over the draft kernel with inputs resident in
HBM and the L2 flushed between steps; the same metric end to end (e2e)
through the binding with host buffers (pinned host -> device copies of the
step's inputs and device -> host copies of its outputs inside the timed
region); the roofline of the draft kernel against the measured HBM peak; SM
clocks sampled during the timed region; and the fp64 CPU oracle timed on a
bounded sample of the same workload (cpu_baseline).

``--impl reference`` times that oracle alone, per step one bounded sample of
the workload, on the host cores (rank 0 only under torchrun).
Multi-GPU: independent replicas, each rank drafts its own batch (weak scaling,
no collective on the data path; the only collectives are the timing barrier
and the max over ranks).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Markov-head draft tokens/s at B=128 K=16 V=151936; % of HBM roofline"
VERIFY_METRIC = "verified draft tokens/s (speculative verification) at B=128 K=16 V=151936"
LABEL_METRIC = "acceptance labels/s (1 - TV of draft and target) at B=128 K=16 V=151936"
SCHEDULE_METRIC = "load-aware verify-window schedules/s at R=128 requests K=16"
STS_METRIC = "sequential temperature scaling fits/s at N=8192 rows K=16"
# the scheduler is one CTA: one SM's 32-bit lanes at the maximum clock
SM_LANE_OPS = 128 * 2.07e9
# the STS fit is one 16-CTA cluster; each cross-entropy evaluation needs four transcendental
# results (exponential, reciprocal, two logarithms), and an SM's special-function units
# deliver 16 a clock
STS_CLUSTER_SMS = 16
STS_SFU_OPS = STS_CLUSTER_SMS * 16 * 2.07e9
STS_SFU_PER_EVAL = 4
L2_FLUSH_BYTES = 512 << 20       # larger than the 129 MB L2
CONF_THRESHOLD = 0.3

WORKLOADS = {
    # name: (config index, description)
    "serving": (2, "serving batch + confidence: B=128 K=16 V=151936 r=256 d=2048"),
    "single": (1, "single request: B=1 K=16 V=151936 r=256"),
    "gated": (3, "gated head: B=64 K=16 V=151936 r=256 d=4096"),
    "rnn": (5, "RNN head (decay and input gates from h): B=64 K=16 V=151936 r=256 d=4096"),
    "selector": (4, "selector top-16 (gated): B=256 K=16 V=151936 r=256 d=4096"),
    "tiny": (0, "tiny: B=1 K=4 V=4096 r=256"),
    "verify": (2, "speculative verification of the serving batch: B=128 K=16 V=151936 r=256, "
                  "synthetic target logits (draft base logits + N(0,1)), T_draft = T_target = 1"),
    "label": (2, "acceptance labels of the serving batch's drafted block: B=128 K=16 V=151936 "
                 "r=256, synthetic target logits (draft base logits + N(0,1)), "
                 "T_draft = T_target = 1"),
    "schedule": (None, "load-aware prefix scheduler: R=128 requests x K=16 extensions, survival "
                       "products of U(0.4, 0.995) confidences, smooth saturating SPS(B)"),
    "sts": (None, "sequential temperature scaling: N=8192 calibration rows x K=16, raw "
                  "confidences of a head 2.5x too sharp, 0/1 acceptance outcomes"),
}
SMALL = {"schedule": dict(R=128, K=16, seed=3003), "sts": dict(N=8192, K=16, seed=3004)}
VERIFY_TARGET_SEED = 2002


def verify_bytes(c: dict) -> int:
    """Bytes one full-window verification must move: every verified target row and
    the bonus row, then, for the draw, W2, each request's base-logit row, its
    embedding row and its target row again."""
    B, K, V, r = c["B"], c["K"], c["V"], c["r"]
    return B * (K + 1) * V * 4 + r * V * 2 + B * V * 4 + B * r * 2 + B * V * 4


def label_bytes(c: dict) -> int:
    """Bytes the labels of a drafted block must move at least once: every base-logit
    row and target row of the K positions, W2 once, the gathered embeddings."""
    B, K, V, r = c["B"], c["K"], c["V"], c["r"]
    return 2 * B * K * V * 4 + r * V * 2 + B * K * r * 2


def metric_of(workload: str) -> str:
    return {"verify": VERIFY_METRIC, "label": LABEL_METRIC, "schedule": SCHEDULE_METRIC,
            "sts": STS_METRIC}.get(workload, METRIC)


def schedule_ops(R: int, K: int) -> int:
    """Element-steps of the scheduler: the bitonic network over the candidates padded to a
    power of two (every stage touches every element), the prefix sum and the cut."""
    n = 1
    while n < R * K:
        n <<= 1
    lg = n.bit_length() - 1
    return n * lg * (lg + 1) // 2 + 2 * R * K


def sts_ops(N: int, K: int) -> int:
    """Special-function results of the fit: four per cross-entropy evaluation, one evaluation
    per row, position, round and grid point."""
    return STS_SFU_PER_EVAL * N * K * 8 * 32


def algorithmic_bytes(cfg: int, c: dict) -> int:
    """Bytes the step must move at least once per position (W2 + U + gathers [+ h, Wg])."""
    B, K, V, r = c["B"], c["K"], c["V"], c["r"]
    if cfg == 4:
        d = c["d"]
        # U scan + 32 gathered rows of A/B per (b, t) + candidate ids and score tables
        # written + the gate's h and Wg
        return (B * K * V * 4 + 2 * B * K * 16 * r * 2 + B * K * (16 * 4 + 16 * 16 * 4)
                + B * K * d * 2 + d * r * 2)
    per_step = r * V * 2 + B * V * 4 + B * r * 2
    total = K * per_step
    if c.get("confidence"):
        total += B * K * c["d"] * 2
    if c.get("gated"):
        total += B * K * c["d"] * 2 + c["d"] * r * 2
    if c.get("rnn"):
        total += c["d"] * r * 2  # the decay gate's weights (h is counted once above)
    return total


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="serving")
    ap.add_argument("--temperature", type=float, default=1.0,
                    help="sampling temperature (0 = greedy); the workloads are quoted at 1.0")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
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


def replica_seed(rank: int, step: int) -> int:
    """Independent replicas draw independent samples: the Philox key differs per rank."""
    return (rank << 32) | step


def job_throughput(tokens_per_rank_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job tokens/s: every rank drafts its own batch; the slowest rank sets the time."""
    return world * tokens_per_rank_step * steps / (max_ms / 1000.0)


def gpu_id(dev) -> str:
    """nvidia-smi -i selector of a torch device (its UUID when torch reports one)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index)


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# Committed ncu summaries by workload, and the sources their kernels are built from:
# a summary's traffic is used only while those sources hash as when it was taken.
_HEADERS = ("sm103.cuh", "philox.cuh", "confidence.cuh", "internal.h")
PROFILES = {
    "serving": ("draft_kernel_serving.md", ("draft.cu",) + _HEADERS),
    "single": ("draft_kernel_single.md", ("draft.cu",) + _HEADERS),
    "label": ("label_step_serving.md",
              ("draft.cu", "label.cu", "rowscan.cuh", "headlogit.cuh") + _HEADERS),
    "verify": ("verify_step_serving.md",
               ("draft.cu", "verify.cu", "rowscan.cuh", "headlogit.cuh") + _HEADERS),
    "selector": ("topk_stream_kernel_selector.md", ("selector.cu", "gate.cu") + _HEADERS),
}


def _code_only(text: str) -> str:
    """C/CUDA source with its comments and blank space removed (none of the kernel
    sources holds a string literal with a comment marker), so that editing a comment
    does not retire a profile taken on the same code."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(" ".join(line.split()) for line in text.splitlines() if line.strip())


def kernel_source_hash(workload: str = "serving") -> str:
    h = hashlib.sha256()
    for name in PROFILES[workload][1]:
        with open(os.path.join(ROOT, "rank_markov_draft_gb300", "csrc", name)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch (per step, for multi-kernel steps) from the committed
    ncu summary, if it was taken on the current kernel sources (else None)."""
    if workload not in PROFILES:
        return None
    path = os.path.join(ROOT, "profiles", PROFILES[workload][0])
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"kernel source hash:\s*`?([0-9a-f]{16})", text)
    m_bytes = re.search(r"dram bytes per launch:\s*`?([0-9]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(workload):
        return None
    return int(m_bytes.group(1))


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(inp, c, n_requests, b0=0, temperature=1.0, seed=0):
    """Run the fp64 oracle on requests b0 .. b0+n-1 of the workload; returns seconds."""
    import oracle
    t0 = time.perf_counter()
    if c.get("gated"):
        # the head's gates of the sampled requests, then their draft
        sl = slice(b0, b0 + n_requests)
        G = oracle.gate(inp.h[sl], inp.Wg)
        if c.get("rnn"):
            A = oracle.gate(inp.h[sl], inp.Wa)
            out = oracle.rnn_draft(inp.U[sl], inp.W1, inp.W2, inp.anchors[sl], A, G=G,
                                   temperature=temperature, seed=seed)
        else:
            out = oracle.markov_draft(inp.U[sl], inp.W1, inp.W2, inp.anchors[sl],
                                      temperature=temperature, seed=seed, H=G)
        return time.perf_counter() - t0
    out = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=temperature,
                              seed=seed, b0=b0, nb=n_requests)
    if c.get("confidence"):
        B = inp.U.shape[0]
        toks = np.zeros((B, c["K"]), np.int32)
        toks[b0:b0 + n_requests] = out["tokens"]
        sl = slice(b0, b0 + n_requests)
        oracle.confidence(inp.h[sl], inp.W1, inp.anchors[sl], toks[sl], inp.w_conf,
                          threshold=CONF_THRESHOLD)
    return time.perf_counter() - t0


def cpu_baseline(inp, c, target_s):
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    K = c["K"]
    done, spent = 0, 0.0
    while spent < target_s and done < c["B"]:
        spent += oracle_sample(inp, c, 1, b0=done)
        done += 1
    return {"value": done * K / spent, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} of {c['B']} requests x {K} positions of the same workload "
                      f"(fp64 oracle, {threads} OpenMP threads, {spent:.1f} s)"}


def verify_cpu_baseline(inp, c, target_s, dtok):
    """The fp64 oracle's verification of whole requests, timed one after the other."""
    import oracle
    from synth import target_logits
    oracle.build()
    threads = oracle.max_threads()
    K, B = c["K"], c["B"]
    tokens = dtok.cpu().numpy()
    P = target_logits(VERIFY_TARGET_SEED, inp.U)
    done, spent = 0, 0.0
    while spent < target_s and done < B:
        t0 = time.perf_counter()
        oracle.verify(P, inp.U, inp.W1, inp.W2, inp.anchors, tokens, draft_temperature=1.0,
                      target_temperature=1.0, seed=done, b0=done, nb=1)
        spent += time.perf_counter() - t0
        done += 1
    return {"value": done * K / spent, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"verification of {done} of {B} requests x {K} positions "
                      f"(fp64 oracle, {threads} OpenMP threads, {spent:.1f} s)"}


def label_cpu_baseline(inp, c, target_s, dtok):
    """The fp64 oracle's labels of whole requests, timed one after the other."""
    import oracle
    from synth import target_logits
    oracle.build()
    threads = oracle.max_threads()
    K, B = c["K"], c["B"]
    tokens = dtok.cpu().numpy() if hasattr(dtok, "cpu") else dtok
    P = target_logits(VERIFY_TARGET_SEED, inp.U)
    done, spent = 0, 0.0
    while spent < target_s and done < B:
        sl = slice(done, done + 1)
        t0 = time.perf_counter()
        oracle.accept_label(P[sl], inp.U[sl], inp.W1, inp.W2, inp.anchors[sl], tokens[sl],
                            draft_temperature=1.0, target_temperature=1.0)
        spent += time.perf_counter() - t0
        done += 1
    return {"value": done * K / spent, "unit": "labels/s", "cores": threads, "kind": "oracle",
            "sample": f"labels of {done} of {B} requests x {K} positions "
                      f"(fp64 oracle, {threads} OpenMP threads, {spent:.1f} s)"}


def small_inputs(workload: str):
    from synth import schedule_inputs, sts_inputs
    c = SMALL[workload]
    if workload == "schedule":
        return schedule_inputs(c["seed"], c["R"], c["K"])
    return sts_inputs(c["seed"], c["N"], c["K"])


def run_reference_small(args, rank, world):
    """The oracle's scheduler or STS fit, one call per step."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    x, y = small_inputs(args.workload)
    c = SMALL[args.workload]

    def one():
        t0 = time.perf_counter()
        if args.workload == "schedule":
            oracle.schedule(x.astype(np.float64), y.astype(np.float64))
        else:
            oracle.sts_fit(x, y)
        return time.perf_counter() - t0
    for _ in range(args.warmup):
        one()
    spent = sum(one() for _ in range(args.steps))
    value = args.steps / spent
    unit = "schedules/s" if args.workload == "schedule" else "fits/s"
    threads = oracle.max_threads()
    print(json.dumps({
        "impl": "reference", "metric": metric_of(args.workload), "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * spent / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload][1], **c},
        "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} whole calls"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_ours_small(args, rank, world, local):
    """The scheduler or the STS fit on the GPU: device time per call, inputs resident, L2
    flushed between calls; roofline against the lanes (scheduler) or special-function units
    (STS fit) of the SMs the kernel runs on."""
    import torch
    from rank_markov_draft_gb300 import binding
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    c = SMALL[args.workload]
    x, y = small_inputs(args.workload)
    X, Y = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    ctx = binding.Context(local, B_max=c.get("R", 1), V_max=8, K_max=c["K"])
    stream = torch.cuda.current_stream(dev)
    if args.workload == "schedule":
        R, K = c["R"], c["K"]
        ell = torch.empty(R, dtype=torch.int32, device=dev)
        theta = torch.empty(1, dtype=torch.float32, device=dev)
        step = lambda: binding.dspark_schedule(ctx, X, R, K, Y, ell, theta, stream)
        ops, unit = schedule_ops(R, K), "schedules/s"
    else:
        N, K = c["N"], c["K"]
        tau = torch.empty(K, dtype=torch.float32, device=dev)
        loss = torch.empty(K, dtype=torch.float32, device=dev)
        step = lambda: binding.dspark_sts_fit(ctx, X, Y, N, K, 1.0 / 64, 64.0, tau, loss, stream)
        ops, unit = sts_ops(N, K), "fits/s"
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(gpu_id(dev))
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.fill_(float(i))
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    if ctx.status() != 0:
        raise RuntimeError(f"device status {ctx.status()} in the timed region")
    per_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms_max = max_over_ranks(sum(per_ms), world, dev)
    value = world * args.steps / (ms_max / 1000.0)
    med = statistics.median(per_ms)
    achieved = ops / (med / 1000.0)
    if args.workload == "schedule":
        peak = SM_LANE_OPS
        peak_source = "one SM's 32-bit lanes (128) at 2070 MHz: the kernel is one CTA by design"
    else:
        peak = STS_SFU_OPS
        peak_source = (f"special-function units of the {STS_CLUSTER_SMS} SMs of the fit's "
                       f"cluster (16 results a clock each) at 2070 MHz; "
                       f"{STS_SFU_PER_EVAL} per evaluation")
    if rank == 0:
        cpu = None
        if not args.skip_cpu:
            import oracle
            oracle.build()
            t0, n = time.perf_counter(), 0
            while time.perf_counter() - t0 < min(args.cpu_seconds, 5.0) or n == 0:
                if args.workload == "schedule":
                    oracle.schedule(x.astype(np.float64), y.astype(np.float64))
                else:
                    oracle.sts_fit(x, y)
                n += 1
            spent = time.perf_counter() - t0
            cpu = {"value": n / spent, "unit": unit, "cores": oracle.max_threads(),
                   "kind": "oracle", "sample": f"{n} whole calls ({spent:.1f} s)"}
        print(json.dumps({
            "metric": metric_of(args.workload), "value": round(value, 1), "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_max / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOADS[args.workload][1], **c,
                       "l2": "flushed between calls (512 MB write)",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "alu", "achieved": round(achieved / 1e9, 3),
                         "peak": round(peak / 1e9, 1), "unit": "Gop/s",
                         "frac": round(achieved / peak, 4), "traffic": None,
                         "peak_source": peak_source,
                         "kernel": "schedule_kernel" if args.workload == "schedule"
                         else "sts_fit_kernel",
                         "ops_per_launch": ops, "median_launch_us": round(med * 1000, 2)},
            "cpu_baseline": cpu, "e2e": None, "clocks": clk, "gpu_launches": args.steps,
        }), flush=True)
    ctx.close()


def run_reference(args, rank, world):
    """The oracle as the reference arm: per step one request of the workload."""
    from synth import CONFIGS, config_inputs
    if args.workload in SMALL:
        run_reference_small(args, rank, world)
        return
    cfg, desc = WORKLOADS[args.workload]
    c = dict(CONFIGS[cfg])
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = config_inputs(cfg)
    K = c["K"]
    if args.workload in ("verify", "label"):
        # the oracle's draft of the batch's first requests, then their verification
        # (or labels)
        from synth import target_logits
        P = target_logits(VERIFY_TARGET_SEED, inp.U)
        n = args.warmup + args.steps
        toks = np.zeros((c["B"], K), np.int32)
        toks[:n] = oracle.markov_draft(inp.U, inp.W1, inp.W2, inp.anchors, temperature=1.0,
                                       seed=77, nb=min(n, c["B"]))["tokens"]

        def one(b):
            t0 = time.perf_counter()
            if args.workload == "verify":
                oracle.verify(P, inp.U, inp.W1, inp.W2, inp.anchors, toks, draft_temperature=1.0,
                              target_temperature=1.0, seed=b, b0=b % c["B"], nb=1)
            else:
                sl = slice(b % c["B"], b % c["B"] + 1)
                oracle.accept_label(P[sl], inp.U[sl], inp.W1, inp.W2, inp.anchors[sl], toks[sl],
                                    draft_temperature=1.0, target_temperature=1.0)
            return time.perf_counter() - t0
    else:
        def one(b):
            return oracle_sample(inp, c, 1, b0=b % c["B"], temperature=args.temperature)
    for i in range(args.warmup):
        one(i)
    spent = 0.0
    for i in range(args.steps):
        spent += one(args.warmup + i)
    value = args.steps * K / spent
    threads = oracle.max_threads()
    unit = "labels/s" if args.workload == "label" else "tokens/s"
    line = {
        "impl": "reference", "metric": metric_of(args.workload),
        "value": value, "unit": "labels/s" if args.workload == "label" else "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * spent / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "B": c["B"], "K": K, "V": c["V"], "r": c["r"],
                   "sample_per_step": "1 request x K positions"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} steps x 1 request x {K} positions"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def run_ours(args, rank, world, local):
    import torch
    from rank_markov_draft_gb300 import binding
    from synth import CONFIGS, config_inputs

    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    cfg, desc = WORKLOADS[args.workload]
    c = dict(CONFIGS[cfg])
    B, K, V, r = c["B"], c["K"], c["V"], c["r"]
    T = float(args.temperature)
    inp = config_inputs(cfg)

    def up(a, bf=False):
        a = np.ascontiguousarray(a)
        if bf:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    ctx = binding.Context(local, B_max=max(B, 1), V_max=V, K_max=K)
    stream = torch.cuda.current_stream(dev)
    U = up(inp.U)
    anchors = up(inp.anchors)
    if cfg == 4:
        A, Bt, h, Wg = up(inp.A, True), up(inp.Bt, True), up(inp.h, True), up(inp.Wg, True)
        cand = torch.empty(B, K, 16, dtype=torch.int32, device=dev)
        cval = torch.empty(B, K, 16, dtype=torch.float32, device=dev)
        scores = torch.empty(B, K, 16, 16, dtype=torch.float32, device=dev)
        tokens = torch.empty(B, K, dtype=torch.int32, device=dev)
        logprobs = torch.empty(B, K, dtype=torch.float32, device=dev)

        def step(seed):
            binding.dspark_selector_scores(ctx, U, A, Bt, anchors, h, Wg, c["d"], B, K, V, r, 16,
                                           cand, cval, scores, stream)
            n = ctx.last_launches
            binding.dspark_selector_walk(ctx, cand, scores, anchors, A, B, K, V, r, 16, T, seed,
                                         tokens, logprobs, None, stream)
            return n + ctx.last_launches
    elif args.workload == "label":
        from synth import target_logits
        W1, W2 = up(inp.W1, True), up(inp.W2, True)
        P = up(target_logits(VERIFY_TARGET_SEED, inp.U))
        dtok = torch.empty(B, K, dtype=torch.int32, device=dev)
        dlp = torch.empty(B, K, dtype=torch.float32, device=dev)
        binding.dspark_markov_draft(ctx, U, W1, W2, anchors, B, K, V, r, T, 77, dtok, dlp, None,
                                    stream)
        label = torch.empty(B, K, dtype=torch.float32, device=dev)

        def step(seed):
            binding.dspark_accept_label(ctx, P, U, W1, W2, anchors, None, None, 0, dtok, dlp, B, K,
                                        V, r, T, T, label, stream)
            return ctx.last_launches
    elif args.workload == "verify":
        from synth import target_logits
        W1, W2 = up(inp.W1, True), up(inp.W2, True)
        P = up(target_logits(VERIFY_TARGET_SEED, inp.U))
        dtok = torch.empty(B, K, dtype=torch.int32, device=dev)
        dlp = torch.empty(B, K, dtype=torch.float32, device=dev)
        binding.dspark_markov_draft(ctx, U, W1, W2, anchors, B, K, V, r, T, 77, dtok, dlp, None,
                                    stream)
        n_acc = torch.empty(B, dtype=torch.int32, device=dev)
        nxt = torch.empty(B, dtype=torch.int32, device=dev)

        def step(seed):
            binding.dspark_verify(ctx, P, U, W1, W2, anchors, None, None, 0, dtok, dlp, None, B, K,
                                  V, r, T, T, seed, n_acc, nxt, None, stream)
            return ctx.last_launches
    else:
        W1, W2 = up(inp.W1, True), up(inp.W2, True)
        tokens = torch.empty(B, K, dtype=torch.int32, device=dev)
        logprobs = torch.empty(B, K, dtype=torch.float32, device=dev)
        conf = None
        if c.get("confidence"):
            conf = binding.Confidence(h=up(inp.h, True), w=up(inp.w_conf, True), bias=0.0,
                                      threshold=CONF_THRESHOLD).allocate(B, K)
        h = up(inp.h, True) if c.get("gated") else None
        Wg = up(inp.Wg, True) if c.get("gated") else None
        Wa = up(inp.Wa, True) if c.get("rnn") else None

        def step(seed):
            if h is None:
                binding.dspark_markov_draft(ctx, U, W1, W2, anchors, B, K, V, r, T, seed, tokens,
                                            logprobs, conf, stream)
            elif Wa is not None:
                binding.dspark_rnn_draft(ctx, U, W1, W2, anchors, h, Wa, Wg, c["d"], B, K, V, r,
                                         T, seed, tokens, logprobs, conf, stream)
            else:
                binding.dspark_gated_draft(ctx, U, W1, W2, anchors, h, Wg, c["d"], B, K, V, r, T,
                                           seed, tokens, logprobs, conf, stream)
            return ctx.last_launches

    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for i in range(args.warmup):
        step(1000 + i)
    torch.cuda.synchronize(dev)
    if ctx.status() != 0:
        raise RuntimeError(f"device status {ctx.status()} after warm-up")

    # -------- device-timed steps (inputs resident, L2 flushed between steps)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(gpu_id(dev))
    launches = 0
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        starts[i].record(stream)
        launches += step(replica_seed(rank, i))
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    barrier(world)
    clk = clocks.stop()
    if ctx.status() != 0:
        raise RuntimeError(f"device status {ctx.status()} in the timed region")
    per_step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    dev_ms = sum(per_step_ms)
    dev_ms_max = max_over_ranks(dev_ms, world, dev)
    value = job_throughput(B * K, args.steps, world, dev_ms_max)
    ms_per_step = dev_ms_max / args.steps

    # -------- roofline of the dominant kernel
    peak, peak_kind = measured_peaks()
    alg = (verify_bytes(c) if args.workload == "verify" else
           label_bytes(c) if args.workload == "label" else algorithmic_bytes(cfg, c))
    kernel_ms = statistics.median(per_step_ms)
    achieved = alg / (kernel_ms / 1000.0) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(args.workload),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s", "algorithmic_bytes_per_launch": alg,
                "kernel": ("verify step (target-row scan with the acceptance tests and the "
                           "draw's per-row prep, residual draw reading the draw rows in place)"
                           if args.workload == "verify" else
                           "label step (target-row scan with per-row offsets, draft kernel in "
                           "label mode)" if args.workload == "label" else
                           "gates + draft_kernel" if c.get("gated") and cfg != 4 else
                           "draft_kernel" if cfg != 4 else
                           "selector step (top-k scan, gate, pair scores, walk)"),
                "median_launch_us": round(kernel_ms * 1000, 2)}

    # -------- end to end through the binding with host buffers
    e2e = None
    if not args.skip_e2e and cfg != 4 and args.workload not in ("verify", "label", "rnn"):
        e2e = run_e2e(args, ctx, inp, c, dev, stream, conf, W1, W2, h, Wg, world)

    line = None
    if rank == 0:
        cpu = None
        if not args.skip_cpu:
            cpu = (verify_cpu_baseline(inp, c, args.cpu_seconds, dtok) if args.workload == "verify"
                   else label_cpu_baseline(inp, c, args.cpu_seconds, dtok)
                   if args.workload == "label" else cpu_baseline(inp, c, args.cpu_seconds))
        line = {
            "metric": metric_of(args.workload),
            "value": round(value, 1), "unit": "labels/s" if args.workload == "label" else "tokens/s",
            "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": desc, "B": B, "K": K, "V": V, "r": r, "d": c.get("d", 0),
                       "temperature": T, "l2": "flushed between steps (512 MB write)",
                       "inputs_bytes": int(inp.U.nbytes), "parallelism": f"replicas x{world}"},
            "us_per_block": round(ms_per_step * 1000, 2),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": launches, "wall_s_timed_region": round(wall, 4),
        }
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line


def run_e2e(args, ctx, inp, c, dev, stream, conf, W1, W2, h, Wg, world):
    """Same metric with host inputs: every step copies its inputs from pinned host memory and
    reads its outputs back.  The copies run on a second stream into one of two device buffers,
    so step i + 1's inputs cross the host link while step i drafts (a buffer is refilled only
    after the step that read it has finished)."""
    import torch
    from rank_markov_draft_gb300 import binding
    B, K, V, r = c["B"], c["K"], c["V"], c["r"]
    T = float(args.temperature)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    U_h = pin(inp.U)
    anc_h = pin(inp.anchors)
    hc_h = pin(inp.h.view(np.int16)) if conf is not None else None
    U_d = [torch.empty_like(U_h, device=dev) for _ in range(2)]
    anc_d = [torch.empty_like(anc_h, device=dev) for _ in range(2)]
    hc_d = [torch.empty_like(hc_h, device=dev) for _ in range(2)] if hc_h is not None else None
    tok_d = torch.empty(B, K, dtype=torch.int32, device=dev)
    lp_d = torch.empty(B, K, dtype=torch.float32, device=dev)
    outs_h = {"tokens": torch.empty(B, K, dtype=torch.int32).pin_memory(),
              "logprobs": torch.empty(B, K, dtype=torch.float32).pin_memory()}
    conf_e = None
    if conf is not None:
        conf_e = [binding.Confidence(h=hc_d[j], w=conf.w, bias=conf.bias,
                                     threshold=conf.threshold).allocate(B, K) for j in range(2)]
        outs_h.update(conf=torch.empty(B, K).pin_memory(), cumprod=torch.empty(B, K).pin_memory(),
                      verify_len=torch.empty(B, dtype=torch.int32).pin_memory())
    h2d = U_h.numel() * 4 + anc_h.numel() * 4 + (hc_h.numel() * 2 if hc_h is not None else 0)
    d2h = sum(t.numel() * t.element_size() for t in outs_h.values())
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    drafted = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        j = i & 1
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(drafted[j])  # the step that last read buffer j is done
            U_d[j].copy_(U_h, non_blocking=True)
            anc_d[j].copy_(anc_h, non_blocking=True)
            if hc_h is not None:
                hc_d[j].copy_(hc_h, non_blocking=True)
            copied[j].record(copy_stream)

    def draft(i, seed):
        j = i & 1
        stream.wait_event(copied[j])
        ce = conf_e[j] if conf_e is not None else None
        if h is None:
            binding.dspark_markov_draft(ctx, U_d[j], W1, W2, anc_d[j], B, K, V, r, T, seed, tok_d,
                                        lp_d, ce, stream)
        else:
            binding.dspark_gated_draft(ctx, U_d[j], W1, W2, anc_d[j], h, Wg, c["d"], B, K, V, r,
                                       T, seed, tok_d, lp_d, ce, stream)
        drafted[j].record(stream)
        outs_h["tokens"].copy_(tok_d, non_blocking=True)
        outs_h["logprobs"].copy_(lp_d, non_blocking=True)
        if ce is not None:
            outs_h["conf"].copy_(ce.conf, non_blocking=True)
            outs_h["cumprod"].copy_(ce.cumprod, non_blocking=True)
            outs_h["verify_len"].copy_(ce.verify_len, non_blocking=True)

    def steps(n, seed0):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            draft(i, seed0 + i)

    with torch.cuda.stream(stream):
        steps(max(1, args.warmup), 2000)
        torch.cuda.synchronize(dev)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        s.record(stream)
        copy_stream.wait_event(s)  # no copy of the timed steps starts before the start event
        steps(args.steps, 3000)
        e.record(stream)
        torch.cuda.synchronize(dev)
    ms = max_over_ranks(s.elapsed_time(e), world, dev)
    return {"value": round(job_throughput(B * K, args.steps, world, ms), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms / args.steps, 4),
            "overlap": "step i + 1's H2D on a second stream during step i's draft"}


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.workload in SMALL:
        run_ours_small(args, rank, world, local)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
