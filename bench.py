"""Throughput of batched speculative-decoding verification on GB300.

One step = one spec_verify call over one batch of the headline workload
(B=256 sequences, K=8 drafts, V=128256, bf16 logits, sampling at T=0.7):
row statistics over every target and draft row, the acceptance scan, and the
residual/bonus draw. Inputs are synthetic (seeded generators), resident in
HBM; two copies of 1.12 GB each are rotated, so no step finds its inputs in
the 129 MB L2.

Prints one JSON line. `value` = verified sequences per second over all ranks.
`roofline` is the row-statistics kernel (pass 1, the dominant one), timed with
CUDA events on its launch stream in a second loop of the same calls (events
between the kernels would break their programmatic-dependent-launch overlap
inside the main timed loop). `e2e` is the same metric
through spec_verify_host (host buffers, copies in the timed region).
`cpu_baseline` is the float64 oracle on this host's cores, on a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference      # the oracle as the reference arm
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified seqs/s and logits HBM GB/s (fraction of GB300 peak) per B×(K+1)×V"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0            # dense bf16, burst (profiling recipe fallback)
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0  # the same, sustained under the power cap
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = ["row_stats.cu", "sv_device.cuh", "sv_internal.h"]


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default=None)
    p.add_argument("--batch", type=int, default=None,
                   help="override B (smaller cases for profiling; not the headline)")
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="wall-clock budget of the CPU-baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--sharded-steps", type=int, default=300,
                   help="timed calls of spec_verify_sharded reported beside the full pass (0: skip)")
    p.add_argument("--shards", type=int, default=8, help="vocabulary shards for that variant")
    p.add_argument("--early-exit-steps", type=int, default=1000,
                   help="timed calls of spec_verify_early_exit reported beside the full pass "
                        "(0: skip)")
    p.add_argument("--filtered-steps", type=int, default=300,
                   help="timed calls of spec_verify_filtered reported beside the full pass "
                        "(0: skip)")
    p.add_argument("--top-k", type=int, default=50, help="top-k of the filtered variant")
    p.add_argument("--top-p", type=float, default=0.9, help="top-p of the filtered variant")
    p.add_argument("--lmhead-steps", type=int, default=100,
                   help="timed calls of spec_verify_lmhead (verification from hidden states, "
                        "the LM head fused with the row statistics) reported beside the full "
                        "pass; 0 = skip")
    p.add_argument("--cpu-threads", type=int, default=0,
                   help="threads for the CPU baseline (0: every core this process may use)")
    return p.parse_args()


def tensor_peaks():
    """(burst, sustained) dense bf16 TFLOP/s and their source."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    return FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _code_of(name: str) -> bytes:
    """A source file without its comments and blank space, so that the sha
    below changes with the code a capture measured, not with its comments."""
    text = open(os.path.join(ROOT, "speculative_decoding_verification_66_gb300", "csrc", name)).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split()).encode()


def kernel_sha():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(_code_of(f))
    return h.hexdigest()[:16]


def profiled_traffic(wl):
    """DRAM bytes per pass-1 launch for this workload, from a committed ncu
    summary (profiles/row_stats_*.md) that names the workload and batch it was
    scaled to and was taken on the current kernel source; None otherwise."""
    want = f"{wl.name} B={wl.B}"
    sha = kernel_sha()
    for path in sorted(glob.glob(os.path.join(PROFILE_DIR, "row_stats_*.md"))):
        text = open(path).read()
        m_wl = re.search(r"traffic_workload:\s*(.+)", text)
        m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
        m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.e+]+)", text)
        if m_wl and m_sha and m_tr and m_wl.group(1).strip() == want and m_sha.group(1) == sha:
            return float(m_tr.group(1))
    return None


LM_SOURCES = ["lmhead.cu", "sv_device.cuh", "sv_internal.h", "sv_stages.h"]


def lm_kernel_sha():
    h = hashlib.sha256()
    for f in LM_SOURCES:
        h.update(_code_of(f))
    return h.hexdigest()[:16]


def profiled_lm_traffic(lw):
    """DRAM bytes per statistics-GEMM launch for this LM-head workload, from a
    committed ncu summary (profiles/lmhead_*.md) taken at this batch on the
    current kernel source; None otherwise."""
    want = f"{lw.name} B={lw.B}"
    sha = lm_kernel_sha()
    for path in sorted(glob.glob(os.path.join(PROFILE_DIR, "lmhead_*.md"))):
        text = open(path).read()
        m_wl = re.search(r"traffic_workload:\s*(.+)", text)
        m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
        m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.e+]+)", text)
        if m_wl and m_sha and m_tr and m_wl.group(1).strip() == want and m_sha.group(1) == sha:
            return float(m_tr.group(1))
    return None


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i] == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": rows[0][1],
                "reasons": reasons, "samples": len(rows)}


def cpu_baseline(wl, host_fn, budget_s: float, threads: int = 0):
    """Time the oracle (as it stands) on this host's cores on a bounded sample of
    the workload: the batch's sequences split over threads, repeated until about
    `budget_s` seconds of wall time have passed."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    if threads > 0:
        cores = min(cores, threads)
    cores = max(1, min(cores, wl.B))  # the oracle splits by sequence
    mode = 0 if wl.mode == "sample" else 1
    t, d, x = host_fn(wl.B)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.verify(t, d, x, wl.temperature, 0x5EED0000 + reps, mode, threads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            break
    return {"value": wl.B * reps / el, "unit": "seqs/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} pass(es) over the {wl.B} sequences of one batch ({wl.label}), "
                      f"float64 C oracle, {cores} threads splitting the sequences, {el:.1f} s wall"}


def reference_arm(args, wl):
    """The oracle timed as the reference arm: each step verifies a bounded
    sample of the workload's sequences on the host's cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch

    import oracle
    from speculative_decoding_verification_66_gb300.workloads import make_inputs, to_host_arrays
    cores = len(os.sched_getaffinity(0))
    inputs = make_inputs(wl.resized(B=max(cores, 1)), 0, "cpu")
    t, d, x = to_host_arrays(inputs)
    mode = 0 if wl.mode == "sample" else 1
    t0 = time.perf_counter()
    oracle.verify(t[:1], None if d is None else d[:1], x[:1], wl.temperature, 1, mode)
    one = time.perf_counter() - t0
    # Size each step so that warm-up plus timed steps stay near two minutes.
    per_step = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(cores, per_step * cores / max(one, 1e-6))))
    for w in range(args.warmup):
        oracle.verify(t[:n], None if d is None else d[:n], x[:n], wl.temperature, w, mode,
                      threads=min(n, cores))
    t0 = time.perf_counter()
    for s in range(args.steps):
        oracle.verify(t[:n], None if d is None else d[:n], x[:n], wl.temperature, 100 + s, mode,
                      threads=min(n, cores))
    el = time.perf_counter() - t0
    value = n * args.steps / el
    del torch
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "seqs/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl),
            "cpu_baseline": {"value": value, "unit": "seqs/s", "cores": min(n, cores),
                             "kind": "oracle",
                             "sample": f"{n} sequence(s) of {wl.label} per step"},
            "e2e": {"value": value, "unit": "seqs/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def early_exit_bytes(nacc, K: int, V: int, es: int, mode: str):
    """Logit bytes spec_verify_early_exit reads for these outcomes, and the
    ideal (rows up to each emitted position only). Its phases cover positions
    [0, 1), [1, 3), [3, 7), ... (lengths 1, 2, 4, ...); a sequence decided at
    position j takes part in every phase that starts at or before j. Sampling
    adds the re-read of the emitted row pair."""
    sampling = mode == "sample"
    phases, p0, ln = [], 0, 1
    while p0 <= K:
        nt = min(ln, K + 1 - p0)
        nd = max(0, min(ln, K - p0)) if sampling else 0
        phases.append((p0, nt, nd))
        p0 += ln
        ln *= 2
    read = ideal = 0
    for j in nacc:
        if j < 0:  # invalid: the first phase read its rows, then it stopped
            read += phases[0][1] + phases[0][2]
            continue
        read += sum(nt + nd for p0, nt, nd in phases if p0 <= j)
        ideal += (j + 1) + (min(j + 1, K) if sampling else 0)
        if sampling:
            again = 2 if j < K else 1
            read += again
            ideal += again
    return read * V * es, ideal * V * es


def max_over_ranks(x: float, dist=None) -> float:
    """The slowest rank's time: every rank's timed region is bracketed by
    barriers, and the job is done when the last rank is."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, seqs_per_rank: int, steps: int, elapsed_s: float) -> float:
    """Weak scaling: every rank verifies its own batch each step, so the job
    verifies world * seqs_per_rank sequences per step."""
    return world * seqs_per_rank * steps / elapsed_s


def config_of(wl):
    return {"workload": wl.label, "B": wl.B, "K": wl.K, "V": wl.V, "logits_dtype": wl.dtype,
            "mode": wl.mode, "temperature": wl.temperature,
            "l2": "inputs larger than L2: two 1.1 GB input sets rotated between steps",
            "parallelism": "independent replicas per GPU (weak scaling, no collective)"}


def main():
    args = parse()
    from speculative_decoding_verification_66_gb300.workloads import HEADLINE, WORKLOADS
    wl = WORKLOADS[args.workload or HEADLINE]
    if args.batch is not None:
        wl = wl.resized(B=args.batch)
    if args.impl == "reference":
        reference_arm(args, wl)
        return

    import torch

    import speculative_decoding_verification_66_gb300 as sv
    from speculative_decoding_verification_66_gb300.workloads import make_inputs, to_host_arrays

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sv.load()

    copies = [make_inputs(wl, 1000 * rank + c, dev) for c in range(2)]
    seeds = [0x5EED0002 + c for c in range(2)]
    B, K, V = wl.B, wl.K, wl.V
    es = 2 if wl.dtype == "bf16" else 4
    mode = wl.mode
    out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    nacc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = torch.empty(sv.sv_workspace_bytes(B, K, V, copies[0]["target"].dtype, mode),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # Per-copy outcome (deterministic for a fixed seed): bytes the step must move.
    rows_pass1 = B * (K + 1) + (B * K if mode == "sample" else 0)
    step_bytes = []
    accepted = []
    for c, inp in enumerate(copies):
        sv.spec_verify(inp["target"], inp["draft"], inp["tokens"], wl.temperature, seeds[c], mode,
                       out_tokens=out, num_accepted=nacc, workspace=ws)
        n = nacc.cpu()
        accepted.append(n.float().mean().item())
        rejected = int(((n >= 0) & (n < K)).sum())
        bonus = int((n == K).sum())
        reread = (2 * rejected + bonus) if mode == "sample" else 0
        step_bytes.append(es * V * (rows_pass1 + reread) + 4 * B * K + 4 * B * (K + 2))
    pass1_bytes = es * V * rows_pass1

    def step(i, ev=None):
        c = i & 1
        inp = copies[c]
        if ev is None:
            sv.spec_verify(inp["target"], inp["draft"], inp["tokens"], wl.temperature, seeds[c],
                           mode, out_tokens=out, num_accepted=nacc, workspace=ws, stream=stream)
        else:
            sv.spec_verify_timed(inp["target"], inp["draft"], inp["tokens"], ev, wl.temperature,
                                 seeds[c], mode, out_tokens=out, num_accepted=nacc, workspace=ws,
                                 stream=stream)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # Timed region: K plain calls (kernels chained by programmatic dependent
    # launch, no events in between).
    with ClockSampler(local) as clocks:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            step(i)
        stop.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), dist)
    # Stage times: the same calls with events recorded on the launch stream
    # between the kernels (this serialises the kernels, so it is timed apart).
    n_staged = max(3, min(args.steps, 300))
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_staged)]
    for i in range(n_staged):
        step(i, events[i])
    torch.cuda.synchronize()
    pass1_ms = sum(e[0].elapsed_time(e[1]) for e in events) / n_staged
    scan_ms = sum(e[1].elapsed_time(e[2]) for e in events) / n_staged
    sample_ms = sum(e[2].elapsed_time(e[3]) for e in events) / n_staged
    ms_per_step = elapsed_ms / args.steps
    value = job_throughput(world, B, args.steps, elapsed_ms / 1e3)
    mean_bytes = sum(step_bytes[i & 1] for i in range(args.steps)) / args.steps
    peak, peak_src = peaks()
    step_gbs = mean_bytes / (ms_per_step / 1e3) / 1e9
    pass1_gbs = pass1_bytes / (pass1_ms / 1e3) / 1e9

    # The early-exit entry on the same inputs (a variant, reported beside the
    # full pass): same outputs, fewer rows read.
    early = None
    if args.early_exit_steps > 0:
        ws_ee = torch.empty(sv.sv_early_exit_workspace_bytes(B, K, V, copies[0]["target"].dtype,
                                                             mode), dtype=torch.uint8, device=dev)

        def ee_step(i):
            c = i & 1
            inp = copies[c]
            sv.spec_verify_early_exit(inp["target"], inp["draft"], inp["tokens"], wl.temperature,
                                      seeds[c], mode, out_tokens=out, num_accepted=nacc,
                                      workspace=ws_ee, stream=stream)

        ee_bytes = []
        for c in range(2):
            ee_step(c)
            ee_bytes.append(early_exit_bytes(nacc.cpu().tolist(), K, V, es, mode))
        for i in range(3):
            ee_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.early_exit_steps):
            ee_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        ee_ms = max_over_ranks(e0.elapsed_time(e1), dist) / args.early_exit_steps
        read = sum(ee_bytes[i & 1][0] for i in range(2)) / 2
        ideal = sum(ee_bytes[i & 1][1] for i in range(2)) / 2
        early = {"value": job_throughput(world, B, 1, ee_ms / 1e3), "unit": "seqs/s",
                 "ms_per_step": ee_ms, "steps": args.early_exit_steps,
                 "bytes_read_per_step": read, "bytes_ideal_per_step": ideal,
                 "hbm_gbs": read / (ee_ms / 1e3) / 1e9}

    # The sharded entry on the same logits split into G vocabulary shards (a
    # variant, reported beside the full pass).
    sharded = None
    G = args.shards
    if args.sharded_steps > 0 and G > 1 and V % G == 0:
        Vs = V // G
        shard_sets = []
        for inp in copies:
            ts = [inp["target"][..., g * Vs:(g + 1) * Vs].contiguous() for g in range(G)]
            ds = ([inp["draft"][..., g * Vs:(g + 1) * Vs].contiguous() for g in range(G)]
                  if mode == "sample" else None)
            shard_sets.append((ts, ds))
        ws_sh = torch.empty(sv.sv_sharded_workspace_bytes(B, K, Vs, G, copies[0]["target"].dtype,
                                                          mode), dtype=torch.uint8, device=dev)

        def sh_step(i):
            c = i & 1
            ts, ds = shard_sets[c]
            sv.spec_verify_sharded(ts, ds, copies[c]["tokens"], wl.temperature, seeds[c], mode,
                                   out_tokens=out, num_accepted=nacc, workspace=ws_sh,
                                   stream=stream)

        for i in range(3):
            sh_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.sharded_steps):
            sh_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        sh_ms = max_over_ranks(e0.elapsed_time(e1), dist) / args.sharded_steps
        # With shard widths of whole 16-byte vectors the sampler reads the
        # shards directly; otherwise a gather reads and writes the pairs once more.
        gathered = mode == "sample" and (Vs * es) % 16 != 0
        sh_bytes = mean_bytes + (2 * (mean_bytes - pass1_bytes) if gathered else 0)
        sharded = {"shards": G, "value": job_throughput(world, B, 1, sh_ms / 1e3),
                   "unit": "seqs/s", "ms_per_step": sh_ms, "steps": args.sharded_steps,
                   "bytes_per_step": sh_bytes, "hbm_gbs": sh_bytes / (sh_ms / 1e3) / 1e9}
        del shard_sets, ws_sh

    # Top-k / top-p on both rows (a variant, reported beside the full pass):
    # the same logits, drafts redrawn from the filtered draft rows. Two cuts:
    # top-k with top-p (the group-maxima thresholds kernel) and top-p alone
    # (the value-count thresholds kernel).
    def run_filtered(tk, tp):
        from speculative_decoding_verification_66_gb300.workloads import draw_from_logits
        gen = torch.Generator(device=dev)
        gen.manual_seed(4321 + rank)
        f_tokens = [draw_from_logits(c["draft"], wl.temperature, gen, tk, tp) for c in copies]
        ws_f = torch.empty(sv.sv_filtered_workspace_bytes(B, K, V, copies[0]["target"].dtype,
                                                          mode), dtype=torch.uint8, device=dev)

        def f_step(i, ev=None):
            c = i & 1
            inp = copies[c]
            sv.spec_verify_filtered(inp["target"], inp["draft"], f_tokens[c], wl.temperature, tk,
                                    tp, seeds[c], mode, out_tokens=out, num_accepted=nacc,
                                    workspace=ws_f, stream=stream, events=ev)

        f_acc = []
        for c in range(2):
            f_step(c)
            f_acc.append(nacc.float().mean().item())
        for i in range(3):
            f_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.filtered_steps):
            f_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        f_ms = max_over_ranks(e0.elapsed_time(e1), dist) / args.filtered_steps
        n_f = max(3, min(args.filtered_steps, 100))
        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_f)]
        for i in range(n_f):
            f_step(i, fev[i])
        torch.cuda.synchronize()
        thr_ms = sum(e[0].elapsed_time(e[1]) for e in fev) / n_f
        f_scan_ms = sum(e[1].elapsed_time(e[2]) for e in fev) / n_f
        f_sample_ms = sum(e[2].elapsed_time(e[3]) for e in fev) / n_f
        # The thresholds pass must read every row once (further sweeps of a
        # row are meant to hit L2): the same algorithmic bytes as pass 1.
        thr_gbs = pass1_bytes / (thr_ms / 1e3) / 1e9
        res = {"top_k": tk, "top_p": tp, "value": job_throughput(world, B, 1, f_ms / 1e3),
               "unit": "seqs/s", "ms_per_step": f_ms, "steps": args.filtered_steps,
               "mean_accepted": sum(f_acc) / len(f_acc),
               "stage_ms": {"thresholds": thr_ms, "scan": f_scan_ms, "sample": f_sample_ms,
                            "steps_timed": n_f},
               "thresholds_kernel": {"kernel": "hist_kernel" if tk == 0 or tk > 64
                                     else "filter_kernel",
                                     "bound": "hbm", "achieved": thr_gbs, "peak": peak,
                                     "unit": "GB/s", "frac": thr_gbs / peak,
                                     "algorithmic_bytes": pass1_bytes}}
        del ws_f, f_tokens
        return res

    filtered = filtered_top_p = None
    if args.filtered_steps > 0 and mode == "sample":
        filtered = run_filtered(args.top_k, args.top_p)
        if args.top_p < 1.0:
            filtered_top_p = run_filtered(0, args.top_p)

    # Verification from the models' last hidden states (a variant, reported
    # beside the full pass): the LM heads run on the tensor cores with the row
    # statistics fused, so no logits are written; only the emitted pairs'
    # logits are made, by a second GEMM. Output matrices of 1.05 GB (target)
    # and 0.5 GB (draft) stream from HBM every step, larger than L2.
    lmhead = None
    if args.lmhead_steps > 0:
        from speculative_decoding_verification_66_gb300.workloads import (LM_WORKLOADS,
                                                                           make_lmhead_inputs)
        lw = LM_WORKLOADS["lm_llama3_bf16" if mode == "sample" else "lm_greedy_bf16"].resized(
            B=B, K=K, V=V, temperature=wl.temperature)
        lin = make_lmhead_inputs(lw, 77 + rank, dev)
        ws_l = torch.empty(sv.sv_lmhead_workspace_bytes(B, K, V, lw.d_target, lw.d_draft, mode),
                           dtype=torch.uint8, device=dev)

        def l_step(i, ev=None):
            sv.spec_verify_lmhead(lin["hidden_t"], lin["weight_t"], lin["hidden_d"],
                                  lin["weight_d"], lin["tokens"], lw.temperature, seeds[i & 1],
                                  mode, out_tokens=out, num_accepted=nacc, workspace=ws_l,
                                  stream=stream, events=ev)

        l_step(0)
        l_acc = nacc.float().mean().item()
        for i in range(3):
            l_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.lmhead_steps):
            l_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        l_ms = max_over_ranks(e0.elapsed_time(e1), dist) / args.lmhead_steps
        n_l = max(3, min(args.lmhead_steps, 50))
        lev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_l)]
        for i in range(n_l):
            l_step(i, lev[i])
        torch.cuda.synchronize()
        st = [sum(e[k].elapsed_time(e[k + 1]) for e in lev) / n_l for k in range(4)]
        Dt, Dd = lw.d_target, lw.d_draft
        rows_d = B * K if mode == "sample" else 0
        stats_flops = 2 * V * (B * (K + 1) * Dt + rows_d * Dd)
        pair_flops = 2 * V * B * (Dt + (Dd if rows_d else 0)) if mode == "sample" else 0
        tpk, tpk_sus, tsrc = tensor_peaks()
        stats_tf = stats_flops / (st[0] / 1e3) / 1e12
        lmhead = {"workload": lw.label, "value": job_throughput(world, B, 1, l_ms / 1e3),
                  "unit": "seqs/s", "ms_per_step": l_ms, "steps": args.lmhead_steps,
                  "mean_accepted": l_acc,
                  "stage_ms": {"stats_gemm": st[0], "scan": st[1], "pair_gemm": st[2],
                               "sample": st[3], "steps_timed": n_l},
                  "stats_kernel": {"bound": "tensor", "achieved": stats_tf, "peak": tpk,
                                   "unit": "TFLOP/s", "frac": stats_tf / tpk,
                                   "frac_of_sustained": stats_tf / tpk_sus, "flops": stats_flops,
                                   "algorithmic_bytes": V * 2 * (Dt + (Dd if rows_d else 0)) +
                                   2 * (B * (K + 1) * Dt + rows_d * Dd),
                                   "traffic": profiled_lm_traffic(lw),
                                   "peak_source": f"{tsrc} bf16_tflops (burst)"}}
        if pair_flops:
            # Near the ridge: its floor is the larger of the tensor time and the
            # time to stream both output matrices once more.
            pair_tf = pair_flops / (st[2] / 1e3) / 1e12
            wbytes = V * 2 * (Dt + Dd)
            floor_ms = max(pair_flops / (tpk * 1e12), wbytes / (peak * 1e9)) * 1e3
            lmhead["pair_kernel"] = {"bound": "tensor+hbm (ridge)", "achieved": pair_tf,
                                     "peak": tpk, "unit": "TFLOP/s", "frac": pair_tf / tpk,
                                     "flops": pair_flops, "weight_bytes": wbytes,
                                     "weight_gbs": wbytes / (st[2] / 1e3) / 1e9,
                                     "floor_ms": floor_ms, "frac_of_floor": floor_ms / st[2]}
        # End to end from host memory: the output matrices stay resident on the
        # device (model parameters); every step copies its hidden states and
        # draft tokens in from pinned host buffers and its results back out.
        hin = {k: lin[k].cpu().pin_memory() for k in ("hidden_t", "hidden_d", "tokens")
               if lin[k] is not None}
        din = {k: torch.empty_like(lin[k]) for k in hin}
        h_lo = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
        h_ln = torch.empty((B,), dtype=torch.int32).pin_memory()

        def l_e2e(i):
            for k in hin:
                din[k].copy_(hin[k], non_blocking=True)
            sv.spec_verify_lmhead(din["hidden_t"], lin["weight_t"], din.get("hidden_d"),
                                  lin["weight_d"], din["tokens"], lw.temperature, seeds[i & 1],
                                  mode, out_tokens=out, num_accepted=nacc, workspace=ws_l,
                                  stream=stream)
            h_lo.copy_(out, non_blocking=True)
            h_ln.copy_(nacc, non_blocking=True)

        n_le = max(3, min(args.lmhead_steps, 20))
        for i in range(2):
            l_e2e(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n_le):
            l_e2e(i)
        torch.cuda.synchronize()
        le_s = max_over_ranks(time.perf_counter() - t0, dist)
        lmhead["e2e"] = {"value": job_throughput(world, B, n_le, le_s), "unit": "seqs/s",
                         "h2d_bytes_per_step": sum(t.numel() * t.element_size()
                                                   for t in hin.values()),
                         "d2h_bytes_per_step": h_lo.numel() * 4 + h_ln.numel() * 4,
                         "steps": n_le, "resident": "output matrices (model parameters)"}
        del lin, ws_l, din, hin

    # End to end through the host entry point: pinned host inputs, copies inside.
    e2e_steps = args.e2e_steps if args.e2e_steps is not None else max(3, min(args.steps, 20))
    h = [{k: (v.cpu().pin_memory() if v is not None else None) for k, v in c.items()}
         for c in copies]
    # Consecutive steps alternate between two streams, each with its own staging
    # buffer and result buffers, as a serving loop would run them: one step's
    # host-to-device copy overlaps the previous step's kernels. Every step still
    # copies its own inputs in and its results out inside the timed region.
    slots = 2
    h_out = [torch.empty((B, K + 1), dtype=torch.int32).pin_memory() for _ in range(slots)]
    h_nacc = [torch.empty((B,), dtype=torch.int32).pin_memory() for _ in range(slots)]
    staging = [torch.empty(sv.sv_host_staging_bytes(B, K, V, copies[0]["target"].dtype, mode),
                           dtype=torch.uint8, device=dev) for _ in range(slots)]
    e2e_streams = [stream] + [torch.cuda.Stream(dev) for _ in range(slots - 1)]

    def e2e_step(i):
        c, q = i & 1, i % slots
        sv.spec_verify_host(h[c]["target"], h[c]["draft"], h[c]["tokens"], wl.temperature,
                            seeds[c], mode, out_tokens=h_out[q], num_accepted=h_nacc[q],
                            staging=staging[q], device=dev, stream=e2e_streams[q],
                            synchronize=False)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    for st in e2e_streams:
        st.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist)
    h2d = sum(t.numel() * t.element_size() for t in h[0].values() if t is not None)
    d2h = h_out[0].numel() * 4 + h_nacc[0].numel() * 4
    del staging

    if rank != 0:
        if dist:
            dist.barrier()
        return
    line = {
        "metric": METRIC, "value": value, "unit": "seqs/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config_of(wl),
        "hbm_gbs": step_gbs, "hbm_frac": step_gbs / peak,
        "stage_ms": {"row_stats": pass1_ms, "scan": scan_ms, "sample": sample_ms,
                     "steps_timed": n_staged},
        "mean_accepted": sum(accepted) / len(accepted),
        "roofline": {"kernel": "row_stats", "bound": "hbm", "achieved": pass1_gbs, "peak": peak,
                     "unit": "GB/s", "frac": pass1_gbs / peak, "traffic": profiled_traffic(wl),
                     "algorithmic_bytes": pass1_bytes, "peak_source": f"{peak_src} hbm_gbs"},
        "e2e": {"value": job_throughput(world, B, e2e_steps, e2e_s), "unit": "seqs/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "streams": slots},
        "clocks": clocks.summary(),
        "gpu_launches": sv.launches(mode, V, copies[0]["target"].dtype) * args.steps,
    }
    if early is not None:
        line["early_exit"] = early
    if sharded is not None:
        line["sharded"] = sharded
    if filtered is not None:
        line["filtered"] = filtered
    if filtered_top_p is not None:
        line["filtered_top_p"] = filtered_top_p
    if lmhead is not None:
        line["lmhead"] = lmhead
    if world == 1 and not args.no_cpu_baseline:
        def host_fn(n):
            sub = {k: (v[:n] if v is not None else None) for k, v in copies[0].items()}
            return to_host_arrays(sub)
        line["cpu_baseline"] = cpu_baseline(wl, host_fn, args.cpu_seconds, args.cpu_threads)
    print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()


if __name__ == "__main__":
    main()
