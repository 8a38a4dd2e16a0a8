#!/usr/bin/env python
"""Throughput of the batched verification step on one GB300.

A step is one pass of the whole hot path over one batch: row statistics of
every verified target and draft row, AV scoring, the left-to-right
acceptance scan, residual/bonus sampling, and one AV refit step (for the
AV-truncated canvas workload also the AV scoring call that trims the canvas
first).  Inputs are seeded synthetic logits resident in HBM; each step uses
its own Philox seed.  The default workload is B=256, K=5, V=128256 bf16
(722 MB of logits per step, larger than the 129 MB L2, so no flush is
needed between steps).

Prints ONE JSON line.  `--impl reference` times the CPU oracle instead (the
only reference this path has), on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified rows/sec (B·(K+1)) and achieved HBM GB/s vs GB300 peak, 1 GPU"
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    "c2": dict(B=64, K=4, V=32000, desc="B=64 K=4 V=32000 bf16, z~N(0,3^2) +8 on one token, draft=z+N(0,1), "
               "tau=1, AV on (omega=1, beta=0), one refit per step"),
    "c3": dict(B=256, K=5, V=128256, desc="B=256 K=5 V=128256 bf16, z~N(0,3^2) with a peaked top token, "
               "draft=0.8z+N(0,1.5^2) (alpha~0.7), tau=1, AV scoring + one refit per step"),
    "c4": dict(B=1024, K=7, V=151936, desc="B=1024 K=7 V=151936 bf16, draft noise sigma_b~U(0.5,3), "
               "tau~U(0.3,1.2), 10% greedy rows, AV scoring + one refit per step"),
    "c5": dict(B=512, K=16, V=128256, desc="B=512 K<=16 V=128256 bf16, AV-truncated canvas (survival >= 0.3), "
               "draft noise 0.5+0.2i, scoring + verify on the kept canvas + one refit per step"),
}


def _dtype_name(dt):
    return {"torch.bfloat16": "bf16", "torch.float32": "f32"}.get(str(dt), str(dt))


def _peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _kernel_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_03_gb300", "csrc")
    for fn in ("rowpass.cu", "api.cu", "rowstats.cuh", "sv_device.cuh", "sv_internal.h", "sample_common.cuh",
               "avfit_common.cuh"):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(workload):
    """DRAM bytes per row-pass launch from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "rowpass_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(workload)
    if not ent or ent.get("kernel_sha") != _kernel_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(device_index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=[], samples=0)
        sm.sort()
        return dict(sm_mhz=sm[len(sm) // 2], sm_max_mhz=max(mx), reasons=sorted(reasons), samples=len(sm))


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _aggregate(elapsed_ms: float, units: float, device):
    """Whole-job timing over the ranks of the default process group: the
    slowest rank's elapsed time (max) and the units all ranks processed
    (sum).  With one process it returns its arguments."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(elapsed_ms), float(units)
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def _bytes_per_step(wl, K, V, esz, kept, accept):
    """Bytes of one step.  Returns (early-exit bytes of the verify row-pass
    launch that the launch events bracket, early-exit bytes of the whole
    step, algorithmic bytes of the bracketed launch).

    Algorithmic bytes (the roofline's numerator): every verified target row
    (k_b + 1 per sequence) and every verified draft row (k_b; on the
    AV-truncated canvas the scoring launch reads the draft rows instead), the
    residual or bonus target row once more (+ the draft row when rejected),
    and 4 B (3K + 4) of small per-sequence inputs and outputs.

    Early-exit bytes: what the acceptance walk cannot avoid -- target rows
    0 .. a_b only (nothing past the first rejection is read) -- plus the same
    draft rows, second pass and small arrays."""
    B = kept.size
    second = int(B + (accept < kept).sum()) * V * esz
    small = 4 * B * (3 * K + 4)
    targets = int((accept + 1).sum()) * V * esz
    if wl == "c5":
        verify_first = targets
        first = verify_first + B * K * V * esz
    else:
        verify_first = first = targets + int(kept.sum()) * V * esz
    # the bracketed verify row pass also samples (second-pass rows) when the
    # rows are 16-byte aligned, as on every workload here
    bracketed = verify_first + second + small
    eager = (int((kept + 1).sum()) + (0 if wl == "c5" else int(kept.sum()))) * V * esz + second + small
    return bracketed, first + second + small, eager


# --------------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import numpy as np
    import torch

    from speculative_decoding_verification_03_gb300 import binding, shard, synth

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    binding.lib()  # fails loudly if the library was not built
    cfg = WORKLOADS[args.workload]
    B, K, V = cfg["B"], cfg["K"], cfg["V"]
    if args.batch:  # a smaller batch of the same rows (profiler captures)
        B = args.batch
    w = getattr(synth, args.workload)(seed=rank, B=B, device=dev)
    theta0 = [1.0] + [0.0] * K if args.workload != "c5" else [0.55] + [0.9 - 0.15 * i for i in range(K)]
    theta = torch.tensor(theta0, dtype=torch.float32, device=dev)
    ws = binding.workspace(B, K, V, dev)
    state = binding.AVState(K, device=dev)
    # every timed step writes its outputs to buffers of its own (nothing is
    # copied inside the timed region to keep the outcomes for the byte count)
    nbuf = max(args.steps, args.warmup)
    outs = [dict(tokens=torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                 accept_len=torch.empty((B,), dtype=torch.int32, device=dev),
                 feature=torch.empty((B, K), dtype=torch.float32, device=dev),
                 conf=torch.empty((B, K), dtype=torch.float32, device=dev)) for _ in range(nbuf)]
    score = None
    if args.workload == "c5":
        score = dict(feature=torch.empty((B, K), dtype=torch.float32, device=dev),
                     conf=torch.empty((B, K), dtype=torch.float32, device=dev),
                     stats=torch.empty((B, K, 4), dtype=torch.int32, device=dev))
        kept = [torch.empty((B,), dtype=torch.int32, device=dev) for _ in range(nbuf)]
    stream = torch.cuda.current_stream(dev)
    # inputs that fit in L2 get it flushed before every timed step (256 MB
    # written), and the steps are then timed by events around each step alone
    first_pass = w.bytes_first_pass()
    flush = torch.zeros(64 << 20, dtype=torch.float32, device=dev) if first_pass <= L2_BYTES else None

    # with several ranks every rank verifies its own block of sequences and
    # the refit is the whole job's: each rank accumulates its labels
    # (round_len 0), the 4K + 2 accumulator values are summed over the ranks
    # (one all-reduce), and every rank solves for the same theta
    sharded = world > 1
    rl = 0 if sharded else 1

    def step(i, seed):
        out = outs[i]
        seed = seed + (rank << 32)  # the ranks' sequences draw independent uniforms
        if score is not None:
            score["kept_len"] = kept[i]
            binding.av_score(w.draft, w.temperature, theta, keep_threshold=0.3, want_stats=True, ws=ws, out=score)
            binding.verify(w.target, w.draft, w.draft_tokens, w.temperature, seed, draft_len=kept[i],
                           theta=theta, draft_stats=score["stats"], want_feature=True, ws=ws, out=out,
                           av_state=state, round_len=rl)
        else:
            binding.verify(w.target, w.draft, w.draft_tokens, w.temperature, seed, theta=theta, want_feature=True,
                           ws=ws, out=out, av_state=state, round_len=rl)
        if sharded:
            shard.end_round(state, theta)

    for i in range(args.warmup):
        step(i, 10**6 + i)
    rc, flags = binding.status(ws)
    if rc != 0:
        raise SystemExit("device status %d (flags %#x) after warm-up" % (rc, flags))

    # per-step events around the row-pass kernel (the dominant kernel)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        a.record(stream)
        b.record(stream)
    step_ev = None
    if flush is not None:
        step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
    clocks = Clocks(local) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        if step_ev is not None:
            _flush_l2(flush)
            step_ev[i][0].record(stream)
        binding.set_launch_events(*ev[i])
        step(i, i)
        if step_ev is not None:
            step_ev[i][1].record(stream)
    binding.set_launch_events(None, None)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks else None
    elapsed_ms = t0.elapsed_time(t1) if step_ev is None else sum(a.elapsed_time(b) for a, b in step_ev)
    rowpass_ms = [a.elapsed_time(b) for a, b in ev]
    rc, flags = binding.status(ws)
    if rc != 0:
        raise SystemExit("device status %d (flags %#x) in the timed region" % (rc, flags))
    # work done: verified rows (sum over sequences of k_b + 1) and algorithmic bytes
    esz = w.target.element_size()
    rows, bytes_rp, bytes_all, bytes_eager = 0, 0, 0, 0
    for i in range(args.steps):
        a = outs[i]["accept_len"].cpu().numpy()
        k = np.full(B, K) if score is None else kept[i].cpu().numpy()
        f, t, e = _bytes_per_step(args.workload, K, V, esz, k, a)
        rows += int((k + 1).sum())
        bytes_rp += f
        bytes_all += t
        bytes_eager += e
    elapsed_ms, rows_all = _aggregate(elapsed_ms, rows, dev)  # max time, summed rows over ranks
    value = rows_all / (elapsed_ms / 1e3)
    # one launch of the row-pass kernel per step (verification, sampling and
    # the refit fused), plus the AV scoring row pass on the truncated canvas;
    # the workspace memset is a driver fill, not a kernel
    launches_per_step = 1 + (1 if score is not None else 0) + (1 if sharded else 0)

    res = dict(metric=METRIC, value=value, unit="rows/s", n_gpus=world, steps=args.steps, warmup=args.warmup,
               ms_per_step=elapsed_ms / args.steps, higher_is_better=True, scaling="weak", vs_baseline=None,
               dtype=_dtype_name(w.target.dtype),
               data="synthetic (seeded; stands in for the pages' model pairs and datasets)")
    peak, peak_kind = _peak()
    # on the AV-truncated canvas both row passes of a step record the same
    # event pair; the later (verify) launch is the one that stays bracketed
    rp_ms = sum(rowpass_ms) / len(rowpass_ms)
    # algorithmic bytes: what the method must read -- target rows 0 .. a_b
    # (the walk stops at the first rejection), every verified draft row (its
    # AV score is an output), the residual or bonus row again, the small
    # per-sequence arrays; fixed by each step's outcome
    ee_bytes = bytes_rp / args.steps
    achieved = ee_bytes / (rp_ms / 1e3) / 1e9
    # the count with every verified target row (k_b + 1 per sequence) read
    # whatever the outcome: an equivalent rate, not a bandwidth
    all_rows = bytes_eager / args.steps
    srt = sorted(rowpass_ms)
    res["roofline"] = dict(bound="hbm", kernel="rowpass_kernel", achieved=achieved, peak=peak, unit="GB/s",
                           frac=achieved / peak, peak_source="%s (MEASURED_PEAKS hbm_gbs)" % peak_kind
                           if peak_kind == "measured" else "fallback 6.8 TB/s",
                           traffic=_traffic(args.workload), algorithmic_bytes_per_launch=ee_bytes,
                           ms_per_launch=rp_ms,
                           ms_per_launch_p10_p50_p90=[srt[len(srt) // 10], srt[len(srt) // 2],
                                                      srt[(9 * len(srt)) // 10]],
                           all_verified_rows_bytes_per_launch=all_rows,
                           equivalent_gbs_all_verified_rows=all_rows / (rp_ms / 1e3) / 1e9)
    res["step_hbm"] = dict(algorithmic_bytes_per_step=bytes_all / args.steps,
                           achieved_gbs=bytes_all / args.steps / (elapsed_ms / args.steps / 1e3) / 1e9)
    res["gpu_launches"] = launches_per_step * args.steps
    res["clocks"] = clk
    res["config"] = dict(workload=args.workload + ": " + cfg["desc"] + (" [batch %d]" % B if args.batch else ""),
                         B=B, K=K, V=V, logits="bf16",
                         global_batch=B * world,
                         l2=("inputs %.0f MB per step > 129 MB L2: no flush" % (first_pass / 1e6)) if flush is None
                         else ("inputs %.0f MB per step fit in the 129 MB L2: 256 MB written before every step; "
                               "steps timed by events around each step alone" % (first_pass / 1e6)),
                         parallelism=("dp%d: a block of B sequences per GPU, one all-reduce of the AV refit "
                                      "accumulators (4K + 2 fp64) per step" % world) if world > 1 else "single GPU")
    if rank == 0 and world == 1 and not args.no_e2e:
        res["e2e"] = run_e2e(args, w, theta0, dev)
    if rank == 0 and world == 1 and not args.no_cpu:
        res["cpu_baseline"] = cpu_baseline(args, budget_s=args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


def run_e2e(args, w, theta0, dev, steps=None):
    """Same metric through the public API with host buffers: each step copies
    its inputs from pinned host memory, verifies, refits, and reads the
    emitted tokens and accept lengths back."""
    import torch

    from speculative_decoding_verification_03_gb300 import binding

    steps = steps or min(args.steps, 20)
    B, K, V = w.B, w.K, w.V
    host = dict(target=w.target.cpu().pin_memory(), draft=w.draft.cpu().pin_memory(),
                draft_tokens=w.draft_tokens.cpu().pin_memory(), temperature=w.temperature.cpu().pin_memory())
    tok_h = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    acc_h = torch.empty((B,), dtype=torch.int32).pin_memory()
    sess = binding.HostSession(B, K, V, w.dtype, dev, theta0)
    for i in range(2):
        sess.step(host, i, tok_h, acc_h)
    torch.cuda.synchronize(dev)
    t = time.perf_counter()
    s = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for i in range(steps):
        sess.step(host, i, tok_h, acc_h)
    e1.record(s)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = tok_h.numel() * 4 + acc_h.numel() * 4
    return dict(value=B * (K + 1) * steps / (ms / 1e3), unit="rows/s", h2d_bytes_per_step=h2d,
                d2h_bytes_per_step=d2h, steps=steps, wall_s=time.perf_counter() - t)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def _oracle_rate(w, K, threads, budget_s, max_seqs=None):
    """Verified rows per second of the oracle (verify + one refit step per
    call) on copies of the workload's sequences until budget_s has passed."""
    import numpy as np

    import oracle

    th = np.array([1.0] + [0.0] * K)
    tgt, drf = synth_logits(w.target), synth_logits(w.draft)
    toks, tau = w.draft_tokens.numpy(), w.temperature.numpy()
    done_rows, done_seqs, calls, t0 = 0, 0, 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s and (max_seqs is None or done_seqs < max_seqs):
        r = oracle.verify(tgt, drf, toks, tau, calls, theta=th, threads=threads)
        fit = oracle.AVFit(th)
        fit.step(r["feature"], r["accept_len"])
        done_rows += int(w.B * (K + 1))
        done_seqs += w.B
        calls += 1
    dt = time.perf_counter() - t0
    return done_rows / dt, done_seqs, dt


def synth_logits(t):
    from speculative_decoding_verification_03_gb300 import synth
    return synth.logits_np(t)


def cpu_baseline(args, budget_s=12.0, max_seqs=None):
    """The oracle as it stands (fp64, plain C) on the host: on every core
    (its sequences split over threads) and on one core, on sequences of the
    same workload, each leg about half of budget_s seconds."""
    from speculative_decoding_verification_03_gb300 import synth

    cfg = WORKLOADS[args.workload]
    B, K, V = cfg["B"], cfg["K"], cfg["V"]
    cores = os.cpu_count() or 1
    n1 = 4 if args.workload != "c4" else 2
    w1 = getattr(synth, args.workload)(seed=0, B=max(n1, 2), device="cpu")
    v1, s1, t1 = _oracle_rate(w1, K, 1, budget_s / 2, max_seqs)
    wn = getattr(synth, args.workload)(seed=0, B=max(2 * cores, n1), device="cpu")
    vn, sn, tn = _oracle_rate(wn, K, cores, budget_s / 2, max_seqs)
    return dict(value=vn, unit="rows/s", cores=cores, kind="oracle", cpu_model=cpu_model(),
                sample="%d sequences of the %s workload (B=%d, K=%d, V=%d) in calls of %d, oracle verify + refit, "
                "sequences split over %d threads, %.1f s" % (sn, args.workload, B, K, V, wn.B, cores, tn),
                single_core=dict(value=v1, cores=1,
                                 sample="%d sequences in calls of %d, one thread, %.1f s" % (s1, w1.B, t1)))


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    import numpy as np

    import oracle
    from speculative_decoding_verification_03_gb300 import synth

    world, rank, _ = _dist()
    if rank != 0:
        return
    oracle.build()
    cfg = WORKLOADS[args.workload]
    B, K, V = cfg["B"], cfg["K"], cfg["V"]
    cores = os.cpu_count() or 1
    # size each step's sample (a multiple of the core count, at most B) so
    # that warm-up + steps take about two minutes on every host core
    pool = min(B, 4 * cores)
    w = getattr(synth, args.workload)(seed=0, B=pool, device="cpu")
    tgt, drf = synth.logits_np(w.target), synth.logits_np(w.draft)
    toks, tau = w.draft_tokens.numpy(), w.temperature.numpy()
    th = np.array([1.0] + [0.0] * K)
    t = time.perf_counter()
    oracle.verify(tgt[:cores], drf[:cores], toks[:cores], tau[:cores], 0, theta=th, threads=cores)
    per_round = time.perf_counter() - t  # one sequence per core
    rounds = int(max(1, min(pool // cores, 120.0 / max(1, args.steps + args.warmup) / per_round)))
    n = min(pool, rounds * cores)

    def step(i):
        s0 = (i * n) % (pool - n + 1)
        sl = slice(s0, s0 + n)
        r = oracle.verify(tgt[sl], drf[sl], toks[sl], tau[sl], i, theta=th, threads=cores)
        fit = oracle.AVFit(th)
        fit.step(r["feature"], r["accept_len"])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = n * (K + 1) * args.steps / dt
    sample = "%d of %d sequences per step (%s workload, V=%d), oracle verify + refit, sequences split over %d " \
        "threads (%s)" % (n, B, args.workload, V, cores, cpu_model())
    res = dict(impl="reference", metric=METRIC, value=value, unit="rows/s", n_gpus=world, steps=args.steps,
               warmup=args.warmup, ms_per_step=dt / args.steps * 1e3, higher_is_better=True, scaling="weak",
               vs_baseline=None, dtype="f64", data="synthetic",
               config=dict(workload=args.workload + ": " + cfg["desc"], B=B, K=K, V=V, logits="bf16"),
               cpu_baseline=dict(value=value, unit="rows/s", cores=cores, kind="oracle", sample=sample),
               e2e=dict(value=value, unit="rows/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(res), flush=True)


# --------------------------------------------------------------------------- the steps around verification
OPS = {
    "budget": "AV global budget: B=512 K=16 confidences (Beta, mean 0.88-0.035i), synthetic cost tables",
    "post": "post-verify update: B=1024 K=7, ragged draft lengths, history capacity 4096",
    "tts": "TTS signal: B=256 K=5 V=128256 bf16 (the c3 rows), weights 0.9^k, KL + bf16 gradient",
    "tree": "tree acceptance: B=256 V=32000 bf16, 16-node trees (levels 3,6,4,2), tau~U(0.4,1.3), 10% greedy",
}


L2_BYTES = 129 * 10**6  # GB300 L2


def _flush_l2(buf):
    buf.add_(1)  # 256 MB written: evicts the 129 MB L2


def run_op(args):
    """Times one of the steps around verification (single GPU) and prints one
    JSON line in the same format as the main benchmark."""
    import numpy as np
    import torch

    from speculative_decoding_verification_03_gb300 import binding, synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.lib()
    stream = torch.cuda.current_stream(dev)
    flush = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    op = args.op
    if op == "budget":
        B, K = 512, 16
        conf, dc, vc = (t.to(dev) for t in synth.budget_inputs(B, K, seed=0))
        out_b = torch.empty(1, dtype=torch.int32, device=dev)
        out_k = torch.empty(B, dtype=torch.int32, device=dev)
        call = lambda i: binding.av_budget(conf, B, dc, vc, out_budget=out_b, out_kept_len=out_k)
        units, unit = B * K, "drafts ranked/s"
        nbytes = B * K * 4 + 2 * (B * K + 1) * 4 + B * 4 + 4
    elif op == "post":
        B, K, H = 1024, 7, 4096
        rng = np.random.default_rng(0)
        kl = rng.integers(0, K + 1, B).astype(np.int32)
        acc = np.array([rng.integers(0, k + 1) for k in kl], np.int32)
        outs = np.full((B, K + 1), -1, np.int32)
        for b in range(B):
            outs[b, :acc[b] + 1] = rng.integers(0, 150000, acc[b] + 1)
        T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        ins, o, a, dl = T(rng.integers(0, 150000, (B, K + 1)).astype(np.int32)), T(outs), T(acc), T(kl)
        sl0 = T(rng.integers(0, H // 2, B).astype(np.int32))
        sl, kv = sl0.clone(), sl0.clone()
        hist = torch.zeros((B, H), dtype=torch.int32, device=dev)
        nxt = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        fl = torch.empty(B, dtype=torch.int32, device=dev)

        def reset():
            sl.copy_(sl0)
            kv.copy_(sl0)

        def call(i):
            binding.post_verify(ins, o, a, sl, kv, history=hist, draft_len=dl, next_in=nxt, flags=fl)
        units, unit = B, "sequences/s"
        nbytes = B * (4 * (K + 1) * 3 + 4 * 5) + int((acc + 1).sum()) * 4
    elif op == "tts":
        w = synth.c3(seed=0, device=dev)
        B, K, V = w.B, w.K, w.V
        wt = torch.tensor([0.9 ** k for k in range(K)], dtype=torch.float32, device=dev)
        kl_out = torch.empty((B, K), dtype=torch.float32, device=dev)
        grad = torch.empty((B, K, V), dtype=torch.bfloat16, device=dev)
        tws = binding.tts_workspace(dev)
        call = lambda i: binding.tts_signal(w.target, w.draft, w.temperature, wt, out_kl=kl_out, out_grad=grad,
                                            workspace=tws)
        units, unit = B * K, "canvas positions/s"
        nbytes = B * K * V * 2 * 3 + B * K * 4  # both rows read once, the gradient written once
    elif op == "tree":
        w = synth.tree(seed=0, B=256, V=32000, device=dev)
        B, N, V = w.B, w.N, w.V
        res = {}

        def call(i):
            res["out"] = binding.verify_tree(w.target, w.draft, w.tokens, w.parents, w.temperature, i)
        units, unit = B, "requests/s"
        nbytes = None  # from the walked paths below
    else:
        raise SystemExit("unknown op " + op)

    for i in range(args.warmup):
        call(10**6 + i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = Clocks(0)
    time.sleep(0.3)
    visited = 0
    for i in range(args.steps):
        _flush_l2(flush)
        if op == "post":
            reset()  # lengths back to the start state, outside the timed launch
        ev[i][0].record(stream)
        call(i)
        ev[i][1].record(stream)
        if op == "tree":
            visited += int((res["out"]["accept_len"] + 1).sum().item()) if i == 0 else 0
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = sorted(a.elapsed_time(b) for a, b in ev)
    mean_ms = sum(ms) / len(ms)
    if op == "tree":
        nbytes = visited * 2 * V * 2  # each visited node's target and draft rows, read once
    value = units / (mean_ms / 1e3)
    peak, kind = _peak()
    achieved = nbytes / (mean_ms / 1e3) / 1e9
    kernel = dict(budget="av_budget_kernel", post="post_verify_kernel", tts="tts_group_kernel", tree="tree_kernel")[op]
    res_line = dict(metric=unit.replace("/s", " per second") + " (" + op + ")", value=value, unit=unit, n_gpus=1,
                    steps=args.steps, warmup=args.warmup, ms_per_step=mean_ms, higher_is_better=True,
                    scaling="weak", vs_baseline=None,
                    dtype=dict(budget="f32", post="int32", tts="bf16", tree="bf16")[op],  # as the verify line: the inputs'
                    data="synthetic",
                    ms_p10_p50_p90=[ms[len(ms) // 10], ms[len(ms) // 2], ms[(9 * len(ms)) // 10]],
                    roofline=dict(bound="hbm", kernel=kernel, achieved=achieved, peak=peak, unit="GB/s",
                                  frac=achieved / peak, traffic=None, algorithmic_bytes_per_launch=nbytes,
                                  peak_source="%s (MEASURED_PEAKS hbm_gbs)" % kind if kind == "measured"
                                  else "fallback 6.8 TB/s"),
                    gpu_launches=args.steps, clocks=clk,
                    config=dict(workload=op + ": " + OPS[op], l2="256 MB written between timed launches",
                                timing="CUDA events around each launch"))
    if not args.no_cpu:
        res_line["cpu_baseline"] = _op_cpu_baseline(op)
    print(json.dumps(res_line), flush=True)


def _op_cpu_baseline(op):
    """The oracle on a bounded sample of the same workload (one host core)."""
    import numpy as np

    import oracle
    from speculative_decoding_verification_03_gb300 import synth

    t0 = time.perf_counter()
    if op == "budget":
        conf, dc, vc = synth.budget_inputs(512, 16, seed=0)
        oracle.av_budget(conf.numpy(), 512, dc.numpy(), vc.numpy())
        units, unit, sample = 512 * 16, "drafts ranked/s", "one call, B=512 K=16"
    elif op == "post":
        rng = np.random.default_rng(0)
        B, K = 1024, 7
        kl = rng.integers(0, K + 1, B)
        acc = np.array([rng.integers(0, k + 1) for k in kl])
        outs = np.full((B, K + 1), 5, np.int32)
        oracle.post_verify(np.zeros((B, K + 1), np.int32), outs, acc, np.zeros(B), np.zeros(B),
                           np.zeros((B, 64), np.int32), draft_len=kl)
        units, unit, sample = B, "sequences/s", "one call, B=1024 K=7"
    elif op == "tts":
        w = synth.c3(seed=0, B=8)
        t = (synth.logits_np(w.target).astype(np.uint32) << 16).view(np.float32)
        d = (synth.logits_np(w.draft).astype(np.uint32) << 16).view(np.float32)
        oracle.tts_signal(t, d, w.temperature.numpy(), [0.9 ** k for k in range(w.K)])
        units, unit, sample = 8 * w.K, "canvas positions/s", "8 requests of the c3 rows"
    else:
        w = synth.tree(seed=0, B=8, V=32000)
        T = (synth.logits_np(w.target).astype(np.uint32) << 16).view(np.float32)
        D = (synth.logits_np(w.draft).astype(np.uint32) << 16).view(np.float32)
        oracle.verify_tree(T, D, w.tokens.numpy(), w.parents.numpy(), w.temperature.numpy(), 0)
        units, unit, sample = 8, "requests/s", "8 requests of the tree workload"
    dt = time.perf_counter() - t0
    return dict(value=units / dt, unit=unit, cores=1, kind="oracle", sample=sample)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="c3")
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences per step instead of the workload's B (for profiler captures on a small case)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--op", choices=["verify"] + sorted(OPS), default="verify",
                    help="verify (the hot path, default) or one of the steps around it")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.op != "verify":
        if args.impl == "reference" or args.gpus != 1:
            raise SystemExit("--op other than verify runs on one GPU, GB300 arm only")
        run_op(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
