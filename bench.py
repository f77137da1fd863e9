#!/usr/bin/env python3
"""Benchmark of the bitwise-reproducible optimizer step on GB300.

One step = replica reduce (R gradient buffers, canonical tree, reciprocal multiply) +
global norm + clip + fused AdamW + Merkle state hash, through the C ABI: by default
repstep_step_fused, one HBM pass from one state buffer into a second whenever the step
does not clip (the benchmark workload never does), else a second pass -- the same bits as
repstep_step, which --two-pass times instead.  Default workload:
n = 1,200,000,000 fp32 parameters, R = 8 fp32 replica gradients N(0, 1e-4) with per-4M-
segment log-uniform scales, hyperparameters lr 3e-4, betas 0.9/0.999, eps 1e-8, wd 0.1,
clip 1.0.  Inputs are synthetic (seeded) and resident in HBM for the device-timed value;
the working set (~77 GB moved per step) is far larger than the 129 MB L2, so no flush is
needed between steps.

Prints ONE JSON line (rank 0).  Metric: parameters per second per bit-exact step, with
the step's algorithmic HBM bytes R*b_g*n + 24n per step as GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain single-threaded restatement of the same
step, the test suite's reference) on the host cores, on a bounded sample of the workload.
Under torchrun with N > 1 every rank runs an independent replica of the whole step (the
single-GPU path does not exchange data); value is the sum over ranks.  --shard runs the
sharded step instead: one model split over the ranks' GPUs, value = n / step time.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "params/s and HBM GB/s (% of roofline) per bit-exact reduce+clip+AdamW+hash step"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
SPEC_HBM_GBS = 8000.0          # the HBM3e figure the metric's own percentage is quoted against
_CSRC = "bitwise_reproducible_step_gb300/csrc/"
# the sources each profiled kernel is built from: a traffic figure recorded under their
# hash stays valid until one of them changes
KERNEL_SOURCES = {k: [_CSRC + f for f in (*srcs, "common.cuh", "kernels.h")]
                  for k, srcs in (("k_reduce", ("k_reduce.cuh",)),
                                  ("k_adamw", ("k_adamw.cuh", "adamw_math.cuh")),
                                  ("k_leaves_b2", ("k_blake2b.cu",)),
                                  ("k_fused", ("k_fused.cuh", "adamw_math.cuh")))}
# BLAKE2b-64 leaves (audit mode) are bound by the SM's integer ALU pipe: per 128-byte block,
# 12 rounds x 8 G functions x 22 32-bit operations (two 3-input and two 2-input 64-bit
# additions at 2 each, four 64-bit XORs at 2, rotations by 24, 16 and 63 at 2 funnel shifts
# each; the rotation by 32 is a word swap), plus the 16 XORs of the feed-forward.
B2_OPS_PER_BLOCK = 12 * 8 * 22 + 16
ALU_LANES_PER_SM = 64           # 4 sub-partitions x 16 lanes of the integer ALU pipe


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; independent replicas)
# ------------------------------------------------------------------------------------
def quiet_nccl():
    """Keep stdout to the one JSON line.  NCCL_DEBUG=VERSION (set in some images) prints a
    version banner on stdout that NCCL_DEBUG_FILE does not redirect, so that level becomes
    WARN for this process; NCCL's debug lines go to stderr."""
    if os.environ.get("NCCL_DEBUG", "").upper() == "VERSION":
        os.environ["NCCL_DEBUG"] = "WARN"
    if os.environ.get("NCCL_DEBUG") and not os.environ.get("NCCL_DEBUG_FILE"):
        os.environ["NCCL_DEBUG_FILE"] = "/dev/stderr"


def dist_init(n_gpus):
    quiet_nccl()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device="cuda") -> float:
    """Slowest rank's time (the job's time) for the weak-scaling replicas."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(params_per_rank: int, ms_max: float, world: int) -> float:
    """Whole-job params/s: every rank runs the whole step on its own replica of the
    workload (no data-path exchange), so the job moves world x n params per step."""
    return params_per_rank / (ms_max * 1e-3) * world


# ------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None      # a private temporary file, read and removed by stop()

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="repstep_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
            if self.path:
                self.fh.close()
                os.remove(self.path)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            lines = fh.readlines()
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------------
# peaks, profiles
# ------------------------------------------------------------------------------------
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 copy measurement)"


def _code_only(text: str) -> str:
    """C++ source without comments and blank space, so that editing a comment keeps a
    recorded traffic figure valid while any change to the code drops it."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel: str):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        h.update(_code_only(open(os.path.join(ROOT, rel), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def alu_peak(dev):
    """Integer ALU pipe peak in T ops/s: SMs x 64 lanes x the maximum SM clock."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    try:
        mhz = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["sm_max_mhz"])
        src = "derived: SMs x 64 ALU lanes x sm_max_mhz of MEASURED_PEAKS.json"
    except (OSError, KeyError, ValueError):
        mhz, src = 2070.0, "derived: SMs x 64 ALU lanes x 2070 MHz (nominal maximum)"
    return sms * ALU_LANES_PER_SM * mhz * 1e6 / 1e12, src


def b2_blocks(n: int) -> int:
    """128-byte BLAKE2b blocks of the audit-mode leaves: the header's one, and ceil(n/32)
    per array (a chunk's 16 KB are 128 blocks, a short last chunk rounds up)."""
    return 1 + 3 * ((n + 31) // 32)


def profiled_traffic(kernel: str):
    """Per-launch DRAM bytes recorded from an ncu capture in profiles/, if the kernel
    sources are unchanged since (the summary stores their hash); else None."""
    src_hash = kernel_source_hash(kernel)
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith(".md"):
            continue
        for line in open(os.path.join(pdir, fn)):
            m = re.match(r"\s*traffic_per_launch:\s*kernel=(\S+)\s+bytes=(\d+)\s+"
                         r"source_hash=(\S+)", line)
            if m and m.group(1) == kernel and m.group(3) == src_hash:
                return int(m.group(2))
    return None


# ------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------
def run_ours(args, rank, world, local):
    from bitwise_reproducible_step_gb300 import inputs as I
    from bitwise_reproducible_step_gb300 import repstep as rs

    wl = I.WORKLOADS[args.workload]
    if args.n:
        import dataclasses
        wl = dataclasses.replace(wl, n=args.n)
    n, R = wl.n, wl.R
    dev = torch.device("cuda", local)
    gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    b_g = 2 if wl.grad_dtype == "bf16" else 4
    hpv = I.default_hparams()

    log(f"[rank {rank}] generating {wl.name}: n={n:,} R={R} on {dev}")
    grads = [I.gen_grad(wl, 1, r, device=dev) for r in range(R)]
    w, m, v = I.gen_state(wl, device=dev)
    pdt = torch.bfloat16 if args.param_dtype == "bf16" else torch.float32
    b_w = 2 if args.param_dtype == "bf16" else 4
    if args.param_dtype == "bf16":
        w = w.to(torch.bfloat16)
    hash_mode = rs.HASH_BLAKE2B if args.hash_mode == "blake2b" else rs.HASH_PF61
    sub_mode = rs.SUBNORMALS_FTZ if args.subnormals == "ftz" else rs.SUBNORMALS_IEEE
    ctx = rs.Repstep(n, grad_dtype=gdt, device=dev, hash_mode=hash_mode, param_dtype=pdt,
                     subnormals=sub_mode, block_threads=args.block_threads)
    if args.decay_mask:
        # a transformer-like layout: no decay on the embedding (first 5%) and on a
        # 4096-element norm gain after every 16.7M-element block of matrices
        segs, e = [(0, False)], n // 20 | 1
        while e < n:
            segs.append((e, True))
            e += 16_777_216 + 3
            if e < n:
                segs.append((e, False))
                e += 4096
        ctx.set_decay_mask(rs.decay_mask_from_segments(n, segs).to(dev))
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)

    def hp(t):
        return rs.hparams(lr=hpv["lr"], beta1=hpv["beta1"], beta2=hpv["beta2"], eps=hpv["eps"],
                          weight_decay=hpv["wd"], clip=hpv["clip"], t=t)

    # the root passes on a second stream, beside the next step's reduce (same bits)
    hash_side = torch.cuda.Stream(dev) if args.hash_stream else None
    ctx.set_hash_stream(hash_side)
    t_step = [0]

    def reduce_only():
        # the paper-exact order (Algorithm 1) when asked for, else the canonical tree
        if args.paper_shard:
            ctx.reduce_paper(grads, args.paper_shard, accum=args.accum or None)
        else:
            ctx.reduce(grads, nodes=args.nodes)

    # one norm and root slot per timed step, read after the timed region
    norms = torch.empty(max(args.steps, 1), dtype=torch.float32, device=dev)
    roots = torch.empty(max(args.steps, 1), dtype=torch.int64, device=dev)

    # the single-pass step writes a second state buffer; the two alternate
    fused_state = None
    if args.fused:
        fused_state = [(w, m, v), (torch.empty_like(w), torch.empty_like(m), torch.empty_like(v))]
    cur = [0]

    # the timed steps' output slots (tensor views), made before the timed region
    timed_out = []

    def one_step(slot=None):
        t_step[0] += 1
        h = hp(t_step[0])
        nr, rt = (norm, root) if slot is None else timed_out[slot]
        if fused_state is not None:
            ctx.step_fused(grads, *fused_state[cur[0]], *fused_state[1 - cur[0]],
                           h, step=t_step[0], norm_out=nr, root_out=rt)
            cur[0] ^= 1
            return
        if not args.paper_shard:
            ctx.step(grads, w, m, v, h, step=t_step[0], norm_out=nr, root_out=rt,
                     nodes=args.nodes)
            return
        reduce_only()
        ctx.clip(h.clip, norm_out=nr)
        ctx.adamw(w, m, v, h)
        ctx.root(t_step[0], root_out=rt)

    # fingerprints that fix the run's bits: the state hash of the initial (w, m, v), and
    # the pre-clip norm and state root after step 1.  They depend only on the workload and
    # the reduction order, so every box and every launch shape must print the same values.
    ctx.hash(0, w, m, v, root_out=root)
    ctx.sync()
    repro = {"initial_state_root": f"{int(root.item()) & (2**64 - 1):016x}"}

    # warm-up (its first step is step 1)
    for i in range(args.warmup):
        one_step()
        if i == 0:
            ctx.sync()
            repro["step1_norm_bits"] = f"{int(norm.view(torch.int32).item()) & 0xFFFFFFFF:08x}"
            repro["step1_norm"] = float(norm.item())
            repro["step1_root"] = f"{int(root.item()) & (2**64 - 1):016x}"
    ctx.sync()

    # ---- timed region: K whole steps, inputs resident in HBM ------------------------
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = ctx.launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] if args.log else []
    # the single pass of every timed step between two events the library records around
    # its launch (repstep_set_pass_events); recorded once here so that they exist
    pass_ev = []
    if fused_state is not None:
        pass_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
        for a_, b_ in pass_ev:
            a_.record(stream)
            b_.record(stream)
        torch.cuda.synchronize(dev)
    t_first = t_step[0] + 1
    timed_out.extend((norms[i:i + 1], roots[i:i + 1]) for i in range(args.steps))
    e0.record(stream)
    for i in range(args.steps):
        if pass_ev:
            ctx.set_pass_events(*pass_ev[i])
        one_step(i)
        if step_ev:
            step_ev[i].record(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    if pass_ev:
        ctx.set_pass_events(None, None)
    clipped_steps = int((norms[:args.steps] > hpv["clip"]).sum().item())
    launches = ctx.launch_count() - launches0
    ms_local = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms_local, world)
    flags = ctx.sync()
    step_records = []
    if step_ev:
        from bitwise_reproducible_step_gb300.policy import f32_bits, root_hex
        nh, rh = norms.cpu().tolist(), roots.cpu().tolist()
        prev = e0
        for i in range(args.steps):
            step_records.append({"workload": wl.name, "step": t_first + i, "norm": nh[i],
                                 "norm_bits": f32_bits(nh[i]), "root": root_hex(rh[i]),
                                 "ms": prev.elapsed_time(step_ev[i])})
            prev = step_ev[i]

    # ---- per-kernel times (same calls, events between them, same stream) ------------
    ctx.set_hash_stream(None)          # the root passes on the timed stream here
    audit = args.hash_mode == "blake2b"
    kt = {"reduce": [], "clip": [], "adamw": [], "root": []}
    if audit:
        kt["leaves"] = []           # the BLAKE2b leaf kernel alone (repstep_leaves)
    # no synchronisation between repetitions: the host stays ahead of the GPU, so each
    # interval is device time, not the host's launch latency (which matters for small n)
    reps = max(3, min(args.steps, 20))
    all_ev = []
    for _ in range(reps + 1):           # the first repetition starts from an idle GPU: dropped
        t_step[0] += 1
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(kt) + 1)]
        h = hp(t_step[0])
        ev[0].record(stream)
        reduce_only()
        ev[1].record(stream)
        ctx.clip(h.clip, norm_out=norm)
        ev[2].record(stream)
        ctx.adamw(w, m, v, h)
        ev[3].record(stream)
        ctx.root(t_step[0], root_out=root)
        ev[4].record(stream)
        if audit:
            ctx.leaves(t_step[0], w, m, v)
            ev[5].record(stream)
        all_ev.append(ev)
    torch.cuda.synchronize(dev)
    for ev in all_ev[1:]:
        for i, k in enumerate(kt):
            kt[k].append(ev[i].elapsed_time(ev[i + 1]))
    kms = {k: statistics.mean(v_) for k, v_ in kt.items()}
    if fused_state is not None:
        # the whole single-pass call (the pass, the norm passes, the three gated two-pass
        # kernels that return at once when the step does not clip, and the root), back to
        # back on one stream
        fev = []
        for _ in range(reps + 1):
            t_step[0] += 1
            e_a = torch.cuda.Event(enable_timing=True)
            e_b = torch.cuda.Event(enable_timing=True)
            e_a.record(stream)
            ctx.step_fused(grads, *fused_state[cur[0]], *fused_state[1 - cur[0]],
                           hp(t_step[0]), step=t_step[0], norm_out=norm, root_out=root)
            cur[0] ^= 1
            e_b.record(stream)
            fev.append((e_a, e_b))
        torch.cuda.synchronize(dev)
        kms["fused_step"] = statistics.mean(a_.elapsed_time(b_) for a_, b_ in fev[1:])
        kms["fused_pass"] = statistics.mean(a_.elapsed_time(b_) for a_, b_ in pass_ev)
    ctx.sync()

    # ---- checkpoint image emit (timed on its own; not part of the step's bytes) --------
    img = torch.empty(rs.image_bytes(n), dtype=torch.uint8, device=dev)
    im_ev = []
    for _ in range(4):                  # back to back, the first dropped as above
        e_a = torch.cuda.Event(enable_timing=True)
        e_b = torch.cuda.Event(enable_timing=True)
        e_a.record(stream)
        ctx.image_write(t_step[0], w, m, v, img)
        e_b.record(stream)
        im_ev.append((e_a, e_b))
    torch.cuda.synchronize(dev)
    del img
    im_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in im_ev[1:])
    image_emit = {"bytes": rs.image_bytes(n), "dst": "device buffer", "ms": im_ms,
                  "gbs_read_plus_write": (b_w + 8 + 12) * n / (im_ms * 1e-3) / 1e9}

    peak, peak_src = hbm_peak()
    mask_b = 0.125 if args.decay_mask else 0.0
    alg_step = int((R * b_g + 16 + 2 * b_w + mask_b) * n)
    alg = {"reduce": (R * b_g + 4) * n, "adamw": int((20 + 2 * b_w + mask_b) * n),
           "fused_pass": int((R * b_g + 16 + 2 * b_w + mask_b) * n)}
    dom = max(("reduce", "adamw", "leaves") if audit else ("reduce", "adamw"),
              key=lambda k: kms[k])
    # the single pass carries the step when no timed step clipped (a step after one that
    # clipped takes the two passes, whose kernels the per-kernel loop times)
    fused_ran = (fused_state is not None and not audit and clipped_steps == 0 and
                 "fused_pass" in kms)
    if fused_ran:
        dom = "fused_pass"
    kname = {"reduce": "k_reduce", "adamw": "k_adamw", "leaves": "k_leaves_b2",
             "fused_pass": "k_fused"}[dom]
    traffic = profiled_traffic(kname)
    if dom == "leaves":
        apeak, apeak_src = alu_peak(dev)
        ops = b2_blocks(n) * B2_OPS_PER_BLOCK
        achieved = ops / (kms[dom] * 1e-3) / 1e12
        roofline = {"bound": "alu", "kernel": kname, "achieved": achieved, "peak": apeak,
                    "unit": "Tops/s", "frac": achieved / apeak, "traffic": traffic,
                    "alg_ops_per_launch": ops, "ops_per_128B_block": B2_OPS_PER_BLOCK,
                    "avg_launch_ms": kms[dom], "peak_source": apeak_src}
    else:
        achieved = alg[dom] / (kms[dom] * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak,
                    "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                    "alg_bytes_per_launch": alg[dom], "avg_launch_ms": kms[dom],
                    "peak_source": peak_src}
        if dom == "fused_pass":
            roofline["timed"] = ("k_fused alone, every step of the timed region: CUDA events "
                                 "the library records on its stream just before and after "
                                 "the launch (repstep_set_pass_events)")

    # ---- end to end: grads from pinned host memory each step, norm+root read back ----
    ctx.set_hash_stream(hash_side)
    e2e = None if args.skip_e2e else run_e2e(args, ctx, wl, grads, w, m, v, hp, t_step, dev,
                                              R, b_g, n, world)

    del grads
    torch.cuda.empty_cache()
    cpu = None
    variant = (args.param_dtype != "f32" or args.decay_mask or args.hash_mode != "pf61"
               or args.subnormals != "ieee" or bool(args.paper_shard) or args.nodes > 1)
    if rank == 0 and not args.skip_cpu_baseline and not variant:
        cpu = cpu_baseline(wl, n, R, dev, args.cpu_seconds)

    value = job_value(n, ms, world)
    step_gbs = alg_step / (ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "n_params": n, "replicas": R,
                   "grad_dtype": wl.grad_dtype, "grad_dist": f"{wl.grad} sigma={wl.sigma}",
                   "bytes_alg_per_step": alg_step,
                   "l2": "inputs larger than L2 (no flush needed): "
                         f"{(R * b_g + (24 if args.fused else 32)) * n / 1e9:.1f} GB "
                         "moved per step",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "launch": "persistent grid (SM count x resident CTAs), "
                             f"{args.block_threads or 512} compute threads",
                   "hash_leaves": args.hash_mode, "param_dtype": args.param_dtype,
                   "decay_mask": bool(args.decay_mask), "subnormals": args.subnormals,
                   "hash_stream": bool(args.hash_stream),
                   "step": ("repstep_step_fused: one HBM pass when the step does not clip, "
                            "two state buffers alternating" if args.fused else
                            "repstep_step: reduce, then clip and AdamW (two HBM passes)"),
                   "reduce_order": (f"paper-exact, dp_shard {args.paper_shard}"
                                    + (f", accum {args.accum}" if args.accum else "")
                                    if args.paper_shard else
                                    "canonical tree" + (f", staged over {args.nodes} nodes"
                                                        if args.nodes > 1 else ""))},
        "hbm_gbs_step": step_gbs,
        "roofline_step": {"bound": "hbm", "achieved": step_gbs, "peak": peak,
                          "unit": "GB/s", "frac": step_gbs / peak, "peak_source": peak_src,
                          "bytes": "R*b_g*n + (16 + 2*b_w)n (+ n/8 with a decay mask) "
                                   "algorithmic bytes per step",
                          "spec_peak": SPEC_HBM_GBS, "frac_of_spec": step_gbs / SPEC_HBM_GBS},
        "roofline": roofline,
        "kernel_ms": kms,
        "clocks": clk,
        "gpu_launches": launches,
        "device_flags": flags,
        "clipped_steps": clipped_steps,
        "repro": repro,
        "image_emit": image_emit,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if args.log and rank == 0:
        from bitwise_reproducible_step_gb300.policy import StepLog
        log_ = StepLog(args.log)
        for r in step_records:
            log_.write(r)
        log_.write({"summary": res})
    return res


def run_sharded(args, rank, world, local):
    """The sharded step (bitwise_reproducible_step_gb300/shard.py): the workload's n split
    into `world` chunk-aligned ranges, one per GPU; each rank holds R/world replica gradients
    of the whole model and its range of the state.  A step is the routing of gradient
    slices, the local reduce (by default the single pass, into a second state buffer), the
    chunk-sum all-gather, the gathered norm and clip, AdamW on the range (when the single
    pass does not stand), the leaf all-gather and the gathered root.  Total work is fixed as the world
    grows (strong scaling): value = n / step time.  One rank routes nothing: it reads its own
    replicas' slices in place."""
    import torch.distributed as dist
    from bitwise_reproducible_step_gb300 import inputs as I
    from bitwise_reproducible_step_gb300 import repstep as rs
    from bitwise_reproducible_step_gb300 import shard as S

    wl = I.WORKLOADS[args.workload]
    if args.n:
        import dataclasses
        wl = dataclasses.replace(wl, n=args.n)
    n, R = wl.n, wl.R
    if R % world:
        raise SystemExit(f"--shard needs the replica count {R} to be a multiple of {world}")
    dev = torch.device("cuda", local)
    gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    b_g = 2 if wl.grad_dtype == "bf16" else 4
    hpv = I.default_hparams()
    step = S.ShardedStep(n, R, rank, world, dev, grad_dtype=gdt)
    plan, Rl = step.plan, R // world
    lo, hi = plan.range_of(rank)
    log(f"[rank {rank}] sharded {wl.name}: n={n:,} R={R}, range [{lo:,}, {hi:,}) of {world}")
    grads = []
    for j in range(Rl):
        grads.append(I.gen_grad(wl, 1, rank * Rl + j, device=dev))
    w_all, m_all, v_all = I.gen_state(wl, device=dev)
    w, m, v = (x[lo:hi].clone() for x in (w_all, m_all, v_all))
    del w_all, m_all, v_all
    torch.cuda.empty_cache()
    # the single-pass step writes a second state buffer; the two alternate
    bufs = [(w, m, v), tuple(torch.empty_like(x) for x in (w, m, v))] if args.fused else None
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    t_step = [0]

    def one():
        t_step[0] += 1
        h = rs.hparams(lr=hpv["lr"], beta1=hpv["beta1"], beta2=hpv["beta2"], eps=hpv["eps"],
                       weight_decay=hpv["wd"], clip=hpv["clip"], t=t_step[0])
        if bufs is not None:
            step.step_fused(grads, *bufs[(t_step[0] - 1) % 2], *bufs[t_step[0] % 2], h,
                            t_step[0], norm_out=norm, root_out=root)
        else:
            step.step(grads, w, m, v, h, t_step[0], norm_out=norm, root_out=root)

    repro = {}
    for i in range(args.warmup):
        one()
        if i == 0:
            step.ctx.sync()
            repro = {"step1_norm_bits": f"{int(norm.view(torch.int32).item()) & 0xFFFFFFFF:08x}",
                     "step1_root": f"{int(root.item()) & (2**64 - 1):016x}"}
    step.ctx.sync()
    clocks = ClockSampler(local)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = step.ctx.launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    peak, peak_src = hbm_peak()
    alg_step = (R * b_g + 24) * n
    step_gbs = alg_step / (ms * 1e-3) / 1e9
    return {
        "metric": METRIC, "value": n / (ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "n_params": n, "replicas": R,
                   "grad_dtype": wl.grad_dtype, "bytes_alg_per_step": alg_step,
                   "parallelism": f"sharded over {world} chunk-aligned ranges (point-to-point "
                                  "routing of gradient slices, all-gathers of chunk sums "
                                  "and leaves)",
                   "step": ("ShardedStep.step_fused: the single pass on each range, state "
                            "buffers alternating" if args.fused else "ShardedStep.step"),
                   "l2": f"inputs larger than L2: {(R * b_g + (24 if args.fused else 32)) * n / 1e9:.1f} "
                         "GB per step"},
        "hbm_gbs_step": step_gbs,
        "roofline_step": {"bound": "hbm", "achieved": step_gbs / world, "peak": peak,
                          "unit": "GB/s per GPU", "frac": step_gbs / world / peak,
                          "peak_source": peak_src},
        "clocks": clk,
        "gpu_launches": step.ctx.launch_count() - launches0,
        "repro": repro,
        "e2e": {"value": None, "unit": UNIT,
                "skipped": "sharded mode: gradients resident on the device"},
        "cpu_baseline": None,
    }


def host_fits(need: int, world: int, avail: int | None = None, device="cuda"):
    """Whether every rank can pin `need` bytes of host memory for the end-to-end leg: the
    ranks of one host (LOCAL_WORLD_SIZE) pin theirs at the same time, so together they may
    take at most 60% of the host's available memory.  Every rank gets the same answer (a
    max over ranks), so none waits in a collective that another one skipped.  Returns
    (fits, reason)."""
    on_node = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    if avail is None:
        try:
            avail = int(re.search(r"MemAvailable:\s+(\d+)",
                                  open("/proc/meminfo").read()).group(1)) * 1024
        except (OSError, AttributeError):
            avail = 0
    fits = not (avail and need * on_node > 0.6 * avail)
    if max_over_ranks(0.0 if fits else 1.0, world, device=device) > 0.0:
        return False, (f"pinned host gradients need {need * on_node / 1e9:.1f} GB on a host; "
                       f"a rank's host has {avail / 1e9:.1f} GB available")
    return True, ""


def run_e2e(args, ctx, wl, grads, w, m, v, hp, t_step, dev, R, b_g, n, world=1):
    """The same step end to end through the C ABI's host-buffer call
    (repstep_step_from_host): every step copies the R gradients from pinned host memory --
    pipelined over chunk-aligned ranges and copy streams, each range reduced as it lands --
    and returns the pre-clip norm and the Merkle root in host memory.  The state (w, m, v)
    stays resident on the device, as an optimizer's state does.  Under torchrun every rank
    does the same on its own replica; the value is the job's (n x world over the slowest
    rank's step time)."""
    need = R * b_g * n
    fits, why = host_fits(need, world)
    if not fits:
        return {"value": None, "unit": UNIT, "skipped": why}
    host = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in grads]
    for h, g in zip(host, grads):
        h.copy_(g)
    steps = max(2, min(args.e2e_steps, args.steps))

    def one():
        t_step[0] += 1
        return ctx.step_from_host(host, grads, w, m, v, hp(t_step[0]), step=t_step[0],
                                  pieces=args.e2e_pieces, copy_streams=args.e2e_copy_streams)

    # the copy floor on this machine: the same bytes host-to-device with nothing else running.
    # The host link is noisy (plain copies of the same 38.4 GB took 182 to 254 ms in one
    # process), so it is sampled 4 times: the fastest is the floor, the median the typical
    # copy.
    side = torch.cuda.Stream(dev)
    floor = []
    for _ in range(4):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(side):
            for h, g in zip(host, grads):
                g.copy_(h, non_blocking=True)
        side.synchronize()
        floor.append(time.perf_counter() - t0)
    one()
    torch.cuda.synchronize(dev)
    per_step = []
    t0 = time.perf_counter()
    for _ in range(steps):
        t1 = time.perf_counter()
        one()
        per_step.append((time.perf_counter() - t1) * 1e3)
    dt = max_over_ranks((time.perf_counter() - t0) / steps, world)
    del host
    fl = min(floor)
    fl_med = statistics.median(floor)
    return {"value": n * world / dt, "unit": UNIT, "ms_per_step": dt * 1e3, "steps": steps,
            "h2d_bytes_per_step": need, "d2h_bytes_per_step": 4 + 8,
            "api": "repstep_step_from_host (C ABI, host gradient buffers, host norm and root)",
            "state": "w, m, v resident on the device",
            "pieces": args.e2e_pieces, "copy_streams": args.e2e_copy_streams,
            "step_ms": [round(x, 2) for x in per_step],
            "h2d_gbs_achieved": round(need / dt / 1e9, 1),
            "h2d_copy_floor_ms": round(fl * 1e3, 2),
            "h2d_copy_gbs": round(need / fl / 1e9, 1),
            "h2d_copy_ms_samples": [round(x * 1e3, 1) for x in floor],
            "frac_of_copy_floor": round(fl / dt, 3),
            "frac_of_median_copy": round(fl_med / dt, 3)}


def cpu_baseline(wl, n, R, dev, seconds):
    """The oracle (plain C, one thread) on the host cores, on the first n_s elements of the
    bench's own workload; repeated until about `seconds` of CPU work."""
    from bitwise_reproducible_step_gb300 import inputs as I
    from oracle import oracle as O

    n_s = min(n, 1 << 24)
    grads = [I.to_numpy(I.gen_grad(wl, 1, r, device=dev)[:n_s]) for r in range(R)]
    w, m, v = (t[:n_s].cpu().numpy() for t in I.gen_state(wl, device=dev))
    hpv = I.default_hparams()
    done, t0, reps = 0, time.perf_counter(), 0
    while True:
        out = O.step(grads, w, m, v, lr=hpv["lr"], beta1=hpv["beta1"], beta2=hpv["beta2"],
                     eps=hpv["eps"], wd=hpv["wd"], clip=hpv["clip"], t=reps + 1)
        w, m, v = out["w"], out["m"], out["v"]
        done += n_s
        reps += 1
        if time.perf_counter() - t0 > seconds or reps >= 8:
            break
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {n_s:,} of {n:,} params of the same workload, R={R}, "
                      f"{reps} full steps (reduce+norm+clip+AdamW+hash) in {dt:.1f} s",
            "host_cpu": _cpu_model(), "host_nproc": os.cpu_count()}


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        m = re.search(r"Model name:\s*(.+)", out)
        return m.group(1).strip() if m else None
    except OSError:
        return None


# ------------------------------------------------------------------------------------
# reference arm: the oracle on host cores
# ------------------------------------------------------------------------------------
def run_reference(args, rank, world, local):
    from bitwise_reproducible_step_gb300 import inputs as I
    from oracle import oracle as O

    wl = I.WORKLOADS[args.workload]
    n, R = wl.n, wl.R
    # bounded sample: ~0.35 s of oracle work per 2^22 params on one Grace core, so that the
    # whole --steps K --warmup W run stays within a couple of minutes
    n_s = min(n, max(1 << 16, min(1 << 22, (1 << 22) * 100 // max(1, args.steps + args.warmup))))
    hpv = I.default_hparams()
    grads = [I.to_numpy(I.gen_grad(wl, 1, r, n=n_s, device="cpu")) for r in range(R)]
    w, m, v = (t.numpy() for t in I.gen_state(wl, n=n_s, device="cpu"))

    def one(t):
        nonlocal w, m, v
        out = O.step(grads, w, m, v, lr=hpv["lr"], beta1=hpv["beta1"], beta2=hpv["beta2"],
                     eps=hpv["eps"], wd=hpv["wd"], clip=hpv["clip"], t=t)
        w, m, v = out["w"], out["m"], out["v"]

    for t in range(1, args.warmup + 1):
        one(t)
    t0 = time.perf_counter()
    for t in range(args.warmup + 1, args.warmup + args.steps + 1):
        one(t)
    dt = (time.perf_counter() - t0) / args.steps
    value = n_s / dt
    sample = (f"{n_s:,} params per step (of the workload's {n:,}) drawn from the same "
              f"distributions, R={R}, seeded on the CPU; one full oracle step each")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "n_params": n, "replicas": R,
                       "grad_dtype": wl.grad_dtype, "sample_params_per_step": n_s},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="flat1200m_r8_segscale")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--e2e-pieces", type=int, default=8,
                    help="chunk-aligned ranges the e2e step pipelines its copies over")
    ap.add_argument("--e2e-copy-streams", type=int, default=2,
                    help="streams the e2e step spreads each range's copies over")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--param-dtype", choices=["f32", "bf16"], default="f32",
                    help="parameter dtype (bf16: widened, updated in fp32, rounded once)")
    ap.add_argument("--subnormals", choices=["ieee", "ftz"], default="ieee",
                    help="ftz: flush-to-zero arithmetic (subnormal operands and tiny results zeroed)")
    ap.add_argument("--decay-mask", action="store_true",
                    help="per-segment weight decay through a device bitmask")
    ap.add_argument("--hash-mode", choices=["pf61", "blake2b"], default="pf61",
                    help="leaf digest of the state hash (blake2b = audit mode)")
    ap.add_argument("--no-hash-stream", dest="hash_stream", action="store_false",
                    help="run the root passes on the step's own stream (no overlap with the "
                         "next step's reduce)")
    ap.add_argument("--nodes", type=int, default=1,
                    help="stage the canonical reduce over this many nodes (same bits)")
    ap.add_argument("--paper-shard", type=int, default=0,
                    help="reduce in the paper-exact order (Algorithm 1) with this dp_shard")
    ap.add_argument("--accum", type=int, default=0,
                    help="with --paper-shard: the replicas are microbatches, accum per rank")
    ap.add_argument("--block-threads", type=int, default=0, choices=[0, 128, 256, 512],
                    help="compute threads per CTA of the streaming kernels (0: default)")
    ap.add_argument("--log", default="",
                    help="append a JSON-lines record per timed step (norm, its bits, root, "
                         "event time) and the summary line to this file")
    ap.add_argument("--two-pass", action="store_true",
                    help="time repstep_step (reduce, then clip and AdamW in place) instead of "
                         "the default repstep_step_fused (one HBM pass from one state buffer "
                         "into a second when the step does not clip; the same bits)")
    ap.add_argument("--shard", action="store_true",
                    help="the sharded step: n split over the ranks' GPUs (all-to-all + "
                         "all-gathers); with one process, a one-rank NCCL group")
    ap.add_argument("--n", type=int, default=0,
                    help="override the workload's parameter count (small profiling cases)")
    args = ap.parse_args()
    # the single pass covers the canonical tree; the paper-exact and staged orders run the
    # two passes
    args.fused = not args.two_pass and not args.paper_shard and args.nodes == 1
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        print(json.dumps(run_reference(args, 0, world, 0)), flush=True)
        return

    rank, world, local = dist_init(args.gpus)
    if args.shard:
        import torch.distributed as dist
        if not dist.is_initialized():          # one process: a one-rank group of its own
            import socket
            with socket.socket() as s_:
                s_.bind(("127.0.0.1", 0))
                port = s_.getsockname()[1]
            dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                                    world_size=1, device_id=torch.device("cuda", local))
        res = run_sharded(args, rank, world, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
        dist.destroy_process_group()
        return
    res = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
