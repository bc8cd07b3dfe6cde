"""Benchmark of the GB300 speculative-decoding verification step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one spec_verify call (one verification round) over one batch of the
B=256, gamma=4, V=128256 bf16 workload (Zipf-shifted N(0, 3^2) target logits,
draft noise sigma ~ U[0.2, 2.0], even sequences greedy, odd ones T=1.0).
Inputs are generated on the host from a seeded generator and copied to HBM
twice, at different addresses; consecutive steps alternate between the two
copies (2 x 591 MB, far more than the 129 MB of L2), so no step reads logits
that the step before left in L2.  Under torchrun each rank verifies its own
batch (seed + rank): weak scaling, no collective on the data path.  Rank 0
prints one JSON line; its "configs" key times the other four workloads the
same way (and the oracle beside each).

--impl reference times the float64 CPU oracle (the method's plain restatement)
on the host cores instead, one bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "spec_verify sequences/s and achieved HBM GB/s vs ~8 TB/s peak (1 GB300)"
UNIT = "sequences/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_DIR = os.path.join(ROOT, "speculative_decoding_verification_45_gb300", "csrc")
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "spec_verify_cfg5_traffic.json")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, group_backend: str | None) -> float:
    """Max over ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if group_backend == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate_value(seqs_per_rank: int, world: int, steps: int, seconds_max: float) -> float:
    """Whole-job sequences per second: every rank's sequences over the slowest rank's time."""
    return seqs_per_rank * world * steps / seconds_max


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    """sha256 over the kernel sources (csrc/*.cu, *.cuh in name order): the
    recorded DRAM traffic holds only for the sources it was measured on."""
    h = hashlib.sha256()
    for name in sorted(os.listdir(KERNEL_DIR)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(KERNEL_DIR, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def recorded_traffic(workload_key: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on this kernel source."""
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_sha256") != kernel_source_hash() or rec.get("workload") != workload_key:
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""

    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4], parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        used = inside
        if not used and rows:
            mid = 0.5 * (t0 + t1)
            used = [min(rows, key=lambda r: abs(r[0] - mid))]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i, v in enumerate(r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": max(r[2] for r in used),
                "reasons": reasons, "samples": len(inside)}


def oracle_baseline(batch, target_seconds: float, threads: int = 0):
    """The float64 oracle on the host cores: whole batches until target_seconds of wall time."""
    import oracle

    cores = threads if threads > 0 else (os.cpu_count() or 1)
    oracle.build()
    n_seq, t_total, reps = 0, 0.0, 0
    while t_total < target_seconds or reps == 0:
        t0 = time.perf_counter()
        oracle.verify_batch(batch, diagnostics=False, nthreads=cores)
        t_total += time.perf_counter() - t0
        n_seq += batch.B
        reps += 1
    return {"value": n_seq / t_total, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} x the full {batch.B}-sequence batch ({n_seq} sequences), {t_total:.1f} s wall, "
                      f"{cores} threads"}


def workload_desc(cfg: int):
    from speculative_decoding_verification_45_gb300 import workloads

    return workloads.CONFIG_NAMES[cfg]


def make_batch(args, rank=0):
    """The timed workload: a config with its default seed (or --seed), shifted per
    rank; --greedy sets every temperature to 0 (config 2 has its own greedy
    variant with argmax drafts)."""
    from speculative_decoding_verification_45_gb300 import workloads

    seed = (workloads.default_seed(args.config) if args.seed is None else args.seed) + rank
    if args.greedy and args.config == 2:
        return workloads.make_config(2, seed=seed, greedy=True)
    batch = workloads.make_config(args.config, seed=seed)
    if args.greedy:
        batch.temperature[:] = 0.0
    return batch


def run_reference(args):
    """Reference arm: the float64 oracle timed on the host cores."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from speculative_decoding_verification_45_gb300 import workloads

    batch = make_batch(args)
    oracle.build()
    cores = os.cpu_count() or 1
    # size one step's sample so the whole run stays within ~60 s of oracle time
    t0 = time.perf_counter()
    cal = min(batch.B, 16)
    sub = _slice(batch, 0, cal)
    oracle.verify_batch(sub, diagnostics=False, nthreads=cores)
    per_seq = (time.perf_counter() - t0) / cal
    total_steps = args.steps + args.warmup
    per_step = max(1, min(batch.B, int(60.0 / max(total_steps, 1) / max(per_seq, 1e-6))))
    # whole multiples of the thread count (the oracle runs one sequence per
    # thread), so that no host core idles in a step
    per_step = min(batch.B, max(cores, per_step // cores * cores))
    samples = [_slice(batch, (i * per_step) % batch.B, per_step) for i in range(4)]
    for i in range(args.warmup):
        oracle.verify_batch(samples[i % 4], diagnostics=False, nthreads=cores)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.verify_batch(samples[i % 4], diagnostics=False, nthreads=cores)
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(args.config), "sequences_per_step": per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} sequences of the {batch.B}-sequence batch per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _slice(batch, start, count):
    import numpy as np

    from speculative_decoding_verification_45_gb300 import workloads

    idx = (np.arange(count) + start) % batch.B
    return workloads.Batch(batch.target[idx], batch.draft[idx], batch.tokens[idx], batch.num_draft[idx],
                           batch.uniforms[idx], batch.temperature[idx], batch.dtype, batch.name)


def est_ms_per_step(step, stream, n=20):
    """Rough device time of one step (sizing the clock window only)."""
    import torch

    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        step()
    z.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(z) / n


def oracle_rate(batch, threads: int, seconds: float):
    """Oracle sequences/s on `threads` host threads over whole batches for about `seconds`."""
    import oracle

    n_seq, t_total = 0, 0.0
    while t_total < seconds or n_seq == 0:
        t0 = time.perf_counter()
        oracle.verify_batch(batch, diagnostics=False, nthreads=threads)
        t_total += time.perf_counter() - t0
        n_seq += batch.B
    return n_seq / t_total


def config_table(args, sv, dev, stream, main_batch, backend):
    """Every workload timed like the headline one (the library's automatic
    choice, and the full sweep and the early exit explicitly), with the oracle
    beside it on 1 host thread and on all of them.  Input sets rotate so that
    they cover at least twice L2 (configs 1 and 2 fit in L2 whatever is done)."""
    import math

    import torch

    from speculative_decoding_verification_45_gb300 import workloads

    peak, _ = measured_peaks()
    cores = os.cpu_count() or 1
    l2 = 129 << 20
    out = {}
    for name in ("1", "2", "2-greedy", "3", "4", "5"):
        cfg = int(name[0])
        batch = main_batch if cfg == args.config and name == str(args.config) else \
            workloads.make_config(cfg, greedy=name.endswith("greedy"))
        base = sv.to_device(batch, dev)
        set_bytes = sum(v.numel() * v.element_size() for v in base.values())
        nsets = max(2, min(8, math.ceil(2 * l2 / set_bytes))) if set_bytes * 8 >= 2 * l2 else 2
        sets = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(nsets - 1)]
        ot = torch.empty((batch.B, batch.gmax + 1), dtype=torch.int32, device=dev)
        on = torch.empty((batch.B,), dtype=torch.int32, device=dev)
        k = max(args.steps, 200 if cfg >= 3 else 1000)
        row = {"workload": workloads.CONFIG_NAMES[cfg] + (" (greedy)" if name.endswith("greedy") else ""),
               "input_sets": nsets, "set_bytes": set_bytes,
               "l2": "rotated sets cover >= 2x L2" if set_bytes * nsets >= 2 * l2 else "inputs fit in L2"}
        algo = batch.algorithmic_bytes()
        _, _, _, auto_kind = sv.launch_shape(batch.B, batch.gmax, batch.V, batch.dtype)
        row["auto_kernel"] = "early_exit" if auto_kind == sv.KERNEL_EARLY else "full_sweep"
        for label, kern in (("auto", sv.KERNEL_AUTO), ("full_sweep", sv.KERNEL_REGISTER),
                            ("early_exit", sv.KERNEL_EARLY)):
            def one(i, kern=kern):
                sv.verify(**sets[i % nsets], out_tokens=ot, out_num_accepted=on, stream=stream, kernel=kern)
            for i in range(max(args.warmup, 3)):
                one(i)
            torch.cuda.synchronize()
            barrier()
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(k):
                one(i)
            z.record(stream)
            torch.cuda.synchronize()
            ms = reduce_max(a.elapsed_time(z), backend) / k
            row[f"{label}_us"] = ms * 1e3
            if label == "auto":
                if auto_kind == sv.KERNEL_EARLY:  # the rows up to each cut, from the outcome
                    import numpy as np

                    n_acc = on.cpu().numpy().astype(np.int64)
                    g_np = np.clip(batch.num_draft.astype(np.int64), 0, batch.gmax)
                    smp = (batch.temperature > 0).astype(np.int64)
                    rows_full = int(((g_np + 1) + smp * g_np).sum())
                    rows_early = int(((np.minimum(n_acc, g_np) + 1) + smp * np.minimum(n_acc + 1, g_np)).sum())
                    algo = algo - (rows_full - rows_early) * batch.V * batch.elem_size
                row.update({"sequences_per_s": batch.B / (ms / 1e3), "rounds_per_s": 1e3 / ms,
                            "algorithmic_bytes": algo, "hbm_gbs_algorithmic": algo / (ms / 1e3) / 1e9,
                            "frac_of_peak": algo / (ms / 1e3) / 1e9 / peak, "gpu_launches": k})
        if not args.no_cpu_baseline:
            row["oracle_1_thread_sequences_per_s"] = oracle_rate(batch, 1, args.cpu_seconds / 8)
            row["oracle_all_cores_sequences_per_s"] = oracle_rate(batch, cores, args.cpu_seconds / 8)
            row["oracle_cores"] = cores
        out[name] = row
        del sets, base
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    backend = None
    if ws > 1:
        backend = "nccl"
        torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import speculative_decoding_verification_45_gb300 as sv
    from speculative_decoding_verification_45_gb300 import workloads

    if rank == 0:
        sv.build()
    barrier()
    sv._native.load()

    batch = make_batch(args, rank)
    B = batch.B
    inputs = sv.to_device(batch, dev)
    # a second copy at other addresses: steps alternate between the two
    sets = [inputs, {k: v.clone() for k, v in inputs.items()}]
    out_tokens = torch.empty((B, batch.gmax + 1), dtype=torch.int32, device=dev)
    out_num = torch.empty((B,), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    full_bytes = batch.algorithmic_bytes()  # every row the full sweep needs
    C, nctas, threads, auto_kind = sv.launch_shape(B, batch.gmax, batch.V, batch.dtype)
    if args.cluster:
        C, nctas = args.cluster, B * args.cluster
    kernel = {"auto": sv.KERNEL_AUTO, "stream": sv.KERNEL_REGISTER, "early": sv.KERNEL_EARLY}[args.kernel]
    ran = auto_kind if args.kernel == "auto" else kernel  # the kernel the steps run

    calls = [0]

    def step():
        sv.verify(**sets[calls[0] & 1], out_tokens=out_tokens, out_num_accepted=out_num, stream=stream,
                  cluster_size=args.cluster, kernel=kernel)
        calls[0] += 1

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()

    sampler = None
    if not args.quick:
        props = torch.cuda.get_device_properties(dev)
        uuid = str(getattr(props, "uuid", ""))
        gpu_id = uuid if uuid.startswith("GPU-") else (f"GPU-{uuid}" if uuid else str(local))
        sampler = ClockSampler(gpu_id)
        sampler.start()
        time.sleep(0.3)

    # The K timed steps run inside a longer busy stretch of the same step
    # (about 0.3 s before and after, enqueued without a synchronisation in
    # between), so that the clock sampler, which reads every 50 ms, sees the
    # clocks the timed steps ran at; only the K steps between the events count.
    n_pad = 0
    if sampler:
        n_pad = max(1, int(0.3 / max(est_ms_per_step(step, stream) / 1e3, 1e-6)))
    start_ev = torch.cuda.Event(enable_timing=True)
    stop_ev = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    w0 = time.time()
    for _ in range(n_pad):
        step()
    start_ev.record(stream)
    for _ in range(args.steps):
        step()
    stop_ev.record(stream)
    for _ in range(n_pad):
        step()
    torch.cuda.synchronize()
    w1 = time.time()
    barrier()
    ms_total = start_ev.elapsed_time(stop_ev)
    ms_max = reduce_max(ms_total, backend)
    clocks = None
    if sampler:
        time.sleep(0.1)
        sampler.stop()
        clocks = sampler.summary(w0, w1)
        clocks["window"] = (f"{n_pad} + {args.steps} + {n_pad} back-to-back steps ({w1 - w0:.2f} s); the "
                            f"{args.steps} timed steps sit in the middle")

    value = aggregate_value(B, ws, args.steps, ms_max / 1e3)
    ms_step = ms_max / args.steps
    # bytes one launch must read: every needed row for the full sweep; for the
    # early exit, the rows up to each sequence's cut (n + 1 target rows, and
    # min(n + 1, g) draft rows when sampled), from this batch's outcome
    import numpy as np

    n_acc = out_num.cpu().numpy().astype(np.int64)
    g_np = batch.num_draft.astype(np.int64)
    smp_np = (batch.temperature > 0).astype(np.int64)
    small_bytes = full_bytes - int(((g_np + 1) + smp_np * g_np).sum()) * batch.V * batch.elem_size
    early_rows = int(((n_acc + 1) + smp_np * np.minimum(n_acc + 1, g_np)).sum())
    algo_bytes = early_rows * batch.V * batch.elem_size + small_bytes if ran == sv.KERNEL_EARLY else full_bytes

    # the distribution of single calls: each of 200 back-to-back calls between
    # its own CUDA events (median, p10 and p90 of the device time)
    per_call = None
    if not args.quick:
        import numpy as np

        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(200)]
        torch.cuda.synchronize()
        for a, z in pairs:
            a.record(stream)
            step()
            z.record(stream)
        torch.cuda.synchronize()
        us = np.array([a.elapsed_time(z) * 1e3 for a, z in pairs])
        per_call = {"median_us": float(np.median(us)), "p10_us": float(np.percentile(us, 10)),
                    "p90_us": float(np.percentile(us, 90)), "calls": len(pairs)}

    # the same steps replayed from a CUDA graph (how a serving loop launches a
    # fixed-shape step): the kernels and bytes are identical; the host launch
    # path is not in the way
    graph = None
    if not args.quick:
        n_cap = 20
        gstream = torch.cuda.Stream(dev)
        gstream.wait_stream(stream)
        with torch.cuda.stream(gstream):
            for _ in range(3):
                sv.verify(**inputs, out_tokens=out_tokens, out_num_accepted=out_num, stream=gstream,
                          cluster_size=args.cluster, kernel=kernel)
        torch.cuda.synchronize()
        cg_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg_, stream=gstream):
            for i in range(n_cap):
                sv.verify(**sets[i & 1], out_tokens=out_tokens, out_num_accepted=out_num, stream=gstream,
                          cluster_size=args.cluster, kernel=kernel)
        reps = max(1, args.steps // n_cap)
        for _ in range(3):
            cg_.replay()
        torch.cuda.synchronize()
        barrier()
        cur = torch.cuda.current_stream(dev)
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for _ in range(reps):
            cg_.replay()
        z.record(cur)
        torch.cuda.synchronize()
        g_ms = reduce_max(a.elapsed_time(z), backend) / (reps * n_cap)
        graph = {"value": aggregate_value(B, ws, 1, g_ms / 1e3), "unit": UNIT, "ms_per_step": g_ms,
                 "hbm_gbs_algorithmic": algo_bytes / (g_ms / 1e3) / 1e9, "steps": reps * n_cap,
                 "gpu_launches": reps * n_cap}
        del cg_

    # the row-ordered early-exit variant on the same inputs (same outputs; it
    # reads n+1 target and min(n+1, g) draft rows per sequence)
    early = None
    if args.kernel == "auto" and not args.quick:
        import numpy as np

        ot_e = torch.empty_like(out_tokens)
        on_e = torch.empty_like(out_num)

        e_calls = [0]

        def step_early():
            sv.verify(**sets[e_calls[0] & 1], out_tokens=ot_e, out_num_accepted=on_e, stream=stream,
                      cluster_size=args.cluster, kernel=sv.KERNEL_EARLY)
            e_calls[0] += 1

        for _ in range(max(args.warmup, 3)):
            step_early()
        torch.cuda.synchronize()
        same = bool(torch.equal(ot_e, out_tokens) and torch.equal(on_e, out_num))
        n_acc = on_e.cpu().numpy().astype(np.int64)
        g = batch.num_draft.astype(np.int64)
        smp = (batch.temperature > 0).astype(np.int64)
        rows = int(((n_acc + 1) + smp * np.minimum(n_acc + 1, g)).sum())
        need = rows * batch.V * batch.elem_size
        barrier()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            step_early()
        z.record(stream)
        torch.cuda.synchronize()
        e_ms = reduce_max(a.elapsed_time(z), backend) / args.steps
        peak_e, _ = measured_peaks()
        early = {"value": aggregate_value(B, ws, 1, e_ms / 1e3), "unit": UNIT, "ms_per_step": e_ms,
                 "rows_read_per_step": rows, "needed_bytes_per_step": need,
                 "hbm_gbs_needed": need / (e_ms / 1e3) / 1e9, "frac_of_peak": need / (e_ms / 1e3) / 1e9 / peak_e,
                 "same_outputs_as_full_sweep": same, "gpu_launches": args.steps}

    # target-only sampling (the round with no drafts): one token per sequence
    # from row t_0 of the same inputs, B rows of V logits
    sampling = None
    if args.kernel == "auto" and not args.quick:
        rows0 = inputs["target_logits"][:, 0].contiguous()
        u0 = inputs["uniforms"][:, -1].contiguous()
        out0 = torch.empty((B,), dtype=torch.int32, device=dev)

        def step_sample():
            sv.sample(rows0, u0, inputs["temperature"], out_tokens=out0, stream=stream)

        for _ in range(max(args.warmup, 3)):
            step_sample()
        torch.cuda.synchronize()
        barrier()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            step_sample()
        z.record(stream)
        torch.cuda.synchronize()
        s_ms = reduce_max(a.elapsed_time(z), backend) / args.steps
        nbytes = rows0.numel() * rows0.element_size()
        peak_s, _ = measured_peaks()
        sampling = {"value": aggregate_value(B, ws, 1, s_ms / 1e3), "unit": UNIT, "ms_per_step": s_ms,
                    "bytes_per_step": nbytes, "hbm_gbs": nbytes / (s_ms / 1e3) / 1e9,
                    "frac_of_peak": nbytes / (s_ms / 1e3) / 1e9 / peak_s, "gpu_launches": args.steps,
                    "note": "B rows of V logits; inputs larger than L2 only together with the rest of the bench"}

    # prompt lookup (n-gram proposer) and point-mass verification of its drafts
    # against the same target rows: contexts of 8192 tokens with repeated spans
    lookup = None
    if args.kernel == "auto" and not args.quick:
        import numpy as np

        ctx_np, lens_np = workloads.ngram_contexts(B, 8192, batch.V, seed=workloads.default_seed(args.config) + 7)
        ctx = torch.from_numpy(ctx_np).to(dev)
        lens = torch.from_numpy(lens_np).to(dev)
        d_tok = torch.empty((B, batch.gmax), dtype=torch.int32, device=dev)
        d_num = torch.empty((B,), dtype=torch.int32, device=dev)
        ot_p = torch.empty_like(out_tokens)
        on_p = torch.empty_like(out_num)

        def step_propose():
            sv.ngram_propose(ctx, lens, 1, 4, batch.gmax, out_tokens=d_tok, out_num=d_num, stream=stream)

        def step_point():
            sv.verify(inputs["target_logits"], None, d_tok, d_num, inputs["uniforms"], inputs["temperature"],
                      out_tokens=ot_p, out_num_accepted=on_p, stream=stream)

        times = {}
        for name, fn in (("propose", step_propose), ("verify_point", step_point)):
            for _ in range(max(args.warmup, 3)):
                fn()
            torch.cuda.synchronize()
            barrier()
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(args.steps):
                fn()
            z.record(stream)
            torch.cuda.synchronize()
            times[name] = reduce_max(a.elapsed_time(z), backend) / args.steps
        g_prop = d_num.cpu().numpy().astype(np.int64)
        rows = int((g_prop + 1).sum())
        vbytes = rows * batch.V * batch.elem_size
        peak_l, _ = measured_peaks()
        lookup = {"contexts": f"B={B} x up to 8192 tokens, repeated spans", "min_n": 1, "max_n": 4,
                  "propose_ms_per_step": times["propose"], "context_bytes": int(ctx_np.nbytes),
                  "mean_drafts": float(g_prop.mean()), "verify_point_ms_per_step": times["verify_point"],
                  "verify_point_rows": rows, "verify_point_hbm_gbs": vbytes / (times["verify_point"] / 1e3) / 1e9,
                  "verify_point_frac_of_peak": vbytes / (times["verify_point"] / 1e3) / 1e9 / peak_l,
                  "gpu_launches": 2 * args.steps}

    # candidate-tree verification: 32 sequences with 64-node Medusa-style trees
    # over the same vocabulary, half greedy and half T = 1; the walk reads the
    # rows on the accepted path only
    tree = None
    if args.kernel == "auto" and not args.quick:
        import numpy as np

        tb = workloads.tree_batch(32, 64, batch.V, dtype=batch.dtype, seed=workloads.default_seed(args.config) + 11,
                                  shape="medusa", temps=(0.0, 1.0), ragged=False)
        tdev = sv.tree_to_device(tb, dev)
        t_tok = torch.empty((tb.B, tb.N), dtype=torch.int32, device=dev)
        t_num = torch.empty((tb.B,), dtype=torch.int32, device=dev)
        t_path = torch.empty((tb.B, tb.N), dtype=torch.int32, device=dev)

        def step_tree():
            sv.tree_verify(**tdev, out_tokens=t_tok, out_num_accepted=t_num, out_path=t_path, stream=stream)

        for _ in range(max(args.warmup, 3)):
            step_tree()
        torch.cuda.synchronize()
        barrier()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            step_tree()
        z.record(stream)
        torch.cuda.synchronize()
        t_ms = reduce_max(a.elapsed_time(z), backend) / args.steps
        acc = t_num.cpu().numpy().astype(np.int64)
        need = tb.path_bytes(acc)
        peak_t, _ = measured_peaks()
        tree = {"value": aggregate_value(tb.B, ws, 1, t_ms / 1e3), "unit": UNIT, "ms_per_step": t_ms,
                "workload": f"B={tb.B}, 64-node Medusa-style trees (4,3,2,2 children per level), V={tb.V} "
                            f"{tb.dtype}, half greedy / half T=1.0",
                "mean_accepted": float(acc.mean()), "rows_read_per_step": int((acc + 1).sum()),
                "needed_bytes_per_step": need, "hbm_gbs_needed": need / (t_ms / 1e3) / 1e9,
                "frac_of_peak": need / (t_ms / 1e3) / 1e9 / peak_t, "gpu_launches": args.steps}
        del tdev

    # acceptance statistics of this batch (outside the timed region): the counts
    # a serving engine exports, and E = (1 - a^(g+1)) / (1 - a) at the measured a
    acceptance = None
    if not args.quick:
        import numpy as np

        cnt = torch.zeros(3, dtype=torch.int64, device=dev)
        hist = torch.zeros(sv.MAX_GAMMA + 1, dtype=torch.int64, device=dev)
        sv.verify(**inputs, stream=stream, counters=cnt, accept_hist=hist)
        torch.cuda.synchronize()
        c, h = cnt.cpu().numpy(), hist.cpu().numpy()
        drafted, accepted, seqs = int(c[0]), int(c[1]), int(c[2])
        a_hat = accepted / drafted if drafted else 0.0
        g = batch.gmax
        acceptance = {"drafted": drafted, "accepted": accepted, "sequences": seqs,
                      "alpha_hat": a_hat, "mean_tokens_per_round": (accepted + seqs) / seqs if seqs else 0.0,
                      "E_at_alpha_hat": (1 - a_hat ** (g + 1)) / (1 - a_hat) if a_hat < 1 else g + 1.0,
                      "accepted_count_hist": [int(x) for x in h[: g + 1]],
                      "note": "alpha_hat pools all positions; E assumes one alpha for every position"}

    configs = None
    if not args.quick and args.kernel == "auto" and not args.cluster and ws == 1:
        configs = config_table(args, sv, dev, stream, batch, backend)

    # end to end through the public API with host buffers.  The main figure
    # keeps every input in page-locked host memory and lets the early-exit
    # kernel read it over the host link (zero copy: only the rows up to each
    # sequence's first rejection cross the link); the outputs come back by a
    # device-to-host copy.  Also timed on the same host buffers: the full sweep
    # (every logit crosses the link) and a staged copy of every input to the
    # device before the call.  A 256 MB device write before every zero-copy
    # step flushes L2, so no step reads logits cached by the one before.
    e2e = None
    if not args.quick:
        host = {k: v.cpu().pin_memory() for k, v in inputs.items()}
        dev_in = {k: torch.empty_like(v) for k, v in inputs.items()}
        h_tok = torch.empty(out_tokens.shape, dtype=torch.int32).pin_memory()
        h_num = torch.empty(out_num.shape, dtype=torch.int32).pin_memory()
        nbytes = {k: v.numel() * v.element_size() for k, v in host.items()}
        h2d_all = sum(nbytes.values())
        small = h2d_all - nbytes["target_logits"] - nbytes["draft_logits"]
        d2h = h_tok.numel() * 4 + h_num.numel() * 4
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        k_e2e = max(3, min(args.steps, 50))

        def zero_copy_step(kern):
            flush.zero_()
            sv.verify(**host, out_tokens=out_tokens, out_num_accepted=out_num, stream=stream,
                      cluster_size=args.cluster, kernel=kern)
            h_tok.copy_(out_tokens, non_blocking=True)
            h_num.copy_(out_num, non_blocking=True)

        def staged_step():
            for k, v in host.items():
                dev_in[k].copy_(v, non_blocking=True)
            sv.verify(**dev_in, out_tokens=out_tokens, out_num_accepted=out_num, stream=stream,
                      cluster_size=args.cluster, kernel=kernel)
            h_tok.copy_(out_tokens, non_blocking=True)
            h_num.copy_(out_num, non_blocking=True)

        def timed(step):
            for _ in range(2):
                step()
            torch.cuda.synchronize()
            barrier()
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(k_e2e):
                step()
            z.record(stream)
            torch.cuda.synchronize()
            return reduce_max(a.elapsed_time(z), backend) / 1e3

        # three rounds of the three paths, interleaved, so that a slow stretch
        # of the shared host link falls on every path; the median round counts
        full_kernel = sv.KERNEL_REGISTER
        rounds = {"zc": [], "full": [], "staged": []}
        for _ in range(3):
            rounds["zc"].append(timed(lambda: zero_copy_step(sv.KERNEL_EARLY)))
            rounds["full"].append(timed(lambda: zero_copy_step(full_kernel)))
            rounds["staged"].append(timed(staged_step))
        t_zc, t_full, t_staged = (statistics.median(rounds[k]) for k in ("zc", "full", "staged"))
        zero_copy_step(sv.KERNEL_EARLY)
        torch.cuda.synchronize()
        n_acc = h_num.numpy().astype(np.int64)
        g = batch.num_draft.astype(np.int64)
        smp = (batch.temperature > 0).astype(np.int64)
        rows_zc = int(((n_acc + 1) + smp * np.minimum(n_acc + 1, g)).sum())
        h2d_zc = rows_zc * batch.V * batch.elem_size + small
        rows_full = int(((g + 1) + smp * g).sum())  # greedy sequences' draft rows are never read
        h2d_full = rows_full * batch.V * batch.elem_size + small
        e2e = {"value": aggregate_value(B, ws, k_e2e, t_zc), "unit": UNIT, "h2d_bytes_per_step": h2d_zc,
               "d2h_bytes_per_step": d2h, "steps": k_e2e, "rounds": 3,
               "path": "zero copy: inputs in page-locked host memory, read by the early-exit kernel over the "
                       "host link (only the rows up to each first rejection cross it, once: pass 2 takes the "
                       "decided rows from shared memory); outputs copied back",
               "host_input_bytes_per_step": h2d_all, "l2_flushed_each_step": True,
               "rounds_sequences_per_s": [aggregate_value(B, ws, k_e2e, t) for t in rounds["zc"]],
               "link_gbs": h2d_zc * k_e2e / t_zc / 1e9,
               "full_sweep_zero_copy": {"value": aggregate_value(B, ws, k_e2e, t_full), "unit": UNIT,
                                        "h2d_bytes_per_step": h2d_full, "d2h_bytes_per_step": d2h,
                                        "link_gbs": h2d_full * k_e2e / t_full / 1e9,
                                        "note": "every row the sweep needs crosses the link; pass 2 reads the "
                                                "decided row over it again"},
               "staged_copy": {"value": aggregate_value(B, ws, k_e2e, t_staged), "unit": UNIT,
                               "h2d_bytes_per_step": h2d_all, "d2h_bytes_per_step": d2h,
                               "note": "every input copied to the device before the call"}}

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return 0

    peak, peak_src = measured_peaks()
    achieved = algo_bytes / (ms_step / 1e3) / 1e9
    kernel_name = "spec_verify_early_kernel" if ran == sv.KERNEL_EARLY else "spec_verify_stream_kernel"
    workload_key = f"cfg{args.config}-B{B}-g{batch.gmax}-V{batch.V}-{batch.dtype}-{kernel_name}"
    traffic = recorded_traffic(workload_key) if args.kernel == "auto" and not args.cluster else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": workload_desc(args.config), "B": B, "gamma": batch.gmax, "V": batch.V,
                   "logits": batch.dtype, "parallelism": f"dp{ws} (independent sequences per rank)",
                   "l2": "two input sets at different addresses, alternating per step (2 x 591 MB >> 129 MB "
                         "of L2): no step reads what the previous one left in L2",
                   "cluster_size": C, "ctas": nctas, "threads_per_cta": threads, "kernel": args.kernel},
        "rounds_per_s": ws * args.steps / (ms_max / 1e3),
        "hbm_gbs_algorithmic": achieved,
        "hbm_gbs_nominal_590MB": batch.nominal_bytes() / (ms_step / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": algo_bytes, "kernel": kernel_name,
                     "bytes_rule": "rows the launch must read (x V x 2 B) + the 4-byte arrays; early exit: "
                                   "n+1 target and min(n+1, g) draft rows per sampled sequence, n+1 target "
                                   "rows per greedy one, from this batch's outcome"},
        "full_sweep_bytes_per_s": full_bytes / (ms_step / 1e3) / 1e9,
        "gpu_launches": args.steps,
        "per_call_us": per_call,
        "graph_replay": graph,
        "early_exit_variant": early,
        "target_only_sampling": sampling,
        "prompt_lookup": lookup,
        "tree_verify": tree,
        "acceptance": acceptance,
        "configs": configs,
        "e2e": e2e,
        "clocks": clocks,
    }
    if ws == 1 and not args.quick and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(batch, args.cpu_seconds, args.cpu_threads)
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--seed", type=int, default=None, help="workload seed (default: 1234 + config)")
    ap.add_argument("--greedy", action="store_true", help="every temperature 0 (argmax verification)")
    ap.add_argument("--kernel", choices=["auto", "stream", "early"], default="auto",
                    help="kernel choice (A/B measurement; auto = the library's default full sweep; "
                         "early = row-ordered early exit)")
    ap.add_argument("--cluster", type=int, default=0, choices=list(range(17)),
                    help="CTAs per sequence (0 = the library's default)")
    ap.add_argument("--quick", action="store_true", help="skip e2e, clocks and the CPU baseline (profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-threads", type=int, default=0, help="oracle baseline threads (0 = all host cores)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and not args.quick:
        log("warning: fewer than 3 warm-up steps")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
