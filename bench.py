"""Benchmark: HBM GB/s of CE fwd+bwd and selective log-softmax, 8192 x 152064 bf16.

One step = the whole hot path over one batch of the packed RL workload
(8 sequences x 1024 tokens = 8192 rows, vocab 152064, bf16 logits ~N(0, 2.5^2),
5% confident rows, temperature 0.9):

  * selective_logsoftmax at K = 4 gathered indices per row, and
  * ce_fwd_bwd_fused (mean reduction, upstream gradient 1) writing dlogits.

``value`` is algorithmic bytes per step (logits read once per op, dlogits
written once, plus indices, labels and log-prob outputs) over the device time
of the step, in GB/s, with inputs resident in HBM.  The logits (2.49 GB) are
larger than L2, so no flush is needed between steps.  ``e2e`` is the same
metric through the public Python API with the inputs copied from pinned host
memory and the results (loss, log-probs) read back every step; the copy goes
in row blocks on a second stream so that each block's compute overlaps the
next block's copy.

``per_config`` times every op of every seeded workload alone (``ms``: a
lone CUDA-graph launch, after an L2 flush for workloads smaller than 256 MB:
a 512 MB write, then a 256 MB read that leaves L2 clean).  For workloads smaller than L2
it adds ``ms_steady``: the same call back to back over rotating copies of
its inputs (more than twice the L2 in all), without the fixed floor of a
lone launch that ``_launch_floor`` records.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same rows instead (the only other place this file runs the oracle is the
``cpu_baseline`` leg of the default arm).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gbce|reference]
Multi-GPU (one process per GPU, torchrun): every rank runs its own replica of
the workload (independent batches, no collective on the data path); rank 0
prints the aggregate over the max-over-ranks time.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "HBM GB/s (% of GB300 peak) for CE fwd+bwd & selective logp, 8192x152064 bf16"
UNIT = "GB/s"
ROWS, VOCAB, K, TEMPERATURE = 8192, 152064, 4, 0.9
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "persistent_fused_kernel_bf16_1024x152064.md")


def algorithmic_bytes(rows=None, vocab=VOCAB, k=K, esize=2, entropy=False):
    """Bytes each op must move at least once: per row, the logits read once per
    op, the dlogits row written once, the K indices, the label and the K fp32
    log-probs (and the fp32 row entropy with --entropy)."""
    rows = ROWS if rows is None else rows
    logits = rows * vocab * esize
    logp = logits + rows * k * 8 + rows * k * 4          # logits + index + fp32 out
    if entropy:
        logp += rows * 4
    ce = 2 * logits + rows * 8                           # logits in, dlogits out, labels
    return {"selective_logsoftmax": logp, "ce_fwd_bwd_fused": ce, "step": logp + ce}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """Hash of the CUDA sources' code: comments and blank space left out,
    so that a comment edit does not void counters taken on the same code
    (a string literal holding a comment marker would be cut too: there is
    none that matters in these sources)."""
    import hashlib
    import re

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "cross_entropy_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            text = re.sub(r"//[^\n]*", " ", text)
            h.update(name.encode())
            h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per fused launch at 8192 rows from the committed ncu summary
    (one-pass counters at 1024 and 2048 rows, scaled by the marginal row),
    if the kernel sources are still the ones captured; else None."""
    try:
        fields = {}
        with open(PROFILE_TRAFFIC) as f:
            for line in f:
                if ":" in line and not line.startswith((" ", "#", "|")):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("kernel_source_sha256") != kernel_source_hash():
            return None
        return int(fields["dram_bytes_per_launch_8192_rows"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.device_index = device_index

    def start(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = os.environ.get("GBCE_DIST_BACKEND") or (
            "nccl" if torch.cuda.is_available() else "gloo")
        dist.init_process_group(backend)
    return world, rank, local


def aggregate_gbs(world: int, bytes_per_step: int, steps: int, max_ms: float) -> float:
    """Whole-job GB/s: every rank moves bytes_per_step per step (weak scaling),
    over the slowest rank's time."""
    return world * bytes_per_step * steps / (max_ms * 1e-3) / 1e9


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def time_oracle_sample(w_rows: dict, n_threads=None):
    """Run the oracle on host rows; returns (seconds, rows)."""
    import oracle

    if n_threads:
        oracle.set_num_threads(n_threads)
    x, idx, lab = w_rows["x"], w_rows["index"], w_rows["labels"]
    t0 = time.perf_counter()
    oracle.selective_logsoftmax(x, idx, TEMPERATURE)
    oracle.cross_entropy(x, lab, temperature=TEMPERATURE, reduction="none",
                         grad_out=w_rows["grad"])
    return time.perf_counter() - t0


def host_sample(w, n_rows: int, seed: int = 1234):
    import numpy as np

    rng = np.random.default_rng(seed)
    sel = np.sort(rng.choice(w.rows, size=n_rows, replace=False))
    sel_t = torch.as_tensor(sel, device=w.logits.device)
    return {"x": workloads.to_numpy_f64(w.logits[sel_t]),
            "index": w.index[sel_t].cpu().numpy(), "labels": w.labels[sel_t].cpu().numpy(),
            "grad": np.full(n_rows, 1.0 / w.rows), "rows": n_rows}


def oracle_rows_for(seconds_target: float, w) -> int:
    """Calibrate how many rows the oracle handles in about `seconds_target`."""
    probe = host_sample(w, 8, seed=99)
    t = time_oracle_sample(probe)
    per_row = max(t / 8, 1e-4)
    return int(max(8, min(w.rows, seconds_target / per_row)))


def run_reference(args):
    """The fp64 CPU oracle as it stands, on a bounded sample per step."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle

    oracle.build()
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    w = workloads.grpo_bf16(device=dev, seed=0, rows=ROWS)
    total_steps = args.steps + args.warmup
    budget = 150.0 / max(total_steps, 1)          # whole run within a few minutes
    n_rows = oracle_rows_for(min(budget, 10.0), w)
    sample = host_sample(w, n_rows)
    del w
    for _ in range(args.warmup):
        time_oracle_sample(sample)
    times = [time_oracle_sample(sample) for _ in range(args.steps)]
    step_s = statistics.median(times)
    bytes_rows = algorithmic_bytes(rows=n_rows)["step"]
    value = bytes_rows / step_s / 1e9
    cores = oracle.num_threads()
    desc = (f"{n_rows} of {ROWS} rows per step (selective logp K=4 + CE fwd+bwd), "
            f"fp64 oracle, OpenMP over rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(world, entropy=False):
    ops = ["selective_logsoftmax" + ("+entropy" if entropy else ""), "ce_fwd_bwd_fused"]
    return {"workload": f"grpo_bf16_{ROWS}x{VOCAB}_k{K}", "rows": ROWS, "vocab": VOCAB,
            "k": K, "temperature": TEMPERATURE, "logits_dtype": "bf16",
            "ops": ops, "reduction": "mean",
            "peaked_rows": "5% with target +8..12", "l2": "inputs larger than L2 (2.49 GB "
            "logits per op), no flush", "parallelism": f"replicas x{world}"}


def run_gbce(args):
    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: the gbce arm needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()
    import cross_entropy_gb300 as gbce

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workloads.grpo_bf16(device=dev, seed=rank, rows=ROWS)
    x, idx, lab = w.logits, w.index, w.labels
    grad = torch.ones(1, device=dev)
    logp_out = torch.empty((ROWS, K), dtype=torch.float32, device=dev)
    ent_out = torch.empty(ROWS, dtype=torch.float32, device=dev) if args.entropy else None
    dlogits = torch.empty_like(x)
    ws = gbce.new_workspace(ROWS, VOCAB, K, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        gbce.selective_logsoftmax(x, idx, TEMPERATURE, out=logp_out, entropy_out=ent_out,
                                  workspace=ws, dev_status=status)
        if evs is not None:
            evs[1].record(stream)
        out = gbce.ce_fwd_bwd_fused(x, lab, grad, temperature=TEMPERATURE, reduction="mean",
                                    dlogits=dlogits, workspace=ws, dev_status=status)
        if evs is not None:
            evs[2].record(stream)
        return out

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0, "device status set during warm-up"

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = gbce.kernel_launches()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    launches = gbce.kernel_launches() - launches0
    barrier(world)
    clocks = sampler.stop() if sampler else None
    total_ms = t_start.elapsed_time(t_end)
    logp_ms = [e[0].elapsed_time(e[1]) for e in evs]
    ce_ms = [e[1].elapsed_time(e[2]) for e in evs]
    total_ms = max_over_ranks(total_ms, world, dev)

    nbytes = algorithmic_bytes(entropy=args.entropy)
    ms_per_step = total_ms / args.steps
    value = aggregate_gbs(world, nbytes["step"], args.steps, total_ms)
    peak, peak_kind = measured_peak()
    ce_avg = statistics.mean(ce_ms)
    lp_avg = statistics.mean(logp_ms)
    achieved = nbytes["ce_fwd_bwd_fused"] / (ce_avg * 1e-3) / 1e9
    traffic = profiled_traffic()

    # ---- end to end through the public API: host inputs in, results out
    e2e = None if args.no_e2e else run_e2e(gbce, w, dev, stream, args, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)
    per_config = None
    if world == 1 and not args.no_configs:
        del x, idx, lab, dlogits
        w = None
        torch.cuda.empty_cache()
        per_config = measure_configs(gbce, dev, stream, peak)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(world, args.entropy),
        "frac_of_peak": value / world / peak,
        "ops": {
            "selective_logsoftmax": {"ms": lp_avg,
                                     "GB/s": nbytes["selective_logsoftmax"] / lp_avg / 1e6,
                                     "frac": nbytes["selective_logsoftmax"] / lp_avg / 1e6 / peak},
            "ce_fwd_bwd_fused": {"ms": ce_avg, "GB/s": achieved, "frac": achieved / peak},
        },
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "ce_fwd_bwd_fused call: persistent_fused_kernel + item count "
                               "+ loss reduction (events around the whole call)",
                     "algorithmic_bytes": nbytes["ce_fwd_bwd_fused"], "peak_kind": peak_kind,
                     "traffic_note": "ncu DRAM read+write of the persistent kernel at 1024 and "
                                     "2048 rows, scaled to 8192 rows by the marginal row"},
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)


def op_bytes(w, op, k=1):
    """Algorithmic bytes of one call: logits of live rows read once, dlogits
    of every row written once, int64 labels / indices and fp32 outputs."""
    es = w.logits.element_size()
    rows, V = w.rows, w.vocab
    if op in ("logp", "logp_ent", "logp_bwd", "logp_ent_bwd"):
        live = rows if w.row_mask is None else int(w.row_mask.sum().item())
        mask = 0 if w.row_mask is None else rows
        if op == "logp":
            return live * V * es + rows * k * 8 + rows * k * 4 + mask
        if op == "logp_ent":  # + one fp32 entropy per row
            return live * V * es + rows * k * 8 + rows * k * 4 + rows * 4 + mask
        # logits in, dlogits out, index + upstream gradient + saved log-probs
        # (+ dL/dH and the saved entropy per row)
        ent = rows * 8 if op == "logp_ent_bwd" else 0
        return live * V * es + rows * V * es + rows * k * (8 + 4 + 4) + mask + ent
    live = int((w.labels != workloads.IGNORE_INDEX).sum().item())
    read = live * V * es + rows * 8
    if op == "ce_fwd":
        return read + rows * 4
    if op == "ce_bwd":
        return read + rows * V * es + rows * 4
    return read + rows * V * es  # fused


class L2Flush:
    """Run before each lone timed call: a 512 MB write, larger than L2, so
    none of the call's inputs stay cached; then a 256 MB read of another
    buffer, so that L2 is left holding clean lines.  After the write alone,
    L2 is full of dirty lines, and a call smaller than L2 then writes about
    as many bytes back to HBM as it reads: the flush's traffic, timed as the
    call's."""

    def __init__(self, dev):
        self.w = torch.empty(128 * 1024 * 1024, dtype=torch.float32, device=dev)
        self.r = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)
        self.acc = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.fill_(1.0)
        torch.sum(self.r, dim=0, out=self.acc)


def time_op(fn, stream, reps, flush=None):
    """Median CUDA-event time (ms) of one call, L2 flushed (L2Flush) before
    each rep.

    The call is captured once in a CUDA graph and replayed, so the time is
    the GPU's and not the Python launch path's (the library's calls never
    synchronize or allocate, so they capture); eager calls if capture fails.
    """
    fn()
    torch.cuda.synchronize()
    run = fn
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        run = graph.replay
    except Exception:  # noqa: BLE001 - fall back to eager timing
        run = fn
    times = []
    for _ in range(reps + 2):
        if flush is not None:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times[2:])


L2_BYTES = 129 * 1024 * 1024  # GB300 L2


def time_op_steady(make, copies, reps=5):
    """Median per-call time (ms) of `copies` calls back to back, call i on
    copy i of the inputs, captured in one CUDA graph.

    For workloads smaller than L2: the copies together hold more than twice
    the L2, so each call's inputs were last touched `copies - 1` calls ago
    and come from HBM, as in time_op after a flush.  Unlike time_op's lone
    call, the call runs among others, so the fixed cost of getting one
    graph onto the GPU (the floor of a lone launch) is not in it.
    """
    fns = [make(i) for i in range(copies)]
    for f in fns:
        f()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for f in fns:
            f()
    times = []
    for _ in range(reps + 1):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) / copies)
    del graph
    return statistics.median(times[1:])


def launch_floor_ms(dev, stream):
    """time_op of a one-element fill after the same L2 flush: the floor that
    a lone launch's event time carries whatever its kernel does."""
    flush = L2Flush(dev)
    e = torch.zeros(1, device=dev)
    ms = time_op(lambda: e.fill_(0.0), stream, 20, flush)
    del flush
    return ms


def measure_configs(gbce, dev, stream, peak):
    """Every seeded workload, each op timed alone: ms, rows/s, GB/s, fraction."""
    flush = L2Flush(dev)
    out = {}

    def record(name, w, op, ms, k=1, steady=None):
        nb = op_bytes(w, op, k)
        gbs = nb / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 5), "rows_per_s": round(w.rows / (ms * 1e-3)),
                     "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4), "bytes": nb}
        if steady is not None:
            # back to back over rotating copies of the inputs (time_op_steady)
            out[name]["ms_steady"] = round(steady, 5)
            out[name]["frac_steady"] = round(nb / (steady * 1e-3) / 1e9 / peak, 4)

    def copies_for(w):
        """Input copies for time_op_steady (None: the workload exceeds L2)."""
        nb = w.logits.numel() * w.logits.element_size()
        if nb >= (256 << 20):
            return None
        return max(2, min(512, -(-(5 * L2_BYTES // 2) // nb)))

    def ce_ops(tag, w, T, red, g, options=False):
        x, lab = w.logits, w.labels
        d = torch.empty_like(x)
        ws = gbce.new_workspace(w.rows, w.vocab, 1, device=dev)
        fwd = gbce.ce_fwd(x, lab, temperature=T, reduction=red, workspace=ws)
        fl = flush if w.logits.numel() * w.logits.element_size() < (256 << 20) else None
        n = copies_for(w)
        xs = [x] + [x.clone() for _ in range(n - 1)] if n else None
        ds = [d] + [torch.empty_like(x) for _ in range(n - 1)] if n else None

        def st(make):
            return time_op_steady(make, n) if n else None

        fused = lambda xi, di: gbce.ce_fwd_bwd_fused(xi, lab, g, temperature=T, reduction=red,  # noqa: E731
                                                     dlogits=di, workspace=ws)
        cfwd = lambda xi: gbce.ce_fwd(xi, lab, temperature=T, reduction=red, workspace=ws)  # noqa: E731
        cbwd = lambda xi, di: gbce.ce_bwd(xi, lab, g, fwd.logp, fwd.n_items, temperature=T,  # noqa: E731
                                          reduction=red, dlogits=di)
        record(f"{tag}/ce_fwd_bwd_fused", w, "fused", time_op(
            lambda: fused(x, d), stream, 10, fl),
            steady=st(lambda i: lambda: fused(xs[i], ds[i])))
        record(f"{tag}/ce_fwd", w, "ce_fwd", time_op(lambda: cfwd(x), stream, 10, fl),
               steady=st(lambda i: lambda: cfwd(xs[i])))
        record(f"{tag}/ce_bwd", w, "ce_bwd", time_op(lambda: cbwd(x, d), stream, 10, fl),
               steady=st(lambda i: lambda: cbwd(xs[i], ds[i])))
        if options:  # label smoothing 0.1 with DFT weights: the smoothing sum in the sweep
            kw = dict(temperature=T, reduction=red, label_smoothing=0.1, dft=True)
            record(f"{tag}/ce_fwd_bwd_fused+smooth+dft", w, "fused", time_op(
                lambda: gbce.ce_fwd_bwd_fused(x, lab, g, dlogits=d, workspace=ws, **kw),
                stream, 10, fl))
            record(f"{tag}/ce_fwd+smooth+dft", w, "ce_fwd", time_op(
                lambda: gbce.ce_fwd(x, lab, workspace=ws, **kw), stream, 10, fl))
            # logit soft-capping at 30: a tanh per element (and the fused
            # call as two passes)
            kc = dict(temperature=T, reduction=red, softcap=30.0)
            record(f"{tag}/ce_fwd_bwd_fused+softcap30", w, "fused", time_op(
                lambda: gbce.ce_fwd_bwd_fused(x, lab, g, dlogits=d, workspace=ws, **kc),
                stream, 10, fl))
            record(f"{tag}/ce_fwd+softcap30", w, "ce_fwd", time_op(
                lambda: gbce.ce_fwd(x, lab, workspace=ws, **kc), stream, 10, fl))

    def logp_op(tag, w, T, backward=False, k=None, entropy=False):
        x, idx = w.logits, (w.index if k is None else w.index[:, :k].contiguous())
        mask = w.row_mask
        K_ = idx.shape[1]
        o = torch.empty((w.rows, K_), dtype=torch.float32, device=dev)
        ws = gbce.new_workspace(w.rows, w.vocab, K_, device=dev)
        fl = flush if w.logits.numel() * w.logits.element_size() < (256 << 20) else None
        n = copies_for(w)
        xs = [x] + [x.clone() for _ in range(n - 1)] if n else None
        lp = lambda xi: gbce.selective_logsoftmax(xi, idx, T, mask, out=o, workspace=ws)  # noqa: E731
        record(f"{tag}/selective_logsoftmax", w, "logp", time_op(
            lambda: lp(x), stream, 10, fl), k=K_,
            steady=time_op_steady(lambda i: lambda: lp(xs[i]), n) if n else None)
        if entropy:
            h = torch.empty(w.rows, dtype=torch.float32, device=dev)
            le = lambda xi: gbce.selective_logsoftmax(xi, idx, T, mask, out=o, entropy_out=h,  # noqa: E731
                                                      workspace=ws)
            record(f"{tag}/selective_logsoftmax+entropy", w, "logp_ent", time_op(
                lambda: le(x), stream, 10, fl), k=K_,
                steady=time_op_steady(lambda i: lambda: le(xs[i]), n) if n else None)
        if backward:
            g = torch.ones((w.rows, K_), device=dev)
            d = torch.empty_like(x)
            record(f"{tag}/selective_logsoftmax_bwd", w, "logp_bwd", time_op(
                lambda: gbce.selective_logsoftmax_bwd(x, idx, g, o, T, mask, dlogits=d),
                stream, 10, fl), k=K_)
            if entropy:
                gh = torch.full((w.rows,), 0.01, device=dev)
                record(f"{tag}/selective_logsoftmax_bwd+entropy", w, "logp_ent_bwd", time_op(
                    lambda: gbce.selective_logsoftmax_bwd(x, idx, g, o, T, mask, grad_entropy=gh,
                                                          saved_entropy=h, dlogits=d),
                    stream, 10, fl), k=K_)

    w = workloads.ce_small_fp32(device=dev)
    ce_ops("ce_small_fp32_64x4096", w, 1.0, "mean", torch.ones(1, device=dev))
    logp_op("ce_small_fp32_64x4096", w, 1.0)
    w = workloads.ce_sparse_bf16(device=dev)
    ce_ops("ce_sparse_bf16_1922x4096", w, 1.0, "none", w.grad_out)
    w = workloads.logp_bf16(device=dev)
    logp_op("logp_bf16_1024x32768_T1.0", w, 1.0)
    logp_op("logp_bf16_1024x32768_T0.9", w, 0.9)
    for dt, tag in ((torch.float32, "fp32"), (torch.bfloat16, "bf16")):
        w = workloads.collapse_stress(dtype=dt, device=dev)
        ce_ops(f"collapse_{tag}_2048x151936", w, 1.0, "mean", torch.ones(1, device=dev))
        logp_op(f"collapse_{tag}_2048x151936", w, 1.0, entropy=True)
        del w
    # few rows, large vocabulary: the split-vocab partial + combine path
    w = workloads.grpo_bf16(device=dev, rows=64, seed=7)
    ce_ops("split_bf16_64x152064", w, TEMPERATURE, "mean", torch.ones(1, device=dev))
    logp_op("split_bf16_64x152064", w, TEMPERATURE, entropy=True)
    # sparse supervision at full size: 25% of the rows carry a label
    w = workloads.sft_sparse_bf16(device=dev)
    ce_ops(w.name, w, 1.0, "mean", torch.ones(1, device=dev))
    del w
    w = workloads.grpo_bf16(device=dev, rows=ROWS)
    ce_ops(f"grpo_bf16_{ROWS}x{VOCAB}", w, TEMPERATURE, "mean", torch.ones(1, device=dev),
           options=True)
    logp_op(f"grpo_bf16_{ROWS}x{VOCAB}_k4", w, TEMPERATURE, backward=True, entropy=True)
    logp_op(f"grpo_bf16_{ROWS}x{VOCAB}_k1", w, TEMPERATURE, backward=True, k=1, entropy=True)
    del w, flush
    torch.cuda.empty_cache()
    out["_launch_floor"] = {"ms": round(launch_floor_ms(dev, stream), 5),
                            "what": "time_op of a one-element fill: the event time of any "
                                    "lone launch after the flush starts here"}
    return out


def run_e2e(gbce, w, dev, stream, args, world, blocks=8):
    """Same metric through the Python API with pinned host buffers copied per step.

    Each step copies all of the step's inputs from pinned host memory and
    reads the log-probs and the loss back.  The rows go in `blocks` row
    blocks: block b's host-to-device copy runs on a copy stream while block
    b-1 computes, so the compute hides behind the copy (which is the bound:
    one pinned copy engine stream moves about 211 GB/s on GB300 machines).  The
    mean over all rows is taken as per-block sums with upstream gradient
    1 / n_items (n_items from the host's own labels) and the partial losses
    added on the host, the same loss and gradient as one mean-reduced call.
    The gradient (dlogits, 2.49 GB) stays on the device, where a training
    step consumes it; only the log-probs and the block losses come back.
    """
    steps = max(3, min(args.steps, 20))
    rows = w.rows
    h_x = w.logits.cpu().pin_memory()
    h_idx = w.index.cpu().pin_memory()
    h_lab = w.labels.cpu().pin_memory()
    d_x = torch.empty_like(w.logits)
    d_idx = torch.empty_like(w.index)
    d_lab = torch.empty_like(w.labels)
    h_logp = torch.empty((rows, K), dtype=torch.float32).pin_memory()
    h_loss = torch.empty((blocks,), dtype=torch.float32).pin_memory()
    d_loss = torch.empty((blocks,), dtype=torch.float32, device=dev)
    d_logp = torch.empty((rows, K), dtype=torch.float32, device=dev)
    dlogits = torch.empty_like(w.logits)
    n_items = int((h_lab != workloads.IGNORE_INDEX).sum().item())
    grad = torch.full((1,), 1.0 / max(n_items, 1), device=dev)
    bounds = [rows * b // blocks for b in range(blocks + 1)]
    wss = [gbce.new_workspace(bounds[b + 1] - bounds[b], VOCAB, K, device=dev)
           for b in range(blocks)]
    copy_stream = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(blocks)]

    def one():
        copy_stream.wait_stream(stream)  # the previous step is done with the buffers
        with torch.cuda.stream(copy_stream):
            for b in range(blocks):
                r0, r1 = bounds[b], bounds[b + 1]
                d_x[r0:r1].copy_(h_x[r0:r1], non_blocking=True)
                d_idx[r0:r1].copy_(h_idx[r0:r1], non_blocking=True)
                d_lab[r0:r1].copy_(h_lab[r0:r1], non_blocking=True)
                ready[b].record(copy_stream)
        for b in range(blocks):
            r0, r1 = bounds[b], bounds[b + 1]
            stream.wait_event(ready[b])
            gbce.selective_logsoftmax(d_x[r0:r1], d_idx[r0:r1], TEMPERATURE,
                                      out=d_logp[r0:r1], workspace=wss[b])
            out = gbce.ce_fwd_bwd_fused(d_x[r0:r1], d_lab[r0:r1], grad, temperature=TEMPERATURE,
                                        reduction="sum", dlogits=dlogits[r0:r1],
                                        workspace=wss[b], want_logp=False)
            d_loss[b:b + 1].copy_(out.loss.reshape(1))
        h_logp.copy_(d_logp, non_blocking=True)
        h_loss.copy_(d_loss, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        one()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    # the step's mean loss from the blocks' sums, as read back
    loss = float(h_loss.double().sum()) / max(n_items, 1)
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    h2d = h_x.numel() * h_x.element_size() + h_idx.numel() * 8 + h_lab.numel() * 8
    d2h = h_logp.numel() * 4 + h_loss.numel() * 4
    value = aggregate_gbs(world, algorithmic_bytes()["step"], steps, ms)
    del h_x, d_x, dlogits
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": ms / steps, "row_blocks": blocks,
            "loss": loss}


def cpu_baseline(w):
    import oracle

    oracle.build()
    n_rows = oracle_rows_for(10.0, w)
    sample = host_sample(w, n_rows)
    secs = time_oracle_sample(sample)
    value = algorithmic_bytes(rows=n_rows)["step"] / secs / 1e9
    return {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n_rows} of {ROWS} rows (selective logp K=4 + CE fwd+bwd), "
                      f"{secs:.1f} s, fp64 oracle, OpenMP over rows"}


PROFILE_CASES = ("ce", "logp", "fused", "split", "slice")


def run_profile_case(case: str, rows: int = 1024):
    """One launch of every op of a kernel family, nothing else, for ncu.

    On `rows` of the packed workload (64 for "split", the few-row cluster
    path): "ce" = ce_fwd plain / label-smoothed / soft-capped
    (30) / capped + smoothed, ce_bwd plain / capped; "logp" = selective
    log-softmax K = 4 with and without the entropy and both backwards;
    "fused" = ce_fwd_bwd_fused plain / smoothed + DFT / capped; "split" =
    selective log-softmax, ce_fwd and the fused call on 64 rows; "slice" =
    vocab_slice_stats on two halves, the combine and one slice's gradient.
    """
    import __graft_entry__

    __graft_entry__.build()
    import cross_entropy_gb300 as gbce

    dev = torch.device("cuda:0")
    rows = 64 if case == "split" else rows
    w = workloads.grpo_bf16(device=dev, rows=rows, seed=3)
    x, idx, lab, V = w.logits, w.index, w.labels, w.vocab
    d = torch.empty_like(x)
    g1 = torch.ones(1, device=dev)
    g4 = torch.ones((rows, K), device=dev)
    ws = gbce.new_workspace(rows, V, K, device=dev)
    o = torch.empty((rows, K), dtype=torch.float32, device=dev)
    h = torch.empty(rows, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    T = TEMPERATURE
    if case == "ce":
        fwd = gbce.ce_fwd(x, lab, temperature=T, workspace=ws)
        gbce.ce_fwd(x, lab, temperature=T, workspace=ws, label_smoothing=0.1)
        gbce.ce_bwd(x, lab, g1, fwd.logp, fwd.n_items, temperature=T, dlogits=d)
        fc = gbce.ce_fwd(x, lab, temperature=T, workspace=ws, softcap=30.0)
        gbce.ce_bwd(x, lab, g1, fc.logp, fc.n_items, temperature=T, dlogits=d, softcap=30.0)
        gbce.ce_fwd(x, lab, temperature=T, workspace=ws, softcap=30.0, label_smoothing=0.1)
    elif case == "logp":
        gbce.selective_logsoftmax(x, idx, T, out=o, workspace=ws)
        gbce.selective_logsoftmax(x, idx, T, out=o, entropy_out=h, workspace=ws)
        gbce.selective_logsoftmax_bwd(x, idx, g4, o, T, dlogits=d)
        gbce.selective_logsoftmax_bwd(x, idx, g4, o, T, dlogits=d, saved_entropy=h,
                                      grad_entropy=torch.full((rows,), 0.01, device=dev))
    elif case == "fused":
        gbce.ce_fwd_bwd_fused(x, lab, g1, temperature=T, dlogits=d, workspace=ws)
        gbce.ce_fwd_bwd_fused(x, lab, g1, temperature=T, dlogits=d, workspace=ws,
                              label_smoothing=0.1, dft=True)
        gbce.ce_fwd_bwd_fused(x, lab, g1, temperature=T, dlogits=d, workspace=ws, softcap=30.0)
    elif case == "split":
        gbce.selective_logsoftmax(x, idx, T, out=o, workspace=ws)
        gbce.ce_fwd(x, lab, temperature=T, workspace=ws)
        gbce.ce_fwd_bwd_fused(x, lab, g1, temperature=T, dlogits=d, workspace=ws)
    elif case == "slice":
        cuts = [0, V // 2, V]
        parts = torch.stack([gbce.vocab_slice_stats(x[:, a:b], idx, a, V, T)
                             for a, b in zip(cuts[:-1], cuts[1:])])
        lp, xt0, state = gbce.vocab_slice_combine(parts, cuts, idx, T)
        gbce.vocab_slice_grad(x[:, :cuts[1]], idx, 0, V, g4, lp, xt0, T, row_state=state)
    torch.cuda.synchronize()
    print(f"profile case {case}: done", flush=True)


def main():
    global ROWS
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gbce", "reference"], default="gbce")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload, per-op timings")
    ap.add_argument("--entropy", action="store_true",
                    help="the step's selective log-softmax also writes each row's entropy")
    ap.add_argument("--rows", type=int, default=None,
                    help="rows of the workload (a smaller case for profiling captures; "
                         f"default {ROWS}, or 1024 with --profile-case)")
    ap.add_argument("--profile-case", choices=PROFILE_CASES,
                    help="launch every op of one kernel family once (for ncu) and exit")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case, args.rows or 1024)
        return
    ROWS = args.rows or ROWS
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gbce(args)


if __name__ == "__main__":
    main()
