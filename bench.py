"""Benchmark: RMSNorm and fused residual-add RMSNorm on GB300, HBM GB/s against the roofline.

One step is one pass of the whole hot path over one batch: ks_rms_norm (x -> y) and
ks_fused_add_rms_norm (x2, residual in place) on the large prefill shape [32768, 8192] bf16,
eps 1e-5, x and residual ~ N(0,1), weight = 1 + 0.1 N(0,1) (seeded, drawn on the device).
Every tensor (512 MiB) is larger than the 129 MB L2, so no flush is needed between steps.

Bytes counted per step are the algorithmic bytes (each element read once and written once):
rms_norm 2*R*H*e + H*e, fused 4*R*H*e + H*e (Triton Kernels, "Kernels" table and "Benchmark
results"; Triton Kernel Lab, "Decode Kernel Results" counts the same four tensor passes plus
the weight for its residual RMSNorm).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ks|reference]

Under torchrun each rank runs one full batch on its own GPU (rows are independent, so no
collective touches the data; weak scaling); rank 0 prints one JSON line with the max time
over ranks. Timing follows the pages' method: CUDA events on the launching stream, warm-up
first, p50 per launch, and no timing is published unless the oracle agrees on sampled rows
(Triton Kernel Lab, "Quick Start": the benchmark refuses to publish when a correctness case
fails). The oracle runs only in the CPU-baseline leg (and in --impl reference).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "RMSNorm / fused-add RMSNorm HBM GB/s (% of GB300 peak) and p50 µs"
# the workload the headline is quoted on; --rows/--hidden name smaller cases (profiling captures)
FULL_ROWS, FULL_HIDDEN = 32768, 8192


def workload(rows: int, hidden: int) -> str:
    kind = "large prefill bf16" if (rows, hidden) == (FULL_ROWS, FULL_HIDDEN) else "bf16"
    return (f"{kind}: rms_norm + fused_add_rms_norm on x, residual [{rows},{hidden}] "
            f"({rows * hidden * 2 / 2**20:.0f} MiB per tensor), weight 1+0.1N(0,1), eps=1e-5")


def device_facts(dev) -> dict:
    """The device's SM count and L2 size, as the runtime reports them."""
    import torch
    p = torch.cuda.get_device_properties(dev)
    return {"sm_count": int(p.multi_processor_count), "l2_bytes": int(p.L2_cache_size)}


def l2_note(rows: int, hidden: int, l2_bytes: int) -> str:
    mib = rows * hidden * 2 / 2**20
    l2 = f"L2 ({l2_bytes / 2**20:.0f} MiB, device query)"
    if rows * hidden * 2 > l2_bytes:
        return f"no flush: every tensor ({mib:.0f} MiB) is larger than {l2}"
    return f"no flush, and the tensors ({mib:.1f} MiB) fit in {l2}: not a bench figure"


FALLBACK_HBM_GBS = 6800.0
C2C_NOMINAL_GBS = 900.0  # NVLink-C2C between Grace and the GPU, both directions together
# what decides the recorded launches' DRAM traffic: the kernels, and the plan code that picks
# their launch shape (a change to either invalidates the record). The generated band table is
# left out of the hash: the record names each launch's plan instead, checked against the plan
# the library picks now, so re-deriving bands of other widths keeps the record.
KERNEL_SOURCES = ["row_wise_rmsnorm_ks_gb300/csrc/ks_kernels.cuh",
                  "row_wise_rmsnorm_ks_gb300/csrc/ks_ptx.cuh",
                  "row_wise_rmsnorm_ks_gb300/csrc/ks_abi.cu"]
GENERATED_BANDS = re.compile(r"// BEGIN GENERATED ROW BANDS\n.*?// END GENERATED ROW BANDS", re.S)
PLAN_FIELDS = ("kernel", "vec_per_thread", "team", "block", "flags", "cluster", "stages")
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "ncu_dram_traffic.json")


def algorithmic_bytes(op: str, rows: int, hidden: int, elem: int) -> int:
    """Bytes an ideal kernel moves: each row element read once and written once, the weight
    read once per launch."""
    passes = 2 if op == "rms_norm" else 4
    return passes * rows * hidden * elem + hidden * elem


def whole_job_gbs(world: int, step_bytes: int, steps: int, elapsed_ms: float) -> float:
    """Aggregate throughput: the bytes every rank moved over the slowest rank's time."""
    return world * step_bytes * steps / (elapsed_ms * 1e-3) / 1e9


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws an independent batch (rows shard across GPUs with no exchange)."""
    return base + 1000 * rank


def max_over_ranks(value: float, device=None) -> float:
    """The maximum of `value` over all ranks of the default process group (or `value` alone)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def code_only(src: str) -> str:
    """C++ source with comments removed and whitespace collapsed: what the compiler sees, so that
    an edit to a comment does not mark recorded counters as stale."""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif src[i] in "\"'":
            q, j = src[i], i + 1
            while j < n and src[j] != q:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(src[i])
            i += 1
    return " ".join("".join(out).split())


def kernel_source_sha() -> str:
    """Hash of the kernel and plan sources' code (comments and layout ignored)."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(GENERATED_BANDS.sub("", f.read())).encode())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured (MEASURED_PEAKS.json)"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback 6.8 TB/s"}


def recorded_traffic(op: str, rows: int = FULL_ROWS, hidden: int = FULL_HIDDEN, plan=None):
    """Per-launch DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) from the
    committed record, if it was taken on the current kernel and plan sources, the launch has the
    recorded shape, and `plan` (the library's plan for it now, a ks_plan_t) is the recorded one
    (else None)."""
    if not os.path.exists(TRAFFIC_RECORD):
        return None
    with open(TRAFFIC_RECORD) as f:
        rec = json.load(f)
    if rec.get("sources_sha") != kernel_source_sha():
        return None
    ent = rec.get("launches", {}).get(op)
    if not ent or [rows, hidden] != ent.get("shape"):
        return None
    if plan is None or ent.get("plan") != {k: getattr(plan, k) for k in PLAN_FIELDS}:
        return None
    return int(ent["dram_read_bytes"]) + int(ent["dram_write_bytes"])


# --------------------------------------------------------------------------- clock sampler

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu_index = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.6)  # let the first samples arrive before the timed region
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = list(csv.reader(io.StringIO(out)))
        load, reasons, maxes, allsm = [], set(), [], []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 10:
                continue
            r = [c.strip() for c in r]
            try:
                ts = time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                sm, smmax = float(r[2]), float(r[3])
            except ValueError:
                continue
            allsm.append(sm)
            maxes.append(smmax)
            if self.t0 is not None and self.t0 - 1 <= ts <= self.t1 + 1:
                load.append(sm)
                for n, v in zip(names, r[6:10]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        samples = load or allsm
        return {"sm_mhz": statistics.median(samples) if samples else None,
                "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples": len(load)}


# ------------------------------------------------------------------------------ ks arm

def run_ks(args) -> int:
    import torch
    import torch.distributed as dist

    from row_wise_rmsnorm_ks_gb300 import _abi, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    _abi.load()
    facts = device_facts(dev)

    R, H, e = args.rows, args.hidden, 2
    eps = 1e-5
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    # Inputs, resident in HBM before the timed region. Each rank draws its own batch.
    x = synth.cast(synth.normal_dev((R, H), rank_seed(synth.SEED_X, rank), dev), "bf16")
    xf = x.clone()
    r = synth.cast(synth.normal_dev((R, H), rank_seed(synth.SEED_RESIDUAL, rank), dev), "bf16")
    w = synth.weight(H, "bf16").to(dev)
    y = torch.empty_like(x)
    torch.cuda.synchronize()

    # Pristine copies of the rows the CPU-baseline leg will recompute.
    S = min(R, args.cpu_rows_max)
    host_in = {"x": x[:S].cpu(), "xf": xf[:S].cpu(), "r": r[:S].cpu(), "w": w.cpu()}

    def ks_plain():
        return _abi.ks_rms_norm(y.data_ptr(), x.data_ptr(), w.data_ptr(), R, H, eps,
                                _abi.KS_DTYPE_BF16, sh)

    def ks_fused():
        return _abi.ks_fused_add_rms_norm(xf.data_ptr(), r.data_ptr(), w.data_ptr(), R, H, eps,
                                          _abi.KS_DTYPE_BF16, sh)

    # First step on pristine inputs: its outputs are what the oracle is compared with.
    _abi.check(ks_plain())
    _abi.check(ks_fused())
    torch.cuda.synchronize()
    gpu_out = {"y": y[:S].cpu(), "x": xf[:S].cpu(), "r": r[:S].cpu()}
    for _ in range(max(0, args.warmup - 1)):
        ks_plain()
        ks_fused()
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps, barrier + synchronize on both sides. One event per
    # kernel boundary: ev[2k] before step k's rms_norm, ev[2k+1] between its two kernels,
    # ev[2k+2] after its fused kernel (and before step k+1's rms_norm); ev[0] and ev[2K] bound
    # the region. Each event record costs the stream about a microsecond on this part, so no
    # boundary carries two.
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps + 1)]
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark_begin()
    ev[0].record(stream)
    for k in range(args.steps):
        ks_plain()
        ev[2 * k + 1].record(stream)
        ks_fused()
        ev[2 * k + 2].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler.mark_end()
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(ev[0].elapsed_time(ev[-1]), dev)

    plain_ms = [ev[2 * k].elapsed_time(ev[2 * k + 1]) for k in range(args.steps)]
    fused_ms = [ev[2 * k + 1].elapsed_time(ev[2 * k + 2]) for k in range(args.steps)]
    b_plain = algorithmic_bytes("rms_norm", R, H, e)
    b_fused = algorithmic_bytes("fused_add_rms_norm", R, H, e)
    step_bytes = b_plain + b_fused
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_gbs(world, step_bytes, args.steps, elapsed_ms)

    peaks = measured_peaks()
    fused_avg_s = statistics.fmean(fused_ms) * 1e-3
    plain_avg_s = statistics.fmean(plain_ms) * 1e-3
    achieved = b_fused / fused_avg_s / 1e9
    ops = {
        "rms_norm": {"bytes_per_launch": b_plain, "p50_us": statistics.median(plain_ms) * 1e3,
                     "avg_us": plain_avg_s * 1e6, "gbs": b_plain / plain_avg_s / 1e9,
                     "frac_of_peak": b_plain / plain_avg_s / 1e9 / peaks["hbm_gbs"]},
        "fused_add_rms_norm": {"bytes_per_launch": b_fused,
                               "p50_us": statistics.median(fused_ms) * 1e3,
                               "avg_us": fused_avg_s * 1e6, "gbs": achieved,
                               "frac_of_peak": achieved / peaks["hbm_gbs"]},
    }

    result = {}
    if rank == 0:
        ops["step_chain"] = step_chain(ks_plain, ks_fused, stream, step_bytes,
                                       measured_peaks()["hbm_gbs"])
        # decode shape (launch-bound): p50 of single cache-cold launches, and graph replay
        if not args.no_decode:
            ops["decode_fused_add_rms_norm_4x1536"] = decode_latency(dev, args)
            ops["pages_latency_shapes"] = pages_shapes_latency(dev, args)
        if not args.no_next_ops:
            ops["next_ops"] = next_ops(dev, args)
        e2e = run_e2e(dev, args, R, H, eps) if not args.no_e2e else None
        cpu = cpu_baseline_and_parity(host_in, gpu_out, R, H, eps, args)
        if not cpu["parity"]["ok"]:
            print(json.dumps({"error": "parity check failed; no timing published",
                              "parity": cpu["parity"]}))
            return 1
        traffic = recorded_traffic("fused_add_rms_norm", R, H, _abi.ks_plan_launch(
            1, R, H, _abi.KS_DTYPE_BF16, True, facts["sm_count"], 0)[1])
        result = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) drawn on the device)",
            "config": {"workload": workload(R, H), "rows": R, "hidden": H, "eps": eps,
                       "accumulate": "f32",
                       "l2": l2_note(R, H, facts["l2_bytes"]),
                       "parallelism": f"rows: one independent batch per GPU x{world}",
                       "kernel_plan": {
                           "rms_norm": _abi.ks_plan_launch(0, R, H, 2, True, facts["sm_count"], 0)[1].as_dict()["kernel_name"],
                           "fused_add_rms_norm": _abi.ks_plan_launch(1, R, H, 2, True, facts["sm_count"], 0)[1].as_dict()["kernel_name"]}},
            "roofline": {"bound": "hbm", "kernel": f"fused_add_rms_norm (bf16 [{R},{H}])",
                         "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "algorithmic_bytes": b_fused, "peak_source": peaks["source"]},
            "cpu_baseline": cpu["baseline"],
            "parity": cpu["parity"],
            "e2e": e2e,
            "gpu_launches": 2 * args.steps,
            "clocks": clocks,
            "ops": ops,
        }
        print(json.dumps(result))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def step_chain(ks_plain, ks_fused, stream, step_bytes: int, peak_gbs: float,
               steps: int = 200) -> dict:
    """The bench step with no event between its kernels, as a model runs it: `steps` steps timed
    by one pair of events, with the library's default launches and with programmatic dependent
    launch (KS_LAUNCH_PDL: each kernel is scheduled while the previous one drains and waits for
    its writes before its first memory access). Reported beside the timed region, whose events
    at every kernel boundary keep each launch apart; this shows what those boundaries cost."""
    import torch

    from row_wise_rmsnorm_ks_gb300 import _abi

    out = {"steps": steps}
    for key, opt in (("no_events", 0), ("no_events_pdl", _abi.KS_LAUNCH_PDL)):
        _abi.check(_abi.ks_set_launch_options(opt))
        try:
            for _ in range(3):
                _abi.check(ks_plain())
                _abi.check(ks_fused())
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(steps):
                ks_plain()
                ks_fused()
            b.record(stream)
            torch.cuda.synchronize()
        finally:
            _abi.ks_set_launch_options(0)
        us = a.elapsed_time(b) * 1e3 / steps
        out[f"us_per_step_{key}"] = us
        out[f"frac_of_peak_{key}"] = step_bytes / us / 1e3 / peak_gbs
    return out


def decode_latency(dev, args) -> dict:
    """Fused op on the decode shape [4, 1536] bf16 (launch-bound). Reported: single launches
    timed with CUDA events around each launch, cold (an L2 flush by a 512 MiB write outside the
    timed pair, the pages' cache-cold method; the flush keeps the GPU busy while the launch is
    queued, so the pair times the kernel) and hot (the GPU idles, so the pair also times this
    Python caller's launch path); and the per-launch time of a CUDA graph of 100 back-to-back
    dependent launches, without and with programmatic dependent launch."""
    import torch

    from row_wise_rmsnorm_ks_gb300 import _abi, synth

    wl = synth.decode()
    x, r, w = wl.x.to(dev), wl.residual.to(dev), wl.weight.to(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def launch(s):
        return _abi.ks_fused_add_rms_norm(x.data_ptr(), r.data_ptr(), w.data_ptr(), 4, 1536,
                                          wl.eps, _abi.KS_DTYPE_BF16, s)

    for _ in range(20):
        launch(stream.cuda_stream)

    def single(cold):
        out = []
        for _ in range(args.decode_samples):
            if cold:
                flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch(stream.cuda_stream)
            b.record(stream)
            b.synchronize()
            out.append(a.elapsed_time(b) * 1e3)
        out.sort()
        return out

    def graph_per_launch(pdl):
        _abi.ks_set_launch_options(_abi.KS_LAUNCH_PDL if pdl else 0)
        try:
            g = torch.cuda.CUDAGraph()
            cs = torch.cuda.Stream(dev)
            cs.wait_stream(stream)
            with torch.cuda.stream(cs):
                launch(cs.cuda_stream)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=cs):
                for _ in range(100):
                    launch(cs.cuda_stream)
        finally:
            _abi.ks_set_launch_options(0)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * 100)

    cold, hot = single(True), single(False)
    q = lambda v, p: v[min(len(v) - 1, int(p * len(v)))]
    return {"bytes_per_launch": algorithmic_bytes("fused_add_rms_norm", 4, 1536, 2),
            "p50_us_cold_event": q(cold, 0.5), "p95_us_cold_event": q(cold, 0.95),
            "p99_us_cold_event": q(cold, 0.99),
            "p50_us_hot_event_incl_python_launch": q(hot, 0.5),
            "us_per_launch_graph_replay": graph_per_launch(False),
            "us_per_launch_graph_replay_pdl": graph_per_launch(True),
            "samples": len(cold)}


# The pages' latency table (Triton Kernel Lab, "Measured Result" and "Decode Kernel Results"; RTX
# 5070 Ti, cache-cold CUDA events, 100 warm-ups, 500 samples, p50), shape for shape: op, dtype,
# rows, hidden, and the pages' p50 in microseconds (context: another GPU).
PAGES_LATENCY_SHAPES = [("rms_norm", "fp16", 128, 1024, 5.8), ("rms_norm", "fp16", 512, 4096, 13.5),
                        ("rms_norm", "fp16", 2048, 4096, 42.7),
                        ("fused_add_rms_norm", "bf16", 4, 1536, 5.1)]


def pages_shapes_latency(dev, args) -> dict:
    """The pages' latency shapes by their method: 100 warm-up launches, then single launches timed
    with CUDA events, each after the L2 is flushed (a 512 MiB write outside the timed pair);
    p50/p95/p99 over --decode-samples samples. Also the per-launch time of 100 back-to-back launches
    replayed from a CUDA graph (inputs hot in L2). N(0,1) inputs; fused residual N(0, var 4)."""
    import torch

    from row_wise_rmsnorm_ks_gb300 import _abi, synth

    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    codes = {"bf16": _abi.KS_DTYPE_BF16, "fp16": _abi.KS_DTYPE_F16}
    out = {}
    for op, dt, R, H, pages_us in PAGES_LATENCY_SHAPES:
        code = codes[dt]
        x = synth.cast(synth.normal_dev((R, H), synth.SEED_X, dev), dt)
        r = synth.cast(synth.normal_dev((R, H), synth.SEED_RESIDUAL, dev, std=2.0), dt)
        w = synth.weight(H, dt).to(dev)
        y = torch.empty_like(x)
        if op == "rms_norm":
            launch = lambda st: _abi.ks_rms_norm(y.data_ptr(), x.data_ptr(), w.data_ptr(), R, H,
                                                 1e-6, code, st)
        else:
            launch = lambda st: _abi.ks_fused_add_rms_norm(x.data_ptr(), r.data_ptr(),
                                                           w.data_ptr(), R, H, 1e-6, code, st)
        for _ in range(100):
            launch(stream.cuda_stream)
        samples = []
        for _ in range(args.decode_samples):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch(stream.cuda_stream)
            b.record(stream)
            b.synchronize()
            samples.append(a.elapsed_time(b) * 1e3)
        samples.sort()
        cs = torch.cuda.Stream(dev)
        cs.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            for _ in range(100):
                launch(cs.cuda_stream)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(10):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        q = lambda p: samples[min(len(samples) - 1, int(p * len(samples)))]
        nb = algorithmic_bytes(op, R, H, 2)
        out[f"{op} {dt} [{R},{H}]"] = {
            "bytes_per_launch": nb, "p50_us_cold_event": q(0.5), "p95_us_cold_event": q(0.95),
            "p99_us_cold_event": q(0.99), "gbs_at_p50": nb / (q(0.5) * 1e-6) / 1e9,
            "us_per_launch_graph_replay": a.elapsed_time(b) * 1e3 / 1000,
            "pages_p50_us_other_gpu": pages_us, "samples": len(samples)}
        del x, r, w, y
    # The floor of this method on this GPU: the same protocol around a one-element torch fill
    one = torch.empty(1, device=dev)
    for _ in range(100):
        one.fill_(0)
    floor = []
    for _ in range(args.decode_samples):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        one.fill_(0)
        b.record(stream)
        b.synchronize()
        floor.append(a.elapsed_time(b) * 1e3)
    floor.sort()
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        for _ in range(100):
            one.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(10):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    out["method floor: one-element torch fill, same protocol"] = {
        "p50_us_cold_event": floor[len(floor) // 2], "samples": len(floor),
        "us_per_launch_graph_replay": a.elapsed_time(b) * 1e3 / 1000}
    return out


def next_ops(dev, args) -> dict:
    """SwiGLU, Softmax and LayerNorm (the library's next operators): HBM GB/s on large bf16
    shapes (CUDA events over back-to-back launches; every tensor larger than L2) and the
    per-launch time of a CUDA graph on the pages' small shapes."""
    import torch

    from row_wise_rmsnorm_ks_gb300 import _abi, synth

    s = torch.cuda.current_stream(dev)
    peak = measured_peaks()["hbm_gbs"]
    BF = _abi.KS_DTYPE_BF16

    def events(fn, n):
        for _ in range(3):
            fn(s.cuda_stream)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(n):
            fn(s.cuda_stream)
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e-3 / n

    def graph_us(fn, n=100, reps=10):
        cs = torch.cuda.Stream(dev)
        cs.wait_stream(s)
        with torch.cuda.stream(cs):
            fn(cs.cuda_stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            for _ in range(n):
                fn(cs.cuda_stream)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(reps):
            g.replay()
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (n * reps)

    out = {}
    R, D = args.next_rows, 8192
    x = synth.cast(synth.normal_dev((R, 2 * D), 11, dev), "bf16")
    y = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
    nb = 3 * R * D * 2
    t = events(lambda st: _abi.ks_silu_and_mul(y.data_ptr(), x.data_ptr(), R, D, BF, st), 100)
    xs = synth.cast(synth.normal_dev((512, 8192), 12, dev), "bf16")
    ys = torch.empty((512, 4096), dtype=torch.bfloat16, device=dev)
    out["silu_and_mul"] = {
        "shape": f"[{R},{2 * D}] -> [{R},{D}] bf16", "bytes_per_launch": nb, "avg_us": t * 1e6,
        "gbs": nb / t / 1e9, "frac_of_peak": nb / t / 1e9 / peak,
        "us_per_launch_graph_512x8192": graph_us(
            lambda st: _abi.ks_silu_and_mul(ys.data_ptr(), xs.data_ptr(), 512, 4096, BF, st))}
    del x, y
    H = 8192
    x = synth.cast(synth.normal_dev((R, H), 13, dev), "bf16")
    y = torch.empty_like(x)
    nb = 2 * R * H * 2
    t = events(lambda st: _abi.ks_softmax(y.data_ptr(), x.data_ptr(), R, H, BF, st), 100)
    xs = synth.cast(synth.normal_dev((512, 1024), 14, dev), "bf16")
    ys = torch.empty_like(xs)
    out["softmax"] = {
        "shape": f"[{R},{H}] bf16", "bytes_per_launch": nb, "avg_us": t * 1e6,
        "gbs": nb / t / 1e9, "frac_of_peak": nb / t / 1e9 / peak,
        "us_per_launch_graph_512x1024": graph_us(
            lambda st: _abi.ks_softmax(ys.data_ptr(), xs.data_ptr(), 512, 1024, BF, st))}
    w = synth.weight(H, "bf16").to(dev)
    bias = synth.cast(synth.normal_dev((H,), 15, dev, std=0.1), "bf16")
    nb = 2 * R * H * 2 + 2 * H * 2
    t = events(lambda st: _abi.ks_layer_norm(y.data_ptr(), x.data_ptr(), w.data_ptr(),
                                             bias.data_ptr(), R, H, 1e-5, BF, st), 100)
    out["layer_norm"] = {"shape": f"[{R},{H}] bf16, weight and bias", "bytes_per_launch": nb,
                         "avg_us": t * 1e6, "gbs": nb / t / 1e9,
                         "frac_of_peak": nb / t / 1e9 / peak}
    return out


def run_e2e(dev, args, R, H, eps) -> dict:
    """The same step through the public API with host buffers: ks.rms_norm_host and
    ks.fused_add_rms_norm_host take pinned host rows. Two modes are timed: direct (the kernels
    read and write the pinned rows over the host link) and staged (chunks copied through a device
    workspace, copies overlapping kernels). Either way every input byte crosses host->device and
    every output byte device->host inside the timed region; the faster mode is the e2e value."""
    import torch

    import row_wise_rmsnorm_ks_gb300 as ks
    from row_wise_rmsnorm_ks_gb300 import synth

    stream = torch.cuda.current_stream(dev)
    xh = synth.cast(synth.normal_dev((R, H), synth.SEED_X, dev), "bf16").cpu().pin_memory()
    x2h = xh.clone().pin_memory()
    rh = synth.cast(synth.normal_dev((R, H), synth.SEED_RESIDUAL, dev), "bf16").cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    w = synth.weight(H, "bf16").to(dev)
    nbytes = algorithmic_bytes("rms_norm", R, H, 2) + algorithmic_bytes("fused_add_rms_norm", R, H, 2)

    def timed(ws):
        def step():
            ks.rms_norm_host(xh, w, eps, workspace=ws, out=yh)
            ks.fused_add_rms_norm_host(x2h, rh, w, eps, workspace=ws)

        for _ in range(2):
            step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.e2e_steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.e2e_steps

    # The host link's own ceiling: pinned copies of 512 MiB one way, the other way, and both at
    # once on two streams (the e2e step moves equal bytes each way).
    blk = 256 << 20  # bf16 elements = 512 MiB
    hsrc = xh.view(-1)[:blk]
    hdst = torch.empty(blk, dtype=torch.bfloat16).pin_memory()
    dbuf = torch.empty(blk, dtype=torch.bfloat16, device=dev)
    dbuf2 = torch.empty(blk, dtype=torch.bfloat16, device=dev)
    s2 = torch.cuda.Stream(dev)

    def copy_time(h2d, d2h, reps=3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            if h2d:
                dbuf.copy_(hsrc, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s2):
                    hdst.copy_(dbuf2, non_blocking=True)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    copy_time(True, True, reps=1)  # warm both directions up
    nblk = blk * 2
    copies = {"h2d_gbs": nblk / copy_time(True, False) / 1e9,
              "d2h_gbs": nblk / copy_time(False, True) / 1e9,
              "both_directions_gbs": 2 * nblk / copy_time(True, True) / 1e9,
              "how": "pinned 512 MiB torch copy_ calls, wall clock over 3 repetitions (the "
                     "copy engines' rate, not the link's: the direct mode beats it)"}
    del hdst, dbuf, dbuf2

    ms_direct = timed(None)
    ws = torch.empty(args.e2e_workspace_mb << 20, dtype=torch.uint8, device=dev)
    ms_staged = timed(ws)
    del ws
    best = "direct" if ms_direct <= ms_staged else "staged"
    ms = min(ms_direct, ms_staged)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"value": gbs, "unit": "GB/s", "ms_per_step": ms,
            "steps": args.e2e_steps, "h2d_bytes_per_step": 3 * R * H * 2,
            "d2h_bytes_per_step": 3 * R * H * 2, "mode": best, "host_copies": copies,
            # every counted byte crosses the host link once (x, residual in; y, x, residual out)
            "link": {"name": "NVLink-C2C", "nominal_gbs_both_directions": C2C_NOMINAL_GBS,
                     "source": "NVIDIA's published Grace-Blackwell figure, not measured here",
                     "frac_of_nominal": gbs / C2C_NOMINAL_GBS},
            "direct_gbs": nbytes / (ms_direct * 1e-3) / 1e9,
            "staged_gbs": nbytes / (ms_staged * 1e-3) / 1e9,
            "api": "rms_norm_host + fused_add_rms_norm_host on pinned host rows (direct: kernels "
                   "address the host rows; staged: chunks through a "
                   f"{args.e2e_workspace_mb} MiB device workspace)"}


def host_cpu_model() -> str:
    """The host CPU's model name, best effort (/proc/cpuinfo on x86; on Arm hosts, whose cpuinfo
    names no model, the implementer and part numbers), else the platform's processor string."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key, val = key.strip().lower(), val.strip()
                if key and val and key not in fields:
                    fields[key] = val
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "cpu implementer" in fields and "cpu part" in fields:
        parts = {("0x41", "0xd4f"): "Arm Neoverse V2", ("0x41", "0xd40"): "Arm Neoverse V1",
                 ("0x41", "0xd0c"): "Arm Neoverse N1", ("0x41", "0xd49"): "Arm Neoverse N2"}
        key = (fields["cpu implementer"].lower(), fields["cpu part"].lower())
        return parts.get(key, f"Arm CPU (implementer {key[0]}, part {key[1]})")
    return platform.processor() or platform.machine()


def oracle_all_cores(host_in, rows: int, H: int, eps: float) -> dict:
    """The same oracle on the first `rows` rows of both ops, the rows split evenly over every
    host core (one thread each; the C oracle keeps no shared state and its calls release the
    interpreter lock). A second, separately labelled CPU figure beside the single-threaded
    baseline."""
    import concurrent.futures as cf

    import oracle

    n = max(1, min(os.cpu_count() or 1, rows))
    per = -(-rows // n)
    chunks = [slice(i, min(rows, i + per)) for i in range(0, rows, per)]

    def work(sl):
        oracle.rms_norm(host_in["x"][sl], host_in["w"], eps)
        oracle.fused_add_rms_norm(host_in["xf"][sl], host_in["r"][sl], host_in["w"], eps)

    oracle.rms_norm(host_in["x"][:1], host_in["w"], eps)  # load the library before the threads
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(work, chunks))
    secs = time.perf_counter() - t0
    nb = algorithmic_bytes("rms_norm", rows, H, 2) + algorithmic_bytes("fused_add_rms_norm", rows, H, 2)
    return {"value": nb / secs / 1e9, "unit": "GB/s", "cores": len(chunks),
            "kind": "oracle, rows split over threads",
            "sample": f"first {rows} rows of both ops ([{rows},{H}] bf16), {secs:.2f} s"}


def cpu_baseline_and_parity(host_in, gpu_out, R, H, eps, args) -> dict:
    """The oracle, as it stands (single-threaded C), on the first rows of the same batch until
    about `cpu_seconds` of work is done; its outputs are also compared with the GPU's."""
    import torch

    import oracle
    from tests.helpers import bits_equal, ulp_dist, within_tol

    S = host_in["x"].shape[0]
    chunk = 256
    done, t_plain, t_fused = 0, 0.0, 0.0
    max_ulp, res_ok, tol_ok = 0, True, True
    while done < S:
        sl = slice(done, min(S, done + chunk))
        t0 = time.perf_counter()
        y_ref, _ = oracle.rms_norm(host_in["x"][sl], host_in["w"], eps)
        t1 = time.perf_counter()
        x_ref, r_ref, _ = oracle.fused_add_rms_norm(host_in["xf"][sl], host_in["r"][sl],
                                                    host_in["w"], eps)
        t2 = time.perf_counter()
        t_plain += t1 - t0
        t_fused += t2 - t1
        res_ok &= bits_equal(gpu_out["r"][sl], r_ref)
        for out, ref in ((gpu_out["y"][sl], y_ref), (gpu_out["x"][sl], x_ref)):
            max_ulp = max(max_ulp, int(ulp_dist(out, ref).max()))
            tol_ok &= within_tol(out, ref, 1e-2, 1e-3)[0]
        done = sl.stop
        if t_plain + t_fused >= args.cpu_seconds:
            break
    nb = algorithmic_bytes("rms_norm", done, H, 2) + algorithmic_bytes("fused_add_rms_norm", done, H, 2)
    secs = t_plain + t_fused
    return {
        "baseline": {"value": nb / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                     "sample": f"first {done} of {R} rows of both ops ([{done},{H}] bf16), "
                               f"{secs:.1f} s single-threaded",
                     "host_cores_total": os.cpu_count(), "host_cpu": host_cpu_model(),
                     "all_cores": oracle_all_cores(host_in, done, H, eps)},
        "parity": {"rows_checked": done, "max_ulp": max_ulp, "residual_bit_exact": res_ok,
                   "within_tolerance": tol_ok, "ok": bool(res_ok and tol_ok and max_ulp <= 1)},
    }


# ------------------------------------------------------------------------ reference arm

def run_reference(args) -> int:
    """The oracle (the plain CPU definition) timed on the host cores on bounded samples of the
    same workload. Rank 0 only; other ranks exit without work."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import torch

    import oracle
    from row_wise_rmsnorm_ks_gb300 import synth

    R, H, eps = args.rows, args.hidden, 1e-5
    budget = args.reference_seconds
    # calibrate one row of each op, then size each step's sample to fit the budget
    x1 = synth.cast(synth.normal_np((1, H), synth.SEED_X), "bf16")
    w = synth.weight(H, "bf16")
    t0 = time.perf_counter()
    oracle.rms_norm(x1, w, eps)
    oracle.fused_add_rms_norm(x1, x1.clone(), w, eps)
    per_row = time.perf_counter() - t0
    rows = max(1, min(R, int(budget / (args.steps + args.warmup) / per_row)))
    x = synth.cast(synth.normal_np((rows, H), synth.SEED_X), "bf16")
    r = synth.cast(synth.normal_np((rows, H), synth.SEED_RESIDUAL), "bf16")

    def step():
        oracle.rms_norm(x, w, eps)
        oracle.fused_add_rms_norm(x, r, w, eps)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = time.perf_counter() - t0
    nb = algorithmic_bytes("rms_norm", rows, H, 2) + algorithmic_bytes("fused_add_rms_norm", rows, H, 2)
    value = nb * args.steps / secs / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), host draw)",
        "config": {"workload": workload(R, H), "rows": R, "hidden": H, "eps": eps},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows} of {R} rows of both ops per step",
                         "host_cores_total": os.cpu_count(), "host_cpu": host_cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


def run_sweep(args) -> int:
    """The configuration sweeps (one JSON line per case; not the contract's line): the large bf16
    shape's rows 1024..32768 at H = 8192, and the odd/wide sweep H in {1536, 5120, 7168, 14336,
    16384} x rows in {1, 7, 333, 65536} x {fp16, bf16}, both ops, on the sweep's own inputs
    (N(0,1) rows for the first, heavy-tailed Student-t rows with 1% scaled by 1e3 for the second).
    Each case: the median of single launches timed with CUDA events, the L2 emptied before each
    (outside the timed pair) by reading a 512 MiB buffer, so no dirty line of another tensor is
    left to write back; algorithmic GB/s and the fraction of the measured copy peak. Cases of at
    most 333 rows also report the per-launch time of 20 back-to-back launches replayed from a
    CUDA graph (inputs hot in L2), the launch-bound figure for decode-sized batches."""
    import torch

    from row_wise_rmsnorm_ks_gb300 import _abi, synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    side = torch.cuda.Stream(dev)
    flush = torch.ones(128 << 20, dtype=torch.float32, device=dev)
    peak = measured_peaks()["hbm_gbs"]
    sms = device_facts(dev)["sm_count"]
    codes = {"bf16": _abi.KS_DTYPE_BF16, "fp16": _abi.KS_DTYPE_F16}

    def median_us(fn, n):
        s = torch.cuda.current_stream(dev)
        fn(s.cuda_stream)
        out = []
        for _ in range(n):
            flush.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn(s.cuda_stream)
            b.record(s)
            b.synchronize()
            out.append(a.elapsed_time(b) * 1e3)
        return statistics.median(out)

    def graph_us(fn, launches=20, replays=20):
        with torch.cuda.stream(side):
            fn(side.cuda_stream)
            side.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _ in range(launches):
                    fn(torch.cuda.current_stream(dev).cuda_stream)
            g.replay()
            side.synchronize()
            out = []
            for _ in range(replays):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(side)
                g.replay()
                b.record(side)
                b.synchronize()
                out.append(a.elapsed_time(b) * 1e3 / launches)
        return statistics.median(out)

    def case(tag, dt, R, H, op, x, r, w, eps):
        code = codes[dt]
        if op == "rms_norm":
            y = torch.empty_like(x)
            fn = lambda st: _abi.check(_abi.ks_rms_norm(y.data_ptr(), x.data_ptr(), w.data_ptr(),
                                                        R, H, eps, code, st))
        else:
            fn = lambda st: _abi.check(_abi.ks_fused_add_rms_norm(x.data_ptr(), r.data_ptr(),
                                                                  w.data_ptr(), R, H, eps, code, st))
        us = median_us(fn, args.sweep_samples)
        nb = algorithmic_bytes(op, R, H, 2)
        plan = _abi.ks_plan_launch(0 if op == "rms_norm" else 1, R, H, code, True, sms, 0)[1]
        line = {"sweep": tag, "op": op, "dtype": dt, "rows": R, "hidden": H, "p50_us": us,
                "gbs": nb / (us * 1e-6) / 1e9, "frac_of_peak": nb / (us * 1e-6) / 1e9 / peak,
                "kernel": plan.as_dict()["kernel_name"], "vec_per_thread": plan.vec_per_thread,
                "prefetch": not plan.flags & _abi.KS_PLAN_NO_PREFETCH}
        if R <= 333:
            line["graph_us"] = graph_us(fn)
        print(json.dumps(line), flush=True)

    for R in (1024, 2048, 4096, 8192, 16384, 32768):
        x = synth.cast(synth.normal_dev((R, 8192), synth.SEED_X, dev), "bf16")
        r = synth.cast(synth.normal_dev((R, 8192), synth.SEED_RESIDUAL, dev), "bf16")
        w = synth.weight(8192, "bf16").to(dev)
        for op in ("rms_norm", "fused_add_rms_norm"):
            case("prefill rows", "bf16", R, 8192, op, x, r, w, 1e-5)
        del x, r
    for dt in ("bf16", "fp16"):
        for H in (1536, 5120, 7168, 14336, 16384):
            for R in (1, 7, 333, 65536):
                for op in ("rms_norm", "fused_add_rms_norm"):
                    wl = synth.wide_device(op, H, R, dt, dev)
                    case("wide", dt, R, H, op, wl.x, wl.residual, wl.weight, wl.eps)
                    del wl
    torch.cuda.empty_cache()
    return 0


def ncu_launch_list(csv_path: str, kernel_prefix: str = "rows_"):
    """(kernel name, gpu__time_duration in microseconds) of each launch in an ncu --csv launch
    list, in launch order, for kernels whose name contains `kernel_prefix`."""
    out = []
    with open(csv_path, newline="") as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(io.StringIO("".join(lines))):
        if row.get("Metric Name") != "gpu__time_duration.sum":
            continue
        name = row.get("Kernel Name", "")
        if kernel_prefix not in name:
            continue
        v = float(row["Metric Value"].replace(",", ""))
        unit = row.get("Metric Unit", "ns")
        out.append((name, v / 1e3 if unit == "ns" else v if unit == "us" else v * 1e3))
    return out


def kernel_times_table(jsonl_path: str, csv_path: str) -> str:
    """A markdown table joining the kernel-times mode's JSON lines with the ncu launch list of the
    same command: per case the median kernel time of its timed launches (ncu; caches flushed
    before each, clocks not locked), the event p50 of the same launches, and the fraction of the
    measured copy peak each implies."""
    peak = measured_peaks()["hbm_gbs"]
    cases = [json.loads(ln) for ln in open(jsonl_path) if ln.startswith('{"kernel_times"')]
    launches = ncu_launch_list(csv_path)
    need = sum(c["launches"] for c in cases)
    if len(launches) != need:
        raise SystemExit(f"the launch list has {len(launches)} launches of this library, the cases "
                         f"made {need}: not the same command")
    rows, i = [], 0
    for c in cases:
        mine = launches[i:i + c["launches"]]
        i += c["launches"]
        k_us = statistics.median(us for _, us in mine[1:])
        p = c["plan"]
        kern = p["kernel_name"] + (f" c{p['cluster']}" if p.get("cluster", 0) >= 2 else "")
        rows.append(f"| {c['kernel_times']} | {c['dtype']} | {c['op']} | [{c['rows']}, {c['hidden']}] "
                    f"| {kern} | {k_us:.2f} | {c['event_p50_us']:.2f} | "
                    f"{c['bytes'] / (k_us * 1e-6) / 1e9 / peak:.3f} | {c['event_frac_of_peak']:.3f} |")
    head = ("| case | dtype | op | [rows, H] | kernel | kernel µs (ncu) | event p50 µs | "
            "of peak by kernel time | of peak by event |\n|---|---|---|---|---|---|---|---|---|")
    return head + "\n" + "\n".join(rows)


KERNEL_TIME_WIDE_H = (1536, 5120, 7168, 14336, 16384)


def kernel_time_cases():
    """The shapes the kernel-times mode runs, in its launch order: (tag, dtype, op, rows, hidden,
    eps). The stated configurations (small [128, 1024]; medium [2048, 4096] fp16 and bf16; fused
    [512, 4096] and decode [4, 1536]; prefill bf16 rows 1024..32768 at 8192; wide fp16/bf16
    H x rows {1, 7, 333, 65536}), both ops where the configuration has both."""
    out = [("small", "bf16", "rms_norm", 128, 1024, 1e-6)]
    out += [("medium", dt, "rms_norm", 2048, 4096, 1e-6) for dt in ("fp16", "bf16")]
    out += [("fused", "bf16", "fused_add_rms_norm", 512, 4096, 1e-6),
            ("decode", "bf16", "fused_add_rms_norm", 4, 1536, 1e-6)]
    out += [("prefill", "bf16", op, R, 8192, 1e-5) for R in (1024, 2048, 4096, 8192, 16384, 32768)
            for op in ("rms_norm", "fused_add_rms_norm")]
    out += [("wide", dt, op, R, H, 1e-6) for dt in ("bf16", "fp16") for H in KERNEL_TIME_WIDE_H
            for R in (1, 7, 333, 65536) for op in ("rms_norm", "fused_add_rms_norm")]
    return out


def run_kernel_times(args) -> int:
    """Every stated configuration, launched a fixed number of times in a fixed order, so that a
    launch list taken by ncu over the same command (gpu__time_duration.sum, one pass) maps onto
    the cases: per case one untimed launch, then --kernel-time-launches single launches, each
    after the L2 is emptied (a 512 MiB read, outside the timed pair) and timed with CUDA events.
    One JSON line per case (not the contract's line) with the event p50 and the number of this
    library's launches it made, in order."""
    import torch

    from row_wise_rmsnorm_ks_gb300 import _abi, synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.ones(128 << 20, dtype=torch.float32, device=dev)
    peak = measured_peaks()["hbm_gbs"]
    sms = device_facts(dev)["sm_count"]
    codes = {"bf16": _abi.KS_DTYPE_BF16, "fp16": _abi.KS_DTYPE_F16}
    n = args.kernel_time_launches
    for tag, dt, op, R, H, eps in kernel_time_cases():
        if tag == "wide":
            wl = synth.wide_device(op, H, R, dt, dev)
            x, r, w = wl.x, wl.residual, wl.weight
        else:
            x = synth.cast(synth.normal_dev((R, H), synth.SEED_X, dev), dt)
            r = synth.cast(synth.normal_dev((R, H), synth.SEED_RESIDUAL, dev, std=2.0), dt)
            w = synth.weight(H, dt).to(dev)
        code = codes[dt]
        st = torch.cuda.current_stream(dev)
        if op == "rms_norm":
            y = torch.empty_like(x)
            fn = lambda: _abi.check(_abi.ks_rms_norm(y.data_ptr(), x.data_ptr(), w.data_ptr(), R,
                                                     H, eps, code, st.cuda_stream))
        else:
            fn = lambda: _abi.check(_abi.ks_fused_add_rms_norm(x.data_ptr(), r.data_ptr(),
                                                               w.data_ptr(), R, H, eps, code,
                                                               st.cuda_stream))
        fn()
        us = []
        for _ in range(n):
            flush.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            fn()
            b.record(st)
            b.synchronize()
            us.append(a.elapsed_time(b) * 1e3)
        nb = algorithmic_bytes(op, R, H, 2)
        plan = _abi.ks_plan_launch(0 if op == "rms_norm" else 1, R, H, code, True, sms, 0)[1]
        p50 = statistics.median(us)
        print(json.dumps({"kernel_times": tag, "dtype": dt, "op": op, "rows": R, "hidden": H,
                          "launches": n + 1, "event_p50_us": p50,
                          "event_frac_of_peak": nb / (p50 * 1e-6) / 1e9 / peak,
                          "bytes": nb, "plan": plan.as_dict()}), flush=True)
        del x, r, w
        if tag == "wide":
            del wl
        torch.cuda.empty_cache()
    return 0


def plan_candidates(op: str, hv: int, elem: int):
    """Every launch plan the heuristic chooses among for a row of hv 16-byte vectors, named as in
    the plan-sweep tables: w1/w1n, w2/w2n, w4/w4n (warp per row, 1, 2 or 4 vectors per lane for
    rows of at most 32, 64 or 128 vectors, with/without prefetch; t8vV/t8vVn and t16vV/t16vVn:
    8- or 16-lane teams, several rows per warp, at the fewest of 1, 2 or 4 vectors per lane that
    cover rows of at most 32 or 64 vectors;
    w6/w6n and w8/w8n: 6 or 8 vectors per lane for rows of 129..192 and 193..256 vectors),
    p2/n2/p4/n4 (CTA per row, 2 or 4 vectors per thread, with/without prefetch), b2 (staged ring,
    2 stages), tBuU (the two-pass kernel, B threads, U vectors per thread per step; rows of at
    least 512 vectors), sCbBuU (the two-pass kernel split over a cluster of C CTAs; rows of at
    least 1024 vectors), both also with a trailing n (no L2 prefetch of the row), sCbBuUp (the
    split kernel with two rows in flight per cluster, no prefetch), and for
    rows wider than 2048 vectors cC (register-resident cluster of C CTAs, 4 vectors per thread)
    and bCsS / bCsSv8 (the staged kernel split over C CTAs, S stages, 4 or 8 vectors per
    thread; bCsS[v8]m, the plain op: the rows kept in shared memory, two in flight, C up to
    16)."""
    from row_wise_rmsnorm_ks_gb300 import _abi

    up32 = lambda n: -(-n // 32) * 32
    fused = op == "fused_add_rms_norm"
    out = []
    for v in (1, 2, 4):  # a warp per row, 8 rows per 256-thread CTA
        if hv <= 32 * v:
            out += [(f"w{v}", _abi.make_plan(_abi.KS_KERNEL_WARP_ROW, v, 256)),
                    (f"w{v}n", _abi.make_plan(_abi.KS_KERNEL_WARP_ROW, v, 256,
                                              flags=_abi.KS_PLAN_NO_PREFETCH))]
    for team in (8, 16):  # sub-warp teams at the fewest vectors per lane that cover the row
        v = next((v for v in (1, 2, 4) if team * v >= hv), None)
        if v:
            out += [(f"t{team}v{v}", _abi.make_plan(_abi.KS_KERNEL_WARP_ROW, v, 256, team=team)),
                    (f"t{team}v{v}n", _abi.make_plan(_abi.KS_KERNEL_WARP_ROW, v, 256, team=team,
                                                     flags=_abi.KS_PLAN_NO_PREFETCH))]
    for v in (6, 8):  # a warp covers rows of up to 32 * v vectors; 4 rows per 128-thread CTA
        if 32 * (v - 2) < hv <= 32 * v:
            out += [(f"w{v}", _abi.make_plan(_abi.KS_KERNEL_WARP_ROW, v, 128)),
                    (f"w{v}n", _abi.make_plan(_abi.KS_KERNEL_WARP_ROW, v, 128,
                                              flags=_abi.KS_PLAN_NO_PREFETCH))]
    for v in (2, 4):
        b = up32(-(-hv // v))
        if b <= (1024 if v == 2 else 512):
            out += [(f"p{v}", _abi.make_plan(_abi.KS_KERNEL_CTA_ROW, v, b)),
                    (f"n{v}", _abi.make_plan(_abi.KS_KERNEL_CTA_ROW, v, b,
                                             flags=_abi.KS_PLAN_NO_PREFETCH))]
    b = up32(-(-hv // 4))
    if b <= 512 and 128 + 2 * hv * 16 * (2 if fused else 1) <= 226 * 1024:
        out.append(("b2", _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, b, 2)))
    npf = _abi.KS_PLAN_NO_PREFETCH
    if hv >= 512:
        for blk, u in ((256, 4), (512, 2), (512, 4), (1024, 2), (1024, 4)):
            out.append((f"t{blk}u{u}", _abi.make_plan(_abi.KS_KERNEL_TWOPASS_ROW, u, blk)))
            out.append((f"t{blk}u{u}n", _abi.make_plan(_abi.KS_KERNEL_TWOPASS_ROW, u, blk,
                                                       flags=npf)))
    if hv >= 1024:
        for c in (2, 4, 8):
            for blk, u in ((256, 4), (512, 2), (512, 4), (1024, 2)):
                if blk * u * (c - 1) < hv:  # at least one step of work per CTA slice
                    out.append((f"s{c}b{blk}u{u}", _abi.make_plan(_abi.KS_KERNEL_TWOPASS_ROW, u,
                                                                  blk, cluster=c)))
                    out.append((f"s{c}b{blk}u{u}n", _abi.make_plan(
                        _abi.KS_KERNEL_TWOPASS_ROW, u, blk, cluster=c, flags=npf)))
                    out.append((f"s{c}b{blk}u{u}p", _abi.make_plan(
                        _abi.KS_KERNEL_TWOPASS_ROW, u, blk, 2, cluster=c, flags=npf)))
    if hv > 2048:
        for c in (2, 4, 8, 16):
            sl = -(-hv // c)
            b = up32(-(-sl // 4))
            if b <= 512 and c <= 8:
                out.append((f"c{c}", _abi.make_plan(_abi.KS_KERNEL_CLUSTER_ROW, 4, b, cluster=c)))
            for vv in ((4,) if fused else (4, 8)):
                b = up32(-(-sl // vv))
                # the shared-memory rows kernel takes up to 1024 threads at 4 vectors
                if b > (1024 if vv == 4 and not fused else 512):
                    continue
                for st in ((2, 3, 4) if c <= 8 and b <= 512 else ()):
                    if 128 + st * sl * 16 * (2 if fused else 1) <= 226 * 1024:
                        out.append((f"b{c}s{st}" + ("v8" if vv == 8 else ""), _abi.make_plan(
                            _abi.KS_KERNEL_BULK_ROW, vv, b, st, cluster=c)))
                for st in (() if fused else (2, 3, 4, 6)):  # rows kept in shared memory
                    if 128 + st * sl * 16 <= 226 * 1024:
                        out.append((f"b{c}s{st}" + ("v8" if vv == 8 else "") + "m", _abi.make_plan(
                            _abi.KS_KERNEL_BULK_ROW, vv, b, st, cluster=c,
                            flags=_abi.KS_PLAN_SMEM_ROWS)))
    return out


def run_plan_sweep(args) -> int:
    """The sweep behind the launch heuristic (one JSON line per dtype, op and width; not the
    contract's line): for rows of hv = 128..2048 16-byte vectors in steps of 64, and 2560, 3072,
    4096, 8192, 16384, every candidate plan of plan_candidates() and the default, at an HBM-bound
    row count (384 MiB per tensor), N(0,1) inputs, back-to-back launches timed with CUDA events;
    the candidates are interleaved over --plan-sweep-rounds rounds and the median kept, as a
    fraction of the measured copy peak."""
    import torch

    from row_wise_rmsnorm_ks_gb300 import _abi, synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    peak = measured_peaks()["hbm_gbs"]
    sms = device_facts(dev)["sm_count"]
    codes = {"bf16": _abi.KS_DTYPE_BF16, "fp16": _abi.KS_DTYPE_F16, "fp32": _abi.KS_DTYPE_F32}

    def timeit(fn, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n * 1e-3

    widths = list(range(128, 2049, 64)) + [2560, 3072, 4096, 8192, 16384, 32768]
    if args.plan_sweep_widths:
        widths = [int(v) for v in args.plan_sweep_widths.split(",")]
    for dt in args.plan_sweep_dtypes.split(","):
        elem = 4 if dt == "fp32" else 2
        code = codes[dt]
        for hv in widths:
            H = hv * 16 // elem
            R = max(64, (384 << 20) // (H * elem))
            x = synth.cast(synth.normal_dev((R, H), synth.SEED_X, dev), dt)
            r = synth.cast(synth.normal_dev((R, H), synth.SEED_RESIDUAL, dev), dt)
            y = torch.empty_like(x)
            w = synth.weight(H, dt).to(dev)
            for op in args.plan_sweep_ops.split(","):
                nb = algorithmic_bytes(op, R, H, elem)
                fns = []
                for name, p in [("default", None)] + plan_candidates(op, hv, elem):
                    if op == "rms_norm":
                        fn = ((lambda p=p: _abi.ks_rms_norm_planned(
                            y.data_ptr(), x.data_ptr(), w.data_ptr(), R, H, 1e-5, code, p, s))
                            if p else (lambda: _abi.ks_rms_norm(
                                y.data_ptr(), x.data_ptr(), w.data_ptr(), R, H, 1e-5, code, s)))
                    else:
                        fn = ((lambda p=p: _abi.ks_fused_add_rms_norm_planned(
                            x.data_ptr(), r.data_ptr(), w.data_ptr(), R, H, 1e-5, code, p, s))
                            if p else (lambda: _abi.ks_fused_add_rms_norm(
                                x.data_ptr(), r.data_ptr(), w.data_ptr(), R, H, 1e-5, code, s)))
                    if fn() == _abi.KS_SUCCESS:  # a plan that does not fit is left out
                        fns.append((name, fn))
                n = max(10, min(60, int(1.5e-2 / (nb / 6e12))))
                res = {name: [] for name, _ in fns}
                for _ in range(args.plan_sweep_rounds):
                    for name, fn in fns:
                        res[name].append(nb / timeit(fn, n) / 1e9 / peak)
                dp = _abi.ks_plan_launch(0 if op == "rms_norm" else 1, R, H, code, True, sms,
                                         0)[1].as_dict()
                line = {"plan_sweep": dt, "op": op, "hv": hv, "hidden": H, "rows": R,
                        "default_plan": {k: dp[k] for k in ("kernel_name", "vec_per_thread",
                                                            "block", "flags", "stages",
                                                            "cluster")}}
                line.update({k: round(statistics.median(v), 4) for k, v in res.items()})
                print(json.dumps(line), flush=True)
            del x, r, y
            torch.cuda.empty_cache()
    st, flags = _abi.ks_device_faults(clear=True)
    if st != _abi.KS_SUCCESS or flags:
        print(json.dumps({"plan_sweep": "device faults", "status": st, "flags": flags}))
        return 1
    return 0


def run_plan_probe(args) -> int:
    """One plan-sweep candidate (--plan-probe NAME, named as in plan_candidates) launched
    --probe-launches times through the planned entry point on --rows x --hidden (--probe-dtype,
    --probe-op), N(0,1) inputs, then one JSON line with the mean event time per launch (not the
    contract's line). A fixed small workload for a profiler to capture one kernel of."""
    import torch

    from row_wise_rmsnorm_ks_gb300 import _abi, synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    dt, op, R, H = args.probe_dtype, args.probe_op, args.rows, args.hidden
    elem = 4 if dt == "fp32" else 2
    code = {"bf16": _abi.KS_DTYPE_BF16, "fp16": _abi.KS_DTYPE_F16, "fp32": _abi.KS_DTYPE_F32}[dt]
    plans = dict(plan_candidates(op, H * elem // 16, elem))
    if args.plan_probe not in plans:
        print(json.dumps({"plan_probe": args.plan_probe, "error": "no such candidate at this width",
                          "candidates": sorted(plans)}))
        return 2
    p = plans[args.plan_probe]
    x = synth.cast(synth.normal_dev((R, H), synth.SEED_X, dev), dt)
    w = synth.weight(H, dt).to(dev)
    y = torch.empty_like(x)
    r = synth.cast(synth.normal_dev((R, H), synth.SEED_RESIDUAL, dev), dt) if op != "rms_norm" else None
    def launch():
        if op == "rms_norm":
            return _abi.ks_rms_norm_planned(y.data_ptr(), x.data_ptr(), w.data_ptr(), R, H, 1e-5,
                                            code, p, s)
        return _abi.ks_fused_add_rms_norm_planned(x.data_ptr(), r.data_ptr(), w.data_ptr(), R, H,
                                                  1e-5, code, p, s)
    _abi.check(launch())  # untimed: the first launch sets the kernel's attributes up
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.probe_launches):
        _abi.check(launch())
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / args.probe_launches
    st, flags = _abi.ks_device_faults(clear=False)
    nb = algorithmic_bytes(op, R, H, elem)
    print(json.dumps({"plan_probe": args.plan_probe, "op": op, "dtype": dt, "rows": R, "hidden": H,
                      "plan": p.as_dict(), "us_per_launch": us,
                      "frac_of_peak": nb / (us * 1e-6) / 1e9 / measured_peaks()["hbm_gbs"],
                      "faults": [st, flags]}))
    return 0 if (st == _abi.KS_SUCCESS and flags == 0) else 1


def run_plan_contexts(args) -> int:
    """The register-kernel candidates (warp and CTA rows, 2 or 4 vectors, with and without
    prefetch; plus the two-pass kernel and the staged ring where they apply) against the default
    plan, per dtype, op and width, in two contexts (one JSON line each; not the contract's line):
    steady (the same plan launched back to back, after 5 untimed launches) and right after one
    launch of the staged ring, a kernel with a large shared-memory carveout, as after a GEMM in a
    model (each launch timed alone). 384 MiB per tensor, N(0,1) inputs; the plans alternate over
    --plan-sweep-rounds rounds and the median is kept, as a fraction of the measured copy peak.
    The plan-sweep mode instead interleaves every candidate, so each block of launches follows a
    different kernel."""
    import torch

    from row_wise_rmsnorm_ks_gb300 import _abi, synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    peak = measured_peaks()["hbm_gbs"]
    sms = device_facts(dev)["sm_count"]
    codes = {"bf16": _abi.KS_DTYPE_BF16, "fp16": _abi.KS_DTYPE_F16, "fp32": _abi.KS_DTYPE_F32}
    keep = ("w1", "w1n", "w2", "w2n", "w4", "w4n", "w6", "w6n", "t8v1", "t8v1n", "t8v2", "t8v2n",
            "t8v4", "t8v4n", "t16v1", "t16v1n", "t16v2", "t16v2n", "t16v4", "t16v4n", "w8", "w8n", "p2", "n2", "p4", "n4", "t256u4", "t512u2",
            "t256u4n", "t512u2n", "b2")

    def steady(fn, n=30):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(5):
            fn()
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n * 1e-3

    def after(fn, pre, n=12):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tot = 0.0
        for _ in range(n):
            pre()
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b) * 1e-3
        return tot / n

    widths = [int(v) for v in (args.plan_sweep_widths or "128,256,512,640,768,1024,1280,1536,2048").split(",")]
    for dt in args.plan_sweep_dtypes.split(","):
        elem = 4 if dt == "fp32" else 2
        code = codes[dt]
        for hv in widths:
            H = hv * 16 // elem
            R = (384 << 20) // (H * elem)
            x = synth.cast(synth.normal_dev((R, H), synth.SEED_X, dev), dt)
            r = synth.cast(synth.normal_dev((R, H), synth.SEED_RESIDUAL, dev), dt)
            w = synth.weight(H, dt).to(dev)
            y = torch.empty_like(x)
            ring = _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, -(-(-(-hv // 4)) // 32) * 32, 2)
            pre = (lambda: _abi.check(_abi.ks_rms_norm_planned(
                y.data_ptr(), x.data_ptr(), w.data_ptr(), R, H, 1e-5, code, ring, s)))
            if 128 + 2 * hv * 16 > 226 * 1024:
                pre = None  # no ring of two stages fits: steady context only
            for op in ("rms_norm", "fused_add_rms_norm"):
                fused = op == "fused_add_rms_norm"
                nb = algorithmic_bytes(op, R, H, elem)

                def mk(p):
                    if fused:
                        return lambda: _abi.check(_abi.ks_fused_add_rms_norm_planned(
                            x.data_ptr(), r.data_ptr(), w.data_ptr(), R, H, 1e-5, code, p, s))
                    return lambda: _abi.check(_abi.ks_rms_norm_planned(
                        y.data_ptr(), x.data_ptr(), w.data_ptr(), R, H, 1e-5, code, p, s))
                def default():
                    if fused:
                        _abi.check(_abi.ks_fused_add_rms_norm(x.data_ptr(), r.data_ptr(),
                                                              w.data_ptr(), R, H, 1e-5, code, s))
                    else:
                        _abi.check(_abi.ks_rms_norm(y.data_ptr(), x.data_ptr(), w.data_ptr(), R, H,
                                                    1e-5, code, s))
                _, dp = _abi.ks_plan_launch(int(fused), R, H, code, True, sms, 0)
                fns = [("default", default)] + [(n, mk(p)) for n, p in plan_candidates(op, hv, elem)
                                                if n in keep]
                line = {"plan_contexts": dt, "op": op, "hv": hv, "hidden": H, "rows": R,
                        "default_plan": {k: dp.as_dict()[k] for k in ("kernel_name", "vec_per_thread",
                                                                       "block", "flags")}}
                for ctx in ("steady", "after_ring") if pre else ("steady",):
                    res = {name: [] for name, _ in fns}
                    for _ in range(args.plan_sweep_rounds):
                        for name, fn in fns:
                            t = steady(fn) if ctx == "steady" else after(fn, pre)
                            res[name].append(nb / t / 1e9 / peak)
                    line[ctx] = {k: round(statistics.median(v), 4) for k, v in res.items()}
                print(json.dumps(line), flush=True)
            del x, r, w, y
            torch.cuda.empty_cache()
    st, flags = _abi.ks_device_faults(clear=False)
    if st != _abi.KS_SUCCESS or flags:
        print(json.dumps({"plan_contexts": "device faults", "status": st, "flags": flags}))
        return 1
    return 0


OPS_BAND_WIDTHS = {
    # rows of 16-byte vectors at the edges of the Softmax and LayerNorm width bands
    "softmax": (16, 32, 33, 44, 45, 52, 53, 63, 64, 65, 72, 80, 81, 96, 127, 128, 129, 168, 169,
                176, 177, 192, 193, 216, 217, 224, 225, 256),
    "layer_norm": (16, 32, 33, 63, 64, 65, 96, 127, 128, 129, 160, 192, 193, 224, 225, 256),
    # the SwiGLU output row's vectors at the edges of its launch shapes
    "silu_and_mul": (32, 64, 128, 159, 160, 161, 192, 193, 256, 287, 288, 447, 448, 512, 1024,
                     2048),
}


def op_band_candidates(op: str, hv: int):
    """The launch plans the next operators' width bands choose among for a row of hv vectors:
    tTvV / tTvVn (a team of T = 8 or 16 lanes per row, V vectors a lane, with / without
    prefetch; where the team covers the row), wV / wVn (a warp per row), cV / cVn (a CTA per
    row, V vectors a thread), for rows wider than 256 vectors xB (the wide multi-pass kernel on
    B threads) and for LayerNorm rS / rSa (the staged ring of S rows per CTA, with the weight and
    bias rows in registers / in shared memory), and for SwiGLU flatB
    (the flat walk on B-thread CTAs) and rowsB (the row kernel with at most B threads)."""
    from row_wise_rmsnorm_ks_gb300 import _abi

    up32 = lambda n: -(-n // 32) * 32
    mk = _abi.make_plan
    npf = _abi.KS_PLAN_NO_PREFETCH
    out = []
    if op == "silu_and_mul":
        out += [("flat256", mk(_abi.KS_KERNEL_FLAT, 2, 256)),
                ("flat128", mk(_abi.KS_KERNEL_FLAT, 2, 128))]
        out += [(f"rows{b}", mk(_abi.KS_KERNEL_CTA_ROW, 2, b)) for b in (96, 128, 256)]
        return out
    for team in (8, 16):  # teams of 8 or 16 lanes: 4 or 2 rows per warp
        for v in (2, 4):
            if team * v >= hv and team * (v - 2) < hv:
                out.append((f"t{team}v{v}", mk(_abi.KS_KERNEL_WARP_ROW, v, 128, team=team)))
                if op == "softmax":
                    out.append((f"t{team}v{v}n", mk(_abi.KS_KERNEL_WARP_ROW, v, 128, flags=npf,
                                                    team=team)))
    for v in (2, 4, 6, 8):
        if 32 * v >= hv:
            out.append((f"w{v}", mk(_abi.KS_KERNEL_WARP_ROW, v, 128)))
            if op == "softmax":
                out.append((f"w{v}n", mk(_abi.KS_KERNEL_WARP_ROW, v, 128, flags=npf)))
    for v in (1, 2, 4):
        b = up32(-(-hv // v))
        if b <= 512:
            out.append((f"c{v}", mk(_abi.KS_KERNEL_CTA_ROW, v, b)))
            if op == "softmax" and v == 4:
                out.append(("c4n", mk(_abi.KS_KERNEL_CTA_ROW, 4, b, flags=npf)))
    if hv > 256:
        # the wide multi-pass kernel at B threads (xB), and for LayerNorm the staged ring of S
        # rows per CTA (rS) where its CTA covers the row and the ring fits
        for blk in (128, 256, 512):
            out.append((f"x{blk}", mk(_abi.KS_KERNEL_TWOPASS_ROW, 4, blk)))
        b = up32(-(-hv // 4))
        if op == "layer_norm" and b <= 1024:
            for st in (2, 3, 4, 6, 8):
                if 128 + st * hv * 16 <= 226 * 1024 and b <= 512:
                    out.append((f"r{st}", mk(_abi.KS_KERNEL_BULK_ROW, 4, b, st)))
                # rSa: the weight and bias rows in shared memory beside the ring (up to 1024
                # threads)
                if 128 + (st + 2) * hv * 16 <= 226 * 1024:
                    out.append((f"r{st}a", mk(_abi.KS_KERNEL_BULK_ROW, 4, b, st,
                                               flags=_abi.KS_PLAN_AFFINE_SMEM)))
    return out


def run_ops_bands(args) -> int:
    """The measurement behind the next operators' width bands (one JSON line per operator, dtype
    and width; not the contract's line): every candidate of op_band_candidates() and the default
    launch, through the *_planned entry points, in two contexts: steady (the same plan launched
    back to back after 5 untimed launches) and right after one launch of a kernel that leaves a
    large shared-memory carveout, as a GEMM would (the RMSNorm staged ring with 196 KiB of shared
    memory; each launch timed alone). 384 MiB per input tensor, N(0,1) rows (SwiGLU gates N(0,4));
    the plans alternate over --plan-sweep-rounds rounds and the median is kept, as a fraction of
    the measured copy peak. A band takes the plan whose worse context scores best
    (--ops-bands-table)."""
    import torch

    from row_wise_rmsnorm_ks_gb300 import _abi, synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    st = torch.cuda.current_stream(dev)
    s = st.cuda_stream
    peak = measured_peaks()["hbm_gbs"]
    sms = device_facts(dev)["sm_count"]
    codes = {"bf16": _abi.KS_DTYPE_BF16, "fp16": _abi.KS_DTYPE_F16, "fp32": _abi.KS_DTYPE_F32}
    op_codes = {"silu_and_mul": _abi.OP_SILU_AND_MUL, "softmax": _abi.OP_SOFTMAX,
                "layer_norm": _abi.OP_LAYER_NORM}
    # the carveout kernel: RMSNorm through the staged ring, 6 stages of 2048 bf16 vectors
    xa = synth.cast(synth.normal_dev((256, 16384), 1, dev), "bf16")
    ya, wa = torch.empty_like(xa), synth.weight(16384, "bf16").to(dev)
    ring = _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 512, 6)
    pre = lambda: _abi.check(_abi.ks_rms_norm_planned(ya.data_ptr(), xa.data_ptr(), wa.data_ptr(),
                                                      256, 16384, 1e-5, _abi.KS_DTYPE_BF16, ring, s))

    def steady(fn, n=30):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(5):
            fn()
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n * 1e-3

    def after(fn, n=12):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tot = 0.0
        for _ in range(n):
            pre()
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b) * 1e-3
        return tot / n

    ops = args.ops_bands_ops.split(",")
    for op in ops:
        widths = ([int(v) for v in args.plan_sweep_widths.split(",")] if args.plan_sweep_widths
                  else OPS_BAND_WIDTHS[op])
        for dt in args.plan_sweep_dtypes.split(","):
            elem = 4 if dt == "fp32" else 2
            code = codes[dt]
            for hv in widths:
                H = hv * 16 // elem
                if op == "silu_and_mul":
                    R = (384 << 20) // (2 * H * elem)
                    x = synth.cast(synth.normal_dev((R, 2 * H), synth.SEED_X, dev, std=2.0), dt)
                    y = torch.empty((R, H), dtype=x.dtype, device=dev)
                    nb = 3 * R * H * elem
                    run = lambda p: _abi.ks_silu_and_mul_planned(y.data_ptr(), x.data_ptr(), R, H,
                                                                 code, p, s)
                    default = lambda: _abi.check(_abi.ks_silu_and_mul(y.data_ptr(), x.data_ptr(),
                                                                      R, H, code, s))
                else:
                    R = (384 << 20) // (H * elem)
                    x = synth.cast(synth.normal_dev((R, H), synth.SEED_X, dev), dt)
                    y = torch.empty_like(x)
                    if op == "softmax":
                        nb = 2 * R * H * elem
                        run = lambda p: _abi.ks_softmax_planned(y.data_ptr(), x.data_ptr(), R, H,
                                                                code, p, s)
                        default = lambda: _abi.check(_abi.ks_softmax(y.data_ptr(), x.data_ptr(),
                                                                     R, H, code, s))
                    else:
                        w = synth.weight(H, dt).to(dev)
                        bias = synth.cast(synth.normal_np((H,), 7, std=0.1), dt).to(dev)
                        nb = 2 * R * H * elem + 2 * H * elem
                        run = lambda p: _abi.ks_layer_norm_planned(
                            y.data_ptr(), x.data_ptr(), w.data_ptr(), bias.data_ptr(), R, H, 1e-5,
                            code, p, s)
                        default = lambda: _abi.check(_abi.ks_layer_norm(
                            y.data_ptr(), x.data_ptr(), w.data_ptr(), bias.data_ptr(), R, H, 1e-5,
                            code, s))
                fns = [("default", default)]
                for name, p in op_band_candidates(op, hv):
                    if run(p) == _abi.KS_SUCCESS:  # a plan that does not fit is left out
                        fns.append((name, (lambda p=p: _abi.check(run(p)))))
                _, dp = _abi.ks_plan_launch(op_codes[op], R, H, code, True, sms, 0)
                line = {"ops_bands": op, "dtype": dt, "hv": hv, "hidden": H, "rows": R,
                        "default_plan": {k: dp.as_dict()[k] for k in ("kernel_name", "vec_per_thread",
                                                                       "block", "flags", "team",
                                                                       "stages")}}
                for ctx in ("steady", "after_ring"):
                    res = {name: [] for name, _ in fns}
                    for _ in range(args.plan_sweep_rounds):
                        for name, fn in fns:
                            t = steady(fn) if ctx == "steady" else after(fn)
                            res[name].append(nb / t / 1e9 / peak)
                    line[ctx] = {k: round(statistics.median(v), 4) for k, v in res.items()}
                print(json.dumps(line), flush=True)
                del x, y
                torch.cuda.empty_cache()
    st_, flags = _abi.ks_device_faults(clear=False)
    if st_ != _abi.KS_SUCCESS or flags:
        print(json.dumps({"ops_bands": "device faults", "status": st_, "flags": flags}))
        return 1
    return 0


def ops_bands_table(jsonl_path: str) -> str:
    """A markdown table from an --ops-bands run: per operator, dtype and width, the default
    launch's score and the best candidate's, each the worse of its two contexts."""
    rows = []
    for ln in open(jsonl_path):
        if not ln.startswith('{"ops_bands"'):
            continue
        d = json.loads(ln)
        if "steady" not in d:
            continue
        score = {k: min(d["steady"][k], d.get("after_ring", d["steady"]).get(k, 0.0))
                 for k in d["steady"]}
        best = max(score, key=score.get)
        dp = d["default_plan"]
        rows.append(f"| {d['ops_bands']} | {d['dtype']} | {d['hv']} | {dp['kernel_name']} v{dp['vec_per_thread']} "
                    f"b{dp['block']}{' n' if dp['flags'] & 1 else ''} | {score['default']:.3f} | "
                    f"{best} | {score[best]:.3f} | {score[best] - score['default']:+.3f} |")
    head = ("| op | dtype | vectors | default plan | default score | best | best score | best - "
            "default |\n|---|---|---|---|---|---|---|---|")
    return head + "\n" + "\n".join(rows)


LN_RING_BYTES = 64 * 1024  # the library's LayerNorm ring: rows of this many bytes per CTA


def band_of(name: str, default_plan: dict, op: str, hv: int):
    """(kind, v, prefetch, team, block) of a band-candidate name, the library's Band fields;
    'default' maps the launch the library made to the same fields, 'g' when it is the general
    rule's CTA row. Kinds: w (a team of `team` lanes per row), c (a CTA per row), r (the
    LayerNorm staged ring, v = its stages), x (the wide multi-pass kernel on `block` threads)."""
    import re
    if name == "default":
        k, v, npf = default_plan["kernel_name"], default_plan["vec_per_thread"], default_plan["flags"] & 1
        if k == "warp_row":
            return ("w", v, not npf, default_plan.get("team", 32) or 32, 0)
        if k == "twopass_row":
            return ("x", 4, True, 32, default_plan["block"])
        if k == "bulk_row":
            st = default_plan.get("stages") or max(2, min(8, LN_RING_BYTES // (hv * 16)))
            return ("R" if default_plan["flags"] & 4 else "r", st, True, 32, 0)
        gen_v = 1 if hv < 64 else (2 if hv < 128 else 4)
        gen_pf = True if op == "layer_norm" else (gen_v != 4 or hv > 1024)
        # for many LayerNorm rows wider than 512 vectors the general rule is the ring or the
        # wide kernel, so a CTA row there is a band of its own
        gen_cta = not (op == "layer_norm" and hv > 512)
        if k == "cta_row" and v == gen_v and (not npf) == gen_pf and gen_cta:
            return ("g", 0, gen_pf, 32, 0)
        return ("c", v, not npf, 32, 0)
    m = re.fullmatch(r"t(\d+)v(\d)(n?)", name)
    if m:
        return ("w", int(m.group(2)), not m.group(3), int(m.group(1)), 0)
    m = re.fullmatch(r"x(\d+)", name)
    if m:
        return ("x", 4, True, 32, int(m.group(1)))
    m = re.fullmatch(r"r(\d)(a?)", name)
    if m:
        return ("R" if m.group(2) else "r", int(m.group(1)), True, 32, 0)
    m = re.fullmatch(r"([wc])(\d)(n?)", name)
    return (m.group(1), int(m.group(2)), not m.group(3), 32, 0)


def ops_candidate_name(plan: dict, hv: int) -> str:
    """The --ops-bands candidate name of a Softmax or LayerNorm launch plan (as the JSON lines
    report it): w / tTEAMv (warp rows), c (CTA rows), r (the LayerNorm ring, its stages; a: the
    weight and bias rows in shared memory), x (the wide kernel, its block); n: no prefetch. hv:
    the row's width in 16-byte vectors (older runs did not report the ring's stages)."""
    k, v, n = plan["kernel_name"], plan["vec_per_thread"], "n" if plan["flags"] & 1 else ""
    if k == "warp_row":
        team = plan.get("team") or 32
        return (f"w{v}" if team == 32 else f"t{team}v{v}") + n
    if k == "cta_row":
        return f"c{v}{n}"
    if k == "bulk_row":
        st = plan.get("stages") or max(2, min(8, LN_RING_BYTES // (hv * 16)))
        return f"r{st}" + ("a" if plan["flags"] & 4 else "")
    if k == "twopass_row":
        return f"x{plan['block']}"
    return k


def ops_bands_record(jsonl_paths) -> dict:
    """The measured record behind the Softmax and LayerNorm width bands, from --ops-bands runs:
    per operator, dtype and width, every candidate's score (the worse of its two contexts, in
    thousandths of the measured copy peak), the band the library's default launch was and that
    launch's candidate name. A width measured by several runs keeps the last."""
    lines = {}
    for path in jsonl_paths:
        for ln in open(path):
            if not ln.startswith('{"ops_bands"'):
                continue
            d = json.loads(ln)
            if d["ops_bands"] not in ("softmax", "layer_norm") or "steady" not in d:
                continue
            sc = {k: round(1000 * min(d["steady"][k], d.get("after_ring", d["steady"]).get(k, 0.0)))
                  for k in d["steady"]}
            lines[(d["ops_bands"], d["dtype"], d["hv"])] = {
                "op": d["ops_bands"], "dtype": d["dtype"], "hv": d["hv"],
                "default_band": list(band_of("default", d["default_plan"], d["ops_bands"], d["hv"])),
                "default_name": ops_candidate_name(d["default_plan"], d["hv"]),
                "scores": sc}
    return {"what": "Softmax and LayerNorm launch scores per width, many rows",
            "score": "worse of steady state and after a large-shared-memory kernel, thousandths "
                     "of the measured copy peak",
            "lines": [lines[k] for k in sorted(lines)]}


def derive_bands(record: dict, op: str, dtypes, min_gain: int = 10):
    """Width bands for op from a record of --ops-bands runs, by one rule: at each measured width,
    score every candidate by its worse context, and over `dtypes` (the dtypes that share one
    table) by its worst dtype; keep the library's current plan unless another candidate scores at
    least `min_gain` thousandths (a point of the copy peak) higher, then take the best. Consecutive
    widths with the same plan merge into one band reaching to the last of them. Returns
    [(hi, kind, v, prefetch, team, block)], closed by the general rule."""
    by_w = {}
    for ln in record["lines"]:
        if ln["op"] == op and ln["dtype"] in dtypes:
            by_w.setdefault(ln["hv"], {})[ln["dtype"]] = ln
    bands = []
    for hv in sorted(by_w):
        per = by_w[hv]
        if set(per) != set(dtypes):
            continue
        names = set.intersection(*(set(ln["scores"]) for ln in per.values()))
        worst = {n: min(per[dt]["scores"][n] for dt in per) for n in names}
        cur = tuple(per[dtypes[0]]["default_band"])
        best = max(sorted(worst), key=worst.get)
        pick = cur if worst[best] - worst["default"] < min_gain else band_of(best, None, op, hv)
        if bands and bands[-1][1:] == pick:
            bands[-1] = (hv,) + pick
        else:
            bands.append((hv,) + pick)
    bands.append((32767, "g", 0, True, 32, 0))
    return bands


OPS_BAND_TABLES = (("kSoftmax16", "softmax", ["bf16", "fp16"]), ("kSoftmax32", "softmax", ["fp32"]),
                   ("kLayerNormBf16", "layer_norm", ["bf16"]),
                   ("kLayerNormF16", "layer_norm", ["fp16"]),
                   ("kLayerNormF32", "layer_norm", ["fp32"]))


def bands_cpp(name: str, bands) -> str:
    """The bands as the library's C++ table."""
    def one(b):
        hi, kind, v, pf, team, block = b
        hi_s = "kBandEnd" if hi == 32767 else str(hi)
        pf_s = "true" if pf else "false"
        if block:
            return f"{{{hi_s}, '{kind}', {v}, {pf_s}, {team}, {block}}}"
        return (f"{{{hi_s}, '{kind}', {v}, {pf_s}, {team}}}" if team != 32
                else f"{{{hi_s}, '{kind}', {v}, {pf_s}}}")
    return f"constexpr Band {name}[] = {{" + ", ".join(one(b) for b in bands) + "};"


# The launch codes of the library's band table for many rows of 1..2048 16-byte vectors (lower
# case: without prefetch): E / e an 8-lane team per row (rows of at most 32 vectors) and H / h a
# 16-lane team (at most 64), at the fewest of 1, 2 or 4 vectors per lane that cover the row;
# W / w a warp per row at the fewest of 1, 2, 4, 6 or 8 vectors per lane (at most 256 vectors);
# T / t a CTA per row at 2 vectors per thread, F / f the same at 4; R the staged ring of 2
# stages; P the two-pass kernel in its default shape (no L2 prefetch).
PLAN_BAND_CODES = "EeHhWwTtFfRP"
PLAN_BAND_ONE_PASS = "EeHhWwTtFf"
PLAN_BAND_LO, PLAN_BAND_HI = 1, 2048


def plan_band_candidate(code: str, op: str, dtype: str, hv: int):
    """The plan-contexts candidate a band code launches at width hv (None where it does not
    apply: teams and warp rows that cannot cover the row)."""
    sfx = "n" if code.islower() else ""
    if code in "EeHh":
        team = 8 if code in "Ee" else 16
        v = next((v for v in (1, 2, 4) if team * v >= hv), None)
        return f"t{team}v{v}{sfx}" if v else None
    if code in "Ww":
        v = next((v for v in (1, 2, 4, 6, 8) if 32 * v >= hv), None)
        return f"w{v}{sfx}" if v else None
    if code == "P":
        return "t512u2n" if (op == "fused_add_rms_norm" and dtype != "fp32") else "t256u4n"
    return {"T": "p2", "t": "n2", "F": "p4", "f": "n4", "R": "b2"}[code]


def plan_bands_record(jsonl_paths, sm_count: int) -> dict:
    """The measured record behind the band table, from one or more --plan-contexts runs: per dtype
    and op, the widths, the row counts, and for every band code its score at each width (the worse
    of its two contexts, as thousandths of the measured copy peak; the mean over runs that
    measured the width)."""
    acc = {}
    for path in jsonl_paths:
        for ln in open(path):
            if not ln.startswith('{"plan_contexts"'):
                continue
            d = json.loads(ln)
            if "steady" not in d or not (PLAN_BAND_LO <= d["hv"] <= PLAN_BAND_HI):
                continue
            sc = {k: min(d["steady"][k], d.get("after_ring", d["steady"]).get(k, 0.0))
                  for k in d["steady"]}
            key = f"{d['plan_contexts']}/{d['op']}"
            slot = acc.setdefault(key, {}).setdefault(d["hv"], {"rows": d["rows"], "runs": []})
            slot["runs"].append({c: sc.get(plan_band_candidate(c, d["op"], d["plan_contexts"],
                                                               d["hv"])) for c in PLAN_BAND_CODES})
    tables = {}
    for key, by_w in sorted(acc.items()):
        hvs = sorted(by_w)
        t = {"hv": hvs, "rows": [by_w[h]["rows"] for h in hvs]}
        for c in PLAN_BAND_CODES:
            col = []
            for h in hvs:
                vals = [r[c] for r in by_w[h]["runs"] if r[c] is not None]
                col.append(round(1000 * sum(vals) / len(vals)) if vals else None)
            t[c] = col
        tables[key] = t
    return {"what": "RMSNorm launch-plan scores for many rows of 1..2048 16-byte vectors",
            "score": "worse of steady state and after a large-shared-memory kernel, thousandths "
                     "of the measured copy peak, mean over runs",
            "sm_count": sm_count, "runs": len(jsonl_paths), "tables": tables}


def derive_plan_bands(record: dict, tol: int = 10) -> dict:
    """The band table a record implies, by one rule: the fewest bands over the measured widths
    such that at every width the band's code scores within `tol` thousandths (a point of the copy
    peak) of that width's best code. Built left to right, each band as wide as the codes common
    to its widths allow (which gives the fewest bands), and among those codes the one with the
    best mean score. A band reaches to its last measured width (the last band to 2048 vectors);
    widths between two measured ones take the next band. The staged ring and the two-pass kernel
    need at least 4 rows per SM, so their bands also name a fallback: the one-pass code with the
    best mean score over the band's widths. Returns {"dtype/op": [(hi, code, fallback)]}."""
    out = {}
    for key, t in record["tables"].items():
        hvs = t["hv"]
        t = {c: t.get(c, [None] * len(hvs)) for c in PLAN_BAND_CODES}  # a code not measured
        ok = []
        for i in range(len(hvs)):
            sc = {c: t[c][i] for c in PLAN_BAND_CODES if t[c][i] is not None}
            best = max(sc.values())
            ok.append({c for c, v in sc.items() if v >= best - tol})
        bands, i = [], 0
        while i < len(hvs):
            common, j = set(ok[i]), i
            while j + 1 < len(hvs) and common & ok[j + 1]:
                common &= ok[j + 1]
                j += 1
            mean = lambda c, lo=i, hi=j: sum(t[c][k] for k in range(lo, hi + 1)) / (hi - lo + 1)
            code = max(sorted(common), key=mean)
            fb = code
            if code in "RP":
                one = [c for c in PLAN_BAND_ONE_PASS
                       if all(t[c][k] is not None for k in range(i, j + 1))]
                fb = max(one, key=mean)
            bands.append((hvs[j], code, fb))
            i = j + 1
        bands[-1] = (PLAN_BAND_HI, bands[-1][1], bands[-1][2])
        out[key] = bands
    return out


WIDE_LO, WIDE_HI = 2049, 32768  # the wide band table: many rows, tensors larger than L2


def wide_plan_fields(name: str):
    """(kernel, cluster, block, v, stages, flags) of a plan-sweep candidate name for rows wider
    than 2048 vectors (block 0: fitted to the slice, ceil(ceil(hv / cluster) / v) rounded up to a
    warp): tBuU[n] the two-pass kernel, sCbBuU[n|p] split over a cluster (p: two rows in
    flight), cC the register-resident cluster kernel, bCsS[v8][m] the staged kernel (m: the rows
    kept in shared memory)."""
    import re
    from row_wise_rmsnorm_ks_gb300 import _abi
    npf = _abi.KS_PLAN_NO_PREFETCH
    m = re.fullmatch(r"t(\d+)u(\d)(n?)", name)
    if m:
        return (_abi.KS_KERNEL_TWOPASS_ROW, 0, int(m.group(1)), int(m.group(2)), 0,
                npf if m.group(3) else 0)
    m = re.fullmatch(r"s(\d)b(\d+)u(\d)([np]?)", name)
    if m:
        return (_abi.KS_KERNEL_TWOPASS_ROW, int(m.group(1)), int(m.group(2)), int(m.group(3)),
                2 if m.group(4) == "p" else 0, npf if m.group(4) else 0)
    m = re.fullmatch(r"c(\d)", name)
    if m:
        return (_abi.KS_KERNEL_CLUSTER_ROW, int(m.group(1)), 0, 4, 0, 0)
    m = re.fullmatch(r"b(\d+)s(\d)(v8)?(m?)", name)
    if m:
        return (_abi.KS_KERNEL_BULK_ROW, int(m.group(1)), 0, 8 if m.group(3) else 4,
                int(m.group(2)), _abi.KS_PLAN_SMEM_ROWS if m.group(4) else 0)
    return None


def wide_bands_record(log_paths, sm_count: int) -> dict:
    """The measured record behind the wide band table, from --plan-sweep runs: per dtype, op and
    width (2049..32768 vectors), the candidates within 5 points of that width's best (thousandths
    of the measured copy peak; a candidate further behind can never be a band's launch under a
    one-point rule) and the default's score. A width measured several times in one run keeps the
    mean; a later run that measured a width replaces the earlier runs' lines for it (a run may
    measure candidates the earlier ones did not)."""
    acc = {}
    for i, path in enumerate(log_paths):
        for ln in open(path):
            if not ln.startswith('{"plan_sweep"'):
                continue
            d = json.loads(ln)
            if "default" not in d or not (WIDE_LO <= d["hv"] <= WIDE_HI):
                continue
            key = (f"{d['plan_sweep']}/{d['op']}", d["hv"])
            slot = acc.get(key)
            if slot is None or slot["run"] != i:
                slot = acc[key] = {"rows": d["rows"], "runs": [], "run": i}
            slot["runs"].append({k: v for k, v in d.items() if isinstance(v, float)})
    tables = {}
    for (key, hv), slot in sorted(acc.items()):
        names = set.intersection(*(set(r) for r in slot["runs"]))
        mean = {n: round(1000 * sum(r[n] for r in slot["runs"]) / len(slot["runs"])) for n in names}
        best = max(v for n, v in mean.items() if n != "default")
        keep = {n: v for n, v in mean.items()
                if n == "default" or (v >= best - 50 and wide_plan_fields(n))}
        tables.setdefault(key, []).append({"hv": hv, "rows": slot["rows"], "scores": keep})
    return {"what": "RMSNorm launch-plan scores for many rows of 2049..32768 16-byte vectors, "
                    "tensors larger than L2",
            "score": "thousandths of the measured copy peak, back-to-back launches, mean over runs; "
                     "candidates within 5 points of the best, and the default",
            "sm_count": sm_count, "runs": len(log_paths), "tables": tables}


def derive_wide_bands(record: dict, tol: int = 10) -> dict:
    """The wide band table a record implies, by the rule of derive_plan_bands: the fewest bands
    such that at every measured width the band's launch scores within `tol` thousandths of that
    width's best; each band as wide as the launches common to its widths allow, the launch with
    the best mean among them; the last band reaching to 32768 vectors. Only portable cluster
    sizes (at most 8 CTAs) are candidates, so the default launch never depends on the device
    placing a larger cluster. Returns {"dtype/op": [(hi, name)]}."""
    out = {}
    for key, lines in record["tables"].items():
        ok = []
        for ln in lines:
            sc = {n: v for n, v in ln["scores"].items()
                  if n != "default" and wide_plan_fields(n)[1] <= 8}
            best = max(sc.values())
            ok.append({n for n, v in sc.items() if v >= best - tol})
        bands, i = [], 0
        while i < len(lines):
            common, j = set(ok[i]), i
            while j + 1 < len(lines) and common & ok[j + 1]:
                common &= ok[j + 1]
                j += 1
            mean = lambda n, lo=i, hi=j: sum(lines[k]["scores"][n] for k in range(lo, hi + 1))
            name = max(sorted(common), key=mean)
            bands.append((lines[j]["hv"], name))
            i = j + 1
        bands[-1] = (WIDE_HI, bands[-1][1])
        out[key] = bands
    return out


WIDE_BAND_TABLES = (("fp32", "kWideBandsF32"), ("fp16", "kWideBandsF16"), ("bf16", "kWideBandsBf16"))


def wide_bands_cpp(bands: dict) -> str:
    """The wide band table as the library's C++ source: {hi, kernel, cluster, block (0: fitted),
    vectors per thread, stages, flags}, one array per dtype and op."""
    lines = []
    for dt, name in WIDE_BAND_TABLES:
        for op, suffix in (("rms_norm", "Plain"), ("fused_add_rms_norm", "Fused")):
            body = ", ".join("{%d, %d, %d, %d, %d, %d, %d}" % ((hi,) + wide_plan_fields(n))
                             for hi, n in bands[f"{dt}/{op}"])
            lines.append(f"constexpr WideBand {name}{suffix}[] = {{{body}}};")
    return "\n".join(lines)


PLAN_BAND_TABLES = (("fp32", "kRowBandsF32"), ("fp16", "kRowBandsF16"), ("bf16", "kRowBandsBf16"))


def plan_bands_cpp(bands: dict) -> str:
    """The band table as the library's C++ source (one array per dtype and op)."""
    lines = []
    for dt, name in PLAN_BAND_TABLES:
        for op, suffix in (("rms_norm", "Plain"), ("fused_add_rms_norm", "Fused")):
            body = ", ".join(f"{{{hi}, '{c}', '{fb}'}}" for hi, c, fb in bands[f"{dt}/{op}"])
            lines.append(f"constexpr RowBand {name}{suffix}[] = {{{body}}};")
    return "\n".join(lines)


def plan_bands_table(record: dict) -> str:
    """A markdown table of a record: per dtype, op and width, the derived band's code and score
    against the best code's."""
    bands = derive_plan_bands(record)
    rows = []
    for key, t in record["tables"].items():
        for i, hv in enumerate(t["hv"]):
            code = next(c for hi, c, _ in bands[key] if hv <= hi)
            sc = {c: t[c][i] for c in PLAN_BAND_CODES if t[c][i] is not None}
            best = max(sc, key=sc.get)
            rows.append(f"| {key} | {hv} | {code} | {sc[code] / 1000:.3f} | {best} | "
                        f"{sc[best] / 1000:.3f} |")
    return ("| dtype/op | vectors | band code | score | best code | best score |\n"
            "|---|---|---|---|---|---|\n" + "\n".join(rows))


def run_ops_scan(args) -> int:
    """The next operators' default launches over row widths (one JSON line per dtype and width;
    not the contract's line): Softmax, LayerNorm (weight and bias) and SwiGLU on rows of
    --plan-sweep-widths 16-byte vectors (SwiGLU: d of that many vectors), 384 MiB per input
    tensor, N(0,1) inputs, each timed in steady state (back-to-back launches) and right after one
    launch of the staged RMSNorm ring, a kernel with a large shared-memory carveout (each launch
    timed alone); the median of --plan-sweep-rounds rounds, as a fraction of the measured copy
    peak."""
    import torch

    from row_wise_rmsnorm_ks_gb300 import _abi, synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    peak = measured_peaks()["hbm_gbs"]
    codes = {"bf16": _abi.KS_DTYPE_BF16, "fp16": _abi.KS_DTYPE_F16, "fp32": _abi.KS_DTYPE_F32}

    def steady(fn, n=25):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(4):
            fn()
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n * 1e-3

    def after(fn, pre, n=10):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tot = 0.0
        for _ in range(n):
            pre()
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b) * 1e-3
        return tot / n

    widths = [int(v) for v in (args.plan_sweep_widths or "64,96,128,160,192,256,512,1024,2048").split(",")]
    for dt in args.plan_sweep_dtypes.split(","):
        e = 4 if dt == "fp32" else 2
        code = codes[dt]
        for hv in widths:
            H = hv * 16 // e
            R = (384 << 20) // (H * e)
            x = synth.cast(synth.normal_dev((R, H), synth.SEED_X, dev), dt)
            y = torch.empty_like(x)
            w = synth.weight(H, dt).to(dev)
            b = synth.weight(H, dt).to(dev)
            ring = _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, -(-(-(-hv // 4)) // 32) * 32, 2)
            pre = (lambda: _abi.check(_abi.ks_rms_norm_planned(
                y.data_ptr(), x.data_ptr(), w.data_ptr(), R, H, 1e-5, code, ring, s)))
            if 128 + 2 * hv * 16 > 226 * 1024 or hv > 2048:
                pre = None  # no ring of two stages fits: steady context only
            R2 = R // 2  # SwiGLU reads x as [R2, 2H] and writes [R2, H] into y
            ops = {
                "softmax": (2 * R * H * e,
                            lambda: _abi.check(_abi.ks_softmax(y.data_ptr(), x.data_ptr(), R, H,
                                                               code, s))),
                "layer_norm": (2 * R * H * e + 2 * H * e,
                               lambda: _abi.check(_abi.ks_layer_norm(
                                   y.data_ptr(), x.data_ptr(), w.data_ptr(), b.data_ptr(), R, H,
                                   1e-5, code, s))),
                "silu_and_mul": (3 * R2 * H * e,
                                 lambda: _abi.check(_abi.ks_silu_and_mul(
                                     y.data_ptr(), x.data_ptr(), R2, H, code, s))),
            }
            line = {"ops_scan": dt, "hv": hv, "hidden": H, "rows": R}
            for name, (nb, fn) in ops.items():
                st, af = [], []
                for _ in range(args.plan_sweep_rounds):
                    st.append(nb / steady(fn) / 1e9 / peak)
                    if pre:
                        af.append(nb / after(fn, pre) / 1e9 / peak)
                line[name] = {"steady": round(statistics.median(st), 4),
                              "after_ring": round(statistics.median(af), 4) if af else None}
            print(json.dumps(line), flush=True)
            del x, y, w, b
            torch.cuda.empty_cache()
    st, flags = _abi.ks_device_faults(clear=False)
    if st != _abi.KS_SUCCESS or flags:
        print(json.dumps({"ops_scan": "device faults", "status": st, "flags": flags}))
        return 1
    return 0


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ks", "reference"], default="ks")
    ap.add_argument("--rows", type=int, default=32768)
    ap.add_argument("--hidden", type=int, default=8192)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-workspace-mb", type=int, default=192)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--decode-samples", type=int, default=500)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-next-ops", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="print the configuration sweeps, one JSON line per case, and exit")
    ap.add_argument("--sweep-samples", type=int, default=15)
    ap.add_argument("--ops-bands", action="store_true",
                    help="time the next operators' band candidates in two contexts (tuning)")
    ap.add_argument("--ops-bands-ops", default="softmax,layer_norm,silu_and_mul")
    ap.add_argument("--ops-bands-table", metavar="JSONL",
                    help="print the markdown table of an --ops-bands run")
    ap.add_argument("--ops-bands-record", nargs="+", metavar="JSONL",
                    help="print the JSON record of one or more --ops-bands runs (the data the "
                         "Softmax and LayerNorm band tables are derived from)")
    ap.add_argument("--ops-bands-derive", metavar="JSON",
                    help="print the Softmax and LayerNorm band tables an --ops-bands-record "
                         "record implies")
    ap.add_argument("--plan-bands-record", nargs="+", metavar="JSONL",
                    help="print the JSON record of one or more --plan-contexts runs (the data the "
                         "RMSNorm band table is derived from)")
    ap.add_argument("--plan-bands-derive", metavar="JSON",
                    help="print the RMSNorm band table a --plan-bands-record record implies")
    ap.add_argument("--plan-bands-table", metavar="JSON",
                    help="print the markdown table of a --plan-bands-record record")
    ap.add_argument("--plan-probe", metavar="NAME",
                    help="launch one plan-sweep candidate a few times on --rows x --hidden and exit "
                         "(a fixed workload for a profiler)")
    ap.add_argument("--probe-launches", type=int, default=4)
    ap.add_argument("--probe-dtype", default="bf16", choices=["bf16", "fp16", "fp32"])
    ap.add_argument("--probe-op", default="rms_norm", choices=["rms_norm", "fused_add_rms_norm"])
    ap.add_argument("--wide-bands-record", nargs="+", metavar="LOG",
                    help="print the JSON record of one or more --plan-sweep runs over rows wider "
                         "than 2048 vectors (the data the wide band table is derived from)")
    ap.add_argument("--wide-bands-derive", metavar="JSON",
                    help="print the wide band table a --wide-bands-record record implies")
    ap.add_argument("--record-sm-count", type=int, default=0,
                    help="the SM count of the box the runs were taken on (default: this GPU's)")
    ap.add_argument("--kernel-times", action="store_true",
                    help="every stated configuration a fixed number of times, for an ncu launch list")
    ap.add_argument("--kernel-time-launches", type=int, default=5)
    ap.add_argument("--kernel-times-table", nargs=2, metavar=("JSONL", "NCU_CSV"),
                    help="print the markdown table joining a kernel-times run with its ncu launch list")
    ap.add_argument("--plan-sweep", action="store_true",
                    help="time every candidate launch plan per dtype, op and width, and exit")
    ap.add_argument("--plan-contexts", action="store_true",
                    help="compare the register-kernel plans per width in steady state and right "
                         "after a large-shared-memory kernel, and exit")
    ap.add_argument("--ops-scan", action="store_true",
                    help="time the next operators' default launches per dtype and width, in steady "
                         "state and right after a large-shared-memory kernel, and exit")
    ap.add_argument("--plan-sweep-rounds", type=int, default=3)
    ap.add_argument("--plan-sweep-dtypes", default="bf16,fp16,fp32")
    ap.add_argument("--plan-sweep-ops", default="rms_norm,fused_add_rms_norm",
                    help="--plan-sweep: the operators, comma-separated")
    ap.add_argument("--plan-sweep-widths", default="",
                    help="comma-separated row widths in 16-byte vectors (default: the full grid)")
    ap.add_argument("--next-rows", type=int, default=32768,
                    help="rows of the next operators' large shapes (width 8192)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-rows-max", type=int, default=8192)
    ap.add_argument("--reference-seconds", type=float, default=90.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.kernel_times:
        return run_kernel_times(args)
    if args.ops_bands:
        return run_ops_bands(args)
    if args.ops_bands_table:
        print(ops_bands_table(args.ops_bands_table))
        return 0
    if args.ops_bands_record:
        print(json.dumps(ops_bands_record(args.ops_bands_record), separators=(",", ":")))
        return 0
    if args.ops_bands_derive:
        rec = json.load(open(args.ops_bands_derive))
        for name, op, dts in OPS_BAND_TABLES:
            print(bands_cpp(name, derive_bands(rec, op, dts)))
        return 0
    if args.kernel_times_table:
        print(kernel_times_table(*args.kernel_times_table))
        return 0
    if args.plan_bands_record:
        sms = args.record_sm_count
        if sms <= 0:
            import torch
            sms = device_facts(torch.device("cuda", 0))["sm_count"]
        print(json.dumps(plan_bands_record(args.plan_bands_record, sms), separators=(",", ":")))
        return 0
    if args.wide_bands_record:
        sms = args.record_sm_count
        if sms <= 0:
            import torch
            sms = device_facts(torch.device("cuda", 0))["sm_count"]
        print(json.dumps(wide_bands_record(args.wide_bands_record, sms), separators=(",", ":")))
        return 0
    if args.wide_bands_derive:
        print(wide_bands_cpp(derive_wide_bands(json.load(open(args.wide_bands_derive)))))
        return 0
    if args.plan_bands_derive:
        print(plan_bands_cpp(derive_plan_bands(json.load(open(args.plan_bands_derive)))))
        return 0
    if args.plan_bands_table:
        print(plan_bands_table(json.load(open(args.plan_bands_table))))
        return 0
    if args.plan_sweep:
        return run_plan_sweep(args)
    if args.plan_contexts:
        return run_plan_contexts(args)
    if args.plan_probe:
        return run_plan_probe(args)
    if args.ops_scan:
        return run_ops_scan(args)
    return run_ks(args)


if __name__ == "__main__":
    sys.exit(main())
