#!/usr/bin/env python
"""Throughput of the fp16 GEMM D = A * B^T on GB300.

One step = one pass of the hot path over one batch of synthetic input: the 8192^3 GEMM and the
MLP up-projection GEMM (M 16384, N 14336, K 4096), inputs resident in HBM.  The line reports
fp16 GEMM TFLOP/s over both (total algorithmic FLOPs 2*M*N*K / total time) with a breakdown per
shape, the dominant kernel's roofline, an end-to-end figure with host copies, clocks sampled
during the timed region, and the CPU oracle's throughput on a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun), every rank runs its own replica of the step on its own GPU (the GEMM
here has no exchange step), the timed region is bracketed by barriers and the maximum time over
ranks is used: value = FLOPs of all ranks / that time ("weak" scaling).
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fp16 GEMM TFLOP/s at 8192³ and MLP shape; % of GB300 dense fp16 peak"
WORKLOADS = ("square_8192", "mlp_up_16384x14336x4096")
FALLBACK_PEAK_TFLOPS = 1900.0
L2_BYTES = 129e6
FLOP_PER_CLK_PER_SM = 8192


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=800)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--variant", type=int, default=0, help="kernel variant (0 = auto)")
    p.add_argument("--e2e-steps", type=int, default=30)
    p.add_argument("--e2e-repeats", type=int, default=3,
                   help="timed regions of the e2e leg; it reports their median (the host link "
                        "is shared with other jobs on the host)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--only", default="", help="comma-separated subset of the step's workloads")
    p.add_argument("--skip-e2e", action="store_true")
    p.add_argument("--sweep", action="store_true",
                   help="time every workload under every kernel variant (with and without a "
                        "stream-K workspace) and print one JSON line per case instead of the "
                        "bench line")
    p.add_argument("--sweep-workloads", default="",
                   help="comma-separated subset of workloads for --sweep (default: all five)")
    p.add_argument("--sweep-variants", default="1,2,3,4,5,6",
                   help="variants for --sweep; 'auto' = the automatic choice only")
    p.add_argument("--sweep-reps", type=int, default=0,
                   help="timed launches per case in --sweep (0: about 0.3 s of work)")
    p.add_argument("--sweep-no-stream-k", action="store_true")
    p.add_argument("--sweep-cold-l2", action="store_true",
                   help="in --sweep, write a 512 MiB scratch buffer before every launch and time "
                        "each launch alone (events around the launch only)")
    p.add_argument("--sweep-processes", type=int, default=1,
                   help="run --sweep in this many fresh processes and report, per case, the "
                        "median of the per-process means")
    p.add_argument("--fused-steps", type=int, default=100,
                   help="steps of the fused leg: bf16 act(A B^T + bias) with GELU on the headline "
                        "step's two shapes (0: skip)")
    p.add_argument("--fused-act", default="gelu", choices=["none", "relu", "gelu"],
                   help="activation of the fused leg")
    p.add_argument("--mx-steps", type=int, default=200,
                   help="steps of the block-scaled FP8 leg (8192^3 and MLP shapes; 0: skip)")
    p.add_argument("--mx-variant", type=int, default=0, help="block-scaled variant (0 = auto)")
    p.add_argument("--gdn-reps", type=int, default=20,
                   help="fewest timed calls per Gated Delta Net scenario (0: skip the leg)")
    p.add_argument("--gdn-min-ms", type=float, default=5.0,
                   help="time at least this many milliseconds of calls per Gated Delta Net "
                        "scenario (0: exactly --gdn-reps calls)")
    p.add_argument("--gdn-scan", default="auto",
                   choices=["auto", "tensor_core", "mma_sync", "tensor_core_16", "tensor_core_32"],
                   help="scan kernel of the Gated Delta Net leg")
    p.add_argument("--gdn-only", action="store_true",
                   help="run only the Gated Delta Net leg and print its JSON")
    p.add_argument("--gdn-scenarios", default="",
                   help="comma-separated Gated Delta Net scenarios to time (default: all six)")
    p.add_argument("--gdn-warm-ms", type=float, default=50.0,
                   help="warm-up time per Gated Delta Net scenario, in batches of 8 calls "
                        "(0: exactly one batch)")
    p.add_argument("--sweep-mx", action="store_true",
                   help="in --sweep, time the block-scaled FP8 workloads instead")
    p.add_argument("--config-ms", type=float, default=200.0,
                   help="back-to-back milliseconds per config in the per_config leg (single tile, "
                        "2048^3, 3000x5000x1000; 0: skip)")
    p.add_argument("--config-processes", type=int, default=3,
                   help="processes the per_config leg runs in (this one and fresh ones); each "
                        "figure is the median of the per-process means")
    p.add_argument("--config-only", action="store_true",
                   help="run only the per_config leg in this process and print it (the fresh "
                        "processes of --config-processes)")
    p.add_argument("--sustained-ms", type=float, default=1500.0,
                   help="length of the sustained leg: the headline step back to back for at "
                        "least this long, with its own clock record (0: skip)")
    p.add_argument("--record-traffic-mx", default="",
                   help="write profiles/ncu_traffic_mx.json from an ncu csv log of the block-scaled "
                        "FP8 step's two launches")
    p.add_argument("--record-traffic-gdn", default="",
                   help="write profiles/ncu_traffic_gdn.json from an ncu csv log of one Gated "
                        "Delta Net call's launches (the roofline scenario)")
    p.add_argument("--record-traffic", default="",
                   help="read an ncu CSV log of the two GEMM launches of one step (metrics "
                        "dram__bytes_read.sum, dram__bytes_write.sum, gpu__time_duration.sum; "
                        "-k regex:gemm_ws) and write profiles/ncu_traffic.json for the current "
                        "kernel sources, then exit")
    p.add_argument("--cublas-steps", type=int, default=-1,
                   help="steps of torch.mm on the same shapes, for context (-1: as many as "
                        "--steps, 0: skip)")
    return p.parse_args()


def step_workloads(args):
    if not args.only:
        return WORKLOADS
    names = tuple(n.strip() for n in args.only.split(",") if n.strip())
    for n in names:
        if n not in WORKLOADS:
            raise SystemExit(f"--only: unknown workload {n!r}; choose from {WORKLOADS}")
    return names


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def clocks_rejected(info) -> bool:
    """True for a clock record the timing rules reject: hw_slowdown, hw_thermal_slowdown or
    sw_thermal_slowdown active, or a median SM clock under 60% of its maximum with no reason
    (sw_power_cap alone is normal under a dense GEMM and is kept)."""
    if not info:
        return False
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(info.get("reasons") or []):
        return True
    sm, mx = info.get("sm_mhz"), info.get("sm_max_mhz")
    return bool(sm and mx and sm < 0.6 * mx and not info.get("reasons"))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's `value` (a job's time is its slowest rank's); the same value
    on every rank.  Works on any initialised process group (NCCL on the GPUs, gloo on the CPU)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, steps: int, flops_step: float, total_ms: float) -> float:
    """Every rank runs the same step on its own GPU (replicas): the job's throughput is all
    ranks' FLOPs over the slowest rank's time."""
    return world * steps * flops_step / (total_ms * 1e-3) / 1e12


GEMM_KERNEL_SOURCES = ("desc.h", "gemm_f16.cu", "gemm_kernels.cuh", "ptx.cuh")
GDN_KERNEL_SOURCES = ("desc.h", "gdn.cu", "gdn_offsets.h", "ptx.cuh")


def kernel_source_hash(sources=GEMM_KERNEL_SOURCES) -> str:
    """sha256 over a kernel's sources (the GEMM's by default): a recorded ncu traffic figure
    applies only while they are unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "blackwell_tensor_core_fp16_gb300", "csrc")
    for f in sources:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0) or 0), "measured"
    except Exception:
        return FALLBACK_PEAK_TFLOPS, 1700.0, "fallback"


# A timed region at least this long runs at the power-capped clock, like the driver's sustained
# cuBLAS loop; a shorter one is compared with the burst figure.
SUSTAINED_REGION_MS = 1000.0


def roofline_peak(peak_burst: float, peak_sustained: float, timed_ms: float):
    """The tensor peak a kernel timed over `timed_ms` of back-to-back launches is measured
    against: the sustained figure for a long region (when one was measured), else the burst."""
    if peak_sustained and timed_ms >= SUSTAINED_REGION_MS:
        return peak_sustained, "bf16_tflops_sustained"
    return peak_burst, "bf16_tflops (burst)"


def measured_hbm_gbs() -> float:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"])
    except Exception:
        return 6800.0


def recorded_traffic(variant_name: str, file="ncu_traffic.json", sources=GEMM_KERNEL_SOURCES):
    """DRAM bytes per launch (or per step or call, as the file says) from a committed ncu
    summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", file)
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_src_sha256") != kernel_source_hash(sources):
        return None
    return d.get("per_launch_dram_bytes", {}).get(variant_name)


_UNIT = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
         "nsecond": 1e-9, "usecond": 1e-6, "msecond": 1e-3, "second": 1.0,
         "ns": 1e-9, "us": 1e-6, "ms": 1e-3, "s": 1.0}


def parse_ncu_csv(path):
    """Per captured launch (in capture order): kernel name and {metric: value in bytes or
    seconds} from an `ncu --csv --log-file` log (lines that are not CSV rows are skipped)."""
    import csv
    lines = [ln for ln in open(path) if ln.startswith('"')]
    launches = {}
    for row in csv.DictReader(lines):
        key = row["ID"]
        d = launches.setdefault(key, {"kernel": row["Kernel Name"], "metrics": {}})
        val = float(row["Metric Value"].replace(",", ""))
        d["metrics"][row["Metric Name"]] = val * _UNIT.get(row.get("Metric Unit", ""), 1.0)
    return [launches[k] for k in sorted(launches, key=int)]


def record_traffic(csv_path, command=""):
    """profiles/ncu_traffic.json from the capture of one step's two launches (8192^3, then the
    MLP shape), tagged with the hash of the kernel sources it describes."""
    launches = parse_ncu_csv(csv_path)
    if len(launches) != len(WORKLOADS):
        raise SystemExit(f"expected {len(WORKLOADS)} launches in {csv_path}, found {len(launches)}")
    by_w, total = {}, 0.0
    for name, l in zip(WORKLOADS, launches):
        m = l["metrics"]
        rd, wr = m["dram__bytes_read.sum"], m["dram__bytes_write.sum"]
        by_w[name] = {"kernel": l["kernel"], "dram_read_bytes": int(rd),
                      "dram_write_bytes": int(wr), "dram_bytes": int(rd + wr),
                      "duration_us": m.get("gpu__time_duration.sum", 0.0) * 1e6}
        total += rd + wr
    out = {"kernel_src_sha256": kernel_source_hash(),
           "source": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,"
                     "gpu__time_duration.sum --clock-control none -k regex:gemm_ws, one launch per "
                     "workload, written by bench.py --record-traffic",
           "command": command,
           "per_launch_dram_bytes_by_workload": {k: v["dram_bytes"] for k, v in by_w.items()},
           "launches": by_w,
           "per_launch_dram_bytes": {"ws_pair": int(total)},
           "per_launch_note": "ws_pair entry is the sum over the two launches of one bench step "
                              "(the unit 'achieved' uses)"}
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=2)
        f.write("\n")
    print(json.dumps(out))
    return 0


def _write_traffic(file, out):
    path = os.path.join(ROOT, "profiles", file)
    with open(path, "w") as f:
        json.dump(out, f, indent=2)
        f.write("\n")
    print(json.dumps(out))
    return 0


def _launch_bytes(l):
    m = l["metrics"]
    rd, wr = m["dram__bytes_read.sum"], m["dram__bytes_write.sum"]
    return {"kernel": l["kernel"], "dram_read_bytes": int(rd), "dram_write_bytes": int(wr),
            "dram_bytes": int(rd + wr), "duration_us": m.get("gpu__time_duration.sum", 0.0) * 1e6}


def record_traffic_mx(csv_path, command=""):
    """profiles/ncu_traffic_mx.json from the capture of the block-scaled FP8 step's two launches
    (8192^3, then the MLP shape), tagged with the hash of the kernel sources."""
    launches = parse_ncu_csv(csv_path)
    if len(launches) != len(MX_STEP):
        raise SystemExit(f"expected {len(MX_STEP)} launches in {csv_path}, found {len(launches)}")
    by_w = {name: _launch_bytes(l) for name, l in zip(MX_STEP, launches)}
    return _write_traffic("ncu_traffic_mx.json", {
        "kernel_src_sha256": kernel_source_hash(),
        "source": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,"
                  "gpu__time_duration.sum --clock-control none, the block-scaled FP8 step's two "
                  "launches, written by bench.py --record-traffic-mx",
        "command": command, "launches": by_w,
        "per_launch_dram_bytes": {"mx_step": sum(v["dram_bytes"] for v in by_w.values())},
        "per_launch_note": "mx_step is the sum over the two launches of one step (the unit the "
                           "leg's 'achieved' uses)"})


def record_traffic_gdn(csv_path, command=""):
    """profiles/ncu_traffic_gdn.json from the capture of one Gated Delta Net call of the roofline
    scenario (its chunk list, prepare and scan launches), tagged with the hash of the Gated Delta
    Net kernel sources."""
    launches = parse_ncu_csv(csv_path)
    if not 2 <= len(launches) <= 3:
        raise SystemExit(f"expected the 2 or 3 launches of one call in {csv_path}, found "
                         f"{len(launches)}")
    ls = [_launch_bytes(l) for l in launches]
    return _write_traffic("ncu_traffic_gdn.json", {
        "kernel_src_sha256": kernel_source_hash(GDN_KERNEL_SOURCES),
        "scenario": GDN_ROOFLINE_SCENARIO,
        "source": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,"
                  "gpu__time_duration.sum --clock-control none, the launches of one call, "
                  "written by bench.py --record-traffic-gdn",
        "command": command, "launches": ls,
        "per_launch_dram_bytes": {GDN_ROOFLINE_SCENARIO: sum(v["dram_bytes"] for v in ls)},
        "per_launch_note": "the entry is the sum over the launches of one call (the unit the "
                           "leg's 'achieved' uses)"})


# ---- clocks --------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid: str | None):
        self.proc = None
        self.uuid = device_uuid
        self.out_path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.fh = open(self.out_path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.out_path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 8:
                rows.append(parts)
        os.unlink(self.out_path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        pw = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w": statistics.median(pw) if pw else None,
                "samples": len(rows)}


# ---- CPU oracle sample ----------------------------------------------------------------------

def host_cpu() -> dict:
    """The host's CPU model (lscpu, else /proc/cpuinfo) and logical CPU count."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() == "Model name":
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            for ln in open("/proc/cpuinfo"):
                if ln.lower().startswith(("model name", "cpu model")):
                    model = ln.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return {"cpu_model": model, "nproc": os.cpu_count()}


def oracle_sample(inputs, seconds_target, rng_seed=0):
    """Time the oracle on random output elements of each GEMM, sized to ~seconds_target.
    Returns (flops, seconds, description)."""
    import numpy as np
    import oracle

    rng = np.random.default_rng(rng_seed)
    total_flops = 0.0
    total_s = 0.0
    desc = []
    per = seconds_target / len(inputs)
    for name, (A, B) in inputs.items():
        M, K = A.shape
        N = B.shape[0]
        # calibrate on a small batch, then size the timed sample
        n0 = 256
        r = rng.integers(0, M, n0)
        c = rng.integers(0, N, n0)
        t = time.perf_counter()
        oracle.gemm_f64_sampled(A, B, r, c)
        dt = max(time.perf_counter() - t, 1e-6)
        count = max(64, int(n0 * per / dt))
        r = rng.integers(0, M, count)
        c = rng.integers(0, N, count)
        t = time.perf_counter()
        oracle.gemm_f64_sampled(A, B, r, c)
        dt = time.perf_counter() - t
        total_flops += 2.0 * K * count
        total_s += dt
        desc.append(f"{count} random output elements of {name} ({M}x{N}x{K})")
    return total_flops, total_s, "; ".join(desc)


def host_inputs(names=WORKLOADS):
    from blackwell_tensor_core_fp16_gb300.workloads import WORKLOADS as W, workload_inputs
    return {n: workload_inputs(W[n]) for n in names}


# ---- reference arm: the oracle, timed on host cores -------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from blackwell_tensor_core_fp16_gb300.workloads import WORKLOADS as W

    oracle.build()
    names = step_workloads(args)
    inputs = host_inputs(names)
    per_step = min(0.25, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(inputs, per_step, rng_seed=1)
    flops = secs = 0.0
    desc = ""
    for s in range(args.steps):
        f, t, desc = oracle_sample(inputs, per_step, rng_seed=100 + s)
        flops += f
        secs += t
    value = flops / secs / 1e12
    cfg = {"workload": "+".join(names),
           "shapes": [[W[n].M, W[n].N, W[n].K] for n in names]}
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "host": host_cpu(),
                         "kind": "oracle",
                         "sample": f"per step, {desc} (binary64 dot products)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---- block-scaled FP8 leg ---------------------------------------------------------------------

MX_STEP = ("mx_square_8192", "mx_mlp_up_16384x14336x4096")
GDN_ROOFLINE_SCENARIO = "packed_n20_t8192_h8_hv16_gva_state"   # the longest call
FP8_OVER_16BIT = 2.0   # nominal dense rate ratio of the FP8 and 16-bit tensor paths (4.5 / 2.25 PF)


def mx_inputs_on_device(g, w, dev):
    import torch
    from blackwell_tensor_core_fp16_gb300.workloads import mx_workload_inputs
    A, B, SA, SB = mx_workload_inputs(w)
    Ad, Bd = A.to(dev), B.to(dev)
    sfa = g.pack_scales(SA.to(dev))
    sfb = g.pack_scales(SB.to(dev))
    D = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    return Ad, Bd, sfa, sfb, D


def mx_launch(g, w, t, variant, stream):
    Ad, Bd, sfa, sfb, D = t
    rc = g.gemm_mxf8_nt(Ad.data_ptr(), Bd.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                        D.data_ptr(), w.M, w.N, w.K, g.FP8_FORMATS[w.fmt_a],
                        g.FP8_FORMATS[w.fmt_b], g.DTYPES["f16"], 0, 0, variant, 0, 0,
                        stream.cuda_stream)
    if rc != g.OK:
        raise g.GemmError(rc, g.gemm_f16_last_error())


def run_fused_leg(args, g, dev, stream, peak16, uuid):
    """The fused linear layer, act(A B^T + bias) with bf16 A, B, bias and D and the exact GELU,
    on the headline step's two shapes (the MLP up-projection with its bias and activation is the
    case the fused epilogue is for), inputs resident, back-to-back launches timed with CUDA events
    at the region's two ends, then each shape alone; cuBLAS on the same buffers for context."""
    import torch
    from blackwell_tensor_core_fp16_gb300.workloads import WORKLOADS as W, workload_inputs
    work = []
    for name in WORKLOADS:
        w = W[name]
        A, B = workload_inputs(w)
        gen = torch.Generator(device="cpu")
        gen.manual_seed(1000 + w.seed)
        bias = (0.1 * torch.randn(w.N, generator=gen)).to(torch.bfloat16)
        Ad, Bd, bd = (t.to(torch.bfloat16).to(dev) for t in (A, B, bias))
        D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
        work.append((w, Ad, Bd, bd, D))
    del A, B

    def launch(item):
        w, Ad, Bd, bd, D = item
        rc = g.gemm_f16_nt_fused(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), w.M, w.N, w.K,
                                 g.DTYPES["bf16"], bd.data_ptr(), g.ACTIVATIONS[args.fused_act],
                                 0, 0, 0, stream.cuda_stream)
        if rc != g.OK:
            raise g.GemmError(rc, g.gemm_f16_last_error())

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            for item in work:
                launch(item)
    torch.cuda.synchronize()
    K = args.fused_steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for _ in range(K):
            for item in work:
                launch(item)
        ev[1].record(stream)
    torch.cuda.synchronize()
    clk = sampler.stop()
    g.check_status(stream)
    total = ev[0].elapsed_time(ev[1])
    flops = sum(item[0].flops for item in work)
    per = {}
    for item in work:
        w = item[0]
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s0.record(stream)
            for _ in range(K):
                launch(item)
            s1.record(stream)
        torch.cuda.synchronize()
        ms = s0.elapsed_time(s1) / K
        per[w.name] = {"M": w.M, "N": w.N, "K": w.K, "ms_per_launch": ms,
                       "tflops": w.flops / (ms * 1e-3) / 1e12,
                       "timing": "this shape alone, as many launches, after the timed region"}
    g.check_status(stream)
    achieved = K * flops / (total * 1e-3) / 1e12
    # cuBLAS for context: one cuBLASLt call with its bias + GELU epilogue (its GELU is the tanh
    # form) where torch offers it, else addmm followed by a separate GELU
    cublas = None
    try:
        if hasattr(torch, "_addmm_activation"):
            def ref_step():
                for w, Ad, Bd, bd, D in work:
                    torch._addmm_activation(bd, Ad, Bd.t(), use_gelu=True, out=D)
            how = "torch._addmm_activation (cuBLASLt bias + GELU epilogue, tanh GELU)"
        else:
            def ref_step():
                for w, Ad, Bd, bd, D in work:
                    torch.nn.functional.gelu(torch.addmm(bd, Ad, Bd.t()), out=D)
            how = "torch.addmm then torch.nn.functional.gelu (two kernels)"
        with torch.cuda.stream(stream):
            for _ in range(3):
                ref_step()
        torch.cuda.synchronize()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            c0.record(stream)
            for _ in range(K):
                ref_step()
            c1.record(stream)
        torch.cuda.synchronize()
        cv = K * flops / (c0.elapsed_time(c1) * 1e-3) / 1e12
        cublas = {"value": cv, "unit": "TFLOP/s", "steps": K, "call": how,
                  "ours_over_cublas": achieved / cv}
    except Exception as e:   # context only
        cublas = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
    return {"metric": "fused linear layer TFLOP/s: bf16 act(A B^T + bias), bf16 out",
            "activation": args.fused_act,
            "value": achieved, "unit": "TFLOP/s", "steps": K, "per_workload": per,
            "clocks": clk, "cublas_same_step": cublas,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak16,
                         "unit": "TFLOP/s", "frac": achieved / peak16, "traffic": None,
                         "peak_source": "measured bf16_tflops (burst): the leg's region is "
                                        "well under a second"},
            "gpu_launches": K * len(work) * 2 + max(3, args.warmup) * len(work)}


def run_mx_leg(args, g, dev, stream, num_sms, peak16, uuid):
    """The block-scaled FP8 GEMM (E4M3 x E4M3, E8M0 scales per 32 K elements, fp16 out) on the
    same two shapes, inputs resident, back-to-back launches timed with CUDA events."""
    import torch
    from blackwell_tensor_core_fp16_gb300.workloads import MX_WORKLOADS
    work = []
    for n in MX_STEP:
        w = MX_WORKLOADS[n]
        v = args.mx_variant or g.gemm_mxf8_choose_variant(w.M, w.N, w.K, num_sms)
        work.append((w, mx_inputs_on_device(g, w, dev), v))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            for w, t, v in work:
                mx_launch(g, w, t, v, stream)
    torch.cuda.synchronize()
    K = args.mx_steps
    # events at the region's two ends only, as in the headline step (and as cuBLAS's below);
    # the per-shape split from separate loops after it
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for _ in range(K):
            for w, t, v in work:
                mx_launch(g, w, t, v, stream)
        ev[1].record(stream)
    torch.cuda.synchronize()
    clk = sampler.stop()
    g.check_status(stream)
    total = ev[0].elapsed_time(ev[1])
    flops = sum(w.flops for w, _, _ in work)
    per = {}
    for w, t, v in work:
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s0.record(stream)
            for _ in range(K):
                mx_launch(g, w, t, v, stream)
            s1.record(stream)
        torch.cuda.synchronize()
        ms = s0.elapsed_time(s1) / K
        per[w.name] = {"M": w.M, "N": w.N, "K": w.K, "variant": v, "ms_per_launch": ms,
                       "tflops": w.flops / (ms * 1e-3) / 1e12,
                       "timing": "this shape alone, as many launches, after the timed region"}
    g.check_status(stream)
    # both shapes run one kernel instance when their variants agree: the region's time is its
    same_kernel = len({v for _, _, v in work}) == 1
    achieved = (K * flops / (total * 1e-3) / 1e12 if same_kernel else
                K * flops / (K * sum(p["ms_per_launch"] for p in per.values()) * 1e-3) / 1e12)
    peak8 = peak16 * FP8_OVER_16BIT

    # cuBLAS's MXFP8 GEMM (torch._scaled_mm) on the same packed inputs, for the same number of
    # steps right after ours: context only.  The tiled scale layout is the one cuBLAS reads, so
    # the same buffers serve both.
    cublas = None
    try:
        e4, e8 = torch.float8_e4m3fn, torch.float8_e8m0fnu
        ops = [(w, t[0].view(e4), t[1].view(e4).t(), t[2].view(e8), t[3].view(e8), t[4])
               for w, t, _ in work]

        def cublas_step():
            for w, a8, b8t, sa, sb, D in ops:
                torch._scaled_mm(a8, b8t, scale_a=sa, scale_b=sb, out_dtype=torch.float16,
                                 out=D)

        with torch.cuda.stream(stream):
            for _ in range(3):
                cublas_step()
        torch.cuda.synchronize()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            c0.record(stream)
            for _ in range(K):
                cublas_step()
            c1.record(stream)
        torch.cuda.synchronize()
        cv = K * flops / (c0.elapsed_time(c1) * 1e-3) / 1e12
        cublas = {"value": cv, "unit": "TFLOP/s", "steps": K,
                  "ours_over_cublas": (K * flops / (total * 1e-3) / 1e12) / cv}
    except Exception as e:  # an older torch without the MX path: report why, not a number
        cublas = {"unavailable": repr(e)[:200]}
    return {"metric": "block-scaled FP8 (MX E4M3, E8M0 per 32) GEMM TFLOP/s, fp16 out",
            "value": K * flops / (total * 1e-3) / 1e12, "unit": "TFLOP/s", "steps": K,
            "per_workload": per, "clocks": clk, "cublas_mxfp8_same_step": cublas,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak8,
                         "unit": "TFLOP/s", "frac": achieved / peak8,
                         "traffic": recorded_traffic("mx_step", "ncu_traffic_mx.json"),
                         "traffic_unit": "DRAM bytes per step (ncu, both launches)",
                         "peak_source": "measured bf16_tflops x 2 (nominal FP8 / 16-bit dense "
                                        "rate ratio, 4.5 / 2.25 PFLOP/s)"},
            "gpu_launches": 2 * K * len(work)}


# ---- Gated Delta Net prefill leg -------------------------------------------------------------------

# The page's own CUDA-event times of its public callable on an H20-3e (sm_90a), for context only:
# another machine, another implementation ("TIRx" (zixuwang.me), "公开版本复测：六个场景").
GDN_PAGE_H20_MS = {
    "single_t512_h8_mha_zero": 0.102550, "single_t1024_h8_mha_state": 0.157430,
    "single_t1024_h8_hv16_gva_state": 0.143251, "single_t4096_h16_mha_zero": 0.263054,
    "packed_n10_t4096_h8_mha_state": 0.173384, "packed_n20_t8192_h8_hv16_gva_state": 0.520107,
}


def run_gdn_leg(args, g, dev, stream, peak16, hbm_peak):
    """Every scenario of the page: inputs resident, the workspace allocated once, CUDA events
    around back-to-back calls (at least `gdn_reps` of them and `gdn_min_ms` of time) after about
    50 ms of warm-up calls."""
    import torch
    from blackwell_tensor_core_fp16_gb300.workloads import GDN_ORDER, GDN_WORKLOADS, \
        gdn_workload_inputs
    if g.gdn_set_scan_kernel(g.GDN_SCAN_KERNELS[args.gdn_scan]) != g.GDN_OK:
        raise g.GemmError(1, g.gdn_last_error())
    out = {}
    names = [n for n in args.gdn_scenarios.split(",") if n] or GDN_ORDER
    for name in names:
        w = GDN_WORKLOADS[name]
        inp = gdn_workload_inputs(w)
        q, k, v = (inp[x].to(dev) for x in ("q", "k", "v"))
        a, b, cu = inp["alpha"].to(dev), inp["beta"].to(dev), inp["cu_seqlens"].to(dev)
        s0 = None if inp["initial_state"] is None else inp["initial_state"].to(dev)
        n = cu.numel() - 1
        o = torch.empty((w.T, w.h_v, w.dv), dtype=torch.bfloat16, device=dev)
        sf = torch.empty((n, w.h_v, w.dv, w.dk), dtype=torch.float32, device=dev) if w.state \
            else None
        need = g.gdn_prefill_workspace_bytes(w.T, n, w.h_v)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

        def call():
            rc = g.gdn_prefill(q.data_ptr(), k.data_ptr(), v.data_ptr(), a.data_ptr(),
                               b.data_ptr(), cu.data_ptr(), n, w.T, w.h_qk, w.h_v, w.dk, w.scale,
                               0 if s0 is None else s0.data_ptr(), o.data_ptr(),
                               0 if sf is None else sf.data_ptr(), ws.data_ptr(), need,
                               stream.cuda_stream)
            if rc != g.GDN_OK:
                raise g.GemmError(rc, g.gdn_last_error())

        # warm up for about 50 ms of calls (at least 3): the leg follows the power-capped GEMM
        # legs, and the SM clock takes tens of milliseconds to climb back once they stop; then
        # time at least `gdn_reps` calls and at least about 5 ms of them
        t_w = time.perf_counter()
        n_w = 0
        while n_w < 3 or time.perf_counter() - t_w < args.gdn_warm_ms * 1e-3:
            with torch.cuda.stream(stream):
                for _ in range(8):
                    call()
            torch.cuda.synchronize()
            n_w += 8
        per_call_s = (time.perf_counter() - t_w) / n_w
        reps = max(args.gdn_reps, int(math.ceil(args.gdn_min_ms * 1e-3 / per_call_s)))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                call()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / max(reps, 1)
        out[name] = {"ms": ms, "reps": reps, "tokens_per_s": w.T / (ms * 1e-3),
                     "recurrence_tflops": w.flops / (ms * 1e-3) / 1e12,
                     "hbm_gbs_algorithmic": w.min_bytes / (ms * 1e-3) / 1e9,
                     "page_h20_ms_context": GDN_PAGE_H20_MS.get(name)}
    # Roofline of the longest scenario: neither the tensor pipe nor HBM is the limit (the scan
    # is a chain of dependent 64-token chunk steps), and both fractions say so.
    big = max(out, key=lambda n: out[n]["ms"])
    tf, gbs = out[big]["recurrence_tflops"], out[big]["hbm_gbs_algorithmic"]
    traffic = (recorded_traffic(big, "ncu_traffic_gdn.json", GDN_KERNEL_SOURCES)
               if big == GDN_ROOFLINE_SCENARIO else None)
    roofline = {"scenario": big, "bound": "tensor", "achieved": tf, "peak": peak16,
                "unit": "TFLOP/s", "frac": tf / peak16, "traffic": traffic,
                "traffic_unit": "DRAM bytes per call (ncu, all launches of one call)",
                "hbm_achieved_gbs": gbs, "hbm_peak_gbs": hbm_peak, "hbm_frac": gbs / hbm_peak,
                "note": "achieved = the token recurrence's 6*T*h_v*dk*dv flops / call time against "
                        "the measured dense bf16 peak; the call is latency-bound: the scan by "
                        "its chain of dependent 64-token chunk steps (about 1.7 us each on the "
                        "tcgen05 scan), the prepare kernel (about a third of the call) by its "
                        "per-chunk chain of products, inverse and stores"}
    g.gdn_set_scan_kernel(g.GDN_SCAN_KERNELS["auto"])
    return {"metric": "Gated Delta Net prefill: ms per call (bf16 q/k/v, head dim 128)",
            "unit": "ms", "higher_is_better": False, "scan_kernel": args.gdn_scan,
            "min_reps": args.gdn_reps,
            "min_timed_ms": args.gdn_min_ms,
            "scenarios": out,
            "roofline": roofline,
            "gpu_launches_per_call": 3,
            "note": "recurrence_tflops counts 6*T*h_v*dk*dv (prediction, rank-one update, "
                    "output) per call; page_h20_ms_context is the page's own time on another "
                    "machine"}


# ---- the other configs: single tile, 2048^3, 3000x5000x1000 ----------------------------------

CONFIGS = ("single_tile_128x128x64", "square_2048", "ragged_3000x5000x1000")


def run_config_leg(args, g, dev, stream, num_sms, peak_burst, hbm_peak, uuid):
    """The three smaller configs on the automatic variant, inputs resident: warm (back-to-back
    launches between two CUDA events, about `config_ms` of work after warm-up) and cold (a 512 MiB
    scratch write before each launch, events around the launch alone), with the clocks sampled
    over the warm loops."""
    import torch
    from blackwell_tensor_core_fp16_gb300.workloads import WORKLOADS as W, workload_inputs
    scratch = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    out = {}
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.2)
    for name in CONFIGS:
        w = W[name]
        A, B = workload_inputs(w)
        Ad, Bd = A.to(dev), B.to(dev)
        D = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
        variant = g.gemm_f16_choose_variant(w.M, w.N, w.K, num_sms)

        def launch():
            rc = g.gemm_f16_nt(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), w.M, w.N, w.K,
                               stream.cuda_stream)
            if rc != g.OK:
                raise g.GemmError(rc, g.gemm_f16_last_error())

        with torch.cuda.stream(stream):
            for _ in range(20):
                launch()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(20):
                launch()
        torch.cuda.synchronize()
        per = (time.perf_counter() - t0) / 20
        reps = max(100, min(200000, int(args.config_ms * 1e-3 / max(per, 1e-6))))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                launch()
            e1.record(stream)
        torch.cuda.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / reps
        # cold L2: 512 MiB written before each launch (outside the events)
        cold_reps = 50
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(cold_reps)]
        with torch.cuda.stream(stream):
            for i in range(cold_reps):
                scratch.fill_(i & 0xFF)
                ev[i][0].record(stream)
                launch()
                ev[i][1].record(stream)
        torch.cuda.synchronize()
        g.check_status(stream)
        cold_us = 1e3 * sum(a.elapsed_time(b) for a, b in ev) / cold_reps
        tf = w.flops / (us * 1e-6) / 1e12
        # the same launches recorded in a CUDA graph (50 per graph) and replayed: the device-side
        # time per launch without the host's per-call cost
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(50):
                launch()
        g_replays = max(2, reps // 50)
        with torch.cuda.stream(stream):
            graph.replay()
            ge0, ge1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ge0.record(stream)
            for _ in range(g_replays):
                graph.replay()
            ge1.record(stream)
        torch.cuda.synchronize()
        g.check_status(stream)
        graph_us = 1e3 * ge0.elapsed_time(ge1) / (50 * g_replays)
        del graph
        # cuBLAS (torch.mm) on the same resident inputs, for context: 50 calls recorded in a
        # CUDA graph and replayed, so that the host's dispatch rate does not set the figure
        cublas_us = None
        if args.cublas_steps != 0:
            with torch.cuda.stream(stream):
                for _ in range(20):
                    torch.mm(Ad, Bd.t(), out=D)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(50):
                    torch.mm(Ad, Bd.t(), out=D)
            replays = max(2, reps // 50)
            with torch.cuda.stream(stream):
                graph.replay()
                c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c0.record(stream)
                for _ in range(replays):
                    graph.replay()
                c1.record(stream)
            torch.cuda.synchronize()
            cublas_us = 1e3 * c0.elapsed_time(c1) / (50 * replays)
            del graph
        out[name] = {"M": w.M, "N": w.N, "K": w.K, "variant": variant, "launches": reps,
                     "us_per_launch_graph": graph_us,
                     "tflops_graph": w.flops / (graph_us * 1e-6) / 1e12,
                     "cublas_us_per_launch_graph_context": cublas_us,
                     "us_per_launch": us, "tflops": tf, "frac_of_burst": tf / peak_burst,
                     "hbm_gbs_algorithmic": w.min_bytes / (us * 1e-6) / 1e9,
                     "hbm_frac": w.min_bytes / (us * 1e-6) / 1e9 / hbm_peak,
                     "cold_l2_us_per_launch": cold_us,
                     "cold_l2_tflops": w.flops / (cold_us * 1e-6) / 1e12}
        del Ad, Bd, D
    clk = sampler.stop()
    del scratch
    return {"metric": "fp16 GEMM per config, automatic variant (gemm_f16_nt)",
            "timing": "warm: back-to-back launches between two CUDA events on the launching "
                      "stream; graph: the same launches recorded 50 to a CUDA graph and "
                      "replayed (no per-call host cost); cold: a 512 MiB scratch write before "
                      "each launch, events around the launch alone",
            "configs": out, "clocks": clk,
            "gpu_launches": sum(v["launches"] + 50 + 50 * (max(2, v["launches"] // 50) + 1)
                                for v in out.values())}


def run_sustained_leg(args, g, stream, work, launch, flops_step, peak_burst, peak_sus, num_sms,
                      uuid):
    """The headline step back to back for at least `sustained_ms` (the power-capped regime the
    sustained peak was measured in), timed with CUDA events on the launching stream at the
    region's two ends, with its own clock record, and each shape alone for as many launches for
    the per-shape split; then cuBLAS (torch.mm) on the same resident inputs the same way, for
    context."""
    import torch
    step_t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(3):
            for item in work:
                launch(item)
    torch.cuda.synchronize()
    step_ms = 1e3 * (time.perf_counter() - step_t0) / 3
    steps = max(10, int(math.ceil(args.sustained_ms / max(step_ms, 1e-3))))

    def timed(fn):
        # the step back to back with events at the two ends only (as the headline region), then
        # each shape alone for as many launches, for the per-shape split
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        sampler = ClockSampler(uuid)
        sampler.start()
        time.sleep(0.2)
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for _ in range(steps):
                for item in work:
                    fn(item)
            ev[1].record(stream)
        torch.cuda.synchronize()
        clk = sampler.stop()
        ms = ev[0].elapsed_time(ev[1])
        per = {}
        for item in work:
            w = item[0]
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                s0.record(stream)
                for _ in range(steps):
                    fn(item)
                s1.record(stream)
            torch.cuda.synchronize()
            m = s0.elapsed_time(s1) / steps
            per[w.name] = {"ms_per_launch": m, "tflops": w.flops / (m * 1e-3) / 1e12}
        tf = steps * flops_step / (ms * 1e-3) / 1e12
        return tf, ms, per, clk

    tf, ms, per, clk = timed(launch)
    g.check_status(stream)
    pj = lambda t, c: (c["power_w"] / (t * 1e12) * 1e12) if c and c.get("power_w") else None
    res = {"value": tf, "unit": "TFLOP/s", "steps": steps, "timed_ms": ms,
           "per_workload": per, "peak_sustained": peak_sus,
           "frac_of_sustained": tf / peak_sus if peak_sus else None,
           "frac_of_burst": tf / peak_burst, "clocks": clk, "gpu_launches": 2 * steps * len(work),
           "pj_per_flop": pj(tf, clk)}
    if clk and clk.get("sm_mhz"):
        cpk = num_sms * FLOP_PER_CLK_PER_SM * clk["sm_mhz"] * 1e6 / 1e12
        res["clock_peak_tflops"] = cpk
        res["frac_of_clock_peak"] = tf / cpk
    if args.cublas_steps != 0:
        def mm(item):
            _w, Ad, Bd, D, _v = item
            torch.mm(Ad, Bd.t(), out=D)
        with torch.cuda.stream(stream):
            for _ in range(3):
                for item in work:
                    mm(item)
        torch.cuda.synchronize()
        ctf, cms, cper, cclk = timed(mm)
        res["cublas_same_step"] = {"value": ctf, "timed_ms": cms, "per_workload": cper,
                                   "clocks": cclk, "ours_over_cublas": tf / ctf,
                                   "pj_per_flop": pj(ctf, cclk)}
    return res


def merge_config_processes(args, first):
    """Runs the per_config leg in args.config_processes - 1 fresh processes as well; per config,
    each time figure becomes the median of the per-process means (all of them listed)."""
    runs = [first]
    cmd = [sys.executable, os.path.abspath(__file__), "--config-only", "--config-ms",
           str(args.config_ms), "--cublas-steps", str(args.cublas_steps)]
    failed = []
    for _ in range(args.config_processes - 1):
        try:
            out = subprocess.run(cmd, check=True, capture_output=True, text=True,
                                 timeout=600).stdout
            runs.append(json.loads([ln for ln in out.splitlines() if ln.startswith("{")][-1]))
        except Exception as e:   # the leg is extra: keep the processes that ran
            failed.append(f"{type(e).__name__}: {e}"[:200])
    merged = dict(first)
    merged["processes"] = len(runs)
    if failed:
        merged["failed_processes"] = failed
    merged["timing"] = (first["timing"] + "; each figure is the median over " + str(len(runs)) +
                        " processes of the per-process means (listed per process)")
    cfgs = {}
    for name, c in first["configs"].items():
        d = dict(c)
        flops = 2.0 * c["M"] * c["N"] * c["K"]
        for key in ("us_per_launch", "us_per_launch_graph", "cold_l2_us_per_launch",
                    "cublas_us_per_launch_graph_context"):
            vals = [r["configs"][name][key] for r in runs if r["configs"][name].get(key)]
            if not vals:
                continue
            d[key] = statistics.median(vals)
            d[key + "_per_process"] = vals
        d["tflops"] = flops / (d["us_per_launch"] * 1e-6) / 1e12
        d["tflops_graph"] = flops / (d["us_per_launch_graph"] * 1e-6) / 1e12
        d["cold_l2_tflops"] = flops / (d["cold_l2_us_per_launch"] * 1e-6) / 1e12
        d["frac_of_burst"] = d["tflops"] * c["frac_of_burst"] / c["tflops"]
        bytes_ = c["hbm_gbs_algorithmic"] * c["us_per_launch"] * 1e-6 * 1e9
        d["hbm_gbs_algorithmic"] = bytes_ / (d["us_per_launch"] * 1e-6) / 1e9
        d["hbm_frac"] = d["hbm_gbs_algorithmic"] * c["hbm_frac"] / c["hbm_gbs_algorithmic"]
        cfgs[name] = d
    merged["configs"] = cfgs
    merged["gpu_launches"] = sum(r["gpu_launches"] for r in runs)
    return merged


def run_config_only(args):
    """--config-only: the per_config leg alone, printed as one JSON line."""
    import torch
    import blackwell_tensor_core_fp16_gb300 as g
    g.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    props = torch.cuda.get_device_properties(dev)
    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    peak_burst, _peak_sus, _src = measured_peaks()
    leg = run_config_leg(args, g, dev, stream, props.multi_processor_count, peak_burst,
                         measured_hbm_gbs(), uuid)
    print(json.dumps(leg), flush=True)
    return 0


# ---- our arm ---------------------------------------------------------------------------------

def run_ours(args):
    import torch
    import torch.distributed as dist

    import blackwell_tensor_core_fp16_gb300 as g
    from blackwell_tensor_core_fp16_gb300.workloads import WORKLOADS as W

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    if args.gdn_only:
        g.build()
        g.load()
        dev = torch.device("cuda", local)
        leg = run_gdn_leg(args, g, dev, torch.cuda.Stream(device=dev),
                          measured_peaks()[0], measured_hbm_gbs())
        print(json.dumps(leg), flush=True)
        return 0
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    g.build()
    g.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    props = torch.cuda.get_device_properties(dev)
    num_sms = props.multi_processor_count

    names = step_workloads(args)
    inputs = host_inputs(names)
    work = []
    for n in names:
        w = W[n]
        A, B = inputs[n]
        Ad, Bd = A.to(dev), B.to(dev)
        D = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
        variant = args.variant or g.gemm_f16_choose_variant(w.M, w.N, w.K, num_sms)
        work.append((w, Ad, Bd, D, variant))
    torch.cuda.synchronize()

    def launch(item):
        w, Ad, Bd, D, variant = item
        rc = g.gemm_f16_nt_variant(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), w.M, w.N, w.K, sh,
                                   variant)
        if rc != g.OK:
            raise g.GemmError(rc, g.gemm_f16_last_error())

    def barrier():
        if world > 1:
            dist.barrier()

    # warm-up
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for item in work:
                launch(item)
    torch.cuda.synchronize()
    g.check_status(stream)

    # Timed region: CUDA events on the launching stream.  When every launch of the step runs the
    # same kernel (both shapes take the CTA-pair kernel), only the region's two ends carry an
    # event: an event recorded between two launches keeps the second from overlapping the first
    # one's end (programmatic dependent launch), which measured 3% per step; the per-shape
    # split is then timed separately after the region.  Otherwise an event follows every launch.
    K = args.steps
    same_kernel = len({item[4] for item in work}) == 1
    events = [torch.cuda.Event(enable_timing=True)
              for _ in range(2 if same_kernel else len(work) * K + 1)]
    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass

    def timed_region():
        clocks = ClockSampler(uuid)
        clocks.start()
        time.sleep(0.3)
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            events[0].record(stream)
            e = 1
            for _ in range(K):
                for item in work:
                    launch(item)
                    if not same_kernel:
                        events[e].record(stream)
                        e += 1
            if same_kernel:
                events[1].record(stream)
        torch.cuda.synchronize()
        barrier()
        wall = time.perf_counter() - t0
        info = clocks.stop()
        g.check_status(stream)
        return wall, info

    wall_s, clock_info = timed_region()
    # A run whose clocks show a hardware or thermal slowdown, or SM clocks stuck far below their
    # maximum with no reason given (a clock lock left by someone), is measured once more; the
    # second run's numbers are reported, with the first run's clocks beside them.
    first_clocks = None
    if clocks_rejected(clock_info):
        first_clocks = clock_info
        wall_s, clock_info = timed_region()
        clock_info = dict(clock_info or {}, remeasured_after=first_clocks)

    total_ms = events[0].elapsed_time(events[-1])
    flops_step = sum(2.0 * w.M * w.N * w.K for (w, *_rest) in work)

    per = {}
    if same_kernel:
        # every launch in the region is the same kernel: its launch time is the region's
        kernel_ms_total = total_ms
        # per shape: the shape alone, K launches back to back, after the timed region
        for (w, Ad, Bd, D, variant) in work:
            item = (w, Ad, Bd, D, variant)
            with torch.cuda.stream(stream):
                for _ in range(2):
                    launch(item)
            torch.cuda.synchronize()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                s0.record(stream)
                for _ in range(K):
                    launch(item)
                s1.record(stream)
            torch.cuda.synchronize()
            mean_ms = s0.elapsed_time(s1) / K
            per[w.name] = {"M": w.M, "N": w.N, "K": w.K, "variant": variant,
                           "ms_per_launch": mean_ms,
                           "tflops": 2.0 * w.M * w.N * w.K / (mean_ms * 1e-3) / 1e12,
                           "timing": "this shape alone, K launches back to back, after the "
                                     "timed region"}
        g.check_status(stream)
    else:
        durs = [events[i].elapsed_time(events[i + 1]) for i in range(len(events) - 1)]
        kernel_ms_total = 0.0
        for j, (w, _, _, _, variant) in enumerate(work):
            ds = durs[j::len(work)]
            mean_ms = sum(ds) / len(ds)
            kernel_ms_total += sum(ds)
            per[w.name] = {"M": w.M, "N": w.N, "K": w.K, "variant": variant,
                           "ms_per_launch": mean_ms,
                           "tflops": 2.0 * w.M * w.N * w.K / (mean_ms * 1e-3) / 1e12}
    total_ms = max_over_ranks(total_ms, world, dev)
    value = whole_job_tflops(world, K, flops_step, total_ms)
    peak_burst, peak_sus, peak_src = measured_peaks()
    peak, peak_kind = roofline_peak(peak_burst, peak_sus, total_ms)
    achieved = K * flops_step / (kernel_ms_total * 1e-3) / 1e12
    for v in per.values():
        v["frac_of_peak"] = v["tflops"] / peak

    variant_names = {val: key for key, val in g.VARIANTS.items()}
    dom = max(work, key=lambda it: 2.0 * it[0].M * it[0].N * it[0].K)
    traffic = recorded_traffic(variant_names.get(dom[4], str(dom[4])))
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src} {peak_kind} (fp16 and bf16 share the kind::f16 "
                               f"tensor path at the same nominal rate); the timed region ran "
                               f"{total_ms:.0f} ms back to back",
                "peak_burst": peak_burst,
                "frac_of_burst": achieved / peak_burst,
                "peak_sustained": peak_sus,
                "frac_of_sustained": achieved / peak_sus if peak_sus else None,
                "kernel": "gemm_ws_kernel",
                "achieved_def": ("algorithmic 2*M*N*K over both launches of a step / the "
                                 "timed region's duration per step (every launch in it is this "
                                 "kernel; events only at the region's ends)") if same_kernel else
                                "algorithmic 2*M*N*K over both launches of a step / summed "
                                "CUDA-event launch durations"}

    # The peak implied by the clock seen during the timed region: 8192 dense fp16 FLOP per
    # clock per SM (one 256x256x16 cta_group::2 MMA per 128 cycles per CTA pair, measured with a
    # bare MMA stream) times the SMs times the median sampled SM clock.
    if clock_info and clock_info.get("sm_mhz"):
        cpk = num_sms * FLOP_PER_CLK_PER_SM * clock_info["sm_mhz"] * 1e6 / 1e12
        roofline["clock_peak_tflops"] = cpk
        roofline["frac_of_clock_peak"] = achieved / cpk

    # cuBLAS (torch.mm) on the same resident inputs and the same step, run back to back for the
    # same number of steps right after ours so both see the same power-capped clocks.  Context
    # only: it is a library kernel, not part of this path.
    cublas = None
    if args.cublas_steps != 0:
        csteps = K if args.cublas_steps < 0 else args.cublas_steps
        with torch.cuda.stream(stream):
            for _ in range(3):
                for (w, Ad, Bd, D, variant) in work:
                    torch.mm(Ad, Bd.t(), out=D)
        torch.cuda.synchronize()
        # timed the way our region is: events at the two ends, the per-shape split after
        cev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        csampler = ClockSampler(uuid)
        csampler.start()
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            cev[0].record(stream)
            for _ in range(csteps):
                for (w, Ad, Bd, D, variant) in work:
                    torch.mm(Ad, Bd.t(), out=D)
            cev[1].record(stream)
        torch.cuda.synchronize()
        cclk = csampler.stop()
        ctot = cev[0].elapsed_time(cev[1])
        cublas = {"value": csteps * flops_step / (ctot * 1e-3) / 1e12, "unit": "TFLOP/s",
                  "steps": csteps, "clocks": cclk, "per_workload": {}}
        for (w, Ad, Bd, D, variant) in work:
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                s0.record(stream)
                for _ in range(csteps):
                    torch.mm(Ad, Bd.t(), out=D)
                s1.record(stream)
            torch.cuda.synchronize()
            ms = s0.elapsed_time(s1) / csteps
            cublas["per_workload"][w.name] = {"ms_per_launch": ms,
                                              "tflops": 2.0 * w.M * w.N * w.K / (ms * 1e-3) / 1e12}
        cublas["ours_over_cublas"] = value / world / cublas["value"]

    sustained = None
    if args.sustained_ms > 0:
        sustained = run_sustained_leg(args, g, stream, work, launch, flops_step, peak_burst,
                                      peak_sus, num_sms, uuid)

    # End to end through the public API: every step copies its inputs from pinned host memory
    # to the device, runs the GEMMs with gemm(), and copies each result back to pinned host
    # memory.  Copies run on their own streams with two buffer slots, so the upload of step
    # i + 1 and the download of step i - 1 overlap the GEMMs of step i; the timed region runs
    # from before the first upload to after the last download.
    e2e_steps = 0 if args.skip_e2e else max(3, min(args.e2e_steps, K))
    e2e_value = None
    e2e_runs = []
    link_gbs = copy_roof = None
    h2d = d2h = 0
    if e2e_steps:
        s_up = torch.cuda.Stream(device=dev)
        s_down = torch.cuda.Stream(device=dev)
        slots = []
        for slot in range(2):
            items = []
            for (w, Ad, Bd, D, variant) in work:
                A, B = inputs[w.name]
                if slot == 0:
                    Ah, Bh = A.pin_memory(), B.pin_memory()
                else:
                    Ah, Bh = slots[0][len(items)][1], slots[0][len(items)][2]
                Dh = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()
                Ad2 = Ad if slot == 0 else torch.empty_like(Ad)
                Bd2 = Bd if slot == 0 else torch.empty_like(Bd)
                D2 = D if slot == 0 else torch.empty_like(D)
                ev = {k: torch.cuda.Event() for k in ("up", "mm", "down")}
                items.append((w, Ah, Bh, Dh, Ad2, Bd2, D2, variant, ev))
            slots.append(items)
        for (w, *_r) in work:
            h2d += 2 * (w.M * w.K + w.N * w.K)
            d2h += 2 * w.M * w.N
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)

        def e2e_region():
            barrier()
            torch.cuda.synchronize()
            ev0.record(stream)
            s_up.wait_event(ev0)
            s_down.wait_event(ev0)
            for i in range(e2e_steps):
                for (w, Ah, Bh, Dh, Ad2, Bd2, D2, variant, ev) in slots[i % 2]:
                    if i >= 2:
                        s_up.wait_event(ev["mm"])       # step i-2 finished reading this slot
                    with torch.cuda.stream(s_up):
                        Ad2.copy_(Ah, non_blocking=True)
                        Bd2.copy_(Bh, non_blocking=True)
                        ev["up"].record(s_up)
                    stream.wait_event(ev["up"])
                    if i >= 2:
                        stream.wait_event(ev["down"])   # step i-2's result has left this slot
                    g.gemm(Ad2, Bd2, out=D2, variant=variant, stream=stream)
                    ev["mm"].record(stream)
                    s_down.wait_event(ev["mm"])
                    with torch.cuda.stream(s_down):
                        Dh.copy_(D2, non_blocking=True)
                        ev["down"].record(s_down)
            stream.wait_stream(s_up)
            stream.wait_stream(s_down)
            ev1.record(stream)
            torch.cuda.synchronize()
            barrier()
            g.check_status(stream)
            return max_over_ranks(ev0.elapsed_time(ev1), world, dev)

        e2e_runs = [whole_job_tflops(world, e2e_steps, flops_step, e2e_region())
                    for _ in range(max(1, args.e2e_repeats))]
        e2e_value = statistics.median(e2e_runs)
        # The copy roofline of this leg: the measured rate of concurrent pinned-host copies in
        # both directions (256 MiB each way, the same streams), and the TFLOP/s a step could
        # reach if its copies ran at that rate and the GEMMs hid under them.
        nb = 256 << 20
        hsrc = torch.empty(nb, dtype=torch.uint8).pin_memory()
        hdst = torch.empty(nb, dtype=torch.uint8).pin_memory()
        dsrc = torch.empty(nb, dtype=torch.uint8, device=dev)
        ddst = torch.empty(nb, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        c0 = time.perf_counter()
        for _ in range(8):
            with torch.cuda.stream(s_up):
                ddst.copy_(hsrc, non_blocking=True)
            with torch.cuda.stream(s_down):
                hdst.copy_(dsrc, non_blocking=True)
        torch.cuda.synchronize()
        link_gbs = 8 * 2 * nb / (time.perf_counter() - c0) / 1e9
        copy_roof = flops_step / ((h2d + d2h) / (link_gbs * 1e9)) / 1e12
        del hsrc, hdst, dsrc, ddst

    config_leg = None
    if args.config_ms > 0 and not args.only:
        config_leg = run_config_leg(args, g, dev, stream, num_sms, peak_burst,
                                    measured_hbm_gbs(), uuid)
        if args.config_processes > 1 and world == 1:
            config_leg = merge_config_processes(args, config_leg)

    mx_leg = None
    if args.mx_steps > 0:
        mx_leg = run_mx_leg(args, g, dev, stream, num_sms, peak_burst, uuid)
    fused_leg = None
    if args.fused_steps > 0 and not args.only:
        fused_leg = run_fused_leg(args, g, dev, stream, peak_burst, uuid)
    gdn_leg = run_gdn_leg(args, g, dev, stream, peak_burst, measured_hbm_gbs()) \
        if args.gdn_reps > 0 else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        f, s, desc = oracle_sample(inputs, args.cpu_seconds)
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
               "host": host_cpu(),
               "kind": "oracle", "sample": desc + " (binary64 dot products, OpenMP)",
               "seconds": s}
        if config_leg is not None:
            # the three smaller configs through the oracle in full (every output element)
            from blackwell_tensor_core_fp16_gb300.workloads import WORKLOADS as W2
            per_cfg = {}
            for name in CONFIGS:
                w = W2[name]
                A, B = host_inputs((name,))[name]
                t = time.perf_counter()
                oracle.gemm_f64(A, B)
                dt = time.perf_counter() - t
                per_cfg[name] = {"seconds": dt, "gflops": w.flops / dt / 1e9,
                                 "gpu_over_cpu": dt / (config_leg["configs"][name]
                                                       ["us_per_launch"] * 1e-6)}
            cpu["per_config_full"] = per_cfg

    in_bytes = [2 * (w.M * w.K + w.N * w.K) for (w, *_r) in work]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {
            "workload": "+".join(names),
            "shapes": [[w.M, w.N, w.K] for (w, *_r) in work],
            "accumulate": "f32", "variant": [it[4] for it in work],
            "parallelism": f"replicas x{world}",
            "l2": f"no flush: every step's inputs ({', '.join(f'{b / 2**20:.0f} MiB' for b in in_bytes)}) "
                  f"exceed the {L2_BYTES / 1e6:.0f} MB L2",
            "device": props.name, "sms": num_sms,
        },
        "per_workload": per,
        "cublas_fp16_same_step": cublas,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "repeats": e2e_runs, "value_def": "median over the repeated timed regions",
                "copy_link_gbs_measured": link_gbs,
                "copy_roofline_tflops": copy_roof,
                "frac_of_copy_roofline": (e2e_value / world / copy_roof) if copy_roof else None,
                "path": "pinned host A,B -> device (copy stream), gemm() public API, "
                        "D -> pinned host (copy stream); two buffer slots, copies of "
                        "neighbouring steps overlap the GEMMs"},
        "gpu_launches": K * len(work),
        "per_config": config_leg,
        "sustained": sustained,
        "mx_fp8": mx_leg,
        "fused_bf16_gelu": fused_leg,
        "gdn_prefill": gdn_leg,
        "clocks": clock_info,
        "wall_s_timed_region": wall_s,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_sweep(args):
    """Per workload and variant: TFLOP/s and algorithmic HBM GB/s of back-to-back launches."""
    import torch

    import blackwell_tensor_core_fp16_gb300 as g
    from blackwell_tensor_core_fp16_gb300.workloads import ORDER, WORKLOADS as W, workload_inputs

    g.build()
    g.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if args.sweep_mx:
        return run_sweep_mx(args, g, dev, stream, sms)
    names = [n.strip() for n in args.sweep_workloads.split(",") if n.strip()] or ORDER
    scratch = (torch.empty(512 << 20, dtype=torch.uint8, device=dev) if args.sweep_cold_l2
               else None)
    for name in names:
        w = W[name]
        A, B = workload_inputs(w)
        Ad, Bd = A.to(dev), B.to(dev)
        D = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
        auto = g.gemm_f16_choose_variant(w.M, w.N, w.K, sms)
        variants = ([auto] if args.sweep_variants == "auto"
                    else [int(v) for v in args.sweep_variants.split(",")])
        for variant in variants:
            for use_ws in ((False,) if args.sweep_no_stream_k else (False, True)):
                # the stream-K leg turns the (default-off) tail on for its launches only
                g.gemm_f16_set_stream_k(1 if use_ws else 0)
                need = g.gemm_f16_workspace_bytes(w.M, w.N, w.K, variant) if use_ws else 0
                if use_ws and need == 0:
                    continue
                ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

                def launch():
                    rc = g.gemm_f16_nt_ex(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), w.M, w.N,
                                          w.K, variant, ws.data_ptr(), need, stream.cuda_stream)
                    if rc != g.OK:
                        raise g.GemmError(rc, g.gemm_f16_last_error())

                with torch.cuda.stream(stream):
                    for _ in range(5):
                        launch()
                torch.cuda.synchronize()
                if args.sweep_cold_l2:
                    reps = args.sweep_reps or 100
                    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                          for _ in range(reps)]
                    with torch.cuda.stream(stream):
                        for i in range(reps):
                            scratch.fill_(i & 0xFF)
                            ev[i][0].record(stream)
                            launch()
                            ev[i][1].record(stream)
                    torch.cuda.synchronize()
                    g.check_status(stream)
                    ms = sum(a.elapsed_time(b) for a, b in ev) / reps
                    print(json.dumps({
                        "workload": name, "M": w.M, "N": w.N, "K": w.K, "variant": variant,
                        "auto_variant": auto, "stream_k": bool(need), "launches": reps,
                        "l2": "cold (512 MiB written before each launch)",
                        "ms_per_launch": ms, "tflops": w.flops / (ms * 1e-3) / 1e12,
                        "hbm_gbs_algorithmic": w.min_bytes / (ms * 1e-3) / 1e9}), flush=True)
                    continue
                # enough launches for ~0.3 s of work
                t0 = time.perf_counter()
                with torch.cuda.stream(stream):
                    launch()
                torch.cuda.synchronize()
                reps = args.sweep_reps or max(10, min(5000, int(0.3 / max(time.perf_counter() - t0,
                                                                           1e-6))))
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    e0.record(stream)
                    for _ in range(reps):
                        launch()
                    e1.record(stream)
                torch.cuda.synchronize()
                g.check_status(stream)
                ms = e0.elapsed_time(e1) / reps
                print(json.dumps({
                    "workload": name, "M": w.M, "N": w.N, "K": w.K, "variant": variant,
                    "auto_variant": auto, "stream_k": bool(need), "launches": reps,
                    "l2": "warm (back-to-back launches)", "ms_per_launch": ms, "tflops": w.flops / (ms * 1e-3) / 1e12,
                    "hbm_gbs_algorithmic": w.min_bytes / (ms * 1e-3) / 1e9}), flush=True)
    g.gemm_f16_set_stream_k(0)
    return 0


def run_sweep_mx(args, g, dev, stream, sms):
    """--sweep over the block-scaled FP8 workloads and variants."""
    import torch
    from blackwell_tensor_core_fp16_gb300.workloads import MX_ORDER, MX_WORKLOADS
    names = [n.strip() for n in args.sweep_workloads.split(",") if n.strip()] or MX_ORDER
    for name in names:
        w = MX_WORKLOADS[name]
        t = mx_inputs_on_device(g, w, dev)
        auto = g.gemm_mxf8_choose_variant(w.M, w.N, w.K, sms)
        variants = ([auto] if args.sweep_variants == "auto"
                    else [int(v) for v in args.sweep_variants.split(",")]
                    if args.sweep_variants != "1,2,3,4,5" else [1, 2, 3, 4])
        for v in variants:
            with torch.cuda.stream(stream):
                for _ in range(5):
                    mx_launch(g, w, t, v, stream)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            with torch.cuda.stream(stream):
                mx_launch(g, w, t, v, stream)
            torch.cuda.synchronize()
            reps = args.sweep_reps or max(10, min(5000, int(0.3 / max(time.perf_counter() - t0,
                                                                       1e-6))))
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(reps):
                    mx_launch(g, w, t, v, stream)
                e1.record(stream)
            torch.cuda.synchronize()
            g.check_status(stream)
            ms = e0.elapsed_time(e1) / reps
            print(json.dumps({
                "workload": name, "M": w.M, "N": w.N, "K": w.K, "variant": v,
                "auto_variant": auto, "stream_k": False, "launches": reps,
                "l2": "warm (back-to-back launches)", "ms_per_launch": ms,
                "tflops": w.flops / (ms * 1e-3) / 1e12,
                "hbm_gbs_algorithmic": w.min_bytes / (ms * 1e-3) / 1e9}), flush=True)
        del t
    return 0


def run_sweep_processes(args):
    """--sweep in several fresh processes; per case, the median of the per-process means."""
    argv = [a for a in sys.argv[1:]]
    i = argv.index("--sweep-processes")
    del argv[i:i + 2]
    cases = {}
    for _ in range(args.sweep_processes):
        out = subprocess.run([sys.executable, os.path.abspath(__file__)] + argv, check=True,
                             capture_output=True, text=True).stdout
        for line in out.splitlines():
            if not line.startswith("{"):
                continue
            d = json.loads(line)
            key = (d["workload"], d["variant"], d["stream_k"], d["l2"])
            cases.setdefault(key, []).append(d)
    for key, runs in cases.items():
        d = dict(runs[0])
        means = [r["ms_per_launch"] for r in runs]
        ms = statistics.median(means)
        w_flops = 2.0 * d["M"] * d["N"] * d["K"]
        w_bytes = 2.0 * (d["M"] * d["K"] + d["N"] * d["K"] + d["M"] * d["N"])
        d.update({"processes": len(runs), "ms_per_launch": ms, "ms_per_process": means,
                  "tflops": w_flops / (ms * 1e-3) / 1e12,
                  "hbm_gbs_algorithmic": w_bytes / (ms * 1e-3) / 1e9})
        print(json.dumps(d), flush=True)
    return 0


def main():
    args = parse_args()
    if args.record_traffic:
        return record_traffic(args.record_traffic, os.environ.get("TRAFFIC_COMMAND", ""))
    if args.record_traffic_mx:
        return record_traffic_mx(args.record_traffic_mx, os.environ.get("TRAFFIC_COMMAND", ""))
    if args.record_traffic_gdn:
        return record_traffic_gdn(args.record_traffic_gdn, os.environ.get("TRAFFIC_COMMAND", ""))
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep and args.sweep_processes > 1:
        return run_sweep_processes(args)
    if args.config_only:
        return run_config_only(args)
    if args.sweep:
        return run_sweep(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
