"""The multi-rank side of bench.py on the CPU: two processes on the gloo backend.

With N GPUs bench.py runs N independent replicas of the step (the GEMMs shard into independent
problems; no collective sits on the data path).  What multi-rank code there is lives on the host:
the slowest rank's time decides the job's time, the job's throughput counts every rank's work,
only rank 0 prints, and the reference arm runs on rank 0 alone.  These tests run that logic in
two gloo processes (127.0.0.1) without a GPU.
"""
from __future__ import annotations

import importlib.util
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench = load_bench()
        w, r, local = bench.dist_env()
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slower replica
        job_ms = bench.max_over_ranks(local_ms, w, "cpu")
        value = bench.whole_job_tflops(w, 4, 1e12, job_ms)
        out.put((rank, w, r, local, job_ms, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_on_gloo():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, w, r, local, job_ms, value in results:
        assert (w, r, local) == (2, rank, rank)
        assert job_ms == 15.0                    # the slowest rank's time, on every rank
        # both replicas' work over the slowest time: 2 ranks x 4 steps x 1 TFLOP / 15 ms
        assert value == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_rank_needs_no_group():
    bench = load_bench()
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.whole_job_tflops(1, 10, 2e12, 20.0) == pytest.approx(10 * 2e12 / 0.02 / 1e12)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Under torchrun every rank but 0 leaves the reference arm at once, printing nothing."""
    bench = load_bench()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(None) == 0
    assert buf.getvalue() == ""


def test_clock_records_that_force_a_second_measurement():
    bench = load_bench()
    ok = {"sm_mhz": 1400.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 20}
    assert not bench.clocks_rejected(ok)                     # the power cap alone is kept
    assert not bench.clocks_rejected(None)                   # no nvidia-smi: nothing to reject
    for reason in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(dict(ok, reasons=["sw_power_cap", reason]))
    locked = {"sm_mhz": 900.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 20}
    assert bench.clocks_rejected(locked)                     # stuck low with no reason
    assert not bench.clocks_rejected(dict(locked, reasons=["sw_power_cap"]))


def test_roofline_peak_follows_the_timed_region():
    bench = load_bench()
    # a long back-to-back region runs at the power-capped clock: the sustained figure
    assert bench.roofline_peak(1919.4, 1711.7, 1500.0) == (1711.7, "bf16_tflops_sustained")
    # a short region (and a peaks file without a sustained figure) takes the burst figure
    assert bench.roofline_peak(1919.4, 1711.7, 20.0)[0] == 1919.4
    assert bench.roofline_peak(1919.4, 0.0, 5000.0)[0] == 1919.4


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle, timed on the host cores) prints exactly one JSON
    line with the keys the benchmark contract names, on the same metric and workload as the
    CUDA arm, with no host-device traffic."""
    import json
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    p = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                       cwd=root, env=env, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    bench = load_bench()
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert (line["steps"], line["warmup"], line["n_gpus"]) == (2, 1, 1)
    assert line["config"]["workload"] == "square_8192+mlp_up_16384x14336x4096"
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == line["value"]
    assert cpu["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_ncu_csv_parsing_scales_units(tmp_path):
    """bench.py --record-traffic reads an ncu --csv log: rows grouped per launch in capture order,
    values scaled by their unit, non-CSV lines skipped."""
    bench = load_bench()
    hdr = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
           '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
           '"Metric Value"')
    rows = [
        ("0", "dram__bytes_read.sum", "Gbyte", "1.03"),
        ("0", "dram__bytes_write.sum", "Mbyte", "124.50"),
        ("0", "gpu__time_duration.sum", "ns", "612500"),
        ("1", "dram__bytes_read.sum", "Mbyte", "743.00"),
        ("1", "dram__bytes_write.sum", "Gbyte", "0.45"),
        ("1", "gpu__time_duration.sum", "msecond", "1.03"),
    ]
    lines = ["==PROF== Connected to process", hdr]
    for i, name, unit, val in rows:
        lines.append(f'"{i}","1","python","h","gemm_ws_kernel","1","7","(192, 1, 1)","(152, 1, 1)",'
                     f'"0","10.3","Command line profiler metrics","{name}","{unit}","{val}"')
    p = tmp_path / "l.csv"
    p.write_text("\n".join(lines) + "\n")
    got = bench.parse_ncu_csv(str(p))
    assert len(got) == 2 and got[0]["kernel"] == "gemm_ws_kernel"
    assert got[0]["metrics"]["dram__bytes_read.sum"] == pytest.approx(1.03e9)
    assert got[0]["metrics"]["dram__bytes_write.sum"] == pytest.approx(124.5e6)
    assert got[1]["metrics"]["gpu__time_duration.sum"] == pytest.approx(1.03e-3)
    assert got[0]["metrics"]["gpu__time_duration.sum"] == pytest.approx(612.5e-6)
    assert got[1]["metrics"]["dram__bytes_write.sum"] == pytest.approx(0.45e9)


def test_traffic_records_follow_their_kernel_sources(tmp_path, monkeypatch):
    """A recorded DRAM figure is reported only while the hash of the sources it was taken on
    matches; the Gated Delta Net record sums the launches of one call and is tagged with the Gated
    Delta Net sources' hash, the block-scaled FP8 record with the GEMM sources'."""
    bench = load_bench()
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash",
                        lambda sources=bench.GEMM_KERNEL_SOURCES: "hash-of-" + sources[1])
    hdr = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
           '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
           '"Metric Value"')

    def log(n_launch, name):
        lines = [hdr]
        for i in range(n_launch):
            for metric, val in (("dram__bytes_read.sum", 1000 * (i + 1)),
                                ("dram__bytes_write.sum", 10 * (i + 1)),
                                ("gpu__time_duration.sum", 5000)):
                unit = "ns" if metric.startswith("gpu") else "byte"
                lines.append(f'"{i}","1","python","h","{name}","1","7","(256, 1, 1)",'
                             f'"(152, 1, 1)","0","10.3","m","{metric}","{unit}","{val}"')
        p = tmp_path / f"{name}.csv"
        p.write_text("\n".join(lines) + "\n")
        return str(p)

    assert bench.record_traffic_gdn(log(3, "gdn"), "cmd") == 0
    big = bench.GDN_ROOFLINE_SCENARIO
    assert bench.recorded_traffic(big, "ncu_traffic_gdn.json", bench.GDN_KERNEL_SOURCES) == \
        1010 + 2020 + 3030
    assert bench.recorded_traffic(big, "ncu_traffic_gdn.json") is None   # another source set
    assert bench.record_traffic_mx(log(2, "mx"), "cmd") == 0
    assert bench.recorded_traffic("mx_step", "ncu_traffic_mx.json") == 1010 + 2020
    with pytest.raises(SystemExit):
        bench.record_traffic_mx(log(3, "mx3"))


def test_per_config_processes_take_the_median(monkeypatch):
    """The per_config leg's figures are the median over its processes of the per-process means;
    a child process that fails leaves the leg with the ones that ran (and says so)."""
    bench = load_bench()

    def leg(us, graph, cold):
        c = {"M": 2048, "N": 2048, "K": 2048, "us_per_launch": us, "us_per_launch_graph": graph,
             "cold_l2_us_per_launch": cold, "cublas_us_per_launch_graph_context": None,
             "tflops": 2 * 2048 ** 3 / (us * 1e-6) / 1e12, "frac_of_burst": 0.5,
             "hbm_gbs_algorithmic": 100.0, "hbm_frac": 0.01}
        return {"timing": "t", "configs": {"square_2048": c}, "gpu_launches": 10}

    children = [leg(14.0, 13.0, 18.0), leg(16.0, 15.0, 20.0)]

    class Done:
        def __init__(self, out):
            self.stdout = out

    def fake_run(cmd, **kw):
        if not children:
            raise RuntimeError("child failed")
        return Done("noise\n" + json.dumps(children.pop(0)) + "\n")

    monkeypatch.setattr(bench.subprocess, "run", fake_run)

    class Args:
        config_ms = 1.0
        cublas_steps = 0
        config_processes = 3

    got = bench.merge_config_processes(Args(), leg(12.0, 11.0, 30.0))
    c = got["configs"]["square_2048"]
    assert got["processes"] == 3 and "failed_processes" not in got
    assert c["us_per_launch"] == 14.0 and c["us_per_launch_per_process"] == [12.0, 14.0, 16.0]
    assert c["us_per_launch_graph"] == 13.0 and c["cold_l2_us_per_launch"] == 20.0
    assert c["tflops"] == pytest.approx(2 * 2048 ** 3 / 14e-6 / 1e12)
    assert c["frac_of_burst"] == pytest.approx(0.5 * 12.0 / 14.0)
    assert got["gpu_launches"] == 30
    # one child fails: two processes remain, and the failure is reported
    children[:] = [leg(14.0, 13.0, 18.0)]
    got = bench.merge_config_processes(Args(), leg(12.0, 11.0, 30.0))
    assert got["processes"] == 2 and len(got["failed_processes"]) == 1
    assert got["configs"]["square_2048"]["us_per_launch"] == 13.0
