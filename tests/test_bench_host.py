"""Host-side logic of bench.py on CPU: algorithmic byte counts, rank aggregation with a
world-size-2 gloo group, clock-sample parsing, and the reference (oracle) arm."""
import datetime
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_per_launch():
    n = 65536 * 7168
    assert bench.kernel_bytes("quant_i8", n) == 1423966208
    assert bench.kernel_bytes("dequant_i8", n) == 1423966208
    assert bench.kernel_bytes("dequant_accum_i8", n) == 2422210560
    assert bench.kernel_bytes("ring_hop_i8", n) == 1908408320
    assert bench.kernel_bytes("quant_mx", 4096 * 7168) == 88997888
    assert bench.kernel_bytes("dequant_mx", 4096 * 43008) == 533987328
    assert bench.kernel_bytes("dequant_accum_mx", n) == 2422210560  # same wire size as INT8
    assert bench.kernel_bytes("ring_hop_mx", n) == 1908408320
    assert bench.kernel_bytes("reduce_quant_i8", n) == 4 * 2 * n + 484442112  # four BF16 shards in, one wire out
    assert bench.kernel_bytes("reduce_quant_e4m3", n) == bench.kernel_bytes("reduce_quant_i8", n)
    assert bench.kernel_bytes("quant_e4m3", n) == bench.kernel_bytes("quant_i8", n)
    assert bench.kernel_bytes("quant_mx_f16", 4096 * 7168) == 88997888
    step = (4 * 1423966208 + 2422210560 + 1423966208 + 1908408320 + 6 * 88997888 + 533987328)
    assert step == 12518424576
    assert bench.step_bytes_of(65536, 4096) == step


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    m = bench.max_over_ranks(10.0 + rank * 5.0, world)
    dist.destroy_process_group()
    q.put((rank, m))


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_clock_summary_keeps_only_the_timed_region():
    c = bench.ClockSampler(0)
    t0 = datetime.datetime(2026, 12, 2, 8, 0, 0)
    c.t0, c.t1 = t0, t0 + datetime.timedelta(seconds=1)
    fmt = "%Y/%m/%d %H:%M:%S.%f"
    c.lines = [
        (t0 - datetime.timedelta(seconds=1)).strftime(fmt) + ", 800, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        (t0 + datetime.timedelta(milliseconds=100)).strftime(fmt) + ", 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        (t0 + datetime.timedelta(milliseconds=300)).strftime(fmt) + ", 1950, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
        (t0 + datetime.timedelta(milliseconds=500)).strftime(fmt) + ", 2000, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2000
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_peaks_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6787.2}))
    assert bench.load_peaks() == (6787.2, "measured")


def _json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_on_cpu():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3", "--ref-budget", "3"], capture_output=True, text=True, timeout=600,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is True
    from oracle import shards
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == shards.host_cores()
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    # the same config as the codec arm's line for this workload
    assert d["config"]["workload"].startswith("prefill pipeline: 4 x BF16 65536x7168")
    assert d["config"]["step_bytes"] == 12518424576 and d["config"]["launches_per_step"] == 14


def test_reference_arm_under_torchrun_world2():
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--ref-budget", "3"],
                       capture_output=True, text=True, timeout=600, env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def test_bench_rejects_too_few_warmup_steps():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_oracle_next_rows_times_every_next_row():
    # the CPU-oracle leg's timing of the next rows: one entry per next-row kernel the GPU
    # side reports (the tiled FP16 variant shares quant_mx_tiled's oracle), each positive
    from block_quantized_wire_gb300 import inputs
    xs = [inputs.prefill_buffer(w, device="cpu", rows=8) for w in range(bench.W_SRC)]
    sl = inputs.mx_slices_4096(device="cpu", rows=8)
    r = bench.oracle_next_rows((xs, sl), 8)
    assert r["rows"] == 8 and r["cores"] == 1 and r["kind"] == "oracle"
    want = {"quant_mx_slices", "quant_mx_tiled", "quant_mx_f16", "dequant_accum_mx", "ring_hop_mx",
            "reduce_quant_i8", "reduce_quant_e4m3", "quant_e4m3", "dequant_e4m3"}
    assert set(r["ops"]) == want
    assert all(v["GB/s"] > 0 for v in r["ops"].values())
