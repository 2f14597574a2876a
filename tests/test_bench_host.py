"""Host-side checks of bench.py (no GPU): the decode layouts, the traffic gate
on the kernel source, and the reference arm's JSON line."""
import json
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from block_scaled_fp4_fp_gb300 import synth  # noqa: E402


def test_layer_groups_cover_the_same_weights():
    split = synth.layer_groups("split")
    assert [(n, k) for n, k, _ in split] == [(p[1], p[2]) for p in synth.LAYER_PROJECTIONS]
    fused = synth.layer_groups("fused")
    assert [(n, k, g) for n, k, g in fused] == [(15360, 5120, [0, 1, 2]), (5120, 5120, [3]),
                                               (34816, 5120, [4, 5]), (5120, 17408, [6])]
    for layout in ("fused", "fused_qkv"):
        groups = synth.layer_groups(layout)
        assert sorted(p for _, _, g in groups for p in g) == list(range(7))
        assert sum(n * k for n, k, _ in groups) == sum(n * k for n, k, _ in split)
    with pytest.raises(ValueError):
        synth.layer_groups("other")


def test_committed_traffic_needs_the_current_source(tmp_path, monkeypatch):
    src = os.path.join(ROOT, "block_scaled_fp4_fp_gb300", "csrc")
    os.makedirs(tmp_path / "block_scaled_fp4_fp_gb300" / "csrc")
    for f in ("qmv_tc.cu", "common.cuh"):
        shutil.copy(os.path.join(src, f), tmp_path / "block_scaled_fp4_fp_gb300" / "csrc" / f)
    os.makedirs(tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash("qmv_tc.cu")
    rec = {"k": {"source_hash": h, "dram_bytes_per_launch": 123}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.committed_traffic("qmv_tc.cu", "k") == 123
    with open(tmp_path / "block_scaled_fp4_fp_gb300" / "csrc" / "qmv_tc.cu", "a") as f:
        f.write("\n// changed\n")
    assert bench.committed_traffic("qmv_tc.cu", "k") is None
    assert bench.committed_traffic("qmv_tc.cu", "missing") is None


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["warmup"] == 0
    assert line["config"]["workload"] == bench.WORKLOAD and line["config"]["layout"] == bench.LAYOUT
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def _ranks_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, e2e = bench.max_over_ranks([1.0 + rank, 10.0 - rank], "cpu")
        q.put((rank, ms, e2e, bench.job_gbs(1000000, ms, world)))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_takes_the_slowest_rank():
    """World size 2 on gloo: both ranks report the maximum of each time, and the
    job throughput counts both replicas' bytes over that time."""
    import multiprocessing as mp
    import socket
    with socket.socket() as s_:
        s_.bind(("127.0.0.1", 0))
        port = s_.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ranks_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1:3] for o in out] == [(2.0, 10.0), (2.0, 10.0)]
    assert all(abs(o[3] - 2 * 1000000 / 2.0 / 1e6) < 1e-12 for o in out)


def test_reference_arm_other_ranks_do_no_work():
    """Under torchrun only rank 0 runs the oracle and prints; rank 1 exits 0 silently."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == "", (r.stdout, r.stderr[-1000:])


def test_nvtx_ranges_and_device_info_never_raise():
    """The bench's NVTX ranges and device record must not break a run: without a
    GPU (or NVTX) the range is a no-op and the record says what it could not read."""
    with bench.nvtx("test range"):
        x = 1 + 1
    assert x == 2
    info = bench.device_info(0)
    assert info["host_cores"] >= 1
    assert ("name" in info and info["sm_count"] >= 1) or "error" in info
