"""The N > 1 path of bench.py: independent replicas, one per rank.

The path has no exchange step, so the only cross-rank work is the timing
aggregation: the job time is the slowest replica's (max over ranks) and the
job throughput counts every replica's bytes.  Checked here with world size 2
on the gloo backend (CPU), plus the reference arm's rule that only rank 0
runs and prints.
"""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # rank 0 is slower on the first time, rank 1 on the second
        mine = [3.0 if rank == 0 else 2.0, 5.0 if rank == 1 else 4.5]
        got = bench.max_over_ranks(mine, world, "cpu")
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_world_2_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == [3.0, 5.0] and res[1] == [3.0, 5.0]


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([1.5, 2], 1, "cpu") == [1.5, 2.0]


def test_job_throughput_counts_every_replica():
    # two replicas, 1 GB each, slowest 2 ms -> 1000 GB/s for the job
    assert bench.job_gbs(1e9, 2.0, 2) == pytest.approx(1000.0)
    assert bench.job_gbs(1e9, 2.0, 1) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_write_traffic_averages_split_launches(tmp_path):
    hdr = '"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'
    rows = [
        '"0","void spec_attn::split_attn_tc_kernel<256, 0, 0>(...)","dram__bytes_read.sum","byte","100"',
        '"0","void spec_attn::split_attn_tc_kernel<256, 0, 0>(...)","dram__bytes_write.sum","byte","10"',
        '"1","void spec_attn::merge_lse_kernel<256>(...)","dram__bytes_read.sum","byte","999"',
        '"2","void spec_attn::split_attn_tc_kernel<256, 0, 0>(...)","dram__bytes_read.sum","byte","200"',
        '"2","void spec_attn::split_attn_tc_kernel<256, 0, 0>(...)","dram__bytes_write.sum","byte","30"',
    ]
    csv_path = tmp_path / "t.csv"
    csv_path.write_text("==PROF== noise\n" + hdr + "\n".join(rows) + "\n")
    out = tmp_path / "traffic.json"
    bench.write_traffic(str(csv_path), str(out))
    d = json.loads(out.read_text())
    assert d["launches"] == 2 and d["dram_bytes_per_launch"] == 170
    assert d["kernel_source_hash"] == bench.kernel_source_hash()


def test_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    """The traffic record stays valid across comment edits of the kernel
    sources, and goes stale on any change to the code itself."""
    import shutil
    src = os.path.join(ROOT, "speculative_decode_verify_paged_gb300", "csrc")
    dst = tmp_path / "speculative_decode_verify_paged_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    f = dst / "merge_lse.cu"
    text = f.read_text()
    f.write_text("// a new comment line\n" + text.replace("\n", "\n\n", 3) + "/* and a block\n comment */\n")
    assert bench.kernel_source_hash() == h0
    f.write_text(text + "\nstatic int spec_attn_unused_probe_value = 1;\n")
    assert bench.kernel_source_hash() != h0
