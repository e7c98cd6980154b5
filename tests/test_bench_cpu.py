"""bench.py on the CPU: the replica aggregation across ranks (two gloo
processes) and the CPU-oracle reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist = bench.init_dist(world, "gloo")
    bench.barrier(dist)
    # rank r "took" 1 + r seconds for 10·(r+1) units of work
    t, w = bench.reduce_time_and_work(dist, 1.0 + rank, 10.0 * (rank + 1))
    q.put((rank, t, w))
    bench.barrier(dist)
    dist.destroy_process_group()


def test_replica_timing_is_max_over_ranks_and_work_sums():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, w in out:
        assert t == 2.0 and w == 30.0, (rank, t, w)


def _bench(args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=e, timeout=600, cwd=ROOT)


@pytest.mark.parametrize("extra", [[], ["--dtype", "bf16"], ["--accumulate", "f16"]])
def test_reference_arm_prints_one_line(extra):
    r = _bench(["--impl", "reference", "--workload", "gemm_256", "--steps", "3", "--warmup", "3",
                "--cpu-seconds", "1", *extra])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "gemm_256" and d["higher_is_better"] is True
    assert d["config"]["accumulate"] == ("f16" if "--accumulate" in extra else "f32")


def test_fp16_accumulator_with_bf16_rejected():
    r = _bench(["--impl", "reference", "--workload", "gemm_256", "--steps", "3", "--warmup", "3",
                "--dtype", "bf16", "--accumulate", "f16"])
    assert r.returncode != 0


def test_reference_arm_non_zero_rank_is_silent():
    r = _bench(["--impl", "reference", "--workload", "gemm_256", "--steps", "3", "--warmup", "3",
                "--gpus", "2"], env={"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_warmup_floor_enforced():
    r = _bench(["--impl", "reference", "--workload", "gemm_256", "--steps", "3", "--warmup", "2"])
    assert r.returncode != 0


def test_roofline_byte_figures():
    """The per-flop byte figures bench.py reports, from the plan and the workload.

    At 8192^3 the kernel delivers every cluster tile its 256 A rows and 256 B
    rows of 128 bytes per k-block: 1024 tiles x 128 k-blocks x 512 rows x 128 B
    = 2^33 bytes into shared memory.  A full Nsight Compute capture of that
    launch counted 8,589,937,024 bytes arriving from L2
    (l1tex__m_xbar2l1tex_read_bytes.sum), the same figure within 2.5 KB."""
    import bench
    import dense_fp16_gemm_gb300 as g
    from dense_fp16_gemm_gb300 import inputs
    w = inputs.WORKLOADS["gemm_8192"]
    pl = g.plan(w.M, w.N, w.K, num_sms=152, max_clusters=76)
    assert bench.l2_to_sm_bytes(pl) == 2 ** 33
    assert abs(bench.l2_to_sm_bytes(pl) - 8_589_937_024) < 2600
    assert w.flops == 2 * 8192 ** 3
    assert w.compulsory_bytes == 3 * 8192 * 8192 * 2          # A and B read, C written, fp16
    # two pairs per cluster: each pair receives the tile's A rows (multicast), plus 512 B rows
    r = inputs.WORKLOADS["ragged_4000x3000x5000"]
    pr = g.plan(r.M, r.N, r.K, num_sms=152, max_clusters=36, lib=g.library_mcast())
    assert pr["cluster_pairs"] == 2
    assert bench.l2_to_sm_bytes(pr) == pr["num_tiles"] * pr["k_blocks"] * 128 * (2 * 256 + 512)


def test_traffic_record_used_only_for_the_same_kernel_source(tmp_path, monkeypatch):
    """The roofline's DRAM figure comes from a machine-readable record of an
    Nsight Compute capture, and only while the kernel sources hash the same."""
    import json

    import bench
    path = tmp_path / "dram_traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.recorded_traffic("gemm_8192") == (None, None)
    rec = {"dram_bytes_per_launch": 1_100_000_000, "kernel_source_sha256_16": bench.kernel_source_hash(),
           "command": "ncu …", "launches": 1}
    path.write_text(json.dumps({"gemm_8192": rec}))
    assert bench.recorded_traffic("gemm_8192")[0] == 1_100_000_000
    assert bench.recorded_traffic("gemm_4096") == (None, None)
    rec["kernel_source_sha256_16"] = "0" * 16
    path.write_text(json.dumps({"gemm_8192": rec}))
    assert bench.recorded_traffic("gemm_8192") == (None, None)
