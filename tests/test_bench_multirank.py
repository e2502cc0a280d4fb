"""Host logic of bench.py's multi-GPU mode on CPU: two gloo ranks stand in for
two GPUs.  Each rank runs the same replica workload; the job's step time is
the maximum over ranks and the job's throughput counts every rank's bytes.
The reference arm runs on rank 0 only."""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 1.0 + 0.5 * rank            # rank 1 is the slow one
        ms = bench.reduce_step_time(ms_local, world)
        value = bench.job_value(1e9, ms, world)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value():
    world = 2
    port = 29500 + (os.getpid() % 1000)
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == pytest.approx(1.5)
    # 2 ranks x 1 GB in 1.5 ms each step
    assert res[0][1] == res[1][1] == pytest.approx(2 * 1e9 / 1.5e-3 / 1e9)


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_step_time(0.25, 1) == 0.25
    assert bench.job_value(5e8, 0.5, 1) == pytest.approx(1000.0)


def test_reference_arm_only_on_rank0():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_profiled_traffic_needs_matching_sources(tmp_path):
    """The roofline's DRAM traffic comes from a committed ncu record (a small
    JSON file) and is used only while the record names the fingerprint of the
    sources being built; otherwise it is null."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    for names in (bench.LM_HEAD_SOURCES, bench.GEMM_SOURCES):
        sha = bench.kernel_source_sha(names)
        good = tmp_path / "good.json"
        good.write_text(json.dumps({"source_sha256": sha, "dram_bytes_read": 389400320,
                                    "dram_bytes_write": 2908160}))
        assert bench.profiled_traffic(str(good), names) == 389400320 + 2908160
        stale = tmp_path / "stale.json"
        stale.write_text(json.dumps({"source_sha256": "0000000000000000", "dram_bytes_read": 1,
                                     "dram_bytes_write": 2}))
        assert bench.profiled_traffic(str(stale), names) is None
        assert bench.profiled_traffic(str(tmp_path / "missing.json"), names) is None
        broken = tmp_path / "broken.json"
        broken.write_text("not json")
        assert bench.profiled_traffic(str(broken), names) is None


def test_device_status_fails_the_bench_leg():
    """A kernel that gave up a bounded wait leaves the device status word set:
    the bench then refuses to print its timings and names the leg."""
    sys.path.insert(0, ROOT)
    import bench

    class FakeLib:
        def __init__(self, status):
            self.status = status

        def get_status(self):
            st, self.status = self.status, 0     # read and cleared, like w4v_get_status
            return st

    bench.check_device_status(FakeLib(0), "clean leg")
    with pytest.raises(RuntimeError, match="36-layer sweep"):
        bench.check_device_status(FakeLib(7), "36-layer sweep")
