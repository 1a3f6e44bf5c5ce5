"""bench.py's multi-GPU path on the CPU: two gloo ranks stand for two GPUs
(independent replicas, no data-path collective). The job time is the slowest
rank's, the job rate counts every rank's units, and the reference arm prints
only on rank 0."""
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(1.0 + rank, world)       # rank r "took" 1 + r seconds
        rate = bench.job_throughput(100.0, slowest, world)
        q.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, slowest, rate in res:
        assert slowest == 2.0                       # max over ranks
        assert rate == pytest.approx(2 * 100.0 / 2.0)


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(10.0, 2.0, 1) == 5.0


def test_l2_label_separates_cold_and_warm_streams():
    sys.path.insert(0, ROOT)
    import bench
    l2 = 126 << 20
    # the sweep: 48 layers x (10 .. 74 experts) x 768,000 B, all far above L2
    cold = bench.l2_label(48, [48 * 10 * 768000, 48 * 74 * 768000], l2)
    assert cold.startswith("inputs larger than L2") and "48-layer" in cold
    # one repeated layer of the hot case (10 experts, 7.7 MB) stays in L2
    warm = bench.l2_label(1, [10 * 768000, 48 * 74 * 768000], l2)
    assert warm.startswith("L2-warm") and "[0]" in warm


def test_case_row_arithmetic():
    sys.path.insert(0, ROOT)
    import bench
    # 48 layer calls of 10 experts (768,000 B each) replayed in 0.48 ms
    row = bench.case_row(2, "hot", [10] * 48, 48 * 10 * 768000, 0.48, 48, 6681.8)
    assert row["us_per_call"] == 10.0 and row["layers_step_ms"] == 0.48
    assert row["effective_GBps"] == pytest.approx(768.0, abs=0.1)
    assert row["pct_of_hbm_peak"] == pytest.approx(100 * 768.0 / 6681.8, abs=0.05)
    assert row["mean_active_experts"] == 10.0 and row["M"] == 2 and row["regime"] == "hot"


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True, env=env,
                       timeout=120, cwd=ROOT)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
