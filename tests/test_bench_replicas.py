"""CPU test of the multi-rank path of bench.py with the gloo backend (world size 2): each
rank runs its own replica and reports its step time; the job's time is the slowest
rank's, and the job throughput counts every rank's work (weak scaling)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = 10.0 + 5.0 * rank  # rank 1 is the slow one
    ms = bench.max_over_ranks(ms_local, world, "cpu")
    value = bench.job_throughput(65536, world, ms)
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_take_max_time_and_sum_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ms, value in out:
        assert ms == pytest.approx(15.0)
        assert value == pytest.approx(65536 * 2 / 0.015)


def test_single_rank_is_local_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_throughput(1000, 1, 2.0) == pytest.approx(500000.0)


def test_algorithmic_counts():
    """The work the roofline figures divide by, against brute-force counts: prefill
    scoring pairs (row i has the i chunks before it), and the training step's valid
    (slot, head) units (4 x 12 x 2004 at 256 chunks, k = 8)."""
    sys.path.insert(0, ROOT)
    import bench
    nc, d = 1000, 64
    assert bench.prefill_flops(nc, d) == 2 * d * sum(len(range(i)) for i in range(nc))
    assert bench.prefill_flops(16384, 768) == 206145847296
    assert bench.algorithmic_flops(4, 256, 12, 64, 8)["units"] == 4 * 12 * 2004
    assert bench.algorithmic_flops(1, 3, 1, 64, 8)["units"] == 1  # rows 0, 1 feed chunks 1, 2
    # Bytes each GCA kernel must move once, counted tensor by tensor at the 128M shape:
    # one [B][L][H][dh] bf16 tensor is 4 * 16384 * 12 * 64 * 2 bytes, one LSE or D row set
    # [B][nQ][H][k][64] f32 is 4 * 256 * 12 * 8 * 64 * 4 bytes.
    t, rows = 4 * 16384 * 12 * 64 * 2, 4 * 256 * 12 * 8 * 64 * 4
    by = bench.algorithmic_bytes(4, 256, 12, 64, 8)
    assert by["gca_fwd"] == 3 * t + t + rows            # reads Q, K, V; writes O, LSE
    assert by["gca_bwd_q"] == 4 * t + rows + t + rows   # reads Q, dO, K, V, LSE; writes dQ, D
    assert by["gca_bwd_kv"] == 4 * t + 2 * rows + 2 * t  # reads Q, dO, K, V, LSE, D; writes dK, dV


def test_traffic_figures_follow_the_sources():
    """A stored DRAM traffic figure is reported only while the kernel's sources still hash
    to the fingerprint taken at capture time."""
    sys.path.insert(0, ROOT)
    import bench
    fp = bench.source_fingerprint("gca_fwd")
    assert bench.measured_traffic("gca_fwd", {"gca_fwd": (123.0, fp)}) == 123.0
    assert bench.measured_traffic("gca_fwd", {"gca_fwd": (123.0, "0" * 16)}) is None
    assert bench.measured_traffic("gca_fwd", {}) is None
