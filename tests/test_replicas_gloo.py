"""bench.py's multi-rank logic on CPU ranks (gloo, world size 2): every rank gets its own
seeded token batch of the workload's shape, the step time reported is the slowest rank's,
and the whole-job throughput counts every rank's tokens.  No GPU is touched."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from mixture_experts_ffn_top_gb300.workloads import WORKLOADS

        wl = WORKLOADS["tiny"]
        base = np.zeros((wl.N, wl.D), np.float32)
        h = bench.rank_hidden(wl, base, rank, world)
        ms = bench.max_over_ranks(1.0 + rank, "cpu")  # rank r took 1 + r ms
        np.save(os.path.join(out_dir, f"h{rank}.npy"), h)
        np.save(os.path.join(out_dir, f"ms{rank}.npy"), np.array([ms, bench.job_throughput(world, wl.N, ms)]))
    finally:
        dist.destroy_process_group()


def test_two_cpu_ranks(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn", join=True)
    h0, h1 = np.load(tmp_path / "h0.npy"), np.load(tmp_path / "h1.npy")
    assert h0.shape == h1.shape == (64, 256)
    assert not np.array_equal(h0, h1)          # independent batches per rank
    assert abs(h0.std() - 1.0) < 0.05 and abs(h1.std() - 1.0) < 0.05
    for r in range(world):
        ms, tput = np.load(tmp_path / f"ms{r}.npy")
        assert ms == 2.0                        # the slowest rank's time on every rank
        assert tput == world * 64 / 2e-3        # all ranks' tokens over that time


def test_single_rank_keeps_workload_batch():
    import sys

    sys.path.insert(0, ROOT)
    import bench
    from mixture_experts_ffn_top_gb300.workloads import WORKLOADS

    wl = WORKLOADS["tiny"]
    base = np.ones((wl.N, wl.D), np.float32)
    assert bench.rank_hidden(wl, base, 0, 1) is base
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_throughput(1, 2048, 1.0) == 2048e3


def test_clock_summary_window_and_reasons():
    """bench.py's clock record: samples inside the timed window, or its two neighbours when the
    window is shorter than the sampling period; throttle reasons read from the 'Active' columns."""
    import bench
    row = "{sm}, 2070, 900.0, 0x0, {hw}, Not Active, Not Active, {cap}"
    lines = [(0.0, row.format(sm=1900, hw="Not Active", cap="Not Active")),
             (1.0, row.format(sm=2070, hw="Not Active", cap="Active")),
             (2.0, row.format(sm=2040, hw="Not Active", cap="Not Active")),
             (3.0, row.format(sm=1500, hw="Active", cap="Not Active")),
             (4.0, "garbage")]
    c = bench.clock_summary(lines, 0.5, 2.5)
    assert c == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 2,
                 "samples_in_window": 2}
    c = bench.clock_summary(lines, 2.2, 2.4)  # no sample inside: the ones at 2.0 and 3.0
    assert c["samples_in_window"] == 0 and c["samples"] == 2
    assert c["sm_mhz"] == 1770.0 and c["reasons"] == ["hw_slowdown"]
    assert bench.clock_summary([], 0.0, 1.0) is None


class _FakeOps:
    """Stands in for the binding's NUMA query (no GPU here)."""

    def __init__(self, node=None, exc=None):
        self.node, self.exc = node, exc

    def moe_device_host_numa_node(self):
        if self.exc is not None:
            raise self.exc
        return self.node


def test_bind_near_gpu_moves_to_the_node_and_reports_the_old_set():
    """The bench's pinned buffers are allocated from the CPUs of the node the device reports;
    the previous CPU set is returned for restoring, and a node without CPUs we may use, no NUMA
    placement, or a failed query leave the affinity alone."""
    import sys

    sys.path.insert(0, ROOT)
    import bench

    before = os.sched_getaffinity(0)
    try:
        nodes = sorted(int(d[4:]) for d in os.listdir("/sys/devices/system/node") if d.startswith("node")
                       and d[4:].isdigit()) if os.path.isdir("/sys/devices/system/node") else []
        if nodes:
            node, prev = bench.bind_near_gpu(_FakeOps(nodes[0]))
            assert node == nodes[0]
            now = os.sched_getaffinity(0)
            assert now <= before and now
            if prev is not None:
                assert prev == before
                os.sched_setaffinity(0, prev)
        assert bench.bind_near_gpu(_FakeOps(-1)) == (None, None)
        assert bench.bind_near_gpu(_FakeOps(exc=RuntimeError("no device"))) == (None, None)
        assert bench.bind_near_gpu(_FakeOps(10 ** 6)) == (None, None)  # no such node directory
        assert os.sched_getaffinity(0) == before
    finally:
        os.sched_setaffinity(0, before)
