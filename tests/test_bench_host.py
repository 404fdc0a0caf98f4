"""Host-side logic of bench.py (no GPU): the roofline entry names the roof
that binds the decode kernel."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6700.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def test_hbm_bound_decode():
    # 80 MB and 18 GFLOP in 30 us: 2667 GB/s (0.40 of HBM), 608 TFLOP/s (0.32 of tensor)
    r = bench.roofline_entry(80e6, 18.25e9, 0.030, PEAKS, 80.5e6, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 80e6 / 30e-6 / 1e9) < 1e-9
    assert abs(r["frac"] - r["achieved"] / 6700.0) < 1e-12
    assert r["traffic"] == 80.5e6


def test_tensor_bound_decode():
    # speculative decode: 720 MB and 310 GFLOP in 300 us: 0.36 of HBM, 0.54 of tensor
    r = bench.roofline_entry(720e6, 310e9, 0.300, PEAKS, None, "measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 310e9 / 300e-6 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / 1900.0) < 1e-12
    assert r["frac"] > 720e6 / 300e-6 / 1e9 / 6700.0


def _free_port():
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica_rank(rank, world, port, out):
    """One rank of a replicas run: its environment as torchrun sets it, a gloo
    group on host cores, the bench's max-over-ranks time and job rate."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_env()
    ms = 10.0 + 5.0 * r  # rank 1 is the slow one
    m = bench.max_over_ranks(ms, dist, "cpu")
    dist.barrier()
    out.put((r, w, local, m, bench.job_rate(w, 1e6, m)))
    dist.destroy_process_group()


def test_two_replicas_are_timed_by_the_slowest_rank():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 and g[2] == g[0] for g in got)
    assert all(g[3] == 15.0 for g in got)  # both ranks see the slowest rank's time
    assert all(abs(g[4] - 2 * 1e6 / 15e-3) < 1e-6 for g in got)  # both ranks' units over that time


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5
    assert bench.job_rate(1, 8e7, 40.0) == 8e7 / 40e-3


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        workload, steps, warmup = "dsv3", 1, 0
    assert bench.run_reference(Args(), 2, 1) is None  # returns before any work


def test_rotation_copies_exceed_l2():
    """The timed loops rotate copies of the cache and of the weights that
    hold more than twice the L2 in all, so no step finds its inputs there:
    the dsv3 cache (75.5 MB) in 4 copies, the one-group weights (33.6 MB)
    in 9, the two-group weights (16.8 MB) in 18, a cache larger than L2
    in one."""
    for nbytes, want in ((16 * 4096 * 1152, 4), (2 * 128 * 128 * 512 * 2, 9), (2 * 128 * 128 * 256 * 2, 18),
                         (900 * 2 ** 20, 1)):
        n = bench.rotation_copies(nbytes)
        assert n == want, (nbytes, n)
        assert n * nbytes >= 2.2 * bench.L2_BYTES or n == 1 and nbytes >= 2.2 * bench.L2_BYTES
