"""The benchmark's multi-rank logic on CPU: world_size 2 over gloo (no GPU).  The path shards
with no data exchange, so N ranks are N replicas; the only collective is the max of the ranks'
timings, and the job value is all ranks' tokens over the slowest rank's time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.5], world)
    value = bench.job_tokens_per_s(8192, world, got[0])
    dist.destroy_process_group()
    q.put((rank, got, value))


def test_max_over_ranks_and_job_value_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == [2.0, 10.0, 3.5]
        assert value == pytest.approx(8192 * 2 / 2.0e-3)


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.job_tokens_per_s(8192, 1, 1.0) == pytest.approx(8192e3)


def test_e2e_input_slices_cover_every_byte():
    """The end-to-end loop cuts each (device, host) input pair into byte slices dealt over the
    H2D streams; copying every slice must reproduce each tensor exactly."""
    import bench

    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(3)
    hosts = [torch.randn(1000, 37, generator=g), torch.arange(12345, dtype=torch.int16),
             torch.randint(0, 255, (3, 5, 7), generator=g, dtype=torch.uint8)]
    devs = [torch.empty_like(h) for h in hosts]
    sl = bench._byte_chunks(list(zip(devs, hosts)), chunk_bytes=4096)
    assert all(d.numel() == h.numel() <= 4096 for d, h in sl)
    assert sum(h.numel() for _, h in sl) == sum(h.numel() * h.element_size() for h in hosts)
    for j in range(3):  # three streams' shares, in any order
        for d, h in sl[j::3]:
            d.copy_(h)
    for d, h in zip(devs, hosts):
        assert torch.equal(d, h)
