"""The benchmark's multi-rank host logic on CPU (gloo, world_size 2).

The operator has no cross-GPU exchange, so ``bench.py`` runs one replica per
rank; ranks meet only at a barrier and at the max-reduction of the step time.
These tests run that host logic with two CPU processes.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    # each rank reports a different step time; every rank must see the maximum
    got = bench.max_over_ranks(1.5 + rank, w, device="cpu")
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_single_rank_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    assert bench.dist_setup() == (1, 0, 0)
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_compulsory_bytes_encoder32():
    """The roofline's byte model for the encoder workload: forward
    V + O + 12 B/sample, backward 2V + O + 24 B/sample."""
    import bench
    from scale_deformable_attention_forward_gb300 import inputs as gen
    w = gen.WORKLOADS["encoder32"]
    fwd, bwd = bench.compulsory_bytes(w)
    V = 2 * 22223 * 8 * 32 * 4
    S = 5689088
    assert fwd == V + V + 12 * S
    assert bwd == 2 * V + V + 24 * S
    assert round((fwd + bwd) / 1e6, 1) == 432.4
