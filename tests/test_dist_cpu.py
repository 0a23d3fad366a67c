"""The replica (N>1) path of bench.py on CPU: two gloo ranks run the barrier and the
max-over-ranks reduction of the timed duration that rank 0 reports."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world)})
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        assert (r, lr, w) == (rank, rank, world)
        bench.barrier(world)
        t = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)


def test_byte_accounting_matches_the_shapes():
    import numpy as np

    import bench

    # MLP: weights 3 * 2560 * 9728 * (1 + 1/32) + per-token activations
    assert bench.mlp_bytes(1) == int(3 * 2560 * 9728 * 33 / 32 + 2560 * 33 / 32 + 2 * 9728 * 33 / 32 + 2560 * 2)
    lens = np.array([234, 4096])
    assert bench.attn_bytes(lens) == (234 + 4096) * 8 * 128 * 2 * 2 + 2 * 32 * 128 * 2 * 2
    parts = bench.step_bytes(np.full(64, 2000))
    assert set(parts) == set(bench.OP_NAMES)
    assert parts["attention_quant"] > parts["mlp"] > parts["qkv_gemm_kv_append"] > parts["o_gemm"]


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
