"""The multi-rank host logic of bench.py on CPU: two gloo ranks (world_size 2).

Under torchrun every rank runs its own replica; the timing is the max over ranks and
the tokens the sum, and only rank 0 prints (and, for the reference arm, works)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    try:
        r, w, lr = bench.dist_env()
        bench.dist_init(w, "gloo")
        bench.barrier(w)
        mx = bench.max_over_ranks(10.0 * (rank + 1), w, "cpu")
        sm = bench.sum_over_ranks(4096.0, w, "cpu")
        # the reference arm works on rank 0 only; the other ranks return nothing
        class A:
            steps, warmup, workload = 1, 3, "tiny"
            reference_seconds = 1.0
            tokens = experts = None
            router_gemm = False
        ref = bench.run_reference(A, r, w) if r != 0 else "skipped"
        q.put((r, w, lr, mx, sm, ref))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timing_and_tokens():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, world, local, mx, sm, ref) in enumerate(got):
        assert (rank, world, local) == (r, 2, r)
        assert mx == 20.0          # the slower rank sets the step time
        assert sm == 8192.0        # tokens of all ranks
    assert got[1][5] is None       # rank 1 does no reference work


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.sum_over_ranks(7.0, 1, "cpu") == 7.0
    bench.barrier(1)
    assert not dist.is_initialized()
