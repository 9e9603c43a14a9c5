"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

Every rank runs an independent copy of the workload; the only collectives
are a barrier and a MAX over the ranks' timings, and the reported rate is the
work of all ranks over the slowest rank's time.  The reference arm runs on
rank 0 only.
"""

import io
import os
import socket
import contextlib

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r times (1 + r) ms for the first quantity and (5 - r) ms for the second
        slowest = bench.max_over_ranks(torch, [1.0 + rank, 5.0 - rank], torch.device("cpu"), world)
        dist.barrier()
        q.put((rank, slowest))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the element-wise maximum: [max(1, 2), max(5, 4)]
    assert results == {0: [2.0, 5.0], 1: [2.0, 5.0]}


def test_max_over_ranks_single_rank_is_identity():
    import torch
    assert bench.max_over_ranks(torch, [3, 1.5], torch.device("cpu"), 1) == [3.0, 1.5]


def test_whole_job_rate_counts_all_ranks_over_slowest_time():
    ops = 2 * 4096 ** 3
    one = bench.whole_job_rate(1, ops, 10, 1.0)          # 10 GEMMs in 1 ms on one GPU
    assert one == pytest.approx(10 * ops / 1e-3 / 1e12)
    # weak scaling: 4 ranks, each the same work, slowest rank 1.25 ms
    assert bench.whole_job_rate(4, ops, 10, 1.25) == pytest.approx(4 * one / 1.25)


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        steps, warmup = 1, 0
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert bench.run_reference(A, rank=1, world=2) is None
    assert out.getvalue() == ""


def test_binding_batch_strides():
    """Host-side stride logic of the batched binding (no GPU): a leading
    dimension of 1 broadcasts (stride 0), a 1-D scale vector is shared."""
    import torch
    import quantized_mixed_precision_gb300 as bq
    a1 = torch.zeros((1, 4, 64), dtype=torch.int8)
    a3 = torch.zeros((3, 4, 64), dtype=torch.int8)
    assert bq._batch_stride(a1, 3, "A") == 0
    assert bq._batch_stride(a3, 3, "A") == 4 * 64
    with pytest.raises(ValueError):
        bq._batch_stride(torch.zeros((2, 4, 64)), 3, "A")
    assert bq._scale_stride(None, 3, "s") == 0
    assert bq._scale_stride(torch.zeros((64,)), 3, "s") == 0
    assert bq._scale_stride(torch.zeros((1, 64)), 3, "s") == 0
    assert bq._scale_stride(torch.zeros((3, 64)), 3, "s") == 64
