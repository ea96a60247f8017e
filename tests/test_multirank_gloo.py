"""Multi-rank host logic on CPU with gloo process groups of 2 and 4 ranks.

1. The data-parallel flow of "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §总结
   with real ranks: each rank takes its block range from the C-ABI's host
   layout, computes its partial sum of squares, the partials are all-reduced
   ("DeepSpeed ZeRO 优化" §七), each rank steps its range, and an all-gather of
   codes and scales rebuilds the whole-buffer result bit for bit.  The per-rank
   arithmetic here is the oracle's: the test is about the ranges and the
   exchanges, which need no GPU.
2. bench.py's max-over-ranks timing and whole-job rate."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

B = 16384


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _dp_worker(rank, world, port, shapes, result_q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    from blockwise_fp8_zero_fold_gb300 import fp8z1 as F

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        L = F.fp8z1_build_layout(shapes, dp_size=world, host_only=True)
        nblk = F.fp8z1_layout_info(L)[0]
        b0, b1 = F.fp8z1_shard_range(L, rank)
        per = -(-nblk // world)
        rng = np.random.default_rng(0)  # every rank draws the same global tensors
        rows = [(rng.standard_normal(s) * 1024e-3).astype(np.float32) for s in shapes]
        master = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
        g = oracle.fold(shapes, rows, b0, b1)
        p = oracle.fold(shapes, master, b0, b1)
        m, v = np.zeros_like(p), np.zeros_like(p)
        # the partial sums of squares, all-reduced
        acc = oracle.SumsqAccumulator()
        acc.add(g)
        part = torch.tensor([acc.result()], dtype=torch.float64)
        dist.all_reduce(part)
        hp = oracle.make_hp(1e-3, 0.9, 0.95, 1e-8, 0.1, 0.5, 1024.0, 1)
        q, sc, _ = oracle.step(hp, float(part.item()), 0, g, p, m, v)
        # all-gather codes and scales (equal-size buffers: pad the short last rank)
        qpad = np.zeros(per * B, np.uint8)
        qpad[:q.size] = q
        spad = np.zeros(per, np.float32)
        spad[:sc.size] = sc
        qs = [torch.zeros(per * B, dtype=torch.uint8) for _ in range(world)]
        ss = [torch.zeros(per, dtype=torch.float32) for _ in range(world)]
        dist.all_gather(qs, torch.from_numpy(qpad))
        dist.all_gather(ss, torch.from_numpy(spad))
        if rank == 0:
            codes = np.concatenate([x.numpy() for x in qs])[:nblk * B]
            scales = np.concatenate([x.numpy() for x in ss])[:nblk]
            result_q.put((b0, b1, codes, scales, float(part.item())))
        else:
            result_q.put((b0, b1, None, None, float(part.item())))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("shapes,world", [([(1, 300, 200)], 2), ([(3, 129, 257), (1, 17, 690)], 2),
                                          ([(1, 300, 200)], 4)])
def test_multi_rank_step_equals_one_rank(shapes, world):
    """world ranks step their block ranges and exchange; with 6 blocks over 4
    ranks the last rank's range is empty and it still joins both exchanges."""
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dp_worker, args=(r, world, port, shapes, q)) for r in range(world)]
    for p in procs:
        p.start()
    outs = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ranges = sorted((o[0], o[1]) for o in outs)
    nblk = oracle.count_blocks(shapes)
    assert ranges == [oracle.shard_range(nblk, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == nblk
    assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
    codes, scales = next((o[2], o[3]) for o in outs if o[2] is not None)
    # the same step on one rank owning everything
    rng = np.random.default_rng(0)
    rows = [(rng.standard_normal(s) * 1024e-3).astype(np.float32) for s in shapes]
    master = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
    g = oracle.fold(shapes, rows)
    p = oracle.fold(shapes, master)
    s_total, _ = oracle.sumsq(g)
    # the partials added in double: within a few roundings of the exact sum
    assert all(o[4] == outs[0][4] for o in outs)
    assert abs(outs[0][4] - s_total) <= world * 2 ** -52 * s_total
    hp = oracle.make_hp(1e-3, 0.9, 0.95, 1e-8, 0.1, 0.5, 1024.0, 1)
    q1, s1, _ = oracle.step(hp, outs[0][4], 0, g, p, np.zeros_like(p), np.zeros_like(p))
    assert np.array_equal(codes, q1) and np.array_equal(scales, s1)


def _timing_worker(rank, world, port, result_q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [3.0, 5.0][rank]
        t = bench.max_over_ranks(mine, dist, "cpu")
        result_q.put((rank, t, bench.whole_job_rate(1000, world, 10, t)))
    finally:
        dist.destroy_process_group()


def test_bench_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_timing_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    outs = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in outs] == [5.0, 5.0]
    assert outs[0][2] == pytest.approx(2 * 1000 * 10 / 5.0)
