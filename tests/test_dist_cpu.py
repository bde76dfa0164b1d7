"""Two-rank (gloo, CPU) checks of the multi-GPU host logic: the expert-parallel
partition of the routing, the sum of the ranks' partial layer outputs, and the
max-over-ranks timing reduction used by bench.py."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

WORLD = 2
GLOBAL = wl.Workload("ep2_T24_E8_top2_H256_I128", T=24, E=8, E_global=8, topk=2, H=256, I=128,
                     routing="softmax", seed=11)
SHARE = wl.Workload("ep2_T24_E4of8_top2_H256_I128", T=24, E=4, E_global=8, topk=2, H=256, I=128,
                    routing="softmax", seed=11)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import oracle
        import bench
        ids, wts = wl.make_routing(SHARE, rank)
        x = wl.make_x(GLOBAL)
        c13, s13 = wl.make_w13(GLOBAL)
        c2, s2 = wl.make_w2(GLOBAL)
        lo = rank * SHARE.E
        w13 = (c13[lo:lo + SHARE.E], s13[lo:lo + SHARE.E])
        w2 = (c2[lo:lo + SHARE.E], s2[lo:lo + SHARE.E])
        part = oracle.moe_layer(x, ids, wts, w13, w2, SHARE.E, block_m=8)
        part32 = torch.from_numpy(wl.bf16_bits_to_f32(part).astype(np.float32))
        dist.all_reduce(part32, op=dist.ReduceOp.SUM)
        counts = torch.tensor([int((ids >= 0).sum())], dtype=torch.int64)
        dist.all_reduce(counts, op=dist.ReduceOp.SUM)
        mx = bench.reduce_max([1.0 + rank, 10.0 - rank], dist, "cpu")
        if rank == 0:
            np.save(os.path.join(out_dir, "sum.npy"), part32.numpy())
            np.save(os.path.join(out_dir, "meta.npy"), np.array([counts.item(), mx[0], mx[1]]))
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_rank_result(tmp_path_factory):
    import oracle
    oracle.build()
    out = tmp_path_factory.mktemp("dist")
    mp.start_processes(_worker, args=(_free_port(), str(out)), nprocs=WORLD, start_method="spawn")
    return np.load(out / "sum.npy"), np.load(out / "meta.npy")


def test_partition_covers_every_pair_once():
    full, _ = wl.make_routing(GLOBAL)
    shares = [wl.make_routing(SHARE, r)[0] for r in range(WORLD)]
    owner = np.full(full.shape, -1)
    for r, ids in enumerate(shares):
        hit = ids >= 0
        assert (owner[hit] == -1).all(), "a pair is local to two ranks"
        owner[hit] = r
        assert (ids[hit] + r * SHARE.E == full[hit]).all()
    assert (owner >= 0).all() and (owner == full // SHARE.E).all()


def test_rank_partials_sum_to_full_layer(two_rank_result):
    import oracle
    summed, meta = two_rank_result
    ids, wts = wl.make_routing(GLOBAL)
    assert meta[0] == int((ids >= 0).sum()) == GLOBAL.T * GLOBAL.topk
    full = oracle.moe_layer(wl.make_x(GLOBAL), ids, wts, wl.make_w13(GLOBAL), wl.make_w2(GLOBAL), GLOBAL.E,
                            block_m=8)
    ref = wl.bf16_bits_to_f32(full).astype(np.float64)
    # each rank rounds its partial to BF16 once; the full layer rounds once
    err = np.abs(summed.astype(np.float64) - ref)
    assert (err <= 1e-2 + 1e-2 * np.abs(ref)).all(), float(err.max())


def test_reduce_max_takes_the_slowest_rank(two_rank_result):
    _, meta = two_rank_result
    assert meta[1] == 2.0 and meta[2] == 10.0
