"""The multi-rank side of all-reduce + RMSNorm, on CPU with gloo ranks
(world size 2): every rank contributes its partial tensor, the ranks
exchange them, each reduces and normalises its own slice of the rows
(row_slice: the two-shot split) through the oracle, and the gathered slices
must equal the one-shot result over all rows.  The partition arithmetic is
checked for many sizes.  (The kernel itself is covered on one GPU by
tests/test_gpu_allreduce.py, with the ranks emulated as separate buffers.)
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri

N, H, MODE = 23, 512, "fp8_per_token"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    wl = ri.make_workload("ar_host", N, H, res_sigma=1.5, seed=61)
    return wl


def _partial(rank):
    return ri.to_bits(ri.normal(300 + rank, 1, N * H), "bf16").reshape(N, H)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = _inputs()
        mine = torch.from_numpy(_partial(rank).view(np.int32).copy())      # bf16 pairs as int32 words
        gathered = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(gathered, mine)                         # the exchange of the all-reduce
        parts = np.stack([g.numpy().view(np.uint16) for g in gathered])
        b, e = rq.row_slice(N, world, rank)
        r = oracle.run_allreduce(parts[:, b:e], wl.residual[b:e], wl.weight, eps=wl.eps, mode=MODE)
        rows = -(-N // world)
        q = np.zeros((rows, H), np.uint8)
        q[: e - b] = r["q"]
        sc = np.zeros(rows, np.float32)
        sc[: e - b] = r["scales"]
        qs = [torch.empty(rows, H // 4, dtype=torch.int32) for _ in range(world)]
        ss = [torch.empty(rows, dtype=torch.float32) for _ in range(world)]
        dist.all_gather(qs, torch.from_numpy(q.view(np.int32).copy()))   # the gather of the two-shot scheme
        dist.all_gather(ss, torch.from_numpy(sc))
        full_q = np.concatenate([qs[k].numpy().view(np.uint8)[: rq.row_slice(N, world, k)[1] - rq.row_slice(N, world, k)[0]]
                                 for k in range(world)])
        full_s = np.concatenate([ss[k].numpy()[: rq.row_slice(N, world, k)[1] - rq.row_slice(N, world, k)[0]]
                                 for k in range(world)])
        out[rank] = (full_q.tobytes(), full_s.tobytes())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_shot_over_gloo_ranks_equals_one_shot():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    wl = _inputs()
    parts = np.stack([_partial(r) for r in range(world)])
    want = oracle.run_allreduce(parts, wl.residual, wl.weight, eps=wl.eps, mode=MODE)
    for r in range(world):
        q, s = out[r]
        assert q == want["q"].tobytes()
        assert s == want["scales"].tobytes()


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_row_slices_cover_the_batch(world):
    for n in (0, 1, 2, 7, 8, 103, 4096):
        spans = [rq.row_slice(n, world, r) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == n
        for (b0, e0), (b1, e1) in zip(spans, spans[1:]):
            assert e0 == b1
        sizes = [e - b for b, e in spans]
        assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 0
    with pytest.raises(ValueError):
        rq.row_slice(4, 2, 2)
