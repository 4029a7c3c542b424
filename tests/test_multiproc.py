"""The multi-GPU path's host logic with world_size 2 on the CPU (gloo): each
process of a run gets its own shard of episodes (distinct LCG seeds and start
bars, the same features and weights: replicas of one policy over one market,
no exchange on the data path) and the timing is the maximum over ranks."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from rl_experience_collection_gb300 import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    try:
        os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                          LOCAL_RANK=str(rank))
        import torch
        import bench
        r, ws, dist = bench.dist_setup("gloo")
        assert (r, ws) == (rank, world)
        w = wl.WORKLOADS["tiny_fp32"]
        inp = wl.generate(w, shard=r)
        digest = lambda a: float(np.asarray(a, np.float64).sum())
        mine = torch.tensor([digest(inp.features), digest(inp.weights), digest(inp.seeds), digest(inp.starts)],
                            dtype=torch.float64)
        allv = [torch.zeros(4, dtype=torch.float64) for _ in range(ws)]
        dist.all_gather(allv, mine)
        seeds = torch.from_numpy(inp.seeds.astype(np.int64))
        all_seeds = [torch.zeros_like(seeds) for _ in range(ws)]
        dist.all_gather(all_seeds, seeds)
        t = bench.max_over_ranks(10.0 + r, dist, "cpu")
        dist.barrier()
        dist.destroy_process_group()
        q.put((r, [v.tolist() for v in allv], [s.tolist() for s in all_seeds], t))
    except Exception as e:                      # reported to the parent, which fails the test
        q.put((rank, repr(e), None, None))


def test_two_ranks_shard_episodes_and_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res = dict((r[0], r[1:]) for r in res)
    for r in (0, 1):
        assert not isinstance(res[r][0], str), res[r][0]
    digests, seeds, tmax = res[0]
    assert digests[0][0] == digests[1][0] and digests[0][1] == digests[1][1]     # same features, same weights
    assert digests[0][2] != digests[1][2] and digests[0][3] != digests[1][3]     # own seeds and starts
    assert not set(seeds[0]) & set(seeds[1])                                     # no episode twice
    assert tmax == 11.0 and res[1][2] == 11.0                                    # the max over ranks
    # shard 0 is the workload's own draw; shard 1's seeds continue the global episode index
    w = wl.WORKLOADS["tiny_fp32"]
    np.testing.assert_array_equal(wl.generate(w).starts, wl.generate(w, shard=0).starts)
    np.testing.assert_array_equal(wl.generate(w, shard=1).seeds, wl.episode_seeds(w.seed, 2 * w.n_episodes)[w.n_episodes:])
