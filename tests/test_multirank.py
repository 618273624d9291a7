"""Multi-rank host logic on CPU (gloo, world size 2): the request-sharded run
(every rank its own requests, ids offset by rank * B, no exchange) gives the
same integer outputs as one batch of all ranks' requests, and the step time is
the max over ranks.  The outputs come from the oracle, so no GPU is needed."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from draft_sampling_verification_gb300 import workloads as W

WORLD = 2
B = 3
V = 301


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _requests(wl, req_ids):
    """Oracle outputs (tokens, greedy and ratio accept lengths / committed) of
    the workload's requests under the given request ids."""
    from oracle import oracle as O
    depth = wl.depth
    x = wl.draft.reshape(wl.B * depth, wl.V)
    counts, ids, nnz, st = O.q_build(x, wl.temperature, wl.top_k)
    tok, _ = O.draft_sample(counts, ids, nnz, wl.top_k, wl.B, depth, wl.seed, req_ids, V=wl.V)
    drafts = tok.reshape(wl.B, depth)
    z = wl.target_f32()
    g = O.verify_greedy(z, drafts)
    r = O.verify_ratio(z, drafts, counts, ids, nnz, wl.top_k, wl.seed, req_ids)
    return (np.asarray(tok), np.asarray(g[0]), np.asarray(g[1]), np.asarray(r[0]),
            np.asarray(r[1]))


def _worker(rank, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        wl = W.config1(B=B, V=V)
        req = bench.rank_request_ids(wl.request_ids, rank, B)
        res = _requests(wl, req)
        gathered = [None] * WORLD
        dist.all_gather_object(gathered, [a.tolist() for a in res])
        t = bench.max_over_ranks(torch.tensor([1.0 + rank, 5.0 - rank], dtype=torch.float64))
        if rank == 0:
            out.put((gathered, t.tolist()))
    finally:
        dist.destroy_process_group()


def test_request_sharding_matches_one_batch():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    gathered, tmax = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert tmax == [2.0, 5.0]
    # one batch of WORLD * B requests: the same rows repeated per rank, ids 0..WORLD*B-1
    wl = W.config1(B=B, V=V)
    big = W.config1(B=B, V=V)
    big.B = WORLD * B
    big.draft = np.concatenate([wl.draft] * WORLD)
    big.target = np.concatenate([wl.target] * WORLD)
    big.temperature = np.concatenate([wl.temperature] * WORLD)
    big.request_ids = np.arange(WORLD * B, dtype=np.uint32)
    ref = _requests(big, big.request_ids)
    for rank in range(WORLD):
        for k, name in enumerate(["tokens", "greedy_len", "greedy_committed", "ratio_len",
                                  "ratio_committed"]):
            part = np.asarray(gathered[rank][k])
            whole = ref[k].reshape((WORLD, -1) + ref[k].shape[1:])[rank].reshape(part.shape)
            assert np.array_equal(part, whole), (rank, name)
    # the ranks' draws differ (their request ids do)
    assert not np.array_equal(np.asarray(gathered[0][0]), np.asarray(gathered[1][0]))
