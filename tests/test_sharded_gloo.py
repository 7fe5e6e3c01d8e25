"""The candidate exchange of the key-sharded top-k on CPU: two gloo ranks, no GPU.

Each rank holds one contiguous shard of a sequence's keys and computes that shard's
(score, global index) candidates (with the oracle here, since CPU ranks run no kernels);
``gather_shard_candidates`` -- the library's exchange step -- all-gathers them in rank
order; merging the gathered lists must give the full-row top-k, and every rank must see
the same gathered tensors.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CASE = dict(T=48, S=90, H=4, D=64, topk=10, q_pos0=42, seed=95)
BOUNDS = [0, 37, 90]   # rank r holds keys BOUNDS[r] .. BOUNDS[r + 1] - 1


def _case():
    import oracle
    import workloads
    c = workloads.dense_case(CASE["T"], CASE["S"], CASE["H"], CASE["D"], CASE["topk"], q_pos0=CASE["q_pos0"],
                             integer=True, int_range=(-1, 1), w_int_range=(-1, 1), seed=CASE["seed"])
    rt, rs, _ = oracle.dense(c.q, c.k, c.w, T=c.T, S=c.S, H=c.H, D=c.D, q_pos0=c.q_pos0, topk_limit=CASE["topk"],
                             k_out=CASE["topk"], want_scores=True)
    n_vis = np.minimum(c.q_pos0 + np.arange(c.T) + 1, c.S)
    return rt, rs, n_vis


def _rank_main(rank: int, world: int, port: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import sparse_attention_token_gb300 as dsa
    from oracle import sharded
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rt, rs, n_vis = _case()
        b0, b1 = BOUNDS[rank], BOUNDS[rank + 1]
        cs, ci = sharded.shard_candidates(rs, n_vis, b0, b1 - b0, CASE["topk"])
        all_idx, all_sc = dsa.gather_shard_candidates(torch.from_numpy(ci), torch.from_numpy(cs.astype(np.float32)))
        merged = sharded.merge_candidates(all_sc.numpy().astype(np.float64), all_idx.numpy(), CASE["topk"],
                                          CASE["topk"])
        out[rank] = (all_idx.numpy().tolist(), merged.tolist(), rt.tolist(), ci.tolist())
    finally:
        dist.destroy_process_group()


def test_gather_shard_candidates_two_gloo_ranks():
    world = 2
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    g0, m0, rt, c0 = res[0]
    g1, m1, _, c1 = res[1]
    assert g0 == g1                      # every rank sees the same gathered candidates
    assert g0[0] == c0 and g0[1] == c1   # in rank order
    assert m0 == m1 == rt                # and their merge is the full-row top-k
