"""Key-sharded top-k on one GPU: the shards of one sequence's keys are scored one after
another (virtual shards), each keeps its (score, global index) candidates, and the merge
kernel keeps the best of their union.

Integer-valued inputs make every score exact in fp32, so the candidates must equal the
oracle's per-shard candidates and the merged top-k the oracle's full-row top-k, bit for
bit, including ties that straddle shard boundaries (small integer ranges give many equal
scores).  Gaussian inputs must give a valid top-k of the oracle's scores within the bf16
tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import sharded
from tests.parity import RTOL, check_topk_row

pytestmark = pytest.mark.gpu

dsa = pytest.importorskip("sparse_attention_token_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _run_shards(c, bounds, k_cand, order=0, topk_limit=None):
    q, w = c.q.cuda(), c.w.cuda()
    qs = None if c.q_scale is None else c.q_scale.cuda()
    idx, sc = [], []
    for b0, b1 in zip(bounds[:-1], bounds[1:]):
        ks = None if c.k_scale is None else c.k_scale[b0:b1].contiguous().cuda()
        ci, cs = dsa.dsa_indexer_shard_candidates(q, c.k[b0:b1].contiguous().cuda(), w, q_pos0=c.q_pos0,
                                                  key_offset=b0, k_cand=k_cand, q_scale=qs, k_scale=ks)
        idx.append(ci)
        sc.append(cs)
    all_idx, all_sc = torch.stack(idx), torch.stack(sc)
    lim = k_cand if topk_limit is None else topk_limit
    out = dsa.dsa_indexer_merge_candidates(all_sc, all_idx, topk_limit=lim, k_out=lim + 5, order=order)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    return all_idx.cpu().numpy(), all_sc.cpu().numpy(), out.cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("bounds", [[0, 1000], [0, 250, 251, 640, 1000], [0, 128, 256, 384, 1000],
                                    [0, 999, 1000], [0, 500, 1000], [0, 3, 1000]])
def test_sharded_integer_exact(dtype, bounds):
    T, S, K, q_pos0 = 300, 1000, 128, 700
    c = workloads.dense_case(T, S, 64, 128, K, q_pos0=q_pos0, dtype=dtype, integer=True, int_range=(-2, 2),
                             w_int_range=(-1, 1), seed=80 + len(bounds))
    ci, cs, got = _run_shards(c, bounds, K)
    rt, rs, _ = oracle.dense(c.q, c.k, c.w, T=T, S=S, H=64, D=128, q_pos0=q_pos0, topk_limit=K, k_out=K + 5,
                             q_scale=c.q_scale, k_scale=c.k_scale, want_scores=True)
    n_vis = np.minimum(q_pos0 + np.arange(T) + 1, S)
    for j, (b0, b1) in enumerate(zip(bounds[:-1], bounds[1:])):
        ocs, oci = sharded.shard_candidates(rs, n_vis, b0, b1 - b0, K)
        assert np.array_equal(ci[j], oci), f"shard {j} indices"
        assert np.array_equal(cs[j].astype(np.float64), ocs), f"shard {j} scores"
    assert np.array_equal(got, rt)
    # the same set in ascending key order
    _, _, got_ix = _run_shards(c, bounds, K, order=1)
    rt_ix = oracle.dense(c.q, c.k, c.w, T=T, S=S, H=64, D=128, q_pos0=q_pos0, topk_limit=K, k_out=K + 5,
                         q_scale=c.q_scale, k_scale=c.k_scale, order=oracle.ORDER_INDEX)[0]
    assert np.array_equal(got_ix, rt_ix)


def test_sharded_rows_that_see_no_shard_keys_and_short_rows():
    # queries at 0..199 against keys split at 150: early rows see nothing of the second shard,
    # and rows with fewer visible keys than k are padded with -1
    T, S, K = 200, 400, 64
    c = workloads.dense_case(T, S, 16, 128, K, q_pos0=0, integer=True, seed=91)
    ci, cs, got = _run_shards(c, [0, 150, 400], K)
    assert np.all(ci[1][:150] == -1) and np.all(np.isinf(cs[1][:150]))
    rt = oracle.dense(c.q, c.k, c.w, T=T, S=S, H=16, D=128, q_pos0=0, topk_limit=K, k_out=K + 5)[0]
    assert np.array_equal(got, rt)


@pytest.mark.parametrize("bounds", [[0, 700, 1500, 2300, 3000], [0, 1400, 3000]])
def test_sharded_gaussian_valid_topk(bounds):
    T, S, K, q_pos0 = 256, 3000, 512, 2744
    c = workloads.dense_case(T, S, 64, 128, K, q_pos0=q_pos0, seed=92)
    _, _, got = _run_shards(c, bounds, K)
    rt, rs, rb = oracle.dense(c.q, c.k, c.w, T=T, S=S, H=64, D=128, q_pos0=q_pos0, topk_limit=K, k_out=K + 5,
                              want_scores=True, want_bound=True)
    for t in range(T):
        n = q_pos0 + t + 1
        check_topk_row(got[t], rt[t], rs[t, :n], RTOL["bf16"] * rb[t, :n], n, K, True)


def test_merge_rejects_bad_arguments_before_launch():
    ci = torch.full((2, 4, 8), -1, dtype=torch.int32, device="cuda")
    cs = torch.full((2, 4, 8), float("-inf"), dtype=torch.float32, device="cuda")
    with pytest.raises(dsa.DsaError):
        dsa.dsa_indexer_merge_candidates(cs, ci, topk_limit=0)
    big_i = torch.full((3, 1, 8192), -1, dtype=torch.int32, device="cuda")
    big_s = torch.zeros((3, 1, 8192), dtype=torch.float32, device="cuda")
    with pytest.raises(dsa.DsaError):   # 3 x 8192 candidates exceed the 16384 a row may hold
        dsa.dsa_indexer_merge_candidates(big_s, big_i, topk_limit=8)
    out = dsa.dsa_indexer_merge_candidates(cs, ci, topk_limit=4)      # nothing valid: all -1
    torch.cuda.synchronize()
    assert np.all(out.cpu().numpy() == -1)
