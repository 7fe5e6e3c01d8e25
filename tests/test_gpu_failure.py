"""Failure detection on the GPU without a GPU fault.

Every wait inside the score kernel is bounded.  dsa_test_arm_score_timeout makes the
next score launch's MMA-issuing thread wait on a barrier that nothing completes, for a
short limit: the wait runs out, the kernel records DSA_ERR_TIMEOUT, every role leaves
its loop, the copies and MMAs already in flight are drained and the tensor memory is
freed.  The tests check that the host reads DSA_ERR_TIMEOUT, that the context stays
usable, and that the next (unarmed) call is bit-exact against the oracle -- on the dense
prefill kernel (one producer) and on the paged decode kernel (two producers, e4m3 keys).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

dsa = pytest.importorskip("sparse_attention_token_gb300")

LIMIT_NS = 2_000_000   # 2 ms: far longer than the copies in flight take to land


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _dense_call(c):
    sc = dsa.dsa_indexer_scores(c.q.cuda(), c.k.cuda(), c.w.cuda(), q_pos0=c.q_pos0)
    tk = dsa.dsa_indexer_topk(sc, T=c.T, S=c.S, q_pos0=c.q_pos0, topk_limit=c.topk_limit)
    return sc, tk


def test_dense_score_wait_times_out_then_recovers():
    c = workloads.dense_case(600, 900, 64, 128, 64, q_pos0=300, integer=True, seed=61)
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    dsa.dsa_test_arm_score_timeout(LIMIT_NS)
    _dense_call(c)
    assert dsa.dsa_check_device_status() == dsa.DSA_ERR_TIMEOUT
    assert dsa.dsa_check_device_status() == dsa.DSA_OK          # the status word was cleared
    sc, tk = _dense_call(c)                                      # the arming was used up
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    rt, rs, _ = oracle.dense(c.q, c.k, c.w, T=c.T, S=c.S, H=c.H, D=c.D, q_pos0=c.q_pos0,
                             topk_limit=c.topk_limit, k_out=c.topk_limit, want_scores=True)
    g = sc.cpu().numpy()[:, :c.S].astype(np.float64)
    vis = np.isfinite(rs)
    assert np.array_equal(g[vis], rs[vis])
    assert np.array_equal(tk.cpu().numpy(), rt)


def test_paged_decode_score_wait_times_out_then_recovers():
    pc = workloads.paged_case([3000, 1800, 700, 65], [1, 1, 1, 1], 64, 128, 256, page_size=64,
                              q_dtype="fp8_e4m3", k_dtype="fp8_e4m3", integer=True, seed=62)
    to = lambda t: None if t is None else t.cuda()
    call = lambda: dsa.dsa_indexer(to(pc.q), to(pc.w), to(pc.k_cache), to(pc.cu_q_lens), to(pc.seq_lens),
                                   to(pc.block_tables), max_seq_len=pc.max_seq_len, topk_limit=pc.topk_limit,
                                   q_scale=to(pc.q_scale), k_scale_cache=to(pc.k_scale_cache))
    dsa.dsa_test_arm_score_timeout(LIMIT_NS)
    call()
    assert dsa.dsa_check_device_status() == dsa.DSA_ERR_TIMEOUT
    got = call()
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    rt = oracle.paged(pc)
    rt = rt[0] if isinstance(rt, tuple) else rt
    assert np.array_equal(got.cpu().numpy(), rt)


def test_disarmed_hook_changes_nothing():
    c = workloads.dense_case(200, 200, 4, 64, 32, q_pos0=0, integer=True, seed=63)
    dsa.dsa_test_arm_score_timeout(LIMIT_NS)
    dsa.dsa_test_arm_score_timeout(0)
    _, tk = _dense_call(c)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    rt = oracle.dense(c.q, c.k, c.w, T=c.T, S=c.S, H=c.H, D=c.D, q_pos0=0, topk_limit=32, k_out=32)
    rt = rt[0] if isinstance(rt, tuple) else rt
    assert np.array_equal(tk.cpu().numpy(), rt)
