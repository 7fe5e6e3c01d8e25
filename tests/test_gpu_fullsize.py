"""GPU parity at the benchmark sizes, in the launch configuration bench.py times.

The oracle computes sampled query rows one by one (first, last, the rows around
the top-k width, and a seeded spread in between); the CUDA path runs the whole
workload exactly as the benchmark does.  Scores must meet the bf16 / FP8
tolerance and every sampled top-k row must be a valid top-k of the oracle's
scores (tests/parity.py).  Properties that hold at any size are checked on every
row: width and -1 padding, indices unique and visible, and (score order) the
GPU's own scores non-increasing along each row.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import RTOL, assert_scores_close, check_topk_row

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

dsa = pytest.importorskip("sparse_attention_token_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def sample_rows(T, k, n=24, seed=0):
    rng = np.random.default_rng(seed)
    fixed = {0, 1, k - 2, k - 1, k, k + 1, T // 2, T - 2, T - 1}
    rest = set(rng.choice(T, size=n, replace=False).tolist())
    return sorted(r for r in fixed | rest if 0 <= r < T)


def test_prefill_8k_full_size_sampled_rows():
    c = workloads.prefill_8k()
    T, S, K = c.T, c.S, c.topk_limit
    q, k, w = c.q.cuda(), c.k.cuda(), c.w.cuda()
    scores = torch.empty((T, S), dtype=torch.float32, device="cuda")
    topk = torch.empty((T, K), dtype=torch.int32, device="cuda")
    dsa.dsa_indexer_scores(q, k, w, q_pos0=0, scores=scores)
    dsa.dsa_indexer_topk(scores, T=T, S=S, q_pos0=0, topk_limit=K, topk=topk)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    tk = topk.cpu().numpy()
    # properties on every row
    n_vis = np.arange(1, T + 1)
    keep = np.minimum(n_vis, K)
    pad_ok = np.array([np.all(tk[t, keep[t]:] == -1) for t in range(T)])
    assert pad_ok.all()
    sel_ok = np.array([tk[t, :keep[t]].min() >= 0 and tk[t, :keep[t]].max() < n_vis[t] for t in range(T)])
    assert sel_ok.all()
    sc = scores.cpu().numpy()
    for t in range(0, T, 97):
        row = sc[t, tk[t, :keep[t]]]
        assert np.all(np.diff(row) <= 0), t
        assert len(np.unique(tk[t, :keep[t]])) == keep[t]
    # oracle on sampled rows
    rows = sample_rows(T, K)
    rt, rs, rb = oracle.dense(c.q, c.k, c.w, T=T, S=S, H=c.H, D=c.D, q_pos0=0, topk_limit=K, k_out=K,
                              rows=rows, want_scores=True, want_bound=True)
    assert_scores_close(sc[rows][:, :S], rs, rb, RTOL["bf16"], exact=False)
    for i, t in enumerate(rows):
        n = t + 1
        check_topk_row(tk[t], rt[i], rs[i, :n], RTOL["bf16"] * rb[i, :n], n, min(K, n), True)


def test_key_sharded_prefill_8k_full_size_sampled_rows():
    # the benchmark's key-sharded configuration: the 8K prefill's keys in two shards
    # (0..4095, 4096..8191), each shard's (score, global index) candidates, then the merge
    c = workloads.prefill_8k()
    T, S, K = c.T, c.S, c.topk_limit
    q, k, w = c.q.cuda(), c.k.cuda(), c.w.cuda()
    bounds = (0, 4096, 8192)
    cands = [dsa.dsa_indexer_shard_candidates(q, k[b0:b1].contiguous(), w, q_pos0=0, key_offset=b0, k_cand=K)
             for b0, b1 in zip(bounds[:-1], bounds[1:])]
    ci = torch.stack([x[0] for x in cands])
    cs = torch.stack([x[1] for x in cands])
    topk = dsa.dsa_indexer_merge_candidates(cs, ci, topk_limit=K)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    tk = topk.cpu().numpy()
    # properties on every row: width, padding, visibility, uniqueness
    n_vis = np.arange(1, T + 1)
    keep = np.minimum(n_vis, K)
    for t in range(T):
        sel = tk[t, :keep[t]]
        assert np.all(tk[t, keep[t]:] == -1), t
        assert sel.min() >= 0 and sel.max() < n_vis[t], t
        assert len(np.unique(sel)) == keep[t], t
    # oracle on sampled rows
    rows = sample_rows(T, K, seed=2)
    rt, rs, rb = oracle.dense(c.q, c.k, c.w, T=T, S=S, H=c.H, D=c.D, q_pos0=0, topk_limit=K, k_out=K,
                              rows=rows, want_scores=True, want_bound=True)
    for i, t in enumerate(rows):
        n = t + 1
        check_topk_row(tk[t], rt[i], rs[i, :n], RTOL["bf16"] * rb[i, :n], n, min(K, n), True)


def test_chunked_prefill_fp8_full_size_sampled_rows():
    pc = workloads.chunked_prefill_fp8()
    to = lambda t: None if t is None else t.cuda()
    got = dsa.dsa_indexer(to(pc.q), to(pc.w), to(pc.k_cache), to(pc.cu_q_lens), to(pc.seq_lens),
                          to(pc.block_tables), max_seq_len=pc.max_seq_len, topk_limit=pc.topk_limit,
                          q_scale=to(pc.q_scale), k_scale_cache=to(pc.k_scale_cache))
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    tk = got.cpu().numpy()
    assert np.all(tk >= 0)  # every row sees >= 57345 keys: no padding
    rows = sample_rows(pc.total_q, 8, n=8, seed=1)
    rt, rs, rb = oracle.paged(pc, rows=rows, want_scores=True, want_bound=True)
    pos = oracle.query_positions(pc)
    for i, r in enumerate(rows):
        n = int(pos[r]) + 1
        check_topk_row(tk[r], rt[i], rs[i, :n], RTOL["fp8_e4m3"] * rb[i, :n], n, pc.topk_limit, True)


def test_decode_b64_bf16_q_fp8_cache_full_size_sampled_rows():
    pc = workloads.decode_b64_fp8()
    to = lambda t: None if t is None else t.cuda()
    got = dsa.dsa_indexer(to(pc.q), to(pc.w), to(pc.k_cache), to(pc.cu_q_lens), to(pc.seq_lens),
                          to(pc.block_tables), max_seq_len=pc.max_seq_len, topk_limit=pc.topk_limit,
                          q_scale=None, k_scale_cache=to(pc.k_scale_cache))
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    tk = got.cpu().numpy()
    assert np.all(tk >= 0)  # every context holds >= 4096 keys: no padding
    rows = sample_rows(pc.B, 4, n=12, seed=2)
    rt, rs, rb = oracle.paged(pc, rows=rows, want_scores=True, want_bound=True)
    lens = pc.seq_lens.numpy()
    for i, r in enumerate(rows):
        n = int(lens[r])
        check_topk_row(tk[r], rt[i], rs[i, :n], RTOL["bf16"] * rb[i, :n], n, pc.topk_limit, True)


def test_indexshare_stack_full_size_bf16_decode():
    """The IndexShare workload at its full size: 12 layers [full, shared, shared] x 4, decode
    B=32 at 32768 keys, bf16 paged caches.  Each full layer's sampled rows are checked
    against the oracle and every row's width and uniqueness; each shared layer's output is
    its source layer's buffer, bytes and all."""
    sc = workloads.indexshare_stack()
    to = lambda t: None if t is None else t.cuda()
    args, keep = [], []
    for pc in sc.layers:
        if pc is None:
            args.append(None)
            continue
        a, kk = dsa.make_indexer_args(to(pc.q), to(pc.w), to(pc.k_cache), to(pc.cu_q_lens), to(pc.seq_lens),
                                      to(pc.block_tables), max_seq_len=pc.max_seq_len, topk_limit=pc.topk_limit)
        args.append(a)
        keep.append(kk)
    ptrs, src = dsa.dsa_indexer_stack(sc.indexer_types, args)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    assert src == [0, 0, 0, 3, 3, 3, 6, 6, 6, 9, 9, 9]
    outs = {}
    fi = 0
    for l, pc in enumerate(sc.layers):
        if pc is None:
            continue
        out = keep[fi][8]
        fi += 1
        assert ptrs[l] == out.data_ptr()
        outs[l] = out.cpu().numpy()
        tk = outs[l]
        assert tk.shape == (32, 2048) and np.all(tk >= 0) and np.all(tk < 32768)
        assert all(len(np.unique(r)) == 2048 for r in tk)
        rows = sample_rows(pc.B, 4, n=4, seed=10 + l)
        rt, rs, rb = oracle.paged(pc, rows=rows, want_scores=True, want_bound=True)
        for i, r in enumerate(rows):
            check_topk_row(tk[r], rt[i], rs[i, :32768], RTOL["bf16"] * rb[i, :32768], 32768, 2048, True)
    # a shared layer's entry is its source layer's buffer: the same memory, the same bytes
    by_ptr = {kk[8].data_ptr(): kk[8] for kk in keep}
    for l, s in enumerate(src):
        assert ptrs[l] == ptrs[s]
        assert np.array_equal(by_ptr[ptrs[l]].cpu().numpy(), outs[s])
