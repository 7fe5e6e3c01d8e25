"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Integer-valued inputs (fp32 accumulation exact) must match bit for bit, scores and
indices including their order; Gaussian inputs must meet the tolerances of
tests/parity.py.  Shapes span several 128-key tiles, ragged tails, every supported
head count, both top-k orders, dense and paged keys, bf16 and FP8.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import RTOL, assert_scores_close, assert_topk_valid

pytestmark = pytest.mark.gpu

dsa = pytest.importorskip("sparse_attention_token_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    yield
    assert dsa.dsa_check_device_status() == dsa.DSA_OK


DEV = "cuda"


def run_dense(c, order=0, topk_limit=None, k_out=None):
    topk_limit = c.topk_limit if topk_limit is None else topk_limit
    k_out = c.k_out if k_out is None else k_out
    q, k, w = c.q.to(DEV), c.k.to(DEV), c.w.to(DEV)
    qs = None if c.q_scale is None else c.q_scale.to(DEV)
    ks = None if c.k_scale is None else c.k_scale.to(DEV)
    sc = dsa.dsa_indexer_scores(q, k, w, q_pos0=c.q_pos0, q_scale=qs, k_scale=ks)
    tk = dsa.dsa_indexer_topk(sc, T=c.T, S=c.S, q_pos0=c.q_pos0, topk_limit=topk_limit, k_out=k_out,
                              order=order)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    return sc.cpu().numpy(), tk.cpu().numpy()


def oracle_dense(c, order=0, topk_limit=None, k_out=None, rows=None):
    return oracle.dense(c.q, c.k, c.w, T=c.T, S=c.S, H=c.H, D=c.D, q_pos0=c.q_pos0,
                        topk_limit=c.topk_limit if topk_limit is None else topk_limit,
                        k_out=c.k_out if k_out is None else k_out, q_scale=c.q_scale, k_scale=c.k_scale,
                        order=order, rows=rows, want_scores=True, want_bound=True)


def n_vis_dense(c, rows=None):
    rows = range(c.T) if rows is None else rows
    return [max(0, min(c.q_pos0 + t + 1, c.S)) for t in rows]


# ----------------------------------------------------------------------------- dense

@pytest.mark.parametrize("order", [0, 1])
def test_tiny_exact_prefill_bit_exact(order):
    c = workloads.tiny_exact_prefill()
    sc, tk = run_dense(c, order=order)
    rt, rs, rb = oracle_dense(c, order=order)
    assert_scores_close(sc[:, :c.S], rs, rb, 0, exact=True)
    assert np.array_equal(tk, rt)


@pytest.mark.parametrize("H,D", [(4, 64), (8, 128), (16, 64), (32, 128), (64, 128), (128, 128), (64, 64)])
def test_dense_integer_exact_all_heads(H, D):
    T, S = 77, 301                 # ragged: 3 key tiles, partial query block
    c = workloads.dense_case(T, S, H, D, 40, q_pos0=S - T, k_out=45, integer=True, int_range=(-2, 2),
                             seed=H + D)
    sc, tk = run_dense(c)
    rt, rs, rb = oracle_dense(c)
    assert_scores_close(sc[:, :S], rs, rb, 0, exact=True)
    assert np.array_equal(tk, rt)


@pytest.mark.parametrize("q_pos0,T,S", [(0, 300, 300), (0, 40, 300), (500, 64, 300), (130, 1, 129)])
def test_dense_positions_and_padding(q_pos0, T, S):
    c = workloads.dense_case(T, S, 64, 128, 100, q_pos0=q_pos0, k_out=128, integer=True, int_range=(-2, 2),
                             seed=3)
    sc, tk = run_dense(c)
    rt, rs, rb = oracle_dense(c)
    assert_scores_close(sc[:, :S], rs, rb, 0, exact=True)
    assert np.array_equal(tk, rt)
    # entries no query may see are not written (the binding pre-fills -inf)
    for t in range(T):
        n = min(q_pos0 + t + 1, S)
        assert np.all(np.isneginf(sc[t, n:S]))


def test_dense_gaussian_bf16_tolerance():
    c = workloads.dense_case(260, 700, 64, 128, 96, q_pos0=440, seed=5, w_std=1 / 8)
    sc, tk = run_dense(c)
    rt, rs, rb = oracle_dense(c)
    assert_scores_close(sc[:, :c.S], rs, rb, RTOL["bf16"], exact=False)
    assert_topk_valid(tk, rt, rs, rb, n_vis_dense(c), c.topk_limit, RTOL["bf16"], exact=False)


def test_dense_fp8_integer_exact():
    c = workloads.dense_case(70, 400, 64, 128, 50, q_pos0=330, dtype="fp8_e4m3", integer=True,
                             int_range=(-3, 3), seed=6)
    sc, tk = run_dense(c)
    rt, rs, rb = oracle_dense(c)
    assert_scores_close(sc[:, :c.S], rs, rb, 0, exact=True)
    assert np.array_equal(tk, rt)


def test_dense_fp8_gaussian_tolerance():
    c = workloads.dense_case(130, 500, 64, 128, 64, q_pos0=370, dtype="fp8_e4m3", seed=7, w_std=1 / 8)
    sc, tk = run_dense(c)
    rt, rs, rb = oracle_dense(c)
    assert_scores_close(sc[:, :c.S], rs, rb, RTOL["fp8_e4m3"], exact=False)
    assert_topk_valid(tk, rt, rs, rb, n_vis_dense(c), c.topk_limit, RTOL["fp8_e4m3"], exact=False)


def test_dense_deterministic():
    c = workloads.dense_case(128, 1000, 64, 128, 256, q_pos0=872, seed=8)
    a = run_dense(c)
    b = run_dense(c)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ----------------------------------------------------------------------------- top-k alone

def _topk_on(scores32: np.ndarray, q_pos0: int, S: int, limit: int, k_out: int, order: int):
    T = scores32.shape[0]
    ld = (S + 3) // 4 * 4
    buf = torch.full((T, ld), float("nan"), dtype=torch.float32)
    buf[:, :S] = torch.from_numpy(scores32)
    tk = dsa.dsa_indexer_topk(buf.to(DEV), T=T, S=S, q_pos0=q_pos0, topk_limit=limit, k_out=k_out, order=order)
    torch.cuda.synchronize()
    nv = [max(0, min(q_pos0 + t + 1, S)) for t in range(T)]
    ref = oracle.topk_of_scores(scores32.astype(np.float64), nv, limit, k_out, order=order)
    return tk.cpu().numpy(), ref


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("S,limit", [(5000, 2048), (20000, 2048), (70000, 4096), (3000, 3000), (9000, 1)])
def test_topk_tie_storms_exact(S, limit, order):
    g = torch.Generator().manual_seed(S + limit)
    T = 6
    sc = torch.randint(-3, 4, (T, S), generator=g).to(torch.float32).numpy()
    sc[1] = 0.0
    sc[2, ::2] = -0.0                       # -0.0 and +0.0 are equal
    sc[3] = np.arange(S, dtype=np.float32)  # strictly increasing: the last keys win
    got, ref = _topk_on(sc, S - T, S, limit, min(limit + 5, 4096), order)
    assert np.array_equal(got, ref)


# row lengths on every kernel: one CTA (<= 8192 keys), clusters of 4 CTAs of 8192 and of
# 16384 keys, clusters of 8, and the streaming kernel beyond 131072 keys
@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("S", [100, 2049, 8192, 16385, 40000, 65536, 100000, 140000])
def test_topk_gaussian_exact(S, order):
    g = torch.Generator().manual_seed(S)
    T = 4
    sc = torch.randn((T, S), generator=g).numpy().astype(np.float32)
    got, ref = _topk_on(sc, S - T, S, 2048, 2048, order)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("S,step", [(3000, 0.05), (8192, 0.02), (30000, 0.01), (8192, 1e-6)])
def test_topk_quantised_scores_exact(S, step, order):
    # values on a grid: tens of equal keys per value, both signs, so the score-order sort
    # meets buckets of 8..64 keys (and, for the coarse grids, more), plus near-zero values
    g = torch.Generator().manual_seed(int(S / step) % 100003)
    T = 5
    sc = (torch.round(torch.randn((T, S), generator=g) / step) * step).numpy().astype(np.float32)
    sc[4, ::3] *= 1e-30
    got, ref = _topk_on(sc, S - T, S, 2048, 2048, order)
    assert np.array_equal(got, ref)


# the linear-bucket paths' limits: few huge outliers (nearly every key in the lowest
# bucket), an infinite score (no finite width), one distinct value among equal ones, a
# heavy tail, and widths of keep from 1 to near the candidate buffer of the cluster form
@pytest.mark.parametrize("kind", ["outliers", "inf", "one_distinct", "heavy_tail"])
@pytest.mark.parametrize("S,limit", [(5000, 1), (5000, 2048), (30000, 64), (30000, 3900), (100000, 2048)])
def test_topk_linear_bucket_edges_exact(kind, S, limit):
    g = torch.Generator().manual_seed(S * 7 + limit)
    T = 3
    sc = torch.randn((T, S), generator=g).numpy().astype(np.float32)
    if kind == "outliers":
        sc[:, ::997] = 1e30
    elif kind == "inf":
        sc[0, S // 2] = np.inf
        sc[1, 3] = -np.inf
        sc[2, -1] = np.inf
    elif kind == "one_distinct":
        sc[:] = 1.5
        sc[:, S // 3] = 2.0
    else:
        sc = np.exp(4.0 * sc).astype(np.float32)
    got, ref = _topk_on(sc, S - T, S, limit, min(limit + 3, 4096), 0)
    assert np.array_equal(got, ref)


# many rows longer than one CTA's registers hold (more rows than half the SMs): one CTA
# streams each row from memory, linear buckets in score order with the general path for the
# rows they decline, and the general path in index order
@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("kind,S,limit", [("gaussian", 20000, 2048), ("gaussian", 70000, 2048),
                                          ("gaussian", 9000, 1), ("heavy_tail", 30000, 3900),
                                          ("outliers", 20000, 2048), ("one_distinct", 12000, 2048),
                                          ("quantised", 20000, 2048), ("ties", 20000, 64),
                                          ("sampled_runs_high", 20000, 2048)])
def test_topk_many_long_rows_exact(kind, S, limit, order):
    g = torch.Generator().manual_seed(S * 13 + limit + len(kind))
    T = 120
    sc = torch.randn((T, S), generator=g).numpy().astype(np.float32)
    if kind == "heavy_tail":
        sc = np.exp(4.0 * sc).astype(np.float32)
    elif kind == "outliers":
        sc[:, ::997] = 1e30
        sc[7, 11] = np.inf
    elif kind == "one_distinct":
        sc[:] = -0.75
        sc[:, S // 5] = 0.5
    elif kind == "quantised":
        sc = (np.round(sc / 0.01) * 0.01).astype(np.float32)
    elif kind == "ties":
        sc = np.round(sc).astype(np.float32)
        sc[3] = 0.0
        sc[4, ::2] = -0.0
    elif kind == "sampled_runs_high":
        # the 32 runs of 128 keys that the one-pass selection samples sit far above the
        # rest of the row, so the threshold it takes from them keeps too few keys and the
        # row is read again in three passes
        for t in range(T):
            n = S - T + t + 1
            for r in range(32):
                o = ((n - 128) * r // 31) & ~3
                sc[t, o:o + 128] += 10.0
    got, ref = _topk_on(sc, S - T, S, limit, min(limit + 3, 4096), order)
    assert np.array_equal(got, ref)


def test_topk_causal_rows_prefill_shape():
    g = torch.Generator().manual_seed(1)
    T = S = 3000
    sc = torch.randn((T, S), generator=g).numpy().astype(np.float32)
    got, ref = _topk_on(sc, 0, S, 2048, 2048, 0)
    assert np.array_equal(got, ref)


# ----------------------------------------------------------------------------- paged

def run_paged(pc, order=0, topk_limit=None, k_out=None):
    to = lambda t: None if t is None else t.to(DEV)
    tk = dsa.dsa_indexer(to(pc.q), to(pc.w), to(pc.k_cache), to(pc.cu_q_lens), to(pc.seq_lens),
                         to(pc.block_tables), max_seq_len=pc.max_seq_len,
                         topk_limit=pc.topk_limit if topk_limit is None else topk_limit,
                         k_out=pc.k_out if k_out is None else k_out, q_scale=to(pc.q_scale),
                         k_scale_cache=to(pc.k_scale_cache), order=order)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    return tk.cpu().numpy()


@pytest.mark.parametrize("page_size", [16, 64, 128])
def test_paged_decode_integer_exact(page_size):
    lens = [1, 63, 64, 65, 129, 1000, 2047, 3000]
    pc = workloads.paged_case(lens, [1] * len(lens), 64, 128, 512, page_size=page_size, integer=True, seed=9)
    got = run_paged(pc)
    ref, _, _ = oracle.paged(pc)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("H", [4, 32, 64, 128])
def test_paged_decode_heads(H):
    lens = [700, 5, 1300]
    pc = workloads.paged_case(lens, [1, 1, 1], H, 128, 256, page_size=64, integer=True, seed=10 + H)
    got = run_paged(pc)
    ref, _, _ = oracle.paged(pc)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("H,k_dtype", [(16, "bf16"), (64, "bf16"), (32, "fp8_e4m3")])
def test_paged_decode_balanced_lists(H, k_dtype):
    # decode-shaped batches (total_q <= B) run on balanced per-CTA work lists: each CTA's
    # equal share of key tiles crosses query blocks and sequences; sequences without a
    # query, several queries per sequence (one block of NQ, or split e4m3 rows per query)
    lens = [(i * 997) % 4999 + 1 for i in range(45)] + [1, 2, 127, 128, 129]
    qlens = [min([1, 0, 2, 1, 0, 1][i % 6], L) for i, L in enumerate(lens)]
    assert sum(qlens) <= len(lens)
    pc = workloads.paged_case(lens, qlens, H, 128, 300, page_size=32, integer=True, seed=70 + H,
                              q_dtype="bf16", k_dtype=k_dtype)
    for order in (0, 1):
        got = run_paged(pc, order=order)
        ref, _, _ = oracle.paged(pc, order=order)
        assert np.array_equal(got, ref)


def test_paged_decode_balanced_many_short():
    # 120 short sequences (1..300 keys): most CTAs' shares are one or two tiles
    lens = [(i * 37) % 300 + 1 for i in range(120)]
    pc = workloads.paged_case(lens, [1] * len(lens), 64, 128, 64, page_size=16, integer=True, seed=77)
    got = run_paged(pc)
    ref, _, _ = oracle.paged(pc)
    assert np.array_equal(got, ref)


def test_paged_decode_many_mixed_lengths_streamed_exact():
    # 100 decode rows from 1 to 30000 keys in one launch: more rows than half the SMs and
    # rows beyond 8192 keys, so every row streams through one CTA -- rows shorter than
    # keep, rows kept whole by the one-pass selection, and sampled rows side by side
    lens = [(i * 7919) % 30000 + 1 for i in range(88)] + [1, 2, 2047, 2048, 2049, 4608, 4609, 6144,
                                                          8192, 8193, 12000, 30000]
    pc = workloads.paged_case(lens, [1] * len(lens), 16, 128, 2048, page_size=64, k_out=2051,
                              integer=True, seed=78)
    for order in (0, 1):
        got = run_paged(pc, order=order)
        ref, _, _ = oracle.paged(pc, order=order)
        assert np.array_equal(got, ref)


def test_paged_varlen_prefill_integer_exact():
    lens, qlens = [900, 40, 1500, 300], [300, 40, 17, 1]
    pc = workloads.paged_case(lens, qlens, 64, 128, 128, page_size=64, integer=True, seed=11)
    for order in (0, 1):
        got = run_paged(pc, order=order)
        ref, _, _ = oracle.paged(pc, order=order)
        assert np.array_equal(got, ref)


def test_paged_fp8_integer_exact():
    lens, qlens = [1000, 257, 64], [3, 257, 1]
    pc = workloads.paged_case(lens, qlens, 64, 128, 200, page_size=64, q_dtype="fp8_e4m3",
                              k_dtype="fp8_e4m3", integer=True, seed=12)
    got = run_paged(pc)
    ref, _, _ = oracle.paged(pc)
    assert np.array_equal(got, ref)


def test_paged_fp8_gaussian_tolerance():
    lens, qlens = [3000, 1200], [1, 200]
    pc = workloads.paged_case(lens, qlens, 64, 128, 300, page_size=64, q_dtype="fp8_e4m3",
                              k_dtype="fp8_e4m3", w_std=1 / 8, seed=13)
    got = run_paged(pc)
    ref, rs, rb = oracle.paged(pc, want_scores=True, want_bound=True)
    pos = oracle.query_positions(pc)
    assert_topk_valid(got, ref, rs, rb, pos + 1, pc.topk_limit, RTOL["fp8_e4m3"], exact=False)

# --------------------------------------------------- bf16 queries, e4m3 paged cache

@pytest.mark.parametrize("page_size", [16, 64])
def test_mixed_decode_every_e4m3_code_exact(page_size):
    pc = workloads.e4m3_code_sweep_decode(seed=40 + page_size, page_size=page_size)
    for order in (0, 1):
        got = run_paged(pc, order=order)
        ref, _, _ = oracle.paged(pc, order=order)
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("H", [4, 16, 64, 128])
def test_mixed_decode_integer_exact(H):
    lens = [1, 64, 65, 129, 700, 1000, 2047, 3000]
    pc = workloads.paged_case(lens, [1] * len(lens), H, 128, 256, page_size=64, q_dtype="bf16",
                              k_dtype="fp8_e4m3", integer=True, seed=41 + H)
    got = run_paged(pc)
    ref, _, _ = oracle.paged(pc)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("page_size,order", [(16, 1), (32, 0), (128, 1)])
def test_mixed_decode_pages_orders_padding(page_size, order):
    # every page size (16..128 keys: 8..1 copies per tile), both orders, rows shorter than
    # index_topk (-1 padding) and k_out wider than the limit
    lens = [1, 7, 129, 500, 1000, 3000]
    pc = workloads.paged_case(lens, [1] * len(lens), 64, 128, 600, page_size=page_size, k_out=640,
                              q_dtype="bf16", k_dtype="fp8_e4m3", integer=True, seed=60 + page_size)
    got = run_paged(pc, order=order)
    ref, _, _ = oracle.paged(pc, order=order)
    assert np.array_equal(got, ref)


def test_mixed_decode_gaussian_tolerance():
    # each bf16 query row is split into e4m3 hi + lo rows: exact for elements within ~2^9
    # of the row's largest, else off by at most 2^-17 of it; the products are exact and
    # the fp32 accumulation order differs: far inside the bf16 bound
    lens = [4096, 5000, 300, 1, 7777]
    pc = workloads.paged_case(lens, [1] * len(lens), 64, 128, 2048, page_size=64, q_dtype="bf16",
                              k_dtype="fp8_e4m3", w_std=1 / 8, seed=45)
    got = run_paged(pc)
    ref, rs, rb = oracle.paged(pc, want_scores=True, want_bound=True)
    pos = oracle.query_positions(pc)
    assert_topk_valid(got, ref, rs, rb, pos + 1, pc.topk_limit, RTOL["bf16"], exact=False)



def test_paged_bad_page_is_reported_not_faulted():
    pc = workloads.paged_case([500, 300], [1, 1], 64, 128, 64, page_size=64, integer=True, seed=14)
    bt = pc.block_tables.clone()
    bt[1, 2] = pc.num_pages + 1000          # out of range: must be skipped and reported
    to = lambda t: t.to(DEV)
    dsa.dsa_indexer(to(pc.q), to(pc.w), to(pc.k_cache), to(pc.cu_q_lens), to(pc.seq_lens), to(bt),
                    max_seq_len=pc.max_seq_len, topk_limit=64)
    assert dsa.dsa_check_device_status() == dsa.DSA_ERR_DEVICE_CHECK
    assert dsa.dsa_check_device_status() == dsa.DSA_OK   # reading clears it


# ----------------------------------------------------------------------------- IndexShare

def test_indexshare_stack_forwards_source_buffers():
    types = ["full", "shared", "shared", "full", "shared"]
    cases = [workloads.paged_case([400, 90], [1, 1], 64, 128, 64, page_size=64, integer=True, seed=20 + i)
             if t == "full" else None for i, t in enumerate(types)]
    keep, args = [], []
    for c in cases:
        if c is None:
            args.append(None)
            continue
        a, kk = dsa.make_indexer_args(c.q.to(DEV), c.w.to(DEV), c.k_cache.to(DEV), c.cu_q_lens.to(DEV),
                                      c.seq_lens.to(DEV), c.block_tables.to(DEV), max_seq_len=c.max_seq_len,
                                      topk_limit=64)
        args.append(a)
        keep.append(kk)
    ptrs, src = dsa.dsa_indexer_stack(types, args)
    torch.cuda.synchronize()
    assert src == [0, 0, 0, 3, 3]
    assert ptrs[1] == ptrs[0] and ptrs[2] == ptrs[0] and ptrs[4] == ptrs[3] and ptrs[0] != ptrs[3]
    ref_src, ref = oracle.stack(types, cases)
    assert ref_src == src
    assert np.array_equal(keep[0][8].cpu().numpy(), ref[0])
    assert np.array_equal(keep[1][8].cpu().numpy(), ref[3])


def test_indexshare_rejects_before_launch():
    c = workloads.paged_case([100], [1], 64, 128, 16, page_size=64, integer=True, seed=30)
    a, _k = dsa.make_indexer_args(c.q.to(DEV), c.w.to(DEV), c.k_cache.to(DEV), c.cu_q_lens.to(DEV),
                                  c.seq_lens.to(DEV), c.block_tables.to(DEV), max_seq_len=100, topk_limit=16)
    with pytest.raises(dsa.DsaError):
        dsa.dsa_indexer_stack(["shared", "full"], [None, a])
    with pytest.raises(dsa.DsaError):
        dsa.dsa_indexer_stack(["full", "full"], [a, None])      # a full layer without its cache


# --------------------------------------------------- host-memory entry point (pipelined)

@pytest.mark.parametrize("chunk_rows,order", [(0, 0), (700, 1), (3000, 0), (97, 0)])
def test_dense_host_matches_oracle(chunk_rows, order):
    # inputs and output in pinned host memory, chunked copies overlapped with the kernels
    c = workloads.dense_case(3000, 3000, 64, 128, 200, integer=True, int_range=(-2, 2), seed=71)
    q, k, w = c.q.pin_memory(), c.k.pin_memory(), c.w.pin_memory()
    tk = dsa.dsa_indexer_dense_host(q, k, w, q_pos0=c.q_pos0, topk_limit=c.topk_limit, k_out=c.k_out,
                                    order=order, chunk_rows=chunk_rows)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    ref, _, _ = oracle_dense(c, order=order)
    assert np.array_equal(tk.numpy(), ref)


def test_dense_host_fp8_longer_keys_than_queries():
    c = workloads.dense_case(900, 2500, 64, 128, 300, q_pos0=1600, dtype="fp8_e4m3", integer=True, seed=72)
    pin = lambda t: None if t is None else t.pin_memory()
    tk = dsa.dsa_indexer_dense_host(pin(c.q), pin(c.k), pin(c.w), q_pos0=c.q_pos0, topk_limit=c.topk_limit,
                                    k_out=c.k_out, q_scale=pin(c.q_scale), k_scale=pin(c.k_scale), chunk_rows=256)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    ref, _, _ = oracle_dense(c)
    assert np.array_equal(tk.numpy(), ref)


# --------------------------------------------------- cache append (the step's new keys)

def _run_append(k_new, slots, cache, scales):
    c_d = cache.clone().to(DEV)
    s_d = None if scales is None else scales.clone().to(DEV)
    dsa.dsa_indexer_cache_append(k_new.to(DEV), slots.to(DEV), c_d, s_d)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    return c_d.cpu(), (None if s_d is None else s_d.cpu())


def _same_bytes(a, b):
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("bf16", 128), ("fp8_e4m3", 128)])
def test_cache_append_matches_oracle(dtype, D):
    g = torch.Generator().manual_seed(D + (7 if dtype == "bf16" else 0))
    n, pages, PS = 300, 12, 64
    k_new = (torch.randn((n, D), generator=g) *
             torch.pow(2.0, torch.randint(-8, 8, (n, 1), generator=g).float())).to(torch.bfloat16)
    k_new[7] = 0
    slots = torch.randperm(pages * PS, generator=g)[:n].to(torch.int64)
    slots[::17] = -1
    if dtype == "bf16":
        cache, scales = torch.randn((pages, PS, D), generator=g).to(torch.bfloat16), None
    else:
        cache = torch.randint(0, 0x7E, (pages, PS, D), generator=g).to(torch.uint8).view(torch.float8_e4m3fn)
        scales = torch.rand((pages, PS), generator=g) + 0.5
    got_c, got_s = _run_append(k_new, slots, cache, scales)
    ref_c, ref_s = oracle.cache_append(k_new, slots, cache, scales)
    assert _same_bytes(got_c, ref_c)
    if scales is not None:
        assert torch.equal(got_s, ref_s)


def test_cache_append_every_e4m3_code_and_tie():
    # rows with amax 448 (scale exactly 1): every finite code, every midpoint between
    # neighbouring codes (round-to-even ties), both signs, zeros, saturating values
    vals = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)
    mids = (vals[:-1] + vals[1:]) / 2
    pool = torch.cat([vals, -vals, mids, -mids, torch.tensor([0.0, -0.0, 460.0, -470.0])])
    rows = []
    for i in range(0, pool.numel(), 127):
        part = pool[i:i + 127]
        rows.append(torch.cat([torch.tensor([448.0]), part, torch.zeros(127 - part.numel())]))
    k_new = torch.stack(rows).to(torch.bfloat16)
    assert torch.equal(k_new.float()[:, 1:].flatten()[:pool.numel()], pool)  # exact in bf16
    n = k_new.shape[0]
    slots = torch.arange(n, dtype=torch.int64)
    cache = torch.zeros((1, 64, 128), dtype=torch.uint8).view(torch.float8_e4m3fn)
    scales = torch.zeros((1, 64))
    got_c, got_s = _run_append(k_new, slots, cache, scales)
    ref_c, ref_s = oracle.cache_append(k_new, slots, cache, scales)
    assert _same_bytes(got_c, ref_c) and torch.equal(got_s, ref_s)


@pytest.mark.parametrize("q_dtype,k_dtype,decode", [("bf16", "bf16", False), ("fp8_e4m3", "fp8_e4m3", False),
                                                     ("bf16", "fp8_e4m3", True)])
def test_indexer_appends_new_keys_before_scoring(q_dtype, k_dtype, decode):
    # the step's own keys are written through slot_mapping first, so every query sees them
    if decode:
        lens, qlens = [1, 300, 1200, 77], [1, 1, 1, 1]
    else:
        lens, qlens = [900, 40, 1500, 300], [300, 40, 17, 1]
    pc = workloads.paged_case(lens, qlens, 64, 128, 128, page_size=64, q_dtype=q_dtype, k_dtype=k_dtype,
                              integer=True, seed=81)
    k_new = workloads.new_keys(pc, seed=82, integer=True)
    if k_dtype == "fp8_e4m3":
        k_new[:, 5] = 448.0  # amax 448: scale exactly 1, every code exact, so scores stay exact
    slots = workloads.new_token_slots(pc)
    to = lambda t: None if t is None else t.to(DEV)
    cache_d, scale_d = to(pc.k_cache.clone()), to(None if pc.k_scale_cache is None else pc.k_scale_cache.clone())
    got = dsa.dsa_indexer(to(pc.q), to(pc.w), cache_d, to(pc.cu_q_lens), to(pc.seq_lens), to(pc.block_tables),
                          max_seq_len=pc.max_seq_len, topk_limit=pc.topk_limit, q_scale=to(pc.q_scale),
                          k_scale_cache=scale_d, k_new=to(k_new), slot_mapping=to(slots))
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    ref_c, ref_s = oracle.cache_append(k_new, slots, pc.k_cache, pc.k_scale_cache)
    assert _same_bytes(cache_d.cpu(), ref_c)
    if ref_s is not None:
        assert torch.equal(scale_d.cpu(), ref_s)
    pc.k_cache, pc.k_scale_cache = ref_c, ref_s
    ref, _, _ = oracle.paged(pc)
    assert np.array_equal(got.cpu().numpy(), ref)


# ----------------------------------------------------------------------------- clock sample

def test_clock_sample_reads_every_sm():
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    a = dsa.dsa_clock_sample(4 * n_sm)
    torch.cuda._sleep(2_000_000)
    b = dsa.dsa_clock_sample(4 * n_sm)
    torch.cuda.synchronize()
    a, b = a.cpu(), b.cpu()
    assert int(a[:, 0].max()) < n_sm and int(a[:, 0].min()) >= 0
    assert len(set(a[:, 0].tolist())) >= n_sm // 2      # blocks spread over the SMs
    import bench
    r = bench.sm_clock_in_band(a, b)
    assert r["sms"] >= n_sm // 2 and 100.0 < r["sm_mhz_min"] <= r["sm_mhz_max"] < 5000.0
