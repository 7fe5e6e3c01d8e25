"""Pins of the CPU oracle to things other than itself (no GPU needed).

* the hand-worked example in tests/golden/hand_worked.json (bf16 and FP8);
* exact rational brute force with a rank-counting top-k on tiny inputs;
* library special cases: H=1, w=1, q,k >= 0 reduces to a matrix product and a
  stable sort (numpy), including the tie order;
* the e4m3 / bf16 decoders against torch's conversions for every code;
* invariants: causality, -1 padding, the tie rule (also -0.0 == +0.0),
  key-permutation equivariance, positive homogeneity in w, the FP8 scale
  shaping against pre-scaled bf16 values, paged == dense;
* IndexShare source resolution and its rejections.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _bits(t):
    if t.dtype == torch.bfloat16:
        return (t.view(torch.int16).to(torch.int32) & 0xFFFF).tolist()
    return t.view(torch.uint8).to(torch.int32).tolist()


# ---------------------------------------------------------------- decoders

def test_e4m3_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).tolist()
    for c, r in zip(range(256), ref):
        v = oracle.decode_e4m3(c)
        if np.isnan(r):
            assert np.isnan(v), c
        else:
            assert v == r, (c, v, r)
            assert brute.e4m3_value(c) == r
    assert oracle.decode_e4m3(0x7E) == 448.0


def test_bf16_decode_all_finite_codes_match_torch():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = codes.view(torch.bfloat16).to(torch.float64).numpy()
    for c in range(0, 65536, 7):
        r = ref[c]
        if not np.isfinite(r):
            continue
        assert oracle.decode_bf16(c) == r, c
        assert float(brute.bf16_value(c)) == r


# ---------------------------------------------------------------- hand-worked

def _golden_case(kind):
    g = json.load(open(GOLDEN))
    q = torch.tensor(g["q"], dtype=torch.float32)
    k = torch.tensor(g["k"], dtype=torch.float32)
    w = torch.tensor(g["w"], dtype=torch.float32)
    qs = ks = None
    if kind == "bf16":
        q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    else:
        q, k = q.to(torch.float8_e4m3fn), k.to(torch.float8_e4m3fn)
        qs = torch.tensor(g["fp8"]["q_scale"], dtype=torch.float32)
        ks = torch.tensor(g["fp8"]["k_scale"], dtype=torch.float32)
    return g, q, k, w, qs, ks


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
def test_hand_worked_example(kind):
    g, q, k, w, qs, ks = _golden_case(kind)
    topk, scores, _ = oracle.dense(q, k, w, T=g["T"], S=g["S"], H=g["H"], D=g["D"],
                                   q_pos0=g["q_pos0"], topk_limit=g["topk_limit"],
                                   k_out=g["k_out"], q_scale=qs, k_scale=ks, want_scores=True)
    exp = g[kind]
    assert topk.tolist() == exp["topk"]
    for t, row in enumerate(exp["scores"]):
        for s, v in enumerate(row):
            if v is None:
                assert scores[t, s] == -np.inf
            else:
                assert scores[t, s] == v, (t, s)


# ---------------------------------------------------------------- brute force

def _brute_dense(c):
    return brute.dense(_bits(c.q), _bits(c.k), c.w.tolist(), dtype="bf16" if c.dtype == "bf16" else "fp8",
                       T=c.T, S=c.S, H=c.H, D=c.D, q_pos0=c.q_pos0, topk_limit=c.topk_limit,
                       k_out=c.k_out,
                       q_scale=None if c.q_scale is None else c.q_scale.tolist(),
                       k_scale=None if c.k_scale is None else c.k_scale.tolist())


def _oracle_dense(c, **kw):
    return oracle.dense(c.q, c.k, c.w, T=c.T, S=c.S, H=c.H, D=c.D, q_pos0=c.q_pos0,
                        topk_limit=c.topk_limit, k_out=c.k_out, q_scale=c.q_scale,
                        k_scale=c.k_scale, **kw)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_brute_force_exact_integer_inputs(seed, dtype):
    # H != D and T != S so a transposed operand or index cannot go unnoticed
    c = workloads.dense_case(9, 12, 3, 5, 4, q_pos0=2, k_out=6, integer=True, dtype=dtype,
                             int_range=(-2, 2), seed=seed)
    bt, bs = _brute_dense(c)
    topk, scores, _ = _oracle_dense(c, want_scores=True)
    assert topk.tolist() == bt
    for t in range(c.T):
        for s, v in enumerate(bs[t]):
            assert scores[t, s] == float(v)
        assert np.all(scores[t, len(bs[t]):] == -np.inf)


@pytest.mark.parametrize("seed", [3, 4])
def test_brute_force_gaussian_inputs(seed):
    c = workloads.dense_case(6, 10, 4, 8, 3, q_pos0=4, k_out=5, seed=seed)
    bt, bs = _brute_dense(c)
    topk, scores, bound = _oracle_dense(c, want_scores=True, want_bound=True)
    for t in range(c.T):
        for s, v in enumerate(bs[t]):
            assert abs(scores[t, s] - float(v)) <= 1e-13 * bound[t, s] + 1e-300
    # continuous random data: no ties, so the exact ranking is the oracle's
    assert topk.tolist() == bt


def test_brute_force_fp8_gaussian_quantised():
    c = workloads.dense_case(5, 7, 2, 6, 3, q_pos0=2, dtype="fp8_e4m3", seed=5)
    bt, bs = _brute_dense(c)
    topk, scores, bound = _oracle_dense(c, want_scores=True, want_bound=True)
    for t in range(c.T):
        for s, v in enumerate(bs[t]):
            assert abs(scores[t, s] - float(v)) <= 1e-13 * bound[t, s] + 1e-300
    assert topk.tolist() == bt


# ---------------------------------------------------------------- library special case

@pytest.mark.parametrize("seed", [0, 1])
def test_single_head_reduces_to_matmul_and_stable_sort(seed):
    g = torch.Generator().manual_seed(100 + seed)
    T, S, D, kk = 20, 40, 16, 9
    q = torch.randint(0, 4, (T, 1, D), generator=g).to(torch.bfloat16)
    k = torch.randint(0, 4, (S, D), generator=g).to(torch.bfloat16)
    w = torch.ones(T, 1)
    q_pos0 = 10
    topk, scores, _ = oracle.dense(q, k, w, T=T, S=S, H=1, D=D, q_pos0=q_pos0, topk_limit=kk,
                                   k_out=kk + 3, want_scores=True)
    ref = q.to(torch.float64)[:, 0, :].numpy() @ k.to(torch.float64).numpy().T
    for t in range(T):
        n = min(q_pos0 + t + 1, S)
        assert np.array_equal(scores[t, :n], ref[t, :n])
        # stable argsort of -score == (score desc, index asc); small integers -> many ties
        order = np.argsort(-ref[t, :n], kind="stable")[:min(kk, n)]
        exp = list(order) + [-1] * (kk + 3 - len(order))
        assert topk[t].tolist() == exp


# ---------------------------------------------------------------- invariants

def test_causality_future_keys_do_not_matter():
    c = workloads.dense_case(16, 24, 4, 8, 5, q_pos0=4, integer=True, seed=7)
    topk, scores, _ = _oracle_dense(c, want_scores=True)
    k2 = c.k.clone()
    g = torch.Generator().manual_seed(9)
    for t in range(c.T):
        pos = c.q_pos0 + t
        k2 = c.k.clone()
        if pos + 1 < c.S:
            k2[pos + 1:] = torch.randint(-4, 5, (c.S - pos - 1, c.D), generator=g).to(torch.bfloat16)
        c2 = workloads.DenseCase(**{**c.__dict__, "k": k2})
        t2, s2, _ = _oracle_dense(c2, rows=[t], want_scores=True)
        assert t2[0].tolist() == topk[t].tolist()
        assert np.array_equal(s2[0, :pos + 1], scores[t, :pos + 1])
        assert topk[t].max() <= pos


@pytest.mark.parametrize("limit,k_out", [(5, 5), (5, 8), (40, 40), (1, 3)])
def test_padding_counts(limit, k_out):
    c = workloads.dense_case(20, 20, 2, 4, limit, q_pos0=0, k_out=k_out, seed=11)
    topk, _, _ = _oracle_dense(c)
    for t in range(c.T):
        keep = min(limit, t + 1, k_out)
        row = topk[t].tolist()
        assert all(v >= 0 for v in row[:keep])
        assert row[keep:] == [-1] * (k_out - keep)
        assert len(set(row[:keep])) == keep


def test_tie_storm_zero_weights_gives_lowest_indices():
    c = workloads.dense_case(10, 30, 4, 8, 7, q_pos0=20, seed=12)
    c.w.zero_()
    topk, scores, _ = _oracle_dense(c, want_scores=True)
    for t in range(c.T):
        keep = min(7, 21 + t)
        assert topk[t].tolist() == list(range(keep))


def test_negative_zero_equals_positive_zero():
    sc = np.array([[0.0, -0.0, 1.0, -0.0, 0.0, -1.0]])
    out = oracle.topk_of_scores(sc, [6], 4, 4)
    assert out[0].tolist() == [2, 0, 1, 3]


def test_key_permutation_equivariance():
    c = workloads.dense_case(8, 32, 4, 8, 6, q_pos0=31, seed=13)   # every query sees every key
    topk, scores, _ = _oracle_dense(c, want_scores=True)
    perm = torch.randperm(c.S, generator=torch.Generator().manual_seed(14))
    c2 = workloads.DenseCase(**{**c.__dict__, "k": c.k[perm].contiguous()})
    t2, s2, _ = _oracle_dense(c2, want_scores=True)
    inv = perm.numpy()
    for t in range(c.T):
        assert np.array_equal(s2[t], scores[t][inv])
        assert sorted(inv[t2[t]].tolist()) == sorted(topk[t].tolist())


def test_positive_homogeneity_in_w():
    c = workloads.dense_case(8, 16, 4, 8, 5, q_pos0=8, integer=True, seed=15)
    topk, scores, _ = _oracle_dense(c, want_scores=True)
    c2 = workloads.DenseCase(**{**c.__dict__, "w": c.w * 2.0})
    t2, s2, _ = _oracle_dense(c2, want_scores=True)
    assert np.array_equal(t2, topk)
    fin = np.isfinite(scores)
    assert np.array_equal(s2[fin], 2.0 * scores[fin])


def test_fp8_scale_shaping_equals_prescaled_bf16():
    c = workloads.dense_case(8, 16, 4, 8, 5, q_pos0=8, integer=True, dtype="fp8_e4m3",
                             int_range=(-3, 3), seed=16)
    topk, scores, _ = _oracle_dense(c, want_scores=True)
    qv = c.q.to(torch.float32) * c.q_scale[:, :, None]
    kv = c.k.to(torch.float32) * c.k_scale[:, None]
    c2 = workloads.DenseCase(**{**c.__dict__, "q": qv.to(torch.bfloat16), "k": kv.to(torch.bfloat16),
                                "q_scale": None, "k_scale": None, "dtype": "bf16"})
    assert torch.equal(c2.q.to(torch.float32), qv) and torch.equal(c2.k.to(torch.float32), kv)
    t2, s2, _ = _oracle_dense(c2, want_scores=True)
    assert np.array_equal(t2, topk)
    assert np.array_equal(s2, scores)


def test_paged_equals_dense():
    pc = workloads.paged_case([37, 5, 64, 130], [3, 5, 1, 7], 4, 8, 6, page_size=16,
                              integer=True, seed=17)
    topk, scores, _ = oracle.paged(pc, want_scores=True)
    pos = oracle.query_positions(pc)
    cu = pc.cu_q_lens.tolist()
    for b, L in enumerate(pc.seq_lens.tolist()):
        npg = (L + 15) // 16
        pages = pc.block_tables[b, :npg].long()
        k_dense = pc.k_cache[pages].reshape(-1, pc.D)[:L].contiguous()
        ql = cu[b + 1] - cu[b]
        td, sd, _ = oracle.dense(pc.q[cu[b]:cu[b + 1]], k_dense, pc.w[cu[b]:cu[b + 1]], T=ql, S=L,
                                 H=pc.H, D=pc.D, q_pos0=L - ql, topk_limit=6, k_out=6,
                                 want_scores=True)
        assert np.array_equal(td, topk[cu[b]:cu[b + 1]])
        assert np.array_equal(sd, scores[cu[b]:cu[b + 1], :L])
        assert pos[cu[b]] == L - ql


def test_index_order_is_sorted_score_order_set():
    c = workloads.dense_case(12, 40, 4, 8, 9, q_pos0=20, integer=True, seed=18)
    t_score, _, _ = _oracle_dense(c)
    t_index, _, _ = _oracle_dense(c, order=oracle.ORDER_INDEX)
    for a, b in zip(t_score, t_index):
        keep = int((a >= 0).sum())
        assert sorted(a[:keep].tolist()) == b[:keep].tolist()
        assert (b[keep:] == -1).all()


def test_row_subset_matches_full_run():
    c = workloads.dense_case(30, 30, 2, 8, 4, q_pos0=0, seed=19)
    full, sf, _ = _oracle_dense(c, want_scores=True)
    rows = [0, 7, 29, 13]
    sub, ss, _ = _oracle_dense(c, rows=rows, want_scores=True)
    assert np.array_equal(sub, full[rows])
    assert np.array_equal(ss, sf[rows])


# ---------------------------------------------------------------- IndexShare

def test_resolve_sources_chain_and_errors():
    assert oracle.resolve_indexer_sources(["full", "shared", "shared", "full", "shared"]) == [0, 0, 0, 3, 3]
    assert oracle.resolve_indexer_sources(workloads.INDEXSHARE_TYPES_12) == [0, 0, 0, 3, 3, 3, 6, 6, 6, 9, 9, 9]
    with pytest.raises(ValueError):
        oracle.resolve_indexer_sources(["shared", "full"])
    with pytest.raises(ValueError):
        oracle.resolve_indexer_sources(["full", "sharded"])
    with pytest.raises(ValueError):
        oracle.resolve_indexer_sources(["full"], num_layers=2)


def test_stack_shared_layers_forward_source_unchanged():
    types = ["full", "shared", "shared", "full", "shared"]
    layers = [workloads.paged_case([40, 70], [1, 1], 4, 8, 8, page_size=16, seed=20 + i)
              if t == "full" else None for i, t in enumerate(types)]
    src, outs = oracle.stack(types, layers)
    assert src == [0, 0, 0, 3, 3]
    assert outs[1] is outs[0] and outs[2] is outs[0] and outs[4] is outs[3]
    assert not np.array_equal(outs[0], outs[3])


# ---------------------------------------------------------------- cache append (encoder, quantiser)

def test_e4m3_encode_matches_torch_rounding():
    # every finite code, every midpoint between neighbours (ties), and random in-range
    # values: torch's float8_e4m3fn cast rounds to nearest, ties to even
    vals = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    mids = (vals[:-1] + vals[1:]) / 2
    g = torch.Generator().manual_seed(3)
    rnd = (torch.rand(4000, generator=g, dtype=torch.float64) * 2 - 1) * 448 * torch.pow(
        2.0, -torch.randint(0, 18, (4000,), generator=g).to(torch.float64))
    x = torch.cat([vals, -vals, mids, -mids, rnd]).to(torch.float32)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x.numpy())
    assert np.array_equal(got, ref)


def test_e4m3_encode_hand_values():
    # derived by hand from the format: 448 = 1.75 * 2^8 (e=15, m=6); 224 = 1.75 * 2^7
    # (e=14, m=6) with the sign; 1 = 2^0 (e=7); 2^-9 is the smallest subnormal; 2^-10 is
    # half of it, a tie between codes 0 and 1 -> the even code 0; 0.05 = 1.6 * 2^-5 lies
    # between 1.5 and 1.625 (m=4, 5) and is nearer 1.625; 500 saturates to 448
    x = [448.0, -224.0, 1.0, 2.0 ** -9, 2.0 ** -10, 0.0, -0.0, 0.05, 500.0, -1e6]
    assert oracle.e4m3_encode(x).tolist() == [0x7E, 0xF6, 0x38, 0x01, 0x00, 0x00, 0x80, 0x15, 0x7E, 0xFE]


def _append_case(cache_dtype, seed=0, n=12, D=128, pages=5, PS=16):
    g = torch.Generator().manual_seed(seed)
    k_new = (torch.randn((n, D), generator=g) * torch.pow(2.0, torch.randint(-6, 6, (n, 1), generator=g))).to(
        torch.bfloat16)
    k_new[3] = 0                                          # all-zero row: scale 1, codes 0
    slots = torch.randperm(pages * PS, generator=g)[:n].to(torch.int64)
    slots[5] = -1                                         # padding token: skipped
    if cache_dtype == "bf16":
        cache = torch.randn((pages, PS, D), generator=g).to(torch.bfloat16)
        return k_new, slots, cache, None
    cache = torch.randint(0, 0x7E, (pages, PS, D), generator=g).to(torch.uint8).view(torch.float8_e4m3fn)
    return k_new, slots, cache, torch.rand((pages, PS), generator=g) + 0.5


def test_cache_append_bf16_copies_rows_and_leaves_the_rest():
    k_new, slots, cache, _ = _append_case("bf16")
    out, _ = oracle.cache_append(k_new, slots, cache)
    flat, before = out.view(-1, 128), cache.view(-1, 128)
    touched = set()
    for i, s in enumerate(slots.tolist()):
        if s >= 0:
            assert torch.equal(flat[s].view(torch.int16), k_new[i].view(torch.int16))
            touched.add(s)
    for s in range(flat.shape[0]):
        if s not in touched:
            assert torch.equal(flat[s].view(torch.int16), before[s].view(torch.int16))


def test_cache_append_e4m3_quantiser_properties():
    k_new, slots, cache, scales = _append_case("fp8", seed=1)
    out, sc = oracle.cache_append(k_new, slots, cache, scales)
    flat, fsc = out.view(-1, 128), sc.view(-1)
    codes = flat.view(torch.uint8)
    for i, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        x = k_new[i].to(torch.float64)
        amax = x.abs().max().item()
        if amax == 0:
            assert fsc[s].item() == 1.0 and codes[s].tolist() == [0] * 128
            continue
        # the scale is amax / 448 rounded once to fp32
        assert fsc[s].item() == float(np.float32(np.float32(amax) / np.float32(448.0)))
        dec = flat[s].to(torch.float64) * fsc[s].item()
        # the amax element lands on +-448 and every element is within half an e4m3 step
        # of its value (relative 1/16 for normals, 2^-10 * scale below 2^-6 * scale)
        j = int(x.abs().argmax())
        assert abs(flat[s].to(torch.float64)[j].item()) == 448.0
        step = torch.maximum(x.abs() / 16, torch.full_like(x, 2.0 ** -10 * fsc[s].item()))
        assert torch.all((dec - x).abs() <= step * 1.0001)
        assert torch.all(torch.sign(dec) * torch.sign(x) >= 0)
    # untouched slots keep their bytes and scales
    touched = {s for s in slots.tolist() if s >= 0}
    before = cache.view(-1, 128).view(torch.uint8)
    for s in range(flat.shape[0]):
        if s not in touched:
            assert torch.equal(codes[s], before[s]) and fsc[s].item() == scales.view(-1)[s].item()


def test_cache_append_e4m3_matches_torch_quantisation():
    # library special case: torch's own per-row scale and cast give the same bytes
    k_new, slots, cache, scales = _append_case("fp8", seed=2)
    out, sc = oracle.cache_append(k_new, slots, cache, scales)
    x = k_new.to(torch.float32)
    amax = x.abs().amax(dim=1, keepdim=True)
    s_ref = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    ref = (x / s_ref).to(torch.float8_e4m3fn).view(torch.uint8)
    flat, fsc = out.view(-1, 128).view(torch.uint8), sc.view(-1)
    for i, s in enumerate(slots.tolist()):
        if s >= 0:
            assert torch.equal(flat[s], ref[i])
            assert fsc[s].item() == s_ref[i, 0].item()


def test_cache_append_rejects_slot_past_the_cache():
    k_new, slots, cache, _ = _append_case("bf16")
    slots[0] = cache.shape[0] * cache.shape[1]
    with pytest.raises(ValueError):
        oracle.cache_append(k_new, slots, cache)


# ---------------------------------------------------------------- indexer front-end (oracle/frontend.py)

from oracle import frontend  # noqa: E402


def test_frontend_hadamard_is_orthogonal_with_sign_entries():
    # Sylvester order: H[i, j] = (-1)^popcount(i & j) / sqrt(D); H H^T = I
    for D in (2, 8, 128):
        Hm = frontend.hadamard(D)
        assert np.allclose(Hm @ Hm.T, np.eye(D), atol=1e-12)
        i, j = np.meshgrid(np.arange(D), np.arange(D), indexing="ij")
        signs = np.vectorize(lambda a: (-1) ** bin(a).count("1"))(i & j)
        assert np.array_equal(Hm * np.sqrt(D), signs.astype(np.float64))
    # the rotation of a basis vector is one column of +-1/sqrt(D); norms are kept
    e = np.zeros((1, 128)); e[0, 5] = 1.0
    r = frontend.rotate_activation(e)
    assert np.allclose(np.abs(r), 1 / np.sqrt(128))
    x = np.random.default_rng(0).standard_normal((3, 128))
    assert np.allclose(np.linalg.norm(frontend.rotate_activation(x), axis=1), np.linalg.norm(x, axis=1))


def test_frontend_rope_identity_quarter_turn_and_norms():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 3, 16))
    for inter in (False, True):
        ones, zeros = np.ones((2, 4)), np.zeros((2, 4))
        assert np.array_equal(frontend.rope(x, ones, zeros, 8, inter), x)      # angle 0
        y = frontend.rope(x, zeros, ones, 8, inter)                              # angle 90 degrees
        if inter:
            assert np.allclose(y[..., 0:8:2], -x[..., 1:8:2]) and np.allclose(y[..., 1:8:2], x[..., 0:8:2])
        else:
            assert np.allclose(y[..., :4], -x[..., 4:8]) and np.allclose(y[..., 4:8], x[..., :4])
        assert np.array_equal(y[..., 8:], x[..., 8:])                          # values past rope_dim untouched
        th = rng.uniform(0, 6.3, (2, 4))
        z = frontend.rope(x, np.cos(th), np.sin(th), 8, inter)
        assert np.allclose(np.linalg.norm(z, axis=-1), np.linalg.norm(x, axis=-1))


def test_frontend_layer_norm_hand_worked():
    # x = [1, 2, 3, 4]: mean 2.5, biased variance 1.25, eps 0 -> (x - 2.5) / sqrt(1.25)
    y = frontend.layer_norm(np.array([[1.0, 2.0, 3.0, 4.0]]), np.ones(4), None, 0.0)
    assert np.allclose(y, [[-1.5 / np.sqrt(1.25), -0.5 / np.sqrt(1.25), 0.5 / np.sqrt(1.25), 1.5 / np.sqrt(1.25)]])
    y2 = frontend.layer_norm(np.array([[1.0, 2.0, 3.0, 4.0]]), np.array([2.0, 2.0, 2.0, 2.0]), np.full(4, 0.5), 0.0)
    assert np.allclose(y2, 2 * y + 0.5)
    x = np.random.default_rng(2).standard_normal((5, 128)) * 3 + 1
    z = frontend.layer_norm(x, np.ones(128), None, 1e-6)
    assert np.allclose(z.mean(axis=1), 0, atol=1e-12) and np.allclose(z.var(axis=1), 1, atol=1e-5)


def test_frontend_linear_brute_force():
    rng = np.random.default_rng(3)
    x, Wm = rng.integers(-3, 4, (3, 5)).astype(np.float64), rng.integers(-3, 4, (4, 5)).astype(np.float64)
    ref = [[sum(x[t, k] * Wm[n, k] for k in range(5)) for n in range(4)] for t in range(3)]
    assert np.array_equal(frontend.linear(x, Wm), np.array(ref))


def test_frontend_quantize_rows_bound_and_zero_row():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4, 128))
    x[2] = 0.0
    codes, scale = frontend.quantize_rows(x)
    assert scale[2] == 1.0 and np.all(codes[2] == 0)
    dq = frontend.dequantize(codes, scale)
    # e4m3 keeps 3 mantissa bits: error at most half a unit in the last place (2^-4 relative),
    # and the row's largest magnitude maps to 448 exactly
    assert np.all(np.abs(dq - x) <= np.abs(x) * 2.0 ** -4 + scale[:, None] * 2.0 ** -10)
    for r in (0, 1, 3):
        assert np.isclose(np.abs(dq[r]).max(), np.abs(x[r]).max(), rtol=1e-6)


def test_frontend_prepare_composition():
    # the pipeline's pieces in order: k is a normalised row rotated by RoPE (and Hadamard),
    # so its norm is the layer norm's (sqrt(D) for a unit weight); w is the plain projection
    g = torch.Generator().manual_seed(5)
    T, Dm, R, H, D, r = 3, 64, 32, 2, 128, 64
    hid = torch.randn((T, Dm), generator=g).to(torch.bfloat16)
    qa = torch.randn((T, R), generator=g).to(torch.bfloat16)
    wq = (torch.randn((H * D, R), generator=g) / 8).to(torch.bfloat16)
    wk = (torch.randn((D, Dm), generator=g) / 8).to(torch.bfloat16)
    wp = (torch.randn((H, Dm), generator=g) / 8).to(torch.bfloat16)
    th = torch.rand((T, r // 2), generator=g) * 6
    for fp8 in (False, True):
        out = frontend.prepare(hid, qa, torch.cos(th), torch.sin(th), wq, wk, wp, torch.ones(D), None, H=H, D=D,
                               rope_dim=r, interleaved=False, eps=1e-6, fp8=fp8)
        assert np.allclose(np.linalg.norm(out["k"], axis=1), np.sqrt(D), rtol=1e-6)
        assert np.allclose(out["w"], frontend.to_f64(hid) @ frontend.to_f64(wp).T)
        q0 = (frontend.to_f64(qa) @ frontend.to_f64(wq).T).reshape(T, H, D)
        assert np.allclose(np.linalg.norm(out["q"], axis=-1), np.linalg.norm(q0, axis=-1))
        if fp8:
            assert out["q_codes"].shape == (T, H, D) and out["q_scale"].shape == (T, H)
            assert out["k_codes"].shape == (T, D) and out["k_scale"].shape == (T,)


# ---------------------------------------------------------------- sparse MLA over top-k (oracle/sparse_mla.py)

from oracle import sparse_mla as smla  # noqa: E402


def _smla(c, topk=None, q_nope=None, q_rope=None):
    return smla.sparse_mla(c.q_nope if q_nope is None else q_nope, c.q_rope if q_rope is None else q_rope,
                           c.cache_c, c.cache_r, c.block_tables, c.cu_q_lens, c.topk if topk is None else topk,
                           page_size=c.page_size, scale=c.scale)


def _latent_rows(c, b, positions):
    cc, cr = frontend.to_f64(c.cache_c), frontend.to_f64(c.cache_r)
    return smla.gather_latent(cc, cr, c.block_tables[b].numpy(), c.page_size, np.asarray(positions))


def test_sparse_mla_single_key_returns_its_latent_row():
    c = workloads.sparse_mla_case([100, 40], [3, 1], 4, 8, kv_rank=32, rope_dim=8, page_size=16, seed=1)
    tk = torch.full_like(c.topk, -1)
    tk[:, 3] = torch.tensor([5, 0, 97, 39], dtype=torch.int32)          # one key per token, anywhere in the row
    out = _smla(c, topk=tk)
    rows = [(0, 5), (0, 0), (0, 97), (1, 39)]
    for t, (b, s) in enumerate(rows):
        lat, _ = _latent_rows(c, b, [s])
        assert np.allclose(out[t], np.broadcast_to(lat[0], out[t].shape), atol=1e-12)


def test_sparse_mla_equal_logits_average_the_selection():
    c = workloads.sparse_mla_case([64], [2], 3, 10, kv_rank=16, rope_dim=8, page_size=16, seed=2)
    zq, zr = torch.zeros_like(c.q_nope), torch.zeros_like(c.q_rope)
    out = _smla(c, q_nope=zq, q_rope=zr)
    for t in range(2):
        sel = c.topk[t][c.topk[t] >= 0].numpy()
        lat, _ = _latent_rows(c, 0, sel)
        assert np.allclose(out[t], lat.mean(axis=0)[None, :], atol=1e-12)


def test_sparse_mla_order_and_padding_do_not_matter():
    c = workloads.sparse_mla_case([300, 90], [2, 2], 4, 24, kv_rank=32, rope_dim=8, page_size=32, seed=3)
    base = _smla(c)
    g = torch.Generator().manual_seed(9)
    tk = torch.full((c.topk.shape[0], 40), -1, dtype=torch.int32)
    for t in range(c.topk.shape[0]):
        sel = c.topk[t][c.topk[t] >= 0]
        slots = torch.randperm(40, generator=g)[:sel.numel()]
        tk[t, slots] = sel[torch.randperm(sel.numel(), generator=g)]
    assert np.allclose(_smla(c, topk=tk), base, atol=1e-12)
    empty = torch.full_like(c.topk, -1)
    assert np.array_equal(_smla(c, topk=empty), np.zeros_like(base))


def test_sparse_mla_all_causal_keys_equals_dense_attention():
    # selecting every visible key reduces to dense causal attention: torch's
    # scaled_dot_product_attention on q = [q_nope, q_rope], k = [c_kv, k_rope], v = c_kv
    L, ql, H, R, rd, P = 96, 5, 3, 16, 8, 16
    c = workloads.sparse_mla_case([L], [ql], H, L, kv_rank=R, rope_dim=rd, page_size=P, seed=4)
    tk = torch.full((ql, L), -1, dtype=torch.int32)
    for i in range(ql):
        pos = L - ql + i
        tk[i, :pos + 1] = torch.arange(pos + 1, dtype=torch.int32)
    out = _smla(c, topk=tk)
    lat, rope = _latent_rows(c, 0, np.arange(L))
    q = torch.cat([c.q_nope.to(torch.float64), c.q_rope.to(torch.float64)], dim=-1).transpose(0, 1)  # [H, ql, R+rd]
    k = torch.from_numpy(np.concatenate([lat, rope], axis=-1))[None].expand(H, L, R + rd)
    v = torch.from_numpy(lat)[None].expand(H, L, R)
    mask = torch.arange(L)[None, :] <= (L - ql + torch.arange(ql))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=c.scale)
    assert np.allclose(out, ref.transpose(0, 1).numpy(), atol=1e-10)


FRONTEND_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "frontend_hand_worked.json")


def _frontend_golden_inputs():
    with open(FRONTEND_GOLDEN) as f:
        g = json.load(f)
    bf = lambda v: torch.tensor(v, dtype=torch.float32).to(torch.bfloat16)
    ins = dict(hidden=bf(g["hidden"]), qa_normed=bf(g["qa_normed"]), wq_b=bf(g["wq_b"]), wk=bf(g["wk"]),
               weights_proj=bf(g["weights_proj"]), k_norm_weight=torch.tensor(g["k_norm_weight"], dtype=torch.float32),
               rope_cos=torch.tensor(g["cos"], dtype=torch.float64), rope_sin=torch.tensor(g["sin"], dtype=torch.float64))
    return g, ins


def _frontend_golden_expected(g, kind):
    e = g[kind]
    return np.array(e["q"], dtype=np.float64), np.array(e["k_times_sqrt6"], dtype=np.float64) / np.sqrt(6.0), \
        np.array(e["w"], dtype=np.float64)


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
def test_frontend_prepare_hand_worked(kind):
    """The front-end's step order (projections, k layer norm, RoPE, then on FP8 the rotation and the
    row scales) against values worked by hand."""
    g, ins = _frontend_golden_inputs()
    out = frontend.prepare(ins["hidden"], ins["qa_normed"], ins["rope_cos"], ins["rope_sin"], ins["wq_b"], ins["wk"],
                           ins["weights_proj"], ins["k_norm_weight"], None, H=g["H"], D=g["D"], rope_dim=g["rope_dim"],
                           interleaved=False, eps=g["eps"], fp8=(kind == "fp8"))
    q, k, w = _frontend_golden_expected(g, kind)
    assert np.allclose(out["q"], q, rtol=0, atol=1e-12)
    assert np.allclose(out["k"], k, rtol=0, atol=1e-12)
    assert np.allclose(out["w"], w, rtol=0, atol=1e-12)
    if kind == "fp8":
        # the scales are fp32 (amax taken to fp32, divided by 448 in fp32)
        assert np.allclose(out["q_scale"], g["fp8"]["q_scale"], rtol=1e-6, atol=0)
        assert np.allclose(out["k_scale"], np.array(g["fp8"]["k_scale_times_sqrt6"]) / np.sqrt(6.0), rtol=1e-6, atol=0)


def test_frontend_hand_worked_values_tell_the_plausible_mistakes_apart():
    """Each misordering of the front-end's steps, built from the oracle's own pieces, misses the
    hand-worked values: the golden case would catch it in prepare."""
    g, ins = _frontend_golden_inputs()
    f64 = frontend.to_f64
    H, D, r = g["H"], g["D"], g["rope_dim"]
    cos, sin = f64(ins["rope_cos"]), f64(ins["rope_sin"])
    ln = lambda x: frontend.layer_norm(x, f64(ins["k_norm_weight"]), None, g["eps"])
    rp = lambda x, c=cos, s=sin: frontend.rope(x, c, s, r, False)
    q0 = frontend.linear(f64(ins["qa_normed"]), f64(ins["wq_b"])).reshape(1, H, D)
    k0 = frontend.linear(f64(ins["hidden"]), f64(ins["wk"]))
    rot = frontend.rotate_activation
    mistakes = {
        "no RoPE": (q0, ln(k0), "bf16"),
        "cos and sin swapped": (rp(q0, sin, cos), rp(ln(k0), sin, cos), "bf16"),
        "layer norm after RoPE": (rp(q0), ln(rp(k0)), "bf16"),
        "rotation before RoPE": (rp(rot(q0)), rp(rot(ln(k0))), "fp8"),
        "projections transposed": (rp((f64(ins["qa_normed"]) @ f64(ins["wq_b"])).reshape(1, H, D)),
                                   rp(ln(f64(ins["hidden"]) @ f64(ins["wk"]))), "bf16"),
    }
    for name, (q, k, kind) in mistakes.items():
        eq, ek, _ = _frontend_golden_expected(g, kind)
        assert not (np.allclose(q, eq, atol=1e-6) and np.allclose(k, ek, atol=1e-6)), name
    # and the right order, built from the same pieces, meets them
    eq, ek, _ = _frontend_golden_expected(g, "fp8")
    assert np.allclose(rot(rp(q0)), eq, atol=1e-12) and np.allclose(rot(rp(ln(k0))), ek, atol=1e-12)


# ---------------------------------------------------------------- key-sharded top-k (oracle/sharded.py)

from oracle import sharded  # noqa: E402


def _sharded_case(seed, T=40, S=70, topk=12, q_pos0=30):
    c = workloads.dense_case(T, S, 4, 64, topk, q_pos0=q_pos0, integer=True, int_range=(-1, 1),
                             w_int_range=(-1, 1), seed=seed)
    rt, rs, _ = oracle.dense(c.q, c.k, c.w, T=T, S=S, H=4, D=64, q_pos0=q_pos0, topk_limit=topk, k_out=topk + 3,
                             want_scores=True)
    n_vis = np.minimum(q_pos0 + np.arange(T) + 1, S)
    return c, rt, rs, n_vis


@pytest.mark.parametrize("bounds", [[0, 70], [0, 17, 40, 70], [0, 1, 2, 69, 70], [0, 35, 70]])
@pytest.mark.parametrize("order", [oracle.ORDER_SCORE, oracle.ORDER_INDEX])
def test_sharded_merge_equals_the_full_row_topk(bounds, order):
    """Merging every shard's best k (score, index) candidates gives the C oracle's own
    full-row top-k, bit for bit, with small-integer scores full of ties across shard
    boundaries and rows that see none of some shards."""
    topk = 12
    c, rt, rs, n_vis = _sharded_case(seed=70 + len(bounds))
    ref = oracle.dense(c.q, c.k, c.w, T=c.T, S=c.S, H=4, D=64, q_pos0=c.q_pos0, topk_limit=topk, k_out=topk + 3,
                       order=order)[0]
    cands = [sharded.shard_candidates(rs, n_vis, b0, b1 - b0, topk) for b0, b1 in zip(bounds[:-1], bounds[1:])]
    cs = np.stack([x[0] for x in cands])
    ci = np.stack([x[1] for x in cands])
    got = sharded.merge_candidates(cs, ci, topk, topk + 3, order)
    assert np.array_equal(got, ref)
    # the shards' order in the gather does not matter
    perm = np.random.default_rng(1).permutation(len(cands))
    assert np.array_equal(sharded.merge_candidates(cs[perm], ci[perm], topk, topk + 3, order), ref)


def test_shard_candidates_brute_force_ranks():
    """Each shard candidate list against rank counting: key s of the shard sits at position
    #{s' in the shard, visible: o[s'] > o[s], or o[s'] == o[s] and s' < s} when that is < k."""
    c, rt, rs, n_vis = _sharded_case(seed=75, T=12, S=30, topk=5, q_pos0=5)
    b0, L, k = 7, 11, 5
    cs, ci = sharded.shard_candidates(rs, n_vis, b0, L, k)
    for t in range(12):
        vis = [s for s in range(b0, b0 + L) if s < n_vis[t]]
        want = [-1] * k
        for s in vis:
            r = sum(1 for s2 in vis if rs[t, s2] > rs[t, s] or (rs[t, s2] == rs[t, s] and s2 < s))
            if r < k:
                want[r] = s
        assert ci[t].tolist() == want
        for i, s in enumerate(want):
            assert (cs[t, i] == rs[t, s]) if s >= 0 else cs[t, i] == -np.inf


def test_sharded_merge_treats_signed_zeros_as_equal():
    # one shard holds +0.0 at key 9, the other -0.0 at key 3: equal scores, the lower index first
    cs = np.array([[[0.0, -1.0]], [[-0.0, -np.inf]]])
    ci = np.array([[[9, 4]], [[3, -1]]], dtype=np.int32)
    assert sharded.merge_candidates(cs, ci, 3, 4).tolist() == [[3, 9, 4, -1]]
    assert sharded.merge_candidates(cs, ci, 2, 2, sharded.ORDER_INDEX).tolist() == [[3, 9]]
