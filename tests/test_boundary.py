"""The C ABI boundary without a GPU: the library loads, exports every function
include/dsa_indexer.h declares, validates arguments before any launch, and the
host-only IndexShare logic and helpers follow the GLM5 TensorCast adaptation
design ("Sparse MLA 配置兼容", "GLM-5.2 IndexShare")."""
import ctypes
import os
import re
import types as _types

import pytest

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa_indexer.h")


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__ as g
    g.build()
    import sparse_attention_token_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**(dsa_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["dsa_indexer_scores", "dsa_indexer_topk", "dsa_indexer", "dsa_indexer_workspace_size",
              "dsa_indexer_stack", "dsa_resolve_indexer_sources", "dsa_check_device_status",
              "dsa_status_string", "dsa_topk_width", "dsa_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(dsa):
    L = ctypes.CDLL(dsa.LIB_PATH)
    for n in declared_functions():
        assert hasattr(L, n), n


def test_status_strings_and_version(dsa):
    assert dsa.dsa_status_string(0) == "DSA_OK"
    assert dsa.dsa_status_string(6) == "DSA_ERR_WORKSPACE"
    assert dsa.dsa_status_string(99) == "DSA_ERR_UNKNOWN"
    assert "sm_103a" in dsa.dsa_version()


@pytest.mark.parametrize("limit,n,exp", [(2048, 100, 100), (2048, 5000, 2048), (64, 0, 0), (64, -3, 0)])
def test_topk_width(dsa, limit, n, exp):
    assert dsa.dsa_topk_width(limit, n) == exp


def test_scores_validation_happens_before_any_launch(dsa):
    L = dsa.lib()
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    ok = lambda *a: L.dsa_indexer_scores(*a)
    base = dict(q=fake, qd=0, qs=None, k=fake, kd=0, ks=None, w=fake, T=4, S=8, H=64, D=128, p0=4,
                sc=fake, ld=8, st=None)

    def call(**kw):
        a = {**base, **kw}
        return ok(a["q"], a["qd"], a["qs"], a["k"], a["kd"], a["ks"], a["w"], a["T"], a["S"], a["H"], a["D"],
                  a["p0"], a["sc"], a["ld"], a["st"])

    assert call(q=None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert call(q=fake + 4) == dsa.DSA_ERR_INVALID_ARGUMENT           # misaligned
    assert call(ld=6) == dsa.DSA_ERR_INVALID_ARGUMENT                 # ld < S
    assert call(ld=10) == dsa.DSA_ERR_INVALID_ARGUMENT                # ld not a multiple of 4
    assert call(H=48) == dsa.DSA_ERR_UNSUPPORTED
    assert call(D=96) == dsa.DSA_ERR_UNSUPPORTED
    assert call(qd=1, kd=0) == dsa.DSA_ERR_UNSUPPORTED                # dtype mix
    assert call(qd=1, kd=1) == dsa.DSA_ERR_INVALID_ARGUMENT           # FP8 without scales
    assert call(qd=1, kd=1, qs=fake, ks=fake, D=64) == dsa.DSA_ERR_UNSUPPORTED
    assert call(qd=7) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert call(T=-1) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert call(p0=-1) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert call(T=0) == dsa.DSA_OK                                    # empty: nothing to do


def test_topk_validation(dsa):
    L = dsa.lib()
    fake = 1 << 20
    assert L.dsa_indexer_topk(fake, 8, 4, 8, 4, 0, 4, 0, fake, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_indexer_topk(fake, 8, 4, 8, 4, 4, 0, 0, fake, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_indexer_topk(fake, 8, 4, 8, 4, 4, 5000, 0, fake, None) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_indexer_topk(fake, 8, 4, 8, 4, 4, 4, 2, fake, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_indexer_topk(fake, 8, 4, 8, 4, 4, 4, 0, None, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_indexer_topk(fake, 8, 0, 8, 4, 4, 4, 0, fake, None) == dsa.DSA_OK


def _args(dsa, **kw):
    a = dsa.dsa_indexer_args()
    a.q_dtype = a.k_dtype = 0
    a.B, a.total_q, a.H, a.D = 2, 2, 64, 128
    a.page_size, a.num_pages, a.max_pages_per_seq, a.max_seq_len = 64, 10, 5, 300
    a.topk_limit, a.k_out, a.order = 64, 64, 0
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_workspace_size_and_paged_validation(dsa):
    n = dsa.dsa_indexer_workspace_size(_args(dsa))
    assert n >= 2 * 300 * 4                               # at least the fp32 score rows
    for bad in [dict(page_size=48), dict(H=3), dict(k_out=5000), dict(max_seq_len=321),
                dict(q_dtype=1, k_dtype=0), dict(order=3), dict(topk_limit=0)]:
        with pytest.raises(dsa.DsaError):
            dsa.dsa_indexer_workspace_size(_args(dsa, **bad))
    # bf16 queries with an e4m3 cache: decode shapes only, and the key scales are required
    n_split = dsa.dsa_indexer_workspace_size(_args(dsa, q_dtype=0, k_dtype=1, k_scale_cache=1 << 20))
    # ... plus the split query rows q8 [total_q, 2H, D] e4m3 and their weights w8 [total_q, H]
    assert n_split - n >= 2 * (2 * 64) * 128 + 2 * 64 * 4
    with pytest.raises(dsa.DsaError):
        dsa.dsa_indexer_workspace_size(_args(dsa, q_dtype=0, k_dtype=1))
    with pytest.raises(dsa.DsaError):
        dsa.dsa_indexer_workspace_size(_args(dsa, q_dtype=0, k_dtype=1, k_scale_cache=1 << 20, total_q=3))
    L = dsa.lib()
    a = _args(dsa)                                        # valid sizes, null pointers
    assert L.dsa_indexer(ctypes.byref(a), None) == dsa.DSA_ERR_INVALID_ARGUMENT
    fake = 1 << 20
    for f in ["q", "w", "cu_q_lens", "seq_lens", "block_tables", "k_cache", "topk"]:
        setattr(a, f, fake)
    assert L.dsa_indexer(ctypes.byref(a), None) == dsa.DSA_ERR_WORKSPACE
    a.workspace, a.workspace_bytes = fake, n - 16
    assert L.dsa_indexer(ctypes.byref(a), None) == dsa.DSA_ERR_WORKSPACE


# ---------------------------------------------------------------- IndexShare host logic

@pytest.mark.parametrize("types", [
    ["full", "shared", "shared"] * 4,
    ["full", "full", "shared", "full"],
    ["full"],
    [],
])
def test_resolve_sources_matches_oracle(dsa, types):
    assert dsa.dsa_resolve_indexer_sources(types) == oracle.resolve_indexer_sources(types)


@pytest.mark.parametrize("types", [["shared"], ["shared", "full"], ["full", "dense"], ["full", None]])
def test_resolve_sources_rejects(dsa, types):
    with pytest.raises(ValueError):
        dsa.dsa_resolve_indexer_sources(types)
    with pytest.raises(ValueError):
        oracle.resolve_indexer_sources(types)


def test_resolve_sources_length_check(dsa):
    with pytest.raises(ValueError):
        dsa.dsa_resolve_indexer_sources(["full", "shared"], num_layers=3)


def test_stack_rejects_bad_lists_before_launch(dsa):
    with pytest.raises(dsa.DsaError):
        dsa.dsa_indexer_stack(["shared", "full"], [None, None])
    with pytest.raises(dsa.DsaError):
        dsa.dsa_indexer_stack(["full", "shared"], [None, None])       # full layer without args
    with pytest.raises(dsa.DsaError):
        dsa.dsa_indexer_stack(["full", "oops"], [None, None])


def test_mtp_extension(dsa):
    base = ["full", "shared", "shared"]
    assert dsa.extend_indexer_types_for_mtp(base, 2) == base + ["full", "full"]
    assert dsa.extend_indexer_types_for_mtp(base, 0) == base
    assert dsa.extend_indexer_types_for_mtp([], 3) == []


def test_topk_limit_resolution_order(dsa):
    ns = _types.SimpleNamespace
    assert dsa.resolve_topk_limit(explicit=7, indexer=ns(topk_limit=8)) == 7
    assert dsa.resolve_topk_limit(indexer=ns(topk_limit=8), config=ns(topk_limit=9)) == 8
    assert dsa.resolve_topk_limit(config=ns(topk_limit=9, index_topk=10)) == 9
    assert dsa.resolve_topk_limit(config=ns(), indexer_config=ns(topk_limit=11)) == 11
    assert dsa.resolve_topk_limit(config=ns(index_topk=2048)) == 2048          # GLM5 style
    assert dsa.resolve_topk_limit(indexer=ns(topk_limit=None), config=ns(topk_limit=None, index_topk=5)) == 5
    with pytest.raises(AttributeError, match="topk_limit"):
        dsa.resolve_topk_limit(config=ns(), indexer_config=ns())


def test_workload_shapes():
    c = workloads.tiny_exact_prefill()
    assert (c.T, c.S, c.H, c.D, c.topk_limit) == (512, 512, 4, 64, 64)
    assert float(c.q.float().abs().max()) <= 4 and float(c.w.abs().max()) <= 2
    st = workloads.indexshare_stack(B=2, ctx=256)
    assert st.indexer_types == workloads.INDEXSHARE_TYPES_12
    assert sum(l is not None for l in st.layers) == 4

def test_dense_host_validation_happens_before_any_cuda_call(dsa):
    L = dsa.lib()
    n = dsa.dsa_indexer_dense_host_workspace_size(8192, 8192, 64, 128, dsa.DSA_BF16, 2048)
    assert n >= 8192 * 64 * 128 * 2 + 8192 * 2048 * 4            # q and the top-k rows at least
    assert dsa.dsa_indexer_dense_host_workspace_size(100, 100, 64, 128, dsa.DSA_BF16, 16, 7) > 0
    with pytest.raises(dsa.DsaError):
        dsa.dsa_indexer_dense_host_workspace_size(0, 10, 64, 128, dsa.DSA_BF16, 16)
    fake = 1 << 20

    def call(qd=0, kd=0, T=10, S=10, k_out=16, order=0, chunk=0, ptrs=True, ws_bytes=1 << 40, qs=None, ks=None):
        p = fake if ptrs else None
        return L.dsa_indexer_dense_host(p, qd, qs, p, kd, ks, p, T, S, 64, 128, 0, 16, k_out, order, chunk, p,
                                        fake, ws_bytes, None)
    assert call(ptrs=False) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert call(order=2) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert call(chunk=-1) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert call(k_out=5000) == dsa.DSA_ERR_UNSUPPORTED
    assert call(qd=1, kd=0) == dsa.DSA_ERR_UNSUPPORTED
    assert call(qd=1, kd=1) == dsa.DSA_ERR_INVALID_ARGUMENT      # e4m3 needs both scale arrays
    assert call(S=0) == dsa.DSA_ERR_UNSUPPORTED
    assert call(ws_bytes=16) == dsa.DSA_ERR_WORKSPACE
    assert call(T=0) == dsa.DSA_OK                               # nothing to do


def test_cache_append_validation_happens_before_any_cuda_call(dsa):
    L = dsa.lib()
    fake = 1 << 20

    def call(n=4, D=128, dt=1, scales=True, ptrs=True, PS=64, pages=3):
        p = fake if ptrs else None
        return L.dsa_indexer_cache_append(p, n, D, p, p, dt, fake if scales else None, PS, pages, None)
    assert call(n=0) == dsa.DSA_OK
    assert call(n=-1) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert call(ptrs=False) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert call(scales=False) == dsa.DSA_ERR_INVALID_ARGUMENT   # e4m3 cache needs its scale cache
    assert call(D=64) == dsa.DSA_ERR_UNSUPPORTED                 # e4m3 rows are D = 128
    assert call(D=96, dt=0) == dsa.DSA_ERR_UNSUPPORTED
    assert call(dt=5) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert call(PS=0) == dsa.DSA_ERR_INVALID_ARGUMENT



def _prepare_args(dsa, **over):
    a = dsa.dsa_indexer_prepare_args()
    fake = 1 << 20
    a.T, a.hidden_dim, a.q_rank, a.H, a.D, a.rope_dim, a.rope_interleaved = 16, 256, 128, 64, 128, 64, 0
    for f in ("hidden", "qa_normed", "rope_cos", "rope_sin", "wq_b", "wk", "weights_proj", "k_norm_weight",
              "slot_mapping", "k_cache", "k_scale_cache", "q_out", "q_scale_out", "w_out", "workspace"):
        setattr(a, f, fake)
    a.k_norm_eps, a.cache_dtype, a.page_size, a.num_pages, a.workspace_bytes = 1e-6, 1, 64, 4, 1 << 30
    for k, v in over.items():
        setattr(a, k, v)
    return a


def test_prepare_workspace_size_and_validation_without_cuda(dsa):
    import ctypes
    L = dsa.lib()
    n = ctypes.c_size_t(0)
    a = _prepare_args(dsa)
    assert L.dsa_indexer_prepare_workspace_size(ctypes.byref(a), ctypes.byref(n)) == dsa.DSA_OK
    # fp32 q [T, H, D] and k [T, D] before the row kernels, each 256-byte rounded
    assert n.value == 16 * 64 * 128 * 4 + 16 * 128 * 4

    def st(**over):
        return L.dsa_indexer_prepare(ctypes.byref(_prepare_args(dsa, **over)), None)
    assert st(T=0) == dsa.DSA_OK                                  # nothing to do, no launch
    assert st(D=64) == dsa.DSA_ERR_UNSUPPORTED                    # rows of 128 (Hadamard, lane quads)
    assert st(H=48) == dsa.DSA_ERR_UNSUPPORTED
    assert st(hidden_dim=100) == dsa.DSA_ERR_UNSUPPORTED          # rows of 16-byte multiples
    assert st(rope_dim=63) == dsa.DSA_ERR_INVALID_ARGUMENT        # pairs
    assert st(rope_dim=130) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert st(rope_dim=60) == dsa.DSA_ERR_UNSUPPORTED             # half-split pairs need rope_dim % 8 == 0
    assert st(cache_dtype=7) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert st(T=-1) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert st(k_norm_eps=-1.0) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_indexer_prepare_workspace_size(None, ctypes.byref(n)) == dsa.DSA_ERR_INVALID_ARGUMENT


def test_prepare_binding_checks_shapes_before_anything_else(dsa):
    import workloads
    c = workloads.frontend_case(5, 64, 32, 4, rope_dim=16, fp8=True, page_size=16)
    base = dict(hidden=c.hidden, qa_normed=c.qa_normed, rope_cos=c.rope_cos, rope_sin=c.rope_sin, wq_b=c.wq_b,
                wk=c.wk, weights_proj=c.weights_proj, k_norm_weight=c.k_norm_weight, k_cache=c.k_cache,
                slot_mapping=c.slot_mapping)

    def call(**over):
        kw = dict(base, **over)
        return dsa.make_prepare_args(kw.pop("hidden"), kw.pop("qa_normed"), kw.pop("rope_cos"), kw.pop("rope_sin"),
                                     kw.pop("wq_b"), kw.pop("wk"), kw.pop("weights_proj"), kw.pop("k_norm_weight"),
                                     kw.pop("k_cache"), kw.pop("slot_mapping"), H=4, rope_dim=16,
                                     k_scale_cache=kw.pop("k_scale_cache", c.k_scale_cache))
    for bad in [dict(rope_cos=c.rope_cos[:, :4]), dict(wq_b=c.wq_b[:100]), dict(slot_mapping=c.slot_mapping[:3]),
                dict(k_scale_cache=None), dict(qa_normed=c.qa_normed[:4]), dict(wk=c.wk[:64])]:
        with pytest.raises(ValueError, match="shape|must be"):
            call(**bad)
    with pytest.raises(ValueError, match="CUDA"):   # right shapes: the next check is the device
        call()


def test_indexer_binding_checks_shapes_before_anything_else(dsa):
    import torch
    pc = workloads.paged_case([300, 70], [2, 1], 64, 128, 32, page_size=64, integer=True, seed=3)

    def call(**over):
        kw = dict(q=pc.q, w=pc.w, k_cache=pc.k_cache, cu_q_lens=pc.cu_q_lens, seq_lens=pc.seq_lens,
                  block_tables=pc.block_tables)
        kw.update(over)
        extra = {k: kw.pop(k) for k in ("q_scale", "k_scale_cache", "topk", "k_new", "slot_mapping") if k in kw}
        return dsa.make_indexer_args(kw["q"], kw["w"], kw["k_cache"], kw["cu_q_lens"], kw["seq_lens"],
                                     kw["block_tables"], max_seq_len=pc.max_seq_len, topk_limit=32, **extra)
    for bad in [dict(w=pc.w[:2]), dict(cu_q_lens=pc.cu_q_lens[:2]), dict(block_tables=pc.block_tables[:1]),
                dict(topk=torch.empty((3, 16), dtype=torch.int32)), dict(k_cache=pc.k_cache[:, :, :64]),
                dict(k_new=torch.zeros((3, 64), dtype=torch.bfloat16), slot_mapping=torch.zeros(3, dtype=torch.int64)),
                dict(q=pc.q[0])]:
        with pytest.raises(ValueError):
            call(**bad)
    with pytest.raises(ValueError, match="CUDA"):   # right shapes: the next check is the device
        call()


def test_dense_bindings_check_shapes(dsa):
    import torch
    q = torch.zeros((4, 8, 64), dtype=torch.bfloat16)
    k = torch.zeros((16, 64), dtype=torch.bfloat16)
    w = torch.zeros((4, 8))
    with pytest.raises(ValueError, match="w must have shape"):
        dsa.dsa_indexer_scores(q, k, w[:3])
    with pytest.raises(ValueError, match="k must have shape"):
        dsa.dsa_indexer_scores(q, k[:, :32], w)
    with pytest.raises(ValueError, match="S = 16 columns"):
        dsa.dsa_indexer_scores(q, k, w, scores=torch.zeros((4, 12)))
    with pytest.raises(ValueError, match="topk must have shape"):
        dsa.dsa_indexer_topk(torch.zeros((4, 16)), T=4, S=16, q_pos0=12, topk_limit=4, topk=torch.zeros((4, 3), dtype=torch.int32))
    with pytest.raises(ValueError, match="at least"):
        dsa.dsa_indexer_topk(torch.zeros((3, 16)), T=4, S=16, q_pos0=12, topk_limit=4)
    with pytest.raises(ValueError, match="slot_mapping must have shape"):
        dsa.dsa_indexer_cache_append(torch.zeros((5, 128), dtype=torch.bfloat16), torch.zeros(4, dtype=torch.int64),
                                     torch.zeros((2, 16, 128), dtype=torch.bfloat16))


def test_seeded_workloads_repeat_byte_for_byte():
    import torch
    a = workloads.paged_case([300, 70], [2, 1], 64, 128, 32, page_size=64, q_dtype="bf16", k_dtype="fp8_e4m3",
                             seed=5)
    b = workloads.paged_case([300, 70], [2, 1], 64, 128, 32, page_size=64, q_dtype="bf16", k_dtype="fp8_e4m3",
                             seed=5)
    for name in ("q", "w", "k_cache", "k_scale_cache", "block_tables", "cu_q_lens", "seq_lens"):
        x, y = getattr(a, name), getattr(b, name)
        assert torch.equal(x.view(torch.uint8) if x.dtype == torch.float8_e4m3fn else x,
                           y.view(torch.uint8) if y.dtype == torch.float8_e4m3fn else y), name
    f1 = workloads.frontend_case(7, 64, 32, 4, fp8=True, seed=3)
    f2 = workloads.frontend_case(7, 64, 32, 4, fp8=True, seed=3)
    assert torch.equal(f1.hidden, f2.hidden) and torch.equal(f1.slot_mapping, f2.slot_mapping)
    s1 = workloads.sparse_mla_case([50], [2], 2, 8, kv_rank=16, rope_dim=8, page_size=16, seed=4)
    s2 = workloads.sparse_mla_case([50], [2], 2, 8, kv_rank=16, rope_dim=8, page_size=16, seed=4)
    assert torch.equal(s1.topk, s2.topk) and torch.equal(s1.cache_c, s2.cache_c)


def test_sharded_validation(dsa):
    L = dsa.lib()
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    import ctypes
    n = ctypes.c_size_t(0)
    assert L.dsa_indexer_shard_candidates_workspace_size(10, 13, ctypes.byref(n)) == dsa.DSA_OK
    assert n.value == 10 * 16 * 4                                     # rows of ceil4(S) fp32 scores
    assert L.dsa_indexer_shard_candidates_workspace_size(-1, 13, ctypes.byref(n)) == dsa.DSA_ERR_INVALID_ARGUMENT

    def shard(**kw):
        a = dict(q=fake, qd=0, qs=None, k=fake, kd=0, ks=None, w=fake, T=4, S=8, H=64, D=128, p0=4, off=8, kc=4,
                 ci=fake, cs=fake, ws=fake, wsb=4 * 8 * 4, st=None)
        a.update(kw)
        return L.dsa_indexer_shard_candidates(a["q"], a["qd"], a["qs"], a["k"], a["kd"], a["ks"], a["w"], a["T"],
                                              a["S"], a["H"], a["D"], a["p0"], a["off"], a["kc"], a["ci"], a["cs"],
                                              a["ws"], a["wsb"], a["st"])
    assert shard(off=-1) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert shard(p0=-1) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert shard(kc=0) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert shard(kc=5000) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert shard(ci=None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert shard(ws=None) == dsa.DSA_ERR_WORKSPACE
    assert shard(wsb=16) == dsa.DSA_ERR_WORKSPACE
    assert shard(ws=fake + 4) == dsa.DSA_ERR_WORKSPACE
    assert shard(H=48) == dsa.DSA_ERR_UNSUPPORTED
    assert shard(T=0) == dsa.DSA_OK

    def merge(**kw):
        a = dict(cs=fake, ci=fake, n=2, T=4, kc=8, lim=8, ko=8, order=0, out=fake, st=None)
        a.update(kw)
        return L.dsa_indexer_merge_candidates(a["cs"], a["ci"], a["n"], a["T"], a["kc"], a["lim"], a["ko"],
                                              a["order"], a["out"], a["st"])
    assert merge(n=0) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert merge(n=33) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert merge(lim=0) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert merge(order=3) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert merge(ko=5000) == dsa.DSA_ERR_UNSUPPORTED
    assert merge(n=3, kc=8192) == dsa.DSA_ERR_UNSUPPORTED              # more than 16384 per row
    assert merge(out=None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert merge(T=0) == dsa.DSA_OK


def test_clock_sample_validation(dsa):
    L = dsa.lib()
    assert L.dsa_clock_sample(None, 4, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_clock_sample(1 << 20, 0, None) == dsa.DSA_ERR_INVALID_ARGUMENT   # never dereferenced


def test_bench_in_band_clock_from_two_samples():
    import torch
    import bench
    # SM 0: 2.07e6 cycles over 1e6 ns (2070 MHz); SM 1: 1.0e6 cycles over 1e6 ns, sampled twice
    a = torch.tensor([[0, 100, 5_000], [1, 50, 5_000], [1, 60, 5_100]], dtype=torch.int64)
    b = torch.tensor([[0, 2_070_100, 1_005_000], [1, 1_000_050, 1_005_000], [1, 999_990, 1_004_900]],
                     dtype=torch.int64)
    r = bench.sm_clock_in_band(a, b)
    assert r["sms"] == 2
    assert abs(r["sm_mhz_max"] - 2070.0) < 1e-9 and abs(r["sm_mhz_min"] - 1000.0) < 1e-9
    assert bench.sm_clock_in_band(a, torch.tensor([[7, 1, 1]], dtype=torch.int64)) is None  # no SM in both


def test_linear_bucket_scale_keeps_the_floor_below_the_bin_count():
    # the top-k kernels' linear buckets: y = RN(RN(x - lo) * RN((4096 - 2^-10) / width)) must
    # stay below 4096 for every x <= hi (the kernels take floor(y) with no clamp); the
    # largest y comes with x = hi, where x - lo is exactly the rounded width
    import numpy as np
    span = np.float32(4096) - np.float32(2.0 ** -10)
    assert float(span) == 4096 - 2.0 ** -10
    rng = np.random.default_rng(0)
    lo = (rng.standard_normal(400_000) * 10.0 ** rng.integers(-20, 20, 400_000)).astype(np.float32)
    hi = (lo + np.abs(rng.standard_normal(400_000)) * 10.0 ** rng.integers(-20, 20, 400_000)).astype(np.float32)
    width = (hi - lo).astype(np.float32)
    ok = (width > 0) & np.isfinite(width)
    lo, hi, width = lo[ok], hi[ok], width[ok]
    scale = (span / width).astype(np.float32)
    ok = np.isfinite(scale) & (scale > 0)
    y = ((hi[ok] - lo[ok]).astype(np.float32) * scale[ok]).astype(np.float32)
    assert (y < 4096).all() and y.max() > 4095
