"""GPU parity of the indexer front-end (dsa_indexer_prepare) against the fp64 oracle.

Tolerances follow from the arithmetic: the projections are bf16 GEMMs accumulated in
fp32 (error at most ~K * 2^-24 of sum |a b|), the layer norm, RoPE and Hadamard rotation
add a few fp32 roundings, and the outputs are rounded once more -- to bf16 (relative
error 2^-8, 2^-7 if an fp32 difference flips a rounding) or to e4m3 (2^-4, 2^-3 with a
flip, plus the subnormal spacing scale * 2^-9).  Every comparison allows the output
rounding plus 2^-12 of the row's rms for the fp32 work before it.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import frontend
import sparse_attention_token_gb300 as dsa
import workloads
from tests.parity import RTOL, assert_topk_valid

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _to(t):
    return None if t is None else t.to(DEV)


def run_gpu(c, interleaved=False, eps=1e-6):
    cache = _to(c.k_cache.clone())
    scales = _to(None if c.k_scale_cache is None else c.k_scale_cache.clone())
    q, qs, w = dsa.dsa_indexer_prepare(_to(c.hidden), _to(c.qa_normed), _to(c.rope_cos), _to(c.rope_sin),
                                       _to(c.wq_b), _to(c.wk), _to(c.weights_proj), _to(c.k_norm_weight), cache,
                                       _to(c.slot_mapping), H=c.H, rope_dim=c.rope_dim, rope_interleaved=interleaved,
                                       k_norm_bias=_to(c.k_norm_bias), k_norm_eps=eps, k_scale_cache=scales)
    torch.cuda.synchronize()
    status = dsa.dsa_check_device_status()
    return dict(q=q.cpu(), q_scale=None if qs is None else qs.cpu(), w=w.cpu(), cache=cache.cpu(),
                scales=None if scales is None else scales.cpu(), status=status)


def run_oracle(c, interleaved=False, eps=1e-6):
    return frontend.prepare(c.hidden, c.qa_normed, c.rope_cos, c.rope_sin, c.wq_b, c.wk, c.weights_proj,
                            c.k_norm_weight, c.k_norm_bias, H=c.H, D=c.D, rope_dim=c.rope_dim,
                            interleaved=interleaved, eps=eps, fp8=c.k_cache.dtype == torch.float8_e4m3fn)


def _rms(ref):
    return np.sqrt((ref ** 2).mean(axis=-1, keepdims=True))


def assert_bf16_close(got, ref, what):
    g = got.to(torch.float64).numpy().reshape(ref.shape)
    tol = np.abs(ref) * 2.0 ** -7 + _rms(ref) * 2.0 ** -12
    bad = np.abs(g - ref) > tol
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, worst {np.max(np.abs(g - ref) - tol)}"


def assert_e4m3_close(codes, scales, ref, ref_scales, what):
    s = scales.to(torch.float64).numpy().reshape(ref_scales.shape)
    assert np.all(np.abs(s - ref_scales) <= ref_scales * 2.0 ** -12), f"{what}: scales"
    c = codes.view(torch.uint8).numpy().reshape(ref.shape)
    dq = frontend.dequantize(c, s)
    tol = np.abs(ref) * 2.0 ** -3 + s[..., None] * 2.0 ** -9 + _rms(ref) * 2.0 ** -12
    bad = np.abs(dq - ref) > tol
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance"
    return c


def assert_w_close(got, c, ref):
    # fp32 accumulation of K products: |error| <= K * 2^-24 * sum |a b| (times 4 for any order)
    A = frontend.linear(np.abs(frontend.to_f64(c.hidden)), np.abs(frontend.to_f64(c.weights_proj)))
    K = c.hidden.shape[1]
    assert np.all(np.abs(got.numpy().astype(np.float64) - ref) <= 4 * K * 2.0 ** -24 * A + 1e-30)


def cache_rows(out, c):
    """The rows the call wrote (valid slots, in token order) and a check that every other
    slot of the cache is untouched (still zero)."""
    slots = c.slot_mapping.numpy()
    n_slots = c.k_cache.shape[0] * c.k_cache.shape[1]
    valid = (slots >= 0) & (slots < n_slots)
    flat = out["cache"].reshape(n_slots, c.D)
    other = np.ones(n_slots, dtype=bool)
    other[slots[valid]] = False
    raw = flat.view(torch.uint8) if flat.dtype == torch.float8_e4m3fn else flat.view(torch.int16)
    assert not raw[torch.from_numpy(other)].any(), "a slot outside slot_mapping was written"
    sc = None if out["scales"] is None else out["scales"].reshape(n_slots)[torch.from_numpy(slots[valid])]
    return raw[torch.from_numpy(slots[valid])].view(flat.dtype), sc, valid


@pytest.mark.parametrize("interleaved", [False, True])
def test_frontend_bf16_cache(interleaved):
    c = workloads.frontend_case(37, 512, 256, 64, rope_dim=64, seed=1)
    got, ref = run_gpu(c, interleaved), run_oracle(c, interleaved)
    assert got["status"] == dsa.DSA_OK
    assert got["q"].dtype == torch.bfloat16 and got["q_scale"] is None
    assert_bf16_close(got["q"], ref["q"], "q")
    assert_w_close(got["w"], c, ref["w"])
    rows, _, valid = cache_rows(got, c)
    assert_bf16_close(rows, ref["k"][valid], "k")


@pytest.mark.parametrize("interleaved,bias,rope_dim,H", [(False, False, 64, 64), (True, True, 64, 32),
                                                         (False, True, 128, 16), (True, False, 0, 8)])
def test_frontend_e4m3_cache(interleaved, bias, rope_dim, H):
    c = workloads.frontend_case(45, 384, 256, H, rope_dim=rope_dim, fp8=True, bias=bias, pos0=1000, seed=2 + H)
    got, ref = run_gpu(c, interleaved), run_oracle(c, interleaved)
    assert got["status"] == dsa.DSA_OK
    assert got["q"].dtype == torch.float8_e4m3fn
    qc = assert_e4m3_close(got["q"], got["q_scale"], ref["q"], ref["q_scale"].astype(np.float64), "q")
    assert (qc == ref["q_codes"]).mean() > 0.99
    assert_w_close(got["w"], c, ref["w"])
    rows, sc, valid = cache_rows(got, c)
    kc = assert_e4m3_close(rows, sc, ref["k"][valid], ref["k_scale"][valid].astype(np.float64), "k")
    assert (kc == ref["k_codes"][valid]).mean() > 0.99


def test_frontend_padding_and_bad_slot():
    c = workloads.frontend_case(24, 256, 128, 64, fp8=True, pad_every=5, seed=9)
    c.slot_mapping[7] = c.k_cache.shape[0] * c.k_cache.shape[1] + 3   # past the cache: skipped, reported
    got, ref = run_gpu(c), run_oracle(c)
    assert got["status"] == dsa.DSA_ERR_DEVICE_CHECK
    c.slot_mapping[7] = -1                                               # compare the rest as a padded token
    rows, sc, valid = cache_rows(got, c)
    assert_e4m3_close(rows, sc, ref["k"][valid], ref["k_scale"][valid].astype(np.float64), "k")
    assert_e4m3_close(got["q"], got["q_scale"], ref["q"], ref["q_scale"].astype(np.float64), "q")


def test_frontend_then_indexer_prefill():
    # one sequence of T new tokens: the front-end writes its keys into the pages of the
    # block table, then dsa_indexer selects from them; the selection matches the oracle
    # run on the same bytes
    T, page = 300, 64
    c = workloads.frontend_case(T, 512, 256, 64, fp8=True, page_size=page, num_pages=8, seed=11)
    perm = torch.randperm(8, generator=torch.Generator().manual_seed(3)).to(torch.int32)
    pos = torch.arange(T)
    c.slot_mapping = (perm[pos // page].to(torch.int64) * page + pos % page)
    got = run_gpu(c)
    assert got["status"] == dsa.DSA_OK
    pc = workloads.PagedCase(q=got["q"], q_scale=got["q_scale"], w=got["w"], k_cache=got["cache"],
                             k_scale_cache=got["scales"], cu_q_lens=torch.tensor([0, T], dtype=torch.int32),
                             seq_lens=torch.tensor([T], dtype=torch.int32), block_tables=perm[None, :].contiguous(),
                             B=1, H=64, D=128, page_size=page, topk_limit=64, k_out=64, q_dtype="fp8_e4m3",
                             k_dtype="fp8_e4m3", max_seq_len=T)
    tk = dsa.dsa_indexer(_to(pc.q), _to(pc.w), _to(pc.k_cache), _to(pc.cu_q_lens), _to(pc.seq_lens),
                         _to(pc.block_tables), max_seq_len=T, topk_limit=64, q_scale=_to(pc.q_scale),
                         k_scale_cache=_to(pc.k_scale_cache))
    torch.cuda.synchronize()
    ref, rs, rb = oracle.paged(pc, want_scores=True, want_bound=True)
    assert_topk_valid(tk.cpu().numpy(), ref, rs, rb, oracle.query_positions(pc) + 1, 64, RTOL["fp8_e4m3"],
                      exact=False)
