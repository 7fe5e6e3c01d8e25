"""GPU parity of sparse MLA over the top-k (dsa_sparse_mla) against the fp64 oracle.

Tolerance from the arithmetic: logits are fp32 sums of 576 exact bf16 products (relative
error ~576 * 2^-24 of sum |q k|, a few 1e-4 after the scale for N(0,1) inputs); the
probabilities enter the P.V product rounded to bf16 (2^-9 relative each) while their sum
is kept in fp32 (another 2^-9 at most), so every output element is within
2^-8 * sum_s p_s |c_s| <= 2^-8 * max_s |c_s| of the exact value; the tests allow 2^-7 times
the largest selected latent magnitude of the row.  Sharper cases pin what that bound
could hide: one selected key returns its latent row exactly (p = 1), equal logits (q = 0)
return the mean of the selected rows to fp32 rounding, and an empty selection returns
zeros -- a dropped, repeated or misplaced key fails these.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import sparse_mla as smla
from oracle import frontend

pytestmark = pytest.mark.gpu

dsa = pytest.importorskip("sparse_attention_token_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _gpu(c, topk=None, q_nope=None, q_rope=None):
    to = lambda t: t.cuda()
    out = dsa.dsa_sparse_mla(to(c.q_nope if q_nope is None else q_nope), to(c.q_rope if q_rope is None else q_rope),
                             to(c.cache_c), to(c.cache_r), to(c.block_tables), to(c.cu_q_lens), to(c.seq_lens),
                             to(c.topk if topk is None else topk), scale=c.scale)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    return out.cpu().numpy().astype(np.float64)


def _oracle(c, topk=None, q_nope=None, q_rope=None):
    return smla.sparse_mla(c.q_nope if q_nope is None else q_nope, c.q_rope if q_rope is None else q_rope,
                           c.cache_c, c.cache_r, c.block_tables, c.cu_q_lens, c.topk if topk is None else topk,
                           page_size=c.page_size, scale=c.scale)


def _row_bound(c, topk):
    """Largest |c_kv| over each query row's selected keys (1 for an empty row)."""
    cc = frontend.to_f64(c.cache_c)
    bt = c.block_tables.numpy()
    cu = c.cu_q_lens.numpy()
    tk = topk.numpy()
    out = np.ones(tk.shape[0])
    for b in range(len(cu) - 1):
        for t in range(cu[b], cu[b + 1]):
            sel = tk[t][tk[t] >= 0]
            if sel.size:
                rows = cc[bt[b][sel // c.page_size], sel % c.page_size]
                out[t] = np.abs(rows).max()
    return out


def _assert_close(got, ref, bound):
    tol = 2.0 ** -7 * bound[:, None, None] + 1e-6
    err = np.abs(got - ref)
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert np.all(err <= tol), f"error {err[worst]:.3e} > {tol[worst]:.3e} at {worst}"


@pytest.mark.parametrize("H,page_size,k", [(64, 64, 160), (16, 16, 64), (32, 64, 300), (128, 32, 200)])
def test_sparse_mla_gaussian(H, page_size, k):
    c = workloads.sparse_mla_case([700, 90, 1500], [2, 1, 3], H, k, page_size=page_size, seed=100 + H)
    got, ref = _gpu(c), _oracle(c)
    _assert_close(got, ref, _row_bound(c, c.topk))


def test_sparse_mla_single_key_is_its_latent_row():
    c = workloads.sparse_mla_case([500, 130], [3, 1], 64, 96, page_size=64, seed=111)
    tk = torch.full_like(c.topk, -1)
    tk[:, 37] = torch.tensor([5, 0, 499, 129], dtype=torch.int32)   # one key anywhere in the row
    got = _gpu(c, topk=tk)
    ref = _oracle(c, topk=tk)
    assert np.array_equal(got, ref)                                # p = 1: the row itself, exactly


def test_sparse_mla_equal_logits_average_the_selection():
    c = workloads.sparse_mla_case([2600, 400], [2, 2], 64, 2048, page_size=64, seed=112)
    zn, zr = torch.zeros_like(c.q_nope), torch.zeros_like(c.q_rope)
    got = _gpu(c, q_nope=zn, q_rope=zr)
    ref = _oracle(c, q_nope=zn, q_rope=zr)
    assert np.allclose(got, ref, rtol=0, atol=2e-6 * np.abs(ref).max() + 1e-7)


def test_sparse_mla_empty_rows_and_padding():
    c = workloads.sparse_mla_case([300, 200], [2, 2], 32, 128, page_size=16, seed=113)
    tk = c.topk.clone()
    tk[1] = -1                                                      # an empty selection
    tk[2, 64:] = -1                                                 # a row of half padding
    got = _gpu(c, topk=tk)
    ref = _oracle(c, topk=tk)
    assert np.all(got[1] == 0)
    _assert_close(got, ref, _row_bound(c, tk))


def test_sparse_mla_decode_b64_topk_2048():
    lens = workloads.decode_lens(64, 2100, 4096, 3)
    c = workloads.sparse_mla_case(lens, [1] * 64, 64, 2048, page_size=64, seed=114)
    got, ref = _gpu(c), _oracle(c)
    _assert_close(got, ref, _row_bound(c, c.topk))
