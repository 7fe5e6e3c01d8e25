"""CPU oracle for sparse MLA over the indexer's top-k -- TEST INFRASTRUCTURE ONLY (numpy, fp64).

The GLM5 TensorCast adaptation design hands the indexer's ``topk_indices`` (and
``topk_limit``) to the multi-head latent attention backend, whose attention length is
capped by the top-k width ("Sparse MLA 配置兼容", the ``_get_backend_kwargs`` hand-off, and
the performance model's sparse prefill / decode length).  The page gives no formula;
the reading taken here is multi-head latent attention in its absorbed form, restricted
to the selected keys:

  for query token t and head h, with the selected logical key positions
  S(t) = { topk[t, j] : topk[t, j] >= 0 } of the token's sequence,

      logit[t, h, s] = scale * (q_nope[t, h] . c_kv[s] + q_rope[t, h] . k_rope[s])
      p[t, h, :]     = softmax over s in S(t)
      out[t, h]      = sum_{s in S(t)} p[t, h, s] * c_kv[s]               (latent output)

where c_kv [.., kv_rank] is the compressed latent row of key s and k_rope [.., rope_dim]
its rotary part, both read from the paged latent cache through block_tables; q_nope is
the query already multiplied into the latent space (the up-projection absorbed), and the
caller applies the value up-projection and output projection to ``out``.  A row whose
selection is empty (all -1) outputs zeros.

Pinned by ``tests/test_oracle_pins.py``: one selected key returns its latent row, equal
logits average the selected rows, the selection's order and -1 padding do not matter,
adding a constant to every logit changes nothing, and selecting every causal key equals
dense causal attention computed by torch's scaled_dot_product_attention.
"""
from __future__ import annotations

import numpy as np
import torch


def _f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to(torch.float64).cpu().numpy()
    return np.asarray(t, dtype=np.float64)


def gather_latent(cache_c: np.ndarray, cache_r: np.ndarray, block_table: np.ndarray, page_size: int,
                  positions: np.ndarray):
    """Latent rows (c_kv, k_rope) of logical key positions of one sequence."""
    pages = block_table[positions // page_size]
    rows = positions % page_size
    return cache_c[pages, rows], cache_r[pages, rows]


def sparse_mla(q_nope, q_rope, cache_c, cache_r, block_tables, cu_q_lens, topk, *, page_size: int,
               scale: float) -> np.ndarray:
    """out [total_q, H, kv_rank] in fp64.

    q_nope [total_q, H, kv_rank], q_rope [total_q, H, rope_dim]; cache_c [pages, page_size,
    kv_rank], cache_r [pages, page_size, rope_dim]; block_tables [B, max_pages]; cu_q_lens
    [B + 1]; topk [total_q, k] int (logical positions, -1 = none)."""
    qn, qr = _f64(q_nope), _f64(q_rope)
    cc, cr = _f64(cache_c), _f64(cache_r)
    bt = np.asarray(block_tables.cpu().numpy() if isinstance(block_tables, torch.Tensor) else block_tables)
    cu = np.asarray(cu_q_lens.cpu().numpy() if isinstance(cu_q_lens, torch.Tensor) else cu_q_lens)
    tk = np.asarray(topk.cpu().numpy() if isinstance(topk, torch.Tensor) else topk)
    total_q, H, R = qn.shape
    out = np.zeros((total_q, H, R), dtype=np.float64)
    for b in range(len(cu) - 1):
        for t in range(int(cu[b]), int(cu[b + 1])):
            sel = tk[t][tk[t] >= 0].astype(np.int64)
            if sel.size == 0:
                continue
            c, r = gather_latent(cc, cr, bt[b], page_size, sel)        # [n, R], [n, rope]
            logits = scale * (qn[t] @ c.T + qr[t] @ r.T)                # [H, n]
            logits -= logits.max(axis=1, keepdims=True)
            p = np.exp(logits)
            p /= p.sum(axis=1, keepdims=True)
            out[t] = p @ c
    return out
