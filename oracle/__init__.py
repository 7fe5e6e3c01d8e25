"""CPU oracle for the DSA indexer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library under
``sparse_attention_token_gb300/`` and never imports it.

Contents:
  * ``dense`` / ``paged``: ctypes wrappers over the plain C oracle
    (``dsa_oracle.c``): fp64 dot products, ReLU, head-weighted sum, full sort
    per row by (score desc, index asc), -1 padding.
  * ``topk_of_scores``: the same full-sort top-k applied to given fp64 scores.
  * ``resolve_indexer_sources`` / ``stack``: GLM-5.2 IndexShare -- a "shared"
    layer forwards the top-k of the nearest earlier "full" layer unchanged
    (GLM5 TensorCast adaptation design, section "GLM-5.2 IndexShare").
  * ``brute``: an exact rational-arithmetic brute force for tiny inputs,
    used to pin the C oracle.
  * ``e4m3_encode`` / ``cache_append``: the FP8 key-cache write (per-token
    amax/448 quantisation through slot_mapping).
  * ``frontend`` (numpy, fp64): the indexer front-end -- projections, k layer
    norm, RoPE, Hadamard rotation, per-row e4m3 quantisation.
  * ``sparse_mla`` (numpy, fp64): absorbed latent attention over each token's
    selected keys (the consumer of the top-k).
  * ``sharded``: the key-sharded top-k -- each shard's best (score, index)
    candidates, and the exact merge of the gathered candidates.

Every function in this package is pinned by ``tests/test_oracle_pins.py``
(hand-worked example, library special cases, invariants, brute force).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

from . import build as _build

ORDER_SCORE = 0   # rows sorted by (score desc, index asc): torch.topk order, ties to lower index
ORDER_INDEX = 1   # the same set, ascending key index

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_dense.restype = i32
        lib.oracle_dense.argtypes = [i32, i32, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                     i32, P, i32, P, P, P, i64, i32]
        lib.oracle_paged.restype = i32
        lib.oracle_paged.argtypes = [i32, i32, P, P, P, P, P, i32, i32, P, i32, P, P, i32, i32,
                                     i32, i32, i32, i32, P, i32, P, P, P, i64, i32]
        lib.oracle_topk.restype = i32
        lib.oracle_topk.argtypes = [P, i64, i32, P, i32, i32, i32, P, i32]
        lib.oracle_max_threads.restype = i32
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_cache_append.restype = i32
        lib.oracle_cache_append.argtypes = [P, i32, i32, P, i32, P, P, i64]
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return 0
    if t.dtype == torch.float8_e4m3fn:
        return 1
    raise TypeError(f"oracle: unsupported storage dtype {t.dtype}")


def _raw(t: Optional[torch.Tensor]):
    """A contiguous CPU numpy view of a tensor's bytes (kept alive by the caller)."""
    if t is None:
        return None
    t = t.detach().to("cpu").contiguous()
    if t.dtype in (torch.bfloat16,):
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def decode_bf16(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits) & 0xFFFF))


def decode_e4m3(code: int) -> float:
    return float(_load().oracle_e4m3_to_double(int(code) & 0xFF))


def dense(q, k, w, *, T: int, S: int, H: int, D: int, q_pos0: int, topk_limit: int, k_out: int,
          q_scale=None, k_scale=None, rows: Optional[Sequence[int]] = None, order: int = ORDER_SCORE,
          want_scores: bool = False, want_bound: bool = False, n_threads: int = 0):
    """Oracle for one dense sequence; returns (topk int32 [n, k_out], scores, bound)."""
    lib = _load()
    qa, ka, wa = _raw(q), _raw(k), _raw(w.to(torch.float32))
    qs = _raw(q_scale.to(torch.float32)) if q_scale is not None else None
    ks = _raw(k_scale.to(torch.float32)) if k_scale is not None else None
    rows_a = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = T if rows is None else len(rows_a)
    topk = np.empty((n, k_out), dtype=np.int32)
    ld = max(S, 1)
    scores = np.empty((n, ld), dtype=np.float64) if want_scores else None
    bound = np.empty((n, ld), dtype=np.float64) if want_bound else None
    rc = lib.oracle_dense(_dtype_code(q), _dtype_code(k), _ptr(qa), _ptr(qs), _ptr(wa), _ptr(ka),
                          _ptr(ks), T, S, H, D, q_pos0, topk_limit, k_out, order, _ptr(rows_a),
                          n, _ptr(topk), _ptr(scores), _ptr(bound), ld, n_threads)
    if rc != 0:
        raise ValueError("oracle_dense: NaN input")
    return topk, scores, bound


def paged(case, *, rows: Optional[Sequence[int]] = None, order: int = ORDER_SCORE,
          want_scores: bool = False, want_bound: bool = False, n_threads: int = 0,
          topk_limit: Optional[int] = None, k_out: Optional[int] = None):
    """Oracle for a paged varlen batch (a ``workloads.PagedCase``-like object)."""
    lib = _load()
    topk_limit = case.topk_limit if topk_limit is None else topk_limit
    k_out = case.k_out if k_out is None else k_out
    qa, ka, wa = _raw(case.q), _raw(case.k_cache), _raw(case.w.to(torch.float32))
    qs = _raw(case.q_scale.to(torch.float32)) if case.q_scale is not None else None
    ks = _raw(case.k_scale_cache.to(torch.float32)) if case.k_scale_cache is not None else None
    bt = _raw(case.block_tables.to(torch.int32))
    cu = _raw(case.cu_q_lens.to(torch.int32))
    sl = _raw(case.seq_lens.to(torch.int32))
    total_q = int(cu[-1])
    rows_a = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = total_q if rows is None else len(rows_a)
    topk = np.empty((n, k_out), dtype=np.int32)
    ld = max(int(sl.max()) if len(sl) else 1, 1)
    scores = np.empty((n, ld), dtype=np.float64) if want_scores else None
    bound = np.empty((n, ld), dtype=np.float64) if want_bound else None
    rc = lib.oracle_paged(_dtype_code(case.q), _dtype_code(case.k_cache), _ptr(qa), _ptr(qs),
                          _ptr(wa), _ptr(ka), _ptr(ks), int(case.k_cache.shape[0]),
                          int(case.k_cache.shape[1]), _ptr(bt), int(bt.shape[1]), _ptr(cu), _ptr(sl),
                          int(len(sl)), int(case.q.shape[1]), int(case.q.shape[2]), topk_limit, k_out,
                          order, _ptr(rows_a), n, _ptr(topk), _ptr(scores), _ptr(bound), ld, n_threads)
    if rc != 0:
        raise ValueError("oracle_paged: NaN input or key outside the page table")
    return topk, scores, bound


def topk_of_scores(scores: np.ndarray, n_visible: Sequence[int], topk_limit: int, k_out: int,
                   order: int = ORDER_SCORE, n_threads: int = 0) -> np.ndarray:
    """Full-sort top-k of given fp64 score rows (row r uses its first n_visible[r] entries)."""
    lib = _load()
    sc = np.ascontiguousarray(scores, dtype=np.float64)
    nv = np.ascontiguousarray(np.asarray(n_visible, dtype=np.int64))
    out = np.empty((sc.shape[0], k_out), dtype=np.int32)
    lib.oracle_topk(_ptr(sc), sc.shape[1], sc.shape[0], _ptr(nv), topk_limit, k_out, order,
                    _ptr(out), n_threads)
    return out


def query_positions(case) -> np.ndarray:
    """Position of every query row of a paged case: seq_len - q_len + i."""
    cu = case.cu_q_lens.tolist()
    sl = case.seq_lens.tolist()
    pos = []
    for b in range(len(sl)):
        ql = cu[b + 1] - cu[b]
        pos.extend(range(sl[b] - ql, sl[b]))
    return np.asarray(pos, dtype=np.int64)


# ---- GLM-5.2 IndexShare ------------------------------------------------------

FULL, SHARED = "full", "shared"


def resolve_indexer_sources(indexer_types: Sequence[str], num_layers: Optional[int] = None):
    """Source layer of every layer: a full layer is its own source; a shared layer
    takes the nearest earlier full layer.  Raises ValueError for a list shorter
    than num_layers, an unknown type, or a shared layer with no earlier full layer
    (GLM5 TensorCast adaptation design, "GLM-5.2 IndexShare")."""
    types = list(indexer_types)
    if num_layers is not None and len(types) < num_layers:
        raise ValueError("indexer_types shorter than the number of layers")
    src = []
    last_full = None
    for i, t in enumerate(types):
        if t == FULL:
            last_full = i
            src.append(i)
        elif t == SHARED:
            if last_full is None:
                raise ValueError(f"shared layer {i} has no earlier full layer")
            src.append(last_full)
        else:
            raise ValueError(f"unknown indexer type {t!r} at layer {i}")
    return src


def stack(indexer_types: Sequence[str], layers, **kw):
    """Per-layer top-k of an IndexShare stack: full layers run the oracle on their own
    inputs, shared layers return their source layer's result object unchanged."""
    src = resolve_indexer_sources(indexer_types)
    out = []
    for i, s in enumerate(src):
        if s == i:
            out.append(paged(layers[i], **kw)[0])
        else:
            out.append(out[s])
    return src, out


def e4m3_encode(values) -> np.ndarray:
    """e4m3 codes (uint8) of fp32 values: nearest finite code, ties to the even code,
    saturating at +-448, sign copied (see ``oracle_e4m3_encode``)."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib.oracle_e4m3_encode(float(x)) for x in v], dtype=np.uint8)


def cache_append(k_new: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                 k_scale_cache: Optional[torch.Tensor] = None):
    """Copies of (k_cache, k_scale_cache) after writing the bf16 rows ``k_new [n, D]`` to
    the slots ``slot_mapping [n]`` (page * page_size + row; negative = skip): a bf16
    cache takes the rows as they are, an e4m3 cache takes them quantised with one
    scale = amax / 448 per token (the GLM5 TensorCast adaptation design's FP8 key and
    scale cache write).  Raises ValueError on a slot past the cache."""
    lib = _load()
    if k_new.dtype != torch.bfloat16:
        raise TypeError("k_new must be bf16")
    n, D = k_new.shape
    kn = np.ascontiguousarray(k_new.contiguous().view(torch.int16).numpy())
    sl = np.ascontiguousarray(slot_mapping.to(torch.int64).numpy())
    fp8 = k_cache.dtype == torch.float8_e4m3fn
    cache = k_cache.clone().contiguous()
    cache_raw = np.ascontiguousarray(cache.view(torch.uint8 if fp8 else torch.int16).numpy())
    scales = None
    if fp8:
        if k_scale_cache is None:
            raise ValueError("an e4m3 cache needs its scale cache")
        scales = np.ascontiguousarray(k_scale_cache.to(torch.float32).clone().numpy())
    n_slots = cache.shape[0] * cache.shape[1]
    rc = lib.oracle_cache_append(_ptr(kn), n, D, _ptr(sl), 1 if fp8 else 0, _ptr(cache_raw), _ptr(scales), n_slots)
    if rc != 0:
        raise ValueError("cache_append: slot outside the cache")
    out = torch.from_numpy(cache_raw).view(k_cache.dtype).reshape(k_cache.shape)
    return out, (torch.from_numpy(scales).reshape(k_scale_cache.shape) if fp8 else k_scale_cache)

