"""Python binding of the GB300 DSA indexer library (libdsa_indexer.so).

Argument marshalling only: every step of the indexer runs in the CUDA kernels
behind the C ABI of include/dsa_indexer.h.  Tensors must be CUDA tensors; the
library is loaded with ctypes and there is no fallback -- if the library is
missing or a call fails, an exception is raised.

Function names mirror the C ABI:
  dsa_indexer_scores, dsa_indexer_topk, dsa_indexer, dsa_indexer_workspace_size,
  dsa_indexer_dense_host, dsa_indexer_dense_host_workspace_size, dsa_indexer_cache_append,
  dsa_resolve_indexer_sources, dsa_indexer_stack, dsa_check_device_status,
  dsa_topk_width, dsa_status_string, dsa_version (and the others the header declares;
  dsa_clock_sample is a diagnostic for measuring the SM clock over an interval).
Host helpers from the GLM5 TensorCast adaptation design ("Sparse MLA 配置兼容",
"GLM-5.2 IndexShare"): resolve_topk_limit, extend_indexer_types_for_mtp,
indexer_types_to_codes.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdsa_indexer.so")

DSA_OK = 0
DSA_ERR_INVALID_ARGUMENT = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_CUDA = 3
DSA_ERR_DEVICE_CHECK = 4
DSA_ERR_TIMEOUT = 5
DSA_ERR_WORKSPACE = 6

DSA_BF16 = 0
DSA_FP8_E4M3 = 1
DSA_LAYER_FULL = 0
DSA_LAYER_SHARED = 1
DSA_ORDER_SCORE = 0
DSA_ORDER_INDEX = 1
DSA_MAX_TOPK = 4096


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {dsa_status_string(status)} ({status})")


class dsa_indexer_args(ctypes.Structure):
    _fields_ = [
        ("q_dtype", ctypes.c_int), ("k_dtype", ctypes.c_int), ("B", ctypes.c_int),
        ("total_q", ctypes.c_int), ("H", ctypes.c_int), ("D", ctypes.c_int),
        ("page_size", ctypes.c_int), ("num_pages", ctypes.c_int),
        ("max_pages_per_seq", ctypes.c_int), ("max_seq_len", ctypes.c_int),
        ("q", ctypes.c_void_p), ("q_scale", ctypes.c_void_p), ("w", ctypes.c_void_p),
        ("cu_q_lens", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p), ("k_cache", ctypes.c_void_p),
        ("k_scale_cache", ctypes.c_void_p), ("topk_limit", ctypes.c_int), ("k_out", ctypes.c_int),
        ("order", ctypes.c_int), ("topk", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t), ("k_new", ctypes.c_void_p), ("slot_mapping", ctypes.c_void_p),
    ]


class dsa_sparse_mla_args(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("total_q", ctypes.c_int), ("H", ctypes.c_int), ("kv_rank", ctypes.c_int),
                ("rope_dim", ctypes.c_int), ("page_size", ctypes.c_int), ("num_pages", ctypes.c_int),
                ("max_pages_per_seq", ctypes.c_int), ("topk_width", ctypes.c_int), ("scale", ctypes.c_float),
                ("q_nope", ctypes.c_void_p), ("q_rope", ctypes.c_void_p), ("cache_c", ctypes.c_void_p),
                ("cache_r", ctypes.c_void_p), ("block_tables", ctypes.c_void_p), ("cu_q_lens", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("topk", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class dsa_indexer_prepare_args(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int), ("hidden_dim", ctypes.c_int), ("q_rank", ctypes.c_int), ("H", ctypes.c_int),
        ("D", ctypes.c_int), ("rope_dim", ctypes.c_int), ("rope_interleaved", ctypes.c_int),
        ("hidden", ctypes.c_void_p), ("qa_normed", ctypes.c_void_p), ("rope_cos", ctypes.c_void_p),
        ("rope_sin", ctypes.c_void_p), ("wq_b", ctypes.c_void_p), ("wk", ctypes.c_void_p),
        ("weights_proj", ctypes.c_void_p), ("k_norm_weight", ctypes.c_void_p), ("k_norm_bias", ctypes.c_void_p),
        ("k_norm_eps", ctypes.c_float), ("cache_dtype", ctypes.c_int), ("slot_mapping", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p), ("k_scale_cache", ctypes.c_void_p), ("page_size", ctypes.c_int),
        ("num_pages", ctypes.c_int), ("q_out", ctypes.c_void_p), ("q_scale_out", ctypes.c_void_p),
        ("w_out", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


_LIB = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        L.dsa_status_string.restype = ctypes.c_char_p
        L.dsa_status_string.argtypes = [I]
        L.dsa_version.restype = ctypes.c_char_p
        L.dsa_topk_width.restype = I
        L.dsa_topk_width.argtypes = [I, I64]
        L.dsa_indexer_scores.restype = I
        L.dsa_indexer_scores.argtypes = [P, I, P, P, I, P, P, I, I, I, I, I, P, I64, P]
        L.dsa_indexer_topk.restype = I
        L.dsa_indexer_topk.argtypes = [P, I64, I, I, I, I, I, I, P, P]
        L.dsa_indexer_workspace_size.restype = I
        L.dsa_indexer_workspace_size.argtypes = [ctypes.POINTER(dsa_indexer_args), ctypes.POINTER(S)]
        L.dsa_indexer.restype = I
        L.dsa_indexer.argtypes = [ctypes.POINTER(dsa_indexer_args), P]
        L.dsa_resolve_indexer_sources.restype = I
        L.dsa_resolve_indexer_sources.argtypes = [I, P, P]
        L.dsa_indexer_stack.restype = I
        L.dsa_indexer_stack.argtypes = [I, P, P, P, P, P]
        L.dsa_check_device_status.restype = I
        L.dsa_check_device_status.argtypes = [P]
        L.dsa_clock_sample.restype = I
        L.dsa_clock_sample.argtypes = [P, I, P]
        L.dsa_indexer_prepare_workspace_size.restype = I
        L.dsa_indexer_prepare_workspace_size.argtypes = [ctypes.POINTER(dsa_indexer_prepare_args), ctypes.POINTER(S)]
        L.dsa_indexer_prepare.restype = I
        L.dsa_indexer_prepare.argtypes = [ctypes.POINTER(dsa_indexer_prepare_args), P]
        L.dsa_indexer_cache_append.restype = I
        L.dsa_indexer_cache_append.argtypes = [P, I, I, P, P, I, P, I, I, P]
        L.dsa_indexer_dense_host_workspace_size.restype = I
        L.dsa_indexer_dense_host_workspace_size.argtypes = [I, I, I, I, I, I, I, ctypes.POINTER(S)]
        L.dsa_indexer_dense_host.restype = I
        L.dsa_indexer_dense_host.argtypes = [P, I, P, P, I, P, P, I, I, I, I, I, I, I, I, I, P, P, S, P]
        L.dsa_indexer_shard_candidates_workspace_size.restype = I
        L.dsa_indexer_shard_candidates_workspace_size.argtypes = [I, I, ctypes.POINTER(S)]
        L.dsa_indexer_shard_candidates.restype = I
        L.dsa_indexer_shard_candidates.argtypes = [P, I, P, P, I, P, P, I, I, I, I, I, I, I, P, P, P, S, P]
        L.dsa_indexer_merge_candidates.restype = I
        L.dsa_indexer_merge_candidates.argtypes = [P, P, I, I, I, I, I, I, P, P]
        L.dsa_sparse_mla_workspace_size.restype = I
        L.dsa_sparse_mla_workspace_size.argtypes = [ctypes.POINTER(dsa_sparse_mla_args), ctypes.POINTER(S)]
        L.dsa_sparse_mla.restype = I
        L.dsa_sparse_mla.argtypes = [ctypes.POINTER(dsa_sparse_mla_args), P]
        L.dsa_test_arm_score_timeout.restype = I
        L.dsa_test_arm_score_timeout.argtypes = [ctypes.c_ulonglong]
        _LIB = L
    return _LIB


def _check(status: int, where: str):
    if status != DSA_OK:
        raise DsaError(status, where)


def dsa_status_string(status: int) -> str:
    return lib().dsa_status_string(int(status)).decode()


def dsa_version() -> str:
    return lib().dsa_version().decode()


def dsa_topk_width(topk_limit: int, active_seq_len: int) -> int:
    return int(lib().dsa_topk_width(int(topk_limit), int(active_seq_len)))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DSA_BF16
    if t.dtype == torch.float8_e4m3fn:
        return DSA_FP8_E4M3
    raise TypeError(f"unsupported element type {t.dtype} (bf16 or float8_e4m3fn)")


def _dev(t: Optional[torch.Tensor], name: str, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    """Raw cudaStream_t of `stream` (default: torch's current stream; NULL without CUDA)."""
    if stream is None:
        if not torch.cuda.is_available():
            return None
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _expect(checks) -> None:
    """Raise ValueError unless every (tensor or None, name, shape) matches; a shape entry
    of None accepts any size in that dimension.  The C ABI sees only pointers and sizes."""
    for t, name, shape in checks:
        if t is None:
            continue
        ok = t.dim() == len(shape) and all(w is None or t.shape[i] == w for i, w in enumerate(shape))
        if not ok:
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def dsa_indexer_scores(q: torch.Tensor, k: torch.Tensor, w: torch.Tensor, *, q_pos0: Optional[int] = None,
                       q_scale: Optional[torch.Tensor] = None, k_scale: Optional[torch.Tensor] = None,
                       scores: Optional[torch.Tensor] = None, ld: Optional[int] = None,
                       fill=float("-inf"), stream=None) -> torch.Tensor:
    """Dense scores [T, ld] fp32 of queries q [T, H, D] against keys k [S, D].

    Entries a query cannot see (s > q_pos0 + t) are left as the output buffer held
    them: a freshly allocated buffer is filled with ``fill`` (by torch) first."""
    T, H, D = q.shape
    S = k.shape[0]
    if q_pos0 is None:
        q_pos0 = S - T
    if ld is None:
        ld = (S + 3) // 4 * 4
    if scores is None:
        scores = torch.full((T, ld), fill, dtype=torch.float32, device=q.device)
    _expect([(k, "k", (S, D)), (w, "w", (T, H)), (q_scale, "q_scale", (T, H)), (k_scale, "k_scale", (S,)),
             (scores, "scores", (T, None))])
    if scores.shape[1] < S:
        raise ValueError(f"scores needs at least S = {S} columns, got {scores.shape[1]}")
    _check(lib().dsa_indexer_scores(
        _dev(q, "q"), _dtype_code(q), _dev(q_scale, "q_scale", torch.float32),
        _dev(k, "k"), _dtype_code(k), _dev(k_scale, "k_scale", torch.float32),
        _dev(w, "w", torch.float32), T, S, H, D, int(q_pos0), _dev(scores, "scores", torch.float32),
        int(scores.stride(0)), _stream_ptr(stream)), "dsa_indexer_scores")
    return scores


def _host(t: Optional[torch.Tensor], name: str, dtype=None):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def dsa_indexer_dense_host_workspace_size(T: int, S: int, H: int, D: int, q_dtype: int, k_out: int,
                                          chunk_rows: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().dsa_indexer_dense_host_workspace_size(T, S, H, D, q_dtype, k_out, chunk_rows, ctypes.byref(n)),
           "dsa_indexer_dense_host_workspace_size")
    return int(n.value)


def dsa_indexer_dense_host(q: torch.Tensor, k: torch.Tensor, w: torch.Tensor, *, topk_limit: int,
                           q_pos0: Optional[int] = None, k_out: Optional[int] = None, order: int = DSA_ORDER_SCORE,
                           q_scale: Optional[torch.Tensor] = None, k_scale: Optional[torch.Tensor] = None,
                           chunk_rows: int = 0, topk: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Scores + top-k of one sequence from HOST tensors q [T, H, D], k [S, D], w [T, H]
    (pin them for overlapped copies) into a host int32 [T, k_out] tensor; the transfers
    are chunked and overlapped with the kernels.  `workspace`: a CUDA uint8 tensor of at
    least dsa_indexer_dense_host_workspace_size bytes (allocated when omitted).  The
    result is final once `stream` (default: torch's current stream) is synchronised."""
    T, H, D = q.shape
    S = k.shape[0]
    if q_pos0 is None:
        q_pos0 = S - T
    if k_out is None:
        k_out = topk_limit
    if topk is None:
        topk = torch.empty((T, k_out), dtype=torch.int32, pin_memory=torch.cuda.is_available())
    _expect([(k, "k", (S, D)), (w, "w", (T, H)), (q_scale, "q_scale", (T, H)), (k_scale, "k_scale", (S,)),
             (topk, "topk", (T, k_out))])
    need = dsa_indexer_dense_host_workspace_size(T, S, H, D, _dtype_code(q), k_out, chunk_rows)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    if not workspace.is_cuda or workspace.dtype != torch.uint8:
        raise TypeError("workspace must be a CUDA uint8 tensor")
    _check(lib().dsa_indexer_dense_host(
        _host(q, "q"), _dtype_code(q), _host(q_scale, "q_scale", torch.float32),
        _host(k, "k"), _dtype_code(k), _host(k_scale, "k_scale", torch.float32),
        _host(w, "w", torch.float32), T, S, H, D, int(q_pos0), int(topk_limit), int(k_out), int(order),
        int(chunk_rows), _host(topk, "topk", torch.int32), workspace.data_ptr(), workspace.numel(),
        _stream_ptr(stream)), "dsa_indexer_dense_host")
    return topk


def dsa_indexer_topk(scores: torch.Tensor, *, T: int, S: int, q_pos0: int, topk_limit: int,
                     k_out: Optional[int] = None, order: int = DSA_ORDER_SCORE,
                     topk: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Per-row top-k [T, k_out] int32 of dense scores (row t sees min(q_pos0 + t + 1, S) keys)."""
    if k_out is None:
        k_out = topk_limit
    if topk is None:
        topk = torch.empty((T, k_out), dtype=torch.int32, device=scores.device)
    _expect([(scores, "scores", (None, None)), (topk, "topk", (T, k_out))])
    if scores.shape[0] < T or scores.shape[1] < S:
        raise ValueError(f"scores must hold at least [{T}, {S}], got {tuple(scores.shape)}")
    _check(lib().dsa_indexer_topk(_dev(scores, "scores", torch.float32), int(scores.stride(0)), T, S,
                                  int(q_pos0), int(topk_limit), int(k_out), int(order),
                                  _dev(topk, "topk", torch.int32), _stream_ptr(stream)), "dsa_indexer_topk")
    return topk


def make_indexer_args(q, w, k_cache, cu_q_lens, seq_lens, block_tables, *, max_seq_len: int, topk_limit: int,
                      k_out: Optional[int] = None, q_scale=None, k_scale_cache=None, topk=None,
                      workspace=None, order: int = DSA_ORDER_SCORE, total_q: Optional[int] = None,
                      k_new=None, slot_mapping=None):
    """Fill a dsa_indexer_args from tensors (allocating topk / workspace with torch if absent).

    Returns (args, keepalive) -- keep the second value alive while the call runs."""
    if q.dim() != 3 or k_cache.dim() != 3 or seq_lens.dim() != 1 or block_tables.dim() != 2:
        raise ValueError("q [total_q, H, D], k_cache [num_pages, page_size, D], seq_lens [B] and "
                         "block_tables [B, max_pages] expected")
    total_q = q.shape[0] if total_q is None else total_q
    H, D = q.shape[1], q.shape[2]
    B = seq_lens.shape[0]
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    if k_out is None:
        k_out = topk_limit
    if topk is None:
        topk = torch.empty((total_q, k_out), dtype=torch.int32, device=q.device)
    # the C ABI sees only pointers and sizes: every tensor's shape is checked here
    want = {"w": (w, (q.shape[0], H)), "q_scale": (q_scale, (q.shape[0], H)),
            "k_scale_cache": (k_scale_cache, (num_pages, page_size)), "cu_q_lens": (cu_q_lens, (B + 1,)),
            "block_tables": (block_tables, (B, block_tables.shape[1])), "topk": (topk, (total_q, k_out)),
            "k_new": (k_new, (total_q, D)), "slot_mapping": (slot_mapping, (total_q,))}
    for name, (t, shape) in want.items():
        if t is not None and tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
    if k_cache.shape[2] != D or q.shape[0] < total_q:
        raise ValueError(f"k_cache rows must have D = {D} values and q at least {total_q} rows")
    a = dsa_indexer_args()
    a.q_dtype, a.k_dtype = _dtype_code(q), _dtype_code(k_cache)
    a.B, a.total_q, a.H, a.D = B, total_q, H, D
    a.page_size, a.num_pages = page_size, num_pages
    a.max_pages_per_seq, a.max_seq_len = block_tables.shape[1], int(max_seq_len)
    a.q = _dev(q, "q")
    a.q_scale = _dev(q_scale, "q_scale", torch.float32)
    a.w = _dev(w, "w", torch.float32)
    a.cu_q_lens = _dev(cu_q_lens, "cu_q_lens", torch.int32)
    a.seq_lens = _dev(seq_lens, "seq_lens", torch.int32)
    a.block_tables = _dev(block_tables, "block_tables", torch.int32)
    a.k_cache = _dev(k_cache, "k_cache")
    a.k_scale_cache = _dev(k_scale_cache, "k_scale_cache", torch.float32)
    a.topk_limit, a.k_out, a.order = int(topk_limit), int(k_out), int(order)
    a.topk = _dev(topk, "topk", torch.int32)
    if workspace is None:
        nbytes = dsa_indexer_workspace_size(a)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    a.workspace = _dev(workspace, "workspace", torch.uint8)
    a.workspace_bytes = workspace.numel()
    if (k_new is None) != (slot_mapping is None):
        raise ValueError("k_new and slot_mapping go together")
    a.k_new = _dev(k_new, "k_new", torch.bfloat16)
    a.slot_mapping = _dev(slot_mapping, "slot_mapping", torch.int64)
    return a, (q, w, k_cache, cu_q_lens, seq_lens, block_tables, q_scale, k_scale_cache, topk, workspace, k_new,
               slot_mapping)


def dsa_indexer_workspace_size(args: dsa_indexer_args) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().dsa_indexer_workspace_size(ctypes.byref(args), ctypes.byref(n)), "dsa_indexer_workspace_size")
    return int(n.value)


def dsa_indexer(q, w, k_cache, cu_q_lens, seq_lens, block_tables, *, max_seq_len: int, topk_limit: int,
                k_out: Optional[int] = None, q_scale=None, k_scale_cache=None, topk=None, workspace=None,
                order: int = DSA_ORDER_SCORE, k_new=None, slot_mapping=None, stream=None) -> torch.Tensor:
    """Fused paged indexer for a varlen batch; returns topk [total_q, k_out] int32.
    With k_new [total_q, D] bf16 and slot_mapping [total_q] int64 the step's keys are
    first written into k_cache (and k_scale_cache), in place."""
    a, keep = make_indexer_args(q, w, k_cache, cu_q_lens, seq_lens, block_tables, max_seq_len=max_seq_len,
                                topk_limit=topk_limit, k_out=k_out, q_scale=q_scale,
                                k_scale_cache=k_scale_cache, topk=topk, workspace=workspace, order=order,
                                k_new=k_new, slot_mapping=slot_mapping)
    _check(lib().dsa_indexer(ctypes.byref(a), _stream_ptr(stream)), "dsa_indexer")
    return keep[8]


def dsa_indexer_cache_append(k_new: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                             k_scale_cache: Optional[torch.Tensor] = None, stream=None) -> None:
    """Write new bf16 key rows k_new [n, D] into k_cache [num_pages, page_size, D] at the
    slots slot_mapping [n] (int64, page * page_size + row; negative = skip), in place;
    an e4m3 cache takes them quantised with one scale amax/448 per token into
    k_scale_cache [num_pages, page_size]."""
    n, D = k_new.shape
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    _expect([(slot_mapping, "slot_mapping", (n,)), (k_cache, "k_cache", (None, None, D)),
             (k_scale_cache, "k_scale_cache", (num_pages, page_size))])
    _check(lib().dsa_indexer_cache_append(
        _dev(k_new, "k_new", torch.bfloat16), n, D, _dev(slot_mapping, "slot_mapping", torch.int64),
        _dev(k_cache, "k_cache"), _dtype_code(k_cache), _dev(k_scale_cache, "k_scale_cache", torch.float32),
        page_size, num_pages, _stream_ptr(stream)), "dsa_indexer_cache_append")


def make_prepare_args(hidden: torch.Tensor, qa_normed: torch.Tensor, rope_cos: Optional[torch.Tensor],
                      rope_sin: Optional[torch.Tensor], wq_b: torch.Tensor, wk: torch.Tensor,
                      weights_proj: torch.Tensor, k_norm_weight: torch.Tensor, k_cache: torch.Tensor,
                      slot_mapping: torch.Tensor, *, H: int, rope_dim: int, rope_interleaved: bool = False,
                      k_norm_bias: Optional[torch.Tensor] = None, k_norm_eps: float = 1e-6,
                      k_scale_cache: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """(args, keepalive, (q, q_scale, w)) for dsa_indexer_prepare: allocates the outputs
    (q [T, H, D] in the cache's element type, q_scale [T, H] for an e4m3 cache, w [T, H])
    and, unless given, the workspace."""
    T, hidden_dim = hidden.shape
    q_rank = qa_normed.shape[1]
    D = wk.shape[0]
    fp8 = k_cache.dtype == torch.float8_e4m3fn
    # the C ABI sees only pointers and sizes: every tensor's shape is checked here
    want = {"qa_normed": (qa_normed, (T, q_rank)), "wq_b": (wq_b, (H * D, q_rank)), "wk": (wk, (D, hidden_dim)),
            "weights_proj": (weights_proj, (H, hidden_dim)), "k_norm_weight": (k_norm_weight, (D,)),
            "slot_mapping": (slot_mapping, (T,))}
    if k_norm_bias is not None:
        want["k_norm_bias"] = (k_norm_bias, (D,))
    if rope_dim > 0:
        want["rope_cos"] = (rope_cos, (T, rope_dim // 2))
        want["rope_sin"] = (rope_sin, (T, rope_dim // 2))
    if k_cache.dim() != 3 or k_cache.shape[2] != D:
        raise ValueError(f"k_cache must be [num_pages, page_size, {D}], got {tuple(k_cache.shape)}")
    if fp8:
        want["k_scale_cache"] = (k_scale_cache, tuple(k_cache.shape[:2]))
    for name, (t, shape) in want.items():
        if t is None or tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {None if t is None else tuple(t.shape)}")
    dev = hidden.device
    q = torch.empty((T, H, D), dtype=k_cache.dtype, device=dev)
    q_scale = torch.empty((T, H), dtype=torch.float32, device=dev) if fp8 else None
    w = torch.empty((T, H), dtype=torch.float32, device=dev)
    a = dsa_indexer_prepare_args()
    a.T, a.hidden_dim, a.q_rank, a.H, a.D = T, hidden_dim, q_rank, H, D
    a.rope_dim, a.rope_interleaved = rope_dim, 1 if rope_interleaved else 0
    a.hidden = _dev(hidden, "hidden", torch.bfloat16)
    a.qa_normed = _dev(qa_normed, "qa_normed", torch.bfloat16)
    a.rope_cos = _dev(rope_cos, "rope_cos", torch.float32)
    a.rope_sin = _dev(rope_sin, "rope_sin", torch.float32)
    a.wq_b = _dev(wq_b, "wq_b", torch.bfloat16)
    a.wk = _dev(wk, "wk", torch.bfloat16)
    a.weights_proj = _dev(weights_proj, "weights_proj", torch.bfloat16)
    a.k_norm_weight = _dev(k_norm_weight, "k_norm_weight", torch.float32)
    a.k_norm_bias = _dev(k_norm_bias, "k_norm_bias", torch.float32)
    a.k_norm_eps = float(k_norm_eps)
    a.cache_dtype = _dtype_code(k_cache)
    a.slot_mapping = _dev(slot_mapping, "slot_mapping", torch.int64)
    a.k_cache = _dev(k_cache, "k_cache")
    a.k_scale_cache = _dev(k_scale_cache, "k_scale_cache", torch.float32)
    a.page_size, a.num_pages = k_cache.shape[1], k_cache.shape[0]
    a.q_out, a.q_scale_out, a.w_out = q.data_ptr(), _dev(q_scale, "q_scale"), w.data_ptr()
    if workspace is None:
        n = ctypes.c_size_t(0)
        _check(lib().dsa_indexer_prepare_workspace_size(ctypes.byref(a), ctypes.byref(n)),
               "dsa_indexer_prepare_workspace_size")
        workspace = torch.empty(max(int(n.value), 1), dtype=torch.uint8, device=dev)
    a.workspace, a.workspace_bytes = workspace.data_ptr(), workspace.numel()
    keep = [hidden, qa_normed, rope_cos, rope_sin, wq_b, wk, weights_proj, k_norm_weight, k_norm_bias, k_cache,
            slot_mapping, k_scale_cache, q, q_scale, w, workspace]
    return a, keep, (q, q_scale, w)


def dsa_indexer_prepare(hidden: torch.Tensor, qa_normed: torch.Tensor, rope_cos: Optional[torch.Tensor],
                        rope_sin: Optional[torch.Tensor], wq_b: torch.Tensor, wk: torch.Tensor,
                        weights_proj: torch.Tensor, k_norm_weight: torch.Tensor, k_cache: torch.Tensor,
                        slot_mapping: torch.Tensor, *, H: int, rope_dim: int, rope_interleaved: bool = False,
                        k_norm_bias: Optional[torch.Tensor] = None, k_norm_eps: float = 1e-6,
                        k_scale_cache: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None):
    """The indexer front-end through the C ABI: returns (q, q_scale, w) for dsa_indexer
    and writes this step's keys (and on an e4m3 cache their scales) through slot_mapping."""
    a, keep, out = make_prepare_args(hidden, qa_normed, rope_cos, rope_sin, wq_b, wk, weights_proj, k_norm_weight,
                                     k_cache, slot_mapping, H=H, rope_dim=rope_dim, rope_interleaved=rope_interleaved,
                                     k_norm_bias=k_norm_bias, k_norm_eps=k_norm_eps, k_scale_cache=k_scale_cache,
                                     workspace=workspace)
    _check(lib().dsa_indexer_prepare(ctypes.byref(a), _stream_ptr(stream)), "dsa_indexer_prepare")
    if stream is not None:  # memory freed here must not be reused ahead of that stream's kernels
        for t in keep:
            if isinstance(t, torch.Tensor):
                t.record_stream(stream)
    del keep
    return out


def indexer_types_to_codes(indexer_types: Sequence) -> list:
    """'full' / 'shared' (or the integer codes) -> dsa_layer_type codes; others -> -1."""
    out = []
    for t in indexer_types:
        if t in ("full", DSA_LAYER_FULL):
            out.append(DSA_LAYER_FULL)
        elif t in ("shared", DSA_LAYER_SHARED):
            out.append(DSA_LAYER_SHARED)
        else:
            out.append(-1)
    return out


def dsa_resolve_indexer_sources(indexer_types: Sequence, num_layers: Optional[int] = None) -> list:
    """Source layer of every layer through the C ABI; ValueError like the reference flow
    for a short list, an unknown type or a shared layer with no earlier full layer."""
    codes = indexer_types_to_codes(indexer_types)
    if num_layers is not None and len(codes) < num_layers:
        raise ValueError("indexer_types shorter than the number of layers")
    L = len(codes)
    types = (ctypes.c_int32 * max(L, 1))(*codes)
    src = (ctypes.c_int32 * max(L, 1))()
    st = lib().dsa_resolve_indexer_sources(L, ctypes.cast(types, ctypes.c_void_p), ctypes.cast(src, ctypes.c_void_p))
    if st == DSA_ERR_INVALID_ARGUMENT:
        raise ValueError("invalid indexer_types: unknown type or shared layer without an earlier full layer")
    _check(st, "dsa_resolve_indexer_sources")
    return list(src[:L])


def dsa_indexer_stack(indexer_types: Sequence, full_layer_args: Sequence, stream=None):
    """Run an IndexShare stack.  full_layer_args[l] is a dsa_indexer_args (full layers)
    or None (shared layers).  Returns (topk device pointers per layer, source layers)."""
    codes = indexer_types_to_codes(indexer_types)
    L = len(codes)
    types = (ctypes.c_int32 * max(L, 1))(*codes)
    arr = (ctypes.POINTER(dsa_indexer_args) * max(L, 1))()
    for i, a in enumerate(full_layer_args):
        arr[i] = ctypes.pointer(a) if a is not None else ctypes.POINTER(dsa_indexer_args)()
    outs = (ctypes.c_void_p * max(L, 1))()
    src = (ctypes.c_int32 * max(L, 1))()
    st = lib().dsa_indexer_stack(L, ctypes.cast(types, ctypes.c_void_p), ctypes.cast(arr, ctypes.c_void_p),
                                 ctypes.cast(outs, ctypes.c_void_p), ctypes.cast(src, ctypes.c_void_p),
                                 _stream_ptr(stream))
    _check(st, "dsa_indexer_stack")
    return [outs[i] for i in range(L)], list(src[:L])


# ---- key-sharded top-k (GLM5 LoRA blog, section 3.1: context parallelism) ---------------

def dsa_indexer_shard_candidates(q: torch.Tensor, k_shard: torch.Tensor, w: torch.Tensor, *, q_pos0: int,
                                 key_offset: int, k_cand: int, q_scale: Optional[torch.Tensor] = None,
                                 k_scale: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                                 stream=None):
    """One key shard's candidates: (cand_idx [T, k_cand] int32 global indices then -1,
    cand_scores [T, k_cand] fp32 then -inf) for keys key_offset .. key_offset + S - 1."""
    T, H, D = q.shape
    S = k_shard.shape[0]
    _expect([(k_shard, "k_shard", (S, D)), (w, "w", (T, H)), (q_scale, "q_scale", (T, H)),
             (k_scale, "k_scale", (S,))])
    nbytes = ctypes.c_size_t(0)
    _check(lib().dsa_indexer_shard_candidates_workspace_size(T, S, ctypes.byref(nbytes)),
           "dsa_indexer_shard_candidates_workspace_size")
    if workspace is None:
        workspace = torch.empty(max(nbytes.value, 16), dtype=torch.uint8, device=q.device)
    cand_idx = torch.empty((T, k_cand), dtype=torch.int32, device=q.device)
    cand_scores = torch.empty((T, k_cand), dtype=torch.float32, device=q.device)
    _check(lib().dsa_indexer_shard_candidates(
        _dev(q, "q"), _dtype_code(q), _dev(q_scale, "q_scale", torch.float32), _dev(k_shard, "k_shard"),
        _dtype_code(k_shard), _dev(k_scale, "k_scale", torch.float32), _dev(w, "w", torch.float32), T, S, H, D,
        int(q_pos0), int(key_offset), int(k_cand), cand_idx.data_ptr(), cand_scores.data_ptr(),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
        "dsa_indexer_shard_candidates")
    return cand_idx, cand_scores


def dsa_indexer_merge_candidates(cand_scores: torch.Tensor, cand_idx: torch.Tensor, *, topk_limit: int,
                                 k_out: Optional[int] = None, order: int = DSA_ORDER_SCORE,
                                 topk: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Top-k [T, k_out] of the union of the shards' candidates [n_shards, T, k_cand]."""
    n_shards, T, k_cand = cand_idx.shape
    k_out = topk_limit if k_out is None else k_out
    _expect([(cand_scores, "cand_scores", (n_shards, T, k_cand))])
    if topk is None:
        topk = torch.empty((T, k_out), dtype=torch.int32, device=cand_idx.device)
    _expect([(topk, "topk", (T, k_out))])
    _check(lib().dsa_indexer_merge_candidates(
        _dev(cand_scores, "cand_scores", torch.float32), _dev(cand_idx, "cand_idx", torch.int32), n_shards, T,
        k_cand, int(topk_limit), int(k_out), int(order), _dev(topk, "topk", torch.int32), _stream_ptr(stream)),
        "dsa_indexer_merge_candidates")
    return topk


def gather_shard_candidates(cand_idx: torch.Tensor, cand_scores: torch.Tensor, group=None):
    """The candidates of every rank of `group`, stacked in rank order: ([world, T, k] int32,
    [world, T, k] fp32).  One all-gather of indices and one of scores (torch.distributed;
    NCCL for device tensors, gloo for host tensors)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    idx = [torch.empty_like(cand_idx) for _ in range(world)]
    sc = [torch.empty_like(cand_scores) for _ in range(world)]
    dist.all_gather(idx, cand_idx.contiguous(), group=group)
    dist.all_gather(sc, cand_scores.contiguous(), group=group)
    return torch.stack(idx), torch.stack(sc)


def dsa_indexer_key_sharded(q: torch.Tensor, k_shard: torch.Tensor, w: torch.Tensor, *, q_pos0: int,
                            key_offset: int, topk_limit: int, k_out: Optional[int] = None,
                            order: int = DSA_ORDER_SCORE, q_scale: Optional[torch.Tensor] = None,
                            k_scale: Optional[torch.Tensor] = None, group=None, stream=None) -> torch.Tensor:
    """Top-k over a sequence whose keys are split over the ranks of `group` (each rank holds
    the queries and its own contiguous key shard): local candidates, one all-gather, merge."""
    k_out = topk_limit if k_out is None else k_out
    ci, cs = dsa_indexer_shard_candidates(q, k_shard, w, q_pos0=q_pos0, key_offset=key_offset,
                                          k_cand=min(topk_limit, k_out), q_scale=q_scale, k_scale=k_scale,
                                          stream=stream)
    all_idx, all_sc = gather_shard_candidates(ci, cs, group)
    return dsa_indexer_merge_candidates(all_sc, all_idx, topk_limit=topk_limit, k_out=k_out, order=order,
                                        stream=stream)


# ---- sparse MLA over the top-k (the attention that consumes topk_indices) -----------------

def make_sparse_mla_args(q_nope, q_rope, cache_c, cache_r, block_tables, cu_q_lens, seq_lens, topk, *,
                         scale: float, out=None, workspace=None):
    """dsa_sparse_mla_args for these tensors (every shape checked); returns (args, kept tensors)."""
    total_q, H, R = q_nope.shape
    rd = q_rope.shape[2]
    num_pages, page_size = cache_c.shape[0], cache_c.shape[1]
    B = seq_lens.shape[0]
    k = topk.shape[1]
    _expect([(q_rope, "q_rope", (total_q, H, rd)), (cache_c, "cache_c", (num_pages, page_size, R)),
             (cache_r, "cache_r", (num_pages, page_size, rd)), (cu_q_lens, "cu_q_lens", (B + 1,)),
             (block_tables, "block_tables", (B, None)), (topk, "topk", (total_q, k))])
    if out is None:
        out = torch.empty((total_q, H, R), dtype=torch.float32, device=q_nope.device)
    _expect([(out, "out", (total_q, H, R))])
    a = dsa_sparse_mla_args()
    a.B, a.total_q, a.H, a.kv_rank, a.rope_dim = B, total_q, H, R, rd
    a.page_size, a.num_pages, a.max_pages_per_seq, a.topk_width = page_size, num_pages, block_tables.shape[1], k
    a.scale = float(scale)
    a.q_nope, a.q_rope = _dev(q_nope, "q_nope", torch.bfloat16), _dev(q_rope, "q_rope", torch.bfloat16)
    a.cache_c, a.cache_r = _dev(cache_c, "cache_c", torch.bfloat16), _dev(cache_r, "cache_r", torch.bfloat16)
    a.block_tables = _dev(block_tables, "block_tables", torch.int32)
    a.cu_q_lens = _dev(cu_q_lens, "cu_q_lens", torch.int32)
    a.seq_lens = _dev(seq_lens, "seq_lens", torch.int32)
    a.topk = _dev(topk, "topk", torch.int32)
    a.out = _dev(out, "out", torch.float32)
    if workspace is None:
        n = ctypes.c_size_t(0)
        _check(lib().dsa_sparse_mla_workspace_size(ctypes.byref(a), ctypes.byref(n)), "dsa_sparse_mla_workspace_size")
        workspace = torch.empty(max(n.value, 16), dtype=torch.uint8, device=q_nope.device)
    a.workspace = _dev(workspace, "workspace")
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a, (q_nope, q_rope, cache_c, cache_r, block_tables, cu_q_lens, seq_lens, topk, out, workspace)


def dsa_sparse_mla(q_nope, q_rope, cache_c, cache_r, block_tables, cu_q_lens, seq_lens, topk, *, scale: float,
                   out=None, workspace=None, stream=None) -> torch.Tensor:
    """Latent attention output [total_q, H, kv_rank] fp32 of each query over its selected keys."""
    a, keep = make_sparse_mla_args(q_nope, q_rope, cache_c, cache_r, block_tables, cu_q_lens, seq_lens, topk,
                                   scale=scale, out=out, workspace=workspace)
    _check(lib().dsa_sparse_mla(ctypes.byref(a), _stream_ptr(stream)), "dsa_sparse_mla")
    return keep[8]


def dsa_test_arm_score_timeout(limit_ns: int) -> None:
    """Failure-path test hook: the next score-kernel launch of this host thread first
    waits up to limit_ns on a barrier nothing completes, then records DSA_ERR_TIMEOUT,
    drains and returns (its outputs are unspecified).  0 disarms."""
    _check(lib().dsa_test_arm_score_timeout(int(limit_ns)), "dsa_test_arm_score_timeout")


def dsa_check_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status (DSA_OK, ...)."""
    return int(lib().dsa_check_device_status(_stream_ptr(stream)))


def dsa_clock_sample(n_ctas: int, stream=None):
    """Device tensor [n_ctas, 3] int64 of (SM id, SM cycle counter, global ns timer), one
    row per one-thread block; two samples bracket an interval (diagnostic)."""
    out = torch.empty((n_ctas, 3), dtype=torch.int64, device="cuda")
    _check(lib().dsa_clock_sample(out.data_ptr(), int(n_ctas), _stream_ptr(stream)), "dsa_clock_sample")
    return out


# ---- host helpers (GLM5 TensorCast adaptation design) -----------------------------

def resolve_topk_limit(explicit=None, indexer=None, config=None, indexer_config=None) -> int:
    """top-k width in the order of section "Sparse MLA 配置兼容": an explicit value, then
    the indexer's own topk_limit, then topk_limit on the attention / indexer config, then
    the GLM5-style index_topk; AttributeError("topk_limit") when none exists."""
    if explicit is not None:
        return int(explicit)
    if indexer is not None and getattr(indexer, "topk_limit", None) is not None:
        return int(indexer.topk_limit)
    for cfg in (config, indexer_config):
        if cfg is not None and getattr(cfg, "topk_limit", None) is not None:
            return int(cfg.topk_limit)
    for cfg in (config, indexer_config):
        if cfg is not None and getattr(cfg, "index_topk", None) is not None:
            return int(cfg.index_topk)
    raise AttributeError("topk_limit")


def extend_indexer_types_for_mtp(indexer_types: Sequence[str], num_mtp_layers: int) -> list:
    """Append one 'full' per MTP block (an MTP block cannot consume the main stack's
    top-k, section "GLM-5.2 IndexShare"); an empty list or zero MTP layers is unchanged."""
    types = list(indexer_types)
    if not types or num_mtp_layers <= 0:
        return types
    return types + ["full"] * int(num_mtp_layers)


# ---- no-allocation variant ----------------------------------------------------------

DSA_STATIC_WORKSPACE_BYTES = 24 << 20


def dsa_indexer_static(q, w, k_cache, cu_q_lens, seq_lens, block_tables, *, max_seq_len: int, topk_limit: int,
                       k_out: Optional[int] = None, q_scale=None, k_scale_cache=None, topk=None,
                       order: int = DSA_ORDER_SCORE, stream=None) -> torch.Tensor:
    """dsa_indexer without a workspace, for callers that cannot allocate device memory
    (plugin hosts that only pass tensors, serving loops that forbid allocation during a
    step).  The library keeps the scratch in a fixed device array of
    DSA_STATIC_WORKSPACE_BYTES; larger problems raise DsaError(DSA_ERR_WORKSPACE).
    Calls that overlap on the GPU share that array and must be serialised."""
    a, keep = make_indexer_args(q, w, k_cache, cu_q_lens, seq_lens, block_tables, max_seq_len=max_seq_len,
                                topk_limit=topk_limit, k_out=k_out, q_scale=q_scale,
                                k_scale_cache=k_scale_cache, topk=topk,
                                workspace=torch.empty(0, dtype=torch.uint8, device=q.device), order=order)
    a.workspace, a.workspace_bytes = None, 0
    fn = lib().dsa_indexer_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(dsa_indexer_args), ctypes.c_void_p]
    _check(fn(ctypes.byref(a), _stream_ptr(stream)), "dsa_indexer_static")
    return keep[8]
