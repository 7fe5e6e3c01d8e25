"""Seeded synthetic inputs for the DSA indexer workloads.

This module only draws random numbers and lays them out; it holds none of the
indexer's arithmetic (no dot products, no ReLU, no head reduction, no top-k).
Both the CPU oracle (``oracle/``) and the CUDA path consume the exact bytes
produced here, so input quantisation is outside every comparison.

Every generator uses a CPU ``torch.Generator`` seeded explicitly, so the same
seed gives the same bytes on any machine.

Shapes and value distributions follow the indexer workloads of the GLM5
``glm_moe_dsa`` DSA indexer (GLM5 TensorCast adaptation design, section
"DSA Indexer 融合语义算子"): query-major ``q[total_q, H, D]``, per-head weights
``w[total_q, H]``, a paged key cache ``k_cache[num_pages, page_size, D]``
addressed through ``block_tables`` and ``seq_lens``, and for the FP8 path a
separate per-token fp32 scale cache.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

E4M3_MAX = 448.0
BF16 = "bf16"
FP8 = "fp8_e4m3"


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def randint_values(shape, lo: int, hi: int, g: torch.Generator) -> torch.Tensor:
    """Integers uniform in [lo, hi] (inclusive), as float32."""
    return torch.randint(lo, hi + 1, tuple(shape), generator=g, dtype=torch.int64).to(torch.float32)


def gaussian(shape, g: torch.Generator, std: float = 1.0) -> torch.Tensor:
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32) * std


def quantize_rows_e4m3(x: torch.Tensor):
    """Quantise the last dimension of ``x`` to e4m3 with one fp32 scale per row.

    scale = amax(|row|) / 448 (1.0 for an all-zero row); codes are torch's
    round-to-nearest float8_e4m3fn conversion of ``row / scale``.  This is input
    preparation only: the oracle and the CUDA path both receive the codes and
    the scales, never the unquantised values.
    """
    amax = x.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = (x / scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return codes, scale.squeeze(-1).to(torch.float32).contiguous()


@dataclass
class DenseCase:
    """One sequence, dense keys ``k[S, D]``; query t sits at position q_pos0 + t."""

    q: torch.Tensor            # [T, H, D] bf16 or float8_e4m3fn
    k: torch.Tensor            # [S, D]    bf16 or float8_e4m3fn
    w: torch.Tensor            # [T, H]    fp32
    q_scale: Optional[torch.Tensor]  # [T, H] fp32 (fp8 only)
    k_scale: Optional[torch.Tensor]  # [S]    fp32 (fp8 only)
    T: int
    S: int
    H: int
    D: int
    q_pos0: int
    topk_limit: int
    k_out: int
    dtype: str
    integer_valued: bool = False


@dataclass
class PagedCase:
    """Varlen batch over a paged key cache (prefill, chunked prefill or decode).

    Sequence b owns queries ``cu_q_lens[b]..cu_q_lens[b+1]-1``; its i-th query
    sits at position ``seq_lens[b] - q_len_b + i`` and its key at logical
    position s lives in ``k_cache[block_tables[b, s // page_size], s % page_size]``.
    """

    q: torch.Tensor              # [total_q, H, D] bf16 or float8_e4m3fn
    q_scale: Optional[torch.Tensor]  # [total_q, H] fp32 or None
    w: torch.Tensor              # [total_q, H] fp32
    k_cache: torch.Tensor        # [num_pages, page_size, D] bf16 or float8_e4m3fn
    k_scale_cache: Optional[torch.Tensor]  # [num_pages, page_size] fp32 or None
    cu_q_lens: torch.Tensor      # [B+1] int32
    seq_lens: torch.Tensor       # [B] int32
    block_tables: torch.Tensor   # [B, max_pages_per_seq] int32
    B: int
    H: int
    D: int
    page_size: int
    topk_limit: int
    k_out: int
    q_dtype: str
    k_dtype: str
    max_seq_len: int
    integer_valued: bool = False

    @property
    def total_q(self) -> int:
        return int(self.cu_q_lens[-1])

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])


def dense_case(T: int, S: int, H: int, D: int, topk_limit: int, *, q_pos0: Optional[int] = None,
               k_out: Optional[int] = None, dtype: str = BF16, integer: bool = False,
               int_range=(-4, 4), w_int_range=(-2, 2), w_std: Optional[float] = None,
               seed: int = 0) -> DenseCase:
    """Dense single-sequence inputs.

    ``integer=True`` draws q and k from the integers of ``int_range`` and w from
    ``w_int_range`` (exact in bf16/fp32); otherwise q, k ~ N(0, 1) and
    w ~ N(0, 1) * w_std (default 1/sqrt(H)).  FP8 cases quantise q per (t, h)
    row and k per token with scale amax/448, except integer FP8 cases, which
    use the integers directly with power-of-two scales so every product stays
    exact.
    """
    g = _gen(seed)
    if q_pos0 is None:
        q_pos0 = S - T
    if k_out is None:
        k_out = topk_limit
    if w_std is None:
        w_std = 1.0 / math.sqrt(H)
    if integer:
        qf = randint_values((T, H, D), int_range[0], int_range[1], g)
        kf = randint_values((S, D), int_range[0], int_range[1], g)
        w = randint_values((T, H), w_int_range[0], w_int_range[1], g)
    else:
        qf = gaussian((T, H, D), g)
        kf = gaussian((S, D), g)
        w = gaussian((T, H), g, w_std)
    q_scale = k_scale = None
    if dtype == BF16:
        q = qf.to(torch.bfloat16)
        k = kf.to(torch.bfloat16)
    elif dtype == FP8:
        if integer:
            q = qf.to(torch.float8_e4m3fn)
            k = kf.to(torch.float8_e4m3fn)
            # powers of two keep every product and sum exact in fp32
            q_scale = torch.pow(2.0, randint_values((T, H), -2, 1, g))
            k_scale = torch.pow(2.0, randint_values((S,), -2, 1, g))
        else:
            q, q_scale = quantize_rows_e4m3(qf)
            k, k_scale = quantize_rows_e4m3(kf)
    else:
        raise ValueError(dtype)
    return DenseCase(q=q.contiguous(), k=k.contiguous(), w=w.contiguous(), q_scale=q_scale,
                     k_scale=k_scale, T=T, S=S, H=H, D=D, q_pos0=q_pos0,
                     topk_limit=topk_limit, k_out=k_out, dtype=dtype, integer_valued=integer)


def paged_case(seq_lens, q_lens, H: int, D: int, topk_limit: int, *, page_size: int = 64,
               k_out: Optional[int] = None, q_dtype: str = BF16, k_dtype: str = BF16,
               integer: bool = False, w_std: Optional[float] = None, spare_pages: int = 3,
               seed: int = 0) -> PagedCase:
    """Paged varlen inputs with physical pages in a seeded random permutation."""
    g = _gen(seed)
    seq_lens = [int(x) for x in seq_lens]
    q_lens = [int(x) for x in q_lens]
    B = len(seq_lens)
    assert len(q_lens) == B and all(0 <= ql <= sl for ql, sl in zip(q_lens, seq_lens))
    if k_out is None:
        k_out = topk_limit
    if w_std is None:
        w_std = 1.0 / math.sqrt(H)
    pages_per_seq = [(sl + page_size - 1) // page_size for sl in seq_lens]
    max_pages = max(1, max(pages_per_seq))
    num_pages = sum(pages_per_seq) + spare_pages
    perm = torch.randperm(num_pages, generator=g)
    block_tables = torch.full((B, max_pages), -1, dtype=torch.int32)
    cursor = 0
    for b, npg in enumerate(pages_per_seq):
        block_tables[b, :npg] = perm[cursor:cursor + npg].to(torch.int32)
        cursor += npg
    total_q = sum(q_lens)
    cu = [0]
    for ql in q_lens:
        cu.append(cu[-1] + ql)
    if integer:
        qf = randint_values((total_q, H, D), -4, 4, g)
        kf = randint_values((num_pages, page_size, D), -4, 4, g)
        w = randint_values((total_q, H), -2, 2, g)
    else:
        qf = gaussian((total_q, H, D), g)
        kf = gaussian((num_pages, page_size, D), g)
        w = gaussian((total_q, H), g, w_std)
    q_scale = k_scale = None
    if q_dtype == BF16:
        q = qf.to(torch.bfloat16)
    elif integer:
        q = qf.to(torch.float8_e4m3fn)
        q_scale = torch.pow(2.0, randint_values((total_q, H), -2, 1, g))
    else:
        q, q_scale = quantize_rows_e4m3(qf)
    if k_dtype == BF16:
        k = kf.to(torch.bfloat16)
    elif integer:
        k = kf.to(torch.float8_e4m3fn)
        k_scale = torch.pow(2.0, randint_values((num_pages, page_size), -2, 1, g))
    else:
        k, k_scale = quantize_rows_e4m3(kf)
    return PagedCase(q=q.contiguous(), q_scale=q_scale, w=w.contiguous(), k_cache=k.contiguous(),
                     k_scale_cache=k_scale, cu_q_lens=torch.tensor(cu, dtype=torch.int32),
                     seq_lens=torch.tensor(seq_lens, dtype=torch.int32), block_tables=block_tables,
                     B=B, H=H, D=D, page_size=page_size, topk_limit=topk_limit, k_out=k_out,
                     q_dtype=q_dtype, k_dtype=k_dtype, max_seq_len=max(seq_lens) if seq_lens else 0,
                     integer_valued=integer)


# ---------------------------------------------------------------------------
# The five indexer workloads, by what they are.
# ---------------------------------------------------------------------------

def tiny_exact_prefill(seed: int = 0) -> DenseCase:
    """T=S=512 causal, H=4, D=64, index_topk=64; bf16 integers in [-4,4], w in [-2,2]."""
    return dense_case(512, 512, 4, 64, 64, integer=True, seed=seed)


def prefill_8k(seed: int = 0) -> DenseCase:
    """T=S=8192 causal, H=64, D=128, index_topk=2048; bf16 N(0,1), w ~ N(0,1)/sqrt(64)."""
    return dense_case(8192, 8192, 64, 128, 2048, seed=seed, w_std=1.0 / 8.0)


def decode_lens(B: int, lo: int, hi: int, seed: int):
    g = _gen(seed + 7919)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).tolist()


def decode_b64_fp8(seed: int = 0, B: int = 64, lo: int = 4096, hi: int = 65536) -> PagedCase:
    """Decode: B=64, one query each, contexts U[4096, 65536], paged e4m3 keys (page 64)
    with per-token fp32 scales, H=64, D=128, index_topk=2048; q bf16 N(0,1), w N(0,1)/8."""
    lens = decode_lens(B, lo, hi, seed)
    return paged_case(lens, [1] * B, 64, 128, 2048, page_size=64, q_dtype=BF16, k_dtype=FP8,
                      w_std=1.0 / 8.0, seed=seed)


def chunked_prefill_fp8(seed: int = 0, n_new: int = 8192, ctx: int = 65536) -> PagedCase:
    """8192 new queries at positions 57344..65535 against a 65536-key causal cache,
    e4m3 q (per-(token, head) scale) and k (per-token scale), H=64, D=128, index_topk=2048."""
    return paged_case([ctx], [n_new], 64, 128, 2048, page_size=64, q_dtype=FP8, k_dtype=FP8,
                      w_std=1.0 / 8.0, seed=seed)


def e4m3_code_sweep_decode(seed: int = 0, B: int = 8, H: int = 64, page_size: int = 64) -> PagedCase:
    """Decode against an e4m3 cache in which every finite e4m3 code (254 of them, both
    zeros and all subnormals included) appears once per sequence in one column d_b.
    Query b is +-1 at d_b in head 0 (other heads random integers), w is +-1 on head 0
    and 0 elsewhere, so each score is one decoded code times its power-of-two key
    scale: exact in any precision, ties only where the ReLU gives 0.  q is bf16."""
    g = _gen(seed)
    codes = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
    n = codes.numel()
    pc = paged_case([n] * B, [1] * B, H, 128, n, page_size=page_size, k_out=n + 2,
                    q_dtype=BF16, k_dtype=FP8, integer=True, seed=seed)
    raw = torch.randint(0, 254, (pc.k_cache.shape[0], page_size, 128), generator=g).to(torch.uint8)
    raw = torch.where(raw >= 0x7F, raw + 1, raw)          # skip the NaN code 0x7F (0xFF is out of range)
    cols = (torch.randperm(128, generator=g)[:B]).tolist()
    q = randint_values((B, H, 128), -4, 4, g)
    w = torch.zeros((B, H))
    for b in range(B):
        perm = codes[torch.randperm(n, generator=g)]
        for j in range(n):
            page = int(pc.block_tables[b, j // page_size])
            raw[page, j % page_size, cols[b]] = perm[j]
        sign = 1.0 if (b % 2 == 0) else -1.0
        q[b, 0, :] = 0
        q[b, 0, cols[b]] = sign
        w[b, 0] = 1.0 if torch.randint(0, 2, (1,), generator=g).item() else -1.0
    pc.k_cache = raw.view(torch.float8_e4m3fn).contiguous()
    pc.q = q.to(torch.bfloat16).contiguous()
    pc.w = w.contiguous()
    return pc


INDEXSHARE_TYPES_12 = ["full", "shared", "shared"] * 4


@dataclass
class StackCase:
    indexer_types: list
    layers: list = field(default_factory=list)   # PagedCase per full layer, None for shared


def indexshare_stack(seed: int = 0, B: int = 32, ctx: int = 32768,
                     types=None, H: int = 64, D: int = 128, topk: int = 2048) -> StackCase:
    """12 layers [full, shared, shared] x 4, decode batch 32 at 32768-token contexts,
    bf16 paged caches (one per full layer), H=64, D=128, index_topk=2048."""
    types = list(INDEXSHARE_TYPES_12 if types is None else types)
    layers = []
    for li, t in enumerate(types):
        if t == "full":
            layers.append(paged_case([ctx] * B, [1] * B, H, D, topk, page_size=64,
                                     w_std=1.0 / 8.0, seed=seed * 1000 + li))
        else:
            layers.append(None)
    return StackCase(indexer_types=types, layers=layers)


def new_token_slots(pc: PagedCase) -> torch.Tensor:
    """Cache slot (page * page_size + row) of every query token of a paged case: query i
    of sequence b is the token at position seq_len - q_len + i, the step's new key."""
    slots = []
    cu = pc.cu_q_lens.tolist()
    for b in range(pc.B):
        q_len, L = cu[b + 1] - cu[b], int(pc.seq_lens[b])
        for i in range(q_len):
            pos = L - q_len + i
            slots.append(int(pc.block_tables[b, pos // pc.page_size]) * pc.page_size + pos % pc.page_size)
    return torch.tensor(slots, dtype=torch.int64)


def new_keys(pc: PagedCase, seed: int = 0, integer: bool = False) -> torch.Tensor:
    """bf16 new key rows [total_q, D] for a paged case (N(0,1) scaled per row by a power of
    two in [2^-6, 2^5], or integers in [-4, 4])."""
    g = _gen(seed)
    total_q = int(pc.cu_q_lens[-1])
    if integer:
        return randint_values((total_q, pc.D), -4, 4, g).to(torch.bfloat16)
    x = gaussian((total_q, pc.D), g) * torch.pow(2.0, torch.randint(-6, 6, (total_q, 1), generator=g).float())
    return x.to(torch.bfloat16)



@dataclass
class FrontendCase:
    """Inputs of the indexer front-end (the fused op's hidden_states, qa_normed, RoPE
    cos / sin, wq_b, wk, weights_proj, k_norm weight, cache and slot_mapping)."""
    hidden: torch.Tensor          # [T, hidden_dim] bf16
    qa_normed: torch.Tensor       # [T, q_rank] bf16
    rope_cos: torch.Tensor        # [T, rope_dim / 2] fp32
    rope_sin: torch.Tensor
    wq_b: torch.Tensor            # [H * D, q_rank] bf16
    wk: torch.Tensor              # [D, hidden_dim] bf16
    weights_proj: torch.Tensor    # [H, hidden_dim] bf16
    k_norm_weight: torch.Tensor   # [D] fp32
    k_norm_bias: Optional[torch.Tensor]
    k_cache: torch.Tensor         # [num_pages, page_size, D] bf16 or e4m3 (zeros)
    k_scale_cache: Optional[torch.Tensor]
    slot_mapping: torch.Tensor    # [T] int64
    H: int
    D: int
    rope_dim: int


def frontend_case(T: int, hidden_dim: int, q_rank: int, H: int, D: int = 128, rope_dim: int = 64, *,
                  fp8: bool = False, bias: bool = False, page_size: int = 64, num_pages: Optional[int] = None,
                  pos0: int = 0, seed: int = 0, pad_every: int = 0) -> FrontendCase:
    """Seeded front-end inputs: activations N(0, 1) in bf16 (qa_normed is the output of a
    norm, so unit scale), projection weights N(0, 1)/sqrt(in_features) in bf16 (unit-scale
    outputs), k_norm weight 1 + N(0, 0.1), RoPE tables of positions pos0 .. pos0 + T - 1 with
    frequencies 10000^(-2i / rope_dim), slots a seeded permutation of the cache's slots
    (every pad_every-th token padded with -1 when pad_every > 0)."""
    g = _gen(seed)
    if num_pages is None:
        num_pages = (T + page_size - 1) // page_size + 2
    hidden = torch.randn((T, hidden_dim), generator=g).to(torch.bfloat16)
    qa = torch.randn((T, q_rank), generator=g).to(torch.bfloat16)
    wq_b = (torch.randn((H * D, q_rank), generator=g) / math.sqrt(q_rank)).to(torch.bfloat16)
    wk = (torch.randn((D, hidden_dim), generator=g) / math.sqrt(hidden_dim)).to(torch.bfloat16)
    wp = (torch.randn((H, hidden_dim), generator=g) / math.sqrt(hidden_dim)).to(torch.bfloat16)
    knw = (1.0 + 0.1 * torch.randn((D,), generator=g)).to(torch.float32)
    knb = (0.1 * torch.randn((D,), generator=g)).to(torch.float32) if bias else None
    half = rope_dim // 2
    pos = torch.arange(pos0, pos0 + T, dtype=torch.float64)[:, None]
    freq = 10000.0 ** (-2.0 * torch.arange(half, dtype=torch.float64) / max(rope_dim, 1))
    ang = pos * freq[None, :]
    cos, sin = torch.cos(ang).to(torch.float32).contiguous(), torch.sin(ang).to(torch.float32).contiguous()
    slots = torch.randperm(num_pages * page_size, generator=g)[:T].to(torch.int64)
    if pad_every > 0:
        slots[::pad_every] = -1
    dt = torch.float8_e4m3fn if fp8 else torch.bfloat16
    cache = torch.zeros((num_pages, page_size, D), dtype=torch.float32).to(dt)
    scales = torch.zeros((num_pages, page_size), dtype=torch.float32) if fp8 else None
    return FrontendCase(hidden, qa, cos, sin, wq_b, wk, wp, knw, knb, cache, scales, slots, H, D, rope_dim)


@dataclass
class SparseMlaCase:
    """Inputs of sparse MLA over top-k: absorbed queries, a paged latent cache and each
    query token's selected logical key positions."""
    q_nope: torch.Tensor        # [total_q, H, kv_rank] bf16
    q_rope: torch.Tensor        # [total_q, H, rope_dim] bf16
    cache_c: torch.Tensor       # [num_pages, page_size, kv_rank] bf16
    cache_r: torch.Tensor       # [num_pages, page_size, rope_dim] bf16
    block_tables: torch.Tensor  # [B, max_pages] int32
    cu_q_lens: torch.Tensor     # [B + 1] int32
    seq_lens: torch.Tensor      # [B] int32
    topk: torch.Tensor          # [total_q, k] int32, -1 = none
    page_size: int
    scale: float


def sparse_mla_case(seq_lens, q_lens, H: int, k: int, *, kv_rank: int = 512, rope_dim: int = 64,
                    page_size: int = 64, seed: int = 0) -> SparseMlaCase:
    """Seeded sparse-MLA inputs: N(0,1) bf16 queries and latent rows, pages in a seeded
    permutation, and for query i of a sequence of length L with q_len new tokens (position
    L - q_len + i) a seeded draw of min(k, position + 1) distinct visible positions in
    random order, -1 padded to k.  scale = (kv_rank + rope_dim)^-1/2."""
    g = _gen(seed)
    seq_lens = [int(x) for x in seq_lens]
    q_lens = [int(x) for x in q_lens]
    B = len(seq_lens)
    pages_per_seq = [(L + page_size - 1) // page_size for L in seq_lens]
    num_pages = sum(pages_per_seq) + 1
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    bt = torch.full((B, max(1, max(pages_per_seq))), -1, dtype=torch.int32)
    cur = 0
    for b, npg in enumerate(pages_per_seq):
        bt[b, :npg] = perm[cur:cur + npg]
        cur += npg
    total_q = sum(q_lens)
    cu = [0]
    for ql in q_lens:
        cu.append(cu[-1] + ql)
    q_nope = torch.randn((total_q, H, kv_rank), generator=g).to(torch.bfloat16)
    q_rope = torch.randn((total_q, H, rope_dim), generator=g).to(torch.bfloat16)
    cache_c = torch.randn((num_pages, page_size, kv_rank), generator=g).to(torch.bfloat16)
    cache_r = torch.randn((num_pages, page_size, rope_dim), generator=g).to(torch.bfloat16)
    topk = torch.full((total_q, k), -1, dtype=torch.int32)
    for b in range(B):
        for i in range(q_lens[b]):
            pos = seq_lens[b] - q_lens[b] + i
            n = min(k, pos + 1)
            sel = torch.randperm(pos + 1, generator=g)[:n].to(torch.int32)
            topk[cu[b] + i, :n] = sel
    return SparseMlaCase(q_nope, q_rope, cache_c, cache_r, bt, torch.tensor(cu, dtype=torch.int32),
                         torch.tensor(seq_lens, dtype=torch.int32), topk, page_size,
                         1.0 / math.sqrt(kv_rank + rope_dim))
