"""Exact brute force for tiny indexer inputs -- TEST INFRASTRUCTURE ONLY.

Pins the C oracle.  Every value is a ``fractions.Fraction`` (bf16, e4m3 and
fp32 values are dyadic rationals, so nothing rounds), scores follow the
definition term by term, and the top-k is chosen by counting, for every key,
how many visible keys beat it -- a different algorithm from the oracle's sort:

  rank(s) = #{s' visible : score[s'] > score[s]  or  (score[s'] == score[s] and s' < s)}

key s is kept iff rank(s) < min(topk_limit, n_visible), and sits at output
slot rank(s) (GLM5 TensorCast adaptation design, "DSA Indexer 融合语义算子";
ties to the lower key index).
"""
from __future__ import annotations

from fractions import Fraction
from typing import List, Optional, Sequence

import struct


def bf16_value(bits: int) -> Fraction:
    """bf16 bits -> exact value (1 sign, 8 exponent bits with bias 127, 7 mantissa bits)."""
    bits &= 0xFFFF
    sign = -1 if bits >> 15 else 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    if e == 0xFF:
        raise ValueError("inf/nan")
    if e == 0:
        return sign * Fraction(m, 128) * Fraction(2) ** (-126)
    return sign * (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)


def e4m3_value(code: int) -> Fraction:
    """OCP e4m3 code -> exact value (bias 7, subnormal at exponent 0, S.1111.111 = NaN)."""
    code &= 0xFF
    sign = -1 if code >> 7 else 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        raise ValueError("nan")
    if e == 0:
        return sign * Fraction(m, 8) * Fraction(2) ** (-6)
    return sign * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def f32_value(x: float) -> Fraction:
    (u,) = struct.unpack("<I", struct.pack("<f", x))
    sign = -1 if u >> 31 else 1
    e = (u >> 23) & 0xFF
    m = u & 0x7FFFFF
    if e == 0xFF:
        raise ValueError("inf/nan")
    if e == 0:
        return sign * Fraction(m, 1 << 23) * Fraction(2) ** (-126)
    return sign * (1 + Fraction(m, 1 << 23)) * Fraction(2) ** (e - 127)


def scores_row(qv, kv, wv, H: int, D: int, n_visible: int, sq=None, sk=None) -> List[Fraction]:
    """qv[h][d], kv[s][d], wv[h] exact values; sq[h], sk[s] scales or None."""
    out = []
    for s in range(n_visible):
        total = Fraction(0)
        for h in range(H):
            x = Fraction(0)
            for d in range(D):
                x += qv[h][d] * kv[s][d]
            if sq is not None:
                x *= sq[h]
            if sk is not None:
                x *= sk[s]
            total += wv[h] * (x if x > 0 else Fraction(0))
        out.append(total)
    return out


def topk_by_rank(scores: Sequence[Fraction], topk_limit: int, k_out: int) -> List[int]:
    n = len(scores)
    keep = min(topk_limit, n, k_out)
    out = [-1] * k_out
    for s in range(n):
        rank = 0
        for s2 in range(n):
            if scores[s2] > scores[s] or (scores[s2] == scores[s] and s2 < s):
                rank += 1
        if rank < keep:
            out[rank] = s
    return out


def dense(q_bits, k_bits, w, *, dtype: str, T: int, S: int, H: int, D: int, q_pos0: int,
          topk_limit: int, k_out: int, q_scale=None, k_scale=None):
    """q_bits[T][H][D], k_bits[S][D] raw codes (bf16 uint16 or e4m3 uint8); w[T][H] floats."""
    dec = bf16_value if dtype == "bf16" else e4m3_value
    kv = [[dec(k_bits[s][d]) for d in range(D)] for s in range(S)]
    sk = None if k_scale is None else [f32_value(x) for x in k_scale]
    all_scores, all_topk = [], []
    for t in range(T):
        qv = [[dec(q_bits[t][h][d]) for d in range(D)] for h in range(H)]
        wv = [f32_value(x) for x in w[t]]
        sq = None if q_scale is None else [f32_value(x) for x in q_scale[t]]
        n_vis = max(0, min(q_pos0 + t + 1, S))
        sc = scores_row(qv, kv, wv, H, D, n_vis, sq, sk)
        all_scores.append(sc)
        all_topk.append(topk_by_rank(sc, topk_limit, k_out))
    return all_topk, all_scores
