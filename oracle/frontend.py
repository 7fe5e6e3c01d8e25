"""CPU oracle for the DSA indexer front-end -- TEST INFRASTRUCTURE ONLY (numpy, fp64).

The GLM5 TensorCast adaptation design ("DSA Indexer 融合语义算子" and its performance
model buckets 1-5, 9 and 10) lists what the fused indexer op does before scoring:
the q projection ``qa_normed @ wq_b``, the k projection ``hidden_states @ wk`` with
``k_norm``, the head-routing projection ``hidden_states @ weights_proj``, RoPE from the
given cos / sin, and on the FP8 path ``rotate_activation`` plus activation
quantisation, with the key (and on FP8 its scale) written into the indexer cache
through ``slot_mapping``.  The page prints no formulas; the readings taken here are:

  * projections are ``x @ W^T`` with ``W`` stored ``[out_features, in_features]``
    (the usual linear-layer layout), computed here in fp64 from the bf16 inputs;
  * ``k_norm`` is a layer norm over the head dimension: (x - mean) / sqrt(var + eps)
    with the biased variance, times ``k_norm_weight``, plus an optional bias (the page
    names only the weight);
  * RoPE rotates the first ``rope_dim`` values of every q head and of k; value pair i
    (pairs ``(i, i + rope_dim/2)``, or ``(2i, 2i+1)`` when interleaved) turns by the
    angle whose cosine and sine are ``cos[t, i]`` and ``sin[t, i]``:
    ``(a, b) -> (a cos - b sin, a sin + b cos)``;
  * ``rotate_activation`` is the Walsh-Hadamard transform in Sylvester (natural)
    order scaled by ``D^-1/2`` (an orthogonal rotation), on q and k after RoPE;
  * activation quantisation is the same per-row reading as the cache write: one fp32
    scale ``amax / 448`` per (token, head) row of q and per token of k (1 for an
    all-zero row), codes the e4m3 value nearest to ``x / scale`` (fp32 division),
    ties to even, saturating;
  * ``weights_proj`` gives the head weights ``w [T, H]`` directly (no extra constant:
    any softmax or head-count scale is folded into the weight by the caller).

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed forms
(Hadamard orthogonality and its entries, rotations by 0 and 90 degrees, a hand-worked
layer norm, a brute-force matrix product, norm preservation).
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import scipy.linalg
import torch

from . import e4m3_encode, decode_e4m3


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact fp64 values of a bf16 / fp32 tensor."""
    return t.detach().to(torch.float64).cpu().numpy()


def linear(x: np.ndarray, weight: np.ndarray) -> np.ndarray:
    """x [T, K] @ weight[N, K]^T in fp64 (the projection buckets 1-3)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(weight, dtype=np.float64).T


def layer_norm(x: np.ndarray, weight: np.ndarray, bias: Optional[np.ndarray], eps: float) -> np.ndarray:
    """Layer norm over the last axis with the biased variance, then weight (and bias)."""
    x = np.asarray(x, dtype=np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    y = (x - mean) / np.sqrt(var + eps) * np.asarray(weight, dtype=np.float64)
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)
    return y


def rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray, rope_dim: int, interleaved: bool) -> np.ndarray:
    """RoPE on the first rope_dim values of the last axis.  x [T, ..., D]; cos / sin
    [T, rope_dim / 2] broadcast over the middle axes."""
    x = np.array(x, dtype=np.float64, copy=True)
    half = rope_dim // 2
    c = np.asarray(cos, dtype=np.float64).reshape((x.shape[0],) + (1,) * (x.ndim - 2) + (half,))
    s = np.asarray(sin, dtype=np.float64).reshape((x.shape[0],) + (1,) * (x.ndim - 2) + (half,))
    if interleaved:
        a, b = x[..., 0:rope_dim:2].copy(), x[..., 1:rope_dim:2].copy()
        x[..., 0:rope_dim:2] = a * c - b * s
        x[..., 1:rope_dim:2] = a * s + b * c
    else:
        a, b = x[..., :half].copy(), x[..., half:rope_dim].copy()
        x[..., :half] = a * c - b * s
        x[..., half:rope_dim] = a * s + b * c
    return x


def hadamard(D: int) -> np.ndarray:
    """Walsh-Hadamard matrix of order D (a power of two), Sylvester order, times D^-1/2."""
    return scipy.linalg.hadamard(D).astype(np.float64) / np.sqrt(D)


def rotate_activation(x: np.ndarray) -> np.ndarray:
    """The normalised Hadamard rotation applied to the last axis (H is symmetric)."""
    D = x.shape[-1]
    return np.asarray(x, dtype=np.float64) @ hadamard(D)


def quantize_rows(x: np.ndarray):
    """Per-row e4m3 quantisation of fp64 values taken to fp32 first: returns
    (codes uint8 [..., D], scales fp32 [...]) with scale = amax / 448 (1 for an all-zero
    row) and code = e4m3(x / scale) in fp32."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.abs(x32).max(axis=-1)
    scale = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0)).astype(np.float32)
    y = (x32 / scale[..., None]).astype(np.float32)
    codes = e4m3_encode(y.ravel()).reshape(x32.shape)
    return codes, scale


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """fp64 values of e4m3 codes times their row scales."""
    table = np.array([decode_e4m3(c) if c not in (0x7F, 0xFF) else np.nan for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.int64)] * np.asarray(scales, dtype=np.float64)[..., None]


def prepare(hidden: torch.Tensor, qa_normed: torch.Tensor, rope_cos: torch.Tensor, rope_sin: torch.Tensor,
            wq_b: torch.Tensor, wk: torch.Tensor, weights_proj: torch.Tensor, k_norm_weight: torch.Tensor,
            k_norm_bias: Optional[torch.Tensor], *, H: int, D: int, rope_dim: int, interleaved: bool,
            eps: float, fp8: bool):
    """The front-end in the page's bucket order.  Returns a dict with the fp64 values
    before any rounding (``q`` [T, H, D], ``k`` [T, D], ``w`` [T, H]) and, when fp8,
    the quantised rows (``q_codes``, ``q_scale``, ``k_codes``, ``k_scale``)."""
    T = hidden.shape[0]
    q = linear(to_f64(qa_normed), to_f64(wq_b)).reshape(T, H, D)          # bucket 1
    k = linear(to_f64(hidden), to_f64(wk))                                  # bucket 2
    k = layer_norm(k, to_f64(k_norm_weight), None if k_norm_bias is None else to_f64(k_norm_bias), eps)
    w = linear(to_f64(hidden), to_f64(weights_proj))                        # bucket 3
    cos, sin = to_f64(rope_cos), to_f64(rope_sin)
    q = rope(q, cos, sin, rope_dim, interleaved)                            # bucket 4
    k = rope(k, cos, sin, rope_dim, interleaved)
    out = {"w": w}
    if fp8:                                                                 # bucket 5
        q = rotate_activation(q)
        k = rotate_activation(k)
        out["q_codes"], out["q_scale"] = quantize_rows(q)
        out["k_codes"], out["k_scale"] = quantize_rows(k)
    out["q"], out["k"] = q, k
    return out
