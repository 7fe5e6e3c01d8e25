"""The exact two-row e4m3 split of bf16 query rows (bf16 q against an e4m3 cache), checked
exhaustively on the CPU with torch's round-to-nearest-even float8 cast.

A query row x is scaled by a power of two s with max |s x| in [128, 256); every scaled
element y is a bf16 value with |y| < 256, written as hi = e4m3(y) and lo = e4m3(y - hi).
Claim: hi + lo == y exactly when |y| >= 2^-2 (within ~2^9 of the row's largest), and
|hi + lo - y| <= 2^-10 below that.
"""
import torch


def _split(y32: torch.Tensor):
    hi = y32.to(torch.float8_e4m3fn).to(torch.float32)
    lo = (y32 - hi).to(torch.float8_e4m3fn).to(torch.float32)   # y - hi is exact in fp32
    return hi, lo


def _bf16_values(lo_exp: int, hi_exp: int) -> torch.Tensor:
    """Every bf16 value with exponent in [lo_exp, hi_exp), both signs, as fp32."""
    bits = torch.arange(0, 1 << 15, dtype=torch.int32)
    v = bits.to(torch.int16).view(torch.bfloat16).to(torch.float32)
    v = v[torch.isfinite(v)]
    e = torch.floor(torch.log2(v.abs().clamp_min(1e-45)))
    keep = (v != 0) & (e >= lo_exp) & (e < hi_exp)
    v = v[keep]
    return torch.cat([v, -v])


def test_split_is_exact_within_nine_binades_of_the_row_max():
    y = _bf16_values(-2, 8)                    # 2^-2 <= |y| < 256
    hi, lo = _split(y)
    assert torch.equal(hi + lo, y)


def test_split_error_below_that_is_at_most_2_to_minus_10():
    y = _bf16_values(-40, -2)                  # tiny elements of a row whose max is >= 128
    hi, lo = _split(y)
    assert torch.all((hi + lo - y).abs() <= 2.0 ** -10)


def test_split_of_zero_and_of_the_row_max_range():
    hi, lo = _split(torch.tensor([0.0, -0.0, 128.0, 255.0, -201.0]))
    assert torch.equal(hi + lo, torch.tensor([0.0, 0.0, 128.0, 255.0, -201.0]))
