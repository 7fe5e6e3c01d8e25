// qsplit.cuh -- one bf16 query row (D = 128) as hi + lo e4m3 rows, for one warp.
// Shared by the split kernel and the decode preparation kernel that runs it beside the
// work-list build.  The reading and its exactness bound are stated in qsplit.cu.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace dsa {

// Two fp32 values -> two e4m3 codes (lo in the low byte), round to nearest even, saturating.
__device__ __forceinline__ uint16_t split_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two e4m3 codes -> their values (exact through f16).
__device__ __forceinline__ float2 split_from_e4m3x2(uint16_t c) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16))));
}

// Row r = (t, h) of q [rows, 128] bf16 -> q8 rows t*2H + h (hi) and t*2H + H + h (lo),
// w8[r] = w[r] / s.  Called by all 32 lanes of a warp.
__device__ __forceinline__ void split_row(const uint2* __restrict__ q, const float* __restrict__ w, long long r,
                                          int H, uint32_t* __restrict__ q8, float* __restrict__ w8, int lane) {
  const int lg = 31 - __clz(H);  // H is a power of two: no 64-bit division
  const long long t = r >> lg;
  const int h = static_cast<int>(r - (t << lg));
  const uint2 raw = q[r * 32 + lane];  // elements 4 lane .. 4 lane + 3 of the row (D = 128)
  const float x0 = __uint_as_float(raw.x << 16), x1 = __uint_as_float(raw.x & 0xFFFF0000u);
  const float x2 = __uint_as_float(raw.y << 16), x3 = __uint_as_float(raw.y & 0xFFFF0000u);
  uint32_t m = max(max(__float_as_uint(fabsf(x0)), __float_as_uint(fabsf(x1))),
                   max(__float_as_uint(fabsf(x2)), __float_as_uint(fabsf(x3))));
  m = __reduce_max_sync(0xffffffffu, m);
  // s = 2^k with the largest |x| * s in [128, 256); k = 0 for an all-zero row
  const int e = static_cast<int>((m >> 23) & 0xFFu) - 127;  // exponent of the largest |x| (subnormal: -127)
  const int k = m == 0 ? 0 : min(max(7 - e, -126), 127);
  const float y0 = ldexpf(x0, k), y1 = ldexpf(x1, k), y2 = ldexpf(x2, k), y3 = ldexpf(x3, k);
  const uint16_t h01 = split_e4m3x2(y0, y1), h23 = split_e4m3x2(y2, y3);
  const float2 d01 = split_from_e4m3x2(h01), d23 = split_from_e4m3x2(h23);
  const uint16_t l01 = split_e4m3x2(y0 - d01.x, y1 - d01.y), l23 = split_e4m3x2(y2 - d23.x, y3 - d23.y);
  uint32_t* rows8 = q8 + (t * 2 * H) * 32;  // 32 words (128 B) per row
  rows8[static_cast<long long>(h) * 32 + lane] = static_cast<uint32_t>(h01) | (static_cast<uint32_t>(h23) << 16);
  rows8[static_cast<long long>(H + h) * 32 + lane] = static_cast<uint32_t>(l01) | (static_cast<uint32_t>(l23) << 16);
  if (lane == 0) w8[r] = ldexpf(w[r], -k);
}

}  // namespace dsa
