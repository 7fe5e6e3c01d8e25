// qsplit.cu -- bf16 query rows as a sum of two e4m3 rows, for decode against an e4m3 cache.
//
// The tensor core takes both operands of one FP8 MMA in FP8 formats and no FP8 kind takes
// a bf16 operand, so bf16 queries against an e4m3 key cache are rewritten once per call:
// every (query, head) row x of D = 128 values gets a power-of-two scale s that puts its
// largest |x| in [128, 256), then hi = e4m3(s x) and lo = e4m3(s x - hi), both rounded to
// nearest.  A bf16 element has 8 significant bits and hi keeps the top 4 (rounded), so the
// residual s x - hi is an integer in [-8, 8] times the element's last-bit weight: lo holds
// it exactly while that weight is at least the smallest e4m3 subnormal 2^-9, i.e. for every
// element no more than ~2^9 below the row's largest.  Smaller elements lose at most 2^-10
// (half that subnormal) after scaling, 2^-17 of the row's largest |s x| >= 128.  The score
// kernel multiplies keys by both rows in one MMA (N = 2H) and
// adds the two halves before the ReLU; w is divided by s here (exact: a power of two), so
//   w/s * relu(k . (hi + lo)) = w * relu(k . x).
// Output: q8 [total_q, 2H, D] (heads 0..H-1 the hi rows, H..2H-1 the lo rows) and
// w8 [total_q, H] = w / s.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kSplitWarps = 8;

// Two fp32 values -> two e4m3 codes (lo in the low byte), round to nearest even, saturating.
__device__ __forceinline__ uint16_t to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two e4m3 codes -> their values (exact through f16).
__device__ __forceinline__ float2 from_e4m3x2(uint16_t c) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16))));
}

__global__ void __launch_bounds__(kSplitWarps * 32) qsplit_kernel(const uint2* __restrict__ q, const float* __restrict__ w,
                                                                  long long rows, int H, uint32_t* __restrict__ q8,
                                                                  float* __restrict__ w8) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * kSplitWarps + (threadIdx.x >> 5);  // (t, h) row
  if (r >= rows) return;
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
  const uint16_t h01 = to_e4m3x2(y0, y1), h23 = to_e4m3x2(y2, y3);
  const float2 d01 = from_e4m3x2(h01), d23 = from_e4m3x2(h23);
  const uint16_t l01 = to_e4m3x2(y0 - d01.x, y1 - d01.y), l23 = to_e4m3x2(y2 - d23.x, y3 - d23.y);
  uint32_t* rows8 = q8 + (t * 2 * H) * 32;  // 32 words (128 B) per row
  rows8[static_cast<long long>(h) * 32 + lane] = static_cast<uint32_t>(h01) | (static_cast<uint32_t>(h23) << 16);
  rows8[static_cast<long long>(H + h) * 32 + lane] = static_cast<uint32_t>(l01) | (static_cast<uint32_t>(l23) << 16);
  if (lane == 0) w8[r] = ldexpf(w[r], -k);
}

}  // namespace

cudaError_t launch_qsplit(const void* q, const float* w, long long rows, int H, void* q8, float* w8,
                          cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + kSplitWarps - 1) / kSplitWarps;
  const cudaError_t e = launch_pdl(qsplit_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kSplitWarps * 32), 0, st,
                                   static_cast<const uint2*>(q), w, rows, H, static_cast<uint32_t*>(q8), w8);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dsa
