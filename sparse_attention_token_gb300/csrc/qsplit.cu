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
#include "qsplit.cuh"

namespace dsa {
namespace {

constexpr int kSplitWarps = 8;

__global__ void __launch_bounds__(kSplitWarps * 32) qsplit_kernel(const uint2* __restrict__ q, const float* __restrict__ w,
                                                                  long long rows, int H, uint32_t* __restrict__ q8,
                                                                  float* __restrict__ w8) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * kSplitWarps + (threadIdx.x >> 5);  // (t, h) row
  if (r >= rows) return;
  split_row(q, w, r, H, q8, w8, lane);
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
