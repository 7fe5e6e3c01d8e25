// cache_append.cu -- write the step's new indexer keys into the paged cache.
//
// The fused indexer op takes the indexer cache as a mutable argument together with
// slot_mapping, and its FP8 path writes the key cache and the scale cache after an
// activation quantisation (GLM5 TensorCast adaptation design, "DSA Indexer 融合语义算子";
// cost buckets 9 and 10).  Reading taken for the quantiser: one fp32 scale per token,
// scale = amax / 448 with amax the largest |k| of the row (1 for an all-zero row), and
// each element the e4m3 value nearest to k / scale, saturating at +-448.
//
// One warp per token, kAppendTokens tokens per warp with all their loads issued first.  A
// bf16 cache takes the row as it is (D = 64 or 128).  An e4m3
// cache (D = 128): lane l holds elements 4l..4l+3, the warp reduces the row's amax on
// the bit patterns of |x| (ordered like the values for non-negative floats), the scale
// and every element are IEEE divisions, and cvt.rn.satfinite.e4m3x2 rounds to nearest
// (ties to even) and saturates.  HBM-bound: 2D bytes read and D (+4) or 2D written per
// token.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dsa_indexer.h"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kAppendWarps = 8;
constexpr int kAppendTokens = 4;  // tokens per warp, their loads all in flight together

// Two fp32 values -> two e4m3 codes (lo in the low byte), round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kAppendWarps * 32) cache_append_kernel(
    const __nv_bfloat16* __restrict__ k_new, int n, int D, const int64_t* __restrict__ slots, void* cache,
    int fp8, float* __restrict__ scale_cache, long long n_slots, unsigned* status) {
  const int lane = threadIdx.x & 31;
  const long long i0 = (static_cast<long long>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5)) * kAppendTokens;
  // every load of the warp's tokens goes out before any is used
  long long slot[kAppendTokens];
  uint2 raw[kAppendTokens];
#pragma unroll
  for (int t = 0; t < kAppendTokens; ++t) {
    const long long i = i0 + t;
    slot[t] = i < n ? slots[i] : -1;
    raw[t] = make_uint2(0u, 0u);
    if (i < n) {
      const __nv_bfloat16* row = k_new + i * D;
      if (fp8 || D == 128) raw[t] = reinterpret_cast<const uint2*>(row)[lane];
      else raw[t].x = reinterpret_cast<const uint32_t*>(row)[lane];
    }
  }
#pragma unroll
  for (int t = 0; t < kAppendTokens; ++t) {
    const long long sl = slot[t];
    if (sl < 0) continue;  // padding token (or past the batch)
    if (sl >= n_slots) {
      if (lane == 0) atomicOr(status, kStatusBadPage);
      continue;
    }
    if (!fp8) {
      // D / 32 bf16 per lane: 8 bytes (D = 128) or 4 bytes (D = 64)
      if (D == 128) reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(cache) + sl * D)[lane] = raw[t];
      else reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(cache) + sl * D)[lane] = raw[t].x;
      continue;
    }
    // elements 4l .. 4l+3
    const float x0 = __uint_as_float(raw[t].x << 16), x1 = __uint_as_float(raw[t].x & 0xFFFF0000u);
    const float x2 = __uint_as_float(raw[t].y << 16), x3 = __uint_as_float(raw[t].y & 0xFFFF0000u);
    uint32_t m = max(max(__float_as_uint(fabsf(x0)), __float_as_uint(fabsf(x1))),
                     max(__float_as_uint(fabsf(x2)), __float_as_uint(fabsf(x3))));
    m = __reduce_max_sync(0xffffffffu, m);
    const float amax = __uint_as_float(m);
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    const uint32_t codes = e4m3x2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale)) |
                           (e4m3x2(__fdiv_rn(x2, scale), __fdiv_rn(x3, scale)) << 16);
    reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(cache) + sl * D)[lane] = codes;
    if (lane == 0) scale_cache[sl] = scale;
  }
}
}  // namespace

cudaError_t launch_cache_append(const void* k_new, int n, int D, const int64_t* slots, void* cache, bool fp8,
                                float* scale_cache, long long n_slots, unsigned* status, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long long per_block = static_cast<long long>(kAppendWarps) * kAppendTokens;
  const int blocks = static_cast<int>((n + per_block - 1) / per_block);
  cache_append_kernel<<<blocks, kAppendWarps * 32, 0, st>>>(static_cast<const __nv_bfloat16*>(k_new), n, D, slots,
                                                            cache, fp8 ? 1 : 0, scale_cache, n_slots, status);
  return cudaGetLastError();
}

}  // namespace dsa
