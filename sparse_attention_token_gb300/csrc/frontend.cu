// frontend.cu -- the indexer front-end: projections, k layer norm, RoPE, Hadamard
// rotation and per-row e4m3 quantisation, ahead of scoring.
//
// GLM5 TensorCast adaptation design, "DSA Indexer 融合语义算子" (the op's inputs:
// hidden_states, qa_normed, RoPE cos / sin, wq_b, wk, weights_proj, k_norm weight,
// indexer cache, slot_mapping) and its performance-model buckets 1-5, 9 and 10:
//   1-3  q = qa_normed @ wq_b^T, k = hidden @ wk^T, w = hidden @ weights_proj^T: bf16
//        products with fp32 accumulation on the tensor cores (proj_gemm.cu), the three
//        chains on the caller's stream and two library-owned streams; with enough tokens
//        the q projection finishes its rows (RoPE, rotation, quantisation) in its own
//        epilogue, otherwise it writes fp32 rows (split over K when the tokens are few)
//        for the q row kernel below;
//   4    RoPE on the first rope_dim values of every q head and of k;
//   5    FP8 cache only: the Walsh-Hadamard rotation (Sylvester order, times D^-1/2) of
//        q and k, then per-row e4m3 quantisation (scale = amax / 448);
//   9-10 k (and on FP8 its scale) written into the paged cache through slot_mapping.
// k_norm is a layer norm over D with the biased variance, times the weight (plus an
// optional bias).  One warp per row of D = 128 values: lane l holds values 4l..4l+3,
// so the Hadamard butterflies with distance 1 and 2 stay in the thread and the other
// five use shuffles; RoPE's half-split pairs are one shuffle of a value quad away.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "dsa_indexer.h"
#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kFrontWarps = 8;

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// RoPE on a row held as lane quads (x[j] = value 4 lane + j).  cs / sn: this row's
// rope_dim / 2 cosines and sines.
__device__ __forceinline__ void rope_row(float (&x)[4], const float* cs, const float* sn, int rope_dim,
                                         bool interleaved, int lane) {
  if (interleaved) {
    // pairs (2i, 2i + 1): this lane's pairs are i = 2 lane and 2 lane + 1
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int i = 2 * lane + p;
      if (2 * i + 1 < rope_dim) {
        const float c = __ldg(cs + i), s = __ldg(sn + i);
        const float a = x[2 * p], b = x[2 * p + 1];
        x[2 * p] = a * c - b * s;
        x[2 * p + 1] = a * s + b * c;
      }
    }
    return;
  }
  // pairs (i, i + rope_dim / 2); rope_dim / 2 is a multiple of 4, so a quad lies in one half
  const int half = rope_dim / 2, qoff = half / 4;
  const int e0 = 4 * lane;
  const bool first = e0 < half, second = !first && e0 < rope_dim;
  const int src = first ? lane + qoff : (second ? lane - qoff : lane);
  float p[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) p[j] = __shfl_sync(0xffffffffu, x[j], src);
  if (first || second) {
    const int i0 = first ? e0 : e0 - half;
    const float4 c = __ldg(reinterpret_cast<const float4*>(cs + i0));
    const float4 s = __ldg(reinterpret_cast<const float4*>(sn + i0));
    const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = first ? x[j] * cc[j] - p[j] * ss[j] : p[j] * ss[j] + x[j] * cc[j];
  }
}

// Normalised Walsh-Hadamard transform (Sylvester order) of a 128-value row.
__device__ __forceinline__ void hadamard_row(float (&x)[4], int lane) {
  float a = x[0] + x[1], b = x[0] - x[1], c = x[2] + x[3], d = x[2] - x[3];
  x[0] = a + c;
  x[1] = b + d;
  x[2] = a - c;
  x[3] = b - d;
#pragma unroll
  for (int bit = 1; bit < 32; bit <<= 1) {
    // the lane holding the upper value of a pair keeps p - x, the other x + p: one
    // fma with a +-1 factor (exact: a single rounding of the sum either way)
    const float sgn = (lane & bit) ? -1.f : 1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float p = __shfl_xor_sync(0xffffffffu, x[j], bit);
      x[j] = fmaf(sgn, x[j], p);
    }
  }
  const float s = 0.08838834764831845f;  // 128^-1/2 rounded to fp32
#pragma unroll
  for (int j = 0; j < 4; ++j) x[j] *= s;
}

// Per-row e4m3 codes of the quad (4 codes in one word) and the row's scale.
__device__ __forceinline__ uint32_t quantize_row(const float (&x)[4], float& scale) {
  uint32_t m = max(max(__float_as_uint(fabsf(x[0])), __float_as_uint(fabsf(x[1]))),
                   max(__float_as_uint(fabsf(x[2])), __float_as_uint(fabsf(x[3]))));
  m = __reduce_max_sync(0xffffffffu, m);
  const float amax = __uint_as_float(m);
  scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  return e4m3x2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale)) |
         (e4m3x2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale)) << 16);
}

__device__ __forceinline__ uint2 to_bf16x4(const float (&x)[4]) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]), hi = __floats2bfloat162_rn(x[2], x[3]);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

// q rows: Qf [T * H, 128] fp32 -> q_out (bf16 or e4m3 with q_scale).
__global__ void __launch_bounds__(kFrontWarps * 32) frontend_q_kernel(const float* __restrict__ Qf, int planes,
                                                                      long long rows,
                                                                      int H, const float* __restrict__ cosb,
                                                                      const float* __restrict__ sinb, int rope_dim,
                                                                      int interleaved, int fp8, void* q_out,
                                                                      float* __restrict__ q_scale) {
  const int lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * kFrontWarps + (threadIdx.x >> 5);
  if (r >= rows) return;
  const long long t = r >> (31 - __clz(H));  // H is a power of two: no 64-bit division
  ptx::grid_dep_wait();  // Qf comes from the projection kernel before this one
  ptx::grid_dep_launch();
  float x[4] = {0.f, 0.f, 0.f, 0.f};
  for (int pl = 0; pl < planes; ++pl) {  // the K splits' partial sums, in order
    const float4 v = reinterpret_cast<const float4*>(Qf + (pl * rows + r) * 128)[lane];
    x[0] += v.x; x[1] += v.y; x[2] += v.z; x[3] += v.w;
  }
  const long long half = rope_dim / 2;
  rope_row(x, cosb + t * half, sinb + t * half, rope_dim, interleaved != 0, lane);
  if (fp8) {
    hadamard_row(x, lane);
    float scale;
    const uint32_t codes = quantize_row(x, scale);
    reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(q_out) + r * 128)[lane] = codes;
    if (lane == 0) q_scale[r] = scale;
  } else {
    reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(q_out) + r * 128)[lane] = to_bf16x4(x);
  }
}

// k rows: Kf [T, 128] fp32 -> layer norm, RoPE, (Hadamard, quantisation) -> cache slot.
__global__ void __launch_bounds__(kFrontWarps * 32) frontend_k_kernel(
    const float* __restrict__ Kf, int planes, int T, const float* __restrict__ cosb, const float* __restrict__ sinb,
    int rope_dim, int interleaved, const float* __restrict__ ln_w, const float* __restrict__ ln_b, float eps,
    int fp8, const int64_t* __restrict__ slots, void* cache, float* __restrict__ scale_cache, long long n_slots,
    unsigned* status) {
  const int lane = threadIdx.x & 31;
  const long long t = static_cast<long long>(blockIdx.x) * kFrontWarps + (threadIdx.x >> 5);
  ptx::grid_dep_wait();  // Kf comes from the projection kernel before this one
  ptx::grid_dep_launch();
  if (t >= T) return;
  const long long slot = slots[t];
  if (slot < 0) return;  // padding token
  if (slot >= n_slots) {
    if (lane == 0) atomicOr(status, kStatusBadPage);
    return;
  }
  float x[4] = {0.f, 0.f, 0.f, 0.f};
  for (int pl = 0; pl < planes; ++pl) {  // the K splits' partial sums, in order
    const float4 v = reinterpret_cast<const float4*>(Kf + (pl * static_cast<long long>(T) + t) * 128)[lane];
    x[0] += v.x; x[1] += v.y; x[2] += v.z; x[3] += v.w;
  }
  const float mean = warp_sum((x[0] + x[1]) + (x[2] + x[3])) * 0.0078125f;  // / 128, exact
  float d2 = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[j] -= mean;
    d2 += x[j] * x[j];
  }
  const float var = warp_sum(d2) * 0.0078125f;
  const float inv = __fdiv_rn(1.f, __fsqrt_rn(var + eps));
  const float4 gw = __ldg(reinterpret_cast<const float4*>(ln_w) + lane);
  const float g[4] = {gw.x, gw.y, gw.z, gw.w};
  float bb[4] = {0.f, 0.f, 0.f, 0.f};
  if (ln_b) {
    const float4 b4 = __ldg(reinterpret_cast<const float4*>(ln_b) + lane);
    bb[0] = b4.x; bb[1] = b4.y; bb[2] = b4.z; bb[3] = b4.w;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) x[j] = x[j] * inv * g[j] + bb[j];
  const long long half = rope_dim / 2;
  rope_row(x, cosb + t * half, sinb + t * half, rope_dim, interleaved != 0, lane);
  if (fp8) {
    hadamard_row(x, lane);
    float scale;
    const uint32_t codes = quantize_row(x, scale);
    reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(cache) + slot * 128)[lane] = codes;
    if (lane == 0) scale_cache[slot] = scale;
  } else {
    reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(cache) + slot * 128)[lane] = to_bf16x4(x);
  }
}

// w [n] = the sum of `planes` partial planes of n values, in order.
__global__ void sum_planes_kernel(const float* __restrict__ P, int planes, long long n, float* __restrict__ out) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float s = 0.f;
    for (int pl = 0; pl < planes; ++pl) s += P[pl * n + i];
    out[i] = s;
  }
}

// Per device: two library-owned streams and the fork / join events.  Created on first
// use; calls on one device are serialised.
struct FrontCtx {
  bool ready = false;
  cudaStream_t side[2] = {};
  cudaEvent_t fork = nullptr, join[2] = {};
};
std::mutex g_front_mu;
FrontCtx g_front[64];

bool front_ctx_init(FrontCtx& c) {
  if (c.ready) return true;
  for (auto& st : c.side)
    if (!st && cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return false;
  const unsigned f = cudaEventDisableTiming;
  if (!c.fork && cudaEventCreateWithFlags(&c.fork, f) != cudaSuccess) return false;
  for (auto& e : c.join)
    if (!e && cudaEventCreateWithFlags(&e, f) != cudaSuccess) return false;
  c.ready = true;
  return true;
}

}  // namespace

namespace {
cudaError_t launch_frontend_q(const float* Qf, int planes, long long rows, int H, const float* cosb,
                              const float* sinb, int rope_dim, bool interleaved, bool fp8, void* q_out,
                              float* q_scale, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + kFrontWarps - 1) / kFrontWarps;
  return launch_pdl(frontend_q_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kFrontWarps * 32), 0, st, Qf,
                    planes, rows, H, cosb, sinb, rope_dim, interleaved ? 1 : 0, fp8 ? 1 : 0, q_out, q_scale);
}

cudaError_t launch_frontend_k(const float* Kf, int planes, int T, const float* cosb, const float* sinb,
                              int rope_dim, bool interleaved, const float* ln_w, const float* ln_b, float eps,
                              bool fp8, const int64_t* slots, void* cache, float* scale_cache, long long n_slots,
                              unsigned* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int blocks = (T + kFrontWarps - 1) / kFrontWarps;
  return launch_pdl(frontend_k_kernel, dim3(blocks), dim3(kFrontWarps * 32), 0, st, Kf, planes, T, cosb, sinb,
                    rope_dim, interleaved ? 1 : 0, ln_w, ln_b, eps, fp8 ? 1 : 0, slots, cache, scale_cache, n_slots,
                    status);
}
}  // namespace

// The fused q projection needs enough token tiles to fill the GPU; below this many
// tokens the projection is split over K instead and the q row kernel finishes the rows.
constexpr int kFusedQMinTokens = 512;

PreparePlan plan_prepare_launch(int T, int hidden_dim, int q_rank, int H, int D, int rope_dim) {
  PreparePlan p{};
  const size_t Tz = static_cast<size_t>(T > 0 ? T : 0);
  p.q_fused = T >= kFusedQMinTokens && proj_q_fused_supported(H, rope_dim);
  p.q_splits = p.q_fused ? 1 : proj_splits(T, H * D, q_rank);
  p.kw_splits = proj_dual_splits(T, hidden_dim);
  auto up = [](size_t b) { return (b + 255) / 256 * 256; };
  p.off_q = 0;
  p.off_k = p.off_q + (p.q_fused ? 0 : up(static_cast<size_t>(p.q_splits) * Tz * H * D * 4));
  p.off_w = p.off_k + up(static_cast<size_t>(p.kw_splits) * Tz * D * 4);
  p.total = p.off_w + (p.kw_splits > 1 ? up(static_cast<size_t>(p.kw_splits) * Tz * H * 4) : 0);
  return p;
}

// The two chains are independent until the end: q (projection and its rows) on the
// caller's stream, k and w (one projection, the k row kernel and cache write, the w
// planes' sum) on a library-owned stream forked from it and joined back.
cudaError_t launch_prepare(const PrepareLaunch& p, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_front_mu);
  FrontCtx& c = g_front[dev];
  if (!front_ctx_init(c)) return cudaErrorUnknown;
  const bool fp8 = p.fp8;
  const PreparePlan& P = p.plan;
  if ((e = cudaEventRecord(c.fork, st)) != cudaSuccess) return e;
  for (auto s2 : c.side)
    if ((e = cudaStreamWaitEvent(s2, c.fork, 0)) != cudaSuccess) return e;
  // q: projection with the rows finished in its epilogue, or fp32 planes and the row kernel
  cudaError_t eq;
  if (P.q_fused) {
    eq = launch_proj_q(p.qa_normed, p.wq_b, p.T, p.H, p.q_rank, p.cosb, p.sinb, p.rope_dim, p.interleaved, fp8,
                       p.q_out, p.q_scale, p.status, st);
  } else {
    eq = launch_proj_f32(p.qa_normed, p.wq_b, p.T, p.H * p.D, p.q_rank, P.q_splits, p.Qf, p.status, st);
    if (eq == cudaSuccess)
      eq = launch_frontend_q(p.Qf, P.q_splits, static_cast<long long>(p.T) * p.H, p.H, p.cosb, p.sinb, p.rope_dim,
                             p.interleaved, fp8, p.q_out, p.q_scale, st);
  }
  // k and w: one projection over hidden_states (its columns 0..127 are k, the rest w), then
  // the k rows (layer norm, RoPE, rotation, quantisation, cache write) and, when split over
  // K, the sum of w's planes
  const int S = P.kw_splits;
  cudaError_t ek = launch_proj_dual(p.hidden, p.wk, p.weights_proj, p.T, p.H, p.hidden_dim, S, p.Kf,
                                    S == 1 ? p.w_out : p.Wp, p.status, c.side[0]);
  if (ek == cudaSuccess)
    ek = launch_frontend_k(p.Kf, S, p.T, p.cosb, p.sinb, p.rope_dim, p.interleaved, p.ln_w, p.ln_b, p.eps, fp8,
                           p.slots, p.cache, p.scale_cache, p.n_slots, p.status, c.side[0]);
  cudaError_t ew = cudaSuccess;
  if (ek == cudaSuccess && S > 1) {
    const long long n = static_cast<long long>(p.T) * p.H;
    const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, 1024));
    ew = launch_pdl(sum_planes_kernel, dim3(blocks), dim3(256), 0, c.side[0], static_cast<const float*>(p.Wp), S, n,
                    p.w_out);
  }
  // join the side streams back into the caller's stream whatever happened above, so no
  // work of this call is left unordered with the caller's later work
  for (int i = 0; i < 2; ++i) {
    if ((e = cudaEventRecord(c.join[i], c.side[i])) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(st, c.join[i], 0)) != cudaSuccess) return e;
  }
  return eq != cudaSuccess ? eq : (ek != cudaSuccess ? ek : ew);
}

}  // namespace dsa
