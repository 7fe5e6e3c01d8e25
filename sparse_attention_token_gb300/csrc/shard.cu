// shard.cu -- key-sharded top-k: one shard's (score, index) candidates and the exact merge
// of the candidates of every shard.
//
// GLM5 LoRA blog, section 3.1 (训练侧): with context parallelism a long sequence is split
// over devices, and a top-k taken on each shard alone matches the full-sequence top-k
// only 68 % of the time; gathering the shards' indexer results (THD layout plus an
// AllGather) makes it 99.97 %.  The exact version of that gather: each shard keeps its
// best min(k, visible) keys as (score, global index) in (score desc, index asc) order;
// the gathered lists are merged under the same order.  A key of the row's best k is
// among the best k of its own shard, so the merge loses nothing.
//
// The merge ranks every candidate directly: its position in its own (sorted) list plus,
// for every other list, the number of that list's entries that beat it (a binary search
// over the list held in shared memory); two lists are merged along a merge path instead
// (one binary search per thread, then a sequential merge of its share of the output).  Candidates compare as one 64-bit word
// (order-preserving score key, complemented index): a larger word is a higher score, or
// the same score at a lower index.  Indices are distinct across shards (disjoint key
// ranges), so ranks are distinct.
#include <cfloat>

#include "dsa_indexer.h"
#include "internal.h"
#include "ptx.cuh"

namespace dsa {

namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeMaxWords = 16384;  // n_shards * k_cand candidates per row in shared memory

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 ranks with +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Global indices and scores of one shard's top-k rows: idx[r, i] (shard-local, -1 padded)
// becomes idx + key_offset with its score, padding becomes (-1, -inf).
__global__ void shard_finish_kernel(int32_t* idx, float* cand_scores, const float* scores, long long ld, int T,
                                    int k, int key_offset) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const long long n = static_cast<long long>(T) * k;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = e / k;
    const int v = idx[e];
    if (v >= 0) {
      cand_scores[e] = scores[r * ld + v];
      idx[e] = v + key_offset;
    } else {
      cand_scores[e] = -INFINITY;
    }
  }
}

// Entries of the descending list w[0..len) greater than x.
__device__ __forceinline__ uint32_t count_greater(const uint64_t* w, uint32_t len, uint64_t x) {
  uint32_t lo = 0, hi = len;
  while (lo < hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if (w[mid] > x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// One CTA per query row: rank the n_shards * k_cand candidates, keep the best `keep`.
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const float* cand_scores, const int32_t* cand_idx,
                                                              int n_shards, int T, int k_cand, int topk_limit,
                                                              int k_out, int order, int32_t* topk, int vec4) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t* W = reinterpret_cast<uint64_t*>(smem);                       // [n_shards][k_cand]
  int32_t* sel = reinterpret_cast<int32_t*>(W + n_shards * k_cand);      // index order staging
  __shared__ uint32_t valid[32];
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int r = blockIdx.x, tid = threadIdx.x;
  const int n = n_shards * k_cand;
  if (tid < n_shards) valid[tid] = 0;
  __syncthreads();
  // padding: 0, below every candidate (a candidate's word is never 0)
  auto word = [](int32_t id, float sc) -> uint64_t {
    return id < 0 ? 0ull
                  : (static_cast<uint64_t>(score_key(sc)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(id));
  };
  if (vec4) {
    // four entries per 16-byte load (k_cand a multiple of 4, 16-byte aligned lists)
    for (int e = 4 * tid; e < n; e += 4 * kMergeThreads) {
      const int j = e / k_cand, p = e - j * k_cand;
      const long long g = (static_cast<long long>(j) * T + r) * k_cand + p;
      const int4 id = *reinterpret_cast<const int4*>(cand_idx + g);
      const float4 sc = *reinterpret_cast<const float4*>(cand_scores + g);
      W[e] = word(id.x, sc.x);
      W[e + 1] = word(id.y, sc.y);
      W[e + 2] = word(id.z, sc.z);
      W[e + 3] = word(id.w, sc.w);
    }
  } else {
    for (int e = tid; e < n; e += kMergeThreads) {
      const int j = e / k_cand, p = e - j * k_cand;
      const long long g = (static_cast<long long>(j) * T + r) * k_cand + p;
      W[e] = word(cand_idx[g], cand_scores[g]);
    }
  }
  __syncthreads();
  // a list's valid entries come first: its count is one past its last candidate
  for (int e = tid; e < n; e += kMergeThreads) {
    const int j = e / k_cand, p = e - j * k_cand;
    if (W[e] != 0 && (p + 1 == k_cand || W[e + 1] == 0)) valid[j] = static_cast<uint32_t>(p + 1);
  }
  __syncthreads();
  uint32_t total = 0;
  for (int j = 0; j < n_shards; ++j) total += valid[j];
  int keep = topk_limit;
  if (static_cast<long long>(keep) > total) keep = static_cast<int>(total);
  if (keep > k_out) keep = k_out;
  int32_t* out = topk + static_cast<long long>(r) * k_out;
  for (int i = keep + tid; i < k_out; i += kMergeThreads) out[i] = -1;
  if (n_shards == 2) {
    // two lists: a merge path.  Thread t writes outputs [o0, o1): one binary search finds
    // how many of the first o0 merged entries come from the first list, then it merges.
    const uint64_t* A = W;
    const uint64_t* Bl = W + k_cand;
    const int nA = static_cast<int>(valid[0]), nB = static_cast<int>(valid[1]);
    const int per = (keep + kMergeThreads - 1) / kMergeThreads;
    const int o0 = tid * per, o1 = min(keep, o0 + per);
    if (o0 < o1) {
      int lo = max(0, o0 - nB), hi = min(o0, nA);
      while (lo < hi) {  // the first i with A[i] not among the first o0
        const int mid = (lo + hi) >> 1;
        if (A[mid] > Bl[o0 - mid - 1]) lo = mid + 1;
        else hi = mid;
      }
      int i = lo, jb = o0 - lo;
      for (int o = o0; o < o1; ++o) {
        const bool take_a = jb >= nB || (i < nA && A[i] > Bl[jb]);
        const uint64_t x = take_a ? A[i++] : Bl[jb++];
        const int32_t id = static_cast<int32_t>(~static_cast<uint32_t>(x));
        if (order == DSA_ORDER_SCORE) out[o] = id;
        else sel[o] = id;
      }
    }
  }
  for (int e = tid; n_shards != 2 && e < n; e += kMergeThreads) {
    const int j = e / k_cand, p = e - j * k_cand;
    if (p >= keep || static_cast<uint32_t>(p) >= valid[j]) continue;  // ranked at least p
    const uint64_t x = W[e];
    uint32_t rank = static_cast<uint32_t>(p);
    for (int j2 = 0; j2 < n_shards && rank < static_cast<uint32_t>(keep); ++j2)
      if (j2 != j) rank += count_greater(W + j2 * k_cand, valid[j2], x);
    if (rank < static_cast<uint32_t>(keep)) {
      const int32_t id = static_cast<int32_t>(~static_cast<uint32_t>(x));
      if (order == DSA_ORDER_SCORE) out[rank] = id;
      else sel[rank] = id;
    }
  }
  if (order == DSA_ORDER_SCORE) return;
  __syncthreads();
  // ascending key index: bitonic sort of sel[0..keep) padded to a power of two
  int m = 1;
  while (m < keep) m <<= 1;
  for (int i = keep + tid; i < m; i += kMergeThreads) sel[i] = INT32_MAX;
  __syncthreads();
  for (int size = 2; size <= m; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < m; i += kMergeThreads) {
        const int jx = i ^ stride;
        if (jx > i) {
          const bool up = (i & size) == 0;
          const int32_t a = sel[i], b = sel[jx];
          if ((a > b) == up) { sel[i] = b; sel[jx] = a; }
        }
      }
      __syncthreads();
    }
  }
  for (int i = tid; i < keep; i += kMergeThreads) out[i] = sel[i];
}

}  // namespace

}  // namespace dsa

using namespace dsa;

extern "C" {

dsa_status dsa_indexer_shard_candidates_workspace_size(int T, int S, size_t* bytes) {
  if (!bytes || T < 0 || S < 0) return DSA_ERR_INVALID_ARGUMENT;
  const size_t ld = (static_cast<size_t>(S > 0 ? S : 1) + 3) & ~static_cast<size_t>(3);
  *bytes = static_cast<size_t>(T) * ld * 4;
  return DSA_OK;
}

dsa_status dsa_indexer_shard_candidates(const void* q, int q_dtype, const float* q_scale, const void* k_shard,
                                        int k_dtype, const float* k_scale, const float* w, int T, int S, int H,
                                        int D, int q_pos0, int key_offset, int k_cand, int32_t* cand_idx,
                                        float* cand_scores, void* workspace, size_t workspace_bytes,
                                        dsa_stream_t stream) {
  if (T < 0 || S < 0 || q_pos0 < 0 || key_offset < 0 || k_cand < 1 || k_cand > DSA_MAX_TOPK)
    return DSA_ERR_INVALID_ARGUMENT;
  if (static_cast<long long>(key_offset) + S > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!cand_idx || !cand_scores) return DSA_ERR_INVALID_ARGUMENT;
  size_t need = 0;
  dsa_indexer_shard_candidates_workspace_size(T, S, &need);
  if (S > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0))
    return DSA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const long long ld = static_cast<long long>((static_cast<size_t>(S > 0 ? S : 1) + 3) & ~static_cast<size_t>(3));
  float* scores = static_cast<float*>(workspace);
  // shard key s is global key key_offset + s: query t (position q_pos0 + t) sees it when
  // s <= q_pos0 - key_offset + t
  const long long shifted = static_cast<long long>(q_pos0) - key_offset;
  if (shifted < INT32_MIN / 2) return DSA_ERR_UNSUPPORTED;
  dsa_status s = DSA_OK;
  if (S > 0) {
    s = dense_scores(q, q_dtype, q_scale, k_shard, k_dtype, k_scale, w, T, S, H, D, static_cast<int>(shifted), scores,
                     ld, st);
    if (s != DSA_OK) return s;
  }
  s = dense_topk(S > 0 ? scores : nullptr, ld, T, S, static_cast<int>(shifted), k_cand, k_cand, DSA_ORDER_SCORE,
                 cand_idx, st);
  if (s != DSA_OK) return s;
  const long long n = static_cast<long long>(T) * k_cand;
  const int grid = static_cast<int>(std::min<long long>((n + 255) / 256, 4096));
  return launch_pdl(shard_finish_kernel, dim3(grid), dim3(256), 0, st, cand_idx, cand_scores,
                    static_cast<const float*>(scores), ld, T, k_cand, key_offset) == cudaSuccess
             ? DSA_OK
             : DSA_ERR_CUDA;
}

dsa_status dsa_indexer_merge_candidates(const float* cand_scores, const int32_t* cand_idx, int n_shards, int T,
                                        int k_cand, int topk_limit, int k_out, int order, int32_t* topk,
                                        dsa_stream_t stream) {
  if (n_shards < 1 || n_shards > 32 || T < 0 || k_cand < 1 || topk_limit < 1 || k_out < 1)
    return DSA_ERR_INVALID_ARGUMENT;
  if (order != DSA_ORDER_SCORE && order != DSA_ORDER_INDEX) return DSA_ERR_INVALID_ARGUMENT;
  if (k_out > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (static_cast<long long>(n_shards) * k_cand > kMergeMaxWords) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!cand_scores || !cand_idx || !topk) return DSA_ERR_INVALID_ARGUMENT;
  int keep_max = topk_limit < k_out ? topk_limit : k_out;
  if (keep_max > n_shards * k_cand) keep_max = n_shards * k_cand;
  int m = 1;
  while (m < keep_max) m <<= 1;
  const size_t smem = static_cast<size_t>(n_shards) * k_cand * 8 + (order == DSA_ORDER_INDEX ? m * 4 : 0);
  auto kern = merge_kernel;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  const int vec4 = (k_cand % 4 == 0 && (reinterpret_cast<uintptr_t>(cand_scores) & 15u) == 0 &&
                    (reinterpret_cast<uintptr_t>(cand_idx) & 15u) == 0)
                       ? 1
                       : 0;
  const cudaError_t e = launch_pdl(kern, dim3(T), dim3(kMergeThreads), smem, reinterpret_cast<cudaStream_t>(stream),
                                   cand_scores, cand_idx, n_shards, T, k_cand, topk_limit, k_out, order, topk, vec4);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // extern "C"
