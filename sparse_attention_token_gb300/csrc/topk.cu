// topk.cu -- per-row top-k of indexer scores (GLM5 TensorCast adaptation design,
// "性能模型设计" bucket 8, top-k selection; output width min(topk_limit, n_visible)).
//
// One CTA of 512 threads per row.  Scores become order-preserving unsigned keys
// (larger score -> larger key; -0.0 folded onto +0.0).  Selecting the best
// `keep` keys under the rule (score desc, index asc) is done in three steps:
//   1. radix select of the threshold key T: histograms of the top 11 bits, then
//      the next 11 and the last 10 bits restricted to the threshold bucket, giving
//      the count of keys above T and `need` = how many keys equal to T to take;
//   2. an ordered compaction in key-index order (block-wide prefix sums), which
//      keeps every key above T and the `need` lowest-index keys equal to T;
//   3. for DSA_ORDER_SCORE, a stable LSD radix sort (8-bit digits, descending) of
//      the kept keys, which leaves equal scores in ascending index order.
// Rows up to cache_cap keys are staged in shared memory once; longer rows are
// re-read from global memory (L2) by each pass.
#include "internal.h"

namespace dsa {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = kThreads * 4;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 compares equal to +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the block (thread order); *total gets the block sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* red, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < kWarps ? red[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kWarps) red[lane] = t;  // inclusive warp totals
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? red[warp - 1] : 0u;
  *total = red[kWarps - 1];
  __syncthreads();  // red is reused by the next call
  return before + x - v;
}

// Warp-aggregated shared-memory histogram increment (all 32 lanes must call).
__device__ __forceinline__ void hist_add(uint32_t* hist, bool active, uint32_t bin) {
  const uint32_t key = active ? bin : 0xFFFFFFFFu;
  const uint32_t peers = __match_any_sync(0xffffffffu, key);
  const int lane = threadIdx.x & 31;
  if (active && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
}

// Find the bucket b (scanning from the top) where the running count reaches `want`:
// out[0] = b, out[1] = keys in buckets above b, out[2] = keys in bucket b.
__device__ __forceinline__ void find_bucket(const uint32_t* hist, int nbins, uint32_t want, uint32_t* red,
                                            uint32_t* out) {
  const int per = nbins / kThreads;  // 4 or 2 bins per thread, highest bins to thread 0
  const int hi = nbins - per * static_cast<int>(threadIdx.x);
  uint32_t s = 0;
  for (int j = 1; j <= per; ++j) s += hist[hi - j];
  uint32_t tot;
  uint32_t run = block_excl_scan(s, red, &tot);
  for (int j = 1; j <= per; ++j) {
    const uint32_t c = hist[hi - j];
    if (run < want && run + c >= want) {
      out[0] = static_cast<uint32_t>(hi - j);
      out[1] = run;
      out[2] = c;
    }
    run += c;
  }
  __syncthreads();
}

struct RowSrc {
  const float* p;
  const uint32_t* cache;  // null when the row is not staged
  long long n;
};

// Keys i..i+3 of the row (cnt valid, the rest unspecified).
__device__ __forceinline__ int load4(const RowSrc& r, long long i, uint32_t (&u)[4]) {
  const long long rem = r.n - i;
  const int cnt = rem >= 4 ? 4 : (rem > 0 ? static_cast<int>(rem) : 0);
  if (r.cache) {
    if (cnt == 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(r.cache + i);
      u[0] = v.x; u[1] = v.y; u[2] = v.z; u[3] = v.w;
    } else {
      for (int j = 0; j < cnt; ++j) u[j] = r.cache[i + j];
    }
  } else {
    if (cnt == 4) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(r.p + i));
      u[0] = order_key(f.x); u[1] = order_key(f.y); u[2] = order_key(f.z); u[3] = order_key(f.w);
    } else {
      for (int j = 0; j < cnt; ++j) u[j] = order_key(__ldg(r.p + i + j));
    }
  }
  return cnt;
}

// Stable LSD radix sort of n <= 4096 (key, value) pairs by key, descending.
// Returns the buffer pair holding the result (a or b).
__device__ uint32_t* radix_sort_desc(uint32_t* ka, uint32_t* va, uint32_t* kb, uint32_t* vb, int n, uint32_t* cnt,
                                     uint32_t* red, uint32_t** vals_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // bits that differ between keys: digits that never change are skipped
  uint32_t diff = 0;
  if (n > 0) {
    const uint32_t k0 = ka[0];
    for (int i = tid; i < n; i += kThreads) diff |= ka[i] ^ k0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) diff |= __shfl_xor_sync(0xffffffffu, diff, o);
  if (lane == 0) red[warp] = diff;
  __syncthreads();
  diff = 0;
  for (int w = 0; w < kWarps; ++w) diff |= red[w];
  __syncthreads();

  const int CH = (((n + kWarps - 1) / kWarps) + 31) & ~31;  // elements per warp, multiple of 32
  const int rounds = CH / 32;                                // <= 8 for n <= 4096
  uint32_t *sk = ka, *sv = va, *dk = kb, *dv = vb;
  for (int sh = 0; sh < 32; sh += 8) {
    if (((diff >> sh) & 255u) == 0) continue;
    for (int i = tid; i < kWarps * 256; i += kThreads) cnt[i] = 0;
    __syncthreads();
    uint32_t offs[8], digs[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      offs[r] = 0;
      digs[r] = 256;
      if (r < rounds) {
        const int e = warp * CH + r * 32 + lane;
        const bool valid = e < n;
        const uint32_t d = valid ? 255u - ((sk[e] >> sh) & 255u) : 256u;
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        const uint32_t rank = __popc(peers & ((1u << lane) - 1u));
        const uint32_t before = valid ? cnt[warp * 256 + d] : 0u;
        __syncwarp();
        if (valid && rank == 0) cnt[warp * 256 + d] = before + __popc(peers);
        __syncwarp();
        offs[r] = before + rank;
        digs[r] = d;
      }
    }
    __syncthreads();
    {
      // exclusive scan in (digit, warp) order: thread t owns digit t/2, warps (t&1)*8 .. +7
      const int d = tid >> 1, w0 = (tid & 1) * 8;
      uint32_t v[8], s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { v[j] = cnt[(w0 + j) * 256 + d]; s += v[j]; }
      uint32_t tot;
      uint32_t ex = block_excl_scan(s, red, &tot);
#pragma unroll
      for (int j = 0; j < 8; ++j) { cnt[(w0 + j) * 256 + d] = ex; ex += v[j]; }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (r < rounds) {
        const int e = warp * CH + r * 32 + lane;
        if (e < n) {
          const uint32_t dest = cnt[warp * 256 + digs[r]] + offs[r];
          dk[dest] = sk[e];
          dv[dest] = sv[e];
        }
      }
    }
    __syncthreads();
    uint32_t* t;
    t = sk; sk = dk; dk = t;
    t = sv; sv = dv; dv = t;
  }
  *vals_out = sv;
  return sk;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a, int cache_cap, int ksel_cap) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint32_t red[32];
  __shared__ uint32_t sel_info[4];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);  // 16 KB: histogram / sort counters
  const int regionB = cache_cap > 2 * ksel_cap ? cache_cap : 2 * ksel_cap;
  uint32_t* cache = hist + kWarps * 256;                 // row cache, later sort scratch
  uint32_t* selk = cache + regionB;
  uint32_t* seli = selk + ksel_cap;
  const int tid = threadIdx.x;

  // ---- which row, how many visible keys
  long long n;
  const float* src;
  int32_t* out;
  if (!a.paged) {
    const int t = blockIdx.x;
    long long v = static_cast<long long>(a.q_pos0) + t + 1;
    if (v > a.S) v = a.S;
    n = v > 0 ? v : 0;
    src = a.scores + static_cast<long long>(t) * a.ld;
    out = a.topk + static_cast<long long>(t) * a.k_out;
  } else {
    const int r = a.row_base + blockIdx.x;
    int lo = 0, hi = a.B;  // last b with cu_q_lens[b] <= r
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.cu_q_lens[mid] <= r) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int q_len = a.cu_q_lens[b + 1] - a.cu_q_lens[b];
    const long long pos = static_cast<long long>(a.seq_lens[b]) - q_len + (r - a.cu_q_lens[b]);
    n = pos + 1 > 0 ? pos + 1 : 0;
    src = a.scores + static_cast<long long>(blockIdx.x) * a.ld;
    out = a.topk + static_cast<long long>(r) * a.k_out;
  }
  if (n > a.max_n) n = a.max_n;
  long long keep_ll = n;
  if (keep_ll > a.topk_limit) keep_ll = a.topk_limit;
  if (keep_ll > a.k_out) keep_ll = a.k_out;
  const int keep = static_cast<int>(keep_ll);
  for (int i = keep + tid; i < a.k_out; i += kThreads) out[i] = -1;
  if (keep == 0) return;

  RowSrc rs{src, nullptr, n};
  uint32_t T = 0;          // threshold key
  uint32_t need = 0;       // keys equal to T to keep (lowest indices first)
  if (n <= keep) {
    need = static_cast<uint32_t>(n);  // every key is kept
  } else {
    const bool cached = n <= cache_cap;
    // ---- pass 1: top 11 bits over the whole row (and stage the row)
    for (int i = tid; i < 2048; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (long long base = 0; base < n; base += kChunk) {
      const long long i = base + 4 * tid;
      uint32_t u[4] = {0u, 0u, 0u, 0u};
      const int c = load4(rs, i, u);
      if (cached) {
        if (c == 4) *reinterpret_cast<uint4*>(cache + i) = make_uint4(u[0], u[1], u[2], u[3]);
        else for (int j = 0; j < c; ++j) cache[i + j] = u[j];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) hist_add(hist, j < c, u[j] >> 21);
    }
    __syncthreads();
    if (cached) rs.cache = cache;
    uint32_t want = static_cast<uint32_t>(keep);
    find_bucket(hist, 2048, want, red, sel_info);
    const uint32_t d1 = sel_info[0];
    uint32_t above = sel_info[1];
    if (sel_info[2] == want - above) {
      T = (d1 << 21) - 1u;  // the whole bucket is kept: select keys >= d1 << 21
      need = 0;
    } else {
      // ---- pass 2: bits 10..20 inside bucket d1
      want -= above;
      uint32_t above_total = above;
      for (int i = tid; i < 2048; i += kThreads) hist[i] = 0;
      __syncthreads();
      for (long long base = 0; base < n; base += kChunk) {
        uint32_t u[4] = {0u, 0u, 0u, 0u};
        const int c = load4(rs, base + 4 * tid, u);
#pragma unroll
        for (int j = 0; j < 4; ++j) hist_add(hist, j < c && (u[j] >> 21) == d1, (u[j] >> 10) & 2047u);
      }
      __syncthreads();
      find_bucket(hist, 2048, want, red, sel_info);
      const uint32_t d2 = sel_info[0];
      above = sel_info[1];
      const uint32_t pre2 = (d1 << 11) | d2;
      if (sel_info[2] == want - above) {
        T = (pre2 << 10) - 1u;
        need = 0;
      } else {
        // ---- pass 3: bits 0..9 inside bucket (d1, d2)
        want -= above;
        above_total += above;
        for (int i = tid; i < 1024; i += kThreads) hist[i] = 0;
        __syncthreads();
        for (long long base = 0; base < n; base += kChunk) {
          uint32_t u[4] = {0u, 0u, 0u, 0u};
          const int c = load4(rs, base + 4 * tid, u);
#pragma unroll
          for (int j = 0; j < 4; ++j) hist_add(hist, j < c && (u[j] >> 10) == pre2, u[j] & 1023u);
        }
        __syncthreads();
        find_bucket(hist, 1024, want, red, sel_info);
        T = (pre2 << 10) | sel_info[0];
        need = want - sel_info[1];
      }
      (void)above_total;
    }
  }

  // ---- ordered compaction: keys > T, then the first `need` keys == T, in index order
  const bool by_score = a.order == 0;
  uint32_t g_run = 0, e_run = 0;  // keys > T and == T seen in earlier chunks
  const bool take_all = n <= keep;
  for (long long base = 0; base < n; base += kChunk) {
    const long long i = base + 4 * tid;
    uint32_t u[4] = {0u, 0u, 0u, 0u};
    const int c = load4(rs, i, u);
    uint32_t cg = 0, ce = 0;
    for (int j = 0; j < c; ++j) {
      if (take_all || u[j] > T) ++cg;
      else if (u[j] == T) ++ce;
    }
    uint32_t tot;
    const uint32_t pre = block_excl_scan((cg << 16) | ce, red, &tot);
    uint32_t g = g_run + (pre >> 16), e = e_run + (pre & 0xFFFFu);
    for (int j = 0; j < c; ++j) {
      int pos = -1;
      if (take_all || u[j] > T) {
        pos = static_cast<int>(g + (e < need ? e : need));
        ++g;
      } else if (u[j] == T) {
        if (e < need) pos = static_cast<int>(g + e);
        ++e;
      }
      if (pos >= 0) {
        if (by_score) {
          selk[pos] = u[j];
          seli[pos] = static_cast<uint32_t>(i + j);
        } else {
          out[pos] = static_cast<int32_t>(i + j);
        }
      }
    }
    g_run += tot >> 16;
    e_run += tot & 0xFFFFu;
  }
  if (!by_score) return;
  __syncthreads();
  uint32_t* vals;
  radix_sort_desc(selk, seli, cache, cache + ksel_cap, keep, hist, red, &vals);
  for (int i = tid; i < keep; i += kThreads) out[i] = static_cast<int32_t>(vals[i]);
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, int max_row_len, cudaStream_t st) {
  if (a.n_rows <= 0) return cudaSuccess;
  int keep_cap = a.k_out < a.topk_limit ? a.k_out : a.topk_limit;
  if (keep_cap > max_row_len) keep_cap = max_row_len;
  if (keep_cap < 1) keep_cap = 1;
  const int ksel_cap = (keep_cap + 3) & ~3;
  const int cache_cap = max_row_len <= 16384 ? ((max_row_len + 3) & ~3) : 0;
  const int regionB = cache_cap > 2 * ksel_cap ? cache_cap : 2 * ksel_cap;
  const size_t smem = (static_cast<size_t>(kWarps) * 256 + regionB + 2 * ksel_cap) * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  topk_kernel<<<a.n_rows, kThreads, smem, st>>>(a, cache_cap, ksel_cap);
  return cudaGetLastError();
}

}  // namespace dsa
