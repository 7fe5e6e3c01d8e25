#pragma once
// topk_kernels.cuh -- per-row top-k of indexer scores (GLM5 TensorCast adaptation design,
// "性能模型设计" bucket 8, top-k selection; output width min(topk_limit, n_visible)).
//
// One CTA of 256 threads per row (rows up to 8192 keys, held in registers), or a cluster
// of CTAs per row (longer rows, few of them), or one CTA streaming the row from memory
// (longer rows when there are enough of them to fill the GPU, and rows of any length).
// The best `keep` keys under (score desc, index asc) are found as follows.
//   Score order -- the linear-bucket path (linear_bucket_topk on a row in registers or
//      streamed from memory, cluster_linear_topk): one histogram of 4096 equal-width buckets between the row's
//      extremes, a descending scan for the threshold bucket and every bucket's start, the
//      keys of the buckets at and above it placed straight at their bucket's slots as
//      (key, bucket, index) words, and each word ranked among its bucket-mates.  It
//      declines rows whose scores are all equal, whose candidate buckets hold more than
//      kBucketLimit keys, or whose candidates overflow the buffers, and the general path
//      takes them.
//   General path (index order, declined rows): scores become
//      order-preserving unsigned keys (larger score -> larger key; -0.0 folded onto
//      +0.0).
//   1. One pass over the row builds a histogram of the top 12 key bits; a suffix
//      scan finds the bucket b where the running count reaches `keep`.
//   2. Fast path (the keys in buckets >= b fit the candidate buffer): an
//      order-preserving compaction (each warp owns a contiguous segment of the row;
//      ballots and warp prefix sums, no block-wide scans) copies every key of
//      bucket >= b with its index, in index order.
//        score order: the candidates are counted into buckets of a compressed key
//        and ranked within them (bucket_rank_out), or, when a bucket is too full, sorted
//        by a stable LSD radix sort over the differing 9-bit digits; the first `keep`
//        are the answer (ties keep ascending index: the input was in index order);
//        index order: the exact threshold inside bucket b is refined on the
//        candidates alone, then one ordered pass writes the selected indices.
//   3. Slow path (a huge threshold bucket, e.g. many equal scores): the exact
//      threshold key T and `need` (how many keys equal to T to keep, lowest index
//      first) are refined over the whole row with two more histogram passes, then
//      the ordered compaction keeps exactly `keep` keys, sorted as above.
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;            // top 12 key bits
constexpr int kMaxRounds = 16;         // sort: candidates per warp / 32
constexpr int kHistWords = kBins + kBins / 16;  // histogram with one pad word per 16 bins
constexpr int kSortBits = 9;           // radix sort digit width
constexpr int kSortBins = 1 << kSortBits;

// Histogram slot of bin b: one pad word after every 16 bins, so a thread reading 16
// consecutive bins while its neighbours read the next 16 hits distinct banks.
__device__ __forceinline__ int hslot(uint32_t b) { return static_cast<int>(b + (b >> 4)); }

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 compares equal to +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the block in thread order; *total gets the block sum.
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
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t r = red[w];
    before += w < warp ? r : 0u;
    tot += r;
  }
  *total = tot;
  __syncthreads();  // red is reused by the next call
  return before + x - v;
}

// Warp-inclusive prefix sum.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Bucket where the running count from the top reaches `want` (nbins = 16 * kThreads
// or 256).  out = {bucket, keys above it, keys in it}.  Thread t scans the bins
// nbins - per*(t+1) .. nbins - per*t - 1, highest first.
__device__ __forceinline__ void find_bucket(const uint32_t* hist, int nbins, uint32_t want, uint32_t* red,
                                            uint32_t* out) {
  const int per = nbins / kThreads;  // 16 or 1
  const int hi = nbins - per * static_cast<int>(threadIdx.x);
  uint32_t c[16];
  uint32_t s = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    c[j] = j < per ? hist[hslot(static_cast<uint32_t>(hi - 1 - j))] : 0u;
    s += c[j];
  }
  uint32_t tot;
  uint32_t run = block_excl_scan(s, red, &tot);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j < per && run < want && run + c[j] >= want) {
      out[0] = static_cast<uint32_t>(hi - 1 - j);
      out[1] = run;
      out[2] = c[j];
    }
    run += c[j];
  }
  __syncthreads();
}

// Four consecutive keys of the row starting at i (cnt of them valid, the rest 0).
__device__ __forceinline__ int load4(const float* p, long long n, long long i, uint32_t (&u)[4]) {
  const long long rem = n - i;
  if (rem >= 4) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(p + i));
    u[0] = order_key(f.x); u[1] = order_key(f.y); u[2] = order_key(f.z); u[3] = order_key(f.w);
    return 4;
  }
  const int c = rem > 0 ? static_cast<int>(rem) : 0;
  for (int j = 0; j < 4; ++j) u[j] = j < c ? order_key(__ldg(p + i + j)) : 0u;
  return c;
}

// Four consecutive scores of the row starting at i as raw fp32 bits (cnt of them valid, the
// rest 0).
__device__ __forceinline__ int load4_raw(const float* p, long long n, long long i, uint32_t (&x)[4]) {
  const long long rem = n - i;
  if (rem >= 4) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(p + i));
    x[0] = __float_as_uint(f.x); x[1] = __float_as_uint(f.y); x[2] = __float_as_uint(f.z); x[3] = __float_as_uint(f.w);
    return 4;
  }
  const int c = rem > 0 ? static_cast<int>(rem) : 0;
  for (int j = 0; j < 4; ++j) x[j] = j < c ? __float_as_uint(__ldg(p + i + j)) : 0u;
  return c;
}

// A row is split into kWarps contiguous segments, one per warp; a segment is read
// in blocks of 128 keys (lane l holds keys 4l..4l+3 of the block), so the order
// (segment, block, lane, element) is the key-index order.
__device__ __forceinline__ long long seg_len(long long n) { return ((n + kWarps - 1) / kWarps + 127) & ~127LL; }

// Segment read from global memory on every pass (any row length).  visit() walks the
// segment in batches of kBatch blocks whose loads are all issued before any is used,
// so a pass over a long row costs a few memory latencies, not one per block.
struct GlobalSeg {
  static constexpr int kBatch = 16;
  const float* p;
  long long s0, s1;
  int nb;
  int nfull;  // blocks full for every lane
  __device__ void init(const float* row, long long n) {
    const long long seg = seg_len(n);
    p = row;
    s0 = (threadIdx.x >> 5) * seg;
    s1 = min(n, s0 + seg);
    nb = s1 > s0 ? static_cast<int>((s1 - s0 + 127) / 128) : 0;
    nfull = s1 > s0 ? static_cast<int>((s1 - s0) / 128) : 0;
  }
  // f(x[4] raw fp32 bits, first index, valid count) for every block of this lane, in index
  // order; batches whose blocks are all full for every lane pass a constant count of 4.
  // Every lane of the warp calls f for the same blocks (f may use warp collectives).
  template <class F>
  __device__ __forceinline__ void visit_f(F f) const {
    const uint32_t i0 = static_cast<uint32_t>(s0) + 4u * (threadIdx.x & 31);
    int j0 = 0;
    for (; j0 + kBatch <= nfull; j0 += kBatch) {
      uint32_t x[kBatch][4];
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p + i0 + 128u * (j0 + jj)));
        x[jj][0] = __float_as_uint(v.x); x[jj][1] = __float_as_uint(v.y);
        x[jj][2] = __float_as_uint(v.z); x[jj][3] = __float_as_uint(v.w);
      }
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) f(x[jj], i0 + 128u * (j0 + jj), 4);
    }
    for (; j0 < nb; j0 += kBatch) {
      uint32_t x[kBatch][4];
      int c[kBatch];
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        const long long i = static_cast<long long>(i0) + 128LL * (j0 + jj);
        x[jj][0] = x[jj][1] = x[jj][2] = x[jj][3] = 0u;
        c[jj] = (j0 + jj < nb && i < s1) ? load4_raw(p, s1, i, x[jj]) : 0;
      }
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj)
        if (j0 + jj < nb) f(x[jj], i0 + 128u * (j0 + jj), c[jj]);
    }
  }
  // f(u[4], first index, valid count) for every block of this lane, in index order.
  template <class F>
  __device__ __forceinline__ void visit(F f) const {
    const int lane = threadIdx.x & 31;
    for (int j0 = 0; j0 < nb; j0 += kBatch) {
      uint32_t u[kBatch][4];
      int c[kBatch];
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        const long long i = s0 + 128LL * (j0 + jj) + 4 * lane;
        c[jj] = (j0 + jj < nb && i < s1) ? load4(p, s1, i, u[jj]) : 0;
      }
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        if (j0 + jj < nb) f(u[jj], s0 + 128LL * (j0 + jj) + 4 * lane, c[jj]);
      }
    }
  }
};

// Segment held in registers as raw fp32 bits (rows up to kWarps * NB * 128 keys).  Every
// load is issued before any loaded value is used, so a row costs one memory latency, not
// one per block.  visit() hands out order-preserving keys (the general path); visit_f()
// hands out the raw bits, and calls f with a constant count of 4 on the blocks that are
// full for every lane of the warp.
template <int NB>
struct RegSeg {
  uint32_t v[NB][4];
  long long s0;
  int len;    // keys of this warp's segment
  int nb;     // blocks holding at least one key
  int nfull;  // blocks full for every lane
  __device__ void init(const float* row, long long n) {
    const long long seg = seg_len(n);
    s0 = (threadIdx.x >> 5) * seg;
    const long long s1 = min(n, s0 + seg);
    len = s1 > s0 ? static_cast<int>(s1 - s0) : 0;
    nb = (len + 127) / 128;
    nfull = len / 128;
    const int l4 = 4 * static_cast<int>(threadIdx.x & 31);
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int r = len - 128 * j - l4;  // keys of block j left from this lane's first one
      const float* p = row + s0 + 128 * j + l4;
      if (r >= 4) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(p));
        v[j][0] = __float_as_uint(f.x); v[j][1] = __float_as_uint(f.y);
        v[j][2] = __float_as_uint(f.z); v[j][3] = __float_as_uint(f.w);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[j][e] = e < r ? __float_as_uint(__ldg(p + e)) : 0u;
      }
    }
  }
  // valid keys of block j for this lane (recomputed instead of held in registers)
  __device__ __forceinline__ int count(int j) const {
    const int r = len - 128 * j - 4 * static_cast<int>(threadIdx.x & 31);
    return r < 0 ? 0 : (r > 4 ? 4 : r);
  }
  template <class F>
  __device__ __forceinline__ void visit(F f) const {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      if (j < nb) {
        uint32_t u[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) u[e] = order_key(__uint_as_float(v[j][e]));
        f(u, s0 + 128LL * j + 4 * lane, count(j));
      }
    }
  }
  template <class F>
  __device__ __forceinline__ void visit_f(F f) const {
    const uint32_t i0 = static_cast<uint32_t>(s0) + 4u * (threadIdx.x & 31);
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      if (j < nfull) f(v[j], i0 + 128u * j, 4);
      else if (j < nb) f(v[j], i0 + 128u * j, count(j));
    }
  }
};

// hist[(u >> shift) & mask] += 1 for every key of the row with (u >> pshift) == pre
// (pshift = 32: every key).
template <class RS>
__device__ __forceinline__ void seg_hist(const RS& rs, uint32_t* hist, int shift, uint32_t mask, int pshift,
                                         uint32_t pre) {
  rs.visit([&](const uint32_t (&u)[4], long long, int c) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < c && (pshift >= 32 || (u[e] >> pshift) == pre)) atomicAdd(&hist[hslot((u[e] >> shift) & mask)], 1u);
  });
}

// Order-preserving compaction: key u (index i) is kept iff
//   u > T, or u == T and it is among the first `need` keys equal to T (index order),
// and kept keys are written to (ck, ci) in index order.  Returns the number kept.
template <class RS>
__device__ uint32_t seg_compact(const RS& rs, uint32_t T, uint32_t need, uint32_t* ck, uint32_t* ci,
                                uint32_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool ties = need != 0 && need != 0xFFFFFFFFu;
  uint32_t eq_before = 0;
  if (ties) {
    uint32_t ce = 0;
    rs.visit([&](const uint32_t (&u)[4], long long, int c) {
#pragma unroll
      for (int e = 0; e < 4; ++e) ce += (e < c && u[e] == T) ? 1u : 0u;
    });
    ce = __reduce_add_sync(0xffffffffu, ce);
    if (lane == 0) red[warp] = ce;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kWarps; ++w) eq_before += w < warp ? red[w] : 0u;
    __syncthreads();
  }
  // pass 1: kept keys per warp
  uint32_t kept = 0;
  {
    uint32_t run = eq_before;
    rs.visit([&](const uint32_t (&u)[4], long long, int c) {
      uint32_t e4 = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) e4 += (e < c && u[e] == T) ? 1u : 0u;
      const uint32_t ie = ties ? warp_incl_scan(e4) : e4;
      uint32_t r = run + ie - e4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (e < c) {
          if (u[e] > T) ++kept;
          else if (u[e] == T) { kept += r < need ? 1u : 0u; ++r; }
        }
      }
      if (ties) run += __shfl_sync(0xffffffffu, ie, 31);
    });
  }
  kept = __reduce_add_sync(0xffffffffu, kept);
  if (lane == 0) red[warp] = kept;
  __syncthreads();
  uint32_t base = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t r = red[w];
    base += w < warp ? r : 0u;
    total += r;
  }
  __syncthreads();
  // pass 2: write
  {
    uint32_t run = eq_before;
    rs.visit([&](const uint32_t (&u)[4], long long i, int c) {
      uint32_t e4 = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) e4 += (e < c && u[e] == T) ? 1u : 0u;
      const uint32_t ie = ties ? warp_incl_scan(e4) : e4;
      uint32_t r = run + ie - e4;
      uint32_t m = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (e < c) {
          if (u[e] > T) m |= 1u << e;
          else if (u[e] == T) { if (r < need) m |= 1u << e; ++r; }
        }
      }
      const uint32_t k = __popc(m);
      const uint32_t incl = warp_incl_scan(k);
      uint32_t pos = base + incl - k;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if ((m >> e) & 1u) {
          ck[pos] = u[e];
          ci[pos] = static_cast<uint32_t>(i + e);
          ++pos;
        }
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
      if (ties) run += __shfl_sync(0xffffffffu, ie, 31);
    });
  }
  __syncthreads();
  return total;
}

// Stable LSD radix sort of n (key, value) pairs by key, descending.  Only the bits
// below the highest bit in which the keys differ are sorted, kSortBits per pass (keys
// of one row's candidates usually differ in their low ~25 bits: 3 passes).
// n <= kWarps * 32 * kMaxRounds.  The sorted buffers come back in sk_out / sv_out.
__device__ void radix_sort_desc(uint32_t* ka, uint32_t* va, uint32_t* kb, uint32_t* vb, int n, uint32_t* cnt,
                                uint32_t* red, uint32_t** sk_out, uint32_t** sv_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t diff = 0;
  if (n > 0) {
    const uint32_t k0 = ka[0];
    for (int i = tid; i < n; i += kThreads) diff |= ka[i] ^ k0;
  }
  diff = __reduce_or_sync(0xffffffffu, diff);
  if (lane == 0) red[warp] = diff;
  __syncthreads();
  diff = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) diff |= red[w];
  __syncthreads();
  const int nbits = 32 - __clz(diff);  // 0 when all keys are equal

  const int CH = (((n + kWarps - 1) / kWarps) + 31) & ~31;  // keys per warp, multiple of 32
  const int rounds = CH / 32;
  uint32_t *sk = ka, *sv = va, *dk = kb, *dv = vb;
  for (int sh = 0; sh < nbits; sh += kSortBits) {
    for (int i = tid; i < kWarps * kSortBins; i += kThreads) cnt[i] = 0;
    __syncthreads();
    uint32_t offs[kMaxRounds];
    uint32_t digs[kMaxRounds];
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
      const int e = warp * CH + r * 32 + lane;
      digs[r] = (r < rounds && e < n) ? (kSortBins - 1) - ((sk[e] >> sh) & (kSortBins - 1)) : kSortBins;
    }
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
      offs[r] = 0;
      if (r < rounds) {
        const uint32_t d = digs[r];
        const bool valid = d < kSortBins;
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        const uint32_t rank = __popc(peers & ((1u << lane) - 1u));
        const uint32_t before = valid ? cnt[warp * kSortBins + d] : 0u;
        __syncwarp();
        if (valid && rank == 0) cnt[warp * kSortBins + d] = before + __popc(peers);
        __syncwarp();
        offs[r] = before + rank;
      }
    }
    __syncthreads();
    {
      // exclusive scan in (digit, warp) order: thread t owns digits 2t and 2t+1 for all warps
      uint32_t v[2][kWarps], s = 0;
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int w = 0; w < kWarps; ++w) { v[q][w] = cnt[w * kSortBins + 2 * tid + q]; s += v[q][w]; }
      uint32_t tot;
      uint32_t ex = block_excl_scan(s, red, &tot);
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int w = 0; w < kWarps; ++w) { cnt[w * kSortBins + 2 * tid + q] = ex; ex += v[q][w]; }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
      if (r < rounds) {
        const int e = warp * CH + r * 32 + lane;
        if (e < n) {
          const uint32_t dest = cnt[warp * kSortBins + digs[r]] + offs[r];
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
  *sk_out = sk;
  *sv_out = sv;
}

// Score order by buckets: the candidates' keys usually span a narrow range, so one
// counting pass over at most 4096 equal-width buckets between their minimum and
// maximum leaves a few keys per bucket; each key's final slot is its bucket's start
// plus the number of bucket-mates that beat it (higher key, or equal key and lower
// index).  Writes out[slot] = index for slots < keep.  Returns false (writing
// nothing) when some bucket holds more than kBucketLimit keys -- many equal or
// clustered scores -- so the caller sorts with the radix sort instead.  bk and bi
// are adjacent scratch arrays (bi == bk + n at least), used together as n 8-byte words.
// |value| bits of an order-preserving key (sign dropped).
__device__ __forceinline__ uint32_t key_mag(uint32_t u) {
  return (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : (~u & 0x7FFFFFFFu);
}
// Order-preserving key with magnitudes below floor_mag clamped to zero (monotone in u).
__device__ __forceinline__ uint32_t bucket_key(uint32_t u, uint32_t floor_mag) {
  const uint32_t m = key_mag(u);
  const uint32_t c = m > floor_mag ? m - floor_mag : 0u;
  return (u & 0x80000000u) ? 0x80000000u + c : 0x80000000u - c;
}

constexpr int kBucketLimit = 64;
constexpr int kScatterQueue = 160;  // a warp's queue: 31 left over + 4 x 32 from one block
constexpr int kSortBuckets = 4096;

__device__ bool bucket_rank_out(uint32_t* ck, const uint32_t* ci, int n, int keep, uint32_t* bk,
                                uint32_t* bi, uint32_t* cur, uint32_t* red, int32_t* out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int i = tid; i < n; i += kThreads) {
    const uint32_t u = ck[i];
    lo = min(lo, u);
    hi = max(hi, u);
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    red[warp] = lo;
    red[kWarps + warp] = hi;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    lo = min(lo, red[w]);
    hi = max(hi, red[kWarps + w]);
  }
  // Buckets are equal-width in a compressed key: magnitudes more than 12 binades below
  // the largest one are clamped to zero.  Key space is logarithmic across binades, so
  // when the candidates straddle zero the raw range covers every exponent of both signs
  // and a few buckets would get most keys; the compressed key is still monotone.
  const uint32_t mbig = max(key_mag(lo), key_mag(hi));
  const uint32_t floor_mag = (mbig >> 23) > 12u ? ((mbig >> 23) - 12u) << 23 : 0u;
  const uint32_t clo = bucket_key(lo, floor_mag), chi = bucket_key(hi, floor_mag);
  int sh = 0;
  while (((chi >> sh) - (clo >> sh)) >= static_cast<uint32_t>(kSortBuckets)) ++sh;
  const uint32_t base = clo >> sh;
  const int nb = static_cast<int>((chi >> sh) - base) + 1;
  for (int b = tid; b < nb; b += kThreads) cur[hslot(b)] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kThreads) atomicAdd(&cur[hslot((bucket_key(ck[i], floor_mag) >> sh) - base)], 1u);
  __syncthreads();
  // descending exclusive scan: start[b] = keys in buckets above b; thread t owns 16 bins
  uint32_t c[16], sum = 0, mx = 0;
  const int b_hi = nb - 16 * tid;  // bins b_hi-1 .. b_hi-16, highest first
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int b = b_hi - 1 - j;
    c[j] = b >= 0 ? cur[hslot(b)] : 0u;
    sum += c[j];
    mx = max(mx, c[j]);
  }
  uint32_t tot;
  uint32_t run = block_excl_scan(sum, red, &tot);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) mx = max(mx, red[w]);
  __syncthreads();  // red is free again before any caller reuses it
  if (mx > static_cast<uint32_t>(kBucketLimit)) return false;  // uniform across the block
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int b = b_hi - 1 - j;
    if (b >= 0) cur[hslot(b)] = run;
    run += c[j];
  }
  __syncthreads();
  // key and complemented index in one word: a larger word is a better key, or the same
  // key at a lower index, so ranking is one 8-byte load and one compare per element
  uint64_t* bw = reinterpret_cast<uint64_t*>(bk);  // bk and bi: 2n adjacent words
  for (int i = tid; i < n; i += kThreads) {
    const uint32_t u = ck[i];
    const uint32_t pos = atomicAdd(&cur[hslot((bucket_key(u, floor_mag) >> sh) - base)], 1u);
    bw[pos] = (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(~ci[i]);
  }
  __syncthreads();
  // cur[b] is now the end of bucket b; bucket b starts where bucket b + 1 ends
  for (int p = tid; p < n; p += kThreads) {
    const uint64_t x = bw[p];
    const int b = static_cast<int>((bucket_key(static_cast<uint32_t>(x >> 32), floor_mag) >> sh) - base);
    const uint32_t q0 = b + 1 < nb ? cur[hslot(b + 1)] : 0u, q1 = cur[hslot(b)];
    uint32_t rank = q0;
    uint32_t q = q0;
    for (; q + 4 <= q1; q += 4)
      rank += (bw[q] > x ? 1u : 0u) + (bw[q + 1] > x ? 1u : 0u) + (bw[q + 2] > x ? 1u : 0u) +
              (bw[q + 3] > x ? 1u : 0u);
    for (; q < q1; ++q) rank += bw[q] > x ? 1u : 0u;
    if (rank < static_cast<uint32_t>(keep)) ck[rank] = ~static_cast<uint32_t>(x);  // ck is free after the scatter
  }
  __syncthreads();
  // coalesced copy-out (scattered 4-byte global stores were a third of the sort's time)
  for (int i = tid; i < keep; i += kThreads) out[i] = static_cast<int32_t>(ck[i]);
  return true;
}

// Exact threshold among the keys of 12-bit bucket d1, of which `want` are still to
// be taken: two histogram passes (the next 12 bits, then the last 8) over the keys
// that `feed(hist, shift, mask, pshift, pre)` counts.  T = the threshold key,
// need = how many keys equal to T to take (lowest index first).
template <class Feed>
__device__ void refine_threshold(Feed feed, uint32_t d1, uint32_t want, uint32_t* hist, uint32_t* red,
                                 uint32_t* info, uint32_t* T_out, uint32_t* need_out) {
  for (int i = threadIdx.x; i < kHistWords; i += kThreads) hist[i] = 0;
  __syncthreads();
  feed(hist, 8, 4095u, 20, d1);
  __syncthreads();
  find_bucket(hist, kBins, want, red, info);
  const uint32_t d2 = info[0];
  want -= info[1];
  const uint32_t pre = (d1 << 12) | d2;  // top 24 bits of the threshold
  for (int i = threadIdx.x; i < kHistWords; i += kThreads) hist[i] = 0;
  __syncthreads();
  feed(hist, 0, 255u, 8, pre);
  __syncthreads();
  find_bucket(hist, 256, want, red, info);
  *T_out = (pre << 8) | info[0];
  *need_out = want - info[1];
}

// Shared-memory layout of every top-k kernel (dynamic part).
struct TopkSmem {
  uint32_t* hist;   // kHistWords counters, later sort counters
  uint32_t* ck;     // candidates: keys
  uint32_t* ci;     //             indices
  uint32_t* tk;     // sort scratch
  uint32_t* ti;
  uint32_t* merged; // cluster kernel: the row's merged histogram
};

__device__ __forceinline__ TopkSmem topk_smem(uint8_t* smem, int cand_cap) {
  TopkSmem m;
  m.hist = reinterpret_cast<uint32_t*>(smem);
  m.ck = m.hist + kHistWords;
  m.ci = m.ck + cand_cap;
  m.tk = m.ci + cand_cap;
  m.ti = m.tk + cand_cap;
  m.merged = m.ti + cand_cap;
  return m;
}

// Zero the n words at p (16-byte aligned, n a multiple of 4) with 16-byte stores.
__device__ __forceinline__ void zero_words(uint32_t* p, int n) {
  uint4* q = reinterpret_cast<uint4*>(p);
  for (int i = threadIdx.x; i < n / 4; i += kThreads) q[i] = make_uint4(0u, 0u, 0u, 0u);
}
// out[0..keep) = src[0..keep) (src 16-byte aligned), 16 bytes per store when out allows.
__device__ __forceinline__ void copy_out(int32_t* out, const uint32_t* src, int keep) {
  int i0 = 0;
  if ((reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
    const int n4 = keep / 4;
    for (int i = threadIdx.x; i < n4; i += kThreads)
      reinterpret_cast<int4*>(out)[i] = reinterpret_cast<const int4*>(src)[i];
    i0 = 4 * n4;
  }
  for (int i = i0 + threadIdx.x; i < keep; i += kThreads) out[i] = static_cast<int32_t>(src[i]);
}

// Score of an order-preserving key (inverse of order_key; -0.0 comes back as +0.0).
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Bucket of score x on a linear grid of kBins equal-width buckets between the row's
// smallest score lo and its largest hi: floor((x - lo) * scale) with
// scale = bucket_scale(hi - lo).  Every step is a correctly rounded IEEE operation (no
// contraction), so the bucket is a non-decreasing function of x and the same score always
// lands in the same bucket.  The floor is taken without a conversion instruction (those
// issue at a quarter of the FP32 rate): for 0 <= y < 2^23, y + 2^23 rounded toward zero is
// 2^23 + floor(y), whose low 23 bits are floor(y).  y = (x - lo) * scale is never negative
// (x >= lo) and below kBins, so no clamp: x - lo <= hi - lo = width (the same rounded
// subtraction at its largest), and scale rounds (kBins - 2^-10) / width, so
// y <= (kBins - 2^-10)(1 + 2^-24)^2 < kBins - 2^-11.
constexpr float kBucketSpan = static_cast<float>(kBins) - 0x1p-10f;
__device__ __forceinline__ float bucket_scale(float width) { return __fdiv_rn(kBucketSpan, width); }
__device__ __forceinline__ uint32_t lin_bucket(float x, float lo, float scale) {
  const float y = __fmul_rn(__fsub_rn(x, lo), scale);
  return __float_as_uint(__fadd_rz(y, 0x1p23f)) & 0x7FFFFFu;
}

// A candidate of the linear-bucket paths as one 8-byte word: the order-preserving key in
// the high half; the bucket (12 bits) and the complemented key index (20 bits) in the low
// half.  Words of one bucket compare like (key, then lower index first), so ranking a
// candidate among its bucket-mates is one compare per mate, and the word itself says
// which bucket to look in.
constexpr int kIndexBits = 20;
__device__ __forceinline__ uint2 cand_word(float x, uint32_t b, uint32_t idx) {
  return make_uint2((b << kIndexBits) | (~idx & ((1u << kIndexBits) - 1u)), order_key(x));
}
__device__ __forceinline__ uint32_t cand_bucket(uint64_t w) { return static_cast<uint32_t>(w) >> kIndexBits; }
__device__ __forceinline__ uint32_t cand_index(uint64_t w) {
  return ~static_cast<uint32_t>(w) & ((1u << kIndexBits) - 1u);
}

// Words in bw[q0, q1) greater than x (x's bucket-mates that beat it), four loads at a time
// so that a bucket of a few keys costs one shared-memory latency.  The loads run up to three
// words past q1 without a bound check: those hold lower buckets' candidates, whose scores
// are below every score of x's bucket (the bucket is a non-decreasing function of the
// score), or the kMatePad zero words the caller keeps after the last candidate -- either
// way smaller than x, so they never count.
constexpr uint32_t kMatePad = 4;
__device__ __forceinline__ uint32_t mates_above(const uint64_t* bw, uint32_t q0, uint32_t q1, uint64_t x) {
  uint32_t n = 0;
  for (uint32_t q = q0; q < q1; q += 4)
    n += (bw[q] > x ? 1u : 0u) + (bw[q + 1] > x ? 1u : 0u) + (bw[q + 2] > x ? 1u : 0u) + (bw[q + 3] > x ? 1u : 0u);
  return n;
}

// Descending exclusive scan of a kBins histogram in place: h[b] becomes the number of keys
// in the buckets above b, the start of bucket b in descending order, for the buckets at
// and above the threshold (a group of 16 wholly below it keeps its counts: nothing reads
// starts there).  Thread t owns bins 4095 - 16t .. 4080 - 16t.  The bucket where the
// running count from the top reaches want goes to info[0] and the keys of the buckets at
// and above it to info[1]; info[2] is set when one of those buckets holds more than
// kBucketLimit keys.  info[2] must be zero and red free at entry; ends with a barrier.
__device__ __forceinline__ void scan_desc_starts(uint32_t* h, uint32_t want, uint32_t* red, uint32_t* info) {
  static_assert(kBins == 16 * kThreads, "one group of 16 bins per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b_hi = kBins - 16 * tid;
  // bins b_hi - 1 - j of this thread's group g = 255 - tid sit at slots 17 g + 15 - j
  uint32_t* hg = h + hslot(static_cast<uint32_t>(b_hi - 1));
  uint32_t c[16], sum = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    c[j] = hg[-j];
    sum += c[j];
  }
  const uint32_t incl = warp_incl_scan(sum);
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  uint32_t r = incl - sum;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) r += w < warp ? red[w] : 0u;
  if (r < want) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t b = static_cast<uint32_t>(b_hi - 1 - j);
      if (r < want) {
        if (c[j] > static_cast<uint32_t>(kBucketLimit)) info[2] = 1u;
        if (r + c[j] >= want) {
          info[0] = b;
          info[1] = r + c[j];
        }
      }
      hg[-j] = r;
      r += c[j];
    }
  }
  __syncthreads();
}

// Score-order top-k of a row held in registers, in one histogram: the keys are counted
// in linear buckets between the row's extremes (Gaussian-like rows leave a few keys per
// bucket around the threshold), a descending scan gives the threshold bucket and every
// bucket's start, the keys of the buckets at and above the threshold go straight from
// registers to their bucket's slots, and each one's final rank is its bucket's start
// plus the bucket-mates that beat it (higher key, or the same key at a lower index).
// Returns false, having written nothing, when a bucket at or above the threshold holds
// more than kBucketLimit keys, the candidates overflow the buffers, or the row's scores
// are all equal; the caller then takes the general path.  RS is a row held in registers
// (RegSeg) or read from memory on each of the three passes (GlobalSeg, rows of at most
// 2^kIndexBits keys: the caller checks).
template <class RS>
__device__ bool linear_bucket_topk(const RS& rs, int keep, int32_t* out, int cand_cap, const TopkSmem& m,
                                   uint32_t* red, uint32_t* info) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the histogram is cleared while the row's loads are still in flight
  static_assert(kHistWords % 4 == 0, "16-byte clears");
  zero_words(m.hist, kHistWords);
  if (tid == 0) info[2] = 0u;
  // the row's extremes
  float fmin = __int_as_float(0x7f800000), fmax = -fmin;
  rs.visit_f([&](const uint32_t (&x)[4], uint32_t, int c) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < c) { fmin = fminf(fmin, __uint_as_float(x[e])); fmax = fmaxf(fmax, __uint_as_float(x[e])); }
  });
  uint32_t kmin = __reduce_min_sync(0xffffffffu, order_key(fmin));
  uint32_t kmax = __reduce_max_sync(0xffffffffu, order_key(fmax));
  if (lane == 0) { red[warp] = kmin; red[kWarps + warp] = kmax; }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kWarps; ++w) { kmin = min(kmin, red[w]); kmax = max(kmax, red[kWarps + w]); }
  const float lo = key_value(kmin), hi = key_value(kmax);
  const float width = __fsub_rn(hi, lo);
  const float scale = bucket_scale(width);
  // all-equal rows, and ranges whose width or scale is not a positive finite number
  if (!(width > 0.f) || !(scale > 0.f) || isinf(width) || isinf(scale)) return false;  // uniform: same inputs
  rs.visit_f([&](const uint32_t (&x)[4], uint32_t, int c) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < c) atomicAdd(&m.hist[hslot(lin_bucket(__uint_as_float(x[e]), lo, scale))], 1u);
  });
  __syncthreads();
  // red is free: its last readers passed the barrier above
  const uint32_t want = static_cast<uint32_t>(keep);
  scan_desc_starts(m.hist, want, red, info);
  const uint32_t d1 = info[0], n_cand = info[1];
  // candidate words (n_cand of 8 bytes, then kMatePad zero words) live in tk and ti,
  // 2 * cand_cap adjacent words
  if (info[2] != 0u || n_cand + kMatePad > static_cast<uint32_t>(cand_cap)) return false;
  uint2* bw2 = reinterpret_cast<uint2*>(m.tk);
  if (tid < static_cast<int>(kMatePad)) bw2[n_cand + tid] = make_uint2(0u, 0u);
  rs.visit_f([&](const uint32_t (&x)[4], uint32_t i, int c) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (e < c) {
        const float f = __uint_as_float(x[e]);
        const uint32_t b = lin_bucket(f, lo, scale);
        if (b >= d1) bw2[atomicAdd(&m.hist[hslot(b)], 1u)] = cand_word(f, b, i + e);
      }
    }
  });
  __syncthreads();
  // hist[b] is now the end of bucket b; bucket b starts where bucket b + 1 ends
  const uint64_t* bw = reinterpret_cast<const uint64_t*>(m.tk);
  for (uint32_t p = tid; p < n_cand; p += kThreads) {
    const uint64_t x = bw[p];
    const uint32_t b = cand_bucket(x);
    const uint32_t q0 = b + 1 < static_cast<uint32_t>(kBins) ? m.hist[hslot(b + 1)] : 0u, q1 = m.hist[hslot(b)];
    const uint32_t rank = q0 + mates_above(bw, q0, q1, x);
    if (rank < want) m.ck[rank] = cand_index(x);
  }
  __syncthreads();
  copy_out(out, m.ck, keep);
  return true;
}

// Score-order top-k of a long row read from memory, in one pass over the row.  A sample of
// the row (32 runs of 128 keys spread over it) gives a value t above which about
// (keep + spec_cap) / 2 of the row's keys should lie; one pass keeps every key >= t, with
// its index, in shared memory (spec, room for spec_cap); when at least `keep` keys were
// kept and they fit, the answer lies among them (the keep-th best key is >= t), and the
// linear-bucket selection runs on them: their extremes (taken in the pass), one histogram
// of 4096 buckets, the descending scan, placement at each bucket's slots, the rank among
// bucket-mates.  Rows of
// at most spec_cap keys are kept whole.  Returns 1 when the output is written; 0 when the
// sample misjudged t (too few kept keys, or too many for spec) -- the caller then reads the
// row in three passes; -1 when the kept keys defeat the buckets (all equal, a bucket of
// more than kBucketLimit keys at or above the threshold) -- the caller takes the general
// path.  Rows of at most 2^kIndexBits keys (the caller checks).
constexpr int kSampleRuns = 32;  // 4 per warp, 128 keys each: 16 keys per thread
__device__ int stream_topk(const GlobalSeg& rs, const float* row, long long n, int keep, int32_t* out, int cand_cap,
                           uint2* spec, int spec_cap, const TopkSmem& m, uint32_t* red, uint32_t* info) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t want = static_cast<uint32_t>(keep);
  // -- the threshold t from a sample (every key of a row that spec holds whole)
  float t = -__int_as_float(0x7f800000);
  zero_words(m.hist, kHistWords);
  if (tid == 0) { info[2] = 0u; info[3] = 0u; }
  if (n > spec_cap) {
    float x[16];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int run = 4 * warp + r;
      const long long o = ((n - 128) * run / (kSampleRuns - 1)) & ~3LL;  // o + 128 <= n, 16-byte aligned
      const float4 v = __ldg(reinterpret_cast<const float4*>(row + o + 4 * lane));
      x[4 * r] = v.x; x[4 * r + 1] = v.y; x[4 * r + 2] = v.z; x[4 * r + 3] = v.w;
    }
    float fmin = x[0], fmax = x[0];
#pragma unroll
    for (int j = 1; j < 16; ++j) { fmin = fminf(fmin, x[j]); fmax = fmaxf(fmax, x[j]); }
    uint32_t kmin = __reduce_min_sync(0xffffffffu, order_key(fmin));
    uint32_t kmax = __reduce_max_sync(0xffffffffu, order_key(fmax));
    if (lane == 0) { red[warp] = kmin; red[kWarps + warp] = kmax; }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kWarps; ++w) { kmin = min(kmin, red[w]); kmax = max(kmax, red[kWarps + w]); }
    const float lo = key_value(kmin), hi = key_value(kmax);
    const float width = __fsub_rn(hi, lo);
    const float scale = bucket_scale(width);
    __syncthreads();  // red is reused below
    if (!(width > 0.f) || !(scale > 0.f) || isinf(width) || isinf(scale)) {
      t = hi;  // a flat or unbounded sample: keep the keys at its top
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) atomicAdd(&m.hist[hslot(lin_bucket(x[j], lo, scale))], 1u);
      __syncthreads();
      // sample keys at and above the bucket that should hold the target count
      const long long target = (static_cast<long long>(keep) + spec_cap) / 2;
      long long r_s = (target * (kSampleRuns * 128) + n - 1) / n;
      if (r_s < 1) r_s = 1;
      find_bucket(m.hist, kBins, static_cast<uint32_t>(r_s), red, info);  // r_s <= the 4096 sample keys
      t = __fadd_rn(lo, __fdiv_rn(static_cast<float>(info[0]), scale));
      zero_words(m.hist, kHistWords);
      if (tid == 0) info[2] = 0u;
    }
  }
  __syncthreads();
  // -- one pass: keep every key >= t with its index.  Each warp takes its segment in
  // batches of 8 blocks (all loads issued first); a lane counts its kept keys in the batch,
  // one warp scan and one shared atomic give every lane its first slot, and the lane
  // writes its keys there in index order (predicated stores, no per-key vote).
  uint32_t* kept = &info[3];
  float fmin = __int_as_float(0x7f800000), fmax = -fmin;  // the kept keys' extremes
  {
    constexpr int kB = 8;  // blocks per batch: 32 keys per lane in registers
    const uint32_t i0 = static_cast<uint32_t>(rs.s0) + 4u * static_cast<uint32_t>(lane);
    const uint32_t s1 = static_cast<uint32_t>(rs.s1);
    // FULL: the batch's blocks are full for every lane (no bound checks)
    auto batch = [&](auto full_tag, int j0) {
      constexpr bool FULL = decltype(full_tag)::value;
      uint32_t x[kB][4];
#pragma unroll
      for (int jj = 0; jj < kB; ++jj) {
        const uint32_t i = i0 + 128u * (j0 + jj);
        if constexpr (FULL) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(rs.p + i));
          x[jj][0] = __float_as_uint(v.x); x[jj][1] = __float_as_uint(v.y);
          x[jj][2] = __float_as_uint(v.z); x[jj][3] = __float_as_uint(v.w);
        } else {
          x[jj][0] = x[jj][1] = x[jj][2] = x[jj][3] = 0u;
          if (j0 + jj < rs.nb && i < s1) load4_raw(rs.p, rs.s1, i, x[jj]);
        }
      }
      auto keeps = [&](int jj, int e) {
        return (FULL || i0 + 128u * (j0 + jj) + e < s1) && __uint_as_float(x[jj][e]) >= t;
      };
      uint32_t cnt = 0;
#pragma unroll
      for (int jj = 0; jj < kB; ++jj)
#pragma unroll
        for (int e = 0; e < 4; ++e) cnt += keeps(jj, e) ? 1u : 0u;
      const uint32_t incl = warp_incl_scan(cnt);
      const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
      if (tot == 0) return;  // uniform in the warp
      uint32_t base = 0;
      if (lane == 31) base = atomicAdd(kept, tot);
      uint32_t pos = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
      if (cnt == 0) return;
#pragma unroll
      for (int jj = 0; jj < kB; ++jj)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (keeps(jj, e)) {
            const float f = __uint_as_float(x[jj][e]);
            fmin = fminf(fmin, f);
            fmax = fmaxf(fmax, f);
            if (pos < static_cast<uint32_t>(spec_cap)) spec[pos] = make_uint2(x[jj][e], i0 + 128u * (j0 + jj) + e);
            ++pos;
          }
        }
    };
    int j0 = 0;
    for (; j0 + kB <= rs.nfull; j0 += kB) batch(std::true_type{}, j0);
    for (; j0 < rs.nb; j0 += kB) batch(std::false_type{}, j0);
  }
  uint32_t kmin = __reduce_min_sync(0xffffffffu, order_key(fmin));
  uint32_t kmax = __reduce_max_sync(0xffffffffu, order_key(fmax));
  if (lane == 0) { red[warp] = kmin; red[kWarps + warp] = kmax; }  // red is free since the sample
  __syncthreads();
  const uint32_t n_spec = *kept;
  if (n_spec < want || n_spec > static_cast<uint32_t>(spec_cap)) return 0;  // uniform: shared value
  // -- the linear-bucket selection on the kept keys (their extremes came with the pass)
#pragma unroll
  for (int w = 0; w < kWarps; ++w) { kmin = min(kmin, red[w]); kmax = max(kmax, red[kWarps + w]); }
  const float lo = key_value(kmin), hi = key_value(kmax);
  const float width = __fsub_rn(hi, lo);
  const float scale = bucket_scale(width);
  if (!(width > 0.f) || !(scale > 0.f) || isinf(width) || isinf(scale)) return -1;  // uniform: same inputs
  for (uint32_t p = tid; p < n_spec; p += kThreads)
    atomicAdd(&m.hist[hslot(lin_bucket(__uint_as_float(spec[p].x), lo, scale))], 1u);
  __syncthreads();
  // red is free: its last readers passed the barrier above
  scan_desc_starts(m.hist, want, red, info);
  const uint32_t d1 = info[0], n_cand = info[1];
  if (info[2] != 0u || n_cand + kMatePad > static_cast<uint32_t>(cand_cap)) return -1;
  uint2* bw2 = reinterpret_cast<uint2*>(m.tk);
  if (tid < static_cast<int>(kMatePad)) bw2[n_cand + tid] = make_uint2(0u, 0u);
  for (uint32_t p = tid; p < n_spec; p += kThreads) {
    const uint2 v = spec[p];
    const float f = __uint_as_float(v.x);
    const uint32_t b = lin_bucket(f, lo, scale);
    if (b >= d1) bw2[atomicAdd(&m.hist[hslot(b)], 1u)] = cand_word(f, b, v.y);
  }
  __syncthreads();
  // hist[b] is now the end of bucket b; bucket b starts where bucket b + 1 ends
  const uint64_t* bw = reinterpret_cast<const uint64_t*>(m.tk);
  for (uint32_t p = tid; p < n_cand; p += kThreads) {
    const uint64_t x = bw[p];
    const uint32_t b = cand_bucket(x);
    const uint32_t q0 = b + 1 < static_cast<uint32_t>(kBins) ? m.hist[hslot(b + 1)] : 0u, q1 = m.hist[hslot(b)];
    const uint32_t rank = q0 + mates_above(bw, q0, q1, x);
    if (rank < want) m.ck[rank] = cand_index(x);
  }
  __syncthreads();
  copy_out(out, m.ck, keep);
  return 1;
}

struct RowInfo {
  long long n;
  const float* src;
  int32_t* out;
  int keep;
};

__device__ __forceinline__ RowInfo row_info(const TopkArgs& a, int r_local) {
  RowInfo R;
  if (!a.paged) {
    const int t = r_local;
    long long v = static_cast<long long>(a.q_pos0) + t + 1;
    if (v > a.S) v = a.S;
    R.n = v > 0 ? v : 0;
    R.src = a.scores + static_cast<long long>(t) * a.ld;
    R.out = a.topk + static_cast<long long>(t) * a.k_out;
  } else {
    const int r = a.row_base + r_local;
    int lo = 0, hi = a.B;  // last b with cu_q_lens[b] <= r
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.cu_q_lens[mid] <= r) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int q_len = a.cu_q_lens[b + 1] - a.cu_q_lens[b];
    const long long pos = static_cast<long long>(a.seq_lens[b]) - q_len + (r - a.cu_q_lens[b]);
    R.n = pos + 1 > 0 ? pos + 1 : 0;
    R.src = a.scores + static_cast<long long>(r_local) * a.ld;
    R.out = a.topk + static_cast<long long>(r) * a.k_out;
  }
  if (R.n > a.max_n) R.n = a.max_n;
  long long keep_ll = R.n;
  if (keep_ll > a.topk_limit) keep_ll = a.topk_limit;
  if (keep_ll > a.k_out) keep_ll = a.k_out;
  R.keep = static_cast<int>(keep_ll);
  return R;
}

// Final output from candidates (ck, ci) in index order:
//   exact    -- the candidates are exactly the kept keys;
//   otherwise every key of 12-bit bucket >= d1 (`want` still to take from bucket d1).
__device__ void finish_row(const TopkSmem& m, uint32_t n_cand, bool exact, uint32_t d1, uint32_t want, int keep,
                           bool by_score, int32_t* out, uint32_t* red, uint32_t* info) {
  const int tid = threadIdx.x;
  if (by_score) {
    if (bucket_rank_out(m.ck, m.ci, static_cast<int>(n_cand), keep, m.tk, m.ti, m.hist, red, out)) return;
    uint32_t *sk, *sv;
    radix_sort_desc(m.ck, m.ci, m.tk, m.ti, static_cast<int>(n_cand), m.hist, red, &sk, &sv);
    for (int i = tid; i < keep; i += kThreads) out[i] = static_cast<int32_t>(sv[i]);
    return;
  }
  if (exact) {
    for (int i = tid; i < keep; i += kThreads) out[i] = static_cast<int32_t>(m.ci[i]);
    return;
  }
  uint32_t T, need;
  const uint32_t nc = n_cand;
  const uint32_t* ckp = m.ck;
  auto feed_cand = [&](uint32_t* h, int shift, uint32_t mask, int pshift, uint32_t pre) {
    for (uint32_t i = tid; i < nc; i += kThreads) {
      const uint32_t u = ckp[i];
      if ((u >> pshift) == pre) atomicAdd(&h[hslot((u >> shift) & mask)], 1u);
    }
  };
  refine_threshold(feed_cand, d1, want, m.hist, red, info, &T, &need);
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t per = ((n_cand + kWarps - 1) / kWarps + 31) & ~31u;
  const uint32_t c0 = warp * per, c1 = min(n_cand, c0 + per);
  uint32_t cgt = 0, ceq = 0;
  for (uint32_t i = c0 + lane; i < c1; i += 32) {
    cgt += m.ck[i] > T ? 1u : 0u;
    ceq += m.ck[i] == T ? 1u : 0u;
  }
  cgt = __reduce_add_sync(0xffffffffu, cgt);
  ceq = __reduce_add_sync(0xffffffffu, ceq);
  if (lane == 0) red[warp] = cgt;
  __syncthreads();
  uint32_t gbase = 0;
  for (int w = 0; w < warp; ++w) gbase += red[w];
  __syncthreads();
  if (lane == 0) red[warp] = ceq;
  __syncthreads();
  uint32_t ebase = 0;
  for (int w = 0; w < warp; ++w) ebase += red[w];
  for (uint32_t i0 = c0; i0 < c1; i0 += 32) {
    const uint32_t i = i0 + lane;
    const bool valid = i < c1;
    const uint32_t u = valid ? m.ck[i] : 0u;
    const bool gt = valid && u > T, eq = valid && u == T;
    const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t g = gbase + __popc(bg & lt), e = ebase + __popc(be & lt);
    if (gt) out[g + (e < need ? e : need)] = static_cast<int32_t>(m.ci[i]);
    else if (eq && e < need) out[g + e] = static_cast<int32_t>(m.ci[i]);
    gbase += __popc(bg);
    ebase += __popc(be);
  }
}

// The whole top-k of one row by one CTA, reading the row through RS.
template <class RS>
__device__ void row_topk(const RS& rs, long long n, int keep, bool by_score, int32_t* out, int cand_cap,
                         const TopkSmem& m, uint32_t* red, uint32_t* info) {
  const int tid = threadIdx.x;
  uint32_t n_cand;
  bool exact = true;
  uint32_t d1 = 0, want = 0;
  if (n <= keep) {
    n_cand = seg_compact(rs, 0u, 0xFFFFFFFFu, m.ck, m.ci, red);  // every key
  } else {
    for (int i = tid; i < kHistWords; i += kThreads) m.hist[i] = 0;
    __syncthreads();
    seg_hist(rs, m.hist, 20, 4095u, 32, 0u);
    __syncthreads();
    find_bucket(m.hist, kBins, static_cast<uint32_t>(keep), red, info);
    d1 = info[0];
    const uint32_t above = info[1], in_b = info[2];
    want = static_cast<uint32_t>(keep) - above;
    if (in_b == want) {
      n_cand = seg_compact(rs, (d1 << 20) - 1u, 0u, m.ck, m.ci, red);  // the whole bucket is kept
    } else if (above + in_b <= static_cast<uint32_t>(cand_cap)) {
      n_cand = seg_compact(rs, (d1 << 20) - 1u, 0u, m.ck, m.ci, red);  // every key of buckets >= d1
      exact = false;
    } else {
      // huge threshold bucket: exact threshold over the row, exactly `keep` keys
      uint32_t T, need;
      auto feed_row = [&](uint32_t* h, int shift, uint32_t mask, int pshift, uint32_t pre) {
        seg_hist(rs, h, shift, mask, pshift, pre);
      };
      refine_threshold(feed_row, d1, want, m.hist, red, info, &T, &need);
      n_cand = seg_compact(rs, T, need, m.ck, m.ci, red);
    }
  }
  finish_row(m, n_cand, exact, d1, want, keep, by_score, out, red, info);
}

template <int NB>  // NB > 0: rows up to kWarps * NB * 128 keys held in registers; 0: any length
__global__ void __launch_bounds__(kThreads, NB == 8 ? 3 : 2) topk_kernel(const TopkArgs a, int cand_cap) {
  ptx::grid_dep_wait();  // the scores come from the previous kernel on the stream
  ptx::grid_dep_launch();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint32_t red[2 * kWarps];
  __shared__ uint32_t info[4];
  const TopkSmem m = topk_smem(smem, cand_cap);
  const RowInfo R = row_info(a, blockIdx.x);
  if (a.prefetch_ahead > 0 && threadIdx.x == 32 && blockIdx.x + a.prefetch_ahead < a.n_rows) {
    // the row a later CTA on this part of the GPU will read: into L2 while this one works
    const RowInfo P = row_info(a, blockIdx.x + a.prefetch_ahead);
    const long long bytes = ((P.n + 3) & ~3LL) * 4;  // whole 16-byte units inside the row's ld
    if (bytes > 0 && (reinterpret_cast<uintptr_t>(P.src) & 15u) == 0)
      ptx::bulk_prefetch_l2(P.src, static_cast<uint32_t>(bytes));
  }
  if (NB == 0 && a.spec_cap > 0 && threadIdx.x == 32 && R.n > a.spec_cap && (reinterpret_cast<uintptr_t>(R.src) & 15u) == 0) {
    // a long row read once: all of it into L2 now, in 64 KB pieces, while the sample that
    // sets the threshold is taken (the pass then reads from L2)
    const long long bytes = ((R.n + 3) & ~3LL) * 4;  // whole 16-byte units inside the row's ld
    for (long long o = 0; o < bytes; o += 65536)
      ptx::bulk_prefetch_l2(reinterpret_cast<const char*>(R.src) + o, static_cast<uint32_t>(min(65536LL, bytes - o)));
  }
  for (int i = R.keep + threadIdx.x; i < a.k_out; i += kThreads) R.out[i] = -1;
  if (R.keep == 0) return;
  using RS = typename std::conditional<NB == 0, GlobalSeg, RegSeg<(NB > 0 ? NB : 1)>>::type;
  static_assert(NB == 0 || kWarps * NB * 128 <= (1 << kIndexBits), "key indices must fit the candidate word");
  RS rs;
  rs.init(R.src, R.n);
  if (a.order == 0 && (NB > 0 || R.n <= (1LL << kIndexBits))) {
    int got = 0;
    if constexpr (NB == 0) {
      if (a.spec_cap > 0) {
        uint2* spec = reinterpret_cast<uint2*>(m.ti + cand_cap);  // after the four candidate arrays
        got = stream_topk(rs, R.src, R.n, R.keep, R.out, cand_cap, spec, a.spec_cap, m, red, info);
        if (got > 0) return;
        __syncthreads();  // the next path reuses the shared buffers
      }
    }
    if (got == 0) {
      if (linear_bucket_topk(rs, R.keep, R.out, cand_cap, m, red, info)) return;
      __syncthreads();  // the general path reuses the shared buffers
    }
  }
  row_topk(rs, R.n, R.keep, a.order == 0, R.out, cand_cap, m, red, info);
}

// ---------------------------------------------------------------- long rows: a cluster of CTAs per row

__device__ __forceinline__ uint32_t dsmem_ld(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void dsmem_st(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st2(uint32_t addr, uint2 v) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa(const void* p, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(d)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
  return d;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void red_add_cluster(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Sum the CL local histograms (m.hist of every CTA) into m.merged of every CTA: each CTA
// adds its non-zero bins into every CTA's merged histogram with remote atomics (a row's
// keys fill a few hundred of the 4096 bins), between two cluster barriers.  Every CTA
// zeroes its own m.merged before the call, after its last read of the previous merge.
template <int CL>
__device__ void cluster_merge_hist(const TopkSmem& m, uint32_t rank, int bmin = 0) {
  cluster_barrier();  // every local histogram complete, every merged histogram zeroed
  for (int b = threadIdx.x + bmin; b < kBins; b += kThreads) {
    const uint32_t c = m.hist[hslot(b)];
    if (c != 0) {
#pragma unroll
      for (int j = 0; j < CL; ++j) red_add_cluster(mapa(&m.merged[hslot(b)], static_cast<uint32_t>(j)), c);
    }
  }
  cluster_barrier();  // every contribution has landed
}


// The score-order fast path of linear_bucket_topk spread over a cluster: the row's extreme
// keys are exchanged between the CL CTAs, each CTA counts its part into linear buckets, the
// merged histogram (the same in every CTA) gives the threshold bucket and every bucket's
// start, the candidates go straight from registers to CTA 0's buffer at their bucket's
// slots (the bucket cursors live in CTA 0), and CTA 0 ranks them inside their buckets.
// Returns false in every CTA, having written no output, when the row's scores are all
// equal, a bucket at or above the threshold holds more than kBucketLimit keys, or the
// candidates overflow CTA 0's buffer; the caller then takes the general path.
template <int NB, int CL>
__device__ bool cluster_linear_topk(const RegSeg<NB>& rs, long long part_lo, long long n, int keep, int32_t* out,
                                    int cand_cap, const TopkSmem& m, uint32_t* red, uint32_t* info, uint32_t* cmm,
                                    uint32_t rank) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  static_assert(CL * kWarps * NB * 128 <= (1 << kIndexBits), "key indices must fit the candidate word");
  if (cand_cap < kBins) return false;  // the bucket cursors need kBins words of m.ci (same in every CTA)
  // the histograms are cleared while the row's loads are still in flight
  zero_words(m.hist, kHistWords);
  zero_words(m.merged, kHistWords);
  float fmin = __int_as_float(0x7f800000), fmax = -fmin;
  rs.visit_f([&](const uint32_t (&x)[4], uint32_t, int c) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < c) { fmin = fminf(fmin, __uint_as_float(x[e])); fmax = fmaxf(fmax, __uint_as_float(x[e])); }
  });
  uint32_t kmin = __reduce_min_sync(0xffffffffu, order_key(fmin));
  uint32_t kmax = __reduce_max_sync(0xffffffffu, order_key(fmax));
  if (lane == 0) { red[warp] = kmin; red[kWarps + warp] = kmax; }
  __syncthreads();
  // Exchange through each CTA's own slots: write this CTA's extremes, one cluster barrier,
  // then warp 0 reads every CTA's slots and reduces them.
  if (tid == 0) {
#pragma unroll
    for (int w = 0; w < kWarps; ++w) { kmin = min(kmin, red[w]); kmax = max(kmax, red[kWarps + w]); }
    cmm[0] = kmin;
    cmm[1] = kmax;
  }
  cluster_barrier();  // every CTA's extremes are in its slots
  if (warp == 0) {
    uint32_t gmin = 0xFFFFFFFFu, gmax = 0u;
    if (lane < CL) {
      gmin = dsmem_ld(mapa(&cmm[0], static_cast<uint32_t>(lane)));
      gmax = dsmem_ld(mapa(&cmm[1], static_cast<uint32_t>(lane)));
    }
    gmin = __reduce_min_sync(0xffffffffu, gmin);
    gmax = __reduce_max_sync(0xffffffffu, gmax);
    if (lane == 0) { red[0] = gmin; red[1] = gmax; }
  }
  __syncthreads();
  const float lo = key_value(red[0]), hi = key_value(red[1]);
  const float width = __fsub_rn(hi, lo);
  const float scale = bucket_scale(width);
  if (!(width > 0.f) || !(scale > 0.f) || isinf(width) || isinf(scale)) return false;  // the same in every CTA
  rs.visit_f([&](const uint32_t (&x)[4], uint32_t, int c) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < c) atomicAdd(&m.hist[hslot(lin_bucket(__uint_as_float(x[e]), lo, scale))], 1u);
  });
  __syncthreads();
  // Only the buckets at and above the lowest of the CTAs' own thresholds for keep / CL keys
  // are merged: every CTA holds at least that many keys there, so the row's threshold
  // bucket is among them (a CTA with fewer keys takes bucket 0, and everything is merged).
  if (tid == 0) info[0] = 0u;
  __syncthreads();  // also: every thread has read lo and hi from red
  find_bucket(m.hist, kBins, static_cast<uint32_t>((keep + CL - 1) / CL), red, info);
  if (tid == 0) {
    cmm[2] = info[0];
    info[2] = 0u;  // the overflow flag of the scan below
  }
  cluster_barrier();  // every CTA's own threshold is in its slot; every local histogram is complete
  if (warp == 0) {
    uint32_t b = 0xFFFFFFFFu;
    if (lane < CL) b = dsmem_ld(mapa(&cmm[2], static_cast<uint32_t>(lane)));
    b = __reduce_min_sync(0xffffffffu, b);
    if (lane == 0) red[0] = b;
  }
  __syncthreads();
  const int bmin = static_cast<int>(red[0]);
  // Each CTA sums the CTAs' local histograms at and above bmin itself, reading them in place
  // (they stay unchanged until the barrier after the placement), and keeps the lower-ranked
  // CTAs' share of every bucket: its own slots in bucket b start after their keys.
  uint32_t* cursor = m.ci;  // kBins words, plain bucket index
  for (int b = tid + bmin; b < kBins; b += kThreads) {
    uint32_t tot = m.hist[hslot(b)], pre = 0;
#pragma unroll
    for (int j = 0; j < CL; ++j) {
      if (j == static_cast<int>(rank)) continue;
      const uint32_t v = dsmem_ld(mapa(&m.hist[hslot(b)], static_cast<uint32_t>(j)));
      tot += v;
      pre += j < static_cast<int>(rank) ? v : 0u;
    }
    m.merged[hslot(b)] = tot;
    cursor[b] = pre;
  }
  __syncthreads();
  // descending exclusive scan of the merged histogram, identical in every CTA (exact at
  // and above bmin, which the threshold bucket is; zero below)
  const uint32_t want = static_cast<uint32_t>(keep);
  scan_desc_starts(m.merged, want, red, info);
  const uint32_t d1 = info[0], n_cand = info[1];
  if (info[2] != 0u || n_cand + kMatePad > static_cast<uint32_t>(cand_cap)) return false;
  for (int b = tid + static_cast<int>(d1); b < kBins; b += kThreads) cursor[b] += m.merged[hslot(b)];
  // CTA 0 keeps kMatePad zero words after the last candidate slot (see mates_above)
  if (rank == 0 && tid < static_cast<int>(kMatePad))
    reinterpret_cast<uint2*>(m.tk)[n_cand + tid] = make_uint2(0u, 0u);
  __syncthreads();
  const uint32_t bw0 = mapa(m.tk, 0);
  // One compare rejects most keys: every score of a bucket >= d1 is at least
  // lo + (d1 - 1) / scale - (|lo| + |hi|) 2^-20 -- a whole bucket below the boundary, less a
  // margin far above the roundings of lin_bucket and of this bound (each at most 2^-24 of
  // |lo| + |hi|).  The exact bucket is taken only for the scores that pass.
  const float tpre = lo + static_cast<float>(d1 > 0 ? d1 - 1 : 0) / scale - (fabsf(lo) + fabsf(hi)) * 0x1p-20f;
  const float fpre = tpre > lo ? tpre : lo;
  // The keys that pass go through a per-warp queue in shared memory (ballots give their
  // slots), and the queue is placed 32 entries at a time with every lane busy: a few
  // percent of a long row's keys pass, so placing them where they lie would run the
  // placement code for most of the warp's key slots with one or two lanes active.
  // m.ck is free until CTA 0 ranks (after the cluster barrier below).
  static_assert(kWarps * kScatterQueue * 2 <= kBins, "scatter queues fit m.ck");
  uint2* q = reinterpret_cast<uint2*>(m.ck) + warp * kScatterQueue;
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t qn = 0;  // entries in this warp's queue (the same in every lane)
  auto place = [&](uint2 w) {
    const float f = __uint_as_float(w.x);
    const uint32_t b = lin_bucket(f, lo, scale);
    if (b >= d1) dsmem_st2(bw0 + 8u * atomicAdd(&cursor[b], 1u), cand_word(f, b, w.y));
  };
  rs.visit_f([&](const uint32_t (&x)[4], uint32_t i, int c4) {
    const uint32_t i0 = static_cast<uint32_t>(part_lo) + i;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool pass = e < c4 && __uint_as_float(x[e]) >= fpre;
      const uint32_t bal = __ballot_sync(0xffffffffu, pass);
      if (pass) q[qn + __popc(bal & lt)] = make_uint2(x[e], i0 + e);
      qn += __popc(bal);
    }
    __syncwarp();
    while (qn >= 32) {
      qn -= 32;
      place(q[qn + lane]);
      __syncwarp();  // the slots just read are refilled by the next block
    }
  });
  if (lane < qn) place(q[lane]);
  cluster_barrier();  // every candidate has landed in CTA 0; nobody touches its memory after this
  if (rank != 0) return true;
  // CTA 0: bucket b spans [start[b], start[b - 1]) (the buckets below follow it); the last
  // candidate bucket d1 ends at n_cand
  const uint64_t* bw = reinterpret_cast<const uint64_t*>(m.tk);
  for (uint32_t p = tid; p < n_cand; p += kThreads) {
    const uint64_t x = bw[p];
    const uint32_t b = cand_bucket(x);
    const uint32_t q0 = m.merged[hslot(b)], q1 = b > d1 ? m.merged[hslot(b - 1)] : n_cand;
    const uint32_t rk = q0 + mates_above(bw, q0, q1, x);
    if (rk < want) m.ck[rk] = cand_index(x);
  }
  __syncthreads();
  copy_out(out, m.ck, keep);
  return true;
}

template <int NB, int CL>  // CL CTAs per row, each holding up to kWarps * NB * 128 keys in registers
__global__ void __launch_bounds__(kThreads, 2) topk_cluster_kernel(const TopkArgs a, int cand_cap) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint32_t red[2 * kWarps];
  __shared__ uint32_t info[4];
  __shared__ uint32_t counts[CL];
  __shared__ uint32_t cmm[3];
  const TopkSmem m = topk_smem(smem, cand_cap);
  const uint32_t rank = cluster_rank();
  const RowInfo R = row_info(a, blockIdx.x / CL);
  const int tid = threadIdx.x;
  if (rank == 0)
    for (int i = R.keep + tid; i < a.k_out; i += kThreads) R.out[i] = -1;
  if (R.keep == 0) return;  // the same decision in every CTA of the cluster
  const bool by_score = a.order == 0;
  // this CTA's contiguous part of the row
  const long long part = ((R.n + CL - 1) / CL + 1023) & ~1023LL;
  const long long lo = min(R.n, static_cast<long long>(rank) * part);
  const long long len = min(R.n - lo, part);
  const int row_id = static_cast<int>(blockIdx.x / CL);
  if (a.prefetch_ahead > 0 && tid == 32 && row_id + a.prefetch_ahead < a.n_rows) {
    // this CTA's part of the row a cluster one resident wave later reads: into L2 now
    const RowInfo P = row_info(a, row_id + a.prefetch_ahead);
    const long long ppart = ((P.n + CL - 1) / CL + 1023) & ~1023LL;
    const long long plo = min(P.n, static_cast<long long>(rank) * ppart);
    const long long plen = min(P.n - plo, ppart);
    const long long bytes = ((plen + 3) & ~3LL) * 4;
    if (plen > 0 && (reinterpret_cast<uintptr_t>(P.src + plo) & 15u) == 0)
      ptx::bulk_prefetch_l2(P.src + plo, static_cast<uint32_t>(bytes));
  }
  RegSeg<NB> rs;
  rs.init(R.src + lo, len);
  if (by_score && cluster_linear_topk<NB, CL>(rs, lo, R.n, R.keep, R.out, cand_cap, m, red, info, cmm, rank))
    return;
  cluster_barrier();  // the general path below starts from clean buffers in every CTA

  const bool take_all = R.n <= R.keep;
  uint32_t T = 0;         // candidates: keys > T (every key when take_all)
  uint32_t d1 = 0, want = 0;
  bool exact = take_all;
  bool fallback = false;  // tie-heavy row: the first CTA finishes it alone
  if (!take_all) {
    for (int i = tid; i < kHistWords; i += kThreads) m.hist[i] = m.merged[i] = 0;
    __syncthreads();
    seg_hist(rs, m.hist, 20, 4095u, 32, 0u);
    __syncthreads();
    cluster_merge_hist<CL>(m, rank);
    find_bucket(m.merged, kBins, static_cast<uint32_t>(R.keep), red, info);
    d1 = info[0];
    const uint32_t above = info[1], in_b = info[2];
    want = static_cast<uint32_t>(R.keep) - above;
    T = (d1 << 20) - 1u;
    exact = in_b == want;
    if (!exact && above + in_b > static_cast<uint32_t>(cand_cap)) {
      // one more level, cluster-wide: bits 8..19 inside bucket d1
      for (int i = tid; i < kHistWords; i += kThreads) m.hist[i] = m.merged[i] = 0;
      __syncthreads();
      seg_hist(rs, m.hist, 8, 4095u, 20, d1);
      __syncthreads();
      cluster_merge_hist<CL>(m, rank);
      find_bucket(m.merged, kBins, want, red, info);
      const uint32_t d2 = info[0], above2 = info[1], in_b2 = info[2];
      const uint32_t pre = (d1 << 12) | d2;
      T = (pre << 8) - 1u;  // candidates: top 24 bits >= pre
      want -= above2;
      exact = in_b2 == want;
      if (!exact) {
        // the threshold sits inside 24-bit bucket pre: keep that level for the refinement
        if (above + above2 + in_b2 > static_cast<uint32_t>(cand_cap)) fallback = true;
        d1 = pre;  // finish_row refines inside (top 24 bits == pre) below
      }
    }
  }
  if (fallback) {
    cluster_barrier();
    if (rank != 0) return;
    GlobalSeg gs;
    gs.init(R.src, R.n);
    row_topk(gs, R.n, R.keep, by_score, R.out, cand_cap, m, red, info);
    return;
  }
  // candidates of this CTA, counted, then written in index order into CTA 0's buffers
  uint32_t cnt = 0;
  rs.visit([&](const uint32_t (&u)[4], long long, int c) {
#pragma unroll
    for (int e = 0; e < 4; ++e) cnt += (e < c && (take_all || u[e] > T)) ? 1u : 0u;
  });
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  const int lane = tid & 31, warp = tid >> 5;
  if (lane == 0) red[warp] = cnt;
  __syncthreads();
  uint32_t wbase = 0, ctotal = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    wbase += w < warp ? red[w] : 0u;
    ctotal += red[w];
  }
  if (tid == 0) dsmem_st(mapa(&counts[rank], 0), ctotal);
  cluster_barrier();
  uint32_t cbase = 0, n_cand = 0;
  if (tid < CL) counts[tid] = rank == 0 ? counts[tid] : dsmem_ld(mapa(&counts[tid], 0));
  __syncthreads();
#pragma unroll
  for (int j = 0; j < CL; ++j) {
    cbase += j < static_cast<int>(rank) ? counts[j] : 0u;
    n_cand += counts[j];
  }
  const bool overflow = n_cand > static_cast<uint32_t>(cand_cap);  // same in every CTA
  if (!overflow) {
    const uint32_t ck0 = mapa(m.ck, 0), ci0 = mapa(m.ci, 0);
    uint32_t base = cbase + wbase;
    rs.visit([&](const uint32_t (&u)[4], long long i, int c) {
      uint32_t msk = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) msk |= ((e < c && (take_all || u[e] > T)) ? 1u : 0u) << e;
      const uint32_t k = __popc(msk);
      const uint32_t incl = warp_incl_scan(k);
      uint32_t pos = base + incl - k;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if ((msk >> e) & 1u) {
          dsmem_st(ck0 + 4u * pos, u[e]);
          dsmem_st(ci0 + 4u * pos, static_cast<uint32_t>(lo + i + e));
          ++pos;
        }
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    });
  }
  cluster_barrier();  // CTA 0 holds every candidate; nobody touches its memory after this
  if (rank != 0) return;
  if (overflow) {
    GlobalSeg gs;
    gs.init(R.src, R.n);
    row_topk(gs, R.n, R.keep, by_score, R.out, cand_cap, m, red, info);
    return;
  }
  if (!by_score && !exact && (d1 >> 12) != 0) {
    // index order with a 24-bit threshold prefix: refine the last 8 bits on the candidates
    uint32_t need;
    const uint32_t nc = n_cand, pre = d1;
    const uint32_t* ckp = m.ck;
    for (int i = tid; i < kHistWords; i += kThreads) m.hist[i] = 0;
    __syncthreads();
    for (uint32_t i = tid; i < nc; i += kThreads)
      if ((ckp[i] >> 8) == pre) atomicAdd(&m.hist[hslot(ckp[i] & 255u)], 1u);
    __syncthreads();
    find_bucket(m.hist, 256, want, red, info);
    const uint32_t Tx = (pre << 8) | info[0];
    need = want - info[1];
    // keep key > Tx and the first `need` keys == Tx (candidates are in index order)
    const uint32_t per = ((nc + kWarps - 1) / kWarps + 31) & ~31u;
    const uint32_t c0 = warp * per, c1 = min(nc, c0 + per);
    uint32_t cgt = 0, ceq = 0;
    for (uint32_t i = c0 + lane; i < c1; i += 32) {
      cgt += ckp[i] > Tx ? 1u : 0u;
      ceq += ckp[i] == Tx ? 1u : 0u;
    }
    cgt = __reduce_add_sync(0xffffffffu, cgt);
    ceq = __reduce_add_sync(0xffffffffu, ceq);
    if (lane == 0) red[warp] = cgt;
    __syncthreads();
    uint32_t gb = 0;
    for (int w = 0; w < warp; ++w) gb += red[w];
    __syncthreads();
    if (lane == 0) red[warp] = ceq;
    __syncthreads();
    uint32_t eb = 0;
    for (int w = 0; w < warp; ++w) eb += red[w];
    for (uint32_t i0 = c0; i0 < c1; i0 += 32) {
      const uint32_t i = i0 + lane;
      const bool valid = i < c1;
      const uint32_t u = valid ? ckp[i] : 0u;
      const bool gt = valid && u > Tx, eq = valid && u == Tx;
      const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
      const uint32_t lt = (1u << lane) - 1u;
      const uint32_t g = gb + __popc(bg & lt), e = eb + __popc(be & lt);
      if (gt) R.out[g + (e < need ? e : need)] = static_cast<int32_t>(m.ci[i]);
      else if (eq && e < need) R.out[g + e] = static_cast<int32_t>(m.ci[i]);
      gb += __popc(bg);
      eb += __popc(be);
    }
    return;
  }
  finish_row(m, n_cand, exact, d1, want, R.keep, by_score, R.out, red, info);
}


// cluster launch of topk_cluster_kernel<NB, CL>: one cluster of CL CTAs per row
template <int NB, int CL>
cudaError_t launch_cluster_rows(const TopkArgs& a, int ccap, size_t csmem, cudaStream_t st) {
  auto kern = topk_cluster_kernel<NB, CL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(csmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(a.n_rows) * CL, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = csmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_off() ? 1 : 2;
  // rows one resident wave of clusters ahead are prefetched into L2 (clusters per SM pair
  // from the occupancy of one CTA; cluster placement only lowers the real count)
  TopkArgs b = a;
  b.prefetch_ahead = 0;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ==
                                                cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, csmem) == cudaSuccess)
    b.prefetch_ahead = sms * per_sm / CL;
  e = cudaLaunchKernelEx(&cfg, kern, b, ccap);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// one translation unit per cluster shape (they compile in parallel)
cudaError_t launch_topk_cluster_8_4(const TopkArgs& a, int ccap, size_t csmem, cudaStream_t st);
cudaError_t launch_topk_cluster_16_4(const TopkArgs& a, int ccap, size_t csmem, cudaStream_t st);
cudaError_t launch_topk_cluster_16_8(const TopkArgs& a, int ccap, size_t csmem, cudaStream_t st);

}  // namespace dsa
