// api.cu -- the C ABI of include/dsa_indexer.h: argument validation, tensor-map
// encoding, work-list construction and kernel launches.
//
// IndexShare (GLM5 TensorCast adaptation design, "GLM-5.2 IndexShare"): full layers
// run the indexer; a shared layer runs nothing and forwards the nearest earlier full
// layer's top-k buffer; a shared layer without an earlier full layer, or an unknown
// type, is rejected before anything is launched.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "dsa_indexer.h"
#include "internal.h"
#include "ptx.cuh"
#include "qsplit.cuh"

namespace dsa {

__device__ unsigned g_device_status;

unsigned* device_status_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
  return static_cast<unsigned*>(p);
}

namespace {

constexpr size_t kMaxSmem = 232448;          // opt-in dynamic shared memory per CTA on sm_100-class parts
// Target bytes of fp32 scores per chunk of query rows (the workspace holds one chunk).
// Large chunks amortise the launch tails of the score and top-k kernels more than they
// lose by the scores leaving L2: chunked prefill of 8192 rows against 65536 keys took
// 9.67 ms with 64 MiB chunks, 9.18 ms with 256 MiB and 8.59 ms with 1 GiB; on later
// kernels 5.70 ms with 1 GiB (two chunks) and 5.65 ms with 2 GiB (one).
constexpr size_t kScoreChunkBudget = 2ull << 30;

// ---------------------------------------------------------------- work list (paged path)
__global__ void prep_items_kernel(const int32_t* cu_q_lens, const int32_t* seq_lens, int NQ, int KC, int R, int cap,
                                  int n_chunks, int max_seq_len, int max_pages_per_seq, int page_size,
                                  int tile_keys, WorkItem* items, int* counts, unsigned* status) {
  const int b = blockIdx.x;
  const int cu0 = cu_q_lens[b], cu1 = cu_q_lens[b + 1];
  const int q_len = cu1 - cu0;
  const int L = seq_lens[b];
  if (q_len <= 0) return;
  if (L > max_seq_len || q_len > L || cu0 < 0 ||
      static_cast<long long>(L) > static_cast<long long>(max_pages_per_seq) * page_size) {
    if (threadIdx.x == 0) atomicOr(status, kStatusUncovered);
    return;
  }
  for (int c = cu0 / R; c <= (cu1 - 1) / R && c < n_chunks; ++c) {
    const int seg0 = max(cu0, c * R), seg1 = min(cu1, (c + 1) * R);
    const int nqb = (seg1 - seg0 + NQ - 1) / NQ;
    for (int j = threadIdx.x; j < nqb; j += blockDim.x) {
      const int row0 = seg0 + j * NQ;
      const int nrows = min(NQ, seg1 - row0);
      const int pos0 = L - q_len + (row0 - cu0);
      const int n_kt = (pos0 + nrows - 1 + tile_keys) / tile_keys;
      const int n_it = KC > 0 ? (n_kt + KC - 1) / KC : 1;
      const int slot = atomicAdd(&counts[c], n_it);
      if (slot + n_it > cap) {
        atomicOr(status, kStatusUncovered);
        continue;
      }
      for (int k = 0; k < n_it; ++k) {
        const int kt0 = KC > 0 ? k * KC : 0;
        const int kt1 = KC > 0 ? min(n_kt, (k + 1) * KC) : n_kt;
        WorkItem w;
        w.row0 = row0;
        w.pos0 = pos0;
        w.kt = kt0 | (kt1 << 16);
        w.bn = b | (nrows << 24);
        items[static_cast<long long>(c) * cap + slot + k] = w;
      }
    }
  }
}

// Exclusive prefix sum of one int per thread over the whole block (blockDim a multiple
// of 32, at most 1024); *total gets the block's sum.  Every thread must call it.
__device__ int block_scan_excl(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int before = warp > 0 ? warp_sums[warp - 1] : 0;
  *total = warp_sums[nw - 1];
  __syncthreads();
  return before + x - v;
}

constexpr int kPrepThreads = 1024;

// Balanced work lists for launches that split long key ranges (few query blocks, e.g.
// decode): the query blocks' key tiles, laid end to end, are cut into one equal share
// (+-1 tile) per CTA of the score grid, and each share into items at query-block
// boundaries.  CTA c's items go to items[c * per_cta ...] and their number to
// cta_counts[c].  One block of kPrepThreads; dynamic shared memory holds q_max query
// blocks (16 bytes each) and q_max + 1 prefix sums.
__device__ __forceinline__ void prep_balanced_body(
    const int32_t* cu_q_lens, const int32_t* seq_lens, int B, int NQ, int G, int per_cta, int q_max,
    int max_seq_len, int max_pages_per_seq, int page_size, int tile_keys, WorkItem* items, int* cta_counts,
    unsigned* status) {
  extern __shared__ int4 blk[];  // row0, pos0, b | nrows << 24, key tiles
  int* pre = reinterpret_cast<int*>(blk + q_max);
  __shared__ int warp_sums[32];
  __shared__ int s_over;
  const int tid = threadIdx.x;
  if (tid == 0) s_over = 0;
  __syncthreads();
  int nq = 0;
  for (int b0 = 0; b0 < B; b0 += blockDim.x) {
    const int b = b0 + tid;
    int nb = 0, cu0 = 0, q_len = 0, L = 0;
    if (b < B) {
      cu0 = cu_q_lens[b];
      q_len = cu_q_lens[b + 1] - cu0;
      L = seq_lens[b];
      if (q_len > 0) {
        if (L > max_seq_len || q_len > L || cu0 < 0 ||
            static_cast<long long>(L) > static_cast<long long>(max_pages_per_seq) * page_size)
          atomicOr(status, kStatusUncovered);
        else
          nb = (q_len + NQ - 1) / NQ;
      }
    }
    int tot;
    const int off = nq + block_scan_excl(nb, warp_sums, &tot);
    for (int j = 0; j < nb; ++j) {
      const int q = off + j;
      if (q >= q_max) {
        s_over = 1;
        break;
      }
      const int row0 = cu0 + j * NQ, nrows = min(NQ, cu0 + q_len - row0);
      const int pos0 = L - q_len + j * NQ;
      blk[q] = make_int4(row0, pos0, b | (nrows << 24), (pos0 + nrows - 1 + tile_keys) / tile_keys);
    }
    nq += tot;
  }
  __syncthreads();
  if (s_over) {
    for (int c = tid; c < G; c += blockDim.x) cta_counts[c] = 0;
    if (tid == 0) atomicOr(status, kStatusUncovered);
    return;
  }
  int carry = 0;
  for (int q0 = 0; q0 < nq; q0 += blockDim.x) {
    const int q = q0 + tid;
    int tot;
    const int off = carry + block_scan_excl(q < nq ? blk[q].w : 0, warp_sums, &tot);
    if (q < nq) pre[q] = off;
    carry += tot;
  }
  if (tid == 0) pre[nq] = carry;
  __syncthreads();
  const long long W = carry;
  for (int c = tid; c < G; c += blockDim.x) {
    const int lo = static_cast<int>(W * c / G), hi = static_cast<int>(W * (c + 1) / G);
    int n = 0;
    if (lo < hi) {
      int l = 0, r = nq - 1;  // first block whose tiles reach past lo
      while (l < r) {
        const int m = (l + r) >> 1;
        if (pre[m + 1] > lo) r = m;
        else l = m + 1;
      }
      for (int j = l; j < nq && pre[j] < hi; ++j) {
        if (n >= per_cta) {
          atomicOr(status, kStatusUncovered);
          break;
        }
        const int4 q = blk[j];
        WorkItem w;
        w.row0 = q.x;
        w.pos0 = q.y;
        w.kt = (max(lo, pre[j]) - pre[j]) | ((min(hi, pre[j + 1]) - pre[j]) << 16);
        w.bn = q.z;
        items[static_cast<long long>(c) * per_cta + n++] = w;
      }
    }
    cta_counts[c] = n;
  }
}

__global__ void __launch_bounds__(kPrepThreads) prep_balanced_kernel(
    const int32_t* cu_q_lens, const int32_t* seq_lens, int B, int NQ, int G, int per_cta, int q_max,
    int max_seq_len, int max_pages_per_seq, int page_size, int tile_keys, WorkItem* items, int* cta_counts,
    unsigned* status) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  prep_balanced_body(cu_q_lens, seq_lens, B, NQ, G, per_cta, q_max, max_seq_len, max_pages_per_seq, page_size,
                     tile_keys, items, cta_counts, status);
}

// Decode against an e4m3 cache needs both the balanced lists and the split query rows;
// neither reads the other's output, so one launch runs both: block 0 builds the lists,
// blocks 1.. split 32 query rows each.
__global__ void __launch_bounds__(kPrepThreads) decode_prep_kernel(
    const int32_t* cu_q_lens, const int32_t* seq_lens, int B, int NQ, int G, int per_cta, int q_max,
    int max_seq_len, int max_pages_per_seq, int page_size, int tile_keys, WorkItem* items, int* cta_counts,
    unsigned* status, const uint2* q, const float* w, long long rows, int H, uint32_t* q8, float* w8) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  if (blockIdx.x == 0) {
    prep_balanced_body(cu_q_lens, seq_lens, B, NQ, G, per_cta, q_max, max_seq_len, max_pages_per_seq, page_size,
                       tile_keys, items, cta_counts, status);
    return;
  }
  const long long r = static_cast<long long>(blockIdx.x - 1) * (kPrepThreads / 32) + (threadIdx.x >> 5);
  if (r < rows) split_row(q, w, r, H, q8, w8, threadIdx.x & 31);
}

// ---------------------------------------------------------------- helpers
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_h(int H) { return H == 4 || H == 8 || H == 16 || H == 32 || H == 64 || H == 128; }

dsa_status check_dtypes(int q_dtype, int k_dtype, int D, bool have_qs, bool have_ks) {
  if ((q_dtype != DSA_BF16 && q_dtype != DSA_FP8_E4M3) || (k_dtype != DSA_BF16 && k_dtype != DSA_FP8_E4M3))
    return DSA_ERR_INVALID_ARGUMENT;
  if (q_dtype != k_dtype) return DSA_ERR_UNSUPPORTED;
  if (q_dtype == DSA_BF16) {
    if (D != 64 && D != 128) return DSA_ERR_UNSUPPORTED;
  } else {
    if (D != 128) return DSA_ERR_UNSUPPORTED;
    if (!have_qs || !have_ks) return DSA_ERR_INVALID_ARGUMENT;
  }
  return DSA_OK;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Row-major [rows, D] operand, 128-byte swizzled boxes of {128 bytes, box_rows}.
bool make_map_2d(CUtensorMap* m, const void* base, bool fp8, int D, long long rows, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Paged cache [num_pages, page_size, D], boxes of {128 bytes, page_size rows, 1 page}.
bool make_map_paged(CUtensorMap* m, const void* base, bool fp8, int D, int page_size, int num_pages) {
  auto enc = encode_fn();
  if (!enc) return false;
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(page_size),
                        static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * esz, static_cast<cuuint64_t>(D) * esz * page_size};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(page_size), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Deepest key-tile ring that fits in shared memory (>= 2), or 0.  Decode tiles (N < 256
// or split queries) have two key producers that own alternate stages: an even ring.
int pick_stages(const ScoreArgs& a) {
  // an even ring depth lets two producer warps alternate tiles (decode tiles, e4m3 tiles)
  const int step = (a.split || a.N != 256 || a.k_fp8) ? 2 : 1;
  for (int s = kMaxKStages - kMaxKStages % step; s >= 2; s -= step)
    if (score_smem_bytes(a, s) <= kMaxSmem) return s;
  return 0;
}

size_t score_launch_smem(const ScoreArgs& a) {
  return std::max<size_t>(score_smem_bytes(a, a.num_k_stages), 120 * 1024);
}

dsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

// One thread per block: {SM id, SM cycle counter, global ns timer} of the block's SM.
__global__ void clock_sample_kernel(uint64_t* out) {
  uint32_t smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  const uint64_t c = clock64();
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  out[3 * blockIdx.x + 0] = smid;
  out[3 * blockIdx.x + 1] = c;
  out[3 * blockIdx.x + 2] = t;
}

struct PagedPlan {
  bool decode, split;
  bool balanced;  // one chunk of split key ranges: per-CTA balanced lists (prep_balanced_kernel)
  int NQ, N, KC, R, n_chunks, cap, tile_keys;
  int G, per_cta, q_max;
  long long ld;
  size_t off_counts, off_items, off_scores, off_q8, off_w8, total;
};

dsa_status plan_paged(const dsa_indexer_args* a, PagedPlan* p) {
  if (!a) return DSA_ERR_INVALID_ARGUMENT;
  if (a->B < 0 || a->total_q < 0 || a->H <= 0 || a->D <= 0 || a->page_size <= 0 || a->num_pages < 0 ||
      a->max_pages_per_seq < 0 || a->max_seq_len < 0 || a->topk_limit < 1 || a->k_out < 1)
    return DSA_ERR_INVALID_ARGUMENT;
  if (a->k_out > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (a->order != DSA_ORDER_SCORE && a->order != DSA_ORDER_INDEX) return DSA_ERR_INVALID_ARGUMENT;
  if (!supported_h(a->H)) return DSA_ERR_UNSUPPORTED;
  if (a->page_size != 16 && a->page_size != 32 && a->page_size != 64 && a->page_size != 128)
    return DSA_ERR_UNSUPPORTED;
  if (static_cast<long long>(a->max_seq_len) > static_cast<long long>(a->max_pages_per_seq) * a->page_size)
    return DSA_ERR_INVALID_ARGUMENT;
  if (a->max_seq_len >= (1 << 16) * kBlockM) return DSA_ERR_UNSUPPORTED;  // key-tile ids are 16-bit
  if (a->max_seq_len > INT_MAX - 2 * kBlockM) return DSA_ERR_UNSUPPORTED;
  p->decode = a->total_q <= a->B;
  p->split = a->q_dtype == DSA_BF16 && a->k_dtype == DSA_FP8_E4M3;
  if (p->split) {
    // bf16 queries against an e4m3 cache (decode shapes): each query row is rewritten as an
    // exact sum of two e4m3 rows and scored by FP8 MMAs
    if (!p->decode || a->D != 128) return DSA_ERR_UNSUPPORTED;
    if (!a->k_scale_cache) return DSA_ERR_INVALID_ARGUMENT;
  } else {
    dsa_status st = check_dtypes(a->q_dtype, a->k_dtype, a->D, a->q_scale != nullptr, a->k_scale_cache != nullptr);
    if (st != DSA_OK) return st;
  }
  const int ns = std::max(num_sms(), 1);
  p->N = p->split ? std::max(64, 2 * a->H) : (p->decode ? std::max(64, a->H) : 256);
  p->NQ = p->split ? 1 : p->N / a->H;
  p->tile_keys = kBlockM;
  p->ld = (std::max(a->max_seq_len, 1) + 3) & ~3LL;
  long long R = static_cast<long long>(kScoreChunkBudget / (static_cast<size_t>(p->ld) * 4));
  R = std::max<long long>(R - R % p->NQ, p->NQ);
  if (R >= a->total_q) R = std::max(a->total_q, 1);
  p->R = static_cast<int>(R);
  p->n_chunks = std::max(1, (a->total_q + p->R - 1) / p->R);
  const long long qb_per_chunk = (p->R + p->NQ - 1) / p->NQ + std::min<long long>(a->B, p->R) + 1;
  p->KC = qb_per_chunk < 2LL * ns ? 16 : 0;
  const long long kt_max = (a->max_seq_len + p->tile_keys - 1) / p->tile_keys;
  const long long per_qb = p->KC > 0 ? (kt_max + p->KC - 1) / p->KC : 1;
  long long cap = qb_per_chunk * std::max<long long>(per_qb, 1);
  p->balanced = p->KC > 0 && p->n_chunks == 1;
  p->G = ns;
  p->q_max = static_cast<int>(qb_per_chunk);
  p->per_cta = p->q_max + 1;  // a CTA's share meets at most every query block
  if (p->balanced) cap = static_cast<long long>(p->G) * p->per_cta;
  if (cap > INT_MAX / 2) return DSA_ERR_UNSUPPORTED;
  p->cap = static_cast<int>(cap);
  size_t off = 0;
  p->off_counts = off;
  off += ((static_cast<size_t>(std::max(p->n_chunks, p->balanced ? p->G : 0)) * 4 + 255) / 256) * 256;
  p->off_items = off;
  off += ((static_cast<size_t>(p->n_chunks) * p->cap * sizeof(WorkItem) + 255) / 256) * 256;
  p->off_scores = off;
  off += static_cast<size_t>(p->R) * static_cast<size_t>(p->ld) * 4;
  off = (off + 255) / 256 * 256;
  p->off_q8 = off;
  if (p->split) off += (static_cast<size_t>(a->total_q) * 2 * a->H * a->D + 255) / 256 * 256;
  p->off_w8 = off;
  if (p->split) off += (static_cast<size_t>(a->total_q) * a->H * 4 + 255) / 256 * 256;
  p->total = off;
  return DSA_OK;
}

dsa_status run_paged(const dsa_indexer_args* a, const PagedPlan& p, cudaStream_t st) {
  if (a->total_q == 0 || a->B == 0) return DSA_OK;
  unsigned* status = device_status_ptr();
  if (!status) return DSA_ERR_CUDA;
  if (a->k_new) {
    // this step's keys go into the cache first, so the step's own queries see them
    const cudaError_t e = launch_cache_append(a->k_new, a->total_q, a->D, a->slot_mapping, a->k_cache,
                                              a->k_dtype == DSA_FP8_E4M3, a->k_scale_cache,
                                              static_cast<long long>(a->num_pages) * a->page_size, status, st);
    if (e != cudaSuccess) return DSA_ERR_CUDA;
  }
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  int* counts = reinterpret_cast<int*>(ws + p.off_counts);
  WorkItem* items = reinterpret_cast<WorkItem*>(ws + p.off_items);
  float* scores = reinterpret_cast<float*>(ws + p.off_scores);
  const bool fp8 = a->q_dtype == DSA_FP8_E4M3;

  ScoreArgs s{};
  s.paged = 1;
  s.q_fp8 = fp8;
  s.k_fp8 = a->k_dtype == DSA_FP8_E4M3;
  s.split = p.split;
  s.H = a->H;
  s.D = a->D;
  s.NQ = p.NQ;
  s.N = p.N;
  s.page_size = a->page_size;
  s.num_pages = a->num_pages;
  s.max_pages_per_seq = a->max_pages_per_seq;
  s.block_tables = a->block_tables;
  s.total_rows = a->total_q;
  s.w = a->w;
  s.q_scale = a->q_scale;
  s.k_scale = a->k_scale_cache;
  s.scores = scores;
  s.ld = p.ld;
  s.status = status;
  s.num_k_stages = pick_stages(s);
  if (s.num_k_stages < 2) return DSA_ERR_UNSUPPORTED;

  CUtensorMap tq, tk;
  void* q8 = ws + p.off_q8;
  float* w8 = reinterpret_cast<float*>(ws + p.off_w8);
  const long long split_rows = static_cast<long long>(a->total_q) * a->H;
  if (p.split) {
    // hi/lo e4m3 rows of every query and the weights divided by the rows' scales (with
    // balanced lists, in the same launch as the lists, below)
    if (!p.balanced && launch_qsplit(a->q, a->w, split_rows, a->H, q8, w8, st) != cudaSuccess) return DSA_ERR_CUDA;
    s.q_fp8 = 1;
    s.w = w8;
    s.q_scale = nullptr;
    s.num_k_stages = pick_stages(s);
    if (s.num_k_stages < 2) return DSA_ERR_UNSUPPORTED;
    if (!make_map_2d(&tq, q8, true, a->D, static_cast<long long>(a->total_q) * 2 * a->H, p.N)) return DSA_ERR_CUDA;
  } else if (!make_map_2d(&tq, a->q, fp8, a->D, static_cast<long long>(a->total_q) * a->H, p.N)) {
    return DSA_ERR_CUDA;
  }
  if (!make_map_paged(&tk, a->k_cache, s.k_fp8 != 0, a->D, a->page_size, std::max(a->num_pages, 1)))
    return DSA_ERR_CUDA;

  cudaError_t e;
  if (p.balanced) {
    const size_t prep_smem = static_cast<size_t>(p.q_max) * 16 + (static_cast<size_t>(p.q_max) + 1) * 4;
    if (p.split) {
      const long long nb = 1 + (split_rows + kPrepThreads / 32 - 1) / (kPrepThreads / 32);
      e = launch_pdl(decode_prep_kernel, dim3(static_cast<unsigned>(nb)), dim3(kPrepThreads), prep_smem, st,
                     a->cu_q_lens, a->seq_lens, a->B, p.NQ, p.G, p.per_cta, p.q_max, a->max_seq_len,
                     a->max_pages_per_seq, a->page_size, p.tile_keys, items, counts, status,
                     static_cast<const uint2*>(a->q), a->w, split_rows, a->H, static_cast<uint32_t*>(q8), w8);
    } else {
      e = launch_pdl(prep_balanced_kernel, dim3(1), dim3(kPrepThreads), prep_smem, st, a->cu_q_lens, a->seq_lens,
                     a->B, p.NQ, p.G, p.per_cta, p.q_max, a->max_seq_len, a->max_pages_per_seq, a->page_size,
                     p.tile_keys, items, counts, status);
    }
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    s.cta_counts = counts;
    s.per_cta = p.per_cta;
  } else {
    if ((e = cudaMemsetAsync(counts, 0, static_cast<size_t>(p.n_chunks) * 4, st)) != cudaSuccess) return DSA_ERR_CUDA;
    prep_items_kernel<<<a->B, 128, 0, st>>>(a->cu_q_lens, a->seq_lens, p.NQ, p.KC, p.R, p.cap, p.n_chunks,
                                            a->max_seq_len, a->max_pages_per_seq, a->page_size, p.tile_keys, items,
                                            counts, status);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return DSA_ERR_CUDA;
  const int ns = std::max(num_sms(), 1);
  const size_t smem = score_launch_smem(s);
  for (int c = 0; c < p.n_chunks; ++c) {
    s.items = items + static_cast<long long>(c) * p.cap;
    s.n_items = counts + c;
    s.items_cap = p.cap;
    s.row_base = c * p.R;
    e = launch_score(s, &tq, &tk, p.balanced ? p.G : ns, smem, st);
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    TopkArgs t{};
    t.scores = scores;
    t.ld = p.ld;
    t.n_rows = std::min(p.R, a->total_q - c * p.R);
    t.paged = 1;
    t.row_base = c * p.R;
    t.B = a->B;
    t.cu_q_lens = a->cu_q_lens;
    t.seq_lens = a->seq_lens;
    t.max_n = p.ld;
    t.topk_limit = a->topk_limit;
    t.k_out = a->k_out;
    t.order = a->order;
    t.topk = a->topk;
    if ((e = launch_topk(t, a->max_seq_len, st)) != cudaSuccess) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

const char* dsa_status_string(int s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARGUMENT: return "DSA_ERR_INVALID_ARGUMENT";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE_CHECK: return "DSA_ERR_DEVICE_CHECK";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    default: return "DSA_ERR_UNKNOWN";
  }
}

const char* dsa_version(void) { return "dsa_indexer sm_103a 0.1"; }

int dsa_topk_width(int topk_limit, int64_t active_seq_len) {
  long long w = std::min<long long>(topk_limit, active_seq_len);
  return w > 0 ? static_cast<int>(w) : 0;
}

dsa_status dsa_indexer_scores(const void* q, int q_dtype, const float* q_scale, const void* k, int k_dtype,
                              const float* k_scale, const float* w, int T, int S, int H, int D, int q_pos0,
                              float* scores, int64_t ld_scores, dsa_stream_t stream) {
  if (q_pos0 < 0) return DSA_ERR_INVALID_ARGUMENT;
  return dense_scores(q, q_dtype, q_scale, k, k_dtype, k_scale, w, T, S, H, D, q_pos0, scores, ld_scores,
                      reinterpret_cast<cudaStream_t>(stream));
}

dsa_status dsa_indexer_topk(const float* scores, int64_t ld_scores, int T, int S, int q_pos0, int topk_limit,
                            int k_out, int order, int32_t* topk, dsa_stream_t stream) {
  if (q_pos0 < 0) return DSA_ERR_INVALID_ARGUMENT;
  return dense_topk(scores, ld_scores, T, S, q_pos0, topk_limit, k_out, order, topk,
                    reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace dsa {

// Dense scoring of T queries (query t at position q_pos0 + t) against keys 0..S-1.  q_pos0
// may be negative: the key-sharded entry points score a shard whose first key sits after
// some queries (those rows see none of its keys).
dsa_status dense_scores(const void* q, int q_dtype, const float* q_scale, const void* k, int k_dtype,
                        const float* k_scale, const float* w, int T, int S, int H, int D, int q_pos0,
                        float* scores, int64_t ld_scores, cudaStream_t stream) {
  if (T < 0 || S < 0 || H <= 0 || D <= 0) return DSA_ERR_INVALID_ARGUMENT;
  if (T == 0 || S == 0) return DSA_OK;
  if (!q || !k || !w || !scores) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(w) || !aligned16(scores) || (q_scale && !aligned16(q_scale)) ||
      (k_scale && !aligned16(k_scale)))
    return DSA_ERR_INVALID_ARGUMENT;
  if (ld_scores < S || (ld_scores & 3) != 0) return DSA_ERR_INVALID_ARGUMENT;
  if (!supported_h(H)) return DSA_ERR_UNSUPPORTED;
  dsa_status st = check_dtypes(q_dtype, k_dtype, D, q_scale != nullptr, k_scale != nullptr);
  if (st != DSA_OK) return st;
  if (static_cast<long long>(T) * H > INT_MAX || static_cast<long long>(q_pos0) + T > INT_MAX)
    return DSA_ERR_UNSUPPORTED;
  if (S >= (1 << 16) * kBlockM) return DSA_ERR_UNSUPPORTED;
  unsigned* status = device_status_ptr();
  if (!status) return DSA_ERR_CUDA;
  const bool fp8 = q_dtype == DSA_FP8_E4M3;

  ScoreArgs a{};
  a.paged = 0;
  a.q_fp8 = fp8;
  a.k_fp8 = fp8;
  a.H = H;
  a.D = D;
  a.N = 256;
  a.NQ = 256 / H;
  a.T = T;
  a.S = S;
  a.q_pos0 = q_pos0;
  a.n_dense_items = (T + a.NQ - 1) / a.NQ;
  a.total_rows = T;
  a.w = w;
  a.q_scale = fp8 ? q_scale : nullptr;
  a.k_scale = fp8 ? k_scale : nullptr;
  a.scores = scores;
  a.ld = ld_scores;
  a.status = status;
  a.num_k_stages = pick_stages(a);
  if (a.num_k_stages < 2) return DSA_ERR_UNSUPPORTED;

  CUtensorMap tq, tk;
  if (!make_map_2d(&tq, q, fp8, D, static_cast<long long>(T) * H, a.N)) return DSA_ERR_CUDA;
  if (!make_map_2d(&tk, k, fp8, D, S, kBlockM)) return DSA_ERR_CUDA;
  const int ns = std::max(num_sms(), 1);
  const int grid = std::min(ns, a.n_dense_items);
  return from_cuda(launch_score(a, &tq, &tk, grid, score_launch_smem(a), stream));
}

// Top-k of dense score rows: row t sees entries 0 .. min(q_pos0 + t, S - 1) (none when
// q_pos0 + t < 0).
dsa_status dense_topk(const float* scores, int64_t ld_scores, int T, int S, int q_pos0, int topk_limit, int k_out,
                      int order, int32_t* topk, cudaStream_t stream) {
  if (T < 0 || S < 0 || topk_limit < 1 || k_out < 1) return DSA_ERR_INVALID_ARGUMENT;
  if (order != DSA_ORDER_SCORE && order != DSA_ORDER_INDEX) return DSA_ERR_INVALID_ARGUMENT;
  if (k_out > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!topk || (S > 0 && !scores)) return DSA_ERR_INVALID_ARGUMENT;
  if (S > 0 && (!aligned16(scores) || ld_scores < S || (ld_scores & 3) != 0)) return DSA_ERR_INVALID_ARGUMENT;
  TopkArgs t{};
  t.scores = scores;
  t.ld = ld_scores;
  t.n_rows = T;
  t.paged = 0;
  t.S = S;
  t.q_pos0 = q_pos0;
  t.max_n = S;
  t.topk_limit = topk_limit;
  t.k_out = k_out;
  t.order = order;
  t.topk = topk;
  const long long longest = std::min<long long>(S, static_cast<long long>(q_pos0) + T);
  return from_cuda(launch_topk(t, static_cast<int>(std::max<long long>(longest, 1)), stream));
}

}  // namespace dsa

extern "C" {

dsa_status dsa_indexer_workspace_size(const dsa_indexer_args* args, size_t* bytes) {
  if (!bytes) return DSA_ERR_INVALID_ARGUMENT;
  PagedPlan p;
  dsa_status st = plan_paged(args, &p);
  if (st != DSA_OK) return st;
  *bytes = p.total;
  return DSA_OK;
}

static dsa_status validate_paged_pointers(const dsa_indexer_args* a, const PagedPlan& p) {
  if (a->total_q == 0 || a->B == 0) return DSA_OK;
  if (!a->q || !a->w || !a->cu_q_lens || !a->seq_lens || !a->block_tables || !a->k_cache || !a->topk)
    return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(a->q) || !aligned16(a->w) || !aligned16(a->k_cache) || (a->q_scale && !aligned16(a->q_scale)) ||
      (a->k_scale_cache && !aligned16(a->k_scale_cache)))
    return DSA_ERR_INVALID_ARGUMENT;
  if (a->num_pages < 1 || a->max_pages_per_seq < 1) return DSA_ERR_INVALID_ARGUMENT;
  if (!a->workspace || a->workspace_bytes < p.total || !aligned16(a->workspace)) return DSA_ERR_WORKSPACE;
  if (a->k_new) {
    // append before scoring: bf16 rows, one slot each; e4m3 caches need their scales
    if (!a->slot_mapping || !aligned16(a->k_new) || (reinterpret_cast<uintptr_t>(a->slot_mapping) & 7u) != 0)
      return DSA_ERR_INVALID_ARGUMENT;
    if (a->k_dtype == DSA_FP8_E4M3 && (a->D != 128 || !a->k_scale_cache)) return DSA_ERR_INVALID_ARGUMENT;
  }
  return DSA_OK;
}

dsa_status dsa_indexer(const dsa_indexer_args* args, dsa_stream_t stream) {
  PagedPlan p;
  dsa_status st = plan_paged(args, &p);
  if (st != DSA_OK) return st;
  if ((st = validate_paged_pointers(args, p)) != DSA_OK) return st;
  return run_paged(args, p, reinterpret_cast<cudaStream_t>(stream));
}

dsa_status dsa_indexer_cache_append(const void* k_new, int n, int D, const int64_t* slot_mapping, void* k_cache,
                                    int cache_dtype, float* k_scale_cache, int page_size, int num_pages,
                                    dsa_stream_t stream) {
  if (n < 0 || D <= 0 || page_size <= 0 || num_pages < 0) return DSA_ERR_INVALID_ARGUMENT;
  if (cache_dtype != DSA_BF16 && cache_dtype != DSA_FP8_E4M3) return DSA_ERR_INVALID_ARGUMENT;
  if (cache_dtype == DSA_BF16 ? (D != 64 && D != 128) : D != 128) return DSA_ERR_UNSUPPORTED;
  if (n == 0) return DSA_OK;
  if (!k_new || !slot_mapping || !k_cache || (cache_dtype == DSA_FP8_E4M3 && !k_scale_cache))
    return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(k_new) || !aligned16(k_cache) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0 ||
      (k_scale_cache && (reinterpret_cast<uintptr_t>(k_scale_cache) & 3u) != 0))
    return DSA_ERR_INVALID_ARGUMENT;
  unsigned* status = device_status_ptr();
  if (!status) return DSA_ERR_CUDA;
  return from_cuda(launch_cache_append(k_new, n, D, slot_mapping, k_cache, cache_dtype == DSA_FP8_E4M3,
                                       k_scale_cache, static_cast<long long>(num_pages) * page_size, status,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
dsa_status plan_prepare(const dsa_indexer_prepare_args* a, PreparePlan* p) {
  if (!a) return DSA_ERR_INVALID_ARGUMENT;
  if (a->T < 0 || a->hidden_dim <= 0 || a->q_rank <= 0 || a->H <= 0 || a->D <= 0 || a->page_size <= 0 ||
      a->num_pages < 0 || a->rope_dim < 0 || a->rope_dim > a->D || (a->rope_dim & 1) || !(a->k_norm_eps >= 0.f))
    return DSA_ERR_INVALID_ARGUMENT;
  if (a->cache_dtype != DSA_BF16 && a->cache_dtype != DSA_FP8_E4M3) return DSA_ERR_INVALID_ARGUMENT;
  if (a->D != 128 || !supported_h(a->H) || (a->hidden_dim & 7) || (a->q_rank & 7)) return DSA_ERR_UNSUPPORTED;
  if (!a->rope_interleaved && (a->rope_dim & 7)) return DSA_ERR_UNSUPPORTED;
  if (static_cast<long long>(a->T) * a->H > INT_MAX) return DSA_ERR_UNSUPPORTED;
  *p = plan_prepare_launch(a->T, a->hidden_dim, a->q_rank, a->H, a->D, a->rope_dim);
  return DSA_OK;
}
}  // namespace

dsa_status dsa_indexer_prepare_workspace_size(const dsa_indexer_prepare_args* a, size_t* bytes) {
  if (!bytes) return DSA_ERR_INVALID_ARGUMENT;
  PreparePlan p;
  const dsa_status st = plan_prepare(a, &p);
  if (st != DSA_OK) return st;
  *bytes = p.total;
  return DSA_OK;
}

dsa_status dsa_indexer_prepare(const dsa_indexer_prepare_args* a, dsa_stream_t stream) {
  PreparePlan p;
  dsa_status st = plan_prepare(a, &p);
  if (st != DSA_OK) return st;
  if (a->T == 0) return DSA_OK;
  const bool fp8 = a->cache_dtype == DSA_FP8_E4M3;
  if (!a->hidden || !a->qa_normed || !a->wq_b || !a->wk || !a->weights_proj || !a->k_norm_weight ||
      !a->slot_mapping || !a->k_cache || !a->q_out || !a->w_out ||
      (a->rope_dim > 0 && (!a->rope_cos || !a->rope_sin)) || (fp8 && (!a->k_scale_cache || !a->q_scale_out)))
    return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(a->hidden) || !aligned16(a->qa_normed) || !aligned16(a->wq_b) || !aligned16(a->wk) ||
      !aligned16(a->weights_proj) || !aligned16(a->k_norm_weight) || (a->k_norm_bias && !aligned16(a->k_norm_bias)) ||
      (a->rope_cos && !aligned16(a->rope_cos)) || (a->rope_sin && !aligned16(a->rope_sin)) ||
      !aligned16(a->k_cache) || (a->k_scale_cache && (reinterpret_cast<uintptr_t>(a->k_scale_cache) & 3u) != 0) ||
      !aligned16(a->q_out) || (a->q_scale_out && (reinterpret_cast<uintptr_t>(a->q_scale_out) & 3u) != 0) ||
      !aligned16(a->w_out) || (reinterpret_cast<uintptr_t>(a->slot_mapping) & 7u) != 0)
    return DSA_ERR_INVALID_ARGUMENT;
  if (!a->workspace || a->workspace_bytes < p.total || !aligned16(a->workspace)) return DSA_ERR_WORKSPACE;
  unsigned* status = device_status_ptr();
  if (!status) return DSA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  PrepareLaunch L{};
  L.T = a->T;
  L.hidden_dim = a->hidden_dim;
  L.q_rank = a->q_rank;
  L.H = a->H;
  L.D = a->D;
  L.rope_dim = a->rope_dim;
  L.interleaved = a->rope_interleaved != 0;
  L.fp8 = fp8;
  L.hidden = a->hidden;
  L.qa_normed = a->qa_normed;
  L.wq_b = a->wq_b;
  L.wk = a->wk;
  L.weights_proj = a->weights_proj;
  L.cosb = a->rope_cos;
  L.sinb = a->rope_sin;
  L.ln_w = a->k_norm_weight;
  L.ln_b = a->k_norm_bias;
  L.eps = a->k_norm_eps;
  L.slots = a->slot_mapping;
  L.cache = a->k_cache;
  L.scale_cache = a->k_scale_cache;
  L.n_slots = static_cast<long long>(a->num_pages) * a->page_size;
  L.q_out = a->q_out;
  L.q_scale = a->q_scale_out;
  L.w_out = a->w_out;
  L.Qf = reinterpret_cast<float*>(ws + p.off_q);
  L.Kf = reinterpret_cast<float*>(ws + p.off_k);
  L.Wp = reinterpret_cast<float*>(ws + p.off_w);
  L.status = status;
  L.plan = p;
  return from_cuda(launch_prepare(L, reinterpret_cast<cudaStream_t>(stream)));
}

dsa_status dsa_resolve_indexer_sources(int L, const int32_t* types, int32_t* src) {
  if (L < 0 || (L > 0 && (!types || !src))) return DSA_ERR_INVALID_ARGUMENT;
  int last_full = -1;
  for (int l = 0; l < L; ++l) {
    if (types[l] == DSA_LAYER_FULL) {
      last_full = l;
      src[l] = l;
    } else if (types[l] == DSA_LAYER_SHARED) {
      if (last_full < 0) return DSA_ERR_INVALID_ARGUMENT;
      src[l] = last_full;
    } else {
      return DSA_ERR_INVALID_ARGUMENT;
    }
  }
  return DSA_OK;
}

dsa_status dsa_indexer_stack(int L, const int32_t* types, const dsa_indexer_args* const* full_args,
                             int32_t** topk_out, int32_t* src_out, dsa_stream_t stream) {
  if (L < 0 || (L > 0 && (!types || !full_args || !topk_out))) return DSA_ERR_INVALID_ARGUMENT;
  int32_t* src = static_cast<int32_t*>(std::malloc(sizeof(int32_t) * static_cast<size_t>(std::max(L, 1))));
  if (!src) return DSA_ERR_INVALID_ARGUMENT;
  dsa_status st = dsa_resolve_indexer_sources(L, types, src);
  // validate every full layer before the first launch
  for (int l = 0; st == DSA_OK && l < L; ++l) {
    if (src[l] == l) {
      if (!full_args[l]) { st = DSA_ERR_INVALID_ARGUMENT; break; }
      PagedPlan p;
      st = plan_paged(full_args[l], &p);
      if (st == DSA_OK) st = validate_paged_pointers(full_args[l], p);
    } else if (full_args[l] != nullptr) {
      st = DSA_ERR_INVALID_ARGUMENT;  // a shared layer owns no indexer inputs or cache
    }
  }
  for (int l = 0; st == DSA_OK && l < L; ++l) {
    if (src[l] == l) {
      st = dsa_indexer(full_args[l], stream);
      topk_out[l] = full_args[l]->topk;
    } else {
      topk_out[l] = topk_out[src[l]];
    }
  }
  if (st == DSA_OK && src_out)
    for (int l = 0; l < L; ++l) src_out[l] = src[l];
  std::free(src);
  return st;
}

dsa_status dsa_test_arm_score_timeout(unsigned long long limit_ns) {
  armed_probe_wait_ns() = limit_ns;
  return DSA_OK;
}

dsa_status dsa_clock_sample(uint64_t* out, int n_ctas, dsa_stream_t stream) {
  if (!out || n_ctas < 1) return DSA_ERR_INVALID_ARGUMENT;
  clock_sample_kernel<<<n_ctas, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(out);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status dsa_check_device_status(dsa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return DSA_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return DSA_ERR_CUDA;
  if (v == 0) return DSA_OK;
  if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess) return DSA_ERR_CUDA;
  if (v & (kStatusSmemAlign | kStatusTmemAlloc)) return DSA_ERR_CUDA;
  if (v & kStatusTimeout) return DSA_ERR_TIMEOUT;
  return DSA_ERR_DEVICE_CHECK;
}

}  // extern "C"
