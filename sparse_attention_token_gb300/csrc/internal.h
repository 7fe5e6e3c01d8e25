// internal.h -- declarations shared by the translation units of the library.
// Nothing here is part of the public C ABI (include/dsa_indexer.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include "dsa_indexer.h"

namespace dsa {

// Bits of the device status word (library-owned __device__ variable).
enum : unsigned {
  kStatusBadPage = 1u,       // a block-table entry outside [0, num_pages)
  kStatusUncovered = 2u,     // a key position the block table does not cover / bad lengths
  kStatusTimeout = 4u,       // a bounded mbarrier wait gave up
  kStatusSmemAlign = 8u,     // dynamic shared memory not 1024-byte aligned
  kStatusTmemAlloc = 16u,    // TMEM allocation returned an unusable address
};

constexpr int kBlockM = 128;             // keys per MMA tile (TMEM lanes)
constexpr int kScoreThreads = 320;       // warp 0 TMA, warp 1 MMA/TMEM, warps 2..9 epilogue
constexpr int kMaxKStages = 12;
constexpr int kTmemCols = 512;           // two accumulators at column 0 and 256
constexpr int kMaxN = 256;               // MMA N (queries x heads per tile)

// One unit of scoring work: NQ (or fewer) consecutive query rows of one
// sequence against key tiles [kt0, kt1).
struct WorkItem {
  int row0;      // first query row (global row of q / w / topk)
  int pos0;      // position of row0 in its sequence
  int kt;        // kt0 | kt1 << 16
  int bn;        // b | nrows << 24
};

struct ScoreArgs {
  int paged;          // 0: dense k[S, D]; 1: paged k_cache[num_pages, page_size, D]
  int q_fp8, k_fp8;   // element type of q / keys (1 = e4m3, 0 = bf16)
  int split;          // decode, bf16 q with e4m3 keys: q comes as 2H e4m3 rows (hi, lo) per query
  int H, D, NQ, N;    // N = NQ * H
  int num_k_stages;   // key ring depth
  // dense single sequence
  int T, S, q_pos0, n_dense_items;
  // paged varlen
  int page_size, num_pages, max_pages_per_seq;
  const int32_t* block_tables;
  const WorkItem* items;
  const int* n_items;
  int items_cap;      // capacity of the items segment (clamps *n_items)
  // balanced lists (per_cta > 0): CTA c runs items[c * per_cta + i], i < cta_counts[c],
  // instead of the strided walk over n_items
  const int* cta_counts;
  int per_cta;
  int row_base;       // global query row stored in scores row 0
  int total_rows;     // rows of q / w (bounds for cp.async of w and q_scale)
  // common
  const float* w;
  const float* q_scale;   // [rows, H] or null
  const float* k_scale;   // dense [S] / paged [num_pages * page_size] or null
  float* scores;
  long long ld;
  unsigned* status;   // device status word
  // two key producers (warps 0 and 10 take alternate tiles, the ring depth even); else
  // warp 0 alone (set by launch_score)
  int two_producers;
  // failure-path test hook (0 = off): the MMA issuer first waits this many ns on a
  // barrier nothing arrives at, so the kernel takes its timeout-and-drain path
  unsigned long long probe_wait_ns;
};

struct TopkArgs {
  const float* scores;
  long long ld;
  int n_rows;          // rows handled by this launch (one CTA each)
  // dense: row t -> n = clamp(q_pos0 + t + 1, 0, S); output row t
  int paged;
  int S, q_pos0;
  // paged: CTA i handles global row row_base + i
  int row_base, B;
  const int32_t* cu_q_lens;
  const int32_t* seq_lens;
  long long max_n;     // no row reads more than this many entries
  int topk_limit, k_out, order;
  int32_t* topk;
  // single-CTA rows: CTA i prefetches into L2 the row of CTA i + prefetch_ahead (about one
  // wave of resident CTAs later); 0 = no prefetch
  int prefetch_ahead;
  // rows streamed from memory in score order: room (keys) for the one-pass selection's
  // kept keys, in shared memory after the candidate arrays; 0 = three passes over the row
  int spec_cap;
};

// Programmatic dependent launch may be switched off for the calling host thread: the
// host-memory pipeline runs chunks on two streams, and a dependent grid's CTAs waiting
// on one stream would hold SM space the other stream's kernels could use.
inline bool& pdl_off() {
  static thread_local bool off = false;
  return off;
}
struct PdlOffScope {
  bool prev;
  PdlOffScope() : prev(pdl_off()) { pdl_off() = true; }
  ~PdlOffScope() { pdl_off() = prev; }
};

// Launch with programmatic stream serialisation: the kernel may be scheduled while the
// previous kernel on the stream drains, runs its prologue, and waits (grid_dep_wait)
// before it touches global memory that kernel may write.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl_off() ? 0 : 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Failure-path test hook: the next score launch of the calling host thread gets this
// probe_wait_ns (set by dsa_test_arm_score_timeout, consumed by launch_score).
inline unsigned long long& armed_probe_wait_ns() {
  static thread_local unsigned long long ns = 0;
  return ns;
}

// Host launchers (return a cudaError_t).
cudaError_t launch_score(const ScoreArgs& a, const CUtensorMap* tmap_q, const CUtensorMap* tmap_k,
                         int grid, size_t smem_bytes, cudaStream_t st);
size_t score_smem_bytes(const ScoreArgs& a, int num_k_stages);
cudaError_t launch_topk(const TopkArgs& a, int max_row_len, cudaStream_t st);
unsigned* device_status_ptr();  // address of the status word on the current device
// New indexer keys through slot_mapping into the paged cache (bf16 copy or per-token
// e4m3 quantisation with its scale); slots >= n_slots set kStatusBadPage.
cudaError_t launch_cache_append(const void* k_new, int n, int D, const int64_t* slots, void* cache, bool fp8,
                                float* scale_cache, long long n_slots, unsigned* status, cudaStream_t st);
// Front-end projections on the tensor cores (proj_gemm.cu).
int proj_splits(int M, int N, int K);  // K splits of an fp32 projection of these shapes
bool proj_q_fused_supported(int H, int rope_dim);
cudaError_t launch_proj_f32(const void* A, const void* B, int M, int N, int K, int splits, float* C,
                            unsigned* status, cudaStream_t st);
int proj_dual_splits(int M, int K);
cudaError_t launch_proj_dual(const void* A, const void* Bk, const void* Bw, int M, int n2, int K, int splits,
                             float* Kf, float* W, unsigned* status, cudaStream_t st);
cudaError_t launch_proj_q(const void* A, const void* B, int M, int H, int K, const float* cosb, const float* sinb,
                          int rope_dim, bool interleaved, bool fp8, void* q_out, float* q_scale, unsigned* status,
                          cudaStream_t st);
// Workspace of the front-end: fp32 planes of the projections that are not finished in
// their own epilogue (one plane per K split).
struct PreparePlan {
  bool q_fused;
  int q_splits, kw_splits;  // the k and head-weight projections run as one kernel
  size_t off_q, off_k, off_w, total;
};
PreparePlan plan_prepare_launch(int T, int hidden_dim, int q_rank, int H, int D, int rope_dim);
// Indexer front-end (frontend.cu): the projections and the q / k row kernels (RoPE, layer
// norm, Hadamard, quantisation, cache write).
struct PrepareLaunch {
  int T, hidden_dim, q_rank, H, D, rope_dim;
  bool interleaved, fp8;
  const void *hidden, *qa_normed, *wq_b, *wk, *weights_proj;
  const float *cosb, *sinb, *ln_w, *ln_b;
  float eps;
  const int64_t* slots;
  void* cache;
  float* scale_cache;
  long long n_slots;
  void* q_out;
  float *q_scale, *w_out, *Qf, *Kf, *Wp;
  unsigned* status;
  PreparePlan plan;
};
cudaError_t launch_prepare(const PrepareLaunch& p, cudaStream_t st);
// Dense scoring and top-k of one sequence (the bodies of dsa_indexer_scores and
// dsa_indexer_topk, with q_pos0 allowed to be negative: rows before the first key see none).
dsa_status dense_scores(const void* q, int q_dtype, const float* q_scale, const void* k, int k_dtype,
                        const float* k_scale, const float* w, int T, int S, int H, int D, int q_pos0, float* scores,
                        int64_t ld_scores, cudaStream_t stream);
dsa_status dense_topk(const float* scores, int64_t ld_scores, int T, int S, int q_pos0, int topk_limit, int k_out,
               int order, int32_t* topk, cudaStream_t stream);
// bf16 q rows [rows = total_q * H, 128] -> q8 [total_q, 2H, 128] e4m3 (hi rows, then lo
// rows, per query) with a power-of-two scale s per row, and w8 = w / s.
cudaError_t launch_qsplit(const void* q, const float* w, long long rows, int H, void* q8, float* w8,
                          cudaStream_t st);

}  // namespace dsa
