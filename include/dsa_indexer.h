/*
 * dsa_indexer.h -- C ABI of the GB300 (sm_103a) DSA indexer library.
 *
 * The DeepSeek-Sparse-Attention indexer that GLM5's glm_moe_dsa layers run
 * scores every causal query/key pair and keeps each query's best keys
 * (GLM5 TensorCast adaptation design, section "DSA Indexer 融合语义算子";
 * cost buckets 6-10 of section "性能模型设计"):
 *
 *     x[t,h,s]   = sq[t,h] * sk[s] * sum_d q[t,h,d] * k[s,d]      (sq = sk = 1 for bf16)
 *     score[t,s] = sum_h w[t,h] * max(x[t,h,s], 0)                 for keys s <= pos(t)
 *     topk[t,:]  = the min(topk_limit, pos(t)+1) keys of highest score, ties to the
 *                  lower key index, then -1 up to k_out
 *
 * and GLM-5.2 IndexShare (same page, section "GLM-5.2 IndexShare"): a layer
 * typed "shared" runs no indexer and forwards the top-k of the nearest earlier
 * "full" layer unchanged.
 *
 * Conventions for every entry point:
 *  - Pointers named q, k, k_cache, w, scales, scores, topk, cu_q_lens,
 *    seq_lens, block_tables and workspace are DEVICE pointers, owned by the
 *    caller; the library keeps none of them after returning and allocates no
 *    device memory per call.  Held for the process lifetime once first used on a
 *    device: the fixed scratch array of dsa_indexer_static, the streams and events
 *    of dsa_indexer_dense_host, and the streams and events of dsa_indexer_prepare.
 *    Pointers named
 *    types / src / full_args / topk_out are host.
 *  - All work is enqueued on `stream` (NULL = legacy default stream) and is
 *    asynchronous; nothing synchronises except dsa_check_device_status.
 *  - Host-side validation happens before any launch; a failing call launches
 *    nothing and returns the status.
 *  - Device-side checks (a page id outside [0, num_pages), a key position that
 *    the block table does not cover, a bounded wait that gave up) never trap:
 *    the kernel records a bit in a library-owned device status word and skips
 *    the access; dsa_check_device_status reports and clears it.
 *  - Tensors are dense row-major with the strides implied by their shapes
 *    (only scores takes an explicit leading dimension).
 *  - Every device pointer must be 16-byte aligned; row pitches of q/k
 *    (D * element size) are then multiples of 16 bytes for the supported D.
 */
#ifndef DSA_INDEXER_H
#define DSA_INDEXER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* the same handle as cudaStream_t */

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, bad indexer_types, ... */
    DSA_ERR_UNSUPPORTED = 2,      /* valid but not implemented: D, H, dtype mix, k_out */
    DSA_ERR_CUDA = 3,             /* a CUDA runtime/driver call or launch failed */
    DSA_ERR_DEVICE_CHECK = 4,     /* a kernel found a bad page id / uncovered key */
    DSA_ERR_TIMEOUT = 5,          /* a bounded device wait gave up */
    DSA_ERR_WORKSPACE = 6         /* workspace missing or smaller than required */
} dsa_status;

typedef enum { DSA_BF16 = 0, DSA_FP8_E4M3 = 1 } dsa_dtype;

typedef enum { DSA_LAYER_FULL = 0, DSA_LAYER_SHARED = 1 } dsa_layer_type;

/* Output order of a top-k row.  Both are unique for a given score row.
 *  DSA_ORDER_SCORE: by (score desc, key index asc) -- torch.topk's sorted order with
 *                   deterministic ties (GLM5 LoRA blog, section 1, on tie order).
 *  DSA_ORDER_INDEX: the same set of keys in ascending key index.             */
typedef enum { DSA_ORDER_SCORE = 0, DSA_ORDER_INDEX = 1 } dsa_topk_order;

/* Largest k_out / topk_limit the top-k kernels accept. */
#define DSA_MAX_TOPK 4096

/* Human-readable name of a status code (static storage; never NULL). */
const char* dsa_status_string(int status);

/* Library version string (static storage). */
const char* dsa_version(void);

/* Width of a top-k row: min(topk_limit, active_seq_len), never negative
 * (GLM5 TensorCast adaptation design, "DSA Indexer 融合语义算子": the op returns
 * (batch, seq_len, min(topk_limit, active_seq_len))). */
int dsa_topk_width(int topk_limit, int64_t active_seq_len);

/*
 * dsa_indexer_scores -- dense scoring of one sequence (cost buckets 6 and 7:
 * q-k index score MMA; head weight multiply, head reduce, FP8 relu / q-scale /
 * k-scale shaping).
 *
 *   q        [T, H, D]  q_dtype        query rows, query t at position q_pos0 + t
 *   q_scale  [T, H]     fp32 > 0       FP8 q only (NULL for bf16 q)
 *   k        [S, D]     k_dtype        keys 0..S-1
 *   k_scale  [S]        fp32 > 0       FP8 k only (NULL for bf16 k)
 *   w        [T, H]     fp32           per-head weights (any sign)
 *   scores   [T, ld_scores] fp32       out: scores[t, s] for s <= min(q_pos0 + t, S - 1);
 *                                      entries with s > q_pos0 + t are NOT written
 *
 * Supported: (q_dtype, k_dtype) in {(BF16, BF16), (FP8, FP8)}; D in {64, 128} for
 * bf16, D = 128 for FP8; H in {4, 8, 16, 32, 64, 128}; ld_scores >= S and a
 * multiple of 4; q_pos0 >= 0.  T == 0 or S == 0 is a no-op.
 * Inputs must be finite; scales must be finite and > 0 (the library applies the
 * q scale to w and the k scale after the head sum, which commutes with ReLU
 * only for positive scales).
 */
dsa_status dsa_indexer_scores(const void* q, int q_dtype, const float* q_scale,
                              const void* k, int k_dtype, const float* k_scale,
                              const float* w, int T, int S, int H, int D, int q_pos0,
                              float* scores, int64_t ld_scores, dsa_stream_t stream);

/*
 * dsa_indexer_topk -- per-row top-k of dense scores (cost bucket 8, top-k selection).
 *
 *   scores [T, ld_scores] fp32   row t has n_t = max(0, min(q_pos0 + t + 1, S)) visible
 *                                entries scores[t, 0..n_t-1]; nothing else is read
 *   topk   [T, k_out] int32      out: min(topk_limit, n_t) key indices, then -1
 *
 * topk_limit >= 1, 1 <= k_out <= DSA_MAX_TOPK, topk_limit <= DSA_MAX_TOPK unless
 * no row is longer than DSA_MAX_TOPK; order is a dsa_topk_order.  Ties between equal
 * scores go to the lower key index; -0.0 and +0.0 are equal.  NaN scores are
 * outside the contract.  Needs no workspace.
 */
dsa_status dsa_indexer_topk(const float* scores, int64_t ld_scores, int T, int S, int q_pos0,
                            int topk_limit, int k_out, int order, int32_t* topk,
                            dsa_stream_t stream);

/*
 * Fused indexer over a paged key cache for a varlen batch: prefill, chunked
 * prefill and decode (op inputs indexer_cache, block_tables, seq_lens of section
 * "DSA Indexer 融合语义算子"; key and scale cache read bytes, buckets 9 and 10).
 *
 * Sequence b owns query rows cu_q_lens[b] .. cu_q_lens[b+1]-1; its i-th query
 * sits at position pos = seq_lens[b] - q_len_b + i and sees keys 0..pos.  Key s
 * of sequence b is k_cache[block_tables[b * max_pages_per_seq + s / page_size]]
 * [s % page_size].  Returned indices are logical key positions in the sequence.
 */
typedef struct {
    int q_dtype;                 /* dsa_dtype of q                                   */
    int k_dtype;                 /* dsa_dtype of k_cache                             */
    int B;                       /* sequences                                        */
    int total_q;                 /* cu_q_lens[B] (host copy; rows of q, w, topk)     */
    int H, D;                    /* indexer heads, head dim                          */
    int page_size;               /* tokens per page: 16, 32, 64 or 128               */
    int num_pages;               /* pages in k_cache                                 */
    int max_pages_per_seq;       /* columns of block_tables                          */
    int max_seq_len;             /* host upper bound of seq_lens[b]                  */
    const void* q;               /* [total_q, H, D]                                  */
    const float* q_scale;        /* [total_q, H] fp32 (FP8 q) or NULL                */
    const float* w;              /* [total_q, H] fp32                                */
    const int32_t* cu_q_lens;    /* [B + 1], cu_q_lens[0] = 0, non-decreasing        */
    const int32_t* seq_lens;     /* [B], q_len_b <= seq_lens[b] <= max_seq_len       */
    const int32_t* block_tables; /* [B, max_pages_per_seq]                           */
    void* k_cache;               /* [num_pages, page_size, D] (written when k_new)   */
    float* k_scale_cache;        /* [num_pages, page_size] fp32 (FP8 k) or NULL      */
    int topk_limit;              /* index_topk / topk_limit                          */
    int k_out;                   /* columns of topk, >= 1                            */
    int order;                   /* dsa_topk_order                                   */
    int32_t* topk;               /* out [total_q, k_out]                             */
    void* workspace;             /* device scratch, >= dsa_indexer_workspace_size    */
    size_t workspace_bytes;
    const void* k_new;           /* NULL, or [total_q, D] bf16: this step's new keys, */
                                 /* appended to the cache before scoring             */
    const int64_t* slot_mapping; /* [total_q] with k_new: cache slot of each new key */
} dsa_indexer_args;

/* Bytes of device workspace dsa_indexer needs for these sizes (pointers may be NULL). */
dsa_status dsa_indexer_workspace_size(const dsa_indexer_args* args, size_t* bytes);

/* Run the fused indexer.  Same dtype / H / D support as dsa_indexer_scores, plus
 * BF16 q against an FP8-e4m3 cache (GLM5 TensorCast adaptation design, background
 * item 5: the indexer cache takes the FP8 dtype when attention is quantised).  That
 * mix is taken on decode batches (total_q <= B) with D = 128 and k_scale_cache set
 * (q_scale is ignored): each bf16 query row x is first rewritten as s x = hi + lo,
 * two e4m3 rows with a power-of-two scale s (largest |s x| in [128, 256)), exact for
 * every element within ~2^9 of the row's largest |x| and within 2^-17 of that largest
 * value otherwise; the keys then meet both rows in FP8 MMAs whose two halves are added
 * before the ReLU, and w is divided by s.  The two e4m3 NaN codes are not accepted in
 * the cache.  On a prefill batch the mix returns DSA_ERR_UNSUPPORTED.  The workspace
 * (which also holds the rewritten queries) must not be used by another call that
 * overlaps on the GPU. */
dsa_status dsa_indexer(const dsa_indexer_args* args, dsa_stream_t stream);

/*
 * dsa_indexer_cache_append -- write this step's new indexer keys into the paged cache
 * (GLM5 TensorCast adaptation design, "DSA Indexer 融合语义算子": the op's indexer cache
 * is a mutable argument written through slot_mapping; its FP8 path writes the key
 * cache and the scale cache after an activation quantisation, cost buckets 9 and 10).
 *
 *   k_new [n, D] bf16 device rows; slot_mapping [n] int64, slot = page * page_size + row
 *   (negative: skip the token); k_cache [num_pages, page_size, D] of cache_dtype;
 *   k_scale_cache [num_pages, page_size] fp32 (e4m3 cache only).
 *   bf16 cache (D = 64 or 128): the row is copied.  e4m3 cache (D = 128): scale =
 *   amax / 448 (fp32; 1 for an all-zero row), each element the e4m3 value nearest to
 *   k / scale (ties to even, saturating at +-448), the scale stored beside the row.
 * A slot past the cache is skipped and reported through dsa_check_device_status.
 * The same append runs first inside dsa_indexer when dsa_indexer_args.k_new is set.
 */
dsa_status dsa_indexer_cache_append(const void* k_new, int n, int D, const int64_t* slot_mapping,
                                    void* k_cache, int cache_dtype, float* k_scale_cache, int page_size,
                                    int num_pages, dsa_stream_t stream);

/*
 * dsa_indexer_prepare -- the indexer front-end: this step's q, k and head weights from
 * the layer's activations (GLM5 TensorCast adaptation design, "DSA Indexer 融合语义算子":
 * the op's inputs hidden_states, qa_normed, RoPE cos / sin, wq_b, wk, weights_proj,
 * k_norm weight, indexer cache, slot_mapping; performance-model buckets 1-5, 9, 10).
 *
 *   q  = RoPE(qa_normed @ wq_b^T), one row of D per head          [T, H, D]
 *   k  = RoPE(layer_norm(hidden @ wk^T) * k_norm_weight + bias)    [T, D]
 *   w  = hidden @ weights_proj^T                                   [T, H] fp32 -> w_out
 * e4m3 cache: q and k are then rotated by the Walsh-Hadamard transform (Sylvester order,
 * times D^-1/2) and quantised per row: scale = amax / 448 (1 for an all-zero row), codes
 * the e4m3 value nearest to x / scale; q -> q_out (e4m3) and q_scale_out [T, H]; k and
 * its scale -> the cache slot.  bf16 cache: q -> q_out (bf16), k -> the cache slot (bf16).
 * The outputs feed dsa_indexer (q, q_scale, w; the cache now holds this step's keys).
 *
 * Readings (the page gives no formulas): projection weights are [out, in] row-major
 * (x @ W^T); k_norm is a layer norm with the biased variance and eps k_norm_eps, times
 * the weight, plus k_norm_bias when not NULL; RoPE turns pair i of the first rope_dim
 * values -- (i, i + rope_dim/2), or (2i, 2i+1) when rope_interleaved -- by the angle with
 * cosine rope_cos[t, i] and sine rope_sin[t, i]: (a, b) -> (a cos - b sin, a sin + b cos).
 *
 * All pointers are device memory, 16-byte aligned (slot_mapping 8-byte).  hidden
 * [T, hidden_dim] and qa_normed [T, q_rank] bf16; wq_b [H*D, q_rank], wk [D, hidden_dim],
 * weights_proj [H, hidden_dim] bf16; rope_cos / rope_sin [T, rope_dim/2] fp32;
 * k_norm_weight [D] fp32, k_norm_bias [D] fp32 or NULL.  D = 128; H a power of two up to
 * 128; rope_dim even, at most D, a multiple of 8 unless interleaved; hidden_dim and
 * q_rank multiples of 8.  The three projections run on the tensor cores as bf16
 * products with fp32 accumulation, in the library's kernels like everything else; with
 * 512 tokens or more and rope_dim 0, 64 or 128 the q projection finishes its rows
 * (RoPE, rotation, quantisation) in its own epilogue.  workspace:
 * dsa_indexer_prepare_workspace_size bytes of device memory (the fp32 partial sums of
 * the projections that are not finished in their epilogue), not shared with
 * overlapping work.  Slots past the cache are skipped and reported through
 * dsa_check_device_status; negative slots are skipped.
 */
typedef struct {
  int T, hidden_dim, q_rank, H, D, rope_dim, rope_interleaved;
  const void* hidden;
  const void* qa_normed;
  const float* rope_cos;
  const float* rope_sin;
  const void* wq_b;
  const void* wk;
  const void* weights_proj;
  const float* k_norm_weight;
  const float* k_norm_bias;
  float k_norm_eps;
  int cache_dtype;           /* DSA_BF16 or DSA_FP8_E4M3 */
  const int64_t* slot_mapping;
  void* k_cache;             /* [num_pages, page_size, D] */
  float* k_scale_cache;      /* [num_pages, page_size] (e4m3 cache) */
  int page_size, num_pages;
  void* q_out;               /* [T, H, D] bf16 or e4m3 */
  float* q_scale_out;        /* [T, H] (e4m3 cache) */
  float* w_out;              /* [T, H] */
  void* workspace;
  size_t workspace_bytes;
} dsa_indexer_prepare_args;

dsa_status dsa_indexer_prepare_workspace_size(const dsa_indexer_prepare_args* args, size_t* bytes);
dsa_status dsa_indexer_prepare(const dsa_indexer_prepare_args* args, dsa_stream_t stream);

/*
 * dsa_indexer_dense_host -- dsa_indexer_scores + dsa_indexer_topk of one sequence whose
 * inputs and output are in HOST memory, with the transfers overlapped with the kernels.
 * The pages describe the indexer on device tensors; this entry point exists for callers
 * that hold the step's inputs on the host (and is what an end-to-end measurement calls).
 *
 *   q_host [T, H, D], w_host [T, H], k_host [S, D] (+ q_scale_host [T, H], k_scale_host [S]
 *   for e4m3): row-major host arrays, pinned (cudaHostAlloc / cudaHostRegister) for the
 *   copies to overlap; pageable memory works but the copies then serialise.
 *   topk_host [T, k_out]: written with the same rows dsa_indexer_topk returns.
 *   chunk_rows: query rows per chunk (0 = max(512, T/16); raised so there are at most
 *   256 chunks).
 *   workspace: device memory of dsa_indexer_dense_host_workspace_size bytes, 256-byte
 *   aligned, owned by the caller and not shared with overlapping work.
 *
 * The query rows travel in chunks (last rows first) on a library-owned copy stream;
 * each chunk is scored and selected as soon as its rows land, alternately on `stream`
 * and on a library-owned compute stream so consecutive chunks' kernels overlap; another
 * library-owned stream copies the chunk's top-k rows back.  The call returns once everything is enqueued; `stream` waits
 * for the last copy, so synchronising it makes topk_host final.  Same element types, H,
 * D and errors as dsa_indexer_scores / dsa_indexer_topk; S = 0 is DSA_ERR_UNSUPPORTED.
 * Concurrent calls from several host threads on one device are serialised internally.
 */
dsa_status dsa_indexer_dense_host_workspace_size(int T, int S, int H, int D, int q_dtype, int k_out,
                                                 int chunk_rows, size_t* bytes);
dsa_status dsa_indexer_dense_host(const void* q_host, int q_dtype, const float* q_scale_host,
                                  const void* k_host, int k_dtype, const float* k_scale_host,
                                  const float* w_host, int T, int S, int H, int D, int q_pos0,
                                  int topk_limit, int k_out, int order, int chunk_rows,
                                  int32_t* topk_host, void* workspace, size_t workspace_bytes,
                                  dsa_stream_t stream);

/*
 * Key-sharded top-k (GLM5 LoRA blog, section 3.1, 训练侧: context parallelism; a top-k
 * taken per shard of a long sequence matches the full-sequence top-k only 68 % of the
 * time, gathering the shards' indexer results 99.97 %).  The exact form: every shard of
 * keys keeps its best min(k, visible) keys as (score, global index) candidates in
 * (score desc, index asc) order; the caller gathers the candidates of all shards (for
 * shards on several devices, one all-gather of [T, k_cand] indices and scores per
 * shard); dsa_indexer_merge_candidates keeps the best of their union under the same
 * order, which equals the top-k of the whole row.
 *
 * dsa_indexer_shard_candidates -- one shard's candidates.
 *   q, q_scale, w, H, D, dtypes   as dsa_indexer_scores; query t at position q_pos0 + t
 *   k_shard [S, D], k_scale [S]   the shard's keys: global key positions
 *                                 key_offset .. key_offset + S - 1 (query t sees global key
 *                                 g when g <= q_pos0 + t)
 *   k_cand                        candidates per row, 1..DSA_MAX_TOPK (use the top-k width)
 *   cand_idx [T, k_cand] int32    out: global key indices, then -1
 *   cand_scores [T, k_cand] fp32  out: their scores, then -inf
 *   workspace                     16-byte aligned device scratch of at least
 *                                 dsa_indexer_shard_candidates_workspace_size(T, S) bytes
 *                                 (the shard's fp32 score rows), caller-owned
 * q_pos0 >= 0, key_offset >= 0.  Same element types, H, D and errors as
 * dsa_indexer_scores; a missing or small workspace is DSA_ERR_WORKSPACE.
 */
dsa_status dsa_indexer_shard_candidates_workspace_size(int T, int S, size_t* bytes);
dsa_status dsa_indexer_shard_candidates(const void* q, int q_dtype, const float* q_scale, const void* k_shard,
                                        int k_dtype, const float* k_scale, const float* w, int T, int S, int H,
                                        int D, int q_pos0, int key_offset, int k_cand, int32_t* cand_idx,
                                        float* cand_scores, void* workspace, size_t workspace_bytes,
                                        dsa_stream_t stream);

/*
 * dsa_indexer_merge_candidates -- the top-k of the union of n_shards candidate lists.
 *   cand_scores [n_shards, T, k_cand] fp32, cand_idx [n_shards, T, k_cand] int32: list j
 *   of row t holds shard j's candidates as written by dsa_indexer_shard_candidates
 *   (valid entries first, in (score desc, index asc) order, then index -1); the shards'
 *   key ranges must not overlap.
 *   topk [T, k_out] int32 out: min(topk_limit, valid candidates) indices in `order`,
 *   then -1.
 * 1 <= n_shards <= 32, n_shards * k_cand <= 16384, 1 <= k_out <= DSA_MAX_TOPK.  Ties go
 * to the lower key index; -0.0 and +0.0 are equal.
 */
dsa_status dsa_indexer_merge_candidates(const float* cand_scores, const int32_t* cand_idx, int n_shards, int T,
                                        int k_cand, int topk_limit, int k_out, int order, int32_t* topk,
                                        dsa_stream_t stream);

/*
 * Sparse MLA over the indexer's top-k (GLM5 TensorCast adaptation design: the fused
 * indexer hands topk_indices / topk_limit to the multi-head latent attention backend,
 * whose attention length is capped by the top-k width -- "Sparse MLA 配置兼容", the
 * performance model's sparse prefill / decode length).  Absorbed multi-head latent
 * attention on the selected keys only: for query row t of sequence b and head h, over the
 * logical key positions s = topk[t, j] >= 0 (s < seq_lens[b]; others are skipped),
 *     logit = scale * (q_nope[t, h] . c_kv[s] + q_rope[t, h] . k_rope[s])
 *     out[t, h, :] = sum_s softmax_s(logit) * c_kv[s]            (fp32, latent space)
 * with c_kv[s] = cache_c[block_tables[b, s / page_size], s % page_size] and k_rope[s] the
 * same row of cache_r.  An empty selection gives zeros.  The value up-projection and the
 * output projection are the caller's.
 *   q_nope [total_q, H, kv_rank] bf16, q_rope [total_q, H, rope_dim] bf16
 *   cache_c [num_pages, page_size, kv_rank] bf16, cache_r [num_pages, page_size, rope_dim] bf16
 *   topk [total_q, topk_width] int32 (any order, -1 padding); out [total_q, H, kv_rank] fp32
 * kv_rank = 512 and rope_dim = 64; H = 16, 32 or a multiple of 64; scale > 0.  workspace:
 * dsa_sparse_mla_workspace_size bytes (the key splits' partial outputs), 16-byte aligned.
 * A selected position whose page is outside the cache is skipped and reported through
 * dsa_check_device_status.  Probabilities enter the P.V product rounded to bf16.
 */
typedef struct {
  int B, total_q, H, kv_rank, rope_dim, page_size, num_pages, max_pages_per_seq, topk_width;
  float scale;
  const void* q_nope;
  const void* q_rope;
  const void* cache_c;
  const void* cache_r;
  const int32_t* block_tables;
  const int32_t* cu_q_lens;
  const int32_t* seq_lens;
  const int32_t* topk;
  float* out;
  void* workspace;
  size_t workspace_bytes;
} dsa_sparse_mla_args;
dsa_status dsa_sparse_mla_workspace_size(const dsa_sparse_mla_args* args, size_t* bytes);
dsa_status dsa_sparse_mla(const dsa_sparse_mla_args* args, dsa_stream_t stream);

/*
 * dsa_indexer_static -- dsa_indexer for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point; it exists for library users.
 *
 * Some callers cannot hand the library a workspace: plugin hosts that pass only the
 * input and output tensors, and serving loops that reserve nearly all device memory
 * up front and forbid allocation during a step (cudaMalloc / cudaFree may synchronise
 * the device and stall every stream).  This call runs the same kernels as dsa_indexer
 * with their scratch (work-list counters, work items, fp32 score rows) in one
 * library-owned device array of DSA_STATIC_WORKSPACE_BYTES, which every GPU that
 * loads this code holds until the process exits.  args->workspace and
 * args->workspace_bytes are ignored; every other field means what it means for
 * dsa_indexer, and the caller still provides every input and the topk output.
 *  - A problem whose dsa_indexer_workspace_size exceeds DSA_STATIC_WORKSPACE_BYTES
 *    returns DSA_ERR_WORKSPACE before anything is launched (use dsa_indexer with a
 *    caller workspace for it).
 *  - The array is placed on a device when the library's device code is loaded there,
 *    which under CUDA's default lazy module loading can be during the first call into
 *    the library on that device, and the first dsa_indexer_static call on a device
 *    looks up the array's device address with that device current.  So make one call
 *    into the library (this one, or any other) on each device before reserving most of
 *    its memory, and make the first dsa_indexer_static call there before any stream
 *    capture.  A failed lookup returns DSA_ERR_CUDA and is tried again by the next call.
 *  - All calls on a device share the array and it keeps the last call's contents; each
 *    call clears the part that must start at zero (the work-list counters).  Calls that
 *    overlap on the GPU (other streams, other host threads) race on the array: serialise them.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define DSA_STATIC_WORKSPACE_BYTES ((size_t)24 << 20)
dsa_status dsa_indexer_static(const dsa_indexer_args* args, dsa_stream_t stream);

/*
 * IndexShare source resolution (host only, GLM5 TensorCast adaptation design,
 * "GLM-5.2 IndexShare"): src[l] = l for a full layer, the nearest earlier full
 * layer for a shared layer.  types[l] is a dsa_layer_type.  An unknown type or a
 * shared layer with no earlier full layer returns DSA_ERR_INVALID_ARGUMENT and
 * leaves src unspecified.
 */
dsa_status dsa_resolve_indexer_sources(int L, const int32_t* types, int32_t* src);

/*
 * dsa_indexer_stack -- an IndexShare stack of L layers.
 *   full_args[l]  host pointer to the args of full layer l (its own cache, q, w and
 *                 output buffer); NULL for shared layers (they own no cache).
 *   topk_out[l]   host array of L device pointers, written by the call: a full layer's
 *                 entry is full_args[l]->topk, a shared layer's entry is its source
 *                 layer's buffer -- the same memory, forwarded unchanged, no launch.
 *   src_out       host [L] or NULL: the resolved source layers.
 * Every argument is validated before the first launch.
 */
dsa_status dsa_indexer_stack(int L, const int32_t* types, const dsa_indexer_args* const* full_args,
                             int32_t** topk_out, int32_t* src_out, dsa_stream_t stream);

/* Synchronise `stream`, then report and clear the device status word of the current
 * device: DSA_OK, DSA_ERR_DEVICE_CHECK or DSA_ERR_TIMEOUT (or DSA_ERR_CUDA). */
dsa_status dsa_check_device_status(dsa_stream_t stream);

/*
 * Clock sample (diagnostic, not part of the method): n_ctas one-thread blocks each write
 * {SM id, that SM's cycle counter (clock64), the global nanosecond timer} as three
 * uint64 to out[3 * i .. 3 * i + 2].  Two samples on a stream bracket an interval; per SM,
 * (cycles after - cycles before) / (ns after - ns before) is its average clock over it.
 *   out     device [3 * n_ctas] uint64, caller-owned
 *   n_ctas  >= 1 (a few per SM reach every SM)
 * Asynchronous on `stream`; DSA_ERR_INVALID_ARGUMENT for a null out or n_ctas < 1.
 */
dsa_status dsa_clock_sample(uint64_t* out, int n_ctas, dsa_stream_t stream);

/*
 * dsa_test_arm_score_timeout -- failure-path test hook; the pages have no counterpart.
 * Every wait inside the library's kernels is bounded: a wait that runs out records
 * DSA_ERR_TIMEOUT in the device status word and makes the kernel stop, wait (bounded)
 * for its own copies and tensor-core work in flight, free its tensor memory and
 * return, so the device stays usable.  This call arms the next score-kernel launch
 * made by the calling host thread (by any entry point) so that its MMA-issuing thread
 * first waits on an internal barrier that nothing ever completes, for at most
 * limit_ns nanoseconds; that launch then takes the path above and its outputs are
 * unspecified.  The arming is used up by that one launch; limit_ns = 0 disarms.
 * Returns DSA_OK.
 */
dsa_status dsa_test_arm_score_timeout(unsigned long long limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* DSA_INDEXER_H */
