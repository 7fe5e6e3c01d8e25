// host_pipe.cu -- dsa_indexer_dense_host: scores + top-k of one sequence whose inputs
// and outputs live in host memory, with the transfers overlapped with the kernels.
//
// The query rows are cut into chunks, handled last rows first.  A library-owned copy
// stream brings the keys, the head weights (and scales), then each chunk's q rows into
// device memory; the caller's
// stream scores each chunk as soon as its rows have landed (dsa_indexer_scores with the
// chunk's query positions, keys up to the chunk's last position) and selects its top-k
// rows (dsa_indexer_topk), every other chunk on a library-owned second compute stream so
// that consecutive chunks' kernels overlap; another library-owned stream copies each
// chunk's top-k rows back to the host as soon as they are ready.  Copies in both directions then run under
// the kernels of other chunks.  Events order the three streams; the caller's stream
// finally waits for the last copy, so synchronising it covers everything.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <mutex>
#include <vector>

#include "dsa_indexer.h"
#include "internal.h"

namespace {

constexpr int kMaxChunks = 256;

struct CopyStreams {
  std::mutex m;
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp = nullptr;
  cudaEvent_t start = nullptr, keys = nullptr, done = nullptr;
  cudaEvent_t in[kMaxChunks] = {}, out[kMaxChunks] = {};
};

CopyStreams& streams_for(int dev) {
  static CopyStreams per_dev[64];
  return per_dev[dev & 63];
}

bool init(CopyStreams& c) {
  if (c.ready) return true;
  if (cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) != cudaSuccess) return false;
  if (cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) != cudaSuccess) return false;
  if (cudaStreamCreateWithFlags(&c.comp, cudaStreamNonBlocking) != cudaSuccess) return false;
  const unsigned f = cudaEventDisableTiming;
  if (cudaEventCreateWithFlags(&c.start, f) != cudaSuccess || cudaEventCreateWithFlags(&c.keys, f) != cudaSuccess ||
      cudaEventCreateWithFlags(&c.done, f) != cudaSuccess)
    return false;
  for (int i = 0; i < kMaxChunks; ++i)
    if (cudaEventCreateWithFlags(&c.in[i], f) != cudaSuccess || cudaEventCreateWithFlags(&c.out[i], f) != cudaSuccess)
      return false;
  c.ready = true;
  return true;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct Layout {
  size_t q, qs, w, k, ks, scores, topk, total;
  long long ld;
  int chunk, n_chunks;
};

bool plan(int T, int S, int H, int D, int q_dtype, int k_out, int chunk_rows, Layout* L) {
  if (T <= 0 || S <= 0 || H <= 0 || D <= 0 || k_out <= 0) return false;
  const int esz = q_dtype == DSA_FP8_E4M3 ? 1 : 2;
  int chunk = chunk_rows > 0 ? chunk_rows : std::max(512, (T + 15) / 16);
  chunk = std::min(chunk, T);
  chunk = std::max(chunk, (T + kMaxChunks - 1) / kMaxChunks);
  L->chunk = chunk;
  L->n_chunks = (T + chunk - 1) / chunk;
  L->ld = (static_cast<long long>(S) + 3) & ~3LL;
  size_t off = 0;
  L->q = off;      off = align256(off + static_cast<size_t>(T) * H * D * esz);
  L->qs = off;     off = align256(off + (esz == 1 ? static_cast<size_t>(T) * H * 4 : 0));
  L->w = off;      off = align256(off + static_cast<size_t>(T) * H * 4);
  L->k = off;      off = align256(off + static_cast<size_t>(S) * D * esz);
  L->ks = off;     off = align256(off + (esz == 1 ? static_cast<size_t>(S) * 4 : 0));
  L->scores = off; off = align256(off + 2 * static_cast<size_t>(chunk) * L->ld * 4);
  L->topk = off;   off = align256(off + static_cast<size_t>(T) * k_out * 4);
  L->total = off;
  return true;
}

dsa_status cuda_ok(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

}  // namespace

extern "C" {

dsa_status dsa_indexer_dense_host_workspace_size(int T, int S, int H, int D, int q_dtype, int k_out, int chunk_rows,
                                                 size_t* bytes) {
  if (!bytes) return DSA_ERR_INVALID_ARGUMENT;
  Layout L;
  if (!plan(T, S, H, D, q_dtype, k_out, chunk_rows, &L)) return DSA_ERR_INVALID_ARGUMENT;
  *bytes = L.total;
  return DSA_OK;
}

dsa_status dsa_indexer_dense_host(const void* q_host, int q_dtype, const float* q_scale_host, const void* k_host,
                                  int k_dtype, const float* k_scale_host, const float* w_host, int T, int S, int H,
                                  int D, int q_pos0, int topk_limit, int k_out, int order, int chunk_rows,
                                  int32_t* topk_host, void* workspace, size_t workspace_bytes,
                                  dsa_stream_t stream) {
  if (T < 0 || S < 0 || q_pos0 < 0 || H <= 0 || D <= 0 || topk_limit < 1 || k_out < 1 || chunk_rows < 0)
    return DSA_ERR_INVALID_ARGUMENT;
  if (order != DSA_ORDER_SCORE && order != DSA_ORDER_INDEX) return DSA_ERR_INVALID_ARGUMENT;
  if (k_out > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (q_dtype != k_dtype || (q_dtype != DSA_BF16 && q_dtype != DSA_FP8_E4M3)) return DSA_ERR_UNSUPPORTED;
  const bool fp8 = q_dtype == DSA_FP8_E4M3;
  if (T == 0) return DSA_OK;
  if (!q_host || !k_host || !w_host || !topk_host || (fp8 && (!q_scale_host || !k_scale_host)))
    return DSA_ERR_INVALID_ARGUMENT;
  if (S == 0) return DSA_ERR_UNSUPPORTED;  // every row would be padding only; use dsa_indexer_topk
  Layout L;
  if (!plan(T, S, H, D, q_dtype, k_out, chunk_rows, &L)) return DSA_ERR_INVALID_ARGUMENT;
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return DSA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  CopyStreams& c = streams_for(dev);
  std::lock_guard<std::mutex> lock(c.m);
  if (!init(c)) return DSA_ERR_CUDA;

  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int esz = fp8 ? 1 : 2;
  const size_t q_row = static_cast<size_t>(H) * D * esz;  // bytes of one query row (all heads)
  uint8_t* q_d = ws + L.q;
  float* qs_d = reinterpret_cast<float*>(ws + L.qs);
  float* w_d = reinterpret_cast<float*>(ws + L.w);
  uint8_t* k_d = ws + L.k;
  float* ks_d = reinterpret_cast<float*>(ws + L.ks);
  int32_t* topk_d = reinterpret_cast<int32_t*>(ws + L.topk);
  // the workspace may still be in use by earlier work on the caller's stream
  dsa_status r;
  if ((r = cuda_ok(cudaEventRecord(c.start, st))) != DSA_OK) return r;
  if ((r = cuda_ok(cudaStreamWaitEvent(c.h2d, c.start, 0))) != DSA_OK) return r;
  if ((r = cuda_ok(cudaStreamWaitEvent(c.d2h, c.start, 0))) != DSA_OK) return r;
  if ((r = cuda_ok(cudaStreamWaitEvent(c.comp, c.start, 0))) != DSA_OK) return r;
  // keys, weights and scales first, then the query rows chunk by chunk
  const size_t k_bytes = static_cast<size_t>(S) * D * esz;
  if ((r = cuda_ok(cudaMemcpyAsync(k_d, k_host, k_bytes, cudaMemcpyHostToDevice, c.h2d))) != DSA_OK) return r;
  if (fp8 && (r = cuda_ok(cudaMemcpyAsync(ks_d, k_scale_host, static_cast<size_t>(S) * 4, cudaMemcpyHostToDevice,
                                          c.h2d))) != DSA_OK)
    return r;
  if ((r = cuda_ok(cudaMemcpyAsync(w_d, w_host, static_cast<size_t>(T) * H * 4, cudaMemcpyHostToDevice, c.h2d))) !=
      DSA_OK)
    return r;
  if (fp8 && (r = cuda_ok(cudaMemcpyAsync(qs_d, q_scale_host, static_cast<size_t>(T) * H * 4,
                                          cudaMemcpyHostToDevice, c.h2d))) != DSA_OK)
    return r;
  // chunks run last rows first: under a causal mask the last rows see the most keys, so
  // the largest kernels start early and run under the remaining copies
  for (int j = 0; j < L.n_chunks; ++j) {
    const int ci = L.n_chunks - 1 - j;
    const int t0 = ci * L.chunk, t1 = std::min(T, t0 + L.chunk);
    const uint8_t* src = static_cast<const uint8_t*>(q_host) + static_cast<size_t>(t0) * q_row;
    if ((r = cuda_ok(cudaMemcpyAsync(q_d + static_cast<size_t>(t0) * q_row, src, static_cast<size_t>(t1 - t0) * q_row,
                                     cudaMemcpyHostToDevice, c.h2d))) != DSA_OK)
      return r;
    if ((r = cuda_ok(cudaEventRecord(c.in[ci], c.h2d))) != DSA_OK) return r;
  }
  // per chunk: score and select, alternating between the caller's stream and a second
  // compute stream so that one chunk's kernels fill the SMs another chunk's tail leaves
  // idle; then copy the chunk's rows back
  // plain launches here: a programmatic dependent grid waiting on one compute stream
  // would hold SM space that the other stream's chunk is meant to fill
  dsa::PdlOffScope no_pdl;
  for (int j = 0; j < L.n_chunks; ++j) {
    const cudaStream_t cs = (j & 1) ? c.comp : st;
    const dsa_stream_t cs_h = reinterpret_cast<dsa_stream_t>(cs);
    const int ci = L.n_chunks - 1 - j;
    const int t0 = ci * L.chunk, t1 = std::min(T, t0 + L.chunk), tc = t1 - t0;
    const int pos0 = q_pos0 + t0;
    const int s_c = static_cast<int>(std::min<long long>(S, static_cast<long long>(q_pos0) + t1));  // visible keys
    float* sc = reinterpret_cast<float*>(ws + L.scores) + static_cast<size_t>(j & 1) * L.chunk * L.ld;
    int32_t* tk = topk_d + static_cast<size_t>(t0) * k_out;
    if ((r = cuda_ok(cudaStreamWaitEvent(cs, c.in[ci], 0))) != DSA_OK) return r;
    if (s_c > 0) {
      r = dsa_indexer_scores(q_d + static_cast<size_t>(t0) * q_row, q_dtype,
                             fp8 ? qs_d + static_cast<size_t>(t0) * H : nullptr, k_d, k_dtype, fp8 ? ks_d : nullptr,
                             w_d + static_cast<size_t>(t0) * H, tc, s_c, H, D, pos0, sc, L.ld, cs_h);
      if (r != DSA_OK) return r;
    }
    r = dsa_indexer_topk(sc, L.ld, tc, s_c, pos0, topk_limit, k_out, order, tk, cs_h);
    if (r != DSA_OK) return r;
    if ((r = cuda_ok(cudaEventRecord(c.out[ci], cs))) != DSA_OK) return r;
    if ((r = cuda_ok(cudaStreamWaitEvent(c.d2h, c.out[ci], 0))) != DSA_OK) return r;
    if ((r = cuda_ok(cudaMemcpyAsync(topk_host + static_cast<size_t>(t0) * k_out, tk,
                                     static_cast<size_t>(tc) * k_out * 4, cudaMemcpyDeviceToHost, c.d2h))) != DSA_OK)
      return r;
  }
  if ((r = cuda_ok(cudaEventRecord(c.done, c.d2h))) != DSA_OK) return r;
  return cuda_ok(cudaStreamWaitEvent(st, c.done, 0));
}

}  // extern "C"
