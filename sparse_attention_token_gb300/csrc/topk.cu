// topk.cu -- per-row top-k: single-CTA kernels and the launch dispatcher.
#include "topk_kernels.cuh"

namespace dsa {

cudaError_t launch_topk(const TopkArgs& a, int max_row_len, cudaStream_t st) {
  if (a.n_rows <= 0) return cudaSuccess;
  int keep_cap = a.k_out < a.topk_limit ? a.k_out : a.topk_limit;
  if (keep_cap > max_row_len) keep_cap = max_row_len;
  if (keep_cap < 1) keep_cap = 1;
  // room for the kept keys plus a threshold bucket of up to max(512, keep/4) keys
  int cap = keep_cap + (keep_cap / 4 > 512 ? keep_cap / 4 : 512);
  const int max_cap = kWarps * 32 * kMaxRounds;
  if (cap > max_cap) cap = max_cap;
  if (cap < keep_cap) return cudaErrorInvalidValue;
  cap = (cap + 31) & ~31;
  const size_t smem = (static_cast<size_t>(kHistWords) + 4 * static_cast<size_t>(cap)) * 4;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 0;
  auto go = [&](auto kern, int spec_cap) -> cudaError_t {
    const size_t ksmem = smem + static_cast<size_t>(spec_cap) * 8;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ksmem));
    if (e != cudaSuccess) return e;
    TopkArgs b = a;
    b.prefetch_ahead = 0;
    b.spec_cap = spec_cap;
    int per_sm = 0;
    // the rows one wave ahead go to L2 only while they and the wave being read take a
    // small part of it (a streamed row may be read three times from L2)
    if (sms > 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, ksmem) == cudaSuccess &&
        static_cast<long long>(sms) * per_sm * max_row_len * 4 <= (32LL << 20))
      b.prefetch_ahead = sms * per_sm;
    e = launch_pdl(kern, dim3(static_cast<unsigned>(a.n_rows)), dim3(kThreads), ksmem, st, b, cap);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  };
  // rows longer than one CTA's registers hold, but within a cluster's: one cluster per row
  // long rows: room for the kept keys plus a wide threshold bucket, so the second
  // histogram level (a cluster-wide pass and merge) is rarely needed
  const int ccap = max_cap;
  const size_t csmem = (static_cast<size_t>(kHistWords) + 4 * static_cast<size_t>(ccap)) * 4 +
                       static_cast<size_t>(kHistWords) * 4;  // + merged histogram
  // streamed rows in score order: room for 2.25 times the kept keys (at least 4096) for the
  // one-pass selection (the sample aims halfway between keep and that), within 200 KB of
  // shared memory per CTA
  int spec_cap = 0;
  if (a.order == 0) {
    long long sc = 9LL * keep_cap / 4;
    if (sc < 4096) sc = 4096;
    const long long room = ((200LL << 10) - static_cast<long long>(smem)) / 8;
    if (sc > room) sc = room;
    sc &= ~31LL;
    if (sc >= 2LL * keep_cap) spec_cap = static_cast<int>(sc);
  }
  if (max_row_len <= kWarps * 8 * 128) return go(topk_kernel<8>, 0);
  // many long rows: one CTA per row reading its row from memory (in score order once, the
  // selection running on the keys above a threshold taken from a sample) keeps every SM
  // busy with several rows; a cluster's rows wait on exchanges between its CTAs
  if (sms > 0 && a.n_rows > sms / 2) return go(topk_kernel<0>, spec_cap);
  // few long rows: a cluster per row, 4 CTAs of 8192 or 16384 keys up to 65536 keys (few
  // CTAs, few merge partners), then 8 of 16384
  if (max_row_len <= 4 * kWarps * 8 * 128) return launch_topk_cluster_8_4(a, ccap, csmem, st);
  if (max_row_len <= 4 * kWarps * 16 * 128) return launch_topk_cluster_16_4(a, ccap, csmem, st);
  if (max_row_len <= 8 * kWarps * 16 * 128) return launch_topk_cluster_16_8(a, ccap, csmem, st);
  return go(topk_kernel<0>, spec_cap);
}

}  // namespace dsa
