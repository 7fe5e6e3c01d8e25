// topk_cluster_16x8.cu -- the cluster top-k for clusters of 8 CTAs of up to 16384 keys.
#include "topk_kernels.cuh"

namespace dsa {
cudaError_t launch_topk_cluster_16_8(const TopkArgs& a, int ccap, size_t csmem, cudaStream_t st) {
  return launch_cluster_rows<16, 8>(a, ccap, csmem, st);
}
}  // namespace dsa
