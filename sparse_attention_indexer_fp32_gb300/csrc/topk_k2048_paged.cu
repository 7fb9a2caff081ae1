// Kernel variants for k <= 2048, paged output (indices mapped through the page table).
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k2048_paged(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_cluster<2048, true>(p, G, dev, stream);
}
int clusters_k2048_paged(int G, int dev) { return max_active_clusters<2048, true>(G, dev); }
}  // namespace tki
