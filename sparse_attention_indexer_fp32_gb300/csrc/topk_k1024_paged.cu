// Kernel variants for k <= 1024, paged output (indices mapped through the page table).
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k1024_paged(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_cluster<1024, true>(p, G, dev, stream);
}
int clusters_k1024_paged(int G, int dev) { return max_active_clusters<1024, true>(G, dev); }
}  // namespace tki
