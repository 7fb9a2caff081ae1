// Kernel variants for k <= 512, paged output (indices mapped through the page table).
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k512_paged(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_cluster<512, true>(p, G, dev, stream);
}
int clusters_k512_paged(int G, int dev) { return max_active_clusters<512, true>(G, dev); }
}  // namespace tki
