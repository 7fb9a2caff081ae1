// Kernel variants for k <= 2048, ragged output (row indices).
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k2048_ragged(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_cluster<2048, false>(p, G, dev, stream);
}
int clusters_k2048_ragged(int G, int dev) { return max_active_clusters<2048, false>(G, dev); }
}  // namespace tki
