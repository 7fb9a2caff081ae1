// Kernel variants for k <= 1024, ragged output (row indices).
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k1024_ragged(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_cluster<1024, false>(p, G, dev, stream);
}
int clusters_k1024_ragged(int G, int dev) { return max_active_clusters<1024, false>(G, dev); }
}  // namespace tki
