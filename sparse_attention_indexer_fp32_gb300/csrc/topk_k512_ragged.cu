// Kernel variants for k <= 512, ragged output (row indices).
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k512_ragged(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_cluster<512, false>(p, G, dev, stream);
}
int clusters_k512_ragged(int G, int dev) { return max_active_clusters<512, false>(G, dev); }
}  // namespace tki
