// Kernel variants for k <= 1024, ragged output (row indices).
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k1024_ragged(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_cluster<1024, false>(p, G, dev, stream);
}
}  // namespace tki
