// Kernel variants for k <= 2048, ragged output (row indices).
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k2048_ragged(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_cluster<2048, false>(p, G, dev, stream);
}
}  // namespace tki
