// Kernel variants for k <= 2048.
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k2048(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_bucket<2048>(p, G, dev, stream);
}
}  // namespace tki
