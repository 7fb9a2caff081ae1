// Kernel variants for k <= 1024.
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k1024(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_bucket<1024>(p, G, dev, stream);
}
}  // namespace tki
