// Kernel variants for k <= 512.
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k512(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_bucket<512>(p, G, dev, stream);
}
}  // namespace tki
