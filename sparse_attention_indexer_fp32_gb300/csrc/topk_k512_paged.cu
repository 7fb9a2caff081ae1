// Kernel variants for k <= 512, paged output (indices mapped through the page table).
#include "topk_launch.cuh"

namespace tki {
topk_status launch_k512_paged(const Params& p, int G, int dev, cudaStream_t stream) {
  return launch_cluster<512, true>(p, G, dev, stream);
}
}  // namespace tki
