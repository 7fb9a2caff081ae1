// Short-row kernel variants for k <= 512 (FP32 and BF16 scores, ragged and paged).
#include "topk_launch.cuh"

namespace tki {
topk_status launch_short_k512(const ShortParams& p, bool bf16, int dev, int sms, cudaStream_t stream) {
  return launch_short_bucket<512>(p, bf16, dev, sms, stream);
}
}  // namespace tki
