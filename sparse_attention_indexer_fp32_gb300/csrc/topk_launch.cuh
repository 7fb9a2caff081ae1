// Launch of one kernel variant (k bucket x cluster size). Each k bucket is
// instantiated in its own translation unit so the variants compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "topk_indexer.h"
#include "topk_kernel.cuh"
#include "topk_short.cuh"
#include "topk_short_bf16.cuh"

namespace tki {

// Per variant, bit d set once the kernel's shared-memory attribute is set on device d.
template <int KMAX, int G, bool PAGED>
std::atomic<uint64_t>& attr_flags() {
  static std::atomic<uint64_t> flags{0};
  return flags;
}

// Sets the variant's kernel attributes on device `dev` (current), once:
// its shared memory, and for clusters of 16 the non-portable cluster size.
template <int KMAX, int G, bool PAGED>
topk_status prepare_variant(int dev) {
  constexpr int C = StashCap<KMAX>::value;
  auto kernel = topk_rows_kernel<KMAX, G, PAGED>;
  const uint64_t bit = 1ull << dev;
  std::atomic<uint64_t>& flags = attr_flags<KMAX, G, PAGED>();
  if ((flags.load(std::memory_order_acquire) & bit) == 0) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(Smem<C, RingStages<KMAX>::value>))) != cudaSuccess)
      return TOPK_ECUDA;
    if (G > 8 && cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                     cudaSuccess)
      return TOPK_ECUDA;
    flags.fetch_or(bit, std::memory_order_acq_rel);
  }
  return TOPK_OK;
}

// Clusters of G CTAs of this variant that can be resident at once on device
// `dev`, as the CUDA driver answers it (cudaOccupancyMaxActiveClusters): a
// cluster's CTAs must share one GPC, so this can fall short of the SM count
// times the CTAs per SM, divided by G. Found once per device; 0 when none fit
// or the query fails.
template <int KMAX, int G, bool PAGED>
int max_active_clusters_variant(int dev) {
  static std::atomic<int> known[64];  // answer + 1; 0 = not asked yet
  const int seen = known[dev].load(std::memory_order_relaxed);
  if (seen > 0) return seen - 1;
  int n = 0;
  if (prepare_variant<KMAX, G, PAGED>(dev) == TOPK_OK) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(Smem<StashCap<KMAX>::value, RingStages<KMAX>::value>);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, topk_rows_kernel<KMAX, G, PAGED>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();  // the query's failure is not a launch error
      n = 0;
    }
  }
  known[dev].store(n + 1, std::memory_order_relaxed);
  return n;
}

template <int KMAX, int G, bool PAGED>
topk_status launch_variant(const Params& p, int dev, cudaStream_t stream) {
  constexpr int C = StashCap<KMAX>::value;
  auto kernel = topk_rows_kernel<KMAX, G, PAGED>;
  const size_t smem = sizeof(Smem<C, RingStages<KMAX>::value>);
  const topk_status prep = prepare_variant<KMAX, G, PAGED>(dev);
  if (prep != TOPK_OK) return prep;
  cudaLaunchConfig_t cfg = {};
  // G CTAs per row, or one per row plus one more per split row.
  const unsigned grid = G > 1 ? static_cast<unsigned>(p.B) * G
                              : static_cast<unsigned>(p.B) + static_cast<unsigned>(p.B - p.split_first);
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (G > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, p) == cudaSuccess ? TOPK_OK : TOPK_ECUDA;
}

template <int KMAX, bool PAGED>
topk_status launch_cluster(const Params& p, int G, int dev, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_variant<KMAX, 1, PAGED>(p, dev, stream);
    case 2: return launch_variant<KMAX, 2, PAGED>(p, dev, stream);
    case 4: return launch_variant<KMAX, 4, PAGED>(p, dev, stream);
    case 8: return launch_variant<KMAX, 8, PAGED>(p, dev, stream);
    case 16: return launch_variant<KMAX, 16, PAGED>(p, dev, stream);
    default: return TOPK_EINVAL;
  }
}

template <int KMAX, bool PAGED>
int max_active_clusters(int G, int dev) {
  switch (G) {
    case 2: return max_active_clusters_variant<KMAX, 2, PAGED>(dev);
    case 4: return max_active_clusters_variant<KMAX, 4, PAGED>(dev);
    case 8: return max_active_clusters_variant<KMAX, 8, PAGED>(dev);
    case 16: return max_active_clusters_variant<KMAX, 16, PAGED>(dev);
    default: return 0;
  }
}


// Launches one short-row kernel (one CTA per row) with its dynamic shared
// memory; `resident` caches, per device, the CTAs an SM holds at once
// (found once, after the kernel's shared-memory attribute is set).
inline topk_status launch_short_grid(void (*kern)(ShortParams), size_t smem, std::atomic<int>* resident,
                                     const ShortParams& p_in, int dev, int sm_count, cudaStream_t stream) {
  int per_sm = resident[dev].load(std::memory_order_acquire);
  if (per_sm == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return TOPK_ECUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess)
      return TOPK_ECUDA;
    resident[dev].store(per_sm, std::memory_order_release);
  }
  ShortParams p = p_in;
  p.ahead = per_sm * sm_count;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? TOPK_OK : TOPK_ECUDA;
}

// FP32 short-row kernel variant (E scores per thread).
template <int E, int KMAX, bool PAGED>
topk_status launch_short_variant(const ShortParams& p, int dev, int sm_count, cudaStream_t stream) {
  static std::atomic<int> resident[64];
  return launch_short_grid(topk_short_kernel<E, KMAX, PAGED>, sizeof(ShortSmem<ShortCap<KMAX>::value>), resident,
                           p, dev, sm_count, stream);
}

// BF16 short-row kernel variant (E scores per thread).
template <int E, int KMAX, bool PAGED>
topk_status launch_short_bf16_variant(const ShortParams& p, int dev, int sm_count, cudaStream_t stream) {
  static std::atomic<int> resident[64];
  return launch_short_grid(topk_short_bf16_kernel<E, KMAX, PAGED>, sizeof(ShortSmemBf16<ShortCap<KMAX>::value>),
                           resident, p, dev, sm_count, stream);
}

// Rows of at most 8192 scores take E = 32, longer ones (up to 16384) E = 64.
template <int KMAX>
topk_status launch_short_bucket(const ShortParams& p, bool bf16, int dev, int sms, cudaStream_t stream) {
  const bool paged = p.page_table != nullptr;
  const bool narrow = p.stride <= 32 * kThreads;
  if (bf16) {
    if (narrow)
      return paged ? launch_short_bf16_variant<32, KMAX, true>(p, dev, sms, stream)
                   : launch_short_bf16_variant<32, KMAX, false>(p, dev, sms, stream);
    return paged ? launch_short_bf16_variant<64, KMAX, true>(p, dev, sms, stream)
                 : launch_short_bf16_variant<64, KMAX, false>(p, dev, sms, stream);
  }
  if (narrow)
    return paged ? launch_short_variant<32, KMAX, true>(p, dev, sms, stream)
                 : launch_short_variant<32, KMAX, false>(p, dev, sms, stream);
  return paged ? launch_short_variant<64, KMAX, true>(p, dev, sms, stream)
               : launch_short_variant<64, KMAX, false>(p, dev, sms, stream);
}

// Defined in topk_short_k{512,1024,2048}.cu.
topk_status launch_short_k512(const ShortParams& p, bool bf16, int dev, int sms, cudaStream_t stream);
topk_status launch_short_k1024(const ShortParams& p, bool bf16, int dev, int sms, cudaStream_t stream);
topk_status launch_short_k2048(const ShortParams& p, bool bf16, int dev, int sms, cudaStream_t stream);

// Defined in topk_k{512,1024,2048}_{ragged,paged}.cu, one translation unit
// each so that they compile in parallel.
topk_status launch_k512_ragged(const Params& p, int G, int dev, cudaStream_t stream);
topk_status launch_k512_paged(const Params& p, int G, int dev, cudaStream_t stream);
topk_status launch_k1024_ragged(const Params& p, int G, int dev, cudaStream_t stream);
topk_status launch_k1024_paged(const Params& p, int G, int dev, cudaStream_t stream);
topk_status launch_k2048_ragged(const Params& p, int G, int dev, cudaStream_t stream);
topk_status launch_k2048_paged(const Params& p, int G, int dev, cudaStream_t stream);
// Resident clusters of G CTAs (see max_active_clusters_variant), same units.
int clusters_k512_ragged(int G, int dev);
int clusters_k512_paged(int G, int dev);
int clusters_k1024_ragged(int G, int dev);
int clusters_k1024_paged(int G, int dev);
int clusters_k2048_ragged(int G, int dev);
int clusters_k2048_paged(int G, int dev);

}  // namespace tki
