// The two-level indexer's helpers on either side of the selection (sglang PR
// 39648 report, 实现拆解 2 table, and the `amax8_varlen` /
// `sort_candidate_blocks` docstrings of candidate_table.py):
//
//  * topk_amax8_varlen: level-one keys, the maximum of every block of 8
//    consecutive scores (+0 above -0), the newest block forced to +inf. A pure stream:
//    each thread reads two blocks (2 x 32 bytes), consecutive threads
//    consecutive blocks, and writes their maxima.
//  * topk_sort_candidate_blocks: the selected block ids of a row rewritten
//    ascending, with their pool slots. One CTA per row sets one bit per
//    selected id in a shared-memory bitmap, then every thread owns a run of
//    bitmap words: a block prefix of their bit counts gives each thread its
//    output positions, and it writes its ids in ascending order (a counting
//    sort, deterministic, no comparison).
#include <cuda_runtime.h>

#include <cstdint>

#include "topk_indexer.h"
#include "topk_kernel.cuh"

namespace tki {

constexpr int kAmaxBlocksPerCta = 2 * kThreads;
constexpr int kMaxBlockWords = 4096;  // bitmap: up to 131072 blocks (rows of 1,048,576 scores)

struct AmaxParams {
  const float* scores;
  int64_t stride;
  const int32_t* lengths;
  int32_t B;
  int32_t topk;
  float* out;
  int64_t out_stride;
  int32_t chunks;  // CTAs per row
};

// Block keys are maxima in the selection's own total order (+0 above -0), so
// the key of a block does not depend on the order of its scores; fmaxf,
// which the page names, leaves the sign of a zero maximum open. The maximum
// is taken over the order-preserving keys and turned back into the float.
__device__ __forceinline__ float key_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

__device__ __forceinline__ uint32_t max_key4(float4 a) {
  return max(max(order_key(a.x), order_key(a.y)), max(order_key(a.z), order_key(a.w)));
}

__global__ void __launch_bounds__(kThreads) amax8_kernel(const AmaxParams p) {
  const int row = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.chunks));
  const int chunk = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.chunks));
  const int64_t len_raw = p.lengths[row];
  const int64_t n = len_raw < 0 ? 0 : (len_raw > p.stride ? p.stride : len_raw);
  const int64_t nb = (n + 7) / 8;
  if (nb == 0 || (p.topk > 0 && nb <= p.topk)) return;  // every block is selected anyway
  const float* rp = p.scores + static_cast<int64_t>(row) * p.stride;
  float* op = p.out + static_cast<int64_t>(row) * p.out_stride;
  const bool vec = (reinterpret_cast<uintptr_t>(rp) & 31u) == 0 && (p.stride & 7) == 0;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int64_t i = static_cast<int64_t>(chunk) * kAmaxBlocksPerCta + u * kThreads + threadIdx.x;
    if (i >= nb) break;
    float m;
    if (i == nb - 1) {
      m = __int_as_float(0x7f800000);  // the newest block: +inf
    } else if (vec) {
      const float4 a = __ldcs(reinterpret_cast<const float4*>(rp + 8 * i));
      const float4 b = __ldcs(reinterpret_cast<const float4*>(rp + 8 * i) + 1);
      m = key_float(max(max_key4(a), max_key4(b)));
    } else {
      uint32_t km = order_key(__ldcs(rp + 8 * i));
#pragma unroll
      for (int j = 1; j < 8; ++j) km = max(km, order_key(__ldcs(rp + 8 * i + j)));
      m = key_float(km);
    }
    op[i] = m;
  }
}

struct SortParams {
  int32_t* blocks;  // [B, k], rewritten in place
  int32_t B;
  int32_t k;
  const int32_t* lengths;
  int64_t stride;
  const int32_t* page_table;
  int64_t pt_stride;
  int32_t bpp;  // blocks per page (page_size / 8, a power of two)
  int32_t* out_pages;
};

__global__ void __launch_bounds__(kThreads) sort_blocks_kernel(const SortParams p) {
  __shared__ uint32_t bm[kMaxBlockWords];
  __shared__ uint32_t tab[kWarps];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int row = static_cast<int>(blockIdx.x);
  const int64_t len_raw = p.lengths[row];
  const int64_t n = len_raw < 0 ? 0 : (len_raw > p.stride ? p.stride : len_raw);
  const int nb = static_cast<int>((n + 7) / 8);
  int32_t* ids = p.blocks + static_cast<int64_t>(row) * p.k;
  int32_t* pages = p.out_pages + static_cast<int64_t>(row) * p.k;
  const int32_t* pt_row = p.page_table + static_cast<int64_t>(row) * p.pt_stride;
  const uint32_t bpp = static_cast<uint32_t>(p.bpp);
  auto slot = [&](uint32_t id) -> int32_t {
    const uint32_t page = id / bpp;
    return static_cast<int32_t>(static_cast<int64_t>(pt_row[page]) * bpp + (id - page * bpp));
  };

  if (nb <= p.k) {  // every block is selected: the identity table, the input is not read
    for (int j = t; j < p.k; j += kThreads) {
      ids[j] = j < nb ? j : INT32_MAX;
      pages[j] = j < nb ? slot(static_cast<uint32_t>(j)) : INT32_MAX;
    }
    return;
  }
  const int words = (nb + 31) / 32;
  for (int q = t; q < words; q += kThreads) bm[q] = 0u;
  __syncthreads();
  for (int j = t; j < p.k; j += kThreads) {
    const int32_t id = ids[j];
    if (id >= 0 && id < nb) atomicOr(&bm[id >> 5], 1u << (id & 31));
  }
  __syncthreads();
  // Thread t owns words [t * wpt, (t + 1) * wpt): their bits, ascending, are
  // the ids this thread writes, after the ids of the lower threads.
  const int wpt = (words + kThreads - 1) / kThreads;
  const int q0 = min(t * wpt, words), q1 = min(q0 + wpt, words);
  uint32_t cnt = 0;
  for (int q = q0; q < q1; ++q) cnt += __popc(bm[q]);
  const uint32_t incl = warp_incl_scan(cnt);
  if (lane == 31) tab[w] = incl;
  __syncthreads();
  const uint32_t e = lane < kWarps ? tab[lane] : 0u;
  uint32_t pos = __reduce_add_sync(0xffffffffu, lane < w ? e : 0u) + incl - cnt;
  const uint32_t total = __reduce_add_sync(0xffffffffu, e);
  for (int q = q0; q < q1; ++q) {
    uint32_t bits = bm[q];
    while (bits != 0u) {
      const uint32_t id = 32u * q + (__ffs(bits) - 1);
      bits &= bits - 1u;
      if (pos < static_cast<uint32_t>(p.k)) {
        ids[pos] = static_cast<int32_t>(id);
        pages[pos] = slot(id);
      }
      ++pos;
    }
  }
  for (int j = static_cast<int>(total) + t; j < p.k; j += kThreads) {
    ids[j] = INT32_MAX;
    pages[j] = INT32_MAX;
  }
}

}  // namespace tki

namespace {

bool aligned4(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; }

topk_status device_ok() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ECUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return TOPK_ECUDA;
  return (major == 10 && minor == 3) ? TOPK_OK : TOPK_EDEVICE;
}

}  // namespace

extern "C" {

topk_status topk_amax8_varlen(const float* scores, int64_t stride, const int32_t* lengths,
                              int32_t B, int32_t topk, float* out, int64_t out_stride,
                              topk_stream_t stream) {
  if (B < 0 || stride < 1 || stride > INT32_MAX || topk < 0) return TOPK_EINVAL;
  if (out_stride < (stride + 7) / 8) return TOPK_EINVAL;
  if (B == 0) return TOPK_OK;
  if (scores == nullptr || lengths == nullptr || out == nullptr) return TOPK_EINVAL;
  if (!aligned4(scores) || !aligned4(lengths) || !aligned4(out)) return TOPK_EINVAL;
  const topk_status st = device_ok();
  if (st != TOPK_OK) return st;
  const int64_t width = (stride + 7) / 8;
  const int64_t chunks = (width + tki::kAmaxBlocksPerCta - 1) / tki::kAmaxBlocksPerCta;
  if (static_cast<int64_t>(B) * chunks > INT32_MAX) return TOPK_EINVAL;
  tki::AmaxParams p = {scores, stride, lengths, B, topk, out, out_stride, static_cast<int32_t>(chunks)};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B * chunks), 1, 1);
  cfg.blockDim = dim3(tki::kThreads, 1, 1);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  return cudaLaunchKernelEx(&cfg, tki::amax8_kernel, p) == cudaSuccess ? TOPK_OK : TOPK_ECUDA;
}

topk_status topk_sort_candidate_blocks(int32_t* blocks, int32_t B, int32_t k,
                                       const int32_t* lengths, int64_t stride,
                                       const int32_t* page_table, int64_t pt_stride,
                                       int32_t page_size, int32_t* out_pages,
                                       topk_stream_t stream) {
  if (B < 0 || k < 1 || stride < 1) return TOPK_EINVAL;
  if ((stride + 7) / 8 > 32LL * tki::kMaxBlockWords) return TOPK_EINVAL;
  if (page_size < 8 || (page_size & (page_size - 1)) != 0) return TOPK_EINVAL;
  const int64_t bpp = page_size / 8;
  if (pt_stride < ((stride + 7) / 8 + bpp - 1) / bpp) return TOPK_EINVAL;
  if (B == 0) return TOPK_OK;
  if (blocks == nullptr || lengths == nullptr || page_table == nullptr || out_pages == nullptr)
    return TOPK_EINVAL;
  if (!aligned4(blocks) || !aligned4(lengths) || !aligned4(page_table) || !aligned4(out_pages))
    return TOPK_EINVAL;
  const topk_status st = device_ok();
  if (st != TOPK_OK) return st;
  tki::SortParams p = {blocks, B, k, lengths, stride, page_table, pt_stride,
                       static_cast<int32_t>(bpp), out_pages};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B), 1, 1);
  cfg.blockDim = dim3(tki::kThreads, 1, 1);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  return cudaLaunchKernelEx(&cfg, tki::sort_blocks_kernel, p) == cudaSuccess ? TOPK_OK : TOPK_ECUDA;
}

}  // extern "C"
