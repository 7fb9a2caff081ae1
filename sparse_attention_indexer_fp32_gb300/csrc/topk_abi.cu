// C ABI of the sm_103a top-k library: argument checks, path selection and
// kernel launches. See include/topk_indexer.h for the contract.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "topk_indexer.h"
#include "topk_launch.cuh"

namespace {

using tki::Params;

constexpr int kMaxDevices = 64;
// Rows at least this long stream against a sampled cutoff by default (the
// dispatch sweep: from 8192-score rows up the sampled cutoff is faster than
// the full stream, 8.1 against 14.7 us for one 16384-score row; shorter rows
// have no room for the 4096-score sample).
constexpr int kDefaultSampleMinN = 8192;
// FP32 rows of at most this width take the short-row kernel by default (its
// whole range). On the dispatch sweep it is faster than the streaming kernel
// at every width up to 16384 from a few hundred rows on: B = 2048 rows of
// 80-100 % of 16384 at k = 2048, 62 against 78 us; of 8192, 32 against 122 us.
constexpr int64_t kShortAutoWidth = 16384;
// Default margin of the sampled rank, in standard deviations. At 5 a row
// whose sampled cutoff lands above its k-th largest score (and is streamed
// again) is a ~3e-7 event for the B=1024 workloads; 4 was 1.4 % faster on
// the 131072-wide rows but makes such a rescan (a latency spike) a few-percent
// event per call, 6 keeps ~6 % more candidates.
constexpr float kDefaultSampleZ = 5.0f;
// Cluster sizes for batches too small to occupy the GPU with one CTA per
// row, from the dispatch sweep (B = 1, 4, 8, 16, 32 and 64 rows of 65536 to
// 262144 scores, k = 512 / 1024 / 2048):
//  - rows under 65536 scores stay on one CTA each (32768-wide rows: one CTA
//    per row was fastest at every batch);
//  - up to 4 rows: clusters of 16 (one row of 131072 at k = 512: 13.1 us
//    against 14.1 on 8);
//  - up to 8 rows: 8 (8 rows of 262144 at k = 2048: 20.2 us against 24.0 on
//    16, which stop fitting well past a handful of rows);
//  - up to 16 rows: 4, except 8 for k <= 512 from 196608 scores (16 rows of
//    131072 at k = 2048: 19.4 against 22.1 us on 8; of 196608 at k = 512:
//    17.6 on 8 against 19.7 on 4);
//  - up to 32 rows: 4 from 131072 scores (32 rows of 262144 at k = 2048: 26.7
//    against 29.6 us on 8), else one CTA per row;
//  - more rows: 4 while each CTA keeps at least 32768 scores (64 rows of
//    131072: 21.1 against 23.9 us on one CTA; 64 rows of 65536: 19.2 on 4
//    against 15.7 on one).
constexpr int64_t kMinClusterWidth = 65536;
constexpr int64_t kMinClusterSliceWide = 32768;
// Workspace layout: per split row one arrival counter (the first 4 KiB,
// which persist between calls and are zero outside a call), two hand-over
// counts (the next 8 KiB), then per split row and half k keys and k indices.
constexpr int kMaxSplitRows = 1024;
constexpr size_t kWsCounterBytes = 4 * kMaxSplitRows;
constexpr size_t kWsHeaderBytes = kWsCounterBytes + 8 * kMaxSplitRows;
// Resident CTAs per SM (shared memory and the launch bounds fix two).
constexpr int kCtasPerSm = 2;

size_t ws_bytes_for(int32_t k, int64_t split_rows) {
  return kWsHeaderBytes + static_cast<size_t>(split_rows) * 2 * static_cast<size_t>(k) * 8;
}

// Rows to split over two CTAs each (one-CTA rows only, with a workspace),
// from the dispatch sweep. Each half pays a row's fixed costs (sampling, its
// own cutoff, the hand-over; one of them the merge), so a split pays only
// when it puts HBM bandwidth to work that one CTA per row leaves idle:
//  - rows under 131072 scores: none (at 65536 one CTA per row was fastest at
//    every batch);
//  - a batch of at least one full wave of one-CTA rows (B >= slots, two CTAs
//    per SM), rows of at least 196608 scores: the rows of the last partial
//    wave, or the ones that fill its idle slots (the B = 1024 x 262144 line);
//  - a partial wave: every row up to half the slots, then the rows that fill
//    the idle slots, while one CTA per row would leave HBM short (up to ~200
//    rows: 192 rows of 262144, 47.7 against 51.2 us unsplit; 256 rows, 52.1
//    against 51.0 unsplit: none); at 131072 to 196608 scores only for k <=
//    1024 beyond 74 rows (128 rows of 131072 at k = 2048: 29.6 split
//    against 26.5 us unsplit; at k = 512: 23.0 against 23.9).
constexpr int64_t kMinSplitWidth = 131072;
constexpr int64_t kMinTailSplitWidth = 196608;
constexpr int32_t kMaxPartialWaveSplitBatch = 200;
constexpr int32_t kMaxWideKSplitBatch = 74;

int auto_split_rows(int32_t B, int64_t stride, int kmax, int sm_count) {
  const int64_t slots = static_cast<int64_t>(kCtasPerSm) * sm_count;
  if (stride < kMinSplitWidth || slots <= 0) return 0;
  if (B >= slots) {
    if (stride < kMinTailSplitWidth) return 0;
    const int64_t r = B % slots;
    return static_cast<int>(r < slots - r ? r : slots - r);
  }
  if (B > kMaxPartialWaveSplitBatch) return 0;
  if (stride < kMinTailSplitWidth && kmax > 1024 && B > kMaxWideKSplitBatch) return 0;
  return static_cast<int>(B < slots - B ? B : slots - B);
}

struct DeviceInfo {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  bool supported = false;
  int sm_count = 0;
};
DeviceInfo g_devices[kMaxDevices];

// Device of the caller's current context, checked once per device for sm_103.
topk_status device_info(int* dev, DeviceInfo** info) {
  if (cudaGetDevice(dev) != cudaSuccess) return TOPK_ECUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return TOPK_EDEVICE;
  DeviceInfo& d = g_devices[*dev];
  std::call_once(d.once, [&]() {
    int major = 0, minor = 0, sms = 0;
    d.err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev);
    if (d.err == cudaSuccess)
      d.err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev);
    if (d.err == cudaSuccess)
      d.err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, *dev);
    d.sm_count = sms;
    d.supported = (major == 10 && minor == 3);
  });
  if (d.err != cudaSuccess) return TOPK_ECUDA;
  if (!d.supported) return TOPK_EDEVICE;
  *info = &d;
  return TOPK_OK;
}

// Resident clusters of G CTAs for the variant of this k bucket and output.
int max_clusters(int kmax, bool paged, int G, int dev) {
  switch (kmax) {
    case 512: return paged ? tki::clusters_k512_paged(G, dev) : tki::clusters_k512_ragged(G, dev);
    case 1024: return paged ? tki::clusters_k1024_paged(G, dev) : tki::clusters_k1024_ragged(G, dev);
    default: return paged ? tki::clusters_k2048_paged(G, dev) : tki::clusters_k2048_ragged(G, dev);
  }
}

// CTAs per row when the batch is too small to occupy the GPU (the table
// above), shrunk while the clusters of every row would not fit on the GPU at
// once (the CUDA driver's answer for clusters of that size, which must each
// sit in one GPC). Clusters of 2 are never chosen: on the dispatch sweep they
// were never faster than one CTA per row, two split halves, or clusters of 4.
int auto_cluster_size(int32_t B, int64_t stride, int kmax, bool paged, int dev, bool can_split_all) {
  // 41 to 74 rows of 131072 to 196608 scores: every row split in two (when
  // the split policy splits them all and a workspace holds them) beat
  // clusters of 4 (64 rows of 131072 at k = 1024: 21.9 against 24.8 us; at
  // 32 rows clusters of 4 still win).
  if (can_split_all && B > 40 && B <= kMaxWideKSplitBatch && stride >= kMinSplitWidth &&
      stride < 262144)
    return 1;
  int G = 1;
  if (B <= 32 && stride >= kMinClusterWidth) {
    if (B <= 4) {
      G = 16;
    } else if (B <= 8) {
      G = 8;
    } else if (B <= 16) {
      G = (kmax <= 512 && stride >= 196608) ? 8 : 4;
    } else {
      G = stride >= 131072 ? 4 : 1;
    }
  } else if (stride / 4 >= kMinClusterSliceWide) {
    G = 4;
  }
  while (G >= 4) {
    const int fit = max_clusters(kmax, paged, G, dev);
    if (fit > 0 && B <= fit) return G;
    G /= 2;
  }
  return 1;
}

bool aligned4(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; }

// log2 of a power-of-two page size, else -1 (the kernels then divide).
int32_t page_shift_of(int32_t page_size) {
  if (page_size < 1 || (page_size & (page_size - 1)) != 0) return -1;
  int32_t s = 0;
  while ((1 << s) < page_size) ++s;
  return s;
}

// Launches the short-row kernel (rows of at most tki::kShortMaxRow scores,
// FP32 or BF16), one CTA per row.
topk_status launch_short(const void* scores, bool bf16, int64_t stride, const int32_t* lengths,
                         int32_t B, int32_t k, const int32_t* page_table, int64_t pt_stride,
                         int32_t page_size, int32_t* out, const topk_debug_opts* opts,
                         cudaStream_t stream) {
  tki::ShortParams p = {};
  p.scores = scores;
  p.stride = stride;
  p.lengths = lengths;
  p.B = B;
  p.k = k;
  p.out = out;
  p.page_table = page_table;
  p.pt_stride = page_table != nullptr ? pt_stride : 0;
  p.page_size = page_table != nullptr ? page_size : 1;
  p.page_shift = page_shift_of(p.page_size);
  p.sample_mode = opts != nullptr ? opts->sample_mode : 0;
  p.sample_z = (opts != nullptr && opts->sample_z != 0.0f) ? opts->sample_z : kDefaultSampleZ;
  p.counters = opts != nullptr ? opts->counters : nullptr;
  int dev = 0;
  DeviceInfo* info = nullptr;
  const topk_status st = device_info(&dev, &info);
  if (st != TOPK_OK) return st;
  if (k <= 512) return tki::launch_short_k512(p, bf16, dev, info->sm_count, stream);
  if (k <= 1024) return tki::launch_short_k1024(p, bf16, dev, info->sm_count, stream);
  return tki::launch_short_k2048(p, bf16, dev, info->sm_count, stream);
}

// Argument checks of every selection entry point; they read no device state,
// and nothing is enqueued when one fails. TOPK_OK with B == 0 means a no-op.
topk_status check_select_args(const void* scores, bool bf16, int64_t stride, const int32_t* lengths,
                              int32_t B, int32_t k, const int32_t* page_table, int64_t pt_stride,
                              int32_t page_size, const int32_t* out) {
  if (B < 0 || stride < 1 || stride > INT32_MAX) return TOPK_EINVAL;
  if (k < 1 || k > TOPK_MAX_K) return TOPK_EUNSUPPORTED_K;
  if (B == 0) return TOPK_OK;
  if (scores == nullptr || lengths == nullptr || out == nullptr) return TOPK_EINVAL;
  const uintptr_t score_align = bf16 ? 1u : 3u;
  if ((reinterpret_cast<uintptr_t>(scores) & score_align) != 0 || !aligned4(lengths) || !aligned4(out))
    return TOPK_EINVAL;
  if (page_table != nullptr) {
    if (page_size < 1 || pt_stride < 1 || !aligned4(page_table)) return TOPK_EINVAL;
    if (pt_stride < (stride + page_size - 1) / page_size) return TOPK_EINVAL;
  }
  return TOPK_OK;
}

topk_status select_impl(const void* scores, bool bf16, int64_t stride, const int32_t* lengths,
                        int32_t B, int32_t k, const int32_t* page_table, int64_t pt_stride,
                        int32_t page_size, int32_t* out, void* workspace, size_t workspace_bytes,
                        const topk_debug_opts* opts, cudaStream_t stream) {
  const topk_status args =
      check_select_args(scores, bf16, stride, lengths, B, k, page_table, pt_stride, page_size, out);
  if (args != TOPK_OK || B == 0) return args;

  const int kmax = k <= 512 ? 512 : (k <= 1024 ? 1024 : 2048);
  const int cap_max = kmax == 512    ? tki::StashCap<512>::value
                      : kmax == 1024 ? tki::StashCap<1024>::value
                                     : tki::StashCap<2048>::value;

  Params p = {};
  p.scores = static_cast<const float*>(scores);
  p.stride = stride;
  p.lengths = lengths;
  p.B = B;
  p.k = k;
  p.out = out;
  p.page_table = page_table;
  p.pt_stride = page_table != nullptr ? pt_stride : 0;
  p.page_size = page_table != nullptr ? page_size : 1;
  p.page_shift = page_shift_of(p.page_size);
  p.cap = cap_max;
  p.sample_mode = 0;
  p.sample_min_n = kDefaultSampleMinN;
  p.sample_z = kDefaultSampleZ;
  p.counters = nullptr;
  p.probe_stage = -1;
  p.probe_wait_us = 0;
  p.split_first = B;

  int G = 0;
  int split_rows = 0;  // 0 automatic, -1 never, m > 0 forced
  if (opts != nullptr) {
    if (opts->sample_mode < 0 || opts->sample_mode > 2) return TOPK_EINVAL;
    p.sample_mode = opts->sample_mode;
    if (opts->stash_capacity != 0) {
      if (opts->stash_capacity < k + tki::kMinStashRoom || opts->stash_capacity > cap_max)
        return TOPK_EINVAL;
      p.cap = opts->stash_capacity;
    }
    if (opts->sample_z != 0.0f) p.sample_z = opts->sample_z;
    if (opts->cluster_size != 0) {
      const int g = opts->cluster_size;
      if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return TOPK_EINVAL;
      G = g;
    }
    if (opts->counters != nullptr && !aligned4(opts->counters)) return TOPK_EINVAL;
    p.counters = opts->counters;
    if (opts->probe_stage < 0 || (opts->probe_stage > 0 && opts->probe_wait_us == 0)) return TOPK_EINVAL;
    if (opts->probe_wait_us > 5000000u) return TOPK_EINVAL;  // the probe wait stays short
    p.probe_stage = opts->probe_stage - 1;
    p.probe_wait_us = opts->probe_wait_us;
    if (opts->split_rows < -1 || opts->split_rows > B) return TOPK_EINVAL;
    split_rows = opts->split_rows;
    if (split_rows > 0 && G > 1) return TOPK_EINVAL;
    if (workspace != nullptr && opts->workspace != nullptr) return TOPK_EINVAL;
    if (opts->workspace != nullptr) {
      workspace = opts->workspace;
      workspace_bytes = opts->workspace_bytes;
    }
  }
  if (workspace != nullptr) {
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0 || workspace_bytes < kWsHeaderBytes)
      return TOPK_EINVAL;
  } else if (split_rows > 0) {
    return TOPK_EINVAL;
  }

  // Short rows: BF16 scores always, FP32 rows of at most kShortMaxRow scores
  // unless an option of the streaming kernel is forced.
  if (opts != nullptr) {
    if (opts->short_rows < -1 || opts->short_rows > 1) return TOPK_EINVAL;
    if (opts->sample_mode < 0 || opts->sample_mode > 2) return TOPK_EINVAL;
    if (opts->counters != nullptr && !aligned4(opts->counters)) return TOPK_EINVAL;
  }
  const bool streaming_opts = opts != nullptr && (opts->cluster_size != 0 || opts->stash_capacity != 0 ||
                                                  opts->probe_stage != 0 || opts->split_rows > 0);
  const int short_rows = opts != nullptr ? opts->short_rows : 0;
  const bool fits_short = stride <= tki::kShortMaxRow;
  if (bf16 || short_rows == 1) {
    if (!fits_short || streaming_opts || short_rows == -1) return TOPK_EINVAL;
    return launch_short(scores, bf16, stride, lengths, B, k, page_table, pt_stride, page_size, out,
                        opts, stream);
  }
  if (short_rows == 0 && stride <= kShortAutoWidth && !streaming_opts)
    return launch_short(scores, false, stride, lengths, B, k, page_table, pt_stride, page_size, out,
                        opts, stream);

  int dev = 0;
  DeviceInfo* info = nullptr;
  const topk_status st = device_info(&dev, &info);
  if (st != TOPK_OK) return st;
  if (split_rows > 0) G = 1;
  const int64_t ws_room = workspace != nullptr
                             ? static_cast<int64_t>((workspace_bytes - kWsHeaderBytes) / (static_cast<size_t>(k) * 16))
                             : 0;
  if (G == 0)
    G = auto_cluster_size(B, stride, kmax, page_table != nullptr, dev,
                          split_rows == 0 && ws_room >= B && B <= kMaxSplitRows &&
                              auto_split_rows(B, stride, kmax, info->sm_count) == B);
  if (static_cast<int64_t>(B) * G > INT32_MAX) return TOPK_EINVAL;

  // Split rows: the last m rows each run as two independent CTAs.
  if (workspace != nullptr && G == 1 && split_rows >= 0) {
    const int64_t hold = ws_room < kMaxSplitRows ? ws_room : kMaxSplitRows;
    int64_t m = split_rows;
    if (m == 0) {
      m = auto_split_rows(B, stride, kmax, info->sm_count);
      if (m > hold) m = hold;
    } else if (m > hold) {
      return TOPK_EINVAL;
    }
    if (static_cast<int64_t>(B) + m > INT32_MAX) return TOPK_EINVAL;
    if (m > 0) {
      unsigned char* ws = static_cast<unsigned char*>(workspace);
      p.split_first = B - static_cast<int32_t>(m);
      p.ws_ctr = reinterpret_cast<uint32_t*>(ws);
      p.ws_cnt = reinterpret_cast<uint32_t*>(ws + kWsCounterBytes);
      p.ws_key = reinterpret_cast<uint32_t*>(ws + kWsHeaderBytes);
      p.ws_idx = p.ws_key + static_cast<size_t>(m) * 2 * static_cast<size_t>(k);
    }
  }

  const bool paged = page_table != nullptr;
  switch (kmax) {
    case 512: return paged ? tki::launch_k512_paged(p, G, dev, stream)
                           : tki::launch_k512_ragged(p, G, dev, stream);
    case 1024: return paged ? tki::launch_k1024_paged(p, G, dev, stream)
                            : tki::launch_k1024_ragged(p, G, dev, stream);
    default: return paged ? tki::launch_k2048_paged(p, G, dev, stream)
                          : tki::launch_k2048_ragged(p, G, dev, stream);
  }
}

// ---- allocation-free entry point ---------------------------------------------
// Scratch of topk_select_noalloc: a fixed array in the library's own device
// memory, which every GPU that loads the library keeps until the process
// exits. 12 KiB of arrival counters and hand-over counts, then room for 128
// split rows at k = 2048 (512 at k = 512): 4 MiB + 12 KiB.
constexpr size_t kStaticWsBytes = kWsHeaderBytes + static_cast<size_t>(4) * 1024 * 1024;
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

struct StaticWs {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  void* ptr = nullptr;
};
StaticWs g_static_ws_state[kMaxDevices];

// Device address of g_static_ws on device `dev` (current). In host code the
// array's name only stands in for it, so the address is looked up once per
// device. The array is zero when the module loads; the first call also
// enqueues a clear of the arrival counters on its own stream, ahead of its
// kernel, and every call that completes leaves them clear again.
topk_status static_workspace(int dev, cudaStream_t stream, void** ptr) {
  StaticWs& st = g_static_ws_state[dev];
  std::call_once(st.once, [&]() {
    st.err = cudaGetSymbolAddress(&st.ptr, g_static_ws);
    if (st.err == cudaSuccess) st.err = cudaMemsetAsync(st.ptr, 0, kWsCounterBytes, stream);
  });
  if (st.err != cudaSuccess) return TOPK_ECUDA;
  *ptr = st.ptr;
  return TOPK_OK;
}

}  // namespace

extern "C" {

topk_status topk_ragged(const float* scores, int64_t stride, const int32_t* lengths, int32_t B,
                        int32_t k, int32_t* out, topk_stream_t stream) {
  return select_impl(scores, false, stride, lengths, B, k, nullptr, 0, 0, out, nullptr, 0, nullptr,
                     reinterpret_cast<cudaStream_t>(stream));
}

topk_status topk_ragged_ws(const float* scores, int64_t stride, const int32_t* lengths, int32_t B,
                           int32_t k, int32_t* out, void* workspace, size_t workspace_bytes,
                           topk_stream_t stream) {
  return select_impl(scores, false, stride, lengths, B, k, nullptr, 0, 0, out, workspace,
                     workspace_bytes, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

topk_status topk_paged_ws(const float* scores, int64_t stride, const int32_t* lengths, int32_t B,
                          int32_t k, const int32_t* page_table, int64_t pt_stride,
                          int32_t page_size, int32_t* out, void* workspace,
                          size_t workspace_bytes, topk_stream_t stream) {
  if (page_table == nullptr && B > 0) return TOPK_EINVAL;
  if (page_size < 1 || pt_stride < 1) return TOPK_EINVAL;
  return select_impl(scores, false, stride, lengths, B, k, page_table, pt_stride, page_size, out,
                     workspace, workspace_bytes, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

topk_status topk_workspace_bytes(int32_t k, int32_t max_split_rows, size_t* bytes) {
  if (k < 1 || k > TOPK_MAX_K) return TOPK_EUNSUPPORTED_K;
  if (bytes == nullptr || max_split_rows < 0 || max_split_rows > kMaxSplitRows) return TOPK_EINVAL;
  int64_t m = max_split_rows;
  if (m == 0) {
    int dev = 0;
    DeviceInfo* info = nullptr;
    const topk_status st = device_info(&dev, &info);
    if (st != TOPK_OK) return st;
    m = info->sm_count < kMaxSplitRows ? info->sm_count : kMaxSplitRows;
  }
  *bytes = ws_bytes_for(k, m);
  return TOPK_OK;
}

topk_status topk_paged(const float* scores, int64_t stride, const int32_t* lengths, int32_t B,
                       int32_t k, const int32_t* page_table, int64_t pt_stride, int32_t page_size,
                       int32_t* out, topk_stream_t stream) {
  if (page_table == nullptr && B > 0) return TOPK_EINVAL;
  if (page_size < 1 || pt_stride < 1) return TOPK_EINVAL;
  return select_impl(scores, false, stride, lengths, B, k, page_table, pt_stride, page_size, out,
                     nullptr, 0, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

topk_status topk_select_ex(const float* scores, int64_t stride, const int32_t* lengths, int32_t B,
                           int32_t k, const int32_t* page_table, int64_t pt_stride,
                           int32_t page_size, int32_t* out, const topk_debug_opts* opts,
                           topk_stream_t stream) {
  return select_impl(scores, false, stride, lengths, B, k, page_table, pt_stride, page_size, out,
                     nullptr, 0, opts, reinterpret_cast<cudaStream_t>(stream));
}

topk_status topk_select_bf16(const uint16_t* scores, int64_t stride, const int32_t* lengths,
                             int32_t B, int32_t k, const int32_t* page_table, int64_t pt_stride,
                             int32_t page_size, int32_t* out, topk_stream_t stream) {
  if (page_table != nullptr && (page_size < 1 || pt_stride < 1)) return TOPK_EINVAL;
  return select_impl(scores, true, stride, lengths, B, k, page_table, pt_stride, page_size, out,
                     nullptr, 0, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

topk_status topk_select_noalloc(const float* scores, int64_t stride, const int32_t* lengths,
                                int32_t B, int32_t k, const int32_t* page_table,
                                int64_t pt_stride, int32_t page_size, int32_t* out,
                                topk_stream_t stream) {
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // Invalid arguments are reported as by topk_ragged / topk_paged, before the
  // scratch is sized.
  if (page_table != nullptr && (page_size < 1 || pt_stride < 1)) return TOPK_EINVAL;
  const topk_status args =
      check_select_args(scores, false, stride, lengths, B, k, page_table, pt_stride, page_size, out);
  if (args != TOPK_OK || B == 0) return args;
  int dev = 0;
  DeviceInfo* info = nullptr;
  topk_status st = device_info(&dev, &info);
  if (st != TOPK_OK) return st;
  // The scratch this call would use, against the fixed array.
  // (the same policy as the call it makes: rows of at most kShortMaxRow scores
  // take the short-row kernel, which splits nothing)
  const int kmax = k <= 512 ? 512 : (k <= 1024 ? 1024 : 2048);
  const int64_t static_room = static_cast<int64_t>((kStaticWsBytes - kWsHeaderBytes) / (static_cast<size_t>(k) * 16));
  const int G = stride <= kShortAutoWidth
                    ? 0
                    : auto_cluster_size(B, stride, kmax, page_table != nullptr, dev,
                                        static_room >= B && B <= kMaxSplitRows &&
                                            auto_split_rows(B, stride, kmax, info->sm_count) == B);
  const int m = G == 1 ? auto_split_rows(B, stride, kmax, info->sm_count) : 0;
  if (ws_bytes_for(k, m) > kStaticWsBytes) return TOPK_ESCRATCH;
  void* ws = nullptr;
  st = static_workspace(dev, cs, &ws);
  if (st != TOPK_OK) return st;
  return select_impl(scores, false, stride, lengths, B, k, page_table, pt_stride, page_size, out, ws,
                     kStaticWsBytes, nullptr, cs);
}

topk_status topk_max_active_clusters(int32_t k, int32_t paged, int32_t cluster_size,
                                     int32_t* clusters) {
  if (k < 1 || k > TOPK_MAX_K) return TOPK_EUNSUPPORTED_K;
  if (clusters == nullptr) return TOPK_EINVAL;
  if (cluster_size != 2 && cluster_size != 4 && cluster_size != 8 && cluster_size != 16)
    return TOPK_EINVAL;
  int dev = 0;
  DeviceInfo* info = nullptr;
  const topk_status st = device_info(&dev, &info);
  if (st != TOPK_OK) return st;
  const int kmax = k <= 512 ? 512 : (k <= 1024 ? 1024 : 2048);
  *clusters = max_clusters(kmax, paged != 0, cluster_size, dev);
  return TOPK_OK;
}

const char* topk_status_string(topk_status status) {
  switch (status) {
    case TOPK_OK: return "success";
    case TOPK_EINVAL: return "invalid argument (null or misaligned pointer, bad size or stride)";
    case TOPK_EUNSUPPORTED_K: return "k outside [1, TOPK_MAX_K]";
    case TOPK_ECUDA: return "a CUDA runtime call failed";
    case TOPK_EDEVICE: return "current device is not an sm_103 GPU";
    case TOPK_ESCRATCH: return "the call needs more scratch than the static workspace of topk_select_noalloc holds";
    default: return "unknown status";
  }
}

int32_t topk_abi_version(void) { return 3; }

}  // extern "C"
