// Batched, ragged, exact per-row top-k over FP32 scores for sm_103a.
//
// One CTA (or one thread-block cluster of G CTAs) owns one row and reads it
// from HBM once:
//
//  1. Order-preserving key. Each float's bit pattern becomes a uint32 whose
//     unsigned order is the float order with -0 below +0 (the `ordered()`
//     transform of vLLM PR 56346, 实现拆解 1).
//  2. Sampled cutoff (DeepSelect-style filter of the same PR, 执行摘要 / 实现拆解 1).
//     Long rows read 16 evenly spread chunks of 256 scores (4096 samples) and
//     take, by two 11-bit radix-histogram passes in shared memory, a cutoff
//     at rank  mu + z*sqrt(mu) + 1  of the sample, mu = k*4096/n, so that the
//     cutoff sits below the row's k-th largest score with overwhelming
//     probability while keeping a few thousand candidates.
//  3. Streaming filter. The row body is brought into shared memory by a ring
//     of four 16 KiB 1-D bulk copies (TMA engine, cp.async.bulk + mbarrier),
//     consumed two stages at a time; every score whose key clears the running
//     threshold is appended, in index order, to a shared-memory stash of
//     (key, index) pairs. Slots come from per-lane hit counts, a warp scan and
//     one block prefix per pair of stages (deterministic, no atomics).
//  4. Compaction instead of truncation. When the stash would overflow, the
//     exact top-k of the stash is found (below) and kept in place, and the
//     threshold rises to just above the new cutoff. Nothing a later step
//     could need is ever dropped, so overflow never loses candidates
//     (the failure of vLLM issue "persistent_topk silently drops ...", 原因分析,
//     and sglang PR 37625) and never costs another HBM pass.
//  5. Underflow rescan. If the sampled cutoff was above the k-th largest
//     score (fewer than k candidates survived), the row is streamed again with
//     no cutoff (the full-row fallback of vLLM PR 56346, 执行摘要 "双回退兜底").
//  6. Exact cutoff. Radix refinement of the stash keys: an 11-bit coarse
//     histogram pass, then 11 and 10 bits under the found prefix (sglang PR
//     37625's exact-key refinement, and `threshold()` of vLLM PR 56346), with
//     early exit as soon as the remaining rank fills a whole bin.
//  7. Emission. Keys strictly above the cutoff and the first r tied keys are
//     written in stash (= index) order; the paged variant maps each index
//     through the page table (sglang PR 39648's PageTransform epilogue).
//
// Cluster split (sglang PR 39648 report, 实现拆解 4): for batches too small to
// fill the GPU, G CTAs of a cluster each stream a contiguous slice of the row
// with their own stash. Rank 0 owns the row's histograms: the other CTAs add
// into it over distributed shared memory, rank 0 finds each cutoff bin and
// sends it to the others (one cluster barrier before and one after), and
// per-CTA counts give each CTA its output offsets.
//
// Split rows (this library's own device, for the last partial wave of a large
// batch): two independent CTAs stream the halves of a row, each leaves its
// exact top-k in a caller workspace, and the one that finishes second merges
// them; no CTA waits for another.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace tki {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStageFloats = 4096;                     // one ring stage: 16 KiB of scores
constexpr int kPerThread = kStageFloats / kThreads;    // 16 consecutive scores per thread
constexpr int kStages = 4;                             // ring depth: 64 KiB (k > 512; see RingStages)
constexpr int kSampleVec4 = 1024;                    // 4096 sampled scores ...
constexpr int kSampleChunkVec4 = 64;                 // ... in 16 chunks of 256
constexpr int kSampleChunks = kSampleVec4 / kSampleChunkVec4;
constexpr int kBins = 2048;
constexpr int kRoundPerThread = 4;                    // stash entries per thread per round ...
constexpr int kRoundEntries = kRoundPerThread * kThreads;  // ... of emission and histograms
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // 2 s: far beyond any stage latency
// Packed per-warp hit counts of a pair of stages: stage A in bits [0, 13),
// stage B in bits [17, 30) (each at most one stage, 4096 < 2^13), and the
// warps' wait-error flags summed in bits [13, 17) (at most 8 < 2^4).
constexpr uint32_t kFieldB = 17;
constexpr uint32_t kFieldMask = 0x1fffu;
constexpr uint32_t kErrUnit = 1u << 13;
constexpr uint32_t kErrMask = 0xfu << 13;

static_assert(kPerThread == 16, "stage layout assumes four float4 per thread");

// Counter slots of the optional diagnostics array (mirrors topk_counter).
enum : int {
  kCntRows = 0,
  kCntTrivial = 1,
  kCntSampled = 2,
  kCntRescan = 3,
  kCntCompactions = 4,
  kCntDeviceErrors = 5,
  kCntClusterRows = 6,
  kCntSplitRows = 7,
};

// Entry count a split-row half hands over when one of its waits timed out.
constexpr uint32_t kHalfFailed = 0xffffffffu;

// Smallest stash capacity beyond k: the hits of half a CTA on one stage.
constexpr int kMinStashRoom = kStageFloats / 2;

template <int KMAX>
struct StashCap {
  // (a multiple of kRoundPerThread, as the round reads assume)
  // k <= 512: room for k kept candidates plus half a stage of new ones (a
  // sampled cutoff keeps ~800 entries), so that a fifth ring stage fits.
  // Larger k: room for k plus one stage, at most 5120 entries, so that two
  // CTAs with a four-stage ring fit on an SM.
  static constexpr int value = KMAX <= 512 ? KMAX + kMinStashRoom
                                           : (KMAX + kStageFloats < 5120 ? KMAX + kStageFloats : 5120);
};

// Ring stages of the k bucket: the smaller stash of k <= 512 leaves shared
// memory for a fifth (80 KiB in flight per CTA; a CTA whose SM neighbour is
// in its fixed per-row phases streams faster).
template <int KMAX>
struct RingStages {
  static constexpr int value = KMAX <= 512 ? 5 : kStages;
};
static_assert(StashCap<512>::value % kRoundPerThread == 0 && StashCap<1024>::value % kRoundPerThread == 0 &&
                  StashCap<2048>::value % kRoundPerThread == 0,
              "round reads must stay inside the stash");
template <int C, int NS>
struct __align__(128) Smem {
  float ring[NS][kStageFloats];
  uint32_t skey[C];
  uint32_t sidx[C];
  uint32_t hist[kBins];
  uint64_t full[NS];
  uint64_t never;                   // an mbarrier nothing arrives on (the wait-limit test)
  uint32_t rel[NS];                 // warps done with each ring slot (the last one refills it)
  uint32_t issued;                  // stages issued into the ring (for the error drain)
  uint32_t tab[2][kWarps];          // per-group per-warp packed hit counts and wait-error flags
  uint32_t rtab[2][kWarps];         // per-round per-warp (above << 16 | tied) counts
  uint32_t scan[kWarps];
  uint32_t res[4];
  uint32_t pub[4];                  // values the other CTAs of the cluster read
  uint32_t off[2];                  // this CTA's emission offsets in a cluster
};

struct Params {
  const float* scores;
  int64_t stride;
  const int32_t* lengths;
  int32_t B;
  int32_t k;
  int32_t* out;
  const int32_t* page_table;
  int64_t pt_stride;
  int32_t page_size;
  int32_t page_shift;    // log2(page_size) when it is a power of two, else -1
  int32_t cap;           // stash capacity in use, in [k + kStageFloats, C]
  int32_t sample_mode;   // 0 automatic, 1 never, 2 whenever the row is long enough
  int32_t sample_min_n;  // automatic sampling gate on the row length
  float sample_z;        // standard deviations of margin on the sampled rank
  uint32_t* counters;    // optional diagnostics
  int32_t probe_stage;   // test only: >= 0 makes that stage's wait run out on a barrier
  uint32_t probe_wait_us;  // that nothing completes, after this many microseconds
  // Split rows (G == 1 only): rows >= split_first are each streamed by two
  // independent CTAs, blocks split_first + 2*(row - split_first) + half.
  // Each half leaves its exact top-k in the workspace; the later one merges.
  int32_t split_first;   // >= B: no split rows
  uint32_t* ws_ctr;      // per split row: halves arrived (zero on entry, reset to zero by the merger)
  uint32_t* ws_cnt;      // per split row and half: entries handed over, or kHalfFailed
  uint32_t* ws_key;      // per split row and half: k keys ...
  uint32_t* ws_idx;      // ... and indices, in index order
};

// Cutoff description: an entry is selected if (key >> shift) > P, or if
// (key >> shift) == P and fewer than r such entries precede it.
struct Cut {
  uint32_t shift;
  uint32_t P;
  uint32_t r;
  bool all_ties;  // r equals the number of entries with (key >> shift) == P
};

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

// The float b whose key is thr: for every non-NaN score x,
// order_key(x) >= thr  <=>  x >= b  (float compare), except when b is a zero,
// where the float compare cannot tell -0 from +0 and the keys must decide.
__device__ __forceinline__ float float_bound(uint32_t thr) {
  if (thr <= 0x007fffffu) return -__int_as_float(0x7f800000);  // every score passes: -inf
  const uint32_t u = (thr & 0x80000000u) ? (thr ^ 0x80000000u) : ~thr;
  return __uint_as_float(u);
}

// Inclusive prefix sum over lanes [0, LANES) of the warp (lanes past LANES
// receive partial sums).
template <int LANES = 32>
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < LANES; d <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += y;
  }
  return v;
}

// The helpers below take any shared-memory layout SM with the members they
// use (scan, res, hist, skey, sidx, rtab): the streaming kernel's Smem<C, NS>
// and the short-row kernel's layout.
template <class SM>
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, SM& S) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_incl_scan(v);
  if (lane == 31) S.scan[w] = v;
  __syncthreads();
  const uint32_t e = lane < kWarps ? S.scan[lane] : 0u;  // warp totals
  return v + __reduce_add_sync(0xffffffffu, lane < w ? e : 0u);
}

// Shared-memory histogram increment; `bin` = 0xffffffff means "no increment".
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin) {
  if (bin != 0xffffffffu) atomicAdd(&hist[bin], 1u);
}

// Where a CTA's histogram increments go. In a cluster (G > 1) rank 0 owns
// the one histogram of the row: its own increments are local shared atomics,
// the other CTAs add remotely into it (h0 = its address in the cluster's
// shared window), and rank 0 alone searches it.
template <int G>
struct HistDst {
  uint32_t h0;
  bool local;
};

template <int G>
__device__ __forceinline__ void hist_inc(uint32_t* hist, HistDst<G> d, uint32_t bin) {
  if (bin == 0xffffffffu) return;
  if (G == 1 || d.local) {
    atomicAdd(&hist[bin], 1u);
  } else {
    red_dsmem_add(d.h0 + 4u * bin, 1u);
  }
}

// Locates the bin holding the target-th largest element (1 <= target <= total).
// Thread t owns BPT consecutive bins, given in DESCENDING bin order in c[].
// Returns the bin; *above = elements in higher bins; *inbin = elements in it.
// With `zero_own`, each thread also clears the BPT/4 vectors of its own bins
// there, after the scan (stores ahead of the scan's shuffles delayed it) and
// before the last barrier (the next histogram adds into them after it).
template <int BPT, class SM>
__device__ uint32_t find_bin(const uint32_t (&c)[BPT], uint32_t target, SM& S,
                             uint32_t* above, uint32_t* inbin, uint4* zero_own = nullptr) {
  constexpr int nbins = BPT * kThreads;
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) s += c[i];
  const uint32_t incl = block_incl_scan(s, S);
  if (zero_own != nullptr) {
#pragma unroll
    for (int q = 0; q < BPT / 4; ++q) zero_own[q] = make_uint4(0, 0, 0, 0);
  }
  uint32_t acc = incl - s;
  if (acc < target && target <= incl) {
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      if (acc < target && acc + c[i] >= target) {
        S.res[0] = nbins - 1 - (BPT * threadIdx.x + i);
        S.res[1] = acc;
        S.res[2] = c[i];
      }
      acc += c[i];
    }
  }
  __syncthreads();
  *above = S.res[1];
  *inbin = S.res[2];
  return S.res[0];
}

// Reads this thread's BPT bins (descending), zeroes them, and finds the bin
// of the target-th largest element. Must be called by every thread (of every
// CTA of the cluster) after the histogram increments. In a cluster (G > 1)
// the histogram is rank 0's (see HistDst): rank 0 searches it and sends the
// result to the other CTAs, two cluster barriers in all.
template <int G, int BPT, class SM>
__device__ uint32_t merged_find(SM& S, uint32_t target, uint32_t* above, uint32_t* inbin,
                                bool rank0 = true) {
  const int lo = (BPT * kThreads) - BPT * (threadIdx.x + 1);  // lowest owned bin
  auto search_own = [&]() -> uint32_t {
    // Only this thread reads or writes its bins here.
    uint32_t c[BPT];
    uint4* h4 = reinterpret_cast<uint4*>(&S.hist[lo]);
#pragma unroll
    for (int q = 0; q < BPT; q += 4) {
      const uint4 v = h4[q / 4];
      c[BPT - 1 - q] = v.x;
      c[BPT - 2 - q] = v.y;
      c[BPT - 3 - q] = v.z;
      c[BPT - 4 - q] = v.w;
    }
    return find_bin<BPT>(c, target, S, above, inbin, h4);  // zeroes these bins
  };
  if constexpr (G == 1) {
    __syncthreads();
    return search_own();
  } else {
    cluster_sync();  // every CTA's increments have reached rank 0's histogram
    if (rank0) {
      (void)search_own();  // leaves the result in S.res[0 .. 2]
      if (threadIdx.x < G - 1) {
#pragma unroll
        for (int j = 0; j < 3; ++j)
          st_dsmem_u32(map_rank(smem_addr(&S.res[j]), threadIdx.x + 1), S.res[j]);
      }
    }
    cluster_sync();  // the result has reached every CTA
    *above = S.res[1];
    *inbin = S.res[2];
    return S.res[0];
  }
}

// This thread's kRoundPerThread consecutive stash words from `base` (zeros
// when base >= n). The stash capacity is a multiple of kRoundPerThread, so
// the vector reads never pass its end.
__device__ __forceinline__ void load_round(const uint32_t* a, int base, int n,
                                           uint32_t (&v)[kRoundPerThread]) {
#pragma unroll
  for (int q = 0; q < kRoundPerThread / 4; ++q) {
    uint4 x = make_uint4(0, 0, 0, 0);
    if (base < n) x = *reinterpret_cast<const uint4*>(&a[base + 4 * q]);
    v[4 * q + 0] = x.x;
    v[4 * q + 1] = x.y;
    v[4 * q + 2] = x.z;
    v[4 * q + 3] = x.w;
  }
}

// Histogram of stash keys: entries e < n with (key >> fshift) == fval (all
// entries when !filter) add one to bin (key >> dshift) & dmask.
template <int G = 1, class SM>
__device__ void stash_hist(SM& S, int n, bool filter, uint32_t fshift, uint32_t fval,
                           uint32_t dshift, uint32_t dmask, HistDst<G> dst = HistDst<G>{0u, true}) {
  for (int base0 = 0; base0 < n; base0 += kRoundEntries) {
    const int base = base0 + kRoundPerThread * threadIdx.x;
    uint32_t kv[kRoundPerThread];
    load_round(S.skey, base, n, kv);
#pragma unroll
    for (int c = 0; c < kRoundPerThread; ++c) {
      const uint32_t key = kv[c];
      const bool ok = (base + c < n) && (!filter || (key >> fshift) == fval);
      hist_inc<G>(S.hist, dst, ok ? ((key >> dshift) & dmask) : 0xffffffffu);
    }
  }
}

// Exact cutoff of the target-th largest key over the stash (merged over the
// cluster when G > 1). 1 <= target <= total entries. Three radix passes: the
// coarse (key >> 21) histogram of the whole stash, then 11 and 10 bits under
// the prefix found, with an early exit once the remaining rank fills a bin.
// (Inserts do not keep the coarse histogram current: the hits of a stage
// share a few coarse bins, and their shared atomics would serialise in the
// streaming loop.) The histogram is all zero on entry and on return.
template <int G, class SM>
__device__ Cut select_stash(SM& S, int n, uint32_t target, HistDst<G> dst = HistDst<G>{0u, true}) {
  uint32_t above, inbin;
  // The last stash writes of every thread are visible; in a cluster, rank 0
  // is also done with its histogram (its own compactions) before any CTA
  // adds into it.
  if constexpr (G > 1) {
    cluster_sync();
  } else {
    __syncthreads();
  }
  stash_hist<G>(S, n, false, 0, 0, 21, 0x7ff, dst);
  const uint32_t b1 = merged_find<G, 8>(S, target, &above, &inbin, dst.local);
  uint32_t rem = target - above;
  if (rem == inbin) return Cut{21, b1, rem, true};
  stash_hist<G>(S, n, true, 21, b1, 10, 0x7ff, dst);
  const uint32_t b2 = merged_find<G, 8>(S, rem, &above, &inbin, dst.local);
  const uint32_t p2 = (b1 << 11) | b2;
  rem -= above;
  if (rem == inbin) return Cut{10, p2, rem, true};
  stash_hist<G>(S, n, true, 10, p2, 0, 0x3ff, dst);
  const uint32_t b3 = merged_find<G, 4>(S, rem, &above, &inbin, dst.local);
  rem -= above;
  return Cut{0, (p2 << 10) | b3, rem, rem == inbin};
}

// Walks stash entries [0, n) in order and calls sink(sel, pos, key, idx) for
// every one (entries past n as key 0, index 0): sel tells whether it is
// selected, and then pos = (#above-cut before it) + min(#tied before it, r),
// the counts starting at gt0 / eq0 (entries of lower-ranked cluster CTAs).
// The sink may compute from idx unconditionally and store only when sel, so
// that its loads (a page-table lookup) can all be in flight together.
// Safe for in-place compaction: pos never exceeds the entry's own position
// and a round's entries are all read before any of them is written.
template <class SM, class Sink>
__device__ void emit_rounds(SM& S, int n, Cut cut, uint32_t gt0, uint32_t eq0, Sink sink) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  if (cut.all_ties) {
    // Every entry at the cutoff is selected: selection is (key >> shift) >= P,
    // and an entry's slot is the number of selected entries before it.
    uint32_t run = gt0 + eq0;
    int par = 0;
    for (int base0 = 0; base0 < n; base0 += kRoundEntries, par ^= 1) {
      const int base = base0 + kRoundPerThread * threadIdx.x;
      uint32_t kv[kRoundPerThread], iv[kRoundPerThread];
      load_round(S.skey, base, n, kv);
      load_round(S.sidx, base, n, iv);
      uint32_t selm = 0, psel = 0, wsel = 0;
#pragma unroll
      for (int c = 0; c < kRoundPerThread; ++c) {
        const bool sel = base + c < n && (kv[c] >> cut.shift) >= cut.P;
        selm |= static_cast<uint32_t>(sel) << c;
        const uint32_t m = __ballot_sync(0xffffffffu, sel);
        psel += __popc(m & lt_mask);
        wsel += __popc(m);
      }
      if (lane == 0) S.rtab[par][w] = wsel;
      __syncthreads();
      const uint32_t e = lane < kWarps ? S.rtab[par][lane] : 0u;  // per-warp counts
      uint32_t pos = run + __reduce_add_sync(0xffffffffu, lane < w ? e : 0u) + psel;
#pragma unroll
      for (int c = 0; c < kRoundPerThread; ++c) {
        const bool sel = (selm >> c) & 1u;
        sink(sel, pos, kv[c], base + c < n ? iv[c] : 0u);  // no stale index reaches the sink
        pos += sel;
      }
      run += __reduce_add_sync(0xffffffffu, e);
    }
    return;
  }
  uint32_t run_gt = gt0, run_eq = eq0;
  int par = 0;
  for (int base0 = 0; base0 < n; base0 += kRoundEntries, par ^= 1) {
    const int base = base0 + kRoundPerThread * threadIdx.x;
    uint32_t kv[kRoundPerThread], iv[kRoundPerThread];
    load_round(S.skey, base, n, kv);
    load_round(S.sidx, base, n, iv);
    uint32_t gtm = 0, eqm = 0, pgt = 0, peq = 0, wgt = 0, weq = 0;
#pragma unroll
    for (int c = 0; c < kRoundPerThread; ++c) {
      const bool valid = base + c < n;
      const uint32_t hi = kv[c] >> cut.shift;
      const bool gt = valid && hi > cut.P;
      const bool eq = valid && hi == cut.P;
      gtm |= static_cast<uint32_t>(gt) << c;
      eqm |= static_cast<uint32_t>(eq) << c;
      const uint32_t mg = __ballot_sync(0xffffffffu, gt);
      const uint32_t me = __ballot_sync(0xffffffffu, eq);
      pgt += __popc(mg & lt_mask);
      peq += __popc(me & lt_mask);
      wgt += __popc(mg);
      weq += __popc(me);
    }
    if (lane == 0) S.rtab[par][w] = (wgt << 16) | weq;
    __syncthreads();
    const uint32_t e = lane < kWarps ? S.rtab[par][lane] : 0u;  // per-warp packed counts
    const uint32_t before = __reduce_add_sync(0xffffffffu, lane < w ? e : 0u);
    const uint32_t total = __reduce_add_sync(0xffffffffu, e);
    uint32_t gb = run_gt + (before >> 16) + pgt;
    uint32_t eb = run_eq + (before & 0xffffu) + peq;
#pragma unroll
    for (int c = 0; c < kRoundPerThread; ++c) {
      const bool gt = (gtm >> c) & 1u, eq = (eqm >> c) & 1u;
      sink(gt || (eq && eb < cut.r), gb + min(eb, cut.r), kv[c], base + c < n ? iv[c] : 0u);
      gb += gt;
      eb += eq;
    }
    run_gt += total >> 16;
    run_eq += total & 0xffffu;
  }
}

// PAGED: the output indices go through the page table (p.page_table is
// not null); the ragged kernel carries no page-table code at all.
template <int KMAX, int G, bool PAGED>
__global__ void __launch_bounds__(kThreads, 2) topk_rows_kernel(const Params p) {
  constexpr int C = StashCap<KMAX>::value;
  constexpr int NS = RingStages<KMAX>::value;  // ring stages
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem<C, NS>& S = *reinterpret_cast<Smem<C, NS>*>(smem_raw);

  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  // The row, and which of its `parts` contiguous slices this CTA streams:
  // the cluster rank for G > 1, the half of a split row, or the whole row.
  int row, part = 0, parts = 1;
  if constexpr (G > 1) {
    row = static_cast<int>(blockIdx.x) / G;
    part = static_cast<int>(cluster_ctarank());
    parts = G;
  } else if (static_cast<int>(blockIdx.x) < p.split_first) {
    row = static_cast<int>(blockIdx.x);
  } else {
    const int q = static_cast<int>(blockIdx.x) - p.split_first;
    row = p.split_first + (q >> 1);
    part = q & 1;
    parts = 2;
  }
  const int rank = (G > 1) ? part : 0;  // rank in the cluster
  const bool split = (G == 1) && parts == 2;

  const int64_t len_raw = p.lengths[row];
  const int n = static_cast<int>(len_raw < 0 ? 0 : (len_raw > p.stride ? p.stride : len_raw));
  int32_t* out_row = p.out + static_cast<int64_t>(row) * p.k;
  const int32_t* pt_row = PAGED ? p.page_table + static_cast<int64_t>(row) * p.pt_stride : nullptr;
  const bool leader = (t == 0 && part == 0);

  // Read-only loads (the table is never written during the call), so the
  // emission's lookups need not wait for its earlier output stores; a
  // power-of-two page size maps with a shift and a mask.
  auto map_index = [&](uint32_t i) -> int32_t {
    if constexpr (!PAGED) return static_cast<int32_t>(i);
    const uint32_t ps = static_cast<uint32_t>(p.page_size);
    const uint32_t page = p.page_shift >= 0 ? (i >> p.page_shift) : i / ps;
    return static_cast<int32_t>(static_cast<int64_t>(__ldg(pt_row + page)) * ps + (i - page * ps));
  };

  if (p.counters != nullptr && leader) {
    atomicAdd(&p.counters[kCntRows], 1u);
    if (G > 1) atomicAdd(&p.counters[kCntClusterRows], 1u);
  }

  // ---- rows with no more than k scores: every index is selected -----------
  if (n <= p.k) {
    if (split && part == 1) return;  // the first half writes the row
    for (int j = rank * kThreads + t; j < p.k; j += kThreads * G)
      out_row[j] = (j < n) ? map_index(static_cast<uint32_t>(j)) : -1;
    if (p.counters != nullptr && leader) atomicAdd(&p.counters[kCntTrivial], 1u);
    return;  // uniform over the cluster: no cluster barrier has been used yet
  }
  const uint32_t kk = static_cast<uint32_t>(p.k);  // n > k: exactly k slots are filled
  const uint32_t cap = static_cast<uint32_t>(p.cap);

  // ---- row geometry: scalar head up to 16-byte alignment, bulk body, tail --
  const float* rp = p.scores + static_cast<int64_t>(row) * p.stride;
  const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(rp) >> 2) & 3);
  const int h = min((4 - mis) & 3, n);
  const int nb = ((n - h) >> 2) << 2;
  const int tail = n - h - nb;
  const float* body = rp + h;
  const int nstages = (nb + kStageFloats - 1) / kStageFloats;
  const int nfull = nb / kStageFloats;  // stages of a full kStageFloats scores
  const int lg_parts = __ffs(parts) - 1;  // parts is 1, 2, 4, 8 or 16
  const int s0 = (nstages * part) >> lg_parts;
  const int s1 = (nstages * (part + 1)) >> lg_parts;
  // This part's scores: its stages of the body, plus the head / the tail.
  const int b0 = s0 * kStageFloats, b1 = min(s1 * kStageFloats, nb);
  const int n_part = (part == 0 ? h : 0) + (b1 - b0) + (part == parts - 1 ? tail : 0);
  // The sampled region: the whole body for one CTA or a cluster (whose CTAs
  // share one cutoff), this half's stages for a split row.
  const float* sbody = split ? body + b0 : body;
  const int snb = split ? b1 - b0 : nb;
  const int sn = split ? n_part : n;

  // ---- sampled cutoff: decision and sample loads (issued first, and only
  // consumed after the ring setup, so that their latency overlaps it) ---------
  uint32_t thr = 0;
  bool sampled = false;
  uint32_t target = 0;
  float4 sx[4];
  uint32_t smask = 0;
  {
    const bool long_enough = snb >= 2 * 4 * kSampleVec4;
    const bool want = long_enough && (p.sample_mode == 2 || (p.sample_mode == 0 && sn >= p.sample_min_n));
    if (want) {
      const float mu = static_cast<float>(kk) * (4.0f * kSampleVec4) * __frcp_rn(static_cast<float>(sn));
      float rf = ceilf(mu + p.sample_z * sqrtf(mu)) + 1.0f;
      rf = fmaxf(rf, 1.0f);
      if (rf < 4.0f * kSampleVec4) {
        sampled = true;
        target = static_cast<uint32_t>(rf);
      }
    }
#pragma unroll
    for (int v = 0; v < 4; ++v) sx[v] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (sampled) {
      const int nb4 = snb >> 2;
      const int step4 = (nb4 - kSampleChunkVec4) / (kSampleChunks - 1);  // float4s between chunk starts
      constexpr int per_rank = kSampleVec4 / G;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int f = t + v * kThreads;
        if (f < per_rank) {
          const int gf = rank * per_rank + f;
          const int chunk = gf / kSampleChunkVec4, within = gf % kSampleChunkVec4;
          const int off4 = chunk * step4 + within;
          sx[v] = __ldg(reinterpret_cast<const float4*>(sbody) + off4);
          smask |= 0xfu << (4 * v);
        }
      }
    }
  }

  // Ring bookkeeping. Stage j of a pass goes to slot (pass start + j - s0) %
  // NS; `consumed` (stages taken from the ring so far) is uniform.
  // Thread 0 fills the ring at the start of a pass; afterwards the last warp
  // to finish with a slot refills it with the stage NS further on.
  uint32_t consumed = 0, t0_seen = 0;
  bool abort = false;

  // One thread; the caller has made the slot's earlier shared-memory reads
  // visible to the bulk copy (fence_proxy_async_smem).
  auto issue_stage = [&](int j, uint32_t slot) {
    const int cnt = min(kStageFloats, nb - j * kStageFloats);
    mbar_arrive_expect_tx(&S.full[slot], static_cast<uint32_t>(cnt) * 4u);
    bulk_load(&S.ring[slot][0], body + static_cast<int64_t>(j) * kStageFloats,
              static_cast<uint32_t>(cnt) * 4u, &S.full[slot]);
  };
  auto prime = [&]() {
    if (t == 0 && !abort) {
      const int m = min(s1 - s0, NS);
      fence_proxy_async_smem();
      for (int u = 0; u < m; ++u) issue_stage(s0 + u, (consumed + u) % NS);
      S.issued += m;
    }
  };
  // Called by every thread once it no longer reads ring slot `slot` (stage
  // j) nor, when `two`, the next slot (stage j + 1). The last warp refills
  // both with the stages NS further on.
  auto release_slots = [&](int j, uint32_t slot, bool two) {
    __syncwarp();
    if (lane == 0 && atom_add_acq_rel_cta(&S.rel[slot], 1u) == kWarps - 1) {
      S.rel[slot] = 0;
      if (!abort && j + NS < s1) {
        fence_proxy_async_smem();
        issue_stage(j + NS, slot);
        uint32_t m = 1;
        if (two && j + 1 + NS < s1) {
          issue_stage(j + 1 + NS, (slot + 1) % NS);
          ++m;
        }
        atomicAdd(&S.issued, m);
      }
    }
  };
  if (t == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      mbar_init(&S.full[s], 1);
      S.rel[s] = 0;
    }
    mbar_init(&S.never, 1);
    S.issued = 0;
    fence_mbar_init();
  }
  prime();  // the first stages are in flight during the setup and the sample passes
  for (int i = t; i < kBins; i += kThreads) S.hist[i] = 0;
  __syncthreads();
  // In a cluster, every CTA's histogram increments go to rank 0's histogram,
  // which is zero before any CTA adds into it (and after every search).
  HistDst<G> hdst{0u, true};
  if constexpr (G > 1) {
    hdst.h0 = map_rank(smem_addr(&S.hist[0]), 0);
    hdst.local = rank == 0;
    cluster_sync();
  }

  // ---- sampled cutoff: two 11-bit radix passes over the sample ---------------
  if (sampled) {
    uint32_t above, inbin;
    uint32_t sk[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      sk[4 * v + 0] = order_key(sx[v].x);
      sk[4 * v + 1] = order_key(sx[v].y);
      sk[4 * v + 2] = order_key(sx[v].z);
      sk[4 * v + 3] = order_key(sx[v].w);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) hist_inc<G>(S.hist, hdst, ((smask >> i) & 1u) ? (sk[i] >> 21) : 0xffffffffu);
    const uint32_t b1 = merged_find<G, 8>(S, target, &above, &inbin, hdst.local);
    const uint32_t rem = target - above;
    if (rem == inbin) {
      thr = b1 << 21;
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const bool ok = ((smask >> i) & 1u) && (sk[i] >> 21) == b1;
        hist_inc<G>(S.hist, hdst, ok ? ((sk[i] >> 10) & 0x7ffu) : 0xffffffffu);
      }
      const uint32_t b2 = merged_find<G, 8>(S, rem, &above, &inbin, hdst.local);
      thr = (b1 << 21) | (b2 << 10);
    }
  }

  // ---- streaming filter into the stash --------------------------------------
  uint32_t n_st = 0;        // stash entries (uniform)
  uint32_t grp = 0;         // groups processed (uniform), selects the count table half
  uint32_t compactions = 0;
  float bound = float_bound(thr);

  auto compact = [&]() {
    const Cut cut = select_stash<1>(S, static_cast<int>(n_st), kk);
    emit_rounds(S, static_cast<int>(n_st), cut, 0u, 0u, [&](bool sel, uint32_t pos, uint32_t key, uint32_t idx) {
      if (sel && pos < kk) {  // exactly kk entries are selected; the guard only bounds a corrupted cut
        S.skey[pos] = key;
        S.sidx[pos] = idx;
      }
    });
    __syncthreads();
    n_st = kk;
    thr = max(thr, (cut.P << cut.shift) + 1u);
    bound = float_bound(thr);
    ++compactions;
  };

  // Exact hit mask: bit e set when score e of this thread's group (index
  // order) has a key >= thr. `bound` is the float whose key is thr, so a float
  // comparison is exact unless bound is a zero, where -0 < +0 must come from
  // the keys.
  auto hit_mask = [&](const float4 (&v)[4], int rot, uint32_t valid) -> uint32_t {
    uint32_t pl = 0;  // in load order: v[j] at bits 4j .. 4j + 3
    if (bound != 0.0f) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pl |= (static_cast<uint32_t>(v[j].x >= bound) | (static_cast<uint32_t>(v[j].y >= bound) << 1) |
               (static_cast<uint32_t>(v[j].z >= bound) << 2) | (static_cast<uint32_t>(v[j].w >= bound) << 3))
              << (4 * j);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pl |= (static_cast<uint32_t>(order_key(v[j].x) >= thr) |
               (static_cast<uint32_t>(order_key(v[j].y) >= thr) << 1) |
               (static_cast<uint32_t>(order_key(v[j].z) >= thr) << 2) |
               (static_cast<uint32_t>(order_key(v[j].w) >= thr) << 3))
              << (4 * j);
      }
    }
    // v[j] holds the scores 4 * ((j + rot) & 3) ..: rotate the 16 bits left by 4 * rot
    const uint32_t pl2 = pl | (pl << 16);
    return (pl2 >> (16 - 4 * rot)) & valid;
  };

  // Hit mask of this thread's 16 scores of a ring stage (ts points at them;
  // scores past the stage's end are stale and masked off by `valid`). The
  // float4 reads are rotated by `rot` so that they are bank-conflict free.
  // (No per-thread maximum is tested first: in a warp of 512 scores some
  // lane nearly always passes, so such a prefilter only added work.)
  // A scalar group (ts == nullptr) has one score, sx, present when bit 0 of
  // `valid` is set.
  auto group_mask = [&](const float* ts, float sx, int rot, uint32_t valid) -> uint32_t {
    if (ts == nullptr) return ((valid & 1u) != 0u && order_key(sx) >= thr) ? 1u : 0u;
    float4 v[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) v[jj] = *reinterpret_cast<const float4*>(ts + 4 * ((jj + rot) & 3));
    return hit_mask(v, rot, valid);
  };

  // Base (lower warps) and total of the packed per-warp counts in table half `par`.
  auto read_table = [&](int par, uint32_t& base, uint32_t& total) {
    const uint32_t e = lane < kWarps ? S.tab[par][lane] : 0u;  // lane i: warp i's word
    base = __reduce_add_sync(0xffffffffu, lane < w ? e : 0u);
    total = __reduce_add_sync(0xffffffffu, e);
  };

  // Publishes this warp's packed count and error flag and synchronises the
  // CTA. Returns this lane's inclusive packed count in the warp, and the
  // packed counts of the lower warps (base) and of all warps (total).
  auto publish = [&](uint32_t cnt, bool err, uint32_t& incl, uint32_t& base, uint32_t& total) {
    const uint32_t wtot = __reduce_add_sync(0xffffffffu, cnt);  // off the scan's critical path
    incl = warp_incl_scan(cnt);
    const bool werr = __any_sync(0xffffffffu, err);
    const int par = static_cast<int>(grp & 1u);
    ++grp;
    if (lane == 0) S.tab[par][w] = wtot + (werr ? kErrUnit : 0u);
    __syncthreads();
    read_table(par, base, total);
  };

  // Appends this lane's hits (bits of m, in index order) from stash position
  // pos on; score e is ts[e] (or sx for a scalar group), its index idx0 + e.
  auto write_hits = [&](uint32_t m, uint32_t pos, const float* ts, float sx, uint32_t idx0) {
    while (m != 0u) {  // two at a time
      const int e0 = __ffs(m) - 1;
      m &= m - 1u;
      const bool two = m != 0u;
      const int e1 = two ? __ffs(m) - 1 : e0;
      if (two) m &= m - 1u;
      const float x0 = ts != nullptr ? ts[e0] : sx;
      const float x1 = ts != nullptr ? ts[e1] : sx;
      const uint32_t k0 = order_key(x0), k1 = order_key(x1);
      S.skey[pos] = k0;
      S.sidx[pos] = idx0 + e0;
      ++pos;
      if (two) {
        S.skey[pos] = k1;
        S.sidx[pos] = idx0 + e1;
        ++pos;
      }
    }
  };

  // One group: two consecutive ring stages A and B (B absent when tsB is
  // null), or one scalar group as A. Thread t's 16 scores of stage A start at
  // tsA and have indices idxA + e (present where bit e of validA is set);
  // likewise for B. Hits of A precede those of B in the stash, each in index
  // order, so the stash stays in index order. One block barrier per group
  // (more only when the stash must be compacted). Every thread of the CTA
  // calls it.
  auto process_group = [&](const float* tsA, const float* tsB, float sx, int rot, uint32_t validA,
                           uint32_t validB, uint32_t idxA, uint32_t idxB, bool err) {
    uint32_t pmA = group_mask(tsA, sx, rot, validA);
    uint32_t pmB = tsB != nullptr ? group_mask(tsB, sx, rot, validB) : 0u;
    uint32_t cnt = __popc(pmA) + (static_cast<uint32_t>(__popc(pmB)) << kFieldB);
    uint32_t incl, base, total;
    publish(cnt, err, incl, base, total);
    if ((total & kErrMask) != 0u) abort = true;
    if (abort) return;  // uniform
    uint32_t tA = total & kFieldMask, tB = (total >> kFieldB) & kFieldMask;
    if (tA + tB == 0u) return;  // uniform
    if (n_st + tA + tB > cap) {
      if (n_st > kk) {  // keep the exact top-k so far and raise the cutoff
        compact();
        pmA = group_mask(tsA, sx, rot, validA);
        pmB = tsB != nullptr ? group_mask(tsB, sx, rot, validB) : 0u;
        cnt = __popc(pmA) + (static_cast<uint32_t>(__popc(pmB)) << kFieldB);
        publish(cnt, false, incl, base, total);
        tA = total & kFieldMask;
        tB = (total >> kFieldB) & kFieldMask;
      }
      if (n_st + tA + tB > cap) {
        // More hits than the stash has room for, even above a raised cutoff.
        // Quarters of the group (half the CTA on one stage, at most
        // kMinStashRoom hits each) append in index order, compacting in
        // between (a quarter overflows only when the stash holds more than
        // k entries).
        for (int part = 0; part < 4; ++part) {
          const bool second = part >= 2;
          if (second && tsB == nullptr) break;  // uniform
          const bool mine = (w >> 2) == (part & 1);
          const float* ts = second ? tsB : tsA;
          const uint32_t valid = second ? validB : validA;
          uint32_t pm = mine ? group_mask(ts, sx, rot, valid) : 0u;
          uint32_t c = __popc(pm);
          publish(c, false, incl, base, total);
          if (n_st + (total & kFieldMask) > cap) {
            compact();
            pm = mine ? group_mask(ts, sx, rot, valid) : 0u;
            c = __popc(pm);
            publish(c, false, incl, base, total);
          }
          write_hits(pm, n_st + (base & kFieldMask) + incl - c, ts, sx, second ? idxB : idxA);
          n_st += total & kFieldMask;
        }
        return;
      }
    }
    const uint32_t before = incl - cnt;  // packed hits of the lower lanes of this warp
    write_hits(pmA, n_st + (base & kFieldMask) + (before & kFieldMask), tsA, sx, idxA);
    write_hits(pmB, n_st + tA + ((base >> kFieldB) & kFieldMask) + ((before >> kFieldB) & kFieldMask),
               tsB, sx, idxB);
    n_st += tA + tB;
  };

  // Scalar group: thread t < cnt holds the score at index first + t.
  auto scalar_group = [&](int first, int cnt) {
    float sx = 0.0f;
    uint32_t valid = 0;
    if (t < cnt) {
      sx = rp[first + t];
      valid = 1u;
    }
    process_group(nullptr, nullptr, sx, 0, valid, 0u, static_cast<uint32_t>(first + t), 0u, false);
  };

  // Takes stage j from the ring: waits for it (bounded) and returns this
  // thread's 16 scores in it, with the mask of those present.
  const bool probing = p.probe_stage >= 0;  // test only
  auto take_stage = [&](int j, bool& err, uint32_t& valid, uint32_t& slot) -> const float* {
    slot = consumed % NS;
    const uint32_t parity = (consumed / NS) & 1u;
    ++consumed;
    if (!abort) {
      if (probing && j - s0 == p.probe_stage) {
        err |= !mbar_wait_bounded(&S.never, 0u, 1000ull * p.probe_wait_us);  // runs out
      } else if (mbar_wait_bounded(&S.full[slot], parity, kWaitLimitNs)) {
        ++t0_seen;  // in order: stages [t0_seen, issued) are unobserved
      } else {
        err = true;
      }
    }
    if (j < nfull) {
      valid = 0xffffu;
    } else {  // the last, partial stage
      const int have = (nb - j * kStageFloats) - kPerThread * t;
      valid = have >= kPerThread ? 0xffffu : (have <= 0 ? 0u : (1u << have) - 1u);
    }
    return &S.ring[slot][kPerThread * t];
  };

  auto stream_pass = [&]() {
    const int rot = (t >> 1) & 3;  // rotates the float4 order: conflict-free shared loads
    if (part == 0 && h > 0) scalar_group(0, h);
    for (int j = s0; j < s1; j += 2) {
      const bool two = j + 1 < s1;
      bool err = false;
      uint32_t validA, validB = 0, slotA, slotB;
      const float* tsA = take_stage(j, err, validA, slotA);
      const float* tsB = two ? take_stage(j + 1, err, validB, slotB) : nullptr;
      const uint32_t idxA = static_cast<uint32_t>(h + j * kStageFloats + kPerThread * t);
      process_group(tsA, tsB, 0.0f, rot, validA, validB, idxA, idxA + kStageFloats, err);
      release_slots(j, slotA, two);
    }
    if (part == parts - 1 && tail > 0) scalar_group(h + nb, tail);
  };

  stream_pass();

  // ---- underflow: the sampled cutoff kept fewer than k candidates -----------
  // (fewer than min(k, its scores) for the half of a split row)
  const uint32_t need = split ? min(kk, static_cast<uint32_t>(n_part)) : kk;
  if (sampled) {
    uint32_t total = n_st;
    if constexpr (G > 1) {
      if (t == 0) S.pub[0] = n_st;
      cluster_sync();
      if (w == 0) {  // lane r reads rank r's count
        uint32_t v = lane < G ? ld_dsmem_u32(map_rank(smem_addr(&S.pub[0]), lane)) : 0u;
        v = __reduce_add_sync(0xffffffffu, v);
        if (lane == 0) S.res[3] = v;
      }
      cluster_sync();  // every CTA has read every count; S.res[3] is visible
      total = S.res[3];
    }
    if (total < need) {  // uniform over the cluster
      if (p.counters != nullptr && t == 0 && rank == 0) atomicAdd(&p.counters[kCntRescan], 1u);
      thr = 0;
      bound = float_bound(thr);
      n_st = 0;
      __syncthreads();  // (the histogram is zero: every search leaves it so)
      prime();
      stream_pass();
    }
  }

  // A wait timed out: let copies still in flight land (bounded) before the
  // CTA leaves, so that no bulk copy writes into shared memory it no longer owns.
  auto drain = [&]() {
    if (abort && t == 0) {
      for (uint32_t u = t0_seen; u < S.issued; ++u)
        (void)mbar_wait_bounded(&S.full[u % NS], (u / NS) & 1u, kWaitLimitNs);
      if (p.counters != nullptr) atomicAdd(&p.counters[kCntDeviceErrors], 1u);
    }
  };
  auto poison_row = [&]() {  // marks the row as failed: no result can be mistaken for one
    for (int j = t; j < p.k; j += kThreads) out_row[j] = static_cast<int32_t>(0x80000000u);
  };

  if (split) {
    // ---- split row: this half's exact top-k goes to the workspace; the half
    // that finishes second merges both (no CTA ever waits for another) -------
    const int slot = row - p.split_first;
    const size_t off = static_cast<size_t>(2 * slot + part) * kk;
    uint32_t handed = 0;
    if (!abort) {
      if (n_st > need) {
        const Cut c = select_stash<1>(S, static_cast<int>(n_st), need);
        emit_rounds(S, static_cast<int>(n_st), c, 0u, 0u, [&](bool sel, uint32_t pos, uint32_t key, uint32_t idx) {
          if (sel && pos < need) {
            p.ws_key[off + pos] = key;
            p.ws_idx[off + pos] = idx;
          }
        });
        handed = need;
      } else {
        // Every thread reads stash entries that others wrote in the last
        // group, after that group's barrier: wait for all of them (a half
        // whose last group is a stage, with no scalar tail after it, has no
        // barrier since).
        __syncthreads();
        for (int e = t; e < static_cast<int>(n_st); e += kThreads) {
          p.ws_key[off + e] = S.skey[e];
          p.ws_idx[off + e] = S.sidx[e];
        }
        handed = n_st;
      }
    }
    drain();
    if (p.counters != nullptr && t == 0) {
      if (compactions) atomicAdd(&p.counters[kCntCompactions], compactions);
      if (part == 0 && sampled) atomicAdd(&p.counters[kCntSampled], 1u);
    }
    if (t == 0) p.ws_cnt[2 * slot + part] = abort ? kHalfFailed : handed;
    __threadfence();  // the hand-over is visible before the arrival is counted
    __syncthreads();
    if (t == 0) S.res[3] = atomicAdd(&p.ws_ctr[slot], 1u);
    __syncthreads();
    if (S.res[3] == 0u) return;  // first to finish: the other half merges
    __threadfence();
    if (t == 0) p.ws_ctr[slot] = 0u;  // both halves have arrived: ready for the next call
    const uint32_t c0 = __ldcg(&p.ws_cnt[2 * slot]), c1 = __ldcg(&p.ws_cnt[2 * slot + 1]);
    if (c0 == kHalfFailed || c1 == kHalfFailed) {
      poison_row();
      return;
    }
    if (PAGED) {  // as below, for the whole row
      const int p1 = (n + p.page_size - 1) / p.page_size;
      for (int q = 32 * t; q < p1; q += 32 * kThreads) prefetch_l2(pt_row + q);
      if (t == 0) prefetch_l2(pt_row + p1 - 1);
    }
    for (int i = t; i < kBins; i += kThreads) S.hist[i] = 0;
    __syncthreads();  // the local emission has read the stash; the histogram is clear
    // Half 0's entries precede half 1's: the merged stash is in index order.
    const size_t base0 = static_cast<size_t>(2 * slot) * kk;
    for (int e = t; e < static_cast<int>(c0 + c1); e += kThreads) {
      const size_t src = static_cast<uint32_t>(e) < c0 ? base0 + e : base0 + kk + (e - c0);
      const uint32_t key = __ldcg(&p.ws_key[src]);
      S.skey[e] = key;
      S.sidx[e] = __ldcg(&p.ws_idx[src]);
    }
    const Cut c = select_stash<1>(S, static_cast<int>(c0 + c1), kk);
    emit_rounds(S, static_cast<int>(c0 + c1), c, 0u, 0u, [&](bool sel, uint32_t pos, uint32_t, uint32_t idx) {
      const int32_t v = map_index(idx);
      if (sel && pos < kk) out_row[pos] = v;
    });
    if (p.counters != nullptr && t == 0) atomicAdd(&p.counters[kCntSplitRows], 1u);
    return;
  }

  if constexpr (G == 1) {
    if (abort) {  // uniform: nothing is selected from an incomplete stash, and
      drain();    // the poison is the only store this CTA makes to its row
      poison_row();
      return;
    }
  }

  // ---- exact cutoff over the stash(es) and emission --------------------------
  if (PAGED && !abort) {
    // The emission maps every selected index through the page table: start
    // bringing this CTA's part of the table row into L2 while the cutoff is
    // found (one line per 32 entries).
    const int first = rank == 0 ? 0 : h + s0 * kStageFloats;
    const int last = rank == G - 1 ? n : h + s1 * kStageFloats;
    const int p0 = first / p.page_size, p1 = (last + p.page_size - 1) / p.page_size;
    for (int q = p0 + 32 * t; q < p1; q += 32 * kThreads) prefetch_l2(pt_row + q);
    if (t == 0 && p1 > p0) prefetch_l2(pt_row + p1 - 1);  // the last line, if no start fell in it
  }
  const Cut cut = select_stash<G>(S, static_cast<int>(n_st), kk, hdst);
  uint32_t gt0 = 0, eq0 = 0;
  if constexpr (G > 1) {
    // Entries above / at the cutoff in this CTA's stash; lower ranks come first.
    if (t == 0) {
      S.pub[1] = 0;
      S.pub[2] = 0;
    }
    __syncthreads();
    uint32_t lg = 0, le = 0;
    for (int e = t; e < static_cast<int>(n_st); e += kThreads) {
      const uint32_t hi = S.skey[e] >> cut.shift;
      lg += hi > cut.P;
      le += hi == cut.P;
    }
    for (int d = 16; d > 0; d >>= 1) {
      lg += __shfl_xor_sync(0xffffffffu, lg, d);
      le += __shfl_xor_sync(0xffffffffu, le, d);
    }
    if (lane == 0) {
      atomicAdd(&S.pub[1], lg);
      atomicAdd(&S.pub[2], le);
    }
    cluster_sync();
    if (w == 0) {  // lane r < rank reads rank r's counts
      uint32_t g = 0, e = 0;
      if (lane < rank) {
        g = ld_dsmem_u32(map_rank(smem_addr(&S.pub[1]), lane));
        e = ld_dsmem_u32(map_rank(smem_addr(&S.pub[2]), lane));
      }
      g = __reduce_add_sync(0xffffffffu, g);
      e = __reduce_add_sync(0xffffffffu, e);
      if (lane == 0) {
        S.off[0] = g;
        S.off[1] = e;
      }
    }
    __syncthreads();
    gt0 = S.off[0];
    eq0 = S.off[1];
  }
  emit_rounds(S, static_cast<int>(n_st), cut, gt0, eq0,
              [&](bool sel, uint32_t pos, uint32_t, uint32_t idx) {
                const int32_t v = map_index(idx);
                if (sel && pos < kk) out_row[pos] = v;
              });

  if constexpr (G > 1) cluster_sync();  // no CTA leaves while others may read its shared memory

  if (p.counters != nullptr && t == 0) {
    if (compactions) atomicAdd(&p.counters[kCntCompactions], compactions);
    if (rank == 0 && sampled) atomicAdd(&p.counters[kCntSampled], 1u);
  }
  if (abort) {  // a cluster CTA: the cluster barrier above orders every
    drain();    // emission store of the cluster before the poison
    poison_row();
  }
}

}  // namespace tki
