// Exact per-row top-k for short rows (at most 16384 scores), FP32 or BF16
// scores: the prefill side of the indexer, where a batch holds thousands of
// rows of a few thousand scores each.
//
// The streaming kernel's per-row fixed costs (sample loads, ring set-up,
// three radix passes, emission rounds) are paid for every row, and with two
// rows in flight per SM they dominate rows this short. Here one CTA of 256
// threads takes a row and keeps it in registers, E consecutive scores per
// thread (E = 32: rows up to 8192; E = 64: up to 16384), so the row is read
// from HBM exactly once and every later step works on registers and a small
// shared-memory stash. The design follows the bf16 small-row top-k of the
// sglang PR 39648 report (实现拆解 2: one CTA per row, the row resident in
// registers, radix passes to the exact k-th value, page-table transform on
// output), with the sampled cutoff of vLLM PR 56346 (实现拆解 1) in front:
//
//  1. Sampled cutoff: E / 16 scores per thread (every 16th score of the row)
//     go through two 11-bit radix passes to the sample's rank
//     mu + z*sqrt(mu) + 1, mu = k * samples / n: a cutoff below the row's
//     k-th largest score with overwhelming probability.
//  2. Filter: the scores whose key clears the cutoff go to the stash as
//     (key, index), in index order (per-thread counts, one block prefix).
//  3. Exact cutoff over the stash and emission in stash (= index) order, with
//     the streaming kernel's select_stash / emit_rounds.
//  4. Exact register path: if the cutoff kept fewer than k scores or more
//     than the stash holds (ties, adversarial rows), or sampling is off, the
//     radix passes run over the registers themselves and the census writes
//     the selection straight from them.
#pragma once

#include <cstdint>

#include "topk_kernel.cuh"

namespace tki {

constexpr int kShortMaxRow = 16384;

// Counter slots of the short-row path (after the streaming kernel's).
enum : int {
  kCntShortRows = 8,   // rows taken by the short-row kernel
  kCntShortExact = 9,  // of them, rows that took the exact register path
};

template <int KMAX>
struct ShortCap {
  // Candidates the stash holds: k plus a margin above the sampled rank.
  static constexpr int value = KMAX + 2048;
};

template <int C>
struct ShortSmem {
  uint32_t skey[C];
  uint32_t sidx[C];
  uint32_t hist[kBins];
  uint32_t tab[2][kWarps];
  uint32_t rtab[2][kWarps];
  uint32_t scan[kWarps];
  uint32_t res[4];
};

struct ShortParams {
  const void* scores;  // float or bf16 (as uint16) rows
  int64_t stride;      // elements between rows, <= kShortMaxRow
  const int32_t* lengths;
  int32_t B;
  int32_t k;
  int32_t* out;
  const int32_t* page_table;
  int64_t pt_stride;
  int32_t page_size;
  int32_t sample_mode;  // 0 automatic, 1 never (exact register path), 2 whenever possible
  float sample_z;
  uint32_t* counters;
  int32_t ahead;  // CTAs resident at once: the block that will take this CTA's slot next
};

template <typename T>
struct ScoreIn;

template <>
struct ScoreIn<float> {
  // E consecutive scores from p (16-byte aligned when `vec`).
  template <int E>
  __device__ __forceinline__ static void load(const float* p, int nv, bool vec, uint32_t (&key)[E]) {
    if (vec) {
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(p) + q);
        key[4 * q + 0] = order_key(x.x);
        key[4 * q + 1] = order_key(x.y);
        key[4 * q + 2] = order_key(x.z);
        key[4 * q + 3] = order_key(x.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < E; ++j) key[j] = j < nv ? order_key(__ldg(p + j)) : 0u;
    }
  }
  static constexpr int kVecAlign = 16;
};

template <>
struct ScoreIn<uint16_t> {
  // bf16 -> fp32 is exact: the bf16 bits are the float's high half.
  __device__ __forceinline__ static uint32_t key_of(uint32_t bits16) {
    return order_key(__uint_as_float(bits16 << 16));
  }
  template <int E>
  __device__ __forceinline__ static void load(const uint16_t* p, int nv, bool vec, uint32_t (&key)[E]) {
    if (vec) {
#pragma unroll
      for (int q = 0; q < E / 8; ++q) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(p) + q);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          key[8 * q + 2 * i + 0] = key_of(w[i] & 0xffffu);
          key[8 * q + 2 * i + 1] = key_of(w[i] >> 16);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < E; ++j) key[j] = j < nv ? key_of(__ldg(p + j)) : 0u;
    }
  }
  static constexpr int kVecAlign = 16;
};

template <int E, int KMAX, bool PAGED, typename T>
__global__ void __launch_bounds__(kThreads, E <= 32 ? 3 : 2) topk_short_kernel(const ShortParams p) {
  constexpr int C = ShortCap<KMAX>::value;
  constexpr int kSamples = E / 16;  // per thread
  static_assert(E % 32 == 0 && E * kThreads <= kShortMaxRow, "a row must fit the CTA's registers");
  __shared__ __align__(16) ShortSmem<C> S;

  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int row = static_cast<int>(blockIdx.x);
  // Start bringing the row of the block that will most likely take this
  // CTA's slot next into L2, so that its loads do not wait on HBM.
  if (t == 0 && p.ahead > 0 && row + p.ahead < p.B) {
    const int nr = row + p.ahead;
    const int64_t ln = p.lengths[nr];
    const int len = static_cast<int>(ln < 0 ? 0 : (ln > p.stride ? p.stride : ln));
    const char* base = reinterpret_cast<const char*>(static_cast<const T*>(p.scores) +
                                                     static_cast<int64_t>(nr) * p.stride);
    const uintptr_t a0 = (reinterpret_cast<uintptr_t>(base) + 15u) & ~static_cast<uintptr_t>(15u);
    const uintptr_t a1 = (reinterpret_cast<uintptr_t>(base) + static_cast<uintptr_t>(len) * sizeof(T)) &
                         ~static_cast<uintptr_t>(15u);
    if (a1 > a0) bulk_prefetch_l2(reinterpret_cast<const void*>(a0), static_cast<uint32_t>(a1 - a0));
  }
  const int64_t len_raw = p.lengths[row];
  const int n = static_cast<int>(len_raw < 0 ? 0 : (len_raw > p.stride ? p.stride : len_raw));
  int32_t* out_row = p.out + static_cast<int64_t>(row) * p.k;
  const int32_t* pt_row = PAGED ? p.page_table + static_cast<int64_t>(row) * p.pt_stride : nullptr;
  auto map_index = [&](uint32_t i) -> int32_t {
    if constexpr (!PAGED) return static_cast<int32_t>(i);
    const uint32_t ps = static_cast<uint32_t>(p.page_size);
    const uint32_t page = i / ps;
    return static_cast<int32_t>(static_cast<int64_t>(pt_row[page]) * ps + (i - page * ps));
  };
  if (p.counters != nullptr && t == 0) {
    atomicAdd(&p.counters[kCntRows], 1u);
    atomicAdd(&p.counters[kCntShortRows], 1u);
  }

  // ---- rows with no more than k scores: every index is selected -----------
  if (n <= p.k) {
    for (int j = t; j < p.k; j += kThreads) out_row[j] = (j < n) ? map_index(static_cast<uint32_t>(j)) : -1;
    if (p.counters != nullptr && t == 0) atomicAdd(&p.counters[kCntTrivial], 1u);
    return;
  }
  const uint32_t kk = static_cast<uint32_t>(p.k);

  // ---- this thread's E consecutive scores, as keys --------------------------
  const T* rp = static_cast<const T*>(p.scores) + static_cast<int64_t>(row) * p.stride;
  const int first = E * t;
  const int nv = min(max(n - first, 0), E);  // valid scores of this thread
  uint32_t key[E];
  {
    const T* tp = rp + first;
    const bool vec = nv == E && (reinterpret_cast<uintptr_t>(tp) % ScoreIn<T>::kVecAlign) == 0;
    if (nv > 0) {
      ScoreIn<T>::template load<E>(tp, nv, vec, key);
    } else {
#pragma unroll
      for (int j = 0; j < E; ++j) key[j] = 0u;
    }
  }
  // valid[q]: bit j of word q set when score 32q + j of the thread exists
  uint32_t valid[E / 32];
#pragma unroll
  for (int q = 0; q < E / 32; ++q) {
    const int m = min(max(nv - 32 * q, 0), 32);
    valid[q] = m >= 32 ? 0xffffffffu : ((1u << m) - 1u);
  }
  for (int i = t; i < kBins; i += kThreads) S.hist[i] = 0;
  __syncthreads();

  int grp = 0;
  // Block prefix of one packed count per thread: returns the count of lower
  // threads (packed) and the total; one barrier.
  auto block_prefix = [&](uint32_t c, uint32_t& before, uint32_t& total) {
    const uint32_t incl = warp_incl_scan(c);
    const int par = grp & 1;
    ++grp;
    if (lane == 31) S.tab[par][w] = incl;
    __syncthreads();
    const uint32_t e = lane < kWarps ? S.tab[par][lane] : 0u;
    before = __reduce_add_sync(0xffffffffu, lane < w ? e : 0u) + incl - c;
    total = __reduce_add_sync(0xffffffffu, e);
  };

  // ---- 1. sampled cutoff ------------------------------------------------------
  bool fast = false;
  uint32_t thr = 0;
  if (p.sample_mode != 1) {
    // Samples: scores 16 s (s < E / 16) of every thread that has them.
    const int a = (n + 15) / 16;  // scores at positions that are multiples of 16
    const float mu = static_cast<float>(kk) * static_cast<float>(a) * __frcp_rn(static_cast<float>(n));
    float rf = ceilf(mu + p.sample_z * sqrtf(mu)) + 1.0f;
    rf = fmaxf(rf, 1.0f);
    if (rf < static_cast<float>(a)) {
      fast = true;
      const uint32_t target = static_cast<uint32_t>(rf);
      uint32_t above, inbin;
#pragma unroll
      for (int s = 0; s < kSamples; ++s)
        hist_add(S.hist, 16 * s < nv ? (key[16 * s] >> 21) : 0xffffffffu);
      const uint32_t b1 = merged_find<1, 8>(S, target, &above, &inbin);
      const uint32_t rem = target - above;
      if (rem == inbin) {
        thr = b1 << 21;
      } else {
#pragma unroll
        for (int s = 0; s < kSamples; ++s) {
          const bool ok = 16 * s < nv && (key[16 * s] >> 21) == b1;
          hist_add(S.hist, ok ? ((key[16 * s] >> 10) & 0x7ffu) : 0xffffffffu);
        }
        const uint32_t b2 = merged_find<1, 8>(S, rem, &above, &inbin);
        thr = (b1 << 21) | (b2 << 10);
      }
    }
  }

  // ---- 2. filter into the stash, 3. exact cutoff and emission ----------------
  if (fast) {
    uint32_t hit[E / 32];
    uint32_t cnt = 0;
#pragma unroll
    for (int q = 0; q < E / 32; ++q) {
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) m |= static_cast<uint32_t>(key[32 * q + j] >= thr) << j;
      hit[q] = m & valid[q];
      cnt += __popc(hit[q]);
    }
    uint32_t before, total;
    block_prefix(cnt, before, total);
    if (total >= kk && total <= static_cast<uint32_t>(C)) {  // uniform
      uint32_t pos = before;
#pragma unroll
      for (int q = 0; q < E / 32; ++q) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if ((hit[q] >> j) & 1u) {
            S.skey[pos] = key[32 * q + j];
            S.sidx[pos] = static_cast<uint32_t>(first + 32 * q + j);
            ++pos;
          }
        }
      }
      if (PAGED) {  // the emission reads the row's page-table entries
        const int p1 = (n + p.page_size - 1) / p.page_size;
        for (int q = 32 * t; q < p1; q += 32 * kThreads) prefetch_l2(pt_row + q);
      }
      const Cut cut = select_stash<1>(S, static_cast<int>(total), kk);
      emit_rounds(S, static_cast<int>(total), cut, 0u, 0u, [&](uint32_t pos, uint32_t, uint32_t idx) {
        if (pos < kk) out_row[pos] = map_index(idx);
      });
      if (p.counters != nullptr && t == 0) atomicAdd(&p.counters[kCntSampled], 1u);
      return;
    }
    // too few or too many candidates: the exact path below
  }

  // ---- 4. exact register path --------------------------------------------------
  if (p.counters != nullptr && t == 0) atomicAdd(&p.counters[kCntShortExact], 1u);
  Cut cut;
  {
    uint32_t above, inbin;
#pragma unroll
    for (int j = 0; j < E; ++j) hist_add(S.hist, ((valid[j / 32] >> (j % 32)) & 1u) ? (key[j] >> 21) : 0xffffffffu);
    const uint32_t b1 = merged_find<1, 8>(S, kk, &above, &inbin);
    uint32_t rem = kk - above;
    if (rem == inbin) {
      cut = Cut{21, b1, rem, true};
    } else {
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const bool ok = ((valid[j / 32] >> (j % 32)) & 1u) && (key[j] >> 21) == b1;
        hist_add(S.hist, ok ? ((key[j] >> 10) & 0x7ffu) : 0xffffffffu);
      }
      const uint32_t b2 = merged_find<1, 8>(S, rem, &above, &inbin);
      const uint32_t p2 = (b1 << 11) | b2;
      rem -= above;
      if (rem == inbin) {
        cut = Cut{10, p2, rem, true};
      } else {
#pragma unroll
        for (int j = 0; j < E; ++j) {
          const bool ok = ((valid[j / 32] >> (j % 32)) & 1u) && (key[j] >> 10) == p2;
          hist_add(S.hist, ok ? (key[j] & 0x3ffu) : 0xffffffffu);
        }
        const uint32_t b3 = merged_find<1, 4>(S, rem, &above, &inbin);
        rem -= above;
        cut = Cut{0, (p2 << 10) | b3, rem, rem == inbin};
      }
    }
  }
  // Census: scores above the cut and the first r tied ones (index order).
  uint32_t gtm[E / 32], eqm[E / 32];
  uint32_t c = 0;
#pragma unroll
  for (int q = 0; q < E / 32; ++q) {
    uint32_t g = 0, e = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint32_t hi = key[32 * q + j] >> cut.shift;
      g |= static_cast<uint32_t>(hi > cut.P) << j;
      e |= static_cast<uint32_t>(hi == cut.P) << j;
    }
    gtm[q] = g & valid[q];
    eqm[q] = e & valid[q];
    c += (static_cast<uint32_t>(__popc(gtm[q])) << 16) + static_cast<uint32_t>(__popc(eqm[q]));
  }
  uint32_t before, total;
  block_prefix(c, before, total);
  uint32_t gb = before >> 16, eb = before & 0xffffu;
#pragma unroll
  for (int q = 0; q < E / 32; ++q) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const bool g = (gtm[q] >> j) & 1u, e = (eqm[q] >> j) & 1u;
      if (g || (e && eb < cut.r)) {
        const uint32_t pos = gb + min(eb, cut.r);
        if (pos < kk) out_row[pos] = map_index(static_cast<uint32_t>(first + 32 * q + j));
      }
      gb += g;
      eb += e;
    }
  }
}

}  // namespace tki
