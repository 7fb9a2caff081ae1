// Exact per-row top-k for short rows (at most 16384 FP32 scores): the
// prefill side of the indexer, where a batch holds thousands of
// rows of a few thousand scores each.
//
// The streaming kernel's per-row fixed costs (sample loads, ring set-up,
// three radix passes, emission rounds) are paid for every row, and with two
// rows in flight per SM they dominate rows this short. Here one CTA of 256
// threads takes a row and keeps it in registers, E scores per thread (E = 32:
// rows up to 8192; E = 64: up to 16384), so the row is read from HBM exactly
// once and every later step works on registers and a small shared-memory
// stash. Each warp owns a contiguous eighth of the row and reads it with
// 16-byte vector loads that cover 512 contiguous bytes per instruction; the
// (vector, lane, element) order of a warp's scores is their index order, and
// one packed warp scan turns per-vector hit counts into stash positions.
// The design follows the bf16 small-row top-k of the sglang PR 39648 report
// (实现拆解 2: one CTA per row, the row resident in registers, radix passes to
// the exact k-th value, page-table transform on output):
//
//  1. Coarse pass over the whole row (it is in registers, so this costs no
//     memory traffic): the 11-bit bin b1 of the k-th largest key, with the
//     counts above it and in it. If the whole bin is selected, the census
//     (4) follows at once.
//  2. Filter: the scores in or above bin b1 go to the stash as (key, index),
//     in index order (per-vector counts, one packed warp scan, one block
//     prefix over the warps).
//  3. The finer passes (11, then 10 bits) over the stash entries of bin b1
//     only, and emission in stash (= index) order with the streaming
//     kernel's emit_rounds. The 11-bit pass also counts its entries per
//     group of 32 bins, so that every warp finds its bin after one barrier
//     (the group among 64 sums, then the bin among 32) instead of scanning
//     all 2048 bins.
//  4. Exact register path: when bin b1 and above hold more entries than the
//     stash (ties, narrow rows), the finer passes run over the registers and
//     a census writes the selection straight from them.
//
// A sampled cutoff (the streaming kernel's) was tried here first and was
// slower: with the row already in registers, its two sample passes cost more
// than the exact coarse pass they replace.
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
  uint32_t hist[kBins];    // (emit_rounds' and the shared helpers' name for hbuf[0])
  uint32_t hist2[kBins];   // the second histogram buffer
  uint32_t sum64[64];      // pass-2 group sums: bins 32g .. 32g + 31 of hist2
  uint32_t tincl[kThreads];  // per-thread inclusive bin sums within the warp
  uint32_t tab[2][kWarps];
  uint32_t rtab[2][kWarps];
  uint32_t scan[kWarps];
  uint32_t res[4];
};

// Finds the bin holding the target-th largest element (1 <= target <= total)
// of histogram `hist` with two CTA barriers and no broadcast: each thread
// sums the BPT consecutive bins it owns, and after the second barrier every
// warp locates, from the warp totals and the per-thread sums, the thread and
// then the bin that holds the target, by itself. The bins are left as they
// are. With ClearOther each thread also zeroes its own bins of `other`, the
// buffer of the previous search, which every warp finished reading before
// the first barrier and which the next histogram fills after the second;
// without it the caller clears `other` itself, off this search's path (the
// coarse search: its stores there delayed the scan, ~3 % of the kernel).
// Returns the bin; *above = elements in higher bins; *inbin = elements in it.
template <int BPT, bool ClearOther = true, class SM>
__device__ uint32_t find_bin_all(SM& S, const uint32_t* hist, uint32_t* other, uint32_t target,
                                 uint32_t* above, uint32_t* inbin) {
  constexpr int nbins = BPT * kThreads;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int lo = nbins - BPT * (t + 1);  // lowest owned bin
  __syncthreads();  // the histogram is complete; the previous search is over in every warp
  uint32_t sum = 0;
#pragma unroll
  for (int q = 0; q < BPT; q += 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(&hist[lo + q]);
    sum += v.x + v.y + v.z + v.w;
  }
  // (all 2048 bins of the other buffer, whatever this search's bin count)
  if constexpr (ClearOther) {
    reinterpret_cast<uint4*>(&other[kBins - 8 * (t + 1)])[0] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(&other[kBins - 8 * (t + 1)])[1] = make_uint4(0, 0, 0, 0);
  }
  const uint32_t incl = warp_incl_scan(sum);
  S.tincl[t] = incl;
  if (lane == 31) S.scan[w] = incl;
  __syncthreads();
  // the warp, then the thread, then the bin (each search redone by every warp)
  const uint32_t e = lane < kWarps ? S.scan[lane] : 0u;
  const uint32_t ie = warp_incl_scan<kWarps>(e);
  const int ws = __ffs(__ballot_sync(0xffffffffu, lane < kWarps && ie >= target)) - 1;
  const uint32_t wbefore = __shfl_sync(0xffffffffu, ie - e, ws);
  const uint32_t ti = S.tincl[ws * 32 + lane];
  const int ls = __ffs(__ballot_sync(0xffffffffu, wbefore + ti >= target)) - 1;
  const uint32_t tprev = __shfl_sync(0xffffffffu, ti, ls > 0 ? ls - 1 : 0);
  const uint32_t tbefore = wbefore + (ls > 0 ? tprev : 0u);
  const int lo_s = nbins - BPT * (ws * 32 + ls + 1);
  const uint32_t c = lane < BPT ? hist[lo_s + BPT - 1 - lane] : 0u;  // descending bins
  const uint32_t ic = warp_incl_scan<BPT>(c);
  const int ib = __ffs(__ballot_sync(0xffffffffu, lane < BPT && tbefore + ic >= target)) - 1;
  *above = tbefore + __shfl_sync(0xffffffffu, ic - c, ib);
  *inbin = __shfl_sync(0xffffffffu, c, ib);
  return static_cast<uint32_t>(lo_s + BPT - 1 - ib);
}

// Finds the bin holding the target-th largest element of a 2048-bin
// histogram that carries per-group sums (sum64[g] = bins 32g .. 32g + 31),
// after one barrier and with no broadcast: every warp locates the group from
// the 64 sums, then the bin among its 32. The bins are left as they are.
__device__ __forceinline__ uint32_t find_bin_grouped(const uint32_t* hist, const uint32_t* sum64, uint32_t target,
                                                     uint32_t* above, uint32_t* inbin) {
  const int lane = threadIdx.x & 31;
  __syncthreads();  // the histogram and its sums are complete
  const uint2 g = *reinterpret_cast<const uint2*>(&sum64[62 - 2 * lane]);  // groups 62 - 2l, 63 - 2l
  const uint32_t s2 = g.x + g.y;
  const uint32_t inc = warp_incl_scan(s2);  // descending groups
  const int ls = __ffs(__ballot_sync(0xffffffffu, inc >= target)) - 1;
  uint32_t before = __shfl_sync(0xffffffffu, inc - s2, ls);
  const uint32_t gy = __shfl_sync(0xffffffffu, g.y, ls);
  int grp = 63 - 2 * ls;
  if (before + gy < target) {
    before += gy;
    --grp;
  }
  const uint32_t c = hist[32 * grp + 31 - lane];  // descending bins
  const uint32_t ic = warp_incl_scan(c);
  const int ib = __ffs(__ballot_sync(0xffffffffu, before + ic >= target)) - 1;
  *above = before + __shfl_sync(0xffffffffu, ic - c, ib);
  *inbin = __shfl_sync(0xffffffffu, c, ib);
  return static_cast<uint32_t>(32 * grp + 31 - ib);
}

// Histogram of stash keys into `hist`: entries e < n with (key >> fshift) ==
// fval add one to bin (key >> dshift) & dmask.
template <class SM>
__device__ void short_stash_hist(SM& S, uint32_t* hist, int n, uint32_t fshift, uint32_t fval,
                                 uint32_t dshift, uint32_t dmask) {
  for (int base0 = 0; base0 < n; base0 += kRoundEntries) {
    const int base = base0 + kRoundPerThread * threadIdx.x;
    uint32_t kv[kRoundPerThread];
    load_round(S.skey, base, n, kv);
#pragma unroll
    for (int c = 0; c < kRoundPerThread; ++c) {
      const uint32_t key = kv[c];
      if (base + c < n && (key >> fshift) == fval) atomicAdd(&hist[(key >> dshift) & dmask], 1u);
    }
  }
}

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
  int32_t page_shift;   // log2(page_size) when it is a power of two, else -1
  int32_t sample_mode;  // 0 automatic, 1 never (exact register path), 2 whenever possible
  float sample_z;
  uint32_t* counters;
  int32_t ahead;  // CTAs resident at once: the block that will take this CTA's slot next
};

// The keys of four consecutive scores (one 16-byte vector).
__device__ __forceinline__ void load_keys4(const float* p, uint32_t* key) {
  const float4 x = __ldg(reinterpret_cast<const float4*>(p));
  key[0] = order_key(x.x);
  key[1] = order_key(x.y);
  key[2] = order_key(x.z);
  key[3] = order_key(x.w);
}

// Positions in index order inside one warp. Lane l's vector q covers the
// warp's scores [q*32V + l*V, q*32V + l*V + V), so the warp's index order is
// (q, lane, element). Given each lane's hit count per vector, run() leaves,
// packed FB bits per vector, the hits of the lower lanes in each vector
// (exc) and the warp's hits in each vector (tot): one inclusive warp scan of
// PW packed words instead of one scan per vector.
template <int NQ, int V>
struct SlabScan {
  static constexpr int FB = (32 * V < 256) ? 8 : 16;  // a field holds up to 32 * V
  static constexpr int PW = (NQ * FB + 31) / 32;
  static constexpr uint32_t kMask = (1u << FB) - 1u;
  uint32_t exc[PW];
  uint32_t tot[PW];

  __device__ __forceinline__ void run(const uint32_t (&cnt)[NQ]) {
    uint32_t inc[PW];
#pragma unroll
    for (int i = 0; i < PW; ++i) inc[i] = 0;
#pragma unroll
    for (int q = 0; q < NQ; ++q) inc[(q * FB) / 32] |= cnt[q] << ((q * FB) % 32);
    uint32_t own[PW];
#pragma unroll
    for (int i = 0; i < PW; ++i) own[i] = inc[i];
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
      for (int i = 0; i < PW; ++i) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc[i], d);
        if (lane >= d) inc[i] += y;  // fields never carry: each sum is at most 32 * V
      }
    }
#pragma unroll
    for (int i = 0; i < PW; ++i) {
      tot[i] = __shfl_sync(0xffffffffu, inc[i], 31);
      exc[i] = inc[i] - own[i];
    }
  }
  __device__ __forceinline__ static uint32_t field(const uint32_t (&a)[PW], int q) {
    return (a[(q * FB) / 32] >> ((q * FB) % 32)) & kMask;
  }
};

template <int E, int KMAX, bool PAGED>
__global__ void __launch_bounds__(kThreads, E <= 32 ? (KMAX <= 1024 ? 5 : 4) : 3) topk_short_kernel(const ShortParams p) {
  constexpr int C = ShortCap<KMAX>::value;
  constexpr int V = 4;        // scores per 16-byte vector
  constexpr int NQ = E / V;  // vectors per lane
  constexpr int CH = 32 * E;  // scores per warp
  constexpr int NW = E / 32;  // words of per-score bit masks
  static_assert(E % 32 == 0 && E * kThreads <= kShortMaxRow, "a row must fit the CTA's registers");
  static_assert(32 % V == 0, "a vector's bits stay in one mask word");
  extern __shared__ __align__(128) unsigned char short_smem_raw[];
  ShortSmem<C>& S = *reinterpret_cast<ShortSmem<C>*>(short_smem_raw);

  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int row = static_cast<int>(blockIdx.x);
  // Start bringing the row of the block that will most likely take this
  // CTA's slot next into L2, so that its loads do not wait on HBM.
  if (t == 0 && p.ahead > 0 && row + p.ahead < p.B) {
    const int nr = row + p.ahead;
    const int64_t ln = p.lengths[nr];
    const int len = static_cast<int>(ln < 0 ? 0 : (ln > p.stride ? p.stride : ln));
    const char* base = reinterpret_cast<const char*>(static_cast<const float*>(p.scores) +
                                                     static_cast<int64_t>(nr) * p.stride);
    const uintptr_t a0 = (reinterpret_cast<uintptr_t>(base) + 15u) & ~static_cast<uintptr_t>(15u);
    const uintptr_t a1 = (reinterpret_cast<uintptr_t>(base) + static_cast<uintptr_t>(len) * sizeof(float)) &
                         ~static_cast<uintptr_t>(15u);
    if (a1 > a0) bulk_prefetch_l2(reinterpret_cast<const void*>(a0), static_cast<uint32_t>(a1 - a0));
  }
  const int64_t len_raw = p.lengths[row];
  const int n = static_cast<int>(len_raw < 0 ? 0 : (len_raw > p.stride ? p.stride : len_raw));
  int32_t* out_row = p.out + static_cast<int64_t>(row) * p.k;
  const int32_t* pt_row = PAGED ? p.page_table + static_cast<int64_t>(row) * p.pt_stride : nullptr;
  auto map_index = [&](uint32_t i) -> int32_t {  // read-only table loads
    if constexpr (!PAGED) return static_cast<int32_t>(i);
    const uint32_t ps = static_cast<uint32_t>(p.page_size);
    const uint32_t page = p.page_shift >= 0 ? (i >> p.page_shift) : i / ps;
    return static_cast<int32_t>(static_cast<int64_t>(__ldg(pt_row + page)) * ps + (i - page * ps));
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

  // ---- this lane's scores, as keys ------------------------------------------
  // Warp w owns the row's scores [w*CH, (w+1)*CH); key[q*V + c] is the score
  // at index w*CH + q*32V + lane*V + c, so each vector load of a warp reads
  // 512 contiguous bytes.
  const float* rp = static_cast<const float*>(p.scores) + static_cast<int64_t>(row) * p.stride;
  const int wbase = w * CH;
  auto index_of = [&](int q, int c) -> uint32_t {
    return static_cast<uint32_t>(wbase + q * 32 * V + lane * V + c);
  };
  uint32_t key[E];
  uint32_t valid[NW];
  const bool aligned = (reinterpret_cast<uintptr_t>(rp) & 15u) == 0;
  if (aligned) {
    // Every vector load is issued unconditionally, so that all of them are in
    // flight together: a vector that starts at or past the row's end re-reads
    // the row's first vector instead (an L1 hit) and is masked off below.
    // The vector holding the last score is the 16-byte block around it: it
    // can end up to 12 bytes past the row's stride when the stride is not a
    // whole number of vectors (never on another page); its scores past the
    // length are masked off too.
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int v0 = static_cast<int>(index_of(q, 0));
      load_keys4(rp + (v0 < n ? v0 : 0), &key[q * V]);
    }
    if (wbase + CH <= n) {  // warp-uniform: the whole warp lies inside the row
#pragma unroll
      for (int i = 0; i < NW; ++i) valid[i] = 0xffffffffu;
    } else {
#pragma unroll
      for (int i = 0; i < NW; ++i) valid[i] = 0;
#pragma unroll
      for (int j = 0; j < E; ++j)
        valid[j / 32] |= static_cast<uint32_t>(static_cast<int>(index_of(j / V, j % V)) < n) << (j % 32);
    }
  } else {
    // A row that does not start on 16 bytes: score by score, every load
    // predicated (none is a branch), so they are all in flight together.
#pragma unroll
    for (int i = 0; i < NW; ++i) valid[i] = 0;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int idx = static_cast<int>(index_of(j / V, j % V));
      const bool ok = idx < n;
      key[j] = order_key(__ldg(rp + (ok ? idx : 0)));
      valid[j / 32] |= static_cast<uint32_t>(ok) << (j % 32);
    }
  }
  const bool full = aligned && wbase + CH <= n;  // warp-uniform
  // (S.hist2 is cleared later, by each path before it adds into it.)
  for (int i = t; i < kBins / 4; i += kThreads) reinterpret_cast<uint4*>(S.hist)[i] = make_uint4(0, 0, 0, 0);
  if (t < 64) S.sum64[t] = 0;
  __syncthreads();

  int grp = 0;
  // Block prefix of one packed count per warp (the warp's lane 0 holds it):
  // returns the count of lower warps (packed) and the total; one barrier.
  auto warp_prefix = [&](uint32_t c, uint32_t& before, uint32_t& total) {
    const int par = grp & 1;
    ++grp;
    if (lane == 0) S.tab[par][w] = c;
    __syncthreads();
    const uint32_t e = lane < kWarps ? S.tab[par][lane] : 0u;
    before = __reduce_add_sync(0xffffffffu, lane < w ? e : 0u);
    total = __reduce_add_sync(0xffffffffu, e);
  };
  auto vec_bits = [&](const uint32_t (&m)[NW], int q) -> uint32_t {
    return (m[(q * V) / 32] >> ((q * V) % 32)) & ((1u << V) - 1u);
  };

  // ---- 1. the coarse bin of the k-th largest score, over the whole row -------
  uint32_t above, inbin;
  if (full) {
#pragma unroll
    for (int j = 0; j < E; ++j) atomicAdd(&S.hist[key[j] >> 21], 1u);
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j) hist_add(S.hist, ((valid[j / 32] >> (j % 32)) & 1u) ? (key[j] >> 21) : 0xffffffffu);
  }
  // Searches alternate between the two buffers: S.hist, S.hist2, S.hist.
  const uint32_t b1 = find_bin_all<8, false>(S, S.hist, S.hist2, kk, &above, &inbin);
  uint32_t rem = kk - above;
  Cut cut;
  if (rem == inbin) {
    cut = Cut{21, b1, rem, true};  // the whole bin is selected: straight to the census
  } else if (p.sample_mode != 1 && above + inbin <= static_cast<uint32_t>(C)) {
    // ---- 2. the scores in or above that bin go to the stash, in index order --
    uint32_t hit[NW];
    const uint32_t lo1 = b1 << 21;  // the lowest key of bin b1
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) m |= static_cast<uint32_t>(key[32 * i + j] >= lo1) << j;
      hit[i] = m & valid[i];
    }
    uint32_t cnt[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) cnt[q] = __popc(vec_bits(hit, q));
    SlabScan<NQ, V> sc;
    sc.run(cnt);
    uint32_t wt = 0;
#pragma unroll
    for (int q = 0; q < NQ; ++q) wt += SlabScan<NQ, V>::field(sc.tot, q);
    uint32_t before, total;
    warp_prefix(wt, before, total);  // total == above + inbin
    uint32_t vbase = before;  // the warp's hits in the vectors before q
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      uint32_t pos = vbase + SlabScan<NQ, V>::field(sc.exc, q);
      const uint32_t m = vec_bits(hit, q);
#pragma unroll
      for (int c = 0; c < V; ++c) {
        if ((m >> c) & 1u) {
          S.skey[pos] = key[q * V + c];
          S.sidx[pos] = index_of(q, c);
          ++pos;
        }
      }
      vbase += SlabScan<NQ, V>::field(sc.tot, q);
    }
    if (PAGED) {  // the emission reads the row's page-table entries
      const int p1 = (n + p.page_size - 1) / p.page_size;
      for (int q = 32 * t; q < p1; q += 32 * kThreads) prefetch_l2(pt_row + q);
    }
    reinterpret_cast<uint4*>(&S.hist2[8 * t])[0] = make_uint4(0, 0, 0, 0);  // for the second pass
    reinterpret_cast<uint4*>(&S.hist2[8 * t])[1] = make_uint4(0, 0, 0, 0);
    // ---- 3. the exact cutoff inside bin b1 (its entries only), emission -------
    __syncthreads();  // the stash is complete, the second histogram clear
    for (int base0 = 0; base0 < static_cast<int>(total); base0 += kRoundEntries) {
      const int base = base0 + kRoundPerThread * t;
      uint32_t kv[kRoundPerThread];
      load_round(S.skey, base, static_cast<int>(total), kv);
#pragma unroll
      for (int c = 0; c < kRoundPerThread; ++c) {
        if (base + c < static_cast<int>(total) && (kv[c] >> 21) == b1) {
          atomicAdd(&S.hist2[(kv[c] >> 10) & 0x7ffu], 1u);
          atomicAdd(&S.sum64[(kv[c] >> 15) & 63u], 1u);
        }
      }
    }
    const uint32_t b2 = find_bin_grouped(S.hist2, S.sum64, rem, &above, &inbin);
    const uint32_t p2 = (b1 << 11) | b2;
    rem -= above;
    if (rem == inbin) {
      cut = Cut{10, p2, rem, true};
    } else {
      // S.hist still holds the coarse counts: clear it for this third pass
      // (every warp is past the search that read it).
      reinterpret_cast<uint4*>(&S.hist[8 * t])[0] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(&S.hist[8 * t])[1] = make_uint4(0, 0, 0, 0);
      __syncthreads();
      short_stash_hist(S, S.hist, static_cast<int>(total), 10, p2, 0, 0x3ff);
      const uint32_t b3 = find_bin_all<4>(S, S.hist, S.hist2, rem, &above, &inbin);
      rem -= above;
      cut = Cut{0, (p2 << 10) | b3, rem, rem == inbin};
    }
    emit_rounds(S, static_cast<int>(total), cut, 0u, 0u, [&](bool sel, uint32_t pos, uint32_t, uint32_t idx) {
      const int32_t v = map_index(idx);
      if (sel && pos < kk) out_row[pos] = v;
    });
    return;
  } else {
    // ---- 4. exact register path: the finer passes over the registers --------
    reinterpret_cast<uint4*>(&S.hist2[8 * t])[0] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(&S.hist2[8 * t])[1] = make_uint4(0, 0, 0, 0);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const bool ok = ((valid[j / 32] >> (j % 32)) & 1u) && (key[j] >> 21) == b1;
      hist_add(S.hist2, ok ? ((key[j] >> 10) & 0x7ffu) : 0xffffffffu);
    }
    const uint32_t b2 = find_bin_all<8>(S, S.hist2, S.hist, rem, &above, &inbin);
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
      const uint32_t b3 = find_bin_all<4>(S, S.hist, S.hist2, rem, &above, &inbin);
      rem -= above;
      cut = Cut{0, (p2 << 10) | b3, rem, rem == inbin};
    }
  }
  // Census: scores above the cut and the first r tied ones (index order).
  if (p.counters != nullptr && t == 0) atomicAdd(&p.counters[kCntShortExact], 1u);
  uint32_t gtm[NW], eqm[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    uint32_t g = 0, e = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint32_t hi = key[32 * i + j] >> cut.shift;
      g |= static_cast<uint32_t>(hi > cut.P) << j;
      e |= static_cast<uint32_t>(hi == cut.P) << j;
    }
    gtm[i] = g & valid[i];
    eqm[i] = e & valid[i];
  }
  uint32_t cg[NQ], ce[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    cg[q] = __popc(vec_bits(gtm, q));
    ce[q] = __popc(vec_bits(eqm, q));
  }
  SlabScan<NQ, V> sg, se;
  sg.run(cg);
  se.run(ce);
  uint32_t wg = 0, we = 0;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    wg += SlabScan<NQ, V>::field(sg.tot, q);
    we += SlabScan<NQ, V>::field(se.tot, q);
  }
  uint32_t before, total;
  warp_prefix((wg << 16) | we, before, total);
  uint32_t gbase = before >> 16, ebase = before & 0xffffu;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    uint32_t gb = gbase + SlabScan<NQ, V>::field(sg.exc, q);
    uint32_t eb = ebase + SlabScan<NQ, V>::field(se.exc, q);
    const uint32_t mg = vec_bits(gtm, q), me = vec_bits(eqm, q);
#pragma unroll
    for (int c = 0; c < V; ++c) {
      const bool g = (mg >> c) & 1u, e = (me >> c) & 1u;
      if (g || (e && eb < cut.r)) {
        const uint32_t pos = gb + min(eb, cut.r);
        if (pos < kk) out_row[pos] = map_index(index_of(q, c));
      }
      gb += g;
      eb += e;
    }
    gbase += SlabScan<NQ, V>::field(sg.tot, q);
    ebase += SlabScan<NQ, V>::field(se.tot, q);
  }
}

}  // namespace tki
