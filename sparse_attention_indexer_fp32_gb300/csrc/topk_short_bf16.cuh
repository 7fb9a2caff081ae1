// Exact per-row top-k for short rows of BF16 scores (at most 16384 each):
// the bf16 small-row top-k of the sglang PR 39648 report (实现拆解 2: one CTA
// per row, the row resident in registers, radix passes over the bf16 bits to
// the exact k-th value, census, page-table transform on output).
//
// The order-preserving key of a BF16 score is 16 bits wide: the high half of
// the FP32 key of the same value, so the two kernels rank alike (+0 above
// -0, lowest indices first among equal scores) and give the same result for
// the same scores. Two keys share a register, and the radix is 11 + 5 bits:
//
//  1. Coarse pass over the row in registers: the 11-bit bin b1 of the k-th
//     largest key (2048 bins), with the counts above it and in it. If the
//     whole bin is selected the census (4) follows at once.
//  2. Filter: the scores in or above b1 go to the stash as one word each,
//     key << 16 | index (a row holds at most 16384 scores), in index order.
//  3. Fine pass over the stash entries of b1: a 32-bin histogram of the low
//     5 key bits, which every warp searches by itself. The cut is then a
//     whole key; the entries above it and the first r equal to it (in index
//     order) are written in index order.
//  4. When b1 and above hold more entries than the stash (ties, narrow rows),
//     the fine pass and a census run over the registers instead.
//
// A slot past the row's end holds key 0. Only a negative NaN has a key below
// that of -inf (0x007f, bin 3), and NaN is excluded, so key 0 sits in bin 0,
// below every score of the row: no pass needs a validity mask. The coarse
// pass counts those slots in bin 0, which is never the cutoff's bin (the row
// has more than k scores when the passes run), the filter and the census
// compare against a bin or cut above it, and the fine passes take bin b1
// only.
#pragma once

#include <cstdint>

#include "topk_short.cuh"

namespace tki {

template <int C>
struct ShortSmemBf16 {
  uint32_t ent[C];           // stash entries: key << 16 | index
  uint32_t hist[kBins];
  uint32_t hist2[kBins];
  uint32_t tincl[kThreads];
  uint32_t tab[2][kWarps];
  uint32_t rtab[2][kWarps];
  uint32_t scan[kWarps];
  uint32_t res[4];
};

// Keys of the two BF16 scores in a word (low half: the lower index): a
// negative score's bits are inverted, a positive one's sign bit set.
__device__ __forceinline__ uint32_t bf16x2_keys(uint32_t w) {
  uint32_t m;
  // each half filled with the sign of its score (byte sign replication)
  asm("prmt.b32 %0, %1, %2, 0xBB99;" : "=r"(m) : "r"(w), "r"(0u));
  return w ^ (m | 0x80008000u);
}

// Key (16 bits) of half h of packed word w.
__device__ __forceinline__ uint32_t half_key(uint32_t w, int h) { return h ? (w >> 16) : (w & 0xffffu); }

// The bin (of 32, descending search) holding the target-th largest entry of
// a 32-bin histogram; every warp runs it after a barrier.
__device__ __forceinline__ uint32_t find_bin32(const uint32_t* hist32, uint32_t target, uint32_t* above,
                                               uint32_t* inbin) {
  const int lane = threadIdx.x & 31;
  const uint32_t c = hist32[31 - lane];
  const uint32_t ic = warp_incl_scan(c);
  const int ib = __ffs(__ballot_sync(0xffffffffu, ic >= target)) - 1;
  *above = __shfl_sync(0xffffffffu, ic - c, ib);
  *inbin = __shfl_sync(0xffffffffu, c, ib);
  return static_cast<uint32_t>(31 - ib);
}

template <int E, int KMAX, bool PAGED>
__global__ void __launch_bounds__(kThreads, E <= 32 ? 6 : 4) topk_short_bf16_kernel(const ShortParams p) {
  constexpr int C = ShortCap<KMAX>::value;
  constexpr int V = 8;        // scores per 16-byte vector
  constexpr int NQ = E / V;   // vectors per lane
  constexpr int NKW = E / 2;  // packed key words per lane
  constexpr int CH = 32 * E;  // scores per warp
  constexpr int NW = E / 32;  // words of per-score bit masks
  static_assert(E % 32 == 0 && E * kThreads <= kShortMaxRow, "a row must fit the CTA's registers");
  extern __shared__ __align__(128) unsigned char short_smem_raw[];
  ShortSmemBf16<C>& S = *reinterpret_cast<ShortSmemBf16<C>*>(short_smem_raw);

  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int row = static_cast<int>(blockIdx.x);
  if (t == 0 && p.ahead > 0 && row + p.ahead < p.B) {
    const int nr = row + p.ahead;
    const int64_t ln = p.lengths[nr];
    const int len = static_cast<int>(ln < 0 ? 0 : (ln > p.stride ? p.stride : ln));
    const char* base = reinterpret_cast<const char*>(static_cast<const uint16_t*>(p.scores) +
                                                     static_cast<int64_t>(nr) * p.stride);
    const uintptr_t a0 = (reinterpret_cast<uintptr_t>(base) + 15u) & ~static_cast<uintptr_t>(15u);
    const uintptr_t a1 = (reinterpret_cast<uintptr_t>(base) + static_cast<uintptr_t>(len) * 2u) &
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
    const uint32_t page = p.page_shift >= 0 ? (i >> p.page_shift) : i / ps;
    return static_cast<int32_t>(static_cast<int64_t>(__ldg(pt_row + page)) * ps + (i - page * ps));
  };
  if (p.counters != nullptr && t == 0) {
    atomicAdd(&p.counters[kCntRows], 1u);
    atomicAdd(&p.counters[kCntShortRows], 1u);
  }
  if (n <= p.k) {
    for (int j = t; j < p.k; j += kThreads) out_row[j] = (j < n) ? map_index(static_cast<uint32_t>(j)) : -1;
    if (p.counters != nullptr && t == 0) atomicAdd(&p.counters[kCntTrivial], 1u);
    return;
  }
  const uint32_t kk = static_cast<uint32_t>(p.k);

  // ---- this lane's keys, two per word ----------------------------------------
  // Warp w owns scores [w*CH, (w+1)*CH); score j of the lane (bit j of the
  // masks) is index w*CH + (j/8)*256 + lane*8 + j%8, held in half j%2 of
  // word j/2.
  const uint16_t* rp = static_cast<const uint16_t*>(p.scores) + static_cast<int64_t>(row) * p.stride;
  const int wbase = w * CH;
  auto index_of = [&](int j) -> uint32_t { return static_cast<uint32_t>(wbase + (j / V) * 32 * V + lane * V + j % V); };
  uint32_t kw[NKW];
  const bool aligned = (reinterpret_cast<uintptr_t>(rp) & 15u) == 0;
  if (aligned) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int v0 = static_cast<int>(index_of(q * V));
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(rp + (v0 < n ? v0 : 0)));
      kw[4 * q + 0] = bf16x2_keys(x.x);
      kw[4 * q + 1] = bf16x2_keys(x.y);
      kw[4 * q + 2] = bf16x2_keys(x.z);
      kw[4 * q + 3] = bf16x2_keys(x.w);
    }
    if (wbase + CH > n) {  // warp-uniform: slots past the row's end get key 0
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const int have = n - static_cast<int>(index_of(q * V));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t lo = 2 * i < have ? 0x0000ffffu : 0u, hi = 2 * i + 1 < have ? 0xffff0000u : 0u;
          kw[4 * q + i] &= lo | hi;
        }
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < NKW; ++i) {
      const int i0 = static_cast<int>(index_of(2 * i)), i1 = i0 + 1;
      const uint32_t lo = __ldg(rp + (i0 < n ? i0 : 0)), hi = __ldg(rp + (i1 < n ? i1 : 0));
      kw[i] = bf16x2_keys(lo | (hi << 16)) & ((i0 < n ? 0x0000ffffu : 0u) | (i1 < n ? 0xffff0000u : 0u));
    }
  }
  // (S.hist2 is cleared later, by each path before it adds into it.)
  for (int i = t; i < kBins / 4; i += kThreads) reinterpret_cast<uint4*>(S.hist)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();

  int grp = 0;
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

  // ---- 1. coarse bin (top 11 bits of the key) ----------------------------------
  uint32_t above, inbin;
#pragma unroll
  for (int i = 0; i < NKW; ++i) {
    atomicAdd(&S.hist[(kw[i] >> 5) & 0x7ffu], 1u);
    atomicAdd(&S.hist[kw[i] >> 21], 1u);
  }
  const uint32_t b1 = find_bin_all<8, false>(S, S.hist, S.hist2, kk, &above, &inbin);
  uint32_t rem = kk - above;
  Cut cut;
  if (rem == inbin) {
    cut = Cut{5, b1, rem, true};
  } else if (p.sample_mode != 1 && above + inbin <= static_cast<uint32_t>(C)) {
    // ---- 2. stash: key << 16 | index for the scores in or above bin b1 --------
    const uint32_t LO = b1 << 21;  // the lowest key of b1, in the high half
    uint32_t hit[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) hit[i] = 0;
#pragma unroll
    for (int i = 0; i < NKW; ++i) {
      const uint32_t h2 = static_cast<uint32_t>((kw[i] << 16) >= LO) | (static_cast<uint32_t>(kw[i] >= LO) << 1);
      hit[(2 * i) / 32] |= h2 << ((2 * i) % 32);
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
    warp_prefix(wt, before, total);
    uint32_t vbase = before;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      uint32_t pos = vbase + SlabScan<NQ, V>::field(sc.exc, q);
      const uint32_t m = vec_bits(hit, q);
#pragma unroll
      for (int c = 0; c < V; ++c) {
        if ((m >> c) & 1u) {
          const uint32_t wd = kw[(q * V + c) / 2];
          S.ent[pos] = ((c & 1) ? (wd & 0xffff0000u) : (wd << 16)) | index_of(q * V + c);
          ++pos;
        }
      }
      vbase += SlabScan<NQ, V>::field(sc.tot, q);
    }
    if (PAGED) {
      const int p1 = (n + p.page_size - 1) / p.page_size;
      for (int q = 32 * t; q < p1; q += 32 * kThreads) prefetch_l2(pt_row + q);
    }
    if (t < 8) reinterpret_cast<uint4*>(&S.hist2[4 * t])[0] = make_uint4(0, 0, 0, 0);
    // ---- 3. fine pass: low 5 bits of the b1 entries, then emission ------------
    __syncthreads();
    const int nt = static_cast<int>(total);
    for (int base0 = 0; base0 < nt; base0 += kRoundEntries) {
      const int base = base0 + kRoundPerThread * t;
      uint32_t ev[kRoundPerThread];
      load_round(S.ent, base, nt, ev);
#pragma unroll
      for (int c = 0; c < kRoundPerThread; ++c)
        if (base + c < nt && (ev[c] >> 21) == b1) atomicAdd(&S.hist2[(ev[c] >> 16) & 31u], 1u);
    }
    __syncthreads();
    const uint32_t b2 = find_bin32(S.hist2, rem, &above, &inbin);
    rem -= above;
    const uint32_t P = (b1 << 5) | b2;
    const bool all = rem == inbin;
    // Emission in stash (= index) order: entries above the cut, then the
    // first rem equal to it. A round gives each thread kRoundPerThread
    // consecutive entries, ordered by one warp scan of packed counts.
    const uint32_t gt_from = all ? P : P + 1u;  // P + 1 <= 0x10000: no wrap
    uint32_t run_gt = 0, run_eq = 0;
    int par = 0;
    for (int base0 = 0; base0 < nt; base0 += kRoundEntries, par ^= 1) {
      const int base = base0 + kRoundPerThread * t;
      uint32_t ev[kRoundPerThread];
      load_round(S.ent, base, nt, ev);
      uint32_t gtm = 0, eqm = 0;
#pragma unroll
      for (int c = 0; c < kRoundPerThread; ++c) {
        const bool ok = base + c < nt;
        const uint32_t key = ev[c] >> 16;
        gtm |= static_cast<uint32_t>(ok && key >= gt_from) << c;
        eqm |= static_cast<uint32_t>(ok && !all && key == P) << c;
      }
      const uint32_t own = (static_cast<uint32_t>(__popc(gtm)) << 16) | static_cast<uint32_t>(__popc(eqm));
      const uint32_t incl = warp_incl_scan(own);
      if (lane == 31) S.rtab[par][w] = incl;
      __syncthreads();
      const uint32_t e = lane < kWarps ? S.rtab[par][lane] : 0u;
      const uint32_t bef = __reduce_add_sync(0xffffffffu, lane < w ? e : 0u) + incl - own;
      const uint32_t tot = __reduce_add_sync(0xffffffffu, e);
      uint32_t gb = run_gt + (bef >> 16);
      uint32_t eb = run_eq + (bef & 0xffffu);
#pragma unroll
      for (int c = 0; c < kRoundPerThread; ++c) {
        const bool gt = (gtm >> c) & 1u, eq = (eqm >> c) & 1u;
        const int32_t v = map_index(base + c < nt ? (ev[c] & 0xffffu) : 0u);
        const uint32_t pos = gb + min(eb, rem);
        if ((gt || (eq && eb < rem)) && pos < kk) out_row[pos] = v;
        gb += gt;
        eb += eq;
      }
      run_gt += tot >> 16;
      run_eq += tot & 0xffffu;
    }
    return;
  } else {
    // ---- 4. register path: the fine pass over the registers ---------------------
    if (t < 8) reinterpret_cast<uint4*>(&S.hist2[4 * t])[0] = make_uint4(0, 0, 0, 0);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NKW; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t key = half_key(kw[i], h);
        hist_add(S.hist2, (key >> 5) == b1 ? (key & 31u) : 0xffffffffu);
      }
    }
    __syncthreads();
    const uint32_t b2 = find_bin32(S.hist2, rem, &above, &inbin);
    rem -= above;
    cut = Cut{0, (b1 << 5) | b2, rem, rem == inbin};
  }
  // Census over the registers: keys above the cut and the first r tied ones.
  if (p.counters != nullptr && t == 0) atomicAdd(&p.counters[kCntShortExact], 1u);
  uint32_t gtm[NW], eqm[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) gtm[i] = eqm[i] = 0;
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const uint32_t hi = half_key(kw[j / 2], j % 2) >> cut.shift;
    gtm[j / 32] |= static_cast<uint32_t>(hi > cut.P) << (j % 32);
    eqm[j / 32] |= static_cast<uint32_t>(hi == cut.P) << (j % 32);
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
        if (pos < kk) out_row[pos] = map_index(index_of(q * V + c));
      }
      gb += g;
      eb += e;
    }
    gbase += SlabScan<NQ, V>::field(sg.tot, q);
    ebase += SlabScan<NQ, V>::field(se.tot, q);
  }
}

}  // namespace tki
