// Plain CPU oracle for batched, ragged, exact per-row top-k over FP32 scores.
//
// TEST INFRASTRUCTURE ONLY. The tests, the package's smoke check and the
// benchmark's CPU-baseline leg call this file; the product path never does.
// It shares no code, header or constant with the CUDA implementation.
//
// What it computes is the plain definition, by a full sort of every row:
//
//   n = clamp(lengths[b], 0, stride)            (negative length = no token)
//   m = min(k, n)
//   order = [0, n) sorted by score, best first, under the total order
//           "larger float ranks higher; +0 ranks above -0"; equal scores keep
//           ascending index order
//   out[b, j] = order[j] for j < m, and -1 for m <= j < k
//   paged:  out[b, j] = page_table[b, i / page_size] * page_size + i % page_size
//           for every valid i = order[j]; -1 slots stay -1
//
// Passages followed:
//  * vLLM issue "persistent_topk silently drops top-k candidates when many
//    values share a coarse histogram bin", 验证方法: the selected values, gathered
//    and sorted, must equal the exact top-k values; repeated calls agree.
//  * vLLM PR 56346 (sampled filtering), 实现拆解 4-5: invalid slots are -1, no
//    duplicate indices, strict equality with an exact top-k; lengths of -1
//    and beyond the width appear in its boundary list.
//  * sglang PR 39648 report, topk.py docstring of topk_transform_bf16_small:
//    row b selects the k best of its first seq_lens[b] scores; index i is
//    written as page_table[b, i // page_size] * page_size + i % page_size; -1
//    fills the slots past min(k, seq_lens[b]); which tied element fills the
//    last slots is arbitrary (this oracle takes the lowest indices).
//  * sglang PR 37625, 评论: signed zero and -inf are part of the coverage;
//    sglang PR 39648, 功能与动机: -inf is a legal score that must not be
//    squeezed out by padding.
//
// NaN is outside the contract. A NaN inside a row's valid prefix makes the
// call return ORACLE_ENAN instead of guessing an order for it.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <numeric>
#include <vector>

namespace {

constexpr int ORACLE_OK = 0;
constexpr int ORACLE_EARG = 1;
constexpr int ORACLE_ENAN = 2;
constexpr int ORACLE_EPAGE = 3;

// True when score a ranks strictly above score b (neither is NaN).
bool ranks_above(float a, float b) {
  if (a > b) return true;
  if (a < b) return false;
  return !std::signbit(a) && std::signbit(b);  // equal floats: only +0 vs -0 differ
}

int64_t valid_length(int32_t len, int64_t stride) {
  if (len < 0) return 0;
  return std::min<int64_t>(len, stride);
}

// Writes the m = min(k, n) best indices of row[0, n) best first, then -1.
int select_row(const float* row, int64_t n, int32_t k, int32_t* out_row) {
  for (int64_t i = 0; i < n; ++i) {
    if (std::isnan(row[i])) return ORACLE_ENAN;
  }
  std::vector<int32_t> order(static_cast<size_t>(n));
  std::iota(order.begin(), order.end(), 0);
  std::sort(order.begin(), order.end(), [row](int32_t i, int32_t j) {
    if (ranks_above(row[i], row[j])) return true;
    if (ranks_above(row[j], row[i])) return false;
    return i < j;
  });
  const int64_t m = std::min<int64_t>(k, n);
  for (int64_t j = 0; j < m; ++j) out_row[j] = order[static_cast<size_t>(j)];
  for (int64_t j = m; j < k; ++j) out_row[j] = -1;
  return ORACLE_OK;
}

// Maps a row index through the page table. Fails when the page lies past the
// table's row or the slot does not fit in int32.
int page_map(int32_t idx, const int32_t* pt_row, int64_t pt_stride, int32_t page_size,
             int32_t* slot_out) {
  const int64_t page = idx / page_size;
  if (page >= pt_stride) return ORACLE_EPAGE;
  const int64_t slot = static_cast<int64_t>(pt_row[page]) * page_size + idx % page_size;
  if (slot < INT32_MIN || slot > INT32_MAX) return ORACLE_EPAGE;
  *slot_out = static_cast<int32_t>(slot);
  return ORACLE_OK;
}

}  // namespace

extern "C" {

int oracle_abi_version(void) { return 2; }

int oracle_topk_ragged(const float* scores, int64_t stride, const int32_t* lengths, int32_t B,
                       int32_t k, int32_t* out) {
  if (B < 0 || k < 1 || stride < 1) return ORACLE_EARG;
  if (B > 0 && (scores == nullptr || lengths == nullptr || out == nullptr)) return ORACLE_EARG;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t n = valid_length(lengths[b], stride);
    const int rc = select_row(scores + static_cast<int64_t>(b) * stride, n, k,
                              out + static_cast<int64_t>(b) * k);
    if (rc != ORACLE_OK) return rc;
  }
  return ORACLE_OK;
}

int oracle_topk_paged(const float* scores, int64_t stride, const int32_t* lengths, int32_t B,
                      int32_t k, const int32_t* page_table, int64_t pt_stride, int32_t page_size,
                      int32_t* out) {
  if (page_size < 1 || pt_stride < 1) return ORACLE_EARG;
  if (B > 0 && page_table == nullptr) return ORACLE_EARG;
  const int rc = oracle_topk_ragged(scores, stride, lengths, B, k, out);
  if (rc != ORACLE_OK) return rc;
  for (int32_t b = 0; b < B; ++b) {
    int32_t* out_row = out + static_cast<int64_t>(b) * k;
    const int32_t* pt_row = page_table + static_cast<int64_t>(b) * pt_stride;
    for (int32_t j = 0; j < k; ++j) {
      if (out_row[j] < 0) continue;
      const int prc = page_map(out_row[j], pt_row, pt_stride, page_size, &out_row[j]);
      if (prc != ORACLE_OK) return prc;
    }
  }
  return ORACLE_OK;
}

// ---------------------------------------------------------------------------
// The two-level indexer's helpers on either side of the selection (sglang PR
// 39648 report, 实现拆解 2 table, and the `amax8_varlen` /
// `sort_candidate_blocks` docstrings of candidate_table.py).

// Level-one keys. For row b: n = clamp(lengths[b], 0, stride) scores,
// nb = ceil(n / 8) blocks of 8 consecutive scores. If topk > 0 and
// nb <= topk the row is left untouched (every block is selected anyway).
// Otherwise out[b, i] = the largest of scores[b, 8i .. 8i + 8) for i < nb - 1,
// and out[b, nb - 1] = +inf (the newest block is always selected); slots from
// nb on are not written. out rows are out_stride >= ceil(stride / 8) floats.
// "Largest" is taken in the same total order as the selection (+0 above -0):
// the page names fmaxf, which leaves the sign of a zero maximum open, and this
// reading makes the key independent of the order of the block's scores.
int oracle_amax8_varlen(const float* scores, int64_t stride, const int32_t* lengths, int32_t B,
                        int32_t topk, float* out, int64_t out_stride) {
  if (B < 0 || stride < 1 || topk < 0 || out_stride < (stride + 7) / 8) return ORACLE_EARG;
  if (B > 0 && (scores == nullptr || lengths == nullptr || out == nullptr)) return ORACLE_EARG;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t n = valid_length(lengths[b], stride);
    const int64_t nb = (n + 7) / 8;
    if (nb == 0 || (topk > 0 && nb <= topk)) continue;
    const float* row = scores + static_cast<int64_t>(b) * stride;
    float* out_row = out + static_cast<int64_t>(b) * out_stride;
    for (int64_t i = 0; i < nb - 1; ++i) {
      float m = row[8 * i];
      for (int64_t j = 8 * i; j < 8 * i + 8; ++j) {
        if (std::isnan(row[j])) return ORACLE_ENAN;
        if (ranks_above(row[j], m)) m = row[j];
      }
      out_row[i] = m;
    }
    out_row[nb - 1] = INFINITY;
  }
  return ORACLE_OK;
}

// Block table. For row b: nb = ceil(clamp(lengths[b], 0, stride) / 8) and
// m = min(k, nb). If nb <= k the table is the identity: blocks[b, j] = j for
// j < nb, whatever the input. Otherwise the input row holds m distinct block
// ids in [0, nb) in any order, -1 padded, and they are rewritten in
// ascending order. Slots from m on hold INT32_MAX. out_pages[b, j] is the
// pool slot of block blocks[b, j], page_table[b, id / bpp] * bpp + id % bpp
// with bpp = page_size / 8 (page_size a power of two >= 8), and INT32_MAX in
// the padded slots. A malformed input row (duplicate or out-of-range ids,
// a wrong count) is an argument error.
int oracle_sort_candidate_blocks(int32_t* blocks, int32_t B, int32_t k, const int32_t* lengths,
                                 int64_t stride, const int32_t* page_table, int64_t pt_stride,
                                 int32_t page_size, int32_t* out_pages) {
  if (B < 0 || k < 1 || stride < 1 || page_size < 8 || (page_size & (page_size - 1)) != 0)
    return ORACLE_EARG;
  if (B > 0 && (blocks == nullptr || lengths == nullptr || page_table == nullptr ||
                out_pages == nullptr))
    return ORACLE_EARG;
  const int64_t bpp = page_size / 8;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t nb = (valid_length(lengths[b], stride) + 7) / 8;
    const int64_t m = std::min<int64_t>(k, nb);
    int32_t* row = blocks + static_cast<int64_t>(b) * k;
    std::vector<int32_t> ids;
    if (nb <= k) {
      for (int64_t j = 0; j < nb; ++j) ids.push_back(static_cast<int32_t>(j));
    } else {
      for (int32_t j = 0; j < k; ++j) {
        if (row[j] < 0) continue;
        if (row[j] >= nb) return ORACLE_EARG;
        ids.push_back(row[j]);
      }
      std::sort(ids.begin(), ids.end());
      if (static_cast<int64_t>(ids.size()) != m) return ORACLE_EARG;
      for (size_t j = 1; j < ids.size(); ++j)
        if (ids[j] == ids[j - 1]) return ORACLE_EARG;
    }
    const int32_t* pt_row = page_table + static_cast<int64_t>(b) * pt_stride;
    int32_t* pages = out_pages + static_cast<int64_t>(b) * k;
    for (int32_t j = 0; j < k; ++j) {
      if (j < m) {
        const int64_t id = ids[static_cast<size_t>(j)];
        const int64_t page = id / bpp;
        if (page >= pt_stride) return ORACLE_EPAGE;
        const int64_t slot = static_cast<int64_t>(pt_row[page]) * bpp + id % bpp;
        if (slot < INT32_MIN || slot > INT32_MAX) return ORACLE_EPAGE;
        row[j] = static_cast<int32_t>(id);
        pages[j] = static_cast<int32_t>(slot);
      } else {
        row[j] = INT32_MAX;
        pages[j] = INT32_MAX;
      }
    }
  }
  return ORACLE_OK;
}

}  // extern "C"
