/*
 * topk_indexer.h - C ABI of the GB300 (sm_103a) batched, ragged, exact per-row
 * top-k over FP32 sparse-attention indexer scores.
 *
 * The operation (vLLM PR 56346 "sampled filtering", 执行摘要 and 实现拆解 1-3;
 * sglang PR 39648 report, topk.py docstring of the paged top-k transform):
 *
 *   for every row b in [0, B):
 *     n_b  = clamp(lengths[b], 0, stride)      negative length = no token,
 *                                              a length past the width is clamped
 *     m_b  = min(k, n_b)
 *     out[b, 0 .. m_b)  = the indices (in [0, n_b)) of the m_b largest scores of
 *                         scores[b, 0 .. n_b), as a set; the order of the slots
 *                         is unspecified (this library writes them in ascending
 *                         index order, the same order on every call)
 *     out[b, m_b .. k)  = -1
 *
 *   Ranking is the float order with -0 below +0; -inf and +inf are ordinary
 *   scores, so -inf outranks the -1 padding (sglang PR 39648 report,
 *   功能与动机). The selected value multiset is exact: it equals the m_b largest
 *   scores bit for bit (vLLM issue "persistent_topk silently drops top-k
 *   candidates ...", 验证方法). Among scores equal to the m_b-th largest the
 *   lowest indices are taken; any tie rule would meet the contract, this one is
 *   fixed so that results are deterministic.
 *
 *   Capacity never truncates a row (the failure documented by that issue,
 *   原因分析, and by sglang PR 37625): an internal candidate buffer that fills up
 *   is compacted to the exact top candidates seen so far, and a sampled cutoff
 *   that keeps fewer than m_b candidates makes the row be scanned again in full.
 *
 * Preconditions that are not checked (they would need a device read):
 *   - no NaN in scores[b, 0 .. n_b); values past n_b never affect the result
 *     (rows of at most 16384 scores that start on 16 bytes may have the rest
 *     of the 16-byte block holding their last score read: when the stride is
 *     not a multiple of 16 bytes that is up to 12 bytes past the row's
 *     stride, past the end of `scores` for its last row, but never on
 *     another page);
 *   - paged: every mapped slot fits in int32 (see topk_paged).
 *
 * Memory and execution:
 *   - every pointer is a DEVICE pointer owned by the caller; the library keeps
 *     no reference after the call returns and allocates nothing per call;
 *   - the call only enqueues work on `stream` (0 = legacy default stream) of
 *     the current CUDA device and never synchronises; results are valid once
 *     that stream reaches this point;
 *   - `scores` needs 4-byte alignment only (rows may start at any float);
 *     `lengths`, `out` and `page_table` need 4-byte alignment;
 *   - `out` must not overlap any input.
 *
 * Errors: argument checks run before anything is enqueued; on any error other
 * than TOPK_ECUDA nothing is written. TOPK_ECUDA reports a failed CUDA runtime
 * call (launch, attribute query or set); the library never aborts the process.
 * A device-side wait that exceeds its time limit (never reached by a correct
 * launch) fills that row of `out` with TOPK_DEVICE_ERROR_INDEX instead of
 * hanging.
 */
#ifndef TOPK_INDEXER_H_
#define TOPK_INDEXER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st* topk_stream_t;

typedef enum topk_status {
  TOPK_OK = 0,
  TOPK_EINVAL = 1,          /* null pointer, misalignment, negative B, bad stride/page size */
  TOPK_EUNSUPPORTED_K = 2,  /* k outside [1, TOPK_MAX_K] */
  TOPK_ECUDA = 3,           /* a CUDA runtime call failed */
  TOPK_EDEVICE = 4,         /* no usable sm_103 device is current */
  TOPK_ESCRATCH = 5         /* topk_select_noalloc: more scratch needed than its static array holds */
} topk_status;

/* Largest supported k. The decode-step indexer uses k = 512, 1024 or 2048. */
#define TOPK_MAX_K 2048

/* Written into every slot of a row whose device-side wait timed out. */
#define TOPK_DEVICE_ERROR_INDEX ((int32_t)0x80000000)

/*
 * topk_ragged - indices of the k largest scores of every row.
 *
 *   scores   [B, stride] float32, row-major: row b starts at scores + b * stride
 *   stride   elements between consecutive rows, >= 1; also the row width
 *   lengths  [B] int32 valid lengths (clamped to [0, stride])
 *   B        number of rows, >= 0 (0 is a no-op)
 *   k        slots per row, 1 <= k <= TOPK_MAX_K
 *   out      [B, k] int32, contiguous; receives the indices and -1 padding
 *   stream   CUDA stream to enqueue on
 *
 * Returns TOPK_OK, or an error code as described above.
 */
topk_status topk_ragged(const float* scores, int64_t stride, const int32_t* lengths, int32_t B,
                        int32_t k, int32_t* out, topk_stream_t stream);

/*
 * topk_paged - as topk_ragged, with each selected index i of row b written as
 *   page_table[b * pt_stride + i / page_size] * page_size + i % page_size
 * (sglang PR 39648 report, topk.py docstring, and its PageTransform epilogue);
 * the -1 slots stay -1. The product is formed in 64-bit and narrowed to int32.
 *
 *   page_table  [B, pt_stride] int32, row-major
 *   pt_stride   entries per page-table row; must be >= ceil(stride / page_size)
 *               so that every valid index has a page entry
 *   page_size   tokens per page, >= 1 (any value; powers of two are not required)
 */
topk_status topk_paged(const float* scores, int64_t stride, const int32_t* lengths, int32_t B,
                       int32_t k, const int32_t* page_table, int64_t pt_stride,
                       int32_t page_size, int32_t* out, topk_stream_t stream);

/*
 * Workspace variants. In a large batch the rows that start last run while
 * most of the GPU has nothing left to do. topk_ragged_ws / topk_paged_ws
 * stream some of those rows with two CTAs each: every CTA finds the exact
 * top-k of its half of the row (same order, same lowest-index tie rule) and
 * leaves it in the workspace; the half that finishes second merges the two
 * and writes the row. No CTA waits for another. Results are identical to
 * topk_ragged / topk_paged, bit for bit and slot for slot. This split of a
 * row over independent CTAs is this library's own scheduling device; the
 * pages' cluster split (sglang PR 39648 report, 实现拆解 4) needs the CTAs of a
 * row to run together.
 *
 * The library chooses how many rows to split from B, the row width, k and
 * the SM count (none when one CTA per row already keeps HBM busy, or when
 * rows are short), at most as many as the workspace holds; a few dozen long
 * rows that it can all split are split rather than given clusters.
 *
 *   workspace        DEVICE memory owned by the caller, 16-byte aligned, at
 *                    least 12 KiB. Its first 4 KiB must be zero before its
 *                    first use, and every call that completes leaves them zero
 *                    again; the rest is scratch. NULL: no row is split (the
 *                    call is then topk_ragged / topk_paged).
 *   workspace_bytes  its size; topk_workspace_bytes tells how much lets every
 *                    row the library would split be split
 *
 * Calls that may run at the same time on the GPU (other streams, concurrent
 * graph launches) need different workspaces: they would race on it.
 */
topk_status topk_ragged_ws(const float* scores, int64_t stride, const int32_t* lengths,
                           int32_t B, int32_t k, int32_t* out, void* workspace,
                           size_t workspace_bytes, topk_stream_t stream);
topk_status topk_paged_ws(const float* scores, int64_t stride, const int32_t* lengths,
                          int32_t B, int32_t k, const int32_t* page_table, int64_t pt_stride,
                          int32_t page_size, int32_t* out, void* workspace,
                          size_t workspace_bytes, topk_stream_t stream);

/*
 * topk_workspace_bytes - writes to *bytes the workspace size that lets a call
 * with this k split up to max_split_rows rows (0 = the most the library ever
 * splits on the current device: its SM count; at most 1024). Errors:
 * TOPK_EUNSUPPORTED_K, TOPK_EINVAL (bytes NULL, max_split_rows out of range),
 * TOPK_ECUDA / TOPK_EDEVICE (device query).
 */
topk_status topk_workspace_bytes(int32_t k, int32_t max_split_rows, size_t* bytes);

/*
 * topk_select_bf16 - the same operation over BF16 scores (raw 16-bit
 * patterns, 2-byte aligned), for rows of at most 16384 scores: `stride` must
 * be <= 16384 (TOPK_EINVAL otherwise). page_table NULL selects the ragged
 * output, otherwise the paged one as in topk_paged. A BF16 value converts
 * exactly to FP32, so the ranking (-0 below +0), the tie rule and the
 * contract are those of topk_ragged / topk_paged on the converted scores.
 * This is the small-row bf16 top-k of the sglang PR 39648 report (实现拆解 2,
 * `topk_transform_bf16_small`: rows <= 16384, k <= 2048, fused page-table
 * transform, NaN unsupported).
 */
topk_status topk_select_bf16(const uint16_t* scores, int64_t stride, const int32_t* lengths,
                             int32_t B, int32_t k, const int32_t* page_table, int64_t pt_stride,
                             int32_t page_size, int32_t* out, topk_stream_t stream);

/*
 * The two-level indexer's helpers on either side of the selection (sglang PR
 * 39648 report, 实现拆解 2 table, and the `amax8_varlen` /
 * `sort_candidate_blocks` docstrings of its candidate_table.py). With n_b =
 * clamp(lengths[b], 0, stride) scores, row b has nb_b = ceil(n_b / 8) blocks.
 *
 * topk_amax8_varlen - level-one keys: out[b * out_stride + i] = the largest
 * of scores[b, 8i .. 8i + 8) for i < nb_b - 1, and +inf for i = nb_b - 1 (the
 * newest block is always selected). "Largest" is in the selection's order,
 * +0 above -0, so a block whose maximum is a zero gets +0 if it holds one,
 * whatever the order of its scores (the page's fmaxf leaves that sign open). Slots from nb_b on are not written. If
 * topk > 0, rows with nb_b <= topk are skipped entirely (every block would be
 * selected); topk = 0 never skips.
 *   scores      [B, stride] float32 (4-byte aligned; rows that start on 32
 *               bytes, i.e. a 32-byte aligned base and stride % 8 == 0, are
 *               read with vector loads); no NaN in a row's valid prefix
 *   out         float32 rows of out_stride >= ceil(stride / 8) entries
 * Errors: TOPK_EINVAL (B < 0, topk < 0, out_stride too small, null or
 * misaligned pointers), TOPK_ECUDA, TOPK_EDEVICE.
 */
topk_status topk_amax8_varlen(const float* scores, int64_t stride, const int32_t* lengths,
                              int32_t B, int32_t topk, float* out, int64_t out_stride,
                              topk_stream_t stream);

/*
 * topk_sort_candidate_blocks - the block table, in place: blocks [B, k]
 * int32 holds row b's selected block ids in any order, -1 padded (for
 * instance the output of topk_ragged over the level-one keys, with lengths
 * nb_b). They are rewritten in ascending order, INT32_MAX past the last.
 * out_pages [B, k] receives each id's pool slot,
 *   page_table[b * pt_stride + id / bpp] * bpp + id % bpp,  bpp = page_size / 8,
 * and INT32_MAX in the padded slots. A row with nb_b <= k gets the identity
 * table (0 .. nb_b - 1) and its input is not read.
 *   page_size   a power of two >= 8
 *   pt_stride   >= ceil(ceil(stride / 8) / bpp)
 *   stride      <= 1,048,576 (at most 131072 blocks per row)
 * Precondition (not checked on the device): a row with nb_b > k holds
 * min(k, nb_b) distinct ids in [0, nb_b); ids outside that range are ignored,
 * duplicates collapse. Errors as above.
 */
topk_status topk_sort_candidate_blocks(int32_t* blocks, int32_t B, int32_t k,
                                       const int32_t* lengths, int64_t stride,
                                       const int32_t* page_table, int64_t pt_stride,
                                       int32_t page_size, int32_t* out_pages,
                                       topk_stream_t stream);

/*
 * topk_select_noalloc - the same operation as topk_ragged (page_table NULL)
 * or topk_paged, for callers that cannot allocate device memory: for
 * instance a serving engine that reserves nearly all of HBM for its KV cache
 * at start-up and forbids allocation on the decode path (cudaMalloc can fail
 * there, and it synchronises the device), or a plugin that runs inside a
 * host framework without access to its allocator. The pages have no
 * counterpart of this call.
 *
 * It allocates nothing and takes no workspace: the scratch for split rows
 * (see topk_ragged_ws) is a fixed 4 MiB + 12 KiB array in the library's own
 * device memory, which every GPU that loads the library holds until the
 * process exits. That is room for 128 split rows at k = 2048, 512 at k = 512.
 * A call that would split more rows than that returns TOPK_ESCRATCH before
 * anything is enqueued.
 *
 * The first call on a device looks up the array's device address and
 * enqueues a clear of its counters on that call's stream, ahead of its
 * kernel (the array is also zero when the library's module loads); make that
 * first call before any stream capture. Every call shares the one array:
 * calls that may run at the same time on the GPU (other streams, other host
 * threads) race on it, so serialise them. The caller still passes inputs and
 * outputs as for topk_ragged / topk_paged, with the same contract; invalid
 * arguments return TOPK_EINVAL / TOPK_EUNSUPPORTED_K exactly as there, before
 * the scratch is sized.
 */
topk_status topk_select_noalloc(const float* scores, int64_t stride, const int32_t* lengths,
                                int32_t B, int32_t k, const int32_t* page_table,
                                int64_t pt_stride, int32_t page_size, int32_t* out,
                                topk_stream_t stream);

/*
 * topk_max_active_clusters - diagnostic: writes to *clusters how many
 * thread-block clusters of cluster_size (2, 4, 8 or 16) CTAs of the streaming
 * kernel for this k (ragged output when paged == 0, paged otherwise) can be
 * resident at once on the current device, as the CUDA driver answers it
 * (cudaOccupancyMaxActiveClusters; the CTAs of a cluster must share one GPC,
 * so this can be less than the SM count times the CTAs per SM, divided by
 * the cluster size). The automatic policy gives a row a cluster only while
 * the clusters of every row fit at once. Errors: TOPK_EUNSUPPORTED_K,
 * TOPK_EINVAL (clusters NULL or another cluster size), TOPK_ECUDA,
 * TOPK_EDEVICE.
 */
topk_status topk_max_active_clusters(int32_t k, int32_t paged, int32_t cluster_size,
                                     int32_t* clusters);

/* Static, human-readable description of a status code. */
const char* topk_status_string(topk_status status);

/* Version of this ABI (bumped on any incompatible change). */
int32_t topk_abi_version(void);

/*
 * Test and diagnostic variant. Same operation and contract as topk_ragged /
 * topk_paged (page_table == NULL selects the ragged output); the options only
 * change which internal path each row takes, never the result. Zero-filled
 * options mean "automatic", exactly like the plain calls.
 *
 *   sample_mode     0 automatic, 1 never use the sampled cutoff,
 *                   2 use it on every row long enough to sample
 *   cluster_size    0 automatic, 1 one CTA per row, or 2 / 4 / 8 / 16 CTAs
 *                   of a thread-block cluster per row (16 is a non-portable
 *                   cluster size; the automatic policy takes 16 only for
 *                   batches of a few long rows)
 *   stash_capacity  0 = default; otherwise the candidate-buffer size to use,
 *                   in [k + 2048, default]: small values force the in-buffer
 *                   compaction path on ordinary inputs. The default is
 *                   b + 2048 entries for b = 512 and min(b + 4096, 5120)
 *                   for b = 1024 or 2048, b the smallest of these not below k
 *   sample_z        0 = default margin; otherwise the number of standard
 *                   deviations added to the sampled rank (negative values make
 *                   the sampled cutoff too high and force the full rescan)
 *   counters        optional DEVICE array of TOPK_NUM_COUNTERS uint32, which
 *                   the kernel increments (see topk_counter); NULL = none
 *   probe_stage     0 = off; s >= 1 makes the wait for streamed stage s-1 of
 *                   every row wait instead on a barrier that nothing completes,
 *                   so it runs out after probe_wait_us microseconds (1 ..
 *                   5,000,000): the row then takes the device-error path
 *                   (TOPK_DEVICE_ERROR_INDEX in every slot, counted). This
 *                   tests the bounded waits without a real fault; results of
 *                   such a call are not a selection.
 *   split_rows      0 automatic; -1 split no row; m > 0 split exactly the last
 *                   m rows (m <= B, the workspace must hold them; forces one
 *                   CTA per row, so cluster_size must be 0 or 1)
 *   workspace,      as for topk_ragged_ws; NULL = none (no row is split, and
 *   workspace_bytes split_rows must be 0 or -1)
 *   short_rows      0 automatic (FP32 rows of width <= 16384 take the short-row
 *                   kernel unless cluster_size, stash_capacity, probe_stage or
 *                   split_rows > 0 is given); -1 never; 1 always (width <= 16384
 *                   and none of those options). In the short-row kernel
 *                   sample_mode 1 selects its register path for every row
 *                   (no stash) and sample_z has no effect.
 */
typedef enum topk_counter {
  TOPK_CNT_ROWS = 0,          /* rows handled */
  TOPK_CNT_TRIVIAL = 1,       /* rows with length <= k (no selection needed) */
  TOPK_CNT_SAMPLED = 2,       /* rows that streamed against a sampled cutoff */
  TOPK_CNT_RESCAN = 3,        /* rows (halves of split rows) rescanned because the cutoff kept too few */
  TOPK_CNT_COMPACTIONS = 4,   /* candidate-buffer compactions (summed over CTAs) */
  TOPK_CNT_DEVICE_ERRORS = 5, /* CTAs whose waits timed out */
  TOPK_CNT_CLUSTER_ROWS = 6,  /* rows split over a cluster of CTAs */
  TOPK_CNT_SPLIT_ROWS = 7,    /* rows streamed by two independent CTAs and merged */
  TOPK_CNT_SHORT_ROWS = 8,    /* rows taken by the short-row kernel */
  TOPK_CNT_SHORT_EXACT = 9,   /* of them, rows selected from registers (no stash) */
  TOPK_NUM_COUNTERS = 16
} topk_counter;

typedef struct topk_debug_opts {
  int32_t sample_mode;
  int32_t cluster_size;
  int32_t stash_capacity;
  float sample_z;
  uint32_t* counters;
  int32_t probe_stage;
  uint32_t probe_wait_us;
  int32_t split_rows;
  void* workspace;
  size_t workspace_bytes;
  int32_t short_rows;
} topk_debug_opts;

topk_status topk_select_ex(const float* scores, int64_t stride, const int32_t* lengths,
                           int32_t B, int32_t k, const int32_t* page_table, int64_t pt_stride,
                           int32_t page_size, int32_t* out, const topk_debug_opts* opts,
                           topk_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* TOPK_INDEXER_H_ */
