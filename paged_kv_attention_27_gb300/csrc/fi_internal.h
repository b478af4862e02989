// Internal declarations shared by the host planner (plan.cpp), the C ABI
// (api.cu) and the kernels. Nothing here is part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "fi.h"

namespace fi {

// One CTA's work. Decode items: tokens [tok_begin, tok_end) of request
// `req` for kv head `head` (all g query heads of its group), pages
// page_indices[page_begin .. page_begin+n_pages), writing either the final
// output row `q_row` (slot < 0) or partial-state slot `slot` of merge task
// `merge`. Prefill items: query rows [q_row, q_row + kPrefillTileM) of
// request `req` (absolute rows of q/out) for query head `head`, over keys
// [tok_begin, tok_end) — tok_end clipped to the causal bound of the tile's
// last row, tok_begin to the page of its first row's window. Shared-prefix
// items: rows [q_row, q_row + kPrefillTileM / g) for all g query heads of
// kv head `head` (the 128 M rows are rows x heads, heads inner).
struct WorkItem {
  int32_t req;
  int32_t head;
  int32_t page_begin;
  int32_t n_pages;
  int32_t tok_begin;
  int32_t tok_end;
  int32_t slot;
  int32_t q_row;
  int32_t merge;   // split decode work: index of its merge task; a prefill piece:
                   // the tile's piece count (row r's state at slot + r * merge);
                   // else -1
};
static_assert(sizeof(WorkItem) == 36, "work item is 9 int32");

// A row whose decode work was split: merge states [slot_base, slot_base +
// n_states) (each [num_qo_heads][head_dim] fp32) into output row out_row.
struct MergeTask {
  int32_t out_row;
  int32_t slot_base;
  int32_t n_states;      // states in slots [slot_base, slot_base + n_states), one per decode CTA
  int32_t extra_slot;    // first shared-prefix state of the row, or -1
  int32_t n_extra;       // shared-prefix states: extra_slot + e * extra_stride, e < n_extra
  int32_t extra_stride;
  int32_t pad[2];
};

constexpr int kPrefillTileM = 128;         // query rows per prefill CTA
constexpr size_t kHeaderBytes = 256;       // device error word, work counter, reserved
constexpr size_t kWorkCounterOffset = 64;  // prefill items handed out (zeroed by the upload)
constexpr size_t kDecodeCounterOffset = 128;  // decode items handed out (decode or mixed kernel)
constexpr size_t kAlign = 256;

// Error bits in the first word of the workspace.
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrBounds = 2u;

inline int decode_tile_tokens(int head_dim) { return 8192 / head_dim; }  // 32 KB of K+V
// A batch with both decode rows and multi-row (chunked prefill) requests runs
// as one persistent launch of the mixed kernel for these shapes (q/out and
// cache of one 16-bit type, head_dim 256, 1, 2 or 4 query heads per kv head).
inline bool mixed_kernel_applies(int head_dim, int group, int dtype, int kv_dtype) {
  return head_dim == 256 && (group == 1 || group == 2 || group == 4) && kv_dtype == dtype &&
         (dtype == FI_DTYPE_BF16 || dtype == FI_DTYPE_FP16);
}
inline int prefill_kv_tile(int head_dim) { return head_dim <= 128 ? 128 : 64; }
// KV split of prefill tiles: at most this many pieces per tile; the cost of a
// piece in KV tiles of one CTA (item start and end, about 2.4; writing its
// fp32 states and reading them back in the merge at an SM's share of HBM,
// about 2.8 at head_dim 128) that the planner weighs against a shorter
// finish; a split only where the estimate is this fraction of the unsplit
// one or less (it leaves out the merge launch), and only when the longest
// tile has kMinSplitTiles KV tiles or more
constexpr int kMaxPrefillPieces = 16;
constexpr int kSplitPieceCost = 5;
constexpr double kSplitMaxRatio = 0.85;
constexpr int kMinSplitTiles = 16;

struct WorkspaceLayout {
  size_t decode_items = 0, prefill_items = 0, prefix_items = 0, prefix_tables = 0,
         prefill_merges = 0, merges = 0, merge_counters = 0, partial_o = 0, partial_lse = 0;
  size_t image_end = 0;   // the run calls upload [0, image_end): header, work lists, merges
  // the page table of a host-buffer call (page indptr | page indices | last
  // page lengths | qo indptr), right after the image, uploaded with it
  size_t hio_tables = 0;
  size_t total = 0;
  // host-buffer calls only, after `total`: the step's q, out and lse
  size_t hio_q = 0, hio_out = 0, hio_lse = 0;
  size_t hio_total = 0;   // bytes of that region
};

struct Plan {
  int32_t mode = 0, batch = 0, num_qo_heads = 0, num_kv_heads = 0, head_dim = 0;
  int32_t page_size = 0, causal = 0, num_sms = 0;
  int32_t window_left = -1;              // -1: no window
  int32_t dtype = FI_DTYPE_BF16;         // q and out
  int32_t kv_dtype = FI_DTYPE_BF16;      // the K/V cache: dtype or FI_DTYPE_E4M3
  std::vector<WorkItem> decode_items;    // launch order
  std::vector<WorkItem> prefill_items;   // launch order
  std::vector<MergeTask> merges;
  // split prefill tiles: one task per row, merging the row's piece states
  // (after the prefill launch, by the merge kernel)
  std::vector<MergeTask> prefill_merges;
  // shared-prefix decode: prefill-kernel items over chunks of each group's
  // prefix (virtual request 2g = group g: its rows of q, one head, the
  // prefix keys; an item's `slot` plus a row of q is the row's state slot),
  // and the virtual requests' qo_indptr / page_indptr / last_page_len (each
  // 2 * groups entries, uploaded with the work lists)
  std::vector<WorkItem> prefix_items;
  std::vector<int32_t> prefix_tables;
  int32_t num_prefix_groups = 0;
  int32_t chunk_tokens = 0;
  int32_t num_split = 0;
  int32_t num_slots = 0;
  int64_t total_kv = 0;
  int64_t total_q = 0;                   // rows of q / out
  int32_t page_entries = 0;              // page_indptr[batch]: length of page_indices
  WorkspaceLayout ws;
};

// Scratch of fi_batch_decode_paged_noalloc: a static device array of this
// size inside the library (noalloc.cu), and a static host buffer of the same
// size from which that call's work list is copied (api.cu).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB

// api.cu: fi_batch_decode_paged with the work-list image filled into the
// static host buffer and copied by an ordinary (pageable) cudaMemcpyAsync,
// which the CUDA driver stages itself: no host or device allocation.
fi_status run_decode_static_upload(fi_plan_t plan, const void* q, const void* k_cache,
                                   const void* v_cache, int32_t kv_layout,
                                   int64_t page_stride_elems, int32_t num_pages,
                                   const int32_t* page_indptr_d, const int32_t* page_indices_d,
                                   const int32_t* last_page_len_d, float sm_scale,
                                   float k_scale, float v_scale, const float* k_head_scale,
                                   const float* v_head_scale, void* out, float* lse,
                                   void* workspace, size_t workspace_bytes, void* stream);

// plan.cpp
fi_status build_plan(int32_t mode, int32_t batch, const int32_t* qo_indptr,
                     const int32_t* page_indptr, const int32_t* last_page_len,
                     int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t page_size, int32_t causal, const fi_plan_options* options,
                     int32_t num_sms, Plan* plan);

}  // namespace fi

struct fi_plan_s {
  fi::Plan p;
};
