// Launch parameters and host-side launchers of the CUDA kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "fi_internal.h"

namespace fi {

constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull;  // 1 s per bounded wait

// Runs `fn` (a kernel's attribute setup and checks) the first time a launch
// site is used on a device; later launches on that device skip it. `mask`
// holds a bit per device (devices 64 and up always run `fn`).
template <class F>
inline cudaError_t once_per_device(std::atomic<uint64_t>& mask, F fn) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const bool tracked = dev >= 0 && dev < 64;
  if (tracked && ((mask.load(std::memory_order_acquire) >> dev) & 1u)) return cudaSuccess;
  const cudaError_t e = fn();
  if (e == cudaSuccess && tracked) mask.fetch_or(uint64_t(1) << dev, std::memory_order_acq_rel);
  return e;
}

struct DecodeParams {
  const WorkItem* items;
  const void* q;
  const int32_t* page_indices;
  int32_t num_pages;
  int32_t page_size;
  int32_t num_qo_heads;
  int32_t layout;
  float sm_scale;           // times the cache's key scale
  float v_scale;            // the cache's value scale, applied to every output state
  const float* k_head_scale;  // [num_kv_heads] factors on sm_scale, or null (all 1)
  const float* v_head_scale;  // [num_kv_heads] factors on v_scale, or null (all 1)
  void* out;
  float* lse;
  float* partial_o;
  float* partial_lse;
  const MergeTask* merges;    // split requests: slots and output row
  uint32_t* merge_counters;   // [merge][kv head], zero at launch
  uint32_t* err;
  uint64_t wait_limit_ns;
  int32_t fault_kind;
  // the decode kernel's persistent launch: items [0, n_items), CTA c starts
  // with item c and takes the next ones from *work_counter (zero at launch)
  int32_t n_items;
  uint32_t* work_counter;
};

struct MergeParams {
  const float* v;          // states [slot][H][d]
  const float* s;          // lse    [slot][H]
  const MergeTask* tasks;  // per output row; null = row r uses slots [r*S, r*S+S)
  int32_t S;
  int32_t H;
  int32_t d;
  void* out;               // [row][H][d], bf16 or fp16
  float* lse;              // [row][H] or null
  int32_t dtype;           // fi_dtype of out
};

struct PrefillParams {
  const WorkItem* items;    // longest first
  int32_t n_items;
  uint32_t* work_counter;   // zero before the launch: items past the first wave taken so far
  const int32_t* qo_indptr;
  const int32_t* page_indptr;
  const int32_t* last_page_len;
  const int32_t* page_indices;
  int32_t num_pages;
  int32_t page_size;
  int32_t num_qo_heads;
  int32_t group;
  int32_t pack;         // query heads per tile (1, or the group size): item.head is the
                        // head block, query heads [head * pack, head * pack + pack)
  int32_t layout;
  int32_t causal;
  int32_t window_left;  // -1: none; else row at key position pos keeps t >= pos - window_left
  float sm_scale;       // times the cache's key scale
  float v_scale;        // the cache's value scale
  const float* k_head_scale;  // [num_kv_heads] factors on sm_scale, or null (all 1)
  const float* v_head_scale;  // [num_kv_heads] factors on v_scale, or null (all 1)
  void* out;
  float* lse;
  // when set, each row's state goes here instead of out / lse: fp32
  // o [slot][head][d] (normalised, times v_scale) and lse [slot][head],
  // slot = item.slot + row of q
  float* state_o;
  float* state_lse;
  // states of split prefill tiles (items with merge > 0): fp32 o
  // [slot][head][d] (normalised, times v_scale) and lse [slot][head], slot =
  // item.slot + row within the tile * item.merge; merged by the merge kernel
  float* piece_o;
  float* piece_lse;
  uint32_t* err;
  uint64_t wait_limit_ns;
  int32_t fault_kind;   // test hook: 1 = CTA 0's K producer skips its first tile
};

// Persistent launch: min(grid, p.n_items) CTAs, one per SM; CTA c starts
// with item c and takes the next ones from p.work_counter.
cudaError_t launch_prefill(int head_dim, int dtype, const CUtensorMap& qm, const CUtensorMap& km,
                           const CUtensorMap& vm, const PrefillParams& p, int grid,
                           cudaStream_t stream);
// The two-tile prefill kernel (prefill_pair.cu): items 2p and 2p + 1 (the
// planner's adjacent query heads h, h + 1 of one tile, h even) run in one
// CTA. It applies to head_dim 64 and 128, even groups, plain prefill (one
// head per tile row, no state output); launch_prefill dispatches to it.
bool prefill_pair_applies(int head_dim, const PrefillParams& p);
cudaError_t launch_prefill_pair(int head_dim, int dtype, const CUtensorMap& qm,
                                const CUtensorMap& km, const CUtensorMap& vm,
                                const PrefillParams& p, int grid, cudaStream_t stream);
// One persistent launch over a mixed batch (prefill.cu): the prefill items
// `p` as launch_prefill runs them (one-tile kernel) and, on other warps of
// the same CTAs, the decode items `dp` (n_dec of them), taken from
// *dec_counter (zero before the launch). Applies to head_dim 256 with 1, 2
// or 4 query heads per kv head and a 16-bit cache (mixed_applies).
bool mixed_applies(int head_dim, int group, int dtype, int kv_dtype);
cudaError_t launch_mixed(int head_dim, int group, int dtype, const CUtensorMap& qm,
                         const CUtensorMap& km, const CUtensorMap& vm, const PrefillParams& p,
                         const DecodeParams& dp, int n_dec, uint32_t* dec_counter, int grid,
                         cudaStream_t stream);
// `dtype` (fi_dtype) selects the element type of q and out, `kv_dtype` that
// of the cache (dtype or FI_DTYPE_E4M3).
cudaError_t launch_decode(int head_dim, int group, int dtype, int kv_dtype, const CUtensorMap& km,
                          const CUtensorMap& vm, const DecodeParams& p, int n_items, int num_sms,
                          cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& p, int n_rows, cudaStream_t stream);

}  // namespace fi
