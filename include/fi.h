/*
 * fi.h — C ABI of the paged-KV attention library (libfi.so), GB300 / sm_103a.
 *
 * The library computes attention over a paged KV cache,
 *     O = softmax(sm_scale * Q K^T + mask) V        (per query head),
 * with the K/V rows of each request reached through a page table. The
 * source pages describe the problem, not a C interface:
 *   - "FlashInfer kernel library deep-dive", section "PageAttention": the KV
 *     cache is cut into fixed-size pages allocated on demand;
 *   - same page, section "KV cache layout": the NHD and HND layouts;
 *   - same page, section "core API usage": single/batch decode and batch
 *     prefill entry points;
 *   - "FlashAttention-3 kernel integration in inference engines", section 2:
 *     variable-length prefill over prefix-sum offsets (cu_seqlens), causal
 *     flag, softmax_scale defaulting to 1/sqrt(head_dim), continuous
 *     batching with chunked prefill over paged KV;
 *   - "FlashInfer Attention Kernel optimisation analysis", section 2.2:
 *     scheduling by sequence length (here: the host planner splits long KV
 *     across CTAs and the partial results are merged by log-sum-exp).
 *
 * Conventions used by every call below
 * ------------------------------------
 * Page table (CSR, int32): request b owns page_indices[page_indptr[b] ..
 *   page_indptr[b+1]-1]; every page is full except the last, which holds
 *   last_page_len[b] in [1, page_size] tokens. kv_len[b] =
 *   (n_pages-1)*page_size + last_page_len[b], or 0 for a request with no
 *   pages (its last_page_len is then ignored). Key t of request b lives on
 *   page page_indices[page_indptr[b] + t/page_size], slot t%page_size.
 * KV layouts (the plan's fi_dtype, bf16 by default):
 *   FI_LAYOUT_NHD = [page][slot][kv_head][dim],
 *   FI_LAYOUT_HND = [page][kv_head][slot][dim]. K and V are separate
 *   buffers of the same layout; page_stride_elems is the distance between
 *   consecutive pages in elements (0 = dense: page_size*num_kv_heads*head_dim),
 *   so K and V may also be two views into one [num_pages][2][...] buffer.
 * Heads: num_qo_heads = g * num_kv_heads; query head h reads kv head h/g.
 * Queries (same type as K/V): decode q is [batch][num_qo_heads][head_dim];
 *   prefill q is the ragged packing [sum qo_len][num_qo_heads][head_dim]
 *   with request b on rows qo_indptr[b] .. qo_indptr[b+1]-1. out has q's
 *   shape and type.
 * Causal (prefill): row i of a request with qo_len rows sees keys
 *   t <= kv_len - qo_len + i (the chunk's queries are the last qo_len
 *   positions of its KV); qo_len > kv_len is rejected. A left window
 *   (fi_plan_options) also hides t < kv_len - qo_len + i - window_left.
 * lse (fp32, optional, may be NULL): natural log of the sum over visible
 *   keys of exp(sm_scale * <q,k>). A row with no visible key gets out = 0
 *   and lse = -inf.
 * Supported shapes: head_dim in {64, 128, 256}; page_size in {16, 32};
 *   g in {1, 2, 4, 8}. Anything else returns FI_ERR_UNSUPPORTED.
 * Memory: every device buffer (inputs, outputs, workspace) is owned by the
 *   caller. The run calls allocate nothing. A plan owns host memory only.
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   Every run call is asynchronous and stream-ordered; host-side argument
 *   errors are returned before anything is enqueued.
 * Device errors: kernels never trap and never wait without a bound. A
 *   page index outside [0, num_pages) is skipped and recorded; a bounded
 *   wait that runs out is recorded. fi_check_device_status() reports
 *   either after the stream has been synchronised. (A run of a plan without
 *   query rows touches nothing, so the workspace's status word is then
 *   whatever the last run before it left.)
 */
#ifndef FI_H
#define FI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FI_OK = 0,
  FI_ERR_INVALID_ARG = 1,         /* malformed sizes, page table or pointers */
  FI_ERR_UNSUPPORTED = 2,         /* valid but not built: head_dim, page_size, g */
  FI_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below what fi_plan asked for */
  FI_ERR_CUDA = 4,                /* a CUDA call failed; see fi_last_error_string() */
  FI_ERR_DEVICE_TIMEOUT = 5,      /* a kernel's bounded wait ran out */
  FI_ERR_DEVICE_BOUNDS = 6,       /* a kernel met a page index outside the cache */
  FI_ERR_NO_DEVICE = 7            /* no usable CUDA device for a run call */
} fi_status;

typedef enum { FI_LAYOUT_NHD = 0, FI_LAYOUT_HND = 1 } fi_kv_layout;
typedef enum { FI_MODE_DECODE = 0, FI_MODE_PREFILL = 1 } fi_mode;

/* Element types: q and out are bf16 or fp16; the K/V cache is the same type
 * or FP8 E4M3 (OCP format; decode plans only). lse and partial states are
 * fp32. */
typedef enum { FI_DTYPE_BF16 = 0, FI_DTYPE_FP16 = 1, FI_DTYPE_E4M3 = 2 } fi_dtype;

/*
 * Options of a plan. Start from FI_PLAN_OPTIONS_DEFAULT (a zero-filled
 * struct means a window of 0, not "no window").
 *   window_left  -1: no window. >= 0: the left half of the window_size pair
 *                of the varlen call on the "FlashAttention-3 kernel
 *                integration in inference engines" page, section 2: the row
 *                standing at key position pos = kv_len - qo_len + i also
 *                loses every key t < pos - window_left, so a causal row sees
 *                at most window_left + 1 keys (a decode row: the last
 *                window_left + 1). The right side is set by `causal`.
 *   dtype        fi_dtype of q and out (FI_DTYPE_BF16 or FI_DTYPE_FP16).
 *   kv_dtype     fi_dtype of the K/V cache: -1 = dtype, or FI_DTYPE_E4M3 for
 *                an FP8 cache (decode plans only; FI_ERR_UNSUPPORTED for
 *                prefill plans). An FP8 cache holds K / k_scale and
 *                V / v_scale; the run calls take the two scales.
 *   num_prefix_groups, prefix_group_indptr, prefix_pages
 *                shared-prefix (cascade) decode: the "FlashInfer kernel
 *                library deep-dive" page, section "batch layer", lists
 *                shared-prefix optimisation (find the prefix that sequences
 *                have in common and reuse it) among the batch kernels'
 *                techniques. Group g is requests
 *                prefix_group_indptr[g] .. prefix_group_indptr[g+1]-1 (host
 *                int32 [num_prefix_groups+1], non-decreasing, groups of
 *                consecutive requests), whose first prefix_pages[g] pages
 *                (host int32 [num_prefix_groups], >= 1, full pages of every
 *                request in the group) are the same physical pages (caller
 *                contract: the library reads the group's first request's
 *                page ids). The prefix is attended once per group for all of
 *                the group's query rows on the tensor cores, each request's
 *                own pages by the decode kernel, and the two states are
 *                merged by log-sum-exp. Decode plans with a 16-bit cache and
 *                no window only (else FI_ERR_UNSUPPORTED); 0 / NULL = none.
 *                The arrays are read by fi_plan only.
 */
typedef struct {
  int32_t window_left;
  int32_t dtype;
  int32_t kv_dtype;
  int32_t num_prefix_groups;
  const int32_t* prefix_group_indptr;
  const int32_t* prefix_pages;
} fi_plan_options;

#define FI_PLAN_OPTIONS_DEFAULT {-1, FI_DTYPE_BF16, -1, 0, NULL, NULL}

typedef struct fi_plan_s* fi_plan_t;

/* Summary of a plan, for logging and tests. */
typedef struct {
  int32_t mode;             /* fi_mode */
  int32_t batch_size;
  int32_t num_items;        /* work items of all launches */
  int32_t num_decode_items; /* of which single-row (decode) work */
  int32_t num_prefill_items;/* multi-row (prefill) work */
  int32_t chunk_tokens;     /* split-KV chunk length of decode work (0 = no split) */
  int32_t num_split_requests;
  int32_t num_partial_slots;/* rows of fp32 partial states in the workspace */
  int64_t workspace_bytes;
  int64_t total_kv_tokens;  /* sum of kv_len */
  int32_t num_prefix_items; /* shared-prefix work (prefix chunk x row tile x head) */
  int32_t num_prefix_groups;
  int64_t host_io_bytes;    /* extra workspace of fi_batch_attention_host */
} fi_plan_info;

/*
 * fi_plan — host-side planning of one batch (no CUDA call, no device memory).
 *
 * Reads the host copies of the page table (and, for prefill, qo_indptr),
 * validates them, decides how each request's KV is split across CTAs for
 * load balance ("FlashInfer Attention Kernel optimisation analysis",
 * section 2.2; "FlashInfer kernel library deep-dive", section
 * "load-balanced scheduling"), builds the work list and sizes the
 * workspace the run calls need.
 *   mode             FI_MODE_DECODE (one query row per request; qo_indptr_h
 *                    must be NULL) or FI_MODE_PREFILL (qo_indptr_h required;
 *                    requests with one row are planned as decode work).
 *   batch_size       number of requests B >= 0 (0 gives an empty plan; a
 *                    plan without query rows, B = 0 or every qo_len 0, makes
 *                    every run call return FI_OK at once, reading no
 *                    argument but the plan).
 *   qo_indptr_h      host int32 [B+1], non-decreasing, qo_indptr_h[0] == 0.
 *   page_indptr_h    host int32 [B+1], non-decreasing, page_indptr_h[0] >= 0.
 *   last_page_len_h  host int32 [B].
 *   causal           prefill only; ignored for decode.
 *   options          window and element type (see fi_plan_options); NULL
 *                    gives FI_PLAN_OPTIONS_DEFAULT. Copied into the plan.
 *   num_sms          SMs of the device the plan will run on (>0).
 *   out_plan         receives the plan; free it with fi_plan_destroy.
 *   workspace_bytes  receives the device workspace size the runs need.
 * The device copies of the same arrays passed to a run must hold the same
 * values (caller contract). A plan is immutable and may be run any number
 * of times, with any inputs of the same page-table structure.
 * Errors: FI_ERR_INVALID_ARG (NULL pointers, negative sizes, decreasing
 * indptr, last_page_len outside [1,page_size] for a request with pages,
 * causal with qo_len > kv_len, num_qo_heads not a multiple of
 * num_kv_heads, window_left < -1, dtype not an fi_dtype, a request of more
 * than INT32_MAX / 2 keys, more than INT32_MAX query rows in all, shared-
 * prefix groups out of order or whose prefix is not made of full pages of
 * every request in the group),
 * FI_ERR_UNSUPPORTED (head_dim, page_size or g not built; an FP8 cache in a
 * prefill plan; shared prefixes with an FP8 cache, a window or a prefill
 * plan).
 */
fi_status fi_plan(int32_t mode, int32_t batch_size, const int32_t* qo_indptr_h,
                  const int32_t* page_indptr_h, const int32_t* last_page_len_h,
                  int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t page_size, int32_t causal, const fi_plan_options* options,
                  int32_t num_sms, fi_plan_t* out_plan, size_t* workspace_bytes);

/* Frees a plan (NULL is accepted). */
fi_status fi_plan_destroy(fi_plan_t plan);

/* Copies a summary of the plan into *info. */
fi_status fi_plan_get_info(fi_plan_t plan, fi_plan_info* info);

/*
 * Copies the plan's work list to host memory: 8 int32 per item, in launch
 * order: {request, kv_head (decode), qo_head (prefill) or kv_head with all
 * its query heads (shared prefix), first page index
 * (into page_indices), number of pages, first key, end key, partial slot or
 * -1, first row of q}. Keys are token positions within the request; the
 * first page holds the first key at slot (first key % page_size), earlier
 * slots of that page lie outside the item's window. Decode items come
 * first, then prefill items, then shared-prefix items (request = 2 x the
 * group index, keys within the group's prefix, slot = the state slot of
 * row 0 of q).
 * `capacity` is in items; *num_items receives the plan's item count.
 */
fi_status fi_plan_get_work(fi_plan_t plan, int32_t* items_h, int32_t capacity,
                           int32_t* num_items);

/*
 * fi_batch_decode_paged — batch decode over a paged KV cache.
 *
 * One query token per request ("FlashInfer kernel library deep-dive",
 * sections "single-request layer" and "batch layer"): for every request b
 * and query head h, out[b][h] = softmax(sm_scale * q[b][h] K_b^T) V_b over
 * all kv_len[b] keys of kv head h/g (the last window_left + 1 of them with
 * a left window). Each K/V page is loaded once and
 * shared by the g query heads of its group. Long requests are split over
 * several CTAs as the plan says; their fp32 partial states are merged by
 * log-sum-exp into out/lse inside the same kernel (the CTA that finishes a
 * split's last chunk merges it).
 *   plan             from fi_plan(FI_MODE_DECODE, ...).
 *   q                device [B][num_qo_heads][head_dim] of the plan's dtype.
 *   k_cache, v_cache device paged caches of the plan's dtype (layout,
 *                    page_stride_elems as in the conventions above),
 *                    num_pages pages each.
 *   page_indptr_d, page_indices_d, last_page_len_d  device int32 copies of
 *                    the planned page table.
 *   sm_scale         score scale, finite and >= 0 (1/sqrt(head_dim) is the
 *                    usual value); anything else is FI_ERR_INVALID_ARG.
 *   k_scale, v_scale dequantisation scales of the cache, finite and > 0:
 *                    the keys and values attended to are k_scale and v_scale
 *                    times the stored ones (1 for a bf16/fp16 cache). k_scale
 *                    is folded into the score scale, v_scale into the output
 *                    (the FP8 scale handling the "FlashAttention-3 kernel
 *                    integration in inference engines" page describes in
 *                    section 1: the quantisation scale fused with the softmax
 *                    scaling instead of extra conversion passes).
 *   k_head_scale, v_head_scale  device fp32 [num_kv_heads] or NULL: a
 *                    further factor per kv head on k_scale and v_scale (an
 *                    FP8 cache quantised with one scale per head: the keys
 *                    and values of kv head h attended to are k_scale *
 *                    k_head_scale[h] and v_scale * v_head_scale[h] times the
 *                    stored ones). NULL means 1 for every head. The values
 *                    must be finite and > 0 (caller contract: they are read
 *                    on the device only); 4-byte aligned.
 *   out              device [B][num_qo_heads][head_dim], the plan's dtype.
 *   lse              device fp32 [B][num_qo_heads] or NULL.
 *   workspace        device buffer of at least the planned size, 256-byte
 *                    aligned; its contents between calls belong to the
 *                    library (it caches the uploaded work list there).
 * Errors: FI_ERR_INVALID_ARG (NULL or misaligned pointers — q, caches and
 * out need 16-byte alignment —, a plan of the other mode, page_stride_elems
 * not a multiple of 8), FI_ERR_WORKSPACE_TOO_SMALL, FI_ERR_NO_DEVICE,
 * FI_ERR_UNSUPPORTED (the stream is being captured into a CUDA graph: the
 * work-list upload reads a reused pinned staging buffer, so a replay would
 * copy another call's list), FI_ERR_CUDA (launch failure).
 * The host keeps, per thread and device, a small ring of pinned staging
 * buffers for the work-list copy (allocated on first use, grown when a
 * plan needs more, never freed).
 */
fi_status fi_batch_decode_paged(fi_plan_t plan, const void* q, const void* k_cache,
                                const void* v_cache, int32_t kv_layout,
                                int64_t page_stride_elems, int32_t num_pages,
                                const int32_t* page_indptr_d, const int32_t* page_indices_d,
                                const int32_t* last_page_len_d, float sm_scale, float k_scale,
                                float v_scale, const float* k_head_scale,
                                const float* v_head_scale, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * fi_batch_decode_paged_noalloc — fi_batch_decode_paged without a workspace
 * argument, for callers that cannot allocate device memory where they run
 * attention (an engine plugin whose framework owns all device memory and
 * exposes no scratch allocator; a latency-critical loop where a cudaMalloc,
 * which can synchronise the device, is not acceptable). None of the cited
 * pages has a counterpart to this call; it is an interface convenience.
 * The scratch (work list, error word, fp32 split partials) is a 16 MiB
 * array inside the library, held by every GPU that loads the library until
 * the process exits. The work list is built in a static 16 MiB host buffer
 * of the library and copied by an ordinary pageable cudaMemcpyAsync (the
 * CUDA driver stages it before the call returns). The call allocates
 * nothing, host or device, pinned or not.
 *   Arguments: as for fi_batch_decode_paged, minus the workspace.
 *   First call on a device: looks up that device's address of the array
 *   (cudaGetSymbolAddress) and caches it.
 *   Graphs: the call cannot be captured; a stream that is capturing is
 *   refused with FI_ERR_UNSUPPORTED before anything touches the device.
 *   Sharing: every call uses the same array, so calls whose GPU work can
 *   overlap (unordered streams) race; order them on one stream.
 *   Limits: a plan whose workspace_bytes exceeds 16 MiB returns
 *   FI_ERR_WORKSPACE_TOO_SMALL before anything is enqueued. Device-side
 *   error flags of this call cannot be read with fi_check_device_status.
 * Errors: as for fi_batch_decode_paged.
 */
fi_status fi_batch_decode_paged_noalloc(fi_plan_t plan, const void* q, const void* k_cache,
                                        const void* v_cache, int32_t kv_layout,
                                        int64_t page_stride_elems, int32_t num_pages,
                                        const int32_t* page_indptr_d,
                                        const int32_t* page_indices_d,
                                        const int32_t* last_page_len_d, float sm_scale,
                                        float k_scale, float v_scale,
                                        const float* k_head_scale,
                                        const float* v_head_scale, void* out, float* lse,
                                        void* stream);

/*
 * fi_batch_prefill_paged — causal (or full) variable-length batch prefill
 * over a paged KV cache, the varlen form of "FlashAttention-3 kernel
 * integration in inference engines", section 2 (cu_seqlens_q is
 * qo_indptr; the keys come from the page table instead of cu_seqlens_k).
 * Requests may mix prompt chunks and single decode rows in one call
 * (continuous batching with chunked prefill, same section).
 *   plan         from fi_plan(FI_MODE_PREFILL, ...); carries `causal`.
 *   q            device [sum qo_len][num_qo_heads][head_dim] of the plan's
 *                dtype.
 *   qo_indptr_d  device int32 copy of the planned qo_indptr.
 *   other arguments as for fi_batch_decode_paged; out has q's shape and
 *   lse is fp32 [sum qo_len][num_qo_heads] or NULL.
 * Errors: as for fi_batch_decode_paged.
 */
fi_status fi_batch_prefill_paged(fi_plan_t plan, const void* q, const int32_t* qo_indptr_d,
                                 const void* k_cache, const void* v_cache, int32_t kv_layout,
                                 int64_t page_stride_elems, int32_t num_pages,
                                 const int32_t* page_indptr_d, const int32_t* page_indices_d,
                                 const int32_t* last_page_len_d, float sm_scale, float k_scale,
                                 float v_scale, const float* k_head_scale,
                                 const float* v_head_scale, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * fi_batch_attention_host — one serving step of a plan with the step's own
 * inputs and outputs in host memory. q and the page table (with qo_indptr
 * for a prefill plan) are copied to the device, the planned kernels run
 * exactly as fi_batch_decode_paged / fi_batch_prefill_paged run them, out
 * and lse are copied back, and the call returns once the step has
 * completed (it synchronises `stream`) with the device status of the step
 * (a device-side error word that fi_check_device_status would read is read
 * and cleared here). The KV cache stays in device memory: it is the cache.
 * The page table is gathered, together with the plan's work list, into a
 * pinned staging buffer of the library and crosses the link in one copy;
 * q, out and lse are copied straight from and to the caller's buffers
 * (page-locked buffers make those copies DMA transfers; pageable ones
 * work, through the driver's staging). A stream that is being captured is
 * refused (FI_ERR_UNSUPPORTED) before anything is copied.
 *   plan             from fi_plan, either mode.
 *   q_h              host [total q rows][num_qo_heads][head_dim], the plan's
 *                    dtype (total q rows = B for a decode plan,
 *                    qo_indptr_h[B] for a prefill plan).
 *   qo_indptr_h      host int32 [B+1] for a prefill plan; NULL for decode.
 *   k_cache, v_cache, kv_layout, page_stride_elems, num_pages, sm_scale,
 *   k_scale, v_scale, k_head_scale, v_head_scale as for fi_batch_decode_paged
 *                    (the caches and the per-head scales are device
 *                    memory).
 *   page_indptr_h, page_indices_h, last_page_len_h  host int32, the planned
 *                    page table (page_indices_h holds page_indptr_h[B]
 *                    entries).
 *   out_h            host, q_h's shape and dtype.
 *   lse_h            host fp32 [total q rows][num_qo_heads] or NULL.
 *   workspace        device, 256-byte aligned, at least workspace_bytes +
 *                    host_io_bytes of the plan (fi_plan_get_info): the
 *                    step's q, out and lse occupy the part after the run
 *                    calls' workspace (the page table has its place inside
 *                    that workspace, after the work lists).
 * Errors: as for fi_batch_decode_paged (FI_ERR_WORKSPACE_TOO_SMALL when the
 * host-IO part does not fit), FI_ERR_DEVICE_TIMEOUT / FI_ERR_DEVICE_BOUNDS
 * from the step's device status.
 */
fi_status fi_batch_attention_host(fi_plan_t plan, const void* q_h, const int32_t* qo_indptr_h,
                                  const void* k_cache, const void* v_cache, int32_t kv_layout,
                                  int64_t page_stride_elems, int32_t num_pages,
                                  const int32_t* page_indptr_h, const int32_t* page_indices_h,
                                  const int32_t* last_page_len_h, float sm_scale, float k_scale,
                                  float v_scale, const float* k_head_scale,
                                  const float* v_head_scale, void* out_h, float* lse_h,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * fi_batch_attention_host_async — fi_batch_attention_host without the wait:
 * the same checks, copies and kernels are enqueued on `stream` and the call
 * returns at once with a ticket for the step in *ticket (0 for an empty
 * plan). The page table (and qo_indptr) is staged before the call returns
 * and may be changed at once; q_h, out_h and lse_h belong to the step
 * until fi_host_step_wait on its ticket returns (the copy engine reads a
 * page-locked q_h when the step's copy runs). This lets a serving loop
 * plan and stage step t+1 while the device runs step t; steps on one
 * stream run in the order they were issued, so consecutive steps may
 * share the workspace.
 *   ticket           receives the step's ticket (must not be NULL).
 * At most 8 steps may be in flight per host thread (issued, not yet
 * waited for); a ticket is waited for on the thread that issued it.
 * Errors: as for fi_batch_attention_host, except the device status, which
 * fi_host_step_wait returns; FI_ERR_INVALID_ARG with 8 steps in flight on
 * this thread, or steps of another device still in flight on it.
 */
fi_status fi_batch_attention_host_async(
    fi_plan_t plan, const void* q_h, const int32_t* qo_indptr_h, const void* k_cache,
    const void* v_cache, int32_t kv_layout, int64_t page_stride_elems, int32_t num_pages,
    const int32_t* page_indptr_h, const int32_t* page_indices_h, const int32_t* last_page_len_h,
    float sm_scale, float k_scale, float v_scale, const float* k_head_scale,
    const float* v_head_scale, void* out_h, float* lse_h, void* workspace, size_t workspace_bytes,
    void* stream, uint64_t* ticket);

/*
 * fi_host_step_wait — blocks until the step of `ticket` has completed (its
 * out and lse are in the caller's host buffers) and returns its device
 * status: FI_OK, FI_ERR_DEVICE_TIMEOUT or FI_ERR_DEVICE_BOUNDS, or
 * FI_ERR_CUDA if the stream failed. Ticket 0 returns FI_OK. A ticket that
 * this thread did not issue, or that was already waited for, gives
 * FI_ERR_INVALID_ARG.
 */
fi_status fi_host_step_wait(uint64_t ticket);

/*
 * fi_merge_states — combine attention states computed over disjoint key
 * sets (split-KV partials) by log-sum-exp. The pages do not spell this
 * step out; it is the standard identity behind tiled online softmax
 * ("FlashAttention-3 kernel integration in inference engines", section 1:
 * softmax aggregated in place across tiles). For row r, head h:
 *   M = max_i s[r][i][h];  w_i = exp(s[r][i][h] - M);
 *   out[r][h] = sum_i w_i v[r][i][h] / sum_i w_i;  lse = M + ln sum_i w_i.
 * States with s = -inf weigh nothing; if all are -inf, out = 0, lse = -inf.
 *   v        device fp32 [n][S][H][d];   s  device fp32 [n][S][H].
 *   out_dtype  fi_dtype of out (bf16 or fp16).
 *   out      device [n][H][d] of out_dtype (16-byte aligned); lse_out fp32
 *            [n][H] or NULL.
 *   d        multiple of 4, at most 1024; n, S, H >= 0 (n == 0 or H == 0: no-op).
 * Errors: FI_ERR_INVALID_ARG, FI_ERR_NO_DEVICE, FI_ERR_CUDA.
 */
fi_status fi_merge_states(const float* v, const float* s, int32_t n, int32_t S, int32_t H,
                          int32_t d, int32_t out_dtype, void* out, float* lse_out, void* stream);

/*
 * fi_check_device_status — synchronises `stream`, reads and clears the
 * device error word kept at the start of `workspace` by the runs that used
 * it. Returns FI_OK, FI_ERR_DEVICE_TIMEOUT (a bounded wait ran out) or
 * FI_ERR_DEVICE_BOUNDS (a page index outside the cache was skipped), or
 * FI_ERR_CUDA if the synchronisation itself failed.
 */
fi_status fi_check_device_status(void* workspace, void* stream);

/* Static description of a status code. */
const char* fi_status_string(fi_status status);

/* Message of the last CUDA error seen by this thread's calls (or ""). */
const char* fi_last_error_string(void);

/*
 * Test hook for the failure path. kind 0 = normal operation; kind 1 = in the
 * next paged run call, the first CTA of each attention kernel (decode, and
 * prefill: its K producer) skips its first tile load, so that the waiting
 * warps' bounded waits run out after about `wait_limit` nanoseconds and the
 * kernel reports FI_ERR_DEVICE_TIMEOUT instead of hanging. wait_limit <= 0
 * restores the default bound. Process-wide: the next run call on any thread
 * takes the fault (once). Meant for tests only.
 */
fi_status fi_debug_set_fault(int32_t kind, int64_t wait_limit);

/*
 * Profiling hook: the next paged run call made by this thread records
 * start_event (a cudaEvent_t) on its stream just before its first attention
 * kernel and stop_event just after its last attention kernel, so that a
 * caller can time the attention kernels alone (without the work-list
 * upload) with
 * cudaEventElapsedTime. One-shot; NULL for both clears a pending request.
 * Errors from the event records are returned by that run call as FI_ERR_CUDA.
 */
fi_status fi_profile_next_launch(void* start_event, void* stop_event);

#ifdef __cplusplus
}
#endif

#endif /* FI_H */
