// The C ABI (include/fi.h): argument validation, tensor-map construction,
// work-list upload and kernel launches. Every numeric step runs in the
// CUDA kernels; this file only checks arguments and enqueues work.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "fi_internal.h"
#include "kernels.cuh"

namespace {

thread_local std::string g_last_error;
// test hook state, process-wide (fi_debug_set_fault may run on any thread)
std::atomic<int32_t> g_fault_kind{0};
std::atomic<uint64_t> g_wait_limit_ns{fi::kDefaultWaitLimitNs};
thread_local cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

fi_status cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return FI_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A side stream and two events per device, created on first use, for the
// calls that run decode and prefill work concurrently (fork/join on events,
// stream-ordered with respect to the caller's stream). No device memory.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

fi_status side_stream(SideStream* out) {
  static std::mutex mu;
  static SideStream per_dev[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FI_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  SideStream& s = per_dev[dev];
  if (!s.stream) {
    if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess) {
      g_last_error = "could not create the side stream for concurrent decode work";
      s = SideStream();
      return FI_ERR_CUDA;
    }
  }
  *out = s;
  return FI_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Pinned staging for the work-list upload. A copy from pageable memory
// makes the host wait until the driver has staged it, which delays the
// kernel launches queued behind it; from pinned memory it is a plain
// asynchronous DMA. Each host thread keeps a small ring of pinned slots for
// its current device; a slot is refilled only once the copy that read it
// has completed (one event per slot). Nothing is freed at exit.
constexpr int kStagingSlots = 8;
struct Staging {
  int device = -1;
  uint8_t* buf = nullptr;
  size_t slot_bytes = 0;
  cudaEvent_t done[kStagingSlots] = {};
  bool pending[kStagingSlots] = {};
  int next = 0;
};
thread_local Staging g_staging;   // work lists (and a host-buffer call's page table)

// The workspace prefix a run uploads: zeroed header (error word, work
// counter), work lists, merge tasks, zeroed merge counters; alignment gaps
// zeroed too. `dst` holds P.ws.image_end bytes.
void fill_image(uint8_t* dst, const fi::Plan& P) {
  // consecutive regions [offset, next offset): the data, then zeros
  struct Region { size_t off, end; const void* src; size_t bytes; };
  const Region regions[] = {
      {0, P.ws.decode_items, nullptr, 0},
      {P.ws.decode_items, P.ws.prefill_items, P.decode_items.data(),
       P.decode_items.size() * sizeof(fi::WorkItem)},
      {P.ws.prefill_items, P.ws.prefix_items, P.prefill_items.data(),
       P.prefill_items.size() * sizeof(fi::WorkItem)},
      {P.ws.prefix_items, P.ws.prefix_tables, P.prefix_items.data(),
       P.prefix_items.size() * sizeof(fi::WorkItem)},
      {P.ws.prefix_tables, P.ws.prefill_merges, P.prefix_tables.data(),
       P.prefix_tables.size() * sizeof(int32_t)},
      {P.ws.prefill_merges, P.ws.merges, P.prefill_merges.data(),
       P.prefill_merges.size() * sizeof(fi::MergeTask)},
      {P.ws.merges, P.ws.image_end, P.merges.data(), P.merges.size() * sizeof(fi::MergeTask)},
  };
  for (const Region& r : regions) {
    if (r.bytes) std::memcpy(dst + r.off, r.src, r.bytes);
    std::memset(dst + r.off + r.bytes, 0, r.end - r.off - r.bytes);
  }
}

// Fills `bytes` bytes of a pinned slot of `s` with `fill` and copies them
// to device `dst` on `stream` (synchronous pageable copy if pinned memory
// cannot be had).
template <class Fill>
fi_status stage_and_copy(Staging& s, void* dst, size_t bytes, Fill fill, cudaStream_t stream,
                         const char* what) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FI_ERR_NO_DEVICE;
  if (s.device != dev || bytes > s.slot_bytes) {
    // (re)build the ring once its copies have completed
    for (int i = 0; i < kStagingSlots; ++i) {
      if (s.done[i]) {
        if (s.pending[i]) cudaEventSynchronize(s.done[i]);
        cudaEventDestroy(s.done[i]);
        s.done[i] = nullptr;
      }
      s.pending[i] = false;
    }
    if (s.buf) cudaFreeHost(s.buf);
    s = Staging();
    size_t slot = size_t(1) << 20;
    while (slot < bytes) slot <<= 1;
    void* p = nullptr;
    bool ok = cudaHostAlloc(&p, slot * kStagingSlots, cudaHostAllocPortable) == cudaSuccess;
    for (int i = 0; ok && i < kStagingSlots; ++i)
      ok = cudaEventCreateWithFlags(&s.done[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      for (int i = 0; i < kStagingSlots; ++i)
        if (s.done[i]) cudaEventDestroy(s.done[i]);
      if (p) cudaFreeHost(p);
      s = Staging();
      cudaGetLastError();   // clear; fall back to a (synchronous) pageable copy
      std::vector<uint8_t> image(bytes);
      fill(image.data());
      const cudaError_t e = cudaMemcpy(dst, image.data(), bytes, cudaMemcpyHostToDevice);
      return e == cudaSuccess ? FI_OK : cuda_fail(e, what);
    }
    s.device = dev;
    s.buf = static_cast<uint8_t*>(p);
    s.slot_bytes = slot;
  }
  const int i = s.next;
  s.next = (s.next + 1) % kStagingSlots;
  cudaError_t e = cudaSuccess;
  if (s.pending[i]) e = cudaEventSynchronize(s.done[i]);
  if (e != cudaSuccess) return cuda_fail(e, what);
  uint8_t* src = s.buf + size_t(i) * s.slot_bytes;
  fill(src);
  e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaEventRecord(s.done[i], stream);
  if (e != cudaSuccess) return cuda_fail(e, what);
  s.pending[i] = true;
  return FI_OK;
}

// Host-buffer steps in flight on this host thread: each holds a pinned word
// that receives the step's device status and an event recorded after the
// step's last copy. A ticket is a sequence number; its slot is the number
// modulo the ring size, and a slot takes a new step only once the ticket it
// held has been waited for. Nothing is freed at exit.
constexpr int kHostSteps = 8;
struct HostSteps {
  int device = -1;
  uint32_t* words = nullptr;           // pinned, kHostSteps words
  cudaEvent_t done[kHostSteps] = {};
  uint64_t ticket[kHostSteps] = {};    // 0: free
  uint64_t next = 1;
};
thread_local HostSteps g_host_steps;

fi_status host_steps_ready(HostSteps& h) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FI_ERR_NO_DEVICE;
  if (h.device == dev) return FI_OK;
  for (int i = 0; i < kHostSteps; ++i)
    if (h.ticket[i]) {
      g_last_error = "host-buffer steps of another device are still in flight on this thread";
      return FI_ERR_INVALID_ARG;
    }
  for (int i = 0; i < kHostSteps; ++i)
    if (h.done[i]) cudaEventDestroy(h.done[i]);
  if (h.words) cudaFreeHost(h.words);
  const uint64_t next = h.next;
  h = HostSteps();
  h.next = next;
  void* p = nullptr;
  cudaError_t e = cudaHostAlloc(&p, kHostSteps * sizeof(uint32_t), cudaHostAllocPortable);
  for (int i = 0; e == cudaSuccess && i < kHostSteps; ++i)
    e = cudaEventCreateWithFlags(&h.done[i], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    for (int i = 0; i < kHostSteps; ++i)
      if (h.done[i]) cudaEventDestroy(h.done[i]);
    if (p) cudaFreeHost(p);
    h = HostSteps();
    h.next = next;
    return cuda_fail(e, "host-step status words");
  }
  h.words = static_cast<uint32_t*>(p);
  h.device = dev;
  return FI_OK;
}

// How a run call gets its work-list image into the workspace: from the
// pinned staging ring, from the static host buffer (the no-allocation call),
// or not at all (the host-buffer call uploads it with the page table).
enum class Upload { kStaged, kStatic, kDone };

fi_status upload_image(void* dst, const fi::Plan& P, cudaStream_t stream) {
  return stage_and_copy(g_staging, dst, P.ws.image_end,
                        [&](uint8_t* p) { fill_image(p, P); }, stream, "work-list upload");
}

// The work-list upload of the no-allocation decode call: the image is built
// in a static host buffer (one per process, guarded by a mutex) and copied
// with an ordinary cudaMemcpyAsync from pageable memory. For such a copy the
// CUDA driver copies the source into its own staging memory before the call
// returns (no device synchronisation), so the buffer may be refilled at once
// and this library allocates nothing, host or device.
std::mutex g_static_image_mutex;
uint8_t g_static_image[fi::kNoAllocScratchBytes];

fi_status upload_image_static(void* dst, const fi::Plan& P, cudaStream_t stream) {
  const size_t bytes = P.ws.image_end;
  if (bytes > sizeof(g_static_image)) return FI_ERR_WORKSPACE_TOO_SMALL;
  std::lock_guard<std::mutex> lock(g_static_image_mutex);
  fill_image(g_static_image, P);
  const cudaError_t e = cudaMemcpyAsync(dst, g_static_image, bytes, cudaMemcpyHostToDevice, stream);
  return e == cudaSuccess ? FI_OK : cuda_fail(e, "work-list upload");
}

// Tensor map over a paged K or V cache that fetches one (page, kv head)
// block per box: page_size rows x 64 dims (128 bytes, 128-byte swizzled)
// for a 16-bit cache; page_size whole rows of head_dim bytes for an FP8
// cache (128-byte swizzled at head_dim 128, unswizzled otherwise).
CUtensorMapDataType tma_type(int dtype) {
  if (dtype == FI_DTYPE_E4M3) return CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return dtype == FI_DTYPE_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

int elem_bytes(int dtype) { return dtype == FI_DTYPE_E4M3 ? 1 : 2; }

fi_status make_kv_map(CUtensorMap* map, const void* base, int layout, int num_pages, int P,
                      int Hkv, int d, int64_t page_stride, int dtype) {
  auto enc = encode_fn();
  if (!enc) {
    g_last_error = "cuTensorMapEncodeTiled is not available from the driver";
    return FI_ERR_CUDA;
  }
  cuuint64_t dims[4];
  cuuint64_t strides[3];
  cuuint32_t box[4];
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const cuuint64_t eb = cuuint64_t(elem_bytes(dtype));
  const cuuint32_t inner = dtype == FI_DTYPE_E4M3 ? cuuint32_t(d) : 64u;
  if (layout == FI_LAYOUT_NHD) {
    dims[0] = d; dims[1] = Hkv; dims[2] = P; dims[3] = num_pages;
    strides[0] = cuuint64_t(d) * eb;
    strides[1] = cuuint64_t(Hkv) * d * eb;
    box[0] = inner; box[1] = 1; box[2] = P; box[3] = 1;
  } else {
    dims[0] = d; dims[1] = P; dims[2] = Hkv; dims[3] = num_pages;
    strides[0] = cuuint64_t(d) * eb;
    strides[1] = cuuint64_t(P) * d * eb;
    box[0] = inner; box[1] = P; box[2] = 1; box[3] = 1;
  }
  strides[2] = cuuint64_t(page_stride) * eb;
  // FP8 rows of 128 bytes are swizzled too (the decode kernel reads MMA
  // fragments from them); other FP8 row lengths are not
  const CUtensorMapSwizzle swizzle = (dtype != FI_DTYPE_E4M3 || d == 128)
                                         ? CU_TENSOR_MAP_SWIZZLE_128B
                                         : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = enc(map, tma_type(dtype), 4, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_error = "cuTensorMapEncodeTiled failed for the KV cache (code " + std::to_string(int(r)) + ")";
    return FI_ERR_CUDA;
  }
  return FI_OK;
}

// Tensor map over the packed queries [rows][num_qo_heads][head_dim] that
// fetches 128 rows x 64 dims of one head per box (128-byte swizzled).
fi_status make_q_map(CUtensorMap* map, const void* q, int64_t rows, int Hq, int pack, int d,
                     int dtype) {
  auto enc = encode_fn();
  if (!enc) {
    g_last_error = "cuTensorMapEncodeTiled is not available from the driver";
    return FI_ERR_CUDA;
  }
  const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(Hq), cuuint64_t(rows)};
  const cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(Hq) * d * 2};
  // 64 dims x `pack` heads x 128 / pack rows: the 128 M rows of a tile,
  // heads inner
  const cuuint32_t box[3] = {64, cuuint32_t(pack), cuuint32_t(fi::kPrefillTileM / pack)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, tma_type(dtype), 3, const_cast<void*>(q), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_error = "cuTensorMapEncodeTiled failed for q (code " + std::to_string(int(r)) + ")";
    return FI_ERR_CUDA;
  }
  return FI_OK;
}

// Encoded tensor maps of recent calls (per host thread). A serving loop
// calls with the same caches, and often the same q buffer, step after step;
// the same arguments encode the same map, so it is reused instead of
// encoded again. Keyed by every argument of the encoding and the device.
struct MapKey {
  const void* base;
  int64_t a, b, c, d, e, f;
  int dev, kind;
  bool operator==(const MapKey& o) const {
    return base == o.base && a == o.a && b == o.b && c == o.c && d == o.d && e == o.e &&
           f == o.f && dev == o.dev && kind == o.kind;
  }
};
constexpr int kMapCache = 8;
struct MapCache {
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  bool used[kMapCache] = {};
  int next = 0;
};
thread_local MapCache g_maps;

template <class Encode>
fi_status cached_map(CUtensorMap* out, const MapKey& k, Encode encode) {
  for (int i = 0; i < kMapCache; ++i)
    if (g_maps.used[i] && g_maps.key[i] == k) {
      *out = g_maps.map[i];
      return FI_OK;
    }
  const fi_status st = encode(out);
  if (st != FI_OK) return st;
  const int i = g_maps.next;
  g_maps.next = (i + 1) % kMapCache;
  g_maps.key[i] = k;
  g_maps.map[i] = *out;
  g_maps.used[i] = true;
  return FI_OK;
}

fi_status kv_map(CUtensorMap* map, const void* base, int layout, int num_pages, int P, int Hkv,
                 int d, int64_t page_stride, int dtype) {
  int dev = -1;
  cudaGetDevice(&dev);
  const MapKey k{base, layout, num_pages, P, Hkv, d * 16 + dtype, page_stride, dev, 0};
  return cached_map(map, k, [&](CUtensorMap* m) {
    return make_kv_map(m, base, layout, num_pages, P, Hkv, d, page_stride, dtype);
  });
}

fi_status q_map(CUtensorMap* map, const void* q, int64_t rows, int Hq, int pack, int d,
                int dtype) {
  int dev = -1;
  cudaGetDevice(&dev);
  const MapKey k{q, rows, Hq, pack, d, dtype, 0, dev, 1};
  return cached_map(map, k, [&](CUtensorMap* m) {
    return make_q_map(m, q, rows, Hq, pack, d, dtype);
  });
}

fi_status check_device() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    g_last_error = std::string("no CUDA device: ") + cudaGetErrorString(e);
    return FI_ERR_NO_DEVICE;
  }
  return FI_OK;
}

// Shared body of the two paged run calls.
// Checks of a run call's layout, scales and page stride (no device access).
fi_status check_run_scalars(const fi::Plan& P, int32_t kv_layout, int64_t page_stride_elems,
                            float sm_scale, float k_scale, float v_scale) {
  if (kv_layout != FI_LAYOUT_NHD && kv_layout != FI_LAYOUT_HND) return FI_ERR_INVALID_ARG;
  if (!(sm_scale >= 0.f) || sm_scale > 3.0e38f) return FI_ERR_INVALID_ARG;  // also rejects NaN
  if (!(k_scale > 0.f) || k_scale > 3.0e38f || !(v_scale > 0.f) || v_scale > 3.0e38f)
    return FI_ERR_INVALID_ARG;
  const int64_t page_elems = int64_t(P.page_size) * P.num_kv_heads * P.head_dim;
  if (page_stride_elems == 0) page_stride_elems = page_elems;
  // page starts 16-byte aligned for TMA
  if (page_stride_elems < page_elems || page_stride_elems % (16 / elem_bytes(P.kv_dtype)) != 0)
    return FI_ERR_INVALID_ARG;
  return FI_OK;
}

fi_status run_paged(fi_plan_t plan, bool prefill_call, const void* q, const int32_t* qo_indptr_d,
                    const void* k_cache, const void* v_cache, int32_t kv_layout,
                    int64_t page_stride_elems, int32_t num_pages, const int32_t* page_indptr_d,
                    const int32_t* page_indices_d, const int32_t* last_page_len_d, float sm_scale,
                    float k_scale, float v_scale, const float* k_head_scale,
                    const float* v_head_scale, void* out, float* lse, void* workspace,
                    size_t workspace_bytes, void* stream_ptr, Upload upload = Upload::kStaged) {
  if (!plan) return FI_ERR_INVALID_ARG;
  const fi::Plan& P = plan->p;
  if (P.mode != (prefill_call ? FI_MODE_PREFILL : FI_MODE_DECODE)) return FI_ERR_INVALID_ARG;
  if (P.batch == 0 || P.total_q == 0) return FI_OK;   // no query rows: nothing to run
  if (!q || !k_cache || !v_cache || !out || !workspace || !page_indptr_d || !last_page_len_d)
    return FI_ERR_INVALID_ARG;
  if (prefill_call && !qo_indptr_d) return FI_ERR_INVALID_ARG;
  if (P.total_kv > 0 && (!page_indices_d || num_pages <= 0)) return FI_ERR_INVALID_ARG;
  if (num_pages < 0) return FI_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(workspace, 256) || (lse && !aligned(lse, 4)) ||
      (k_head_scale && !aligned(k_head_scale, 4)) || (v_head_scale && !aligned(v_head_scale, 4)))
    return FI_ERR_INVALID_ARG;
  fi_status st = check_run_scalars(P, kv_layout, page_stride_elems, sm_scale, k_scale, v_scale);
  if (st != FI_OK) return st;
  const int64_t page_elems = int64_t(P.page_size) * P.num_kv_heads * P.head_dim;
  if (page_stride_elems == 0) page_stride_elems = page_elems;
  if (workspace_bytes < P.ws.total) return FI_ERR_WORKSPACE_TOO_SMALL;
  st = check_device();
  if (st != FI_OK) return st;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  // A captured copy would replay from a staging slot that later calls
  // refill, so run calls refuse stream capture instead of recording it.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
    g_last_error = "run calls cannot be captured into a CUDA graph";
    return FI_ERR_UNSUPPORTED;
  }
  // Upload header (zeroed error word and counters) + work lists + merge
  // tasks in one copy.
  if (upload == Upload::kStaged) st = upload_image(ws, P, stream);
  else if (upload == Upload::kStatic) st = upload_image_static(ws, P, stream);
  if (st != FI_OK) return st;
  cudaError_t e = cudaSuccess;

  CUtensorMap kmap, vmap;
  if (P.total_kv > 0) {
    st = kv_map(&kmap, k_cache, kv_layout, num_pages, P.page_size, P.num_kv_heads, P.head_dim,
                page_stride_elems, P.kv_dtype);
    if (st != FI_OK) return st;
    st = kv_map(&vmap, v_cache, kv_layout, num_pages, P.page_size, P.num_kv_heads, P.head_dim,
                page_stride_elems, P.kv_dtype);
    if (st != FI_OK) return st;
  } else {
    std::memset(&kmap, 0, sizeof(kmap));
    std::memset(&vmap, 0, sizeof(vmap));
  }
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);
  float* partial_o = reinterpret_cast<float*>(ws + P.ws.partial_o);
  float* partial_lse = reinterpret_cast<float*>(ws + P.ws.partial_lse);

  CUtensorMap qmap;
  if (!P.prefill_items.empty() || !P.prefix_items.empty()) {
    // prefill tiles hold 128 rows of one head; shared-prefix tiles 128 / g
    // rows of the g heads of a kv head (a decode plan has only the latter)
    st = q_map(&qmap, q, P.total_q, P.num_qo_heads,
                    P.prefix_items.empty() ? 1 : P.num_qo_heads / P.num_kv_heads, P.head_dim,
                    P.dtype);
    if (st != FI_OK) return st;
  }

  cudaEvent_t prof_start = g_prof_start, prof_stop = g_prof_stop;
  g_prof_start = g_prof_stop = nullptr;
  const int32_t fault_kind = g_fault_kind.exchange(0);  // one-shot
  const uint64_t wait_limit_ns = g_wait_limit_ns.load();
  if (prof_start) {
    e = cudaEventRecord(prof_start, stream);
    if (e != cudaSuccess) return cuda_fail(e, "profiling event");
  }

  // The launch parameters of the plan's prefill and decode work (both read
  // the work lists uploaded above).
  fi::PrefillParams pp;
  pp.items = reinterpret_cast<const fi::WorkItem*>(ws + P.ws.prefill_items);
  pp.qo_indptr = qo_indptr_d;
  pp.page_indptr = page_indptr_d;
  pp.last_page_len = last_page_len_d;
  pp.page_indices = page_indices_d;
  pp.num_pages = num_pages;
  pp.page_size = P.page_size;
  pp.num_qo_heads = P.num_qo_heads;
  pp.group = P.num_qo_heads / P.num_kv_heads;
  pp.pack = 1;
  pp.layout = kv_layout;
  pp.causal = P.causal;
  pp.window_left = P.window_left;
  pp.sm_scale = sm_scale * k_scale;   // the key scale folds into the score scale
  pp.v_scale = v_scale;
  pp.k_head_scale = k_head_scale;
  pp.v_head_scale = v_head_scale;
  pp.out = out;
  pp.lse = lse;
  pp.err = err;
  pp.wait_limit_ns = wait_limit_ns;
  pp.fault_kind = fault_kind;
  pp.n_items = int(P.prefill_items.size());
  pp.work_counter = reinterpret_cast<uint32_t*>(ws + fi::kWorkCounterOffset);
  pp.state_o = nullptr;
  pp.state_lse = nullptr;
  pp.piece_o = partial_o;
  pp.piece_lse = partial_lse;

  fi::DecodeParams dp;
  dp.items = reinterpret_cast<const fi::WorkItem*>(ws + P.ws.decode_items);
  dp.q = q;
  dp.page_indices = page_indices_d;
  dp.num_pages = num_pages;
  dp.page_size = P.page_size;
  dp.num_qo_heads = P.num_qo_heads;
  dp.layout = kv_layout;
  dp.sm_scale = sm_scale * k_scale;   // the key scale folds into the score scale
  dp.v_scale = v_scale;
  dp.k_head_scale = k_head_scale;
  dp.v_head_scale = v_head_scale;
  dp.out = out;
  dp.lse = lse;
  dp.partial_o = partial_o;
  dp.partial_lse = partial_lse;
  dp.merges = reinterpret_cast<const fi::MergeTask*>(ws + P.ws.merges);
  dp.merge_counters = reinterpret_cast<uint32_t*>(ws + P.ws.merge_counters);
  dp.err = err;
  dp.wait_limit_ns = wait_limit_ns;
  dp.fault_kind = fault_kind;
  dp.n_items = int(P.decode_items.size());
  // the decode kernel's item counter (the mixed kernel's decode side uses the
  // same word; a call launches one or the other)
  dp.work_counter = reinterpret_cast<uint32_t*>(ws + fi::kDecodeCounterOffset);

  const int group = P.num_qo_heads / P.num_kv_heads;
  const bool both = !P.prefill_items.empty() && !P.decode_items.empty();
  if (both && P.prefix_items.empty() &&
      fi::mixed_applies(P.head_dim, group, P.dtype, P.kv_dtype)) {
    // Chunked prefill and decode rows in one persistent launch: every CTA
    // runs prefill items on its tensor-core warps and decode items on its
    // decode warps, each side taking work from its own counter, so the
    // HBM-bound decode streams overlap the tensor-bound prefill tiles on
    // the same SMs.
    e = fi::launch_mixed(P.head_dim, group, P.dtype, qmap, kmap, vmap, pp, dp,
                         int(P.decode_items.size()),
                         reinterpret_cast<uint32_t*>(ws + fi::kDecodeCounterOffset), P.num_sms,
                         stream);
    if (e != cudaSuccess) return cuda_fail(e, "mixed launch");
  } else {
    // Otherwise, with both kinds of work, the decode kernel (HBM-bound) runs
    // on a side stream concurrently with the prefill kernel (tensor-bound),
    // which is launched first; the streams join at the end. Split decode
    // work is merged inside the decode kernel.
    SideStream side;
    cudaStream_t dstream = stream;
    if (both) {
      st = side_stream(&side);
      if (st != FI_OK) return st;
      e = cudaEventRecord(side.fork, stream);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(side.stream, side.fork, 0);
      if (e != cudaSuccess) return cuda_fail(e, "fork to the side stream");
      dstream = side.stream;
    }
    if (!P.prefill_items.empty()) {
      e = fi::launch_prefill(P.head_dim, P.dtype, qmap, kmap, vmap, pp, P.num_sms, stream);
      if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    }
    if (!P.prefill_merges.empty()) {
      // Split prefill tiles: each row's piece states, merged by log-sum-exp
      // into out and lse (same stream, after the prefill launch)
      fi::MergeParams mp;
      mp.v = partial_o;
      mp.s = partial_lse;
      mp.tasks = reinterpret_cast<const fi::MergeTask*>(ws + P.ws.prefill_merges);
      mp.S = 0;
      mp.H = P.num_qo_heads;
      mp.d = P.head_dim;
      mp.out = out;
      mp.lse = lse;
      mp.dtype = P.dtype;
      e = fi::launch_merge(mp, int(P.prefill_merges.size()), stream);
      if (e != cudaSuccess) return cuda_fail(e, "prefill merge launch");
    }
    if (!P.prefix_items.empty()) {
      // Shared prefixes: each group's rows of q against chunks of its prefix,
      // on the prefill kernel, writing fp32 states (row r of q -> slot
      // item.slot + r) that the decode kernel merges with the rest. Same
      // stream, before the decode launch.
      const int32_t* tables = reinterpret_cast<const int32_t*>(ws + P.ws.prefix_tables);
      const int G2 = 2 * P.num_prefix_groups;
      fi::PrefillParams xp = pp;
      xp.items = reinterpret_cast<const fi::WorkItem*>(ws + P.ws.prefix_items);
      xp.qo_indptr = tables;
      xp.page_indptr = tables + G2;
      xp.last_page_len = tables + 2 * G2;
      xp.pack = xp.group;
      xp.causal = 0;
      xp.window_left = -1;
      xp.out = nullptr;
      xp.lse = nullptr;
      xp.state_o = partial_o;
      xp.state_lse = partial_lse;
      xp.fault_kind = 0;
      xp.n_items = int(P.prefix_items.size());
      e = fi::launch_prefill(P.head_dim, P.dtype, qmap, kmap, vmap, xp, P.num_sms, stream);
      if (e != cudaSuccess) return cuda_fail(e, "shared-prefix launch");
    }
    if (!P.decode_items.empty()) {
      e = fi::launch_decode(P.head_dim, group, P.dtype, P.kv_dtype, kmap, vmap, dp,
                            int(P.decode_items.size()), P.num_sms, dstream);
      if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    }
    if (both) {
      e = cudaEventRecord(side.join, side.stream);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, side.join, 0);
      if (e != cudaSuccess) return cuda_fail(e, "join from the side stream");
    }
  }
  if (prof_stop) {
    e = cudaEventRecord(prof_stop, stream);
    if (e != cudaSuccess) return cuda_fail(e, "profiling event");
  }
  return FI_OK;
}

}  // namespace

fi_status fi::run_decode_static_upload(
    fi_plan_t plan, const void* q, const void* k_cache, const void* v_cache, int32_t kv_layout,
    int64_t page_stride_elems, int32_t num_pages, const int32_t* page_indptr_d,
    const int32_t* page_indices_d, const int32_t* last_page_len_d, float sm_scale, float k_scale,
    float v_scale, const float* k_head_scale,
    const float* v_head_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
    void* stream) {
  return run_paged(plan, false, q, nullptr, k_cache, v_cache, kv_layout, page_stride_elems,
                   num_pages, page_indptr_d, page_indices_d, last_page_len_d, sm_scale, k_scale,
                   v_scale, k_head_scale, v_head_scale, out, lse, workspace, workspace_bytes,
                   stream, Upload::kStatic);
}

extern "C" {

fi_status fi_plan(int32_t mode, int32_t batch_size, const int32_t* qo_indptr_h,
                  const int32_t* page_indptr_h, const int32_t* last_page_len_h,
                  int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t page_size, int32_t causal, const fi_plan_options* options,
                  int32_t num_sms, fi_plan_t* out_plan, size_t* workspace_bytes) {
  if (!out_plan || !workspace_bytes) return FI_ERR_INVALID_ARG;
  *out_plan = nullptr;
  fi_plan_s* p = new (std::nothrow) fi_plan_s;
  if (!p) return FI_ERR_INVALID_ARG;
  fi_status st = fi::build_plan(mode, batch_size, qo_indptr_h, page_indptr_h, last_page_len_h,
                                num_qo_heads, num_kv_heads, head_dim, page_size, causal, options,
                                num_sms, &p->p);
  if (st != FI_OK) {
    delete p;
    return st;
  }
  const fi::Plan& P = p->p;
  *out_plan = p;
  *workspace_bytes = P.ws.total;
  return FI_OK;
}

fi_status fi_plan_destroy(fi_plan_t plan) {
  delete plan;
  return FI_OK;
}

fi_status fi_plan_get_info(fi_plan_t plan, fi_plan_info* info) {
  if (!plan || !info) return FI_ERR_INVALID_ARG;
  const fi::Plan& P = plan->p;
  info->mode = P.mode;
  info->batch_size = P.batch;
  info->num_decode_items = int32_t(P.decode_items.size());
  info->num_prefill_items = int32_t(P.prefill_items.size());
  info->num_prefix_items = int32_t(P.prefix_items.size());
  info->num_prefix_groups = P.num_prefix_groups;
  info->num_items = info->num_decode_items + info->num_prefill_items + info->num_prefix_items;
  info->chunk_tokens = P.chunk_tokens;
  info->num_split_requests = P.num_split;
  info->num_partial_slots = P.num_slots;
  info->workspace_bytes = int64_t(P.ws.total);
  info->total_kv_tokens = P.total_kv;
  info->host_io_bytes = int64_t(P.ws.hio_total);
  return FI_OK;
}

fi_status fi_plan_get_work(fi_plan_t plan, int32_t* items_h, int32_t capacity,
                           int32_t* num_items) {
  if (!plan || !num_items) return FI_ERR_INVALID_ARG;
  const fi::Plan& P = plan->p;
  const int32_t n =
      int32_t(P.decode_items.size() + P.prefill_items.size() + P.prefix_items.size());
  *num_items = n;
  if (!items_h) return FI_OK;
  if (capacity < n) return FI_ERR_INVALID_ARG;
  // the first 8 fields of each item, as the header documents
  int32_t* dst = items_h;
  for (const auto* list : {&P.decode_items, &P.prefill_items, &P.prefix_items}) {
    for (const fi::WorkItem& w : *list) {
      const int32_t f[8] = {w.req, w.head, w.page_begin, w.n_pages, w.tok_begin, w.tok_end,
                            w.slot, w.q_row};
      std::memcpy(dst, f, sizeof(f));
      dst += 8;
    }
  }
  return FI_OK;
}

fi_status fi_batch_decode_paged(fi_plan_t plan, const void* q, const void* k_cache,
                                const void* v_cache, int32_t kv_layout,
                                int64_t page_stride_elems, int32_t num_pages,
                                const int32_t* page_indptr_d, const int32_t* page_indices_d,
                                const int32_t* last_page_len_d, float sm_scale, float k_scale,
                                float v_scale, const float* k_head_scale,
                                const float* v_head_scale, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return run_paged(plan, false, q, nullptr, k_cache, v_cache, kv_layout, page_stride_elems,
                   num_pages, page_indptr_d, page_indices_d, last_page_len_d, sm_scale, k_scale,
                   v_scale, k_head_scale, v_head_scale, out, lse, workspace, workspace_bytes,
                   stream);
}

fi_status fi_batch_prefill_paged(fi_plan_t plan, const void* q, const int32_t* qo_indptr_d,
                                 const void* k_cache, const void* v_cache, int32_t kv_layout,
                                 int64_t page_stride_elems, int32_t num_pages,
                                 const int32_t* page_indptr_d, const int32_t* page_indices_d,
                                 const int32_t* last_page_len_d, float sm_scale, float k_scale,
                                 float v_scale, const float* k_head_scale,
                                 const float* v_head_scale, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return run_paged(plan, true, q, qo_indptr_d, k_cache, v_cache, kv_layout, page_stride_elems,
                   num_pages, page_indptr_d, page_indices_d, last_page_len_d, sm_scale, k_scale,
                   v_scale, k_head_scale, v_head_scale, out, lse, workspace, workspace_bytes,
                   stream);
}

fi_status fi_batch_attention_host_async(
    fi_plan_t plan, const void* q_h, const int32_t* qo_indptr_h, const void* k_cache,
    const void* v_cache, int32_t kv_layout, int64_t page_stride_elems, int32_t num_pages,
    const int32_t* page_indptr_h, const int32_t* page_indices_h, const int32_t* last_page_len_h,
    float sm_scale, float k_scale, float v_scale, const float* k_head_scale,
    const float* v_head_scale, void* out_h, float* lse_h, void* workspace, size_t workspace_bytes,
    void* stream_ptr, uint64_t* ticket_out) {
  if (!plan || !ticket_out) return FI_ERR_INVALID_ARG;
  *ticket_out = 0;
  const fi::Plan& P = plan->p;
  const bool prefill = P.mode == FI_MODE_PREFILL;
  if (P.batch == 0 || P.total_q == 0) return FI_OK;   // no query rows: nothing to run
  if (!q_h || !out_h || !page_indptr_h || !last_page_len_h || !workspace || !k_cache ||
      !v_cache || (prefill && !qo_indptr_h) || (P.page_entries > 0 && !page_indices_h))
    return FI_ERR_INVALID_ARG;
  if (P.total_kv > 0 && num_pages <= 0) return FI_ERR_INVALID_ARG;
  if (num_pages < 0 || !aligned(workspace, 256) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return FI_ERR_INVALID_ARG;
  fi_status st = check_run_scalars(P, kv_layout, page_stride_elems, sm_scale, k_scale, v_scale);
  if (st != FI_OK) return st;
  if (workspace_bytes < P.ws.total + P.ws.hio_total) return FI_ERR_WORKSPACE_TOO_SMALL;
  st = check_device();
  if (st != FI_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t q_bytes = size_t(P.total_q) * P.num_qo_heads * P.head_dim * 2;
  const size_t lse_bytes = size_t(P.total_q) * P.num_qo_heads * sizeof(float);
  // device copies of the step's inputs, in the host-IO part of the workspace
  int32_t* tab = reinterpret_cast<int32_t*>(ws + P.ws.hio_tables);
  int32_t* indptr_d = tab;
  int32_t* indices_d = indptr_d + (P.batch + 1);
  int32_t* last_d = indices_d + P.page_entries;
  int32_t* qo_d = prefill ? last_d + P.batch : nullptr;
  const size_t table_bytes =
      (size_t(P.batch + 1) + P.page_entries + P.batch + (prefill ? P.batch + 1 : 0)) *
      sizeof(int32_t);
  // A captured copy would replay from a staging slot that later calls
  // refill (as in the run calls).
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
    g_last_error = "run calls cannot be captured into a CUDA graph";
    return FI_ERR_UNSUPPORTED;
  }
  HostSteps& hs = g_host_steps;
  st = host_steps_ready(hs);
  if (st != FI_OK) return st;
  const int slot = int(hs.next % kHostSteps);
  if (hs.ticket[slot]) {
    g_last_error = "more than 8 host-buffer steps in flight on this thread";
    return FI_ERR_INVALID_ARG;
  }
  // the work-list image and, right after it in the workspace, the page
  // table (and qo_indptr): one pinned staging fill, one copy; q comes
  // straight from the caller's buffer
  st = stage_and_copy(
      g_staging, ws, P.ws.hio_tables + table_bytes,
      [&](uint8_t* p) {
        fill_image(p, P);
        int32_t* t = reinterpret_cast<int32_t*>(p + P.ws.hio_tables);
        std::memcpy(t, page_indptr_h, size_t(P.batch + 1) * sizeof(int32_t));
        t += P.batch + 1;
        if (P.page_entries > 0)
          std::memcpy(t, page_indices_h, size_t(P.page_entries) * sizeof(int32_t));
        t += P.page_entries;
        std::memcpy(t, last_page_len_h, size_t(P.batch) * sizeof(int32_t));
        t += P.batch;
        if (prefill) std::memcpy(t, qo_indptr_h, size_t(P.batch + 1) * sizeof(int32_t));
      },
      stream, "work-list and page-table upload");
  if (st != FI_OK) return st;
  cudaError_t e = cudaMemcpyAsync(ws + P.ws.hio_q, q_h, q_bytes, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(e, "q upload");
  void* out_d = ws + P.ws.hio_out;
  float* lse_d = lse_h ? reinterpret_cast<float*>(ws + P.ws.hio_lse) : nullptr;
  st = run_paged(plan, prefill, ws + P.ws.hio_q, qo_d, k_cache, v_cache, kv_layout,
                 page_stride_elems, num_pages, indptr_d, indices_d, last_d, sm_scale, k_scale,
                 v_scale, k_head_scale, v_head_scale, out_d, lse_d, workspace, P.ws.total,
                 stream_ptr, Upload::kDone);
  if (st != FI_OK) return st;
  e = cudaMemcpyAsync(out_h, out_d, q_bytes, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess && lse_h)
    e = cudaMemcpyAsync(lse_h, lse_d, lse_bytes, cudaMemcpyDeviceToHost, stream);
  // the step's device status (error word at the start of the workspace)
  // into the slot's pinned word; the next step's upload zeroes the header
  hs.words[slot] = 0;
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&hs.words[slot], workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                        stream);
  if (e == cudaSuccess) e = cudaEventRecord(hs.done[slot], stream);
  if (e != cudaSuccess) return cuda_fail(e, "host-buffer step");
  hs.ticket[slot] = hs.next;
  *ticket_out = hs.next++;
  return FI_OK;
}

fi_status fi_host_step_wait(uint64_t ticket) {
  if (ticket == 0) return FI_OK;   // an empty step
  HostSteps& hs = g_host_steps;
  const int slot = int(ticket % kHostSteps);
  if (hs.device < 0 || hs.ticket[slot] != ticket) {
    g_last_error = "not a host-buffer step of this thread that is still to be waited for";
    return FI_ERR_INVALID_ARG;
  }
  const cudaError_t e = cudaEventSynchronize(hs.done[slot]);
  hs.ticket[slot] = 0;
  if (e != cudaSuccess) return cuda_fail(e, "host-buffer step");
  const uint32_t word = hs.words[slot];
  if (word & fi::kErrTimeout) return FI_ERR_DEVICE_TIMEOUT;
  if (word & fi::kErrBounds) return FI_ERR_DEVICE_BOUNDS;
  return FI_OK;
}

fi_status fi_batch_attention_host(fi_plan_t plan, const void* q_h, const int32_t* qo_indptr_h,
                                  const void* k_cache, const void* v_cache, int32_t kv_layout,
                                  int64_t page_stride_elems, int32_t num_pages,
                                  const int32_t* page_indptr_h, const int32_t* page_indices_h,
                                  const int32_t* last_page_len_h, float sm_scale, float k_scale,
                                  float v_scale, const float* k_head_scale,
                                  const float* v_head_scale, void* out_h, float* lse_h, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  uint64_t ticket = 0;
  const fi_status st = fi_batch_attention_host_async(
      plan, q_h, qo_indptr_h, k_cache, v_cache, kv_layout, page_stride_elems, num_pages,
      page_indptr_h, page_indices_h, last_page_len_h, sm_scale, k_scale, v_scale, k_head_scale,
      v_head_scale, out_h, lse_h, workspace, workspace_bytes, stream, &ticket);
  if (st != FI_OK) return st;
  return fi_host_step_wait(ticket);
}

fi_status fi_merge_states(const float* v, const float* s, int32_t n, int32_t S, int32_t H,
                          int32_t d, int32_t out_dtype, void* out, float* lse_out, void* stream) {
  if (n < 0 || S < 0 || H < 0 || d <= 0 || d % 4 != 0 || d > 1024) return FI_ERR_INVALID_ARG;
  if (out_dtype != FI_DTYPE_BF16 && out_dtype != FI_DTYPE_FP16) return FI_ERR_INVALID_ARG;
  if (n == 0 || H == 0) return FI_OK;
  if (!out || (S > 0 && (!v || !s))) return FI_ERR_INVALID_ARG;
  if (!aligned(out, 16) || (v && !aligned(v, 16)) || (s && !aligned(s, 4)) ||
      (lse_out && !aligned(lse_out, 4)))
    return FI_ERR_INVALID_ARG;
  fi_status st = check_device();
  if (st != FI_OK) return st;
  fi::MergeParams mp;
  mp.v = v;
  mp.s = s;
  mp.tasks = nullptr;
  mp.S = S;
  mp.H = H;
  mp.d = d;
  mp.out = out;
  mp.lse = lse_out;
  mp.dtype = out_dtype;
  cudaError_t e = fi::launch_merge(mp, n, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return FI_OK;
}

fi_status fi_check_device_status(void* workspace, void* stream_ptr) {
  if (!workspace) return FI_ERR_INVALID_ARG;
  fi_status st = check_device();
  if (st != FI_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(word), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "device status read");
  if (word & fi::kErrTimeout) return FI_ERR_DEVICE_TIMEOUT;
  if (word & fi::kErrBounds) return FI_ERR_DEVICE_BOUNDS;
  return FI_OK;
}

const char* fi_status_string(fi_status status) {
  switch (status) {
    case FI_OK: return "ok";
    case FI_ERR_INVALID_ARG: return "invalid argument";
    case FI_ERR_UNSUPPORTED: return "unsupported configuration";
    case FI_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FI_ERR_CUDA: return "CUDA error";
    case FI_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case FI_ERR_DEVICE_BOUNDS: return "page index outside the cache";
    case FI_ERR_NO_DEVICE: return "no CUDA device";
  }
  return "unknown status";
}

const char* fi_last_error_string(void) { return g_last_error.c_str(); }

fi_status fi_profile_next_launch(void* start_event, void* stop_event) {
  g_prof_start = static_cast<cudaEvent_t>(start_event);
  g_prof_stop = static_cast<cudaEvent_t>(stop_event);
  return FI_OK;
}

fi_status fi_debug_set_fault(int32_t kind, int64_t wait_limit) {
  if (kind < 0 || kind > 1) return FI_ERR_INVALID_ARG;
  g_wait_limit_ns.store(wait_limit > 0 ? uint64_t(wait_limit) : fi::kDefaultWaitLimitNs);
  g_fault_kind.store(kind);
  return FI_OK;
}

}  // extern "C"
