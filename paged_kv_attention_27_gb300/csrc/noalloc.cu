// fi_batch_decode_paged_noalloc: batch decode for callers that cannot hand
// the library a workspace buffer.
//
// Some callers cannot allocate device memory at the point where they run
// attention: an engine plugin whose host framework owns every device byte
// and offers no scratch allocator, or a hot loop where a cudaMalloc (which
// may synchronise the device) is not acceptable. For them, the decode path's
// scratch — the uploaded work list, the device error word and the fp32
// split-KV partial states — lives in one file-scope device array of this
// library, kNoAllocScratchBytes (16 MiB) long. Every GPU that loads the
// library keeps that array until the process exits. The work list reaches it
// from a static host buffer of the same size, by an ordinary pageable
// cudaMemcpyAsync that the CUDA driver stages itself, so the call needs no
// pinned host memory either.
//
// Properties callers must know:
//   * the first call on a device looks up the array's device address for
//     that device (cudaGetSymbolAddress, with that device current) and caches
//     it;
//   * the call cannot be captured into a CUDA graph: a capturing stream is
//     refused with FI_ERR_UNSUPPORTED, checked before anything else touches
//     the device;
//   * every call, on every stream, shares the one array: calls whose GPU work
//     overlaps (different streams without ordering between them) race on it;
//   * plans whose workspace need exceeds kNoAllocScratchBytes are rejected
//     with FI_ERR_WORKSPACE_TOO_SMALL before anything is enqueued;
//   * the error word inside the array is cleared by each call's upload, but
//     it cannot be read back through fi_check_device_status (the caller has
//     no pointer to it); bounded waits and page-index checks still keep a
//     faulty input from hanging or faulting the GPU.
// This call allocates nothing, on the host or the device: it validates,
// resolves the array's address and runs the same decode kernel as
// fi_batch_decode_paged with that array as the workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "fi_internal.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[fi::kNoAllocScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" fi_status fi_batch_decode_paged_noalloc(
    fi_plan_t plan, const void* q, const void* k_cache, const void* v_cache, int32_t kv_layout,
    int64_t page_stride_elems, int32_t num_pages, const int32_t* page_indptr_d,
    const int32_t* page_indices_d, const int32_t* last_page_len_d, float sm_scale, float k_scale,
    float v_scale, const float* k_head_scale,
    const float* v_head_scale, void* out, float* lse, void* stream) {
  if (!plan) return FI_ERR_INVALID_ARG;
  if (plan->p.ws.total > fi::kNoAllocScratchBytes) return FI_ERR_WORKSPACE_TOO_SMALL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FI_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return FI_ERR_UNSUPPORTED;
  // refuse capture before the symbol lookup, which may load the module
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap) != cudaSuccess ||
      cap != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return FI_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return FI_ERR_CUDA;
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return fi::run_decode_static_upload(plan, q, k_cache, v_cache, kv_layout, page_stride_elems,
                                      num_pages, page_indptr_d, page_indices_d, last_page_len_d,
                                      sm_scale, k_scale, v_scale, k_head_scale, v_head_scale,
                                      out, lse, scratch,
                                      fi::kNoAllocScratchBytes, stream);
}
