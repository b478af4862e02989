// Batch decode over a paged KV cache (one query row per request): one CTA
// per planned work item, a (request, kv head, KV chunk), with one producer
// warp and four consumer warps. The pipeline itself (TMA page gather into a
// ring, online softmax on CUDA cores or m16n8k16 MMAs, cross-warp and
// split-KV merges) is in decode_roles.cuh, shared with the mixed kernel.
#include "decode_roles.cuh"

namespace fi {

namespace {

template <int HEAD_DIM, int GROUP, class E, class KV>
__global__ void __launch_bounds__(
    (DecodeCfg<HEAD_DIM, GROUP, std::is_same<KV, E4m3>::value ? 1 : 2>::THREADS),
    (DecodeCfg<HEAD_DIM, GROUP, std::is_same<KV, E4m3>::value ? 1 : 2>::MIN_BLOCKS))
decode_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
              DecodeParams prm) {
  constexpr bool FP8 = std::is_same<KV, E4m3>::value;
  using C = DecodeCfg<HEAD_DIM, GROUP, FP8 ? 1 : 2>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::NSTAGE];
  __shared__ __align__(8) uint64_t empty_bar[C::NSTAGE];
  __shared__ int abort_flag;
  __shared__ int merge_last;

  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem_base - smem_u32(smem_raw));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WorkItem item = prm.items[blockIdx.x];
  // Tokens are counted from the start of the item's first page; the first
  // `lead` slots of that page precede the first visible key (a left window).
  const int lead = item.tok_begin % prm.page_size;
  const int n_tok = item.tok_end - item.tok_begin + lead;
  const int n_tiles = (n_tok + C::TILE - 1) / C::TILE;
  const bool skip_first = prm.fault_kind == 1 && blockIdx.x == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), C::NCW);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == C::NCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
    }
    const DecRing ring = contiguous_ring(smem_base, C::NSTAGE, full_bar, empty_bar);
    const int issued = decode_produce<HEAD_DIM, GROUP, KV, C::NSTAGE>(
        prm, item, n_tok, n_tiles, 0, skip_first, ring, &abort_flag, &k_map, &v_map);
    // Before leaving, make sure no copy this CTA issued is still in flight,
    // whether or not a consumer gave up (in a normal run the consumers have
    // already seen these phases complete, so the waits return at once).
    if (lane == 0) {
      for (int i = max(0, issued - C::NSTAGE); i < issued; ++i) {
        if (skip_first && i == 0) continue;
        mbar_wait_bounded(smem_u32(&full_bar[i % C::NSTAGE]), (i / C::NSTAGE) & 1,
                          prm.wait_limit_ns, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    // per-warp states for the cross-warp merge (the ring is idle by then)
    float* red_o = reinterpret_cast<float*>(smem_gen);               // [NCW][GROUP][D]
    float* red_m = red_o + C::NCW * GROUP * HEAD_DIM;                // [NCW][GROUP]
    float* red_l = red_m + C::NCW * GROUP;                           // exact weight sums
    float* red_lp = red_l + C::NCW * GROUP;                          // weights applied to O
    const DecRing ring = contiguous_ring(smem_base, C::NSTAGE, full_bar, empty_bar);
    bool aborted;
    if constexpr (!C::MMA)
      aborted = simt_consumer<HEAD_DIM, GROUP, E, KV, C::NSTAGE>(
          prm, item, n_tok, lead, n_tiles, 0, false, warp, ring, &abort_flag, red_o, red_m,
          red_l, red_lp);
    else
      aborted = mma_consumer<HEAD_DIM, GROUP, E, KV, C::NSTAGE>(
          prm, item, n_tok, lead, n_tiles, 0, false, warp, ring, &abort_flag, red_o, red_m,
          red_l, red_lp);
    if (!aborted)
      decode_finish<HEAD_DIM, GROUP, E, KV>(prm, item, threadIdx.x, true, red_o, red_m, red_l,
                                            red_lp, &merge_last);
  }
}

template <int HEAD_DIM, int GROUP, class E, class KV>
cudaError_t launch_decode_t(const CUtensorMap& km, const CUtensorMap& vm, const DecodeParams& p,
                            int n_items, cudaStream_t stream) {
  using C = DecodeCfg<HEAD_DIM, GROUP, std::is_same<KV, E4m3>::value ? 1 : 2>;
  auto kern = decode_kernel<HEAD_DIM, GROUP, E, KV>;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = once_per_device(configured, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::SMEM_BYTES);
  });
  if (e != cudaSuccess) return e;
  kern<<<n_items, C::THREADS, C::SMEM_BYTES, stream>>>(km, vm, p);
  return cudaGetLastError();
}

template <int HEAD_DIM, class E, class KV>
cudaError_t launch_decode_d(int group, const CUtensorMap& km, const CUtensorMap& vm,
                            const DecodeParams& p, int n_items, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_decode_t<HEAD_DIM, 1, E, KV>(km, vm, p, n_items, stream);
    case 2: return launch_decode_t<HEAD_DIM, 2, E, KV>(km, vm, p, n_items, stream);
    case 4: return launch_decode_t<HEAD_DIM, 4, E, KV>(km, vm, p, n_items, stream);
    case 8: return launch_decode_t<HEAD_DIM, 8, E, KV>(km, vm, p, n_items, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <class E, class KV>
cudaError_t launch_decode_e(int head_dim, int group, const CUtensorMap& km, const CUtensorMap& vm,
                            const DecodeParams& p, int n_items, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_decode_d<64, E, KV>(group, km, vm, p, n_items, stream);
    case 128: return launch_decode_d<128, E, KV>(group, km, vm, p, n_items, stream);
    case 256: return launch_decode_d<256, E, KV>(group, km, vm, p, n_items, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(int head_dim, int group, int dtype, int kv_dtype, const CUtensorMap& km,
                          const CUtensorMap& vm, const DecodeParams& p, int n_items,
                          cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  const bool fp8 = kv_dtype == FI_DTYPE_E4M3;
  if (dtype == FI_DTYPE_BF16)
    return fp8 ? launch_decode_e<Bf16, E4m3>(head_dim, group, km, vm, p, n_items, stream)
               : launch_decode_e<Bf16, Bf16>(head_dim, group, km, vm, p, n_items, stream);
  if (dtype == FI_DTYPE_FP16)
    return fp8 ? launch_decode_e<Fp16, E4m3>(head_dim, group, km, vm, p, n_items, stream)
               : launch_decode_e<Fp16, Fp16>(head_dim, group, km, vm, p, n_items, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fi
