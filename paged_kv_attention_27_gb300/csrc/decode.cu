// Batch decode over a paged KV cache (one query row per request). Work items
// are (request, kv head, KV chunk); each CTA has one producer warp and the
// consumer warps of its configuration. The pipeline itself (TMA page gather
// into a ring, online softmax on CUDA cores or m16n8k16 MMAs, cross-warp and
// split-KV merges) is in decode_roles.cuh, shared with the mixed kernel.
//
// With the SIMT consumer (DecodeCfg::PERSISTENT) the launch is persistent:
// as many CTAs as fit on the GPU at once, each starting with the item of its
// index and taking the next ones from a global counter (the planner lists
// items longest first). The producer runs on into the next item's pages
// while the consumers finish the current one, so no CTA pays a start-up
// (barriers, Q, the first page-table read and copy latency) per item. An
// item's cross-warp reduction uses the stage of its last tile, which the
// consumers release once the item is written. The other configurations run
// one item per CTA and reduce in the idle ring.
#include "decode_roles.cuh"

namespace fi {

namespace {

constexpr int kDecItemRing = 8;   // item indices handed from the producer to the consumers

template <int HEAD_DIM, int GROUP, class E, class KV>
__device__ __forceinline__ void decode_persistent(const CUtensorMap* k_map,
                                                  const CUtensorMap* v_map,
                                                  const DecodeParams& prm, uint32_t smem_base,
                                                  uint8_t* smem_gen) {
  constexpr bool FP8 = std::is_same<KV, E4m3>::value;
  using C = DecodeCfg<HEAD_DIM, GROUP, FP8 ? 1 : 2>;
  __shared__ __align__(8) uint64_t full_bar[C::NSTAGE];
  __shared__ __align__(8) uint64_t empty_bar[C::NSTAGE];
  __shared__ __align__(8) uint64_t item_full[kDecItemRing];
  __shared__ __align__(8) uint64_t item_empty[kDecItemRing];
  __shared__ int item_ring[kDecItemRing];
  __shared__ int abort_flag;
  __shared__ int merge_last;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = prm.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), C::NCW);
    }
    for (int s = 0; s < kDecItemRing; ++s) {
      mbar_init(smem_u32(&item_full[s]), 1);
      mbar_init(smem_u32(&item_empty[s]), C::NCW);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const DecRing ring = contiguous_ring(smem_base, C::NSTAGE, full_bar, empty_bar);

  if (warp == C::NCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(k_map);
      prefetch_tensormap(v_map);
    }
    bool ok = true;
    int r = 0;          // ring position of the next tile
    int issued = 0;     // ring positions whose copies were issued
    int skip_pos = -1;  // test hook: the position left without copies
    for (int n = 0; ok; ++n) {
      // the next item: this CTA's own first, then from the counter; handed
      // to the consumers through the item ring (-1: no more work)
      int idx = -1;
      if (lane == 0) {
        idx = n == 0 ? int(blockIdx.x) : int(gridDim.x + atomicAdd(prm.work_counter, 1u));
        if (idx >= prm.n_items || abort_flag) idx = -1;
        const int s = n % kDecItemRing;
        if (n >= kDecItemRing &&
            !mbar_wait_bounded(smem_u32(&item_empty[s]), ((n / kDecItemRing) & 1) ^ 1, limit,
                               &abort_flag)) {
          ok = false;
        } else {
          item_ring[s] = idx;
          mbar_arrive(smem_u32(&item_full[s]));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
      idx = __shfl_sync(0xffffffffu, idx, 0);
      if (!ok || idx < 0) break;
      const WorkItem item = prm.items[idx];
      const int lead = item.tok_begin % prm.page_size;
      const int n_tok = item.tok_end - item.tok_begin + lead;
      const int n_tiles = (n_tok + C::TILE - 1) / C::TILE;
      const bool skip = prm.fault_kind == 1 && blockIdx.x == 0 && n == 0 && n_tiles > 0;
      if (skip) skip_pos = r;
      const int done = decode_produce<HEAD_DIM, GROUP, KV, C::NSTAGE>(
          prm, item, n_tok, n_tiles, r, skip, ring, &abort_flag, k_map, v_map);
      issued = r + done;
      if (done < n_tiles) ok = false;
      r += n_tiles;
    }
    if (!ok && lane == 0) {
      abort_flag = 1;
      atomicOr(prm.err, kErrTimeout);
    }
    // Before leaving, make sure no copy this CTA issued is still in flight,
    // whether or not a consumer gave up (in a normal run the consumers have
    // already seen these phases complete, so the waits return at once).
    if (lane == 0) {
      for (int i = max(0, issued - C::NSTAGE); i < issued; ++i) {
        if (i == skip_pos) continue;
        mbar_wait_bounded(smem_u32(&full_bar[i % C::NSTAGE]), (i / C::NSTAGE) & 1, limit,
                          nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    int r = 0;
    for (int n = 0;; ++n) {
      int idx = -1;
      bool good = true;
      if (lane == 0) {
        const int s = n % kDecItemRing;
        good = mbar_wait_bounded(smem_u32(&item_full[s]), (n / kDecItemRing) & 1, limit,
                                 &abort_flag);
        if (good) idx = *reinterpret_cast<volatile int*>(&item_ring[s]);
        mbar_arrive(smem_u32(&item_empty[s]));
      }
      good = __shfl_sync(0xffffffffu, good, 0) != 0;
      idx = __shfl_sync(0xffffffffu, idx, 0);
      // the consumer warps leave together (a warp that left alone would
      // never reach their named barriers); all read the same index
      if (named_bar_or(2, C::NCW * 32, !good || idx < 0)) break;
      const WorkItem item = prm.items[idx];
      const int lead = item.tok_begin % prm.page_size;
      const int n_tok = item.tok_end - item.tok_begin + lead;
      const int n_tiles = (n_tok + C::TILE - 1) / C::TILE;
      // the reduction area: the stage of the item's last tile, held until
      // the item is written (an item without keys needs none)
      const bool hold = n_tiles > 0;
      const int last_stage = (r + n_tiles - 1) % C::NSTAGE;
      float* red_o = hold ? reinterpret_cast<float*>(smem_gen + last_stage * C::STAGE_BYTES)
                          : nullptr;
      float* red_m = red_o + C::NCW * GROUP * HEAD_DIM;
      float* red_l = red_m + C::NCW * GROUP;
      float* red_lp = red_l + C::NCW * GROUP;
      bool aborted;
      if (!hold)
        aborted = named_bar_or(1, C::NCW * 32, abort_flag != 0);
      else if constexpr (C::MMA)
        aborted = mma_consumer<HEAD_DIM, GROUP, E, KV, C::NSTAGE>(
            prm, item, n_tok, lead, n_tiles, r, true, warp, ring, &abort_flag, red_o, red_m,
            red_l, red_lp);
      else
        aborted = simt_consumer<HEAD_DIM, GROUP, E, KV, C::NSTAGE>(
            prm, item, n_tok, lead, n_tiles, r, true, warp, ring, &abort_flag, red_o, red_m,
            red_l, red_lp);
      if (aborted) break;   // voted: all consumer warps agree
      decode_finish<HEAD_DIM, GROUP, E, KV>(prm, item, threadIdx.x, hold, red_o, red_m, red_l,
                                            red_lp, &merge_last);
      if (hold) {
        // every consumer warp is done with the reduction area
        named_bar_sync(1, C::NCW * 32);
        if (lane == 0) mbar_arrive(smem_u32(&empty_bar[last_stage]));
      }
      r += n_tiles;
    }
  }
}

// One item per CTA (configurations whose reduction does not fit a stage):
// the consumers reduce in the ring, idle once the item's tiles are consumed.
template <int HEAD_DIM, int GROUP, class E, class KV>
__device__ __forceinline__ void decode_one_item(const CUtensorMap* k_map,
                                                const CUtensorMap* v_map,
                                                const DecodeParams& prm, uint32_t smem_base,
                                                uint8_t* smem_gen) {
  constexpr bool FP8 = std::is_same<KV, E4m3>::value;
  using C = DecodeCfg<HEAD_DIM, GROUP, FP8 ? 1 : 2>;
  __shared__ __align__(8) uint64_t full_bar[C::NSTAGE];
  __shared__ __align__(8) uint64_t empty_bar[C::NSTAGE];
  __shared__ int abort_flag;
  __shared__ int merge_last;
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
  const DecRing ring = contiguous_ring(smem_base, C::NSTAGE, full_bar, empty_bar);

  if (warp == C::NCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(k_map);
      prefetch_tensormap(v_map);
    }
    const int issued = decode_produce<HEAD_DIM, GROUP, KV, C::NSTAGE>(
        prm, item, n_tok, n_tiles, 0, skip_first, ring, &abort_flag, k_map, v_map);
    // no copy of this CTA may still be in flight when it leaves
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
__global__ void __launch_bounds__(
    (DecodeCfg<HEAD_DIM, GROUP, std::is_same<KV, E4m3>::value ? 1 : 2>::THREADS),
    (DecodeCfg<HEAD_DIM, GROUP, std::is_same<KV, E4m3>::value ? 1 : 2>::MIN_BLOCKS))
decode_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
              DecodeParams prm) {
  using C = DecodeCfg<HEAD_DIM, GROUP, std::is_same<KV, E4m3>::value ? 1 : 2>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem_base - smem_u32(smem_raw));
  if constexpr (C::PERSISTENT)
    decode_persistent<HEAD_DIM, GROUP, E, KV>(&k_map, &v_map, prm, smem_base, smem_gen);
  else
    decode_one_item<HEAD_DIM, GROUP, E, KV>(&k_map, &v_map, prm, smem_base, smem_gen);
}

template <int HEAD_DIM, int GROUP, class E, class KV>
cudaError_t launch_decode_t(const CUtensorMap& km, const CUtensorMap& vm, const DecodeParams& p,
                            int n_items, int num_sms, cudaStream_t stream) {
  using C = DecodeCfg<HEAD_DIM, GROUP, std::is_same<KV, E4m3>::value ? 1 : 2>;
  auto kern = decode_kernel<HEAD_DIM, GROUP, E, KV>;
  static std::atomic<uint64_t> configured{0};
  static int per_sm = 1;   // resident CTAs per SM (the same on every device of a process)
  cudaError_t e = once_per_device(configured, [&] {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    int b = 0;
    if (r == cudaSuccess)
      r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, C::THREADS, C::SMEM_BYTES);
    if (r == cudaSuccess) per_sm = b > 0 ? b : 1;
    return r;
  });
  if (e != cudaSuccess) return e;
  DecodeParams q = p;
  q.n_items = n_items;
  int grid = n_items;
  if (C::PERSISTENT) {
    const long long slots = (long long)(num_sms > 0 ? num_sms : 1) * per_sm;
    grid = int(slots < n_items ? slots : n_items);
  }
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(km, vm, q);
  return cudaGetLastError();
}

template <int HEAD_DIM, class E, class KV>
cudaError_t launch_decode_d(int group, const CUtensorMap& km, const CUtensorMap& vm,
                            const DecodeParams& p, int n_items, int num_sms,
                            cudaStream_t stream) {
  switch (group) {
    case 1: return launch_decode_t<HEAD_DIM, 1, E, KV>(km, vm, p, n_items, num_sms, stream);
    case 2: return launch_decode_t<HEAD_DIM, 2, E, KV>(km, vm, p, n_items, num_sms, stream);
    case 4: return launch_decode_t<HEAD_DIM, 4, E, KV>(km, vm, p, n_items, num_sms, stream);
    case 8: return launch_decode_t<HEAD_DIM, 8, E, KV>(km, vm, p, n_items, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <class E, class KV>
cudaError_t launch_decode_e(int head_dim, int group, const CUtensorMap& km, const CUtensorMap& vm,
                            const DecodeParams& p, int n_items, int num_sms,
                            cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_decode_d<64, E, KV>(group, km, vm, p, n_items, num_sms, stream);
    case 128: return launch_decode_d<128, E, KV>(group, km, vm, p, n_items, num_sms, stream);
    case 256: return launch_decode_d<256, E, KV>(group, km, vm, p, n_items, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(int head_dim, int group, int dtype, int kv_dtype, const CUtensorMap& km,
                          const CUtensorMap& vm, const DecodeParams& p, int n_items, int num_sms,
                          cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  const bool fp8 = kv_dtype == FI_DTYPE_E4M3;
  if (dtype == FI_DTYPE_BF16)
    return fp8 ? launch_decode_e<Bf16, E4m3>(head_dim, group, km, vm, p, n_items, num_sms, stream)
               : launch_decode_e<Bf16, Bf16>(head_dim, group, km, vm, p, n_items, num_sms, stream);
  if (dtype == FI_DTYPE_FP16)
    return fp8 ? launch_decode_e<Fp16, E4m3>(head_dim, group, km, vm, p, n_items, num_sms, stream)
               : launch_decode_e<Fp16, Fp16>(head_dim, group, km, vm, p, n_items, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fi
