// Batch decode over a paged KV cache (one query row per request).
//
// One CTA per planned work item: a (request, kv head, KV chunk). The g query
// heads of the kv head's group share every K/V page the CTA loads (GQA
// sharing). Work is HBM-bound (about 1 flop per KV byte for g = 1), so the
// design is about moving bytes:
//   * a producer warp walks the page table and issues one TMA box per
//     (page, 64-dim slice) for K and for V, into a 3-stage shared-memory
//     ring (32 KB of K+V per stage) completed on mbarriers — no register
//     staging, as "FlashAttention-3 kernel integration in inference
//     engines", section 1 describes for TMA;
//   * 4 consumer warps read the staged rows (128-byte-swizzled, so reads
//     are bank-conflict free), compute scores with warp-shuffle reductions
//     ("FlashInfer Attention Kernel optimisation analysis", sections 1.3 and
//     2.1: warp-level reductions via __shfl_sync, no global sync) and keep a
//     running max / sum / accumulator (the online softmax of section 1 of the
//     FlashAttention-3 page), rescaling whenever the max grows;
//   * the warps' states are merged in shared memory; the CTA writes either
//     the final bf16 row + lse, or an fp32 partial state that the merge
//     kernel combines by log-sum-exp.
// Scores are kept in the log2 domain (q pre-scaled by sm_scale*log2(e)).
#include <cuda_bf16.h>

#include "fi_internal.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace fi {

namespace {

using namespace dev;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int HEAD_DIM, int GROUP>
struct DecodeCfg {
  static constexpr int TILE = 8192 / HEAD_DIM;         // tokens per stage (32 KB of K+V)
  static constexpr int NSTAGE = 3;
  static constexpr int NCW = 4;                        // consumer warps
  static constexpr int THREADS = 32 * (NCW + 1);       // + one producer warp
  static constexpr int LPT = HEAD_DIM / 8;             // lanes per token row (8 dims each)
  static constexpr int TPP = 32 / LPT;                 // token rows per warp pass
  static constexpr int TOK_PER_WARP = TILE / NCW;
  static constexpr int PASSES = TOK_PER_WARP / TPP;    // 8 for every head_dim
  static constexpr int SUB = GROUP >= 8 ? 2 : (GROUP >= 4 ? 4 : 8);  // passes per softmax step
  static constexpr int DBLK = HEAD_DIM / 64;           // 128-byte slices per row
  static constexpr int KBYTES = TILE * HEAD_DIM * 2;   // one K (or V) stage
  static constexpr int STAGE_BYTES = 2 * KBYTES;
  static constexpr int SMEM_BYTES = NSTAGE * STAGE_BYTES + 1024;  // + alignment slack
  static_assert(PASSES % SUB == 0, "");
  static_assert(NCW * GROUP * HEAD_DIM * 4 + 2 * NCW * GROUP * 4 <= NSTAGE * STAGE_BYTES, "");
};

// Byte offset of 16-byte chunk `c8` (0..7) of row `r` inside a 128-byte-row
// slice written by TMA with 128-byte swizzling (slice base 1024-aligned).
__device__ __forceinline__ uint32_t swz(int r, int c8) {
  return uint32_t(r * 128 + ((c8 ^ (r & 7)) << 4));
}

template <int HEAD_DIM, int GROUP>
__global__ void __launch_bounds__(DecodeCfg<HEAD_DIM, GROUP>::THREADS, 2)
decode_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
              DecodeParams prm) {
  using C = DecodeCfg<HEAD_DIM, GROUP>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::NSTAGE];
  __shared__ __align__(8) uint64_t empty_bar[C::NSTAGE];
  __shared__ int abort_flag;

  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem_base - smem_u32(smem_raw));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WorkItem item = prm.items[blockIdx.x];
  const int n_tok = item.tok_end - item.tok_begin;
  const int n_tiles = (n_tok + C::TILE - 1) / C::TILE;

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
    const int pages_per_tile = C::TILE / prm.page_size;
    const uint32_t box_bytes = uint32_t(prm.page_size) * 128u;
    int issued = 0;
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i % C::NSTAGE;
      if (i >= C::NSTAGE) {
        const uint32_t ph = ((i / C::NSTAGE) & 1) ^ 1;
        if (!mbar_wait_warp(smem_u32(&empty_bar[s]), ph, prm.wait_limit_ns, &abort_flag)) {
          if (lane == 0) { abort_flag = 1; atomicOr(prm.err, kErrTimeout); }
          break;
        }
      }
      const int tok0 = i * C::TILE;                         // relative to tok_begin
      const int tok_in_tile = min(C::TILE, n_tok - tok0);
      const int np = (tok_in_tile + prm.page_size - 1) / prm.page_size;
      int page = -1;
      bool valid = false;
      if (lane < np) {
        page = prm.page_indices[item.page_begin + i * pages_per_tile + lane];
        valid = page >= 0 && page < prm.num_pages;
        if (!valid) atomicOr(prm.err, kErrBounds);
      }
      const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
      const uint32_t bytes = uint32_t(__popc(vmask)) * 2u * C::DBLK * box_bytes;
      const uint32_t fb = smem_u32(&full_bar[s]);
      const bool skip = (prm.fault_kind == 1 && blockIdx.x == 0 && i == 0);
      if (lane == 0 && !skip) mbar_arrive_expect_tx(fb, bytes);
      __syncwarp();
      if (valid && !skip) {
        const uint32_t kdst = smem_base + s * C::STAGE_BYTES + lane * box_bytes;
        const uint32_t vdst = kdst + C::KBYTES;
#pragma unroll
        for (int c = 0; c < C::DBLK; ++c) {
          const uint32_t off = uint32_t(c) * C::TILE * 128u;
          if (prm.layout == FI_LAYOUT_NHD) {
            tma_load_4d(kdst + off, &k_map, fb, c * 64, item.head, 0, page);
            tma_load_4d(vdst + off, &v_map, fb, c * 64, item.head, 0, page);
          } else {
            tma_load_4d(kdst + off, &k_map, fb, c * 64, 0, item.head, page);
            tma_load_4d(vdst + off, &v_map, fb, c * 64, 0, item.head, page);
          }
        }
      }
      issued = i + 1;
    }
    // Before leaving, make sure no copy this CTA issued is still in flight.
    if (abort_flag) {
      for (int i = max(0, issued - C::NSTAGE); i < issued; ++i) {
        const bool skipped = (prm.fault_kind == 1 && blockIdx.x == 0 && i == 0);
        if (skipped) continue;
        mbar_wait_bounded(smem_u32(&full_bar[i % C::NSTAGE]), (i / C::NSTAGE) & 1,
                          prm.wait_limit_ns, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int ch = lane % C::LPT;            // 16-byte chunk of the row this lane owns
    const int ts = lane / C::LPT;            // token slot within a pass
    const int blk = ch >> 3, c8 = ch & 7;
    const float qscale = prm.sm_scale * kLog2e;
    float q[GROUP][8];
    {
      const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(prm.q) +
                                (size_t(item.q_row) * prm.num_qo_heads + item.head * GROUP) * HEAD_DIM +
                                ch * 8;
#pragma unroll
      for (int h = 0; h < GROUP; ++h) {
        const uint4 u = *reinterpret_cast<const uint4*>(qp + h * HEAD_DIM);
        unpack8(u, q[h]);
#pragma unroll
        for (int j = 0; j < 8; ++j) q[h][j] *= qscale;
      }
    }
    float m[GROUP], l[GROUP], acc[GROUP][8];
#pragma unroll
    for (int h = 0; h < GROUP; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[h][j] = 0.f;
    }

    for (int i = 0; i < n_tiles; ++i) {
      const int s = i % C::NSTAGE;
      if (!mbar_wait_warp(smem_u32(&full_bar[s]), (i / C::NSTAGE) & 1, prm.wait_limit_ns,
                          &abort_flag)) {
        if (lane == 0) { abort_flag = 1; atomicOr(prm.err, kErrTimeout); }
        break;
      }
      const int ntok = min(C::TILE, n_tok - i * C::TILE);
      const uint32_t kbase = smem_base + s * C::STAGE_BYTES + blk * C::TILE * 128;
      const uint32_t vbase = kbase + C::KBYTES;
#pragma unroll
      for (int p0 = 0; p0 < C::PASSES; p0 += C::SUB) {
        float sc[C::SUB][GROUP];
#pragma unroll
        for (int p = 0; p < C::SUB; ++p) {
          const int r = warp * C::TOK_PER_WARP + (p0 + p) * C::TPP + ts;
          float kf[8];
          unpack8(lds128(kbase + swz(r, c8)), kf);
#pragma unroll
          for (int h = 0; h < GROUP; ++h) {
            float d0 = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) d0 = fmaf(q[h][j], kf[j], d0);
#pragma unroll
            for (int off = C::LPT / 2; off >= 1; off >>= 1)
              d0 += __shfl_xor_sync(0xffffffffu, d0, off);
            sc[p][h] = (r < ntok) ? d0 : -INFINITY;
          }
        }
        float ref[GROUP];
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
          float mt = sc[0][h];
#pragma unroll
          for (int p = 1; p < C::SUB; ++p) mt = fmaxf(mt, sc[p][h]);
          const float m_new = fmaxf(m[h], mt);
          ref[h] = (m_new == -INFINITY) ? 0.f : m_new;
          const float alpha = ex2(m[h] - ref[h]);
          l[h] *= alpha;
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[h][j] *= alpha;
          m[h] = m_new;
        }
#pragma unroll
        for (int p = 0; p < C::SUB; ++p) {
          const int r = warp * C::TOK_PER_WARP + (p0 + p) * C::TPP + ts;
          if (r < ntok) {
            float vf[8];
            unpack8(lds128(vbase + swz(r, c8)), vf);
#pragma unroll
            for (int h = 0; h < GROUP; ++h) {
              const float pr = ex2(sc[p][h] - ref[h]);
              l[h] += pr;
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[h][j] = fmaf(pr, vf[j], acc[h][j]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
    }

    // merge the token slots of this warp
#pragma unroll
    for (int off = C::LPT; off < 32; off <<= 1) {
#pragma unroll
      for (int h = 0; h < GROUP; ++h) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
        const float lo = __shfl_xor_sync(0xffffffffu, l[h], off);
        const float mn = fmaxf(m[h], mo);
        const float rf = (mn == -INFINITY) ? 0.f : mn;
        const float a = ex2(m[h] - rf), b = ex2(mo - rf);
        l[h] = l[h] * a + lo * b;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float ao = __shfl_xor_sync(0xffffffffu, acc[h][j], off);
          acc[h][j] = acc[h][j] * a + ao * b;
        }
        m[h] = mn;
      }
    }

    // merge the consumer warps through shared memory (the ring is idle now)
    // every consumer thread takes the same decision (abort_flag may still
    // change while warps arrive, so it is voted on at the barrier)
    const bool aborted = named_bar_or(1, C::NCW * 32, abort_flag != 0);
    if (!aborted) {
      float* red_o = reinterpret_cast<float*>(smem_gen);               // [NCW][GROUP][D]
      float* red_m = red_o + C::NCW * GROUP * HEAD_DIM;                // [NCW][GROUP]
      float* red_l = red_m + C::NCW * GROUP;
      if (lane < C::LPT) {
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
          float4* dst = reinterpret_cast<float4*>(red_o + (warp * GROUP + h) * HEAD_DIM + ch * 8);
          dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
          dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
          if (lane == 0) {
            red_m[warp * GROUP + h] = m[h];
            red_l[warp * GROUP + h] = l[h];
          }
        }
      }
      named_bar_sync(1, C::NCW * 32);
      const int tid = threadIdx.x;
      for (int idx = tid; idx < GROUP * HEAD_DIM; idx += C::NCW * 32) {
        const int h = idx / HEAD_DIM, dd = idx % HEAD_DIM;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NCW; ++w) M = fmaxf(M, red_m[w * GROUP + h]);
        const float rf = (M == -INFINITY) ? 0.f : M;
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < C::NCW; ++w) {
          const float sc = ex2(red_m[w * GROUP + h] - rf);
          L = fmaf(red_l[w * GROUP + h], sc, L);
          O = fmaf(red_o[(w * GROUP + h) * HEAD_DIM + dd], sc, O);
        }
        const float o = (L > 0.f) ? O / L : 0.f;
        const float lse = (L > 0.f) ? (rf + lg2(L)) * kLn2 : -INFINITY;
        const int hq = item.head * GROUP + h;
        if (item.slot < 0) {
          reinterpret_cast<__nv_bfloat16*>(prm.out)[(size_t(item.q_row) * prm.num_qo_heads + hq) *
                                                        HEAD_DIM + dd] = __float2bfloat16_rn(o);
          if (dd == 0 && prm.lse) prm.lse[size_t(item.q_row) * prm.num_qo_heads + hq] = lse;
        } else {
          prm.partial_o[(size_t(item.slot) * prm.num_qo_heads + hq) * HEAD_DIM + dd] = o;
          if (dd == 0) prm.partial_lse[size_t(item.slot) * prm.num_qo_heads + hq] = lse;
        }
      }
    }
  }
}

template <int HEAD_DIM, int GROUP>
cudaError_t launch_decode_t(const CUtensorMap& km, const CUtensorMap& vm, const DecodeParams& p,
                            int n_items, cudaStream_t stream) {
  using C = DecodeCfg<HEAD_DIM, GROUP>;
  auto kern = decode_kernel<HEAD_DIM, GROUP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<n_items, C::THREADS, C::SMEM_BYTES, stream>>>(km, vm, p);
  return cudaGetLastError();
}

template <int HEAD_DIM>
cudaError_t launch_decode_d(int group, const CUtensorMap& km, const CUtensorMap& vm,
                            const DecodeParams& p, int n_items, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_decode_t<HEAD_DIM, 1>(km, vm, p, n_items, stream);
    case 2: return launch_decode_t<HEAD_DIM, 2>(km, vm, p, n_items, stream);
    case 4: return launch_decode_t<HEAD_DIM, 4>(km, vm, p, n_items, stream);
    case 8: return launch_decode_t<HEAD_DIM, 8>(km, vm, p, n_items, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(int head_dim, int group, const CUtensorMap& km, const CUtensorMap& vm,
                          const DecodeParams& p, int n_items, cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  switch (head_dim) {
    case 64: return launch_decode_d<64>(group, km, vm, p, n_items, stream);
    case 128: return launch_decode_d<128>(group, km, vm, p, n_items, stream);
    case 256: return launch_decode_d<256>(group, km, vm, p, n_items, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fi
