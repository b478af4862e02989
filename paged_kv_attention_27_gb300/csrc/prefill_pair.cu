// Causal variable-length batch prefill over a paged KV cache, two query
// tiles per CTA: the two query heads of a pair within one kv group, on the
// same 128 rows, against every K/V tile they share.
//
// Why two tiles: with one 128-row tile per CTA the tensor core finishes a
// tile's two MMA groups (S = Q K^T, O += P V; 1024 cycles at its full rate)
// well before the softmax warps have turned that tile's scores into P, and
// then waits. With two tiles, each with its own softmax warpgroup and its own
// MMA-issuing warp, one tile's MMAs run while the other tile's softmax works
// (the ping-pong of the FlashAttention-3 page, section 1: two warpgroups
// alternating between softmax and GEMM, here on sm_103a's tcgen05 MMAs with
// TMEM accumulators), and each K/V tile copied into shared memory feeds
// twice the MMA work.
//
// Layout:
//   * TMEM (512 columns): S_0, S_1 (128 columns each), O_0, O_1 (head_dim
//     columns each). P_i, packed 16-bit pairs, is written over the first 64
//     columns of S_i once S_i has been read.
//   * shared memory: Q_0, Q_1 (both MMA operands of S come from shared
//     memory), a two-deep K ring and a two-deep V ring.
// Roles (12 warps):
//   * warps 0-3 / 4-7: softmax of tile 0 / tile 1 (thread = query row = TMEM
//     lane), then the epilogue of their tile;
//   * warp 8 / 9: MMA issuer of tile 0 / tile 1 (warp 8 owns the TMEM
//     allocation). Before issuing S_i of the next KV tile a warp waits for
//     its previous O_i += P_i V: P_i lives in S_i's columns, and O_i is then
//     settled for the softmax's rescale. The other tile's MMAs keep the
//     tensor core busy meanwhile;
//   * warp 10: Q of both tiles and the K tiles (one TMA box per page and
//     64-dim slice), and the work items; warp 11: the V tiles.
// The launch is persistent over pairs of the planner's work items (items 2p
// and 2p + 1: the same rows and keys, query heads h and h + 1 of one kv
// group), longest first, as in the one-tile kernel.
#include <cfloat>
#include <climits>
#include <type_traits>

#include "elem.cuh"
#include "fi_internal.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace fi {

namespace {

using namespace dev;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale when the max grows by > 2^8
constexpr int kItemRing = 8;

template <int HEAD_DIM, class E>
struct PairCfg {
  static_assert(HEAD_DIM == 64 || HEAD_DIM == 128, "two 128-row tiles fit TMEM up to d = 128");
  static constexpr int M = kPrefillTileM;                   // 128 query rows per tile
  static constexpr int N = 128;                             // KV tokens per tile
  static constexpr int DBLK = HEAD_DIM / 64;                // 128-byte slices of a row
  static constexpr int THREADS = 384;
  // registers per thread: 168 at launch (384 x 168 = 64512); the softmax
  // warpgroups take 224, the helper warpgroup (MMA issuers, copy producers)
  // keeps 56: 2 x 128 x 224 + 128 x 56 = 64512
  static constexpr uint32_t LAUNCH_REGS = 168, SOFTMAX_REGS = 224, HELPER_REGS = 56;
  static_assert(2 * 128 * SOFTMAX_REGS + 128 * HELPER_REGS == THREADS * LAUNCH_REGS, "");
  static constexpr int NST = 2;                             // K (and V) ring depth
  static constexpr int Q_BYTES = DBLK * M * 128;            // one tile's Q
  static constexpr int KV_BYTES = DBLK * N * 128;           // one K (or V) tile
  static constexpr int OFF_Q = 0;                           // Q_0, Q_1
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NST * KV_BYTES;
  static constexpr int USED = OFF_V + NST * KV_BYTES;
  // keep one CTA per SM (each CTA takes all 512 TMEM columns)
  static constexpr int SMEM_BYTES = (USED < 120 * 1024 ? 120 * 1024 : USED) + 1024;
  static_assert(SMEM_BYTES <= 226 * 1024, "shared-memory budget");
  static constexpr uint32_t TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t col_s(int i) { return uint32_t(i * N); }
  __host__ __device__ static constexpr uint32_t col_o(int i) {
    return uint32_t(2 * N + i * HEAD_DIM);
  }
  static_assert(2 * N + 2 * HEAD_DIM <= TMEM_COLS, "TMEM budget");
  // K-major Q and K (both from shared memory); K-major P (TMEM) with MN-major V
  static constexpr uint32_t IDESC_QK = idesc_f16kind(M, N, 0, 0, E::kMmaFmt);
  static constexpr uint32_t IDESC_PV = idesc_f16kind(M, HEAD_DIM, 0, 1, E::kMmaFmt);
};

struct PairBarriers {
  uint64_t item_full[kItemRing], item_empty[kItemRing];
  uint64_t q_full, q_empty;
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2], o_final[2], drain[2];
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

template <int N>
__device__ __forceinline__ int item_tiles(const WorkItem& w) {
  return (w.tok_end - w.tok_begin + N - 1) / N;
}

template <int HEAD_DIM, class E>
__global__ void __launch_bounds__(PairCfg<HEAD_DIM, E>::THREADS, 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap q_map,
                    const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, PrefillParams prm) {
  using C = PairCfg<HEAD_DIM, E>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) PairBarriers bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int item_ring[kItemRing];

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_pairs = prm.n_items / 2;
  const uint64_t limit = prm.wait_limit_ns;
  // pair indices, published one ahead by warp 10 in a shared-memory ring
  auto item_at = [&](int n, int& idx) {
    if (!mbar_wait_bounded(smem_u32(&bars.item_full[n % kItemRing]), (n / kItemRing) & 1,
                           limit, &abort_flag))
      return false;
    idx = *reinterpret_cast<volatile int*>(&item_ring[n % kItemRing]);
    return true;
  };
  auto item_done = [&](int n) { mbar_arrive(smem_u32(&bars.item_empty[n % kItemRing])); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(smem_u32(&bars.item_full[s]), 1);
      mbar_init(smem_u32(&bars.item_empty[s]), 11);   // 8 softmax warps, 2 MMA warps, V producer
    }
    mbar_init(smem_u32(&bars.q_full), 1);
    mbar_init(smem_u32(&bars.q_empty), 2);            // both tiles' last S of the item
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.k_empty[s]), 2);       // S of both tiles
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.v_empty[s]), 2);       // O of both tiles
      mbar_init(smem_u32(&bars.s_full[s]), 1);
      mbar_init(smem_u32(&bars.p_full[s]), 4);        // the tile's 4 softmax warps
      mbar_init(smem_u32(&bars.pv_done[s]), 1);
      mbar_init(smem_u32(&bars.o_final[s]), 1);
      mbar_init(smem_u32(&bars.drain[s]), 1);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(&tmem_base_sh), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  int issued = 0;   // producers: KV tiles whose copies this warp has issued
  int q_loads = 0;  // warp 10: Q pairs it has loaded

  // The launch holds exactly LAUNCH_REGS per thread (checked on the host
  // before the launch), so the register split of the two branches adds up.
  if (warp >= 8) {
    setmaxnreg_dec<C::HELPER_REGS>();
    if (warp >= 10) {
      // ------------------------------------------------------------ producers
      const bool is_v = warp == 11;
      if (lane == 0) {
        prefetch_tensormap(is_v ? &v_map : &k_map);
        if (!is_v) prefetch_tensormap(&q_map);
      }
      const CUtensorMap* map = is_v ? &v_map : &k_map;
      uint64_t* full = is_v ? bars.v_full : bars.k_full;
      uint64_t* empty = is_v ? bars.v_empty : bars.k_empty;
      const uint32_t ring = base + (is_v ? C::OFF_V : C::OFF_K);
      const int P = prm.page_size;
      const int ppt = C::N / P;
      const uint32_t box = uint32_t(P) * 128u;
      auto pages_in = [&](const WorkItem& w, int j) {
        return (min(C::N, w.tok_end - w.tok_begin - j * C::N) + P - 1) / P;
      };
      bool ok = true;
      int g = 0;
      auto publish = [&](int n, int value) {
        if (n >= kItemRing &&
            !mbar_wait_bounded(smem_u32(&bars.item_empty[n % kItemRing]),
                               ((n / kItemRing) & 1) ^ 1, limit, &abort_flag))
          return false;
        item_ring[n % kItemRing] = value;
        mbar_arrive(smem_u32(&bars.item_full[n % kItemRing]));   // release: the index is visible
        return true;
      };
      // pair n + 1 (n = -1: the first): warp 10 takes it from the global
      // counter (the first is blockIdx.x) and publishes it; warp 11 reads it
      auto next_pair = [&](int n, int& idx) {
        int v = -1;
        bool good = true;
        if (lane == 0) {
          if (!is_v) {
            v = n < 0 ? int(blockIdx.x) : int(gridDim.x + atomicAdd(prm.work_counter, 1u));
            if (v >= n_pairs) v = -1;
            good = publish(n + 1, v);
          } else {
            good = item_at(n + 1, v);
            item_done(n + 1);
          }
        }
        idx = __shfl_sync(0xffffffffu, v, 0);
        return __shfl_sync(0xffffffffu, good, 0) != 0;
      };
      int it = -1;
      ok = next_pair(-1, it);
      WorkItem w;
      if (ok && it >= 0) w = prm.items[2 * it];
      int next_page = -1;
      if (ok && it >= 0 && item_tiles<C::N>(w) > 0 && lane < pages_in(w, 0))
        next_page = prm.page_indices[w.page_begin + lane];
      for (int n = 0; ok && it >= 0; ++n) {
        const int nt = item_tiles<C::N>(w);
        const int kv_head = w.head / prm.group;
        const int c1 = prm.layout == FI_LAYOUT_NHD ? kv_head : 0;
        const int c2 = prm.layout == FI_LAYOUT_NHD ? 0 : kv_head;
        int it_next = -1;
        if (!next_pair(n, it_next)) {
          ok = false;
          break;
        }
        WorkItem wn;
        if (it_next >= 0) wn = prm.items[2 * it_next];
        if (!is_v) {
          // Q of both tiles, once both have issued their last S of the previous pair
          if (n >= 1) {
            ok = mbar_wait_warp(smem_u32(&bars.q_empty), (n - 1) & 1, limit, &abort_flag);
            if (!ok) break;
          }
          if (lane == 0) {
            const uint32_t qb = smem_u32(&bars.q_full);
            mbar_arrive_expect_tx(qb, 2 * C::Q_BYTES);
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
              for (int c = 0; c < C::DBLK; ++c)
                tma_load_3d(base + C::OFF_Q + i * C::Q_BYTES + c * C::M * 128, &q_map, qb, c * 64,
                            w.head + i, w.q_row);
          }
          q_loads = n + 1;
        }
        for (int j = 0; j < nt; ++j, ++g) {
          const int st = g % C::NST;
          const int np = pages_in(w, j);
          int page = -1;
          bool valid = false;
          if (lane < np) {
            page = next_page;
            valid = page >= 0 && page < prm.num_pages;
            if (!valid && !is_v) atomicOr(prm.err, kErrBounds);
          }
          if (j + 1 < nt) {
            if (lane < pages_in(w, j + 1))
              next_page = prm.page_indices[w.page_begin + (j + 1) * ppt + lane];
          } else if (it_next >= 0 && item_tiles<C::N>(wn) > 0 && lane < pages_in(wn, 0)) {
            next_page = prm.page_indices[wn.page_begin + lane];
          }
          const uint32_t bytes =
              uint32_t(__popc(__ballot_sync(0xffffffffu, valid))) * C::DBLK * box;
          if (g >= C::NST && !mbar_wait_warp(smem_u32(&empty[st]), ((g / C::NST) & 1) ^ 1,
                                             limit, &abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[st]);
          const bool skip = !is_v && g == 0 && prm.fault_kind == 1 && blockIdx.x == 0;
          if (lane == 0 && !skip) mbar_arrive_expect_tx(fb, bytes);
          __syncwarp();
          if (valid && !skip) {
            const uint32_t dst = ring + st * C::KV_BYTES + lane * box;
#pragma unroll
            for (int c = 0; c < C::DBLK; ++c)
              tma_load_4d(dst + c * C::N * 128, map, fb, c * 64, c1, c2, page);
          }
          issued = g + 1;
        }
        if (nt == 0 && it_next >= 0 && item_tiles<C::N>(wn) > 0 && lane < pages_in(wn, 0))
          next_page = prm.page_indices[wn.page_begin + lane];
        w = wn;
        it = it_next;
      }
      if (!ok && lane == 0) { abort_flag = 1; atomicOr(prm.err, kErrTimeout); }
      __syncwarp();
    } else {
      // ------------------------------------------------------------ MMA issuers
      const int i = warp - 8;   // this warp's tile
      if (lane == 0) {
        // descriptors are linear in the address field (bits 0-13 = addr >> 4),
        // so each MMA's descriptor is a base plus a compile-time offset
        const uint64_t qd0 = sdesc_sw128(base + C::OFF_Q + i * C::Q_BYTES, 16, 1024);
        const uint64_t kd0 = sdesc_sw128(base + C::OFF_K, 16, 1024);
        const uint64_t vd0 = sdesc_sw128(base + C::OFF_V, C::N * 128, 1024);
        const uint32_t s_col = tmem + C::col_s(i), o_col = tmem + C::col_o(i);
        bool ok = true;
        int g = 0;   // KV tiles of earlier pairs
        for (int n = 0; ok; ++n) {
          int it = -1;
          ok = item_at(n, it);
          item_done(n);
          if (!ok || it < 0) break;
          const int nt = item_tiles<C::N>(prm.items[2 * it]);
          ok = mbar_wait_bounded(smem_u32(&bars.q_full), n & 1, limit, &abort_flag);
          for (int j = 0; ok && j < nt; ++j) {
            const int gq = g + j, st = gq % C::NST;
            // (the K of later tiles was waited for while the previous tile's
            // softmax ran)
            if (j == 0)
              ok = mbar_wait_bounded(smem_u32(&bars.k_full[st]), (gq / C::NST) & 1, limit,
                                     &abort_flag);
            // S_i and P_i share columns, and the softmax rescales O_i after S_i
            // is full: the previous O_i += P_i V completes first
            if (ok && gq >= 1)
              ok = mbar_wait_bounded(smem_u32(&bars.pv_done[i]), (gq - 1) & 1, limit,
                                     &abort_flag);
            if (!ok) break;
            tc_fence_after();
            const uint64_t kd = kd0 + uint64_t((st * C::KV_BYTES) >> 4);
#pragma unroll
            for (int k = 0; k < HEAD_DIM / 16; ++k) {
              const uint64_t a = qd0 + uint64_t(((k >> 2) * C::M * 128 + (k & 3) * 32) >> 4);
              const uint64_t b = kd + uint64_t(((k >> 2) * C::N * 128 + (k & 3) * 32) >> 4);
              tc_mma_ss(s_col, a, b, C::IDESC_QK, k > 0 ? 1u : 0u);
            }
            tc_commit(smem_u32(&bars.s_full[i]));
            tc_commit(smem_u32(&bars.k_empty[st]));
            if (j == nt - 1) tc_commit(smem_u32(&bars.q_empty));
            // The next tile's K and this tile's V are waited for here, while the
            // softmax works on S_i: a wait costs this thread a few hundred
            // cycles even when its phase has long completed, and after P_i
            // that sat between the softmax and the PV (+5 % at 1K-16K).
            if (j + 1 < nt)
              ok = mbar_wait_bounded(smem_u32(&bars.k_full[(gq + 1) % C::NST]),
                                     ((gq + 1) / C::NST) & 1, limit, &abort_flag);
            if (ok)
              ok = mbar_wait_bounded(smem_u32(&bars.v_full[st]), (gq / C::NST) & 1, limit,
                                     &abort_flag);
            if (ok)
              ok = mbar_wait_bounded(smem_u32(&bars.p_full[i]), gq & 1, limit, &abort_flag);
            if (!ok) break;
            tc_fence_after();
            const uint64_t vd = vd0 + uint64_t((st * C::KV_BYTES) >> 4);
#pragma unroll
            for (int k = 0; k < C::N / 16; ++k) {
              // MN-major V: 16 tokens per step; the next 64 dims one slice further
              const uint64_t b = vd + uint64_t((k * 16 * 128) >> 4);
              tc_mma_ts(o_col, s_col + k * 8, b, C::IDESC_PV, (j > 0 || k > 0) ? 1u : 0u);
            }
            tc_commit(smem_u32(&bars.v_empty[st]));
            tc_commit(smem_u32(&bars.pv_done[i]));
          }
          if (!ok) break;
          if (nt == 0) tc_commit(smem_u32(&bars.q_empty));
          tc_commit(smem_u32(&bars.o_final[i]));
          g += nt;
        }
        if (!ok) {
          abort_flag = 1;
          atomicOr(prm.err, kErrTimeout);
          // every MMA issued so far completes before the TMEM is released
          tc_commit(smem_u32(&bars.drain[i]));
          mbar_wait_bounded(smem_u32(&bars.drain[i]), 0, limit, nullptr);
        }
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<C::SOFTMAX_REGS>();
    // ------------------------------------------------------------ softmax + epilogue
    const int i = warp >> 2;                          // this warpgroup's tile
    const int t = (warp & 3) * 32 + lane;             // M row of the tile = TMEM lane
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_off + C::col_s(i);
    const uint32_t o_col = tmem + lane_off + C::col_o(i);
    const float scale0 = prm.sm_scale * kLog2e;
    // Row bounds of pair w for this thread's row: the last key it may see
    // (causal bound, clipped to the keys), the first (left window; INT_MIN:
    // none) and the end of the request's rows.
    struct RowBounds { int q_end, t_max, t_min; };
    auto bounds_of = [&](const WorkItem& w) {
      const int q_start = prm.qo_indptr[w.req], q_end = prm.qo_indptr[w.req + 1];
      const int np_req = prm.page_indptr[w.req + 1] - prm.page_indptr[w.req];
      const int kv_len =
          np_req > 0 ? (np_req - 1) * prm.page_size + prm.last_page_len[w.req] : 0;
      const int pos = kv_len - (q_end - q_start) + (w.q_row - q_start + t);  // key position
      RowBounds r;
      r.q_end = q_end;
      r.t_max = min(prm.causal ? pos : kv_len - 1, kv_len - 1);
      r.t_min = prm.window_left >= 0 ? pos - prm.window_left : INT_MIN;
      return r;
    };
    auto take_item = [&](int n, int& idx) {
      int v = -1;
      bool good = true;
      if (lane == 0) {
        good = item_at(n, v);
        item_done(n);
      }
      idx = __shfl_sync(0xffffffffu, v, 0);
      return __shfl_sync(0xffffffffu, good, 0) != 0;
    };
    int g = 0;   // KV tiles of earlier pairs
    int it = -1;
    bool ok = take_item(0, it);
    WorkItem w;
    RowBounds rb;
    if (ok && it >= 0) {
      w = prm.items[2 * it];
      rb = bounds_of(w);
    }
    for (int n = 0; ok && it >= 0; ++n) {
      const int nt = item_tiles<C::N>(w);
      const int kv_head = w.head / prm.group;
      // this item's kv head: its key scale joins the score scale (at least
      // FLT_MIN: a hidden score is -inf, and -inf * 0 would be NaN; with
      // sm_scale = 0 every weight is still exactly 2^0 = 1), its value scale
      // the output
      const float scale =
          fmaxf(scale0 * (prm.k_head_scale ? prm.k_head_scale[kv_head] : 1.f), FLT_MIN);
      const float v_scale = prm.v_scale * (prm.v_head_scale ? prm.v_head_scale[kv_head] : 1.f);
      int it_next = -1;
      if (!take_item(n + 1, it_next)) {
        ok = false;
        break;
      }
      // l: sum of the exact weights (gives lse); lp: of the rounded weights
      // the PV MMA multiplies (normalises O)
      float m = -INFINITY, l = 0.f, lp = 0.f;
      // lp differs from l only where a row of the warp sees fewer than N keys
      // in all (from its first visible key to its last; one or two are
      // possible there): in the tiles that cross such a row's bounds, lp
      // adds the rounded weights. Elsewhere the rounding errors of many
      // weights average out and lp = l. The two cases run separate copies
      // of the tile loop: with the rounded sums compiled out, the loop
      // measured 1K +4 %, 4K +3 %.
      const bool few_keys =
          __any_sync(0xffffffffu, rb.t_max - (rb.t_min > 0 ? rb.t_min : 0) + 1 < C::N);
      auto tiles = [&](auto rounded_sums) {
      constexpr bool RS = decltype(rounded_sums)::value;
      for (int j = 0; j < nt; ++j, ++g) {
        const int kvst = g % C::NST;
        // The warpgroups take turns: tile g of warpgroup 1 after tile g of
        // warpgroup 0, tile g of warpgroup 0 after tile g - 1 of warpgroup 1,
        // so that one softmax runs while the tensor core works on the other
        // tile (run side by side, the two would share the schedulers and
        // keep pace, and the MMAs of both tiles would wait for both).
        const bool turn = i == 1 ? mbar_wait_warp(smem_u32(&bars.p_full[0]), g & 1, limit,
                                                  &abort_flag)
                                 : (g == 0 || mbar_wait_warp(smem_u32(&bars.p_full[1]),
                                                             (g - 1) & 1, limit, &abort_flag));
        if (!turn || !mbar_wait_warp(smem_u32(&bars.s_full[i]), g & 1, limit, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int col0 = w.tok_begin + j * C::N;   // key position of column 0
        // the columns of this tile the row may see: lo .. hi (a window's lower
        // bound, INT_MIN when there is none, gives lo = 0)
        const int hi = rb.t_max - col0;
        const int lo = rb.t_min > col0 ? rb.t_min - col0 : 0;
        const bool need_mask = __any_sync(0xffffffffu, hi < C::N - 1 || lo > 0);
        // The tile body in two copies: tiles that cross some row's bounds
        // (the mask, the rounded sums, the V zeroing of a last tile) and the
        // rest, which need none of it.
        auto body = [&](auto masked) -> bool {
        constexpr bool MK = decltype(masked)::value;
        // The row's 128 scores in registers (one wait), the row max
        // (sm_scale >= 0 commutes with max; two scores per three-input max)
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_col + c * 32, sr[c]);
        tmem_wait_ld();
        // In a tile that crosses the row's bounds the hidden scores become
        // -inf once, here: their weights are then exactly 0 (2^-inf), and the
        // rest of the softmax is the same code as in every other tile.
        if (MK) {
          if (prm.window_left < 0) {
#pragma unroll
            for (int k = 0; k < C::N; ++k)
              if (k > hi) sr[k >> 5][k & 31] = 0xff800000u;
          } else {
#pragma unroll
            for (int k = 0; k < C::N; ++k)
              if (k > hi || k < lo) sr[k >> 5][k & 31] = 0xff800000u;
          }
        }
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
        for (int k = 0; k < C::N; k += 2)
          mx8[(k >> 1) & 7] = fmax3(mx8[(k >> 1) & 7], __uint_as_float(sr[k >> 5][k & 31]),
                                    __uint_as_float(sr[k >> 5][(k + 1) & 31]));
        const float mx_raw = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                                   fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        const float m_tile = (mx_raw == -INFINITY) ? -INFINITY : mx_raw * scale;
        const float m_new = fmaxf(m, m_tile);
        const bool grow = m_new > m + kRescaleThreshold;
        const bool o_live = grow && (m != -INFINITY);  // O row holds data that must be rescaled
        float alpha = 1.f;
        if (grow) {
          alpha = ex2(m - m_new);
          l *= alpha;
          lp *= alpha;
          m = m_new;
        }
        // O_i is settled: its MMA warp issued this S only after the previous
        // O_i += P_i V had completed
        if (__any_sync(0xffffffffu, o_live)) {
#pragma unroll 1
          for (int c = 0; c < HEAD_DIM / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(o_col + c * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 y = __fmul2_rn(
                  make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                  make_float2(alpha, alpha));
              r[e] = __float_as_uint(y.x);
              r[e + 1] = __float_as_uint(y.y);
            }
            tmem_st32(o_col + c * 32, r);
          }
          tmem_wait_st();
        }
        const float ref = (m == -INFINITY) ? 0.f : m;
        // p = 2^(s * scale - ref): a packed FFMA per two scores, one ex2 each
        float s[C::N];
        const float2 sc2 = make_float2(scale, scale), nr2 = make_float2(-ref, -ref);
#pragma unroll
        for (int k = 0; k < C::N; k += 2) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[k >> 5][k & 31]),
                                                  __uint_as_float(sr[k >> 5][(k + 1) & 31])),
                                      sc2, nr2);
          s[k] = ex2(x.x);
          s[k + 1] = ex2(x.y);
        }
        float2 rs4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) rs4[e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < C::N; k += 2)
          rs4[(k >> 1) & 3] = __fadd2_rn(rs4[(k >> 1) & 3], make_float2(s[k], s[k + 1]));
        // P as packed 16-bit pairs over S_i's first 64 columns (all read
        // above). With RS, lp adds the rounded values the tensor core
        // multiplies in tiles that cross the row's bounds, the exact sum
        // elsewhere.
        float2 rsp2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          uint32_t wv[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) wv[e] = E::pack2(s[kb * 64 + 2 * e], s[kb * 64 + 2 * e + 1]);
          if (RS && MK) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              rsp2[e & 1] = __fadd2_rn(rsp2[e & 1], make_float2(E::lo(wv[e]), E::hi(wv[e])));
          }
          tmem_st32(s_col + kb * 32, wv);
        }
        tmem_wait_st();
        const float2 rs2 = __fadd2_rn(__fadd2_rn(rs4[0], rs4[1]), __fadd2_rn(rs4[2], rs4[3]));
        const float rs_tile = rs2.x + rs2.y;
        l += rs_tile;
        lp += (RS && MK) ? (rsp2[0].x + rsp2[0].y) + (rsp2[1].x + rsp2[1].y) : rs_tile;
        // Last tile: V rows past the valid keys may hold unused page slots or
        // stale data; zero them so that P = 0 there cannot meet a NaN. (Both
        // warpgroups write the same zeros; each orders its own writes before
        // its tile's MMA.)
        const int valid = w.tok_end - col0;
        if (MK && valid < C::N) {
          if (!mbar_wait_warp(smem_u32(&bars.v_full[kvst]), (g / C::NST) & 1, limit,
                              &abort_flag))
            return false;
          if (t >= valid) {
#pragma unroll
            for (int c = 0; c < C::DBLK; ++c)
#pragma unroll
              for (int c8 = 0; c8 < 8; ++c8)
                st_shared_v4(base + C::OFF_V + kvst * C::KV_BYTES + c * C::N * 128 + t * 128 +
                                 c8 * 16, 0u, 0u, 0u, 0u);
          }
        }
        return true;
        };
        if (!(need_mask ? body(std::true_type{}) : body(std::false_type{}))) {
          ok = false;
          break;
        }
        fence_proxy_async_smem();   // zeroed V rows (generic writes) before the MMA reads them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars.p_full[i]));
      }
      };
      if (few_keys)
        tiles(std::true_type{});
      else
        tiles(std::false_type{});
      if (!ok) break;
      // the next pair's bounds load while this pair's last PV completes
      WorkItem wn;
      RowBounds rn;
      if (it_next >= 0) {
        wn = prm.items[2 * it_next];
        rn = bounds_of(wn);
      }
      if (!mbar_wait_warp(smem_u32(&bars.o_final[i]), n & 1, limit, &abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // ---- epilogue: O / lp (the inputs' type), lse = ln(l) + m ln 2
      // (a piece of a split tile writes the row's fp32 state instead: O / l
      // times v_scale and lse, at slot item.slot + t * item.merge)
      const bool row_ok = w.q_row + t < rb.q_end;
      const float inv = lp > 0.f ? v_scale / lp : 0.f;
      const size_t out_row = size_t(w.q_row) + t;
      const int qo_head = w.head + i;
      const bool piece = w.merge > 0;
      const size_t srow = piece ? size_t(w.slot) + size_t(t) * size_t(w.merge) : 0;
      uint16_t* op = reinterpret_cast<uint16_t*>(prm.out) +
                     (out_row * prm.num_qo_heads + qo_head) * HEAD_DIM;
#pragma unroll 1
      for (int c0 = 0; c0 < HEAD_DIM / 32; c0 += 2) {
        uint32_t rb2[2][32];
        if (nt > 0) {
          tmem_ld32(o_col + c0 * 32, rb2[0]);
          tmem_ld32(o_col + (c0 + 1) * 32, rb2[1]);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int e = 0; e < 32; ++e) rb2[b][e] = 0u;
        }
        if (row_ok && piece) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            float4* dst = reinterpret_cast<float4*>(
                prm.piece_o + (srow * prm.num_qo_heads + qo_head) * HEAD_DIM + (c0 + b) * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float* f = reinterpret_cast<const float*>(rb2[b]) + q4 * 4;
              dst[q4] = make_float4(f[0] * inv, f[1] * inv, f[2] * inv, f[3] * inv);
            }
          }
        } else if (row_ok) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            uint4* dst = reinterpret_cast<uint4*>(op + (c0 + b) * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const float* f = reinterpret_cast<const float*>(rb2[b]) + q4 * 8;
              dst[q4] = make_uint4(E::pack2(f[0] * inv, f[1] * inv),
                                   E::pack2(f[2] * inv, f[3] * inv),
                                   E::pack2(f[4] * inv, f[5] * inv),
                                   E::pack2(f[6] * inv, f[7] * inv));
            }
          }
        }
      }
      float* lse_dst = piece ? prm.piece_lse : prm.lse;
      const size_t lrow = piece ? srow : out_row;
      if (row_ok && lse_dst)
        lse_dst[lrow * prm.num_qo_heads + qo_head] = l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
      // O has been read: the next pair's first PV (issued only after this
      // warp's next p_full arrival) may overwrite it
      tc_fence_before();
      w = wn;
      rb = rn;
      it = it_next;
    }
    if (!ok && lane == 0) {
      abort_flag = 1;
      atomicOr(prm.err, kErrTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // Each producer lets every copy it issued land before the CTA exits, also
  // after a timeout anywhere in the CTA.
  if ((warp == 10 || warp == 11) && lane == 0) {
    const bool is_v = warp == 11;
    uint64_t* full = is_v ? bars.v_full : bars.k_full;
    for (int j = max(0, issued - C::NST); j < issued; ++j) {
      if (!is_v && j == 0 && prm.fault_kind == 1 && blockIdx.x == 0) continue;  // never issued
      mbar_wait_bounded(smem_u32(&full[j % C::NST]), (j / C::NST) & 1, limit, nullptr);
    }
    if (!is_v && q_loads > 0)
      mbar_wait_bounded(smem_u32(&bars.q_full), (q_loads - 1) & 1, limit, nullptr);
  }
}

template <int HEAD_DIM, class E>
cudaError_t launch_pair_t(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                          const PrefillParams& p, int grid, cudaStream_t stream) {
  using C = PairCfg<HEAD_DIM, E>;
  auto kern = prefill_pair_kernel<HEAD_DIM, E>;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = once_per_device(configured, [&] {
    // the per-warpgroup register split assumes this launch allocation
    cudaFuncAttributes fa;
    cudaError_t r = cudaFuncGetAttributes(&fa, kern);
    if (r != cudaSuccess) return r;
    if (fa.numRegs != int(C::LAUNCH_REGS)) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::SMEM_BYTES);
  });
  if (e != cudaSuccess) return e;
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(qm, km, vm, p);
  return cudaGetLastError();
}

template <class E>
cudaError_t launch_pair_e(int head_dim, const CUtensorMap& qm, const CUtensorMap& km,
                          const CUtensorMap& vm, const PrefillParams& p, int grid,
                          cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_pair_t<64, E>(qm, km, vm, p, grid, stream);
    case 128: return launch_pair_t<128, E>(qm, km, vm, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool prefill_pair_applies(int head_dim, const PrefillParams& p) {
  return (head_dim == 64 || head_dim == 128) && p.pack == 1 && p.state_o == nullptr &&
         p.group % 2 == 0 && p.n_items % 2 == 0;
}

cudaError_t launch_prefill_pair(int head_dim, int dtype, const CUtensorMap& qm,
                                const CUtensorMap& km, const CUtensorMap& vm,
                                const PrefillParams& p, int grid, cudaStream_t stream) {
  const int n_pairs = p.n_items / 2;
  if (n_pairs <= 0 || grid <= 0) return cudaSuccess;
  grid = grid < n_pairs ? grid : n_pairs;
  switch (dtype) {
    case FI_DTYPE_BF16: return launch_pair_e<Bf16>(head_dim, qm, km, vm, p, grid, stream);
    case FI_DTYPE_FP16: return launch_pair_e<Fp16>(head_dim, qm, km, vm, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fi
