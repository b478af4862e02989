// Causal variable-length batch prefill over a paged KV cache, on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// A work item is 128 query rows of one request and one query head, against
// keys [tok_begin, tok_end) of that request (tok_end clipped to the causal
// bound of the tile's last row, tok_begin to the left window of its first).
// The launch is persistent: one CTA per SM works through items in the
// planner's longest-first order, taking the next one from a global counter
// when it starts loading the current one, so that one item's epilogue and
// the next item's first loads and scores overlap, and the per-CTA setup
// (barriers, TMEM allocation, pipeline fill) is paid once per SM.
// Warp-specialised, as the FlashAttention-3 page describes for Hopper
// (section 1: TMA producer warps, consumer warps driving the tensor cores,
// hardware barriers between them, ping-pong buffers), rebuilt for sm_103a:
//   * warps 4 and 6 (producers): TMA loads of each item's Q tile and, per KV
//     tile of N tokens, one 128B-swizzled box per (page, 64-dim slice) of K
//     (warp 4) and of V (warp 6) into K and V rings (three deep for
//     head_dim <= 128) that run on across items;
//   * warp 5 (MMA issuer; also owns the TMEM allocation): one thread issues
//     S_j = Q K_j^T into a double-buffered S region of TMEM, then
//     O += P_{j-1} V_{j-1} into an O region of TMEM, so that the tensor core
//     computes the next scores while the softmax warps work. The A operands
//     (Q and P) are read from TMEM: with both operands in shared memory an
//     M=128, N=128 MMA alone would use all of the shared memory bandwidth,
//     which the K/V copies also need. At head_dim 256, O and Q leave no
//     TMEM columns for P, so P is written over the S buffer it came from;
//   * warps 0-3 (softmax, thread = query row = TMEM lane): copy their Q row
//     into TMEM per item, then per tile read the S row with tcgen05.ld, apply the
//     causal mask, keep the running max and sums (online softmax, the
//     section-1 FA-1/2 idea), write P as packed 16-bit pairs (the inputs'
//     type, bf16 or fp16) into TMEM for the PV MMA, and rescale the O row in
//     TMEM only when the running max grew by more than 2^8 (the rescale guard
//     the same page's section 4 says must stay on; skipping smaller growths
//     is exact because O and the row sums share the stale reference);
//   * the same warps finish with O / l, write out (inputs' type) and the
//     fp32 lse.
// Fully masked KV tiles are never visited: the planner clips tok_end.
#include <cfloat>
#include <climits>
#include <type_traits>

#include "decode_roles.cuh"
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

// DG > 0: the mixed kernel, which also runs batch decode (groups of DG query
// heads per kv head) on warps 7-11 of the same CTA.
template <int HEAD_DIM, class E, int DG = 0>
struct PrefillCfg {
  static constexpr int M = kPrefillTileM;                   // 128 query rows
  static constexpr int N = HEAD_DIM <= 128 ? 128 : 64;      // KV tokens per tile
  static constexpr int DBLK = HEAD_DIM / 64;                // 128-byte slices of a row
  static constexpr bool MIXED = DG > 0;
  using DC = DecodeCfg<HEAD_DIM, (DG > 0 ? DG : 1), 2>;
  // 4 softmax warps, K producer, MMA issuer, V producer; the mixed kernel
  // adds a decode producer (warp 7) and four decode consumer warps (8-11):
  // on CUDA cores, or as two sets of two m16n8k16 warps taking turns on
  // stages (two warps alone could not keep pace with one SM's share of HBM)
  static constexpr int DEC_PAIRS = (MIXED && DC::MMA) ? 2 : 1;
  static constexpr int DEC_WARPS = DC::NCW * DEC_PAIRS;
  static constexpr int THREADS = MIXED ? 256 + 32 * DEC_WARPS : 224;
  static_assert(!MIXED || DEC_WARPS * DG * HEAD_DIM * 4 + 3 * DEC_WARPS * DG * 4 <=
                              DC::STAGE_BYTES, "reduction area within one decode stage");
  // d = 256 leaves no TMEM columns for P: P of tile g is written over its
  // S buffer (g & 1), which the MMA issuer then frees after that tile's PV
  static constexpr bool P_IN_S = HEAD_DIM > 128;
  static constexpr int NST = HEAD_DIM <= 128 ? 3 : 2;       // K (and V) ring depth
  static constexpr int Q_BYTES = DBLK * M * 128;
  static constexpr int KV_BYTES = DBLK * N * 128;           // one K (or V) tile
  // The mixed kernel stages each item's Q through two slots of the K ring
  // (the K producer loads it there, the softmax warps copy it into TMEM and
  // the MMA issuer frees the slots), which leaves room for the decode ring.
  static constexpr bool Q_IN_RING = MIXED;
  static_assert(!Q_IN_RING || Q_BYTES == 2 * KV_BYTES, "Q fills two K-ring slots");
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + (Q_IN_RING ? 0 : Q_BYTES);
  static constexpr int OFF_V = OFF_K + NST * KV_BYTES;
  static constexpr int OFF_DEC = OFF_V + NST * KV_BYTES;    // decode ring (mixed kernel)
  static constexpr int USED = OFF_DEC + (MIXED ? DC::NSTAGE * DC::STAGE_BYTES : 0);
  // mixed kernel: once a CTA's prefill side has no more items, the prefill K
  // and V rings (contiguous from OFF_K) join the decode ring as further stages
  static constexpr int DEC_STAGES_EXT =
      MIXED ? DC::NSTAGE + (OFF_DEC - OFF_K) / DC::STAGE_BYTES : 1;
  static_assert(!MIXED || (OFF_DEC - OFF_K) % DC::STAGE_BYTES == 0, "");
  // mixed kernel (384 threads): the softmax warpgroup raises its registers
  // to 224 per thread, the helper warpgroup (prefill producers, MMA issuer,
  // decode producer) lowers them to 64, the decode consumer warpgroup raises
  // them to 184. The shares fit the launch allocation of R per thread when
  // 128 x (224 + 64 + 184) <= 384 x R, i.e. R >= 158 (the compiler's cap for
  // 384 threads is 168); the host checks the compiled R before the launch.
  static constexpr uint32_t SOFTMAX_REGS = 224, HELPER_REGS = 64, DECODE_REGS = 184;
  static constexpr uint32_t MIN_LAUNCH_REGS =
      (128 * (SOFTMAX_REGS + HELPER_REGS + DECODE_REGS) + 383) / 384;
  static_assert(!MIXED || THREADS == 384, "four warpgroups");
  static_assert(!MIXED || HEAD_DIM == 256, "mixed kernel: head_dim 256");
  // keep one CTA per SM (each CTA takes all 512 TMEM columns)
  static constexpr int SMEM_BYTES = (USED < 120 * 1024 ? 120 * 1024 : USED) + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM columns: two S buffers, O, then (packed 16-bit pairs) Q and P
  static constexpr uint32_t COL_S = 0;                      // [0,N), [N,2N)
  static constexpr uint32_t COL_O = 2 * N;                  // [2N, 2N+HEAD_DIM)
  static constexpr uint32_t COL_Q = COL_O + HEAD_DIM;       // HEAD_DIM/2 columns
  static constexpr uint32_t COL_P = COL_Q + HEAD_DIM / 2;   // N/2 columns (unless P_IN_S)
  static_assert((P_IN_S ? COL_P : COL_P + N / 2) <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared-memory budget");
  // K-major Q and K; K-major P with MN-major V; A and B of the element type
  static constexpr uint32_t IDESC_QK = idesc_f16kind(M, N, 0, 0, E::kMmaFmt);
  static constexpr uint32_t IDESC_PV = idesc_f16kind(M, HEAD_DIM, 0, 1, E::kMmaFmt);
};

constexpr int kItemRing = 8;   // item indices handed from the K producer to the other roles

template <int NST, int DNST, int DNST2>
struct PrefillBarriers {
  uint64_t item_full[kItemRing], item_empty[kItemRing];
  uint64_t q_full, q_tmem;
  uint64_t k_full[NST], k_empty[NST];
  uint64_t v_full[NST], v_empty[NST];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, pv_done, o_final, drain;
  // mixed kernel: the decode ring and the decode items handed from the
  // decode producer to the decode consumers
  uint64_t d_full[DNST], d_empty[DNST];
  uint64_t ditem_full[kItemRing], ditem_empty[kItemRing];
  // the extended decode ring (the decode stages plus the prefill K and V
  // rings, once this CTA's prefill side has no more work)
  uint64_t e_full[DNST2], e_empty[DNST2];
};




__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Number of KV tiles of an item: keys [tok_begin, tok_end), N per tile.
template <int N>
__device__ __forceinline__ int item_tiles(const WorkItem& w) {
  return (w.tok_end - w.tok_begin + N - 1) / N;
}

// The kernel body, shared by prefill_kernel (DG = 0) and mixed_kernel
// (DG > 0: decode work items dprm.items[0 .. n_dec) run on warps 7-11 of the
// same CTAs, taken from *dec_counter).
template <int HEAD_DIM, class E, int DG>
__device__ __forceinline__ void prefill_body(const CUtensorMap& q_map, const CUtensorMap& k_map,
                                             const CUtensorMap& v_map, const PrefillParams& prm,
                                             const DecodeParams& dprm, int n_dec,
                                             uint32_t* dec_counter) {
  using C = PrefillCfg<HEAD_DIM, E, DG>;
  using DC = typename C::DC;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8)
      PrefillBarriers<C::NST, C::MIXED ? DC::NSTAGE : 1, C::MIXED ? C::DEC_STAGES_EXT : 1> bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int item_ring[kItemRing];
  __shared__ int ditem_ring[C::MIXED ? kItemRing : 1];
  __shared__ int dec_merge_last;
  __shared__ int prefill_free;   // mixed kernel: the prefill side is done, its rings are idle

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = prm.n_items;
  const uint64_t limit = prm.wait_limit_ns;
  // Items are handed out in the planner's longest-first order as CTAs get
  // free: a CTA's first item is blockIdx.x, later ones come from a global
  // counter, so the items in flight across the GPU stay neighbours in the
  // list (they share K/V through the L2) and the load stays balanced. The K
  // producer takes the indices and publishes them, one item ahead, in a
  // small shared-memory ring that the other roles read in order; all
  // barrier phases count this CTA's items (n) or KV tiles (g).
  auto item_at = [&](int n, int& idx) {   // consumer side, one thread per role-warp
    if (!mbar_wait_bounded(smem_u32(&bars.item_full[n % kItemRing]), (n / kItemRing) & 1,
                           limit, &abort_flag))
      return false;
    idx = *reinterpret_cast<volatile int*>(&item_ring[n % kItemRing]);
    return true;
  };
  auto item_done = [&](int n) {
    mbar_arrive(smem_u32(&bars.item_empty[n % kItemRing]));
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(smem_u32(&bars.item_full[s]), 1);
      mbar_init(smem_u32(&bars.item_empty[s]), 6);   // V producer, MMA issuer, 4 softmax warps
    }
    mbar_init(smem_u32(&bars.q_full), 1);
    mbar_init(smem_u32(&bars.q_tmem), 4);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.k_empty[s]), 1);
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.v_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars.s_full[s]), 1);
      // S buffer free: read by the 4 softmax warps, or (P over S) read by the PV
      mbar_init(smem_u32(&bars.s_free[s]), C::P_IN_S ? 1 : 4);
    }
    mbar_init(smem_u32(&bars.p_full), 4);
    mbar_init(smem_u32(&bars.pv_done), 1);
    mbar_init(smem_u32(&bars.o_final), 1);
    mbar_init(smem_u32(&bars.drain), 1);
    if constexpr (C::MIXED) {
      for (int s = 0; s < DC::NSTAGE; ++s) {
        mbar_init(smem_u32(&bars.d_full[s]), 1);
        mbar_init(smem_u32(&bars.d_empty[s]), DC::NCW);
      }
      for (int s = 0; s < kItemRing; ++s) {
        mbar_init(smem_u32(&bars.ditem_full[s]), 1);
        mbar_init(smem_u32(&bars.ditem_empty[s]), C::DEC_WARPS);
      }
      for (int s = 0; s < C::DEC_STAGES_EXT; ++s) {
        mbar_init(smem_u32(&bars.e_full[s]), 1);
        mbar_init(smem_u32(&bars.e_empty[s]), DC::NCW);
      }
    }
    prefill_free = 0;
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&tmem_base_sh), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  int issued = 0;    // producers: ring positions whose copies this warp has issued
  int q_loads = 0;   // K producer: Q tiles it has loaded (Q outside the K ring)
  int skip_pos = -1; // K producer: the ring position the test hook left unloaded
  bool dec_extended = false;  // mixed kernel, decode producer: on the extended ring

  // Role dispatch by warpgroup; in the mixed kernel each warpgroup sets its
  // register share first (one setmaxnreg per warpgroup, so that every code
  // path after it stays within that share): warps 0-3 compute the softmax of
  // whole rows, the helpers (warps 4-7) need few registers, the decode
  // consumers (warps 8-11) hold the MMA fragments of a 256-dim row.
  if (warp < 4) {
    if constexpr (C::MIXED) setmaxnreg_inc<C::SOFTMAX_REGS>();
    // ------------------------------------------------------------ softmax + epilogue
    const int t = threadIdx.x;                       // M row of the tile = TMEM lane
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    // M row t holds query head head * pack + t % pack of q row q_row + t / pack
    // (pack > 1: heads of one kv head sharing every K/V tile)
    const int t_row = t / prm.pack, t_head = t % prm.pack;
    const float scale0 = prm.sm_scale * kLog2e;
    // Row bounds of item w for this thread's row: the last key it may see
    // (causal bound, clipped to the keys), the first (left window; INT_MIN:
    // none) and the end of the request's rows.
    struct RowBounds { int q_end, t_max, t_min; };
    auto bounds_of = [&](const WorkItem& w) {
      const int q_start = prm.qo_indptr[w.req], q_end = prm.qo_indptr[w.req + 1];
      const int np_req = prm.page_indptr[w.req + 1] - prm.page_indptr[w.req];
      const int kv_len =
          np_req > 0 ? (np_req - 1) * prm.page_size + prm.last_page_len[w.req] : 0;
      const int pos = kv_len - (q_end - q_start) + (w.q_row - q_start + t_row);  // key position
      RowBounds r;
      r.q_end = q_end;
      r.t_max = min(prm.causal ? pos : kv_len - 1, kv_len - 1);
      r.t_min = prm.window_left >= 0 ? pos - prm.window_left : INT_MIN;
      return r;
    };
    // Q of item n: from the swizzled TMA tile into this thread's TMEM lane
    // (16-bit pairs), then one arrival per warp on q_tmem.
    // (Q staged in the K ring: its slots are at K-ring positions kq, kq + 1,
    // 64-dim slices 2h and 2h + 1 in slot h.)
    auto copy_q = [&](int n, int kq) {
      if constexpr (C::Q_IN_RING) {
        if (!mbar_wait_warp(smem_u32(&bars.k_full[kq % C::NST]), (kq / C::NST) & 1, limit,
                            &abort_flag) ||
            !mbar_wait_warp(smem_u32(&bars.k_full[(kq + 1) % C::NST]), ((kq + 1) / C::NST) & 1,
                            limit, &abort_flag))
          return false;
      } else {
        if (!mbar_wait_warp(smem_u32(&bars.q_full), n & 1, limit, &abort_flag)) return false;
      }
#pragma unroll
      for (int b = 0; b < C::DBLK; ++b) {
        uint32_t r[32];
        const uint32_t slice =
            C::Q_IN_RING ? base + C::OFF_K + ((kq + b / 2) % C::NST) * C::KV_BYTES +
                               (b % 2) * C::M * 128
                         : base + C::OFF_Q + b * C::M * 128;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const uint4 v = lds128(slice + swz(t, c8));
          r[c8 * 4 + 0] = v.x;
          r[c8 * 4 + 1] = v.y;
          r[c8 * 4 + 2] = v.z;
          r[c8 * 4 + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + C::COL_Q + b * 32, r);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.q_tmem));
      return true;
    };

    // index of item n from the ring (lane 0 reads, the warp gets a copy)
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
    int g = 0;    // KV tiles of earlier items
    int kq = 0;   // K-ring position of the current item's Q (Q staged in the K ring)
    int it = -1;
    bool ok = take_item(0, it);
    WorkItem w;
    RowBounds rb;
    if (ok && it >= 0) {
      w = prm.items[it];
      rb = bounds_of(w);
      ok = copy_q(0, 0);
    }
    for (int n = 0; ok && it >= 0; ++n) {
      const int nt = item_tiles<C::N>(w);
      // this item's kv head: its key scale joins the score scale, its value
      // scale the output
      const int kv_head = w.head * prm.pack / prm.group;
      // (at least FLT_MIN: a hidden score is -inf, and -inf * 0 would be NaN;
      // with sm_scale = 0 every weight is still exactly 2^0 = 1)
      const float scale =
          fmaxf(scale0 * (prm.k_head_scale ? prm.k_head_scale[kv_head] : 1.f), FLT_MIN);
      const float v_scale = prm.v_scale * (prm.v_head_scale ? prm.v_head_scale[kv_head] : 1.f);
      int it_next = -1;
      if (!take_item(n + 1, it_next)) {
        ok = false;
        break;
      }
      const bool has_next = it_next >= 0;
      // l: sum of the exact weights (gives lse); lp: sum of the rounded
      // weights the PV MMA multiplies (normalises O)
      float m = -INFINITY, l = 0.f, lp = 0.f;
      for (int j = 0; j < nt; ++j, ++g) {
        const int st = g & 1;                 // S buffer
        const int kvst = g % C::NST;          // K/V ring stage
        if (!mbar_wait_warp(smem_u32(&bars.s_full[st]), (g >> 1) & 1, limit, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[C::N / 32][32];
#pragma unroll
        for (int c = 0; c < C::N / 32; ++c)
          tmem_ld32(tmem + lane_off + C::COL_S + st * C::N + c * 32, sr[c]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (!C::P_IN_S && lane == 0) mbar_arrive(smem_u32(&bars.s_free[st]));

        // Row max of the raw scores (sm_scale >= 0 commutes with max). Eight
        // independent accumulators keep the dependency chains short; the mask
        // is applied only in tiles that cross this warp's bounds.
        const int col0 = w.tok_begin + j * C::N;   // key position of column 0
        // the columns of this tile the row may see: lo .. hi (a window's lower
        // bound, INT_MIN when there is none, gives lo = 0)
        const int hi = rb.t_max - col0;
        const int lo = rb.t_min > col0 ? rb.t_min - col0 : 0;
        const bool need_mask = __any_sync(0xffffffffu, hi < C::N - 1 || lo > 0);
        auto body = [&](auto masked) -> bool {
        constexpr bool MK = decltype(masked)::value;
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
        for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
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
        for (int i = 0; i < 4; ++i) rs4[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < C::N; k += 2)
          rs4[(k >> 1) & 3] = __fadd2_rn(rs4[(k >> 1) & 3], make_float2(s[k], s[k + 1]));
        const float2 rs2 = __fadd2_rn(__fadd2_rn(rs4[0], rs4[1]), __fadd2_rn(rs4[2], rs4[3]));
        const float rs_tile = rs2.x + rs2.y;
        l += rs_tile;

        // P buffer and O are free once the previous PV of this item has
        // completed (the last PV of the previous item completed before its
        // epilogue read O)
        if (j >= 1) {
          if (!mbar_wait_warp(smem_u32(&bars.pv_done), (g - 1) & 1, limit, &abort_flag))
            return false;
          tc_fence_after();
          if (__any_sync(0xffffffffu, o_live)) {
#pragma unroll 1
            for (int c = 0; c < HEAD_DIM / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(tmem + lane_off + C::COL_O + c * 32, r);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                const float2 y = __fmul2_rn(
                    make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                    make_float2(alpha, alpha));
                r[e] = __float_as_uint(y.x);
                r[e + 1] = __float_as_uint(y.y);
              }
              tmem_st32(tmem + lane_off + C::COL_O + c * 32, r);
            }
            tmem_wait_st();
          }
        }
        // Last tile: V rows past the valid keys may hold unused page slots or
        // stale data; zero them so that P = 0 there cannot meet a NaN.
        const int valid = w.tok_end - col0;
        if (MK && valid < C::N) {
          if (!mbar_wait_warp(smem_u32(&bars.v_full[kvst]), (g / C::NST) & 1, limit,
                              &abort_flag))
            return false;
          if (t >= valid && t < C::N) {
#pragma unroll
            for (int c = 0; c < C::DBLK; ++c)
#pragma unroll
              for (int c8 = 0; c8 < 8; ++c8)
                st_shared_v4(base + C::OFF_V + kvst * C::KV_BYTES + c * C::N * 128 + t * 128 +
                                 c8 * 16, 0u, 0u, 0u, 0u);
          }
        }
        // P row t as packed 16-bit pairs into TMEM (the A operand of the PV
        // MMA). lp adds the same rounded values the tensor core multiplies, so
        // that the final division normalises exactly the weights applied.
        // In tiles on the causal diagonal a row may have only a few visible
        // keys, so lp adds exactly the rounded values there; elsewhere the
        // rounding errors of many weights average out and the exact sum is used.
        float2 rsp2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int kb = 0; kb < C::N / 64; ++kb) {
          uint32_t wv[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) wv[e] = E::pack2(s[kb * 64 + 2 * e], s[kb * 64 + 2 * e + 1]);
          if (MK) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              rsp2[e & 1] = __fadd2_rn(rsp2[e & 1], make_float2(E::lo(wv[e]), E::hi(wv[e])));
          }
          tmem_st32(tmem + lane_off + (C::P_IN_S ? C::COL_S + st * C::N : C::COL_P) + kb * 32,
                    wv);
        }
        tmem_wait_st();
        lp += MK ? (rsp2[0].x + rsp2[0].y) + (rsp2[1].x + rsp2[1].y) : rs_tile;
        return true;
        };
        if (!(need_mask ? body(std::true_type{}) : body(std::false_type{}))) {
          ok = false;
          break;
        }
        fence_proxy_async_smem();   // zeroed V rows (generic writes) before the MMA reads them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars.p_full));
      }
      if (!ok) break;
      // Every QK MMA of this item has completed (the last S was read), so the
      // TMEM Q region may take the next item's Q now: the MMA issuer then
      // computes the next item's first scores while this item's last PV
      // and epilogue finish. (Copying it inside the tile loop instead, right
      // after the last S read, made the loop measurably slower.)
      kq += 2 + nt;
      if (has_next && !copy_q(n + 1, kq)) {
        ok = false;
        break;
      }
      // the next item's bounds load while this item's last PV completes
      WorkItem wn;
      RowBounds rn;
      if (has_next) {
        wn = prm.items[it_next];
        rn = bounds_of(wn);
      }
      if (!mbar_wait_warp(smem_u32(&bars.o_final), n & 1, limit, &abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // ---- epilogue: O / lp (bf16 or fp16) and lse = ln(l) + m ln 2
      const bool row_ok = w.q_row + t_row < rb.q_end;
      const float inv = lp > 0.f ? v_scale / lp : 0.f;
      const size_t out_row = size_t(w.q_row) + t_row;
      const int qo_head = w.head * prm.pack + t_head;
      // state slot of the row: shared-prefix items item.slot + row of q; a
      // piece of a split tile item.slot + row within the tile * item.merge
      // (mixed plans are never split)
      const bool piece = !C::MIXED && w.merge > 0;
      const size_t srow = piece ? size_t(w.slot) + size_t(t_row) * size_t(w.merge)
                                : size_t(w.slot) + out_row;
      uint16_t* op = reinterpret_cast<uint16_t*>(prm.out) +
                     (out_row * prm.num_qo_heads + qo_head) * HEAD_DIM;
      // O is read 64 columns (two loads) per wait, to halve the round trips
      constexpr int BATCH = HEAD_DIM >= 64 ? 2 : 1;
#pragma unroll 1
      for (int c0 = 0; c0 < HEAD_DIM / 32; c0 += BATCH) {
        uint32_t rb2[BATCH][32];
        if (nt > 0) {
#pragma unroll
          for (int b = 0; b < BATCH; ++b)
            tmem_ld32(tmem + lane_off + C::COL_O + (c0 + b) * 32, rb2[b]);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int b = 0; b < BATCH; ++b)
#pragma unroll
            for (int e = 0; e < 32; ++e) rb2[b][e] = 0u;
        }
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
          const int c = c0 + b;
          const uint32_t (&r)[32] = rb2[b];
          if (row_ok && (prm.state_o || piece)) {
            // fp32 state for a later log-sum-exp merge (shared-prefix decode,
            // or a piece of a split tile)
            float4* dst = reinterpret_cast<float4*>(
                (piece ? prm.piece_o : prm.state_o) + (srow * prm.num_qo_heads + qo_head) *
                HEAD_DIM + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float* f = reinterpret_cast<const float*>(r) + q4 * 4;
              dst[q4] = make_float4(f[0] * inv, f[1] * inv, f[2] * inv, f[3] * inv);
            }
          } else if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(op + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const float* f = reinterpret_cast<const float*>(r) + q4 * 8;
              dst[q4] = make_uint4(E::pack2(f[0] * inv, f[1] * inv),
                                   E::pack2(f[2] * inv, f[3] * inv),
                                   E::pack2(f[4] * inv, f[5] * inv),
                                   E::pack2(f[6] * inv, f[7] * inv));
            }
          }
        }
      }
      float* lse_dst = piece ? prm.piece_lse : (prm.state_o ? prm.state_lse : prm.lse);
      const size_t lrow = (piece || prm.state_o) ? srow : out_row;
      if (row_ok && lse_dst)
        lse_dst[lrow * prm.num_qo_heads + qo_head] = l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
      // O has been read: the next item's first PV (issued only after this
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
    if constexpr (C::MIXED) {
      // No prefill item is left for this CTA: every MMA of its last item has
      // completed (its epilogue waited for them) and no copy into the K and V
      // rings is pending, so the decode side may take those rings over.
      if (!named_bar_or(3, 128, !ok) && threadIdx.x == 0) {
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&prefill_free) = 1;
      }
    }
  } else if (warp < 8) {
    if constexpr (C::MIXED) setmaxnreg_dec<C::HELPER_REGS>();
    if (warp == 4 || warp == 6) {
      // ------------------------------------------------------------ producers
      // Warp 4 loads Q and the K tiles, warp 6 the V tiles: each page needs one
      // TMA instruction per 64-dim slice, and their issue, not the bytes,
      // bounded a single producer warp. Copies run ahead across item
      // boundaries: the next item's Q and first tiles load while the current
      // item is still computing.
      const bool is_v = warp == 6;
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
      // K producer, lane 0: publish item n's index in the ring (-1: no more)
      auto publish = [&](int n, int value) {
        if (n >= kItemRing &&
            !mbar_wait_bounded(smem_u32(&bars.item_empty[n % kItemRing]),
                               ((n / kItemRing) & 1) ^ 1, limit, &abort_flag))
          return false;
        item_ring[n % kItemRing] = value;
        mbar_arrive(smem_u32(&bars.item_full[n % kItemRing]));   // release: the index is visible
        return true;
      };
      // index of item 0 (both producers); a mixed launch may have more CTAs
      // than prefill items
      int it = int(blockIdx.x) < n_items ? int(blockIdx.x) : -1;
      if (is_v) {
        int v = -1;
        if (lane == 0) {
          ok = item_at(0, v);
          item_done(0);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        it = __shfl_sync(0xffffffffu, v, 0);
      } else if (lane == 0) {
        ok = publish(0, it);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      WorkItem w;
      if (ok && it >= 0) w = prm.items[it];
      // page ids of the next tile are loaded while the current tile's copies
      // are issued, so the dependent global load is off the critical path
      int next_page = -1;
      if (ok && it >= 0 && item_tiles<C::N>(w) > 0 && lane < pages_in(w, 0))
        next_page = prm.page_indices[w.page_begin + lane];
      for (int n = 0; ok && it >= 0; ++n) {
        const int nt = item_tiles<C::N>(w);
        const int kv_head = w.head * prm.pack / prm.group;
        const int c1 = prm.layout == FI_LAYOUT_NHD ? kv_head : 0;
        const int c2 = prm.layout == FI_LAYOUT_NHD ? 0 : kv_head;
        // the next item: taken from the counter and published by the K
        // producer, read from the ring by the V producer
        int it_next = -1;
        if (lane == 0) {
          if (is_v) {
            ok = item_at(n + 1, it_next);
            item_done(n + 1);
          } else {
            it_next = int(gridDim.x + atomicAdd(prm.work_counter, 1u));
            if (it_next >= n_items) it_next = -1;
            ok = publish(n + 1, it_next);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        it_next = __shfl_sync(0xffffffffu, it_next, 0);
        if (!ok) break;
        WorkItem wn;
        if (it_next >= 0) wn = prm.items[it_next];
        if (!is_v && !C::Q_IN_RING) {
          // Q of item n, once the buffer is free: its previous contents have
          // been copied into TMEM
          if (n >= 1) {
            ok = mbar_wait_warp(smem_u32(&bars.q_tmem), (n - 1) & 1, limit, &abort_flag);
            if (!ok) break;
          }
          if (lane == 0) {
            const uint32_t qb = smem_u32(&bars.q_full);
            mbar_arrive_expect_tx(qb, C::Q_BYTES);
  #pragma unroll
            for (int c = 0; c < C::DBLK; ++c)
              // 128 M rows = (128 / pack rows of q) x (pack heads), heads inner
              tma_load_3d(base + C::OFF_Q + c * C::M * 128, &q_map, qb, c * 64, w.head * prm.pack,
                          w.q_row);
          }
          q_loads = n + 1;
        } else if (!is_v) {
          // Q of item n into the next two K-ring slots (64-dim slices 2h and
          // 2h + 1 in slot h), released by the MMA issuer once the softmax
          // warps have copied Q into TMEM
          for (int h = 0; h < 2; ++h, ++g) {
            const int st = g % C::NST;
            if (g >= C::NST && !mbar_wait_warp(smem_u32(&empty[st]), ((g / C::NST) & 1) ^ 1,
                                               limit, &abort_flag)) {
              ok = false;
              break;
            }
            if (lane == 0) {
              const uint32_t fb = smem_u32(&full[st]);
              mbar_arrive_expect_tx(fb, C::KV_BYTES);
  #pragma unroll
              for (int c = 0; c < 2; ++c)
                tma_load_3d(ring + st * C::KV_BYTES + c * C::M * 128, &q_map, fb, (2 * h + c) * 64,
                            w.head * prm.pack, w.q_row);
            }
            issued = g + 1;
          }
          if (!ok) break;
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
          const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
          const uint32_t bytes = uint32_t(__popc(vmask)) * C::DBLK * box;
          if (g >= C::NST && !mbar_wait_warp(smem_u32(&empty[st]), ((g / C::NST) & 1) ^ 1,
                                             limit, &abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[st]);
          const bool skip = !is_v && n == 0 && j == 0 && prm.fault_kind == 1 && blockIdx.x == 0;
          if (skip) skip_pos = g;
          if (lane == 0 && !skip) mbar_arrive_expect_tx(fb, bytes);
          __syncwarp();
          // one copy per lane: box lane % DBLK of the tile's page lane / DBLK
          // (at most 32); one lane issuing its page's boxes in turn paced
          // the ring
          const int pi = min(lane / C::DBLK, 31);
          const int opage = __shfl_sync(0xffffffffu, page, pi);
          if (((vmask >> pi) & 1u) && lane < np * C::DBLK && !skip) {
            const int c = lane % C::DBLK;
            tma_load_4d(ring + st * C::KV_BYTES + pi * box + c * C::N * 128, map, fb, c * 64, c1,
                        c2, opage);
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
    } else if (warp == 5) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        // descriptors are linear in the address field (bits 0-13 = addr >> 4),
        // so each MMA's descriptor is a base plus a compile-time offset
        const uint64_t kd0 = sdesc_sw128(base + C::OFF_K, 16, 1024);
        const uint64_t vd0 = sdesc_sw128(base + C::OFF_V, C::N * 128, 1024);
        bool ok = true;
        int g = 0;    // KV tiles of earlier items (V ring, S buffers)
        int kq = 0;   // K-ring position of the item's first K tile (Q slots included)
        for (int n = 0; ok; ++n) {
          int it = -1;
          ok = item_at(n, it);
          item_done(n);
          if (!ok || it < 0) break;
          const int nt = item_tiles<C::N>(prm.items[it]);
          ok = mbar_wait_bounded(smem_u32(&bars.q_tmem), n & 1, limit, &abort_flag);
          if (ok && C::Q_IN_RING) {
            // Q is in TMEM: its two K-ring slots are free for K tiles again
            mbar_arrive(smem_u32(&bars.k_empty[kq % C::NST]));
            mbar_arrive(smem_u32(&bars.k_empty[(kq + 1) % C::NST]));
            kq += 2;
          }
          for (int j = 0; ok && j <= nt; ++j) {
            if (j < nt) {
              const int gq = g + j, sb = gq & 1;
              const int kp = kq + j, st = kp % C::NST;   // K-ring position of this tile
              ok = mbar_wait_bounded(smem_u32(&bars.k_full[st]), (kp / C::NST) & 1, limit,
                                     &abort_flag);
              if (ok && gq >= 2)
                ok = mbar_wait_bounded(smem_u32(&bars.s_free[sb]), ((gq >> 1) & 1) ^ 1, limit,
                                       &abort_flag);
              if (!ok) break;
              tc_fence_after();
              const uint64_t kd = kd0 + uint64_t((st * C::KV_BYTES) >> 4);
              const uint32_t s_col = tmem + C::COL_S + sb * C::N;
  #pragma unroll
              for (int k = 0; k < HEAD_DIM / 16; ++k) {
                const uint64_t bd = kd + uint64_t(((k >> 2) * C::N * 128 + (k & 3) * 32) >> 4);
                tc_mma_ts(s_col, tmem + C::COL_Q + k * 8, bd, C::IDESC_QK, k > 0 ? 1u : 0u);
              }
              tc_commit(smem_u32(&bars.s_full[sb]));
              tc_commit(smem_u32(&bars.k_empty[st]));
            }
            if (j >= 1) {
              const int gp = g + j - 1, st = gp % C::NST;
              ok = mbar_wait_bounded(smem_u32(&bars.p_full), gp & 1, limit, &abort_flag);
              if (ok)
                ok = mbar_wait_bounded(smem_u32(&bars.v_full[st]), (gp / C::NST) & 1, limit,
                                       &abort_flag);
              if (!ok) break;
              tc_fence_after();
              const uint64_t vd = vd0 + uint64_t((st * C::KV_BYTES) >> 4);
  #pragma unroll
              for (int k = 0; k < C::N / 16; ++k) {
                // MN-major V: 16 tokens per step; the next 64 dims one K-tile slice further
                const uint64_t bd = vd + uint64_t((k * 16 * 128) >> 4);
                const uint32_t p_col = C::P_IN_S ? C::COL_S + (gp & 1) * C::N : C::COL_P;
                tc_mma_ts(tmem + C::COL_O, tmem + p_col + k * 8, bd, C::IDESC_PV,
                          (j > 1 || k > 0) ? 1u : 0u);
              }
              tc_commit(smem_u32(&bars.v_empty[st]));
              tc_commit(smem_u32(&bars.pv_done));
              if (C::P_IN_S) tc_commit(smem_u32(&bars.s_free[gp & 1]));
            }
          }
          if (!ok) break;
          tc_commit(smem_u32(&bars.o_final));
          g += nt;
          kq += nt;
        }
        if (!ok) {
          abort_flag = 1;
          atomicOr(prm.err, kErrTimeout);
          // every MMA issued so far completes before the TMEM is released
          tc_commit(smem_u32(&bars.drain));
          mbar_wait_bounded(smem_u32(&bars.drain), 0, limit, nullptr);
        }
      }
      __syncwarp();
    } else {
      if constexpr (C::MIXED) {
        // ------------------------------------------------------------ decode producer (mixed kernel)
        // Takes decode items from a global counter in the planner's
        // longest-first order, hands their indices to the decode consumers
        // through a small ring, and streams their pages into the decode ring.
        // Once the CTA's prefill side has no more work, the decode ring grows
        // into the prefill K and V rings: between two items the producer
        // waits until the consumers have released every stage of the short
        // ring, then sends them a switch marker (-2), and both sides go on
        // from position 0 of the long ring (barriers of its own).
        const DecRing ring_a = contiguous_ring(base + C::OFF_DEC, DC::NSTAGE, bars.d_full,
                                               bars.d_empty);
        const DecRing ring_b{base + C::OFF_DEC, base + C::OFF_K, DC::NSTAGE, C::DEC_STAGES_EXT,
                             bars.e_full, bars.e_empty};
        bool ok = true;
        int r = 0;   // position in the current ring
        for (int dn = 0; ok; ++dn) {
          int grow = 0;
          if (lane == 0)
            grow = !dec_extended && *reinterpret_cast<volatile int*>(&prefill_free) != 0;
          grow = __shfl_sync(0xffffffffu, grow, 0);
          if (grow) {
            // every stage of the short ring released by the consumers
            for (int q = max(0, r - DC::NSTAGE); ok && q < r; ++q)
              ok = mbar_wait_warp(smem_u32(&bars.d_empty[q % DC::NSTAGE]), (q / DC::NSTAGE) & 1,
                                  limit, &abort_flag);
            if (!ok) break;
          }
          int idx = -1;
          if (lane == 0) {
            if (grow) idx = -2;
            else idx = abort_flag ? -1 : int(atomicAdd(dec_counter, 1u));
            if (idx >= n_dec) idx = -1;
            if (dn >= kItemRing &&
                !mbar_wait_bounded(smem_u32(&bars.ditem_empty[dn % kItemRing]),
                                   ((dn / kItemRing) & 1) ^ 1, limit, &abort_flag)) {
              ok = false;
            } else {
              ditem_ring[dn % kItemRing] = idx;
              mbar_arrive(smem_u32(&bars.ditem_full[dn % kItemRing]));
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
          idx = __shfl_sync(0xffffffffu, idx, 0);
          if (!ok) break;
          if (idx == -2) {
            dec_extended = true;
            r = 0;
            issued = 0;
            continue;
          }
          if (idx < 0) break;
          const WorkItem item = dprm.items[idx];
          const int lead = item.tok_begin % dprm.page_size;
          const int n_tok = item.tok_end - item.tok_begin + lead;
          const int n_tiles = (n_tok + DC::TILE - 1) / DC::TILE;
          const int done = decode_produce<HEAD_DIM, DG, E, 0>(
              dprm, item, n_tok, n_tiles, r, false, dec_extended ? ring_b : ring_a, &abort_flag,
              &k_map, &v_map);
          issued = r + done;
          if (done < n_tiles) ok = false;
          r += n_tiles;
        }
        if (!ok && lane == 0) {
          abort_flag = 1;
          atomicOr(dprm.err, kErrTimeout);
        }
        __syncwarp();
      }
    }
  } else {
    if constexpr (C::MIXED) {
      setmaxnreg_inc<C::DECODE_REGS>();
      // ------------------------------------------------------------ decode consumers (mixed kernel)
      // Batch decode on the same SM: the decode producer (warp 7) takes
      // decode items from a global counter in the planner's longest-first
      // order and streams their pages through the decode ring; the decode
      // consumers (warps 8-11) work through them in order. The HBM-bound
      // decode work thus runs beside the tensor-bound prefill tiles of the
      // same CTA instead of after them. An item's reduction area is the ring
      // stage of its last tile, released once the item is written.
      const DecRing ring_a = contiguous_ring(base + C::OFF_DEC, DC::NSTAGE, bars.d_full,
                                             bars.d_empty);
      const DecRing ring_b{base + C::OFF_DEC, base + C::OFF_K, DC::NSTAGE, C::DEC_STAGES_EXT,
                           bars.e_full, bars.e_empty};
      bool extended = false;                      // on the long ring (switch marker seen)
      const int cw = warp - 8;                    // consumer warp 0..DEC_WARPS-1
      const int ctid = int(threadIdx.x) - 256;    // consumer thread
      int r = 0;
      for (int dn = 0;; ++dn) {
        int idx = -1;
        bool good = true;
        if (lane == 0) {
          good = mbar_wait_bounded(smem_u32(&bars.ditem_full[dn % kItemRing]),
                                   (dn / kItemRing) & 1, limit, &abort_flag);
          if (good) idx = *reinterpret_cast<volatile int*>(&ditem_ring[dn % kItemRing]);
          mbar_arrive(smem_u32(&bars.ditem_empty[dn % kItemRing]));
        }
        good = __shfl_sync(0xffffffffu, good, 0) != 0;
        idx = __shfl_sync(0xffffffffu, idx, 0);
        // the consumer warps leave together (a warp that left alone would
        // never reach their named barriers); all read the same index
        if (named_bar_or(2, C::DEC_WARPS * 32, !good || idx == -1)) break;
        if (idx == -2) {                          // the ring grows: position 0 of the long one
          extended = true;
          r = 0;
          continue;
        }
        const DecRing& ring = extended ? ring_b : ring_a;
        const WorkItem item = dprm.items[idx];
        const int lead = item.tok_begin % dprm.page_size;
        const int n_tok = item.tok_end - item.tok_begin + lead;
        const int n_tiles = (n_tok + DC::TILE - 1) / DC::TILE;
        const bool hold = n_tiles > 0;
        const int last_stage = ring_stage<0>(ring, r + n_tiles - 1);
        const uint32_t red_addr = ring_addr(ring, last_stage, DC::STAGE_BYTES);
        float* red_o = hold ? reinterpret_cast<float*>(smem_raw + (red_addr - smem_u32(smem_raw)))
                            : nullptr;
        float* red_m = red_o + C::DEC_WARPS * DG * HEAD_DIM;
        float* red_l = red_m + C::DEC_WARPS * DG;
        float* red_lp = red_l + C::DEC_WARPS * DG;
        bool aborted;
        if (hold)
          aborted = DC::MMA
                        ? mma_consumer<HEAD_DIM, DG, E, E, 0, C::DEC_PAIRS>(
                              dprm, item, n_tok, lead, n_tiles, r, true, cw, ring, &abort_flag,
                              red_o, red_m, red_l, red_lp)
                        : simt_consumer<HEAD_DIM, DG, E, E, 0>(dprm, item, n_tok, lead, n_tiles,
                                                               r, true, cw, ring, &abort_flag,
                                                               red_o, red_m, red_l, red_lp);
        else
          aborted = named_bar_or(1, C::DEC_WARPS * 32, abort_flag != 0);
        if (aborted) break;                      // voted: all consumer warps agree
        decode_finish<HEAD_DIM, DG, E, E, C::DEC_WARPS>(dprm, item, ctid, hold, red_o, red_m,
                                                        red_l, red_lp, &dec_merge_last);
        if (hold) {
          // every consumer warp is done with the reduction area; the set that
          // consumed the last tile releases its stage
          named_bar_sync(1, C::DEC_WARPS * 32);
          if (lane == 0 && cw / DC::NCW == (r + n_tiles - 1) % C::DEC_PAIRS)
            mbar_arrive(smem_u32(&ring.empty[last_stage]));
        }
        r += n_tiles;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // Each producer lets every copy it issued land before the CTA exits, also
  // after a timeout anywhere in the CTA (in a normal run the consumers have
  // already seen these phases complete, so the waits return at once).
  if ((warp == 4 || warp == 6) && lane == 0) {
    const bool is_v = warp == 6;
    uint64_t* full = is_v ? bars.v_full : bars.k_full;
    for (int j = max(0, issued - C::NST); j < issued; ++j) {
      if (!is_v && j == skip_pos) continue;  // never issued
      mbar_wait_bounded(smem_u32(&full[j % C::NST]), (j / C::NST) & 1, limit, nullptr);
    }
    if (!is_v && q_loads > 0)
      mbar_wait_bounded(smem_u32(&bars.q_full), (q_loads - 1) & 1, limit, nullptr);
  }
  if constexpr (C::MIXED) {
    // the decode producer's copies, on the ring it ended on
    if (warp == 7 && lane == 0) {
      const int n = dec_extended ? C::DEC_STAGES_EXT : DC::NSTAGE;
      uint64_t* full = dec_extended ? bars.e_full : bars.d_full;
      for (int j = max(0, issued - n); j < issued; ++j)
        mbar_wait_bounded(smem_u32(&full[j % n]), (j / n) & 1, limit, nullptr);
    }
  }
}

template <int HEAD_DIM, class E>
__global__ void __launch_bounds__(PrefillCfg<HEAD_DIM, E>::THREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
               const __grid_constant__ CUtensorMap v_map, PrefillParams prm) {
  DecodeParams none{};
  prefill_body<HEAD_DIM, E, 0>(q_map, k_map, v_map, prm, none, 0, nullptr);
}

// One persistent launch over a mixed batch: the prefill items as in
// prefill_kernel, and on warps 7-11 of the same CTAs the decode items
// (dprm.items[0 .. n_dec), groups of DG query heads per kv head), handed out
// longest first from *dec_counter (zero before the launch).
template <int HEAD_DIM, class E, int DG>
__global__ void __launch_bounds__(PrefillCfg<HEAD_DIM, E, DG>::THREADS, 1)
mixed_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
             const __grid_constant__ CUtensorMap v_map, PrefillParams prm, DecodeParams dprm,
             int n_dec, uint32_t* dec_counter) {
  prefill_body<HEAD_DIM, E, DG>(q_map, k_map, v_map, prm, dprm, n_dec, dec_counter);
}

template <int HEAD_DIM, class E>
cudaError_t launch_prefill_t(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                             const PrefillParams& p, int grid, cudaStream_t stream) {
  using C = PrefillCfg<HEAD_DIM, E>;
  auto kern = prefill_kernel<HEAD_DIM, E>;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = once_per_device(configured, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::SMEM_BYTES);
  });
  if (e != cudaSuccess) return e;
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(qm, km, vm, p);
  return cudaGetLastError();
}

template <class E>
cudaError_t launch_prefill_e(int head_dim, const CUtensorMap& qm, const CUtensorMap& km,
                             const CUtensorMap& vm, const PrefillParams& p, int grid,
                             cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_prefill_t<64, E>(qm, km, vm, p, grid, stream);
    case 128: return launch_prefill_t<128, E>(qm, km, vm, p, grid, stream);
    case 256: return launch_prefill_t<256, E>(qm, km, vm, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <class E, int DG>
cudaError_t launch_mixed_t(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                           const PrefillParams& p, const DecodeParams& dp, int n_dec,
                           uint32_t* dec_counter, int grid, cudaStream_t stream) {
  using C = PrefillCfg<256, E, DG>;
  auto kern = mixed_kernel<256, E, DG>;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = once_per_device(configured, [&] {
    // the per-warpgroup register split assumes this launch allocation
    cudaFuncAttributes fa;
    cudaError_t r = cudaFuncGetAttributes(&fa, kern);
    if (r != cudaSuccess) return r;
    if (fa.numRegs < int(C::MIN_LAUNCH_REGS)) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::SMEM_BYTES);
  });
  if (e != cudaSuccess) return e;
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(qm, km, vm, p, dp, n_dec, dec_counter);
  return cudaGetLastError();
}

}  // namespace

bool mixed_applies(int head_dim, int group, int dtype, int kv_dtype) {
  return mixed_kernel_applies(head_dim, group, dtype, kv_dtype);
}

cudaError_t launch_mixed(int head_dim, int group, int dtype, const CUtensorMap& qm,
                         const CUtensorMap& km, const CUtensorMap& vm, const PrefillParams& p,
                         const DecodeParams& dp, int n_dec, uint32_t* dec_counter, int grid,
                         cudaStream_t stream) {
  if (head_dim != 256) return cudaErrorInvalidValue;
  const int want = p.n_items > n_dec ? p.n_items : n_dec;
  grid = grid < want ? grid : want;
  if (grid <= 0) return cudaSuccess;
#define FI_MIXED_CASE(E)                                                                      \
  switch (group) {                                                                            \
    case 1: return launch_mixed_t<E, 1>(qm, km, vm, p, dp, n_dec, dec_counter, grid, stream); \
    case 2: return launch_mixed_t<E, 2>(qm, km, vm, p, dp, n_dec, dec_counter, grid, stream); \
    case 4: return launch_mixed_t<E, 4>(qm, km, vm, p, dp, n_dec, dec_counter, grid, stream); \
    default: return cudaErrorInvalidValue;                                                    \
  }
  if (dtype == FI_DTYPE_BF16) FI_MIXED_CASE(Bf16)
  if (dtype == FI_DTYPE_FP16) FI_MIXED_CASE(Fp16)
#undef FI_MIXED_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill(int head_dim, int dtype, const CUtensorMap& qm, const CUtensorMap& km,
                           const CUtensorMap& vm, const PrefillParams& p, int grid,
                           cudaStream_t stream) {
  if (p.n_items <= 0 || grid <= 0) return cudaSuccess;
  if (prefill_pair_applies(head_dim, p))
    return launch_prefill_pair(head_dim, dtype, qm, km, vm, p, grid, stream);
  grid = grid < p.n_items ? grid : p.n_items;
  switch (dtype) {
    case FI_DTYPE_BF16: return launch_prefill_e<Bf16>(head_dim, qm, km, vm, p, grid, stream);
    case FI_DTYPE_FP16: return launch_prefill_e<Fp16>(head_dim, qm, km, vm, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fi
