// The batch-decode pipeline as per-item role functions, shared by the decode
// kernel (one work item per CTA, decode.cu) and the persistent mixed kernel
// (mixed.cu), whose decode warps work through many items on one ring.
//
// A decode work item is a (request, kv head, KV chunk); the g query heads of
// the kv head's group share every K/V page loaded (GQA sharing). Work is
// HBM-bound (about 1 flop per KV byte for g = 1), so the design is about
// moving bytes:
//   * a producer warp walks the page table and issues one TMA box per
//     (page, 64-dim slice) for K and for V, into a shared-memory ring
//     completed on mbarriers, with no register staging, as
//     "FlashAttention-3 kernel integration in inference engines", section 1
//     describes for TMA;
//   * 4 consumer warps read the staged rows (128-byte-swizzled, so reads are
//     bank-conflict free) and keep a running max / sum / accumulator (the
//     online softmax of section 1 of the FlashAttention-3 page), rescaling
//     when the max grows. With four or eight heads per kv head, or an FP8
//     cache, at head_dim <= 128 they compute with m16n8k16 MMAs that take the
//     tokens as rows and the heads as columns; otherwise with warp-shuffle
//     reductions ("FlashInfer Attention Kernel optimisation analysis",
//     sections 1.3 and 2.1: warp-level reductions via __shfl_sync, no global
//     sync);
//   * the warps' states are merged in shared memory; the item ends with
//     either the final row (bf16 or fp16, the inputs' type) + lse, or an fp32
//     partial state, and the CTA that completes a split request's last chunk
//     combines its partial states by log-sum-exp (no second launch).
// Scores are kept in the log2 domain (q pre-scaled by sm_scale*log2(e)).
//
// Ring positions: an item's tiles occupy consecutive positions r0, r0 + 1,
// ... of the ring (stage r % NSTAGE, phase (r / NSTAGE) & 1); a kernel that
// runs several items on one ring carries r0 on from item to item.
#pragma once

#include <type_traits>

#include "elem.cuh"
#include "fi_internal.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace fi {
namespace {

using namespace dev;

constexpr float kDecLog2e = 1.4426950408889634f;
constexpr float kDecLn2 = 0.6931471805599453f;

template <int HEAD_DIM, int GROUP, int KVB>   // KVB: bytes per cache element (2, or 1 for FP8)
struct DecodeCfg {
  // GQA groups of 4 or 8 heads at head_dim <= 128 use the tensor cores:
  // m16n8k16 MMAs with 16 tokens as the rows and the g heads as the 8 columns
  // (zero-padded); so do FP8 caches with 1 or 2 heads, where the MMAs replace
  // the SIMT consumer's shuffle-reduced dot products. At head_dim 256 a
  // 16-bit cache with 2 or more heads per kv head takes them too: a shuffle-
  // reduced dot product of 256 dims costs a warp far more instructions per
  // token than the 16 + 16 MMAs of a 16-token chunk (and 8 heads did not fit
  // the SIMT consumer's registers); so does an FP8 cache with 8 heads, whose
  // SIMT consumer spilled.
  static constexpr bool MMA = (HEAD_DIM <= 128 && (GROUP >= 4 || KVB == 1)) ||
                              (HEAD_DIM == 256 && KVB == 2 && GROUP >= 2) ||
                              (HEAD_DIM == 256 && KVB == 1 && GROUP >= 8);
  // tokens per stage: 32 KB of K+V, for 16-bit caches and the FP8 tensor-core
  // consumer (two 16-token chunks per consumer warp and stage); 16 KB for
  // the FP8 SIMT consumer, which runs three CTAs per SM
  static constexpr int TILE = (KVB == 1 && MMA ? 16384 : 8192) / HEAD_DIM;
  // tensor-core consumer: two 32 KB stages per CTA, three CTAs per SM;
  // 16-bit SIMT: three; FP8 SIMT: 16 KB stages, four deep
  static constexpr int NSTAGE = MMA ? 2 : (KVB == 2 ? 3 : 4);
  // consumer warps: a stage's tokens split into 16-token MMA chunks, two at
  // head_dim 256 (32 tokens per 32 KB stage)
  static constexpr int NCW = (MMA && HEAD_DIM == 256) ? 2 : 4;
  static constexpr int THREADS = 32 * (NCW + 1);       // + one producer warp
  static constexpr int LPT = HEAD_DIM / 8;             // lanes per token row (8 dims each)
  static constexpr int TPP = 32 / LPT;                 // token rows per warp pass
  static constexpr int TOK_PER_WARP = TILE / NCW;
  static constexpr int PASSES = TOK_PER_WARP / TPP;    // 8 for every head_dim
  static constexpr int SUB = GROUP >= 8 ? 2 : (GROUP >= 4 ? 4 : 8);  // passes per softmax step
  static constexpr int DBLK = HEAD_DIM / 64;           // 128-byte slices of a 16-bit row
  static constexpr int KBYTES = TILE * HEAD_DIM * KVB; // one K (or V) stage
  static constexpr int STAGE_BYTES = 2 * KBYTES;
  // FP8 rows of 128 bytes (head_dim 128) arrive 128-byte swizzled, and the
  // tensor-core consumer then loads its MMA fragments straight from them;
  // at head_dim 64 it widens 16 tokens of K and of V at a time into 16-bit
  // rows laid out as the TMA writes a 16-bit stage
  static constexpr bool SWZ8 = KVB == 1 && HEAD_DIM == 128;
  static constexpr int CONV_BYTES = (KVB == 1 && MMA && !SWZ8) ? NCW * 2 * 16 * HEAD_DIM * 2 : 0;
  static constexpr int SMEM_BYTES = NSTAGE * STAGE_BYTES + CONV_BYTES + 1024;  // + alignment
  // CTAs per SM: three for the tensor-core consumer (two 32 KB stages, at
  // most 136 registers) and for the FP8 SIMT consumer of 1 or 2 heads (65 KB),
  // for more warps to hide their latency; two otherwise, and for the FP8
  // tensor-core consumer at head_dim 256, whose 32 KB widening scratch
  // makes a CTA 97 KB
  static constexpr int MIN_BLOCKS =
      ((MMA && !(KVB == 1 && HEAD_DIM == 256)) || (KVB == 1 && GROUP <= 2)) ? 3 : 2;
  // The decode kernel is persistent (items from a counter, the ring running
  // on from item to item) for the SIMT consumer, whose ring has three or
  // more stages, when an item's cross-warp reduction fits in the stage of
  // its last tile (held by the consumers until the item is written). The
  // tensor-core consumer's ring has two stages: holding one for a reduction
  // leaves one to carry the next item, and one item per CTA, three CTAs per
  // SM overlapping their starts and ends, measured faster (70B GQA 0.295 vs
  // 0.299 ms, FP8 0.197 vs 0.204, shared prefix 0.210 vs 0.221; Llama-7B, on
  // the SIMT consumer, 0.371 vs 0.364 ms the other way round).
  static constexpr bool PERSISTENT =
      NSTAGE >= 3 && NCW * GROUP * HEAD_DIM * 4 + 3 * NCW * GROUP * 4 <= STAGE_BYTES;
  static_assert(PASSES % SUB == 0, "");
  static_assert(!MMA || TOK_PER_WARP % 16 == 0, "");
  static_assert(NCW * GROUP * HEAD_DIM * 4 + 3 * NCW * GROUP * 4 <= NSTAGE * STAGE_BYTES, "");
  static_assert(SMEM_BYTES <= 113 * 1024, "two CTAs per SM");
};

// Byte offset of 16-byte chunk `c8` (0..7) of row `r` inside a 128-byte-row
// slice written by TMA with 128-byte swizzling (slice base 1024-aligned).
__device__ __forceinline__ uint32_t swz(int r, int c8) {
  return uint32_t(r * 128 + ((c8 ^ (r & 7)) << 4));
}

// A ring of decode stages: `n` stages of `stage_bytes`, the first `n_lo` at
// shared address `lo`, the rest at `hi` (two separate blocks of shared
// memory, each 1024-aligned), completed on `full[s]` (the producer's bytes)
// and `empty[s]` (one arrival per consumer warp).
struct DecRing {
  uint32_t lo, hi;
  int n_lo, n;
  uint64_t* full;
  uint64_t* empty;
};

__device__ __forceinline__ DecRing contiguous_ring(uint32_t base, int n, uint64_t* full,
                                                   uint64_t* empty) {
  return DecRing{base, base, n, n, full, empty};
}

// Stage and phase of ring position r, and the stage's shared address. NS > 0
// is the stage count known at compile time (the decode kernel's ring); 0
// takes R.n.
template <int NS>
__device__ __forceinline__ int ring_stage(const DecRing& R, int r) {
  return NS > 0 ? r % NS : r % R.n;
}
template <int NS>
__device__ __forceinline__ uint32_t ring_phase(const DecRing& R, int r) {
  return uint32_t((NS > 0 ? r / NS : r / R.n) & 1);
}
__device__ __forceinline__ uint32_t ring_addr(const DecRing& R, int s, int stage_bytes) {
  return s < R.n_lo ? R.lo + uint32_t(s * stage_bytes) : R.hi + uint32_t((s - R.n_lo) * stage_bytes);
}

// Tensor-core consumer warp for GQA groups of 4 or 8 heads, token-major: per
// 16-token chunk of its share of a stage,
//   S^T (16 tokens x 8 heads) = K Q^T by m16n8k16 MMAs, K the A operand
//     (ldmatrix from the swizzled stage), Q^T the B operand held in
//     registers (groups of 4 pad heads 4-7 with zeros);
//   P^T = 2^(S^T - ref) per head column, rounded to the MMA type and moved
//     into B-fragment order by two register transposes (movmatrix);
//   O^T (head_dim x 8) += V^T P^T, V^T the A operand (ldmatrix.trans).
// The tokens fill the MMAs' 16 rows and the heads their 8 columns, so no
// MMA work is padding for groups of 8. A lane holds two head columns (2c,
// 2c + 1, c = lane % 4) of every fragment; each head's reference grows only
// when a score exceeds it by more than 2^8 (the rescale then needs the
// chunk's exact maximum, a reduction over the 8 lanes sharing the column).
// With an FP8 cache at head_dim 128 the K and V fragments come straight from
// the FP8 rows (see the comments at the loads); at head_dim 64 each 16-token
// chunk of K and V is widened (exactly) into the warp's 16-bit scratch,
// laid out as the TMA writes a 16-bit stage.
// Leaves the warp's (m, l, lp, O) in shared memory and returns whether any
// consumer aborted (voted, so all agree). Ring positions, `cw`, `hold_last`
// and the reduction arrays as for simt_consumer. With NPAIR = 2 there are
// two sets of NCW consumer warps (cw = set * NCW + warp in the set) that
// take turns on stages: set (r % 2) consumes ring position r, so a stage
// needs NCW arrivals, and twice as many warps work on the item.
template <int HEAD_DIM, int GROUP, class E, class KV, int NS, int NPAIR = 1>
__device__ __forceinline__ bool mma_consumer(const DecodeParams& prm, const WorkItem& item,
                                             int n_tok, int lead, int n_tiles, int r0,
                                             bool hold_last, int cw, const DecRing& R,
                                             int* abort_flag, float* red_o, float* red_m,
                                             float* red_l, float* red_lp) {
  constexpr bool FP8 = std::is_same<KV, E4m3>::value;
  using C = DecodeCfg<HEAD_DIM, GROUP, FP8 ? 1 : 2>;
  // With an FP8 cache the P V MMAs run in fp16: e4m3 widens to fp16 in one
  // instruction per pair, exactly, and P is rounded to fp16. K Q^T runs in
  // fp16 too at head_dim 64 (q converted once, exact within fp16's range)
  // and in e4m3 at head_dim 128 (below).
  using ME = std::conditional_t<FP8, Fp16, E>;
  constexpr int KS = HEAD_DIM / 16;       // k-steps of K Q^T
  constexpr int MB = HEAD_DIM / 16;       // 16-dim row blocks of O^T
  const int warp = cw % C::NCW, lane = threadIdx.x & 31;   // warp: its part of a stage
  const int set = cw / C::NCW;                               // its turn among the stages
  const int g = lane >> 2;                // fragment row group (token g / g + 8; B column g)
  const int c = lane & 3;                 // this lane's head columns 2c, 2c + 1
  // score scale in the log2 domain, with the kv head's key scale
  const float scale =
      prm.sm_scale * kDecLog2e * (prm.k_head_scale ? prm.k_head_scale[item.head] : 1.f);

  // Q^T as B fragments: column = head g, rows (k) 2c, 2c + 1 and 2c + 8, 2c + 9
  // of each k-step. With fp16 MMAs on FP8 K rows (fp16 q), k index 2c + j of
  // a k-step is dim 4c + j and 2c + 8 + j is dim 4c + 2 + j, so that a lane's
  // four consecutive bytes of a key row feed both halves of its A fragment;
  // Q's k order follows.
  uint32_t qb[C::SWZ8 && std::is_same<E, Bf16>::value ? 1 : KS][2];
  // With FP8 K rows of 128 bytes and bf16 q, K Q^T runs as e4m3 MMAs
  // (m16n8k32) on the cache bytes themselves: an ldmatrix of the rows gives a lane four
  // consecutive dims 4c..4c+3 (and 16 + 4c..) of token g (and g + 8), the A
  // fragment's layout, so K is never widened. Q enters as a sum of two e4m3
  // terms, each the e4m3 rounding of what the terms before it left: the
  // first after a power-of-two scale per head that puts the head's largest
  // |element| in [128, 256), the others (whose inputs are at most 8 there)
  // after a further 2^5, so that they do not fall into e4m3's subnormal
  // range. Each term accumulates on its own and the two sums are scaled
  // back when the scores are formed. The two terms hold a bf16 element (8
  // significant bits) exactly for every element above 2^-14 of the head's
  // largest; the error below that is under 2^-22 of the largest. B
  // fragment: dims 32 ks + 4c..4c+3 and 32 ks + 16 + 4c.. of head g, one
  // byte each. (fp16 q, 11 bits, would take three terms, which do not fit
  // the registers: it keeps the fp16 MMAs.)
  constexpr bool K8 = C::SWZ8 && std::is_same<E, Bf16>::value;
  constexpr int KS8 = HEAD_DIM / 32;
  constexpr int NQ = 2;
  uint32_t q8[K8 ? KS8 : 1][NQ][2];
  float qinv[2] = {1.f, 1.f};   // 2^-qe of heads 2c, 2c + 1 (this lane's score columns)
  if constexpr (K8) {
    const uint16_t* qh = reinterpret_cast<const uint16_t*>(prm.q) +
        (size_t(item.q_row) * prm.num_qo_heads + item.head * GROUP + (g < GROUP ? g : 0)) *
            HEAD_DIM;
    float qf[KS8][2][4];
    float amax = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS8; ++ks)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const uint2 u = g < GROUP
            ? *reinterpret_cast<const uint2*>(qh + ks * 32 + hf * 16 + 4 * c)
            : make_uint2(0u, 0u);
        qf[ks][hf][0] = E::lo(u.x);
        qf[ks][hf][1] = E::hi(u.x);
        qf[ks][hf][2] = E::lo(u.y);
        qf[ks][hf][3] = E::hi(u.y);
#pragma unroll
        for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fabsf(qf[ks][hf][j]));
      }
    // the head's largest |element| (its four lanes); a non-finite one gives NaN scores
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int ex = 0;
    if (amax > 0.f && amax <= 3.0e38f) frexpf(amax, &ex);   // amax in [2^(ex-1), 2^ex)
    ex = max(ex, -100);   // (a head of subnormal q: fewer bits, no overflow of the scale)
    const float qsc = ldexpf(1.f, 8 - ex);
    const float inv = amax <= 3.0e38f ? ldexpf(1.f, ex - 8) : __int_as_float(0x7fffffff);
    qinv[0] = __shfl_sync(0xffffffffu, inv, 8 * c);
    qinv[1] = __shfl_sync(0xffffffffu, inv, 8 * c + 4);
#pragma unroll
    for (int ks = 0; ks < KS8; ++ks)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = qf[ks][hf][j] * qsc;
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          const uint32_t lo = E4m3::from_f32x2(x[0], x[1]), hi = E4m3::from_f32x2(x[2], x[3]);
          q8[ks][t][hf] = lo | (hi << 16);
          if (t + 1 < NQ) {
            float r[4];
            E4m3::unpack4(q8[ks][t][hf], r);
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] = (x[j] - r[j]) * 32.f;
          }
        }
      }
  } else {
    const uint32_t* qp = reinterpret_cast<const uint32_t*>(
        reinterpret_cast<const uint16_t*>(prm.q) +
        (size_t(item.q_row) * prm.num_qo_heads + item.head * GROUP + (g < GROUP ? g : 0)) *
            HEAD_DIM);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int w0i = C::SWZ8 ? (ks * 16 + 4 * c) >> 1 : (ks * 16 + 2 * c) >> 1;
      const int w1i = C::SWZ8 ? w0i + 1 : (ks * 16 + 8 + 2 * c) >> 1;
      uint32_t w0 = g < GROUP ? qp[w0i] : 0u;
      uint32_t w1 = g < GROUP ? qp[w1i] : 0u;
      if constexpr (!std::is_same<ME, E>::value) {
        w0 = ME::pack2(E::lo(w0), E::hi(w0));
        w1 = ME::pack2(E::lo(w1), E::hi(w1));
      }
      qb[ks][0] = w0;
      qb[ks][1] = w1;
    }
  }
  // O^T accumulators: block mb, rows (dims) g and g + 8, columns (heads) 2c, 2c + 1
  float o[MB][4];
#pragma unroll
  for (int t = 0; t < MB; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  // per head column of this lane: reference, sum of weights, sum of rounded weights
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f}, lp[2] = {0.f, 0.f};

  for (int i = 0; i < n_tiles; ++i) {
    if (NPAIR > 1 && (r0 + i) % NPAIR != set) continue;   // the other set's stage
    const int s = ring_stage<NS>(R, r0 + i);
    if (!mbar_wait_warp(smem_u32(&R.full[s]), ring_phase<NS>(R, r0 + i), prm.wait_limit_ns,
                        abort_flag)) {
      if (lane == 0) { *abort_flag = 1; atomicOr(prm.err, kErrTimeout); }
      break;
    }
    const int ntok = min(C::TILE, n_tok - i * C::TILE);
    const int lo = i == 0 ? lead : 0;        // rows below lo are outside the window
    const uint32_t kstage = ring_addr(R, s, C::STAGE_BYTES);
    const uint32_t vstage = kstage + C::KBYTES;
#pragma unroll 1
    for (int cb = warp * C::TOK_PER_WARP; cb < (warp + 1) * C::TOK_PER_WARP; cb += 16) {
      if (cb >= ntok) break;
      // 16-bit K and V rows of this chunk: in the stage (row cb + t of slices
      // TILE rows long) or, for FP8, in the warp's scratch (row t of 16-row slices)
      uint32_t kbase = kstage, vbase = vstage, slice = C::TILE * 128;
      int row0 = cb;
      if constexpr (C::SWZ8) {
        if (cb + 16 > ntok) {
          // FP8 V rows past the last key: zero them (P = 0 must not meet a NaN)
          for (int idx = lane; idx < 16 * 8; idx += 32) {
            const int row = cb + idx / 8;
            if (row >= ntok) {
              const uint32_t a = vstage + row * 128 + (idx % 8) * 16;
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u)
                           : "memory");
            }
          }
          __syncwarp();
        }
      } else if constexpr (FP8) {
        // (the decode kernel's FP8 scratch follows its ring)
        kbase = R.lo + C::NSTAGE * C::STAGE_BYTES + warp * (2 * 16 * HEAD_DIM * 2);
        vbase = kbase + 16 * HEAD_DIM * 2;
        slice = 16 * 128;
        row0 = 0;
        // 16 tokens x HEAD_DIM bytes of each of K and V; one 16-byte FP8
        // chunk becomes two 16-byte chunks of the 16-bit layout. Rows past
        // the last key become zeros (P = 0 there must not meet a NaN).
        constexpr int CPR = HEAD_DIM / 16;   // 16-byte FP8 chunks per row
#pragma unroll 1
        for (int idx = lane; idx < 2 * 16 * CPR; idx += 32) {
          const int is_v = idx >= 16 * CPR;
          const int rem = idx - is_v * 16 * CPR;
          const int t = rem / CPR, c = rem % CPR;
          uint32_t w[8];
          if (cb + t < ntok) {
            const uint4 u = lds128((is_v ? vstage : kstage) + (cb + t) * HEAD_DIM + c * 16);
            const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              w[2 * e] = E4m3::to_f16x2(uw[e]);
              w[2 * e + 1] = E4m3::to_f16x2(uw[e] >> 16);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = 0u;
          }
          const uint32_t dst = (is_v ? vbase : kbase);
          const int c8 = 2 * c;                       // first 8-dim chunk of the 16 dims
          const uint32_t a0 = dst + (c8 >> 3) * slice + swz(t, c8 & 7);
          const uint32_t a1 = dst + ((c8 + 1) >> 3) * slice + swz(t, (c8 + 1) & 7);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "r"(w[0]), "r"(w[1]),
                       "r"(w[2]), "r"(w[3]) : "memory");
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a1), "r"(w[4]), "r"(w[5]),
                       "r"(w[6]), "r"(w[7]) : "memory");
        }
        __syncwarp();
      } else if (cb + 16 > ntok) {
        // V rows past the last key hold unused slots or stale data: zero them
        // so that P = 0 there cannot meet a NaN in the MMA
        for (int idx = lane; idx < 16 * (HEAD_DIM / 8); idx += 32) {
          const int row = cb + idx / (HEAD_DIM / 8), c = idx % (HEAD_DIM / 8);
          if (row >= ntok) {
            const uint32_t a = vbase + (c >> 3) * C::TILE * 128 + swz(row, c & 7);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
          }
        }
        __syncwarp();
      }
      // S^T accumulators by k-step parity (two dependent chains of KS / 2)
      float sacc2[2][4] = {};
      // ldmatrix lanes 0-7 / 8-15 / 16-23 / 24-31 address matrices 0..3
      const int ltok = (lane & 7) + ((lane >> 3) & 1) * 8;   // token row this lane addresses
      if constexpr (K8) {
        // K straight from the FP8 rows as the e4m3 A fragment: each 8x8
        // matrix of byte pairs is 8 tokens x 16 dims, so a lane's register is
        // dims 4c..4c+3 of one token. Matrices: (tokens 0-7 | 8-15) x (dims
        // 32 ks .. +15 | 32 ks + 16 .. +31). Term 0 of Q goes to
        // accumulator 0, term 1 (2^5 finer) to accumulator 1.
        const int tok = cb + ltok;
#pragma unroll
        for (int ks = 0; ks < KS8; ++ks) {
          const int ch = 2 * ks + (lane >> 4);
          uint32_t a[4];
          ldsm_x4(kstage + tok * 128 + ((ch ^ (tok & 7)) << 4), a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int t = 0; t < NQ; ++t) E4m3::mma16832(sacc2[t > 0], a, q8[ks][t][0], q8[ks][t][1]);
        }
      } else if constexpr (C::SWZ8) {
        // fp16 q: K widened from the FP8 rows. Each 8x8 matrix of byte pairs
        // is 8 tokens x 16 dims, and a lane's register is 4 consecutive dims
        // 4c..4c+3 of token g: widened, dims 4c, 4c+1 and 4c+2, 4c+3 are the A
        // fragment's (row g, k 2c..) and (row g, k 2c+8..) halves.
        // Matrices: (tokens 0-7 | 8-15) x (k-steps ks | ks+1).
        const int tok = cb + ltok;
#pragma unroll
        for (int ks = 0; ks < KS; ks += 2) {
          const int step = ks + (lane >> 4);
          uint32_t q0, q1, q2, q3;
          ldsm_x4(kstage + tok * 128 + ((step ^ (tok & 7)) << 4), q0, q1, q2, q3);
          const uint32_t a0[4] = {E4m3::to_f16x2(q0), E4m3::to_f16x2(q1),
                                  E4m3::to_f16x2(q0 >> 16), E4m3::to_f16x2(q1 >> 16)};
          const uint32_t a1[4] = {E4m3::to_f16x2(q2), E4m3::to_f16x2(q3),
                                  E4m3::to_f16x2(q2 >> 16), E4m3::to_f16x2(q3 >> 16)};
          ME::mma16816(sacc2[0], a0, qb[ks][0], qb[ks][1]);
          ME::mma16816(sacc2[1], a1, qb[ks + 1][0], qb[ks + 1][1]);
        }
      } else {
        // matrices: (tokens 0-7 | 8-15) x (dims 0-7 | 8-15 of the k-step)
        const int mi = lane >> 3;
        const int trow = row0 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int dim = ks * 16 + (mi >> 1) * 8;
          uint32_t a[4];
          ldsm_x4(kbase + (dim >> 6) * slice + swz(trow, (dim & 63) >> 3), a[0], a[1], a[2], a[3]);
          ME::mma16816(sacc2[ks & 1], a, qb[ks][0], qb[ks][1]);
        }
      }
      // scores of tokens g (e = 0, 1) and g + 8 (e = 2, 3), heads 2c + (e & 1)
      float sv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = cb + g + (e >> 1) * 8;
        const float acc = K8 ? fmaf(sacc2[1][e], 1.f / 32.f, sacc2[0][e])
                                  : sacc2[0][e] + sacc2[1][e];
        sv[e] = (tok < ntok && tok >= lo) ? acc * (scale * qinv[e & 1]) : -INFINITY;
      }
      float mx[2] = {fmaxf(sv[0], sv[2]), fmaxf(sv[1], sv[3])};
      // Lazy rescale: a head's reference changes only when one of its scores
      // exceeds it by more than 2^8 (exact: O and both sums share the stale
      // reference). Then the chunk's maximum over the 8 lanes of the column
      // becomes the reference, the same in every lane that holds the head.
      if (__any_sync(0xffffffffu, mx[0] > m[0] + 8.0f || mx[1] > m[1] + 8.0f)) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float v = mx[h];
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
          const float m_new = fmaxf(m[h], v);
          if (m_new > m[h] + 8.0f) {
            const float alpha = ex2(m[h] - m_new);
            l[h] *= alpha;
            lp[h] *= alpha;
#pragma unroll
            for (int t = 0; t < MB; ++t) {
              o[t][h] *= alpha;
              o[t][h + 2] *= alpha;
            }
            m[h] = m_new;
          }
        }
      }
      const float ref0 = (m[0] == -INFINITY) ? 0.f : m[0];
      const float ref1 = (m[1] == -INFINITY) ? 0.f : m[1];
      const float p0 = ex2(sv[0] - ref0), p1 = ex2(sv[1] - ref1);
      const float p2 = ex2(sv[2] - ref0), p3 = ex2(sv[3] - ref1);
      l[0] += p0 + p2;
      l[1] += p1 + p3;
      // P^T (tokens x heads) as the B fragment of the PV MMA: the C layout's
      // 8x8 blocks (tokens 0-7, 8-15) x heads, transposed in registers
      const uint32_t x0 = ME::pack2(p0, p1), x1 = ME::pack2(p2, p3);
      lp[0] += ME::lo(x0) + ME::lo(x1);
      lp[1] += ME::hi(x0) + ME::hi(x1);
      const uint32_t pb0 = movmatrix_trans(x0), pb1 = movmatrix_trans(x1);
      if constexpr (C::SWZ8) {
        // V straight from the FP8 rows: a transposed 8x8 matrix of byte pairs
        // gives a lane dims 2g, 2g+1 of tokens 2c, 2c+1; a byte permute splits
        // them into the even dim's and the odd dim's token pairs, which are
        // taken as rows g and g + 8 of the 16-dim block (O^T's rows permuted
        // accordingly, undone when O is written out). Matrices: (tokens 0-7 |
        // 8-15) x (16-dim blocks j | j+1).
        const int tok = cb + ltok;
#pragma unroll
        for (int j = 0; j < MB; j += 2) {
          const int grp = j + (lane >> 4);
          uint32_t v0, v1, v2, v3;
          ldsm_x4_trans(vstage + tok * 128 + ((grp ^ (tok & 7)) << 4), v0, v1, v2, v3);
          const uint32_t a0[4] = {E4m3::to_f16x2(__byte_perm(v0, 0, 0x0020)),
                                  E4m3::to_f16x2(__byte_perm(v0, 0, 0x0031)),
                                  E4m3::to_f16x2(__byte_perm(v1, 0, 0x0020)),
                                  E4m3::to_f16x2(__byte_perm(v1, 0, 0x0031))};
          const uint32_t a1[4] = {E4m3::to_f16x2(__byte_perm(v2, 0, 0x0020)),
                                  E4m3::to_f16x2(__byte_perm(v2, 0, 0x0031)),
                                  E4m3::to_f16x2(__byte_perm(v3, 0, 0x0020)),
                                  E4m3::to_f16x2(__byte_perm(v3, 0, 0x0031))};
          ME::mma16816(o[j], a0, pb0, pb1);
          ME::mma16816(o[j + 1], a1, pb0, pb1);
        }
      } else {
        // V^T blocks: matrices (tokens 0-7 | 8-15) x (dims 0-7 | 8-15 of the
        // block), transposed by ldmatrix into the A fragment's order
        const int mi = lane >> 3;
        const int trow = row0 + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
          const int dim = mb * 16 + (mi & 1) * 8;
          uint32_t a[4];
          ldsm_x4_trans(vbase + (dim >> 6) * slice + swz(trow, (dim & 63) >> 3), a[0], a[1], a[2],
                        a[3]);
          ME::mma16816(o[mb], a, pb0, pb1);
        }
      }
    }
    fence_proxy_async_smem();   // any zeroed rows before the producer's next TMA into the stage
    __syncwarp();
    if (lane == 0 && !(hold_last && i == n_tiles - 1)) mbar_arrive(smem_u32(&R.empty[s]));
  }
  // a head's sums are spread over the 8 lanes of its column
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], x);
      lp[h] += __shfl_xor_sync(0xffffffffu, lp[h], x);
    }
  }
  const bool aborted = named_bar_or(1, C::NCW * NPAIR * 32, *abort_flag != 0);
  if (!aborted) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int head = 2 * c + h;
      if (head < GROUP) {
        float* op = red_o + (cw * GROUP + head) * HEAD_DIM;
#pragma unroll
        for (int t = 0; t < MB; ++t) {
          // rows g and g + 8 of block t: dims 16t + g and + 8, or with FP8
          // fragments dims 16t + 2g and + 1
          const int d0 = C::SWZ8 ? 16 * t + 2 * g : 16 * t + g;
          const int d1 = C::SWZ8 ? d0 + 1 : d0 + 8;
          op[d0] = o[t][h];
          op[d1] = o[t][h + 2];
        }
        if (g == 0) {
          red_m[cw * GROUP + head] = m[h];
          red_l[cw * GROUP + head] = l[h];
          red_lp[cw * GROUP + head] = lp[h];
        }
      }
    }
  }
  return aborted;
}


// Producer warp: the TMA copies of one item's tiles into ring positions r0,
// r0 + 1, ... One box per (page, 64-dim slice) of a 16-bit cache, per page
// of an FP8 cache. The lanes read a tile's page ids (up to 32) at once, after
// the wait for its stage. On a ring sized at run time (NS = 0: the mixed
// kernel, where the decode copies share the SM with prefill work) the page
// ids are read 32 at a time instead (lane j holds page j of the batch), the
// next batch as soon as the current one is started, and each tile takes its
// 1-16 pages from the batch by a shuffle, so that a freed stage is refilled
// without a page-table round trip. (In the decode kernel, three CTAs per SM
// hide that round trip, and the batched form measured 1-2 % slower.)
// `skip_first` (test hook) leaves the first tile's copies out, so that the
// consumers' bounded waits run out. Returns the number of tiles whose copies
// were issued (n_tiles, unless a wait for a free stage ran out).
template <int HEAD_DIM, int GROUP, class KV, int NS>
__device__ __forceinline__ int decode_produce(const DecodeParams& prm, const WorkItem& item,
                                               int n_tok, int n_tiles, int r0, bool skip_first,
                                               const DecRing& R, int* abort_flag,
                                               const CUtensorMap* k_map, const CUtensorMap* v_map) {
  constexpr bool FP8 = std::is_same<KV, E4m3>::value;
  using C = DecodeCfg<HEAD_DIM, GROUP, FP8 ? 1 : 2>;
  const int lane = threadIdx.x & 31;
  const int pages_per_tile = C::TILE / prm.page_size;
  const uint32_t box_bytes = uint32_t(prm.page_size) * (FP8 ? HEAD_DIM : 128u);
  constexpr int BOXES = FP8 ? 1 : C::DBLK;
  // pages per tile: 1-16 (page size 16 or 32), a divisor of 32
  const int item_pages = (n_tok + prm.page_size - 1) / prm.page_size;
  const int tiles_per_batch = 32 / pages_per_tile;
  auto batch_ids = [&](int b) {   // this lane's page id of 32-page batch b (-1 past the item)
    const int p = b * 32 + lane;
    return p < item_pages ? prm.page_indices[item.page_begin + p] : -1;
  };
  constexpr bool BATCHED = NS == 0;
  int cur = BATCHED && n_tiles > 0 ? batch_ids(0) : -1;
  int nxt = BATCHED && item_pages > 32 ? batch_ids(1) : -1;
  for (int i = 0; i < n_tiles; ++i) {
    const int r = r0 + i;
    const int s = ring_stage<NS>(R, r);
    int page = -1;
    if constexpr (BATCHED) {
      const int k = i % tiles_per_batch;
      if (k == 0 && i > 0) {
        const int b = i / tiles_per_batch;
        cur = nxt;
        if ((b + 1) * 32 < item_pages) nxt = batch_ids(b + 1);
      }
      page = __shfl_sync(0xffffffffu, cur, k * pages_per_tile + lane % pages_per_tile);
    }
    if (r >= (NS > 0 ? NS : R.n)) {
      const uint32_t ph = ring_phase<NS>(R, r) ^ 1u;
      if (!mbar_wait_warp(smem_u32(&R.empty[s]), ph, prm.wait_limit_ns, abort_flag)) {
        if (lane == 0) { *abort_flag = 1; atomicOr(prm.err, kErrTimeout); }
        return i;
      }
    }
    const int np = (min(C::TILE, n_tok - i * C::TILE) + prm.page_size - 1) / prm.page_size;
    bool valid = false;
    if (lane < np) {
      if constexpr (!BATCHED) page = prm.page_indices[item.page_begin + i * pages_per_tile + lane];
      valid = page >= 0 && page < prm.num_pages;
      if (!valid) atomicOr(prm.err, kErrBounds);
    }
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
    const uint32_t bytes = uint32_t(__popc(vmask)) * 2u * BOXES * box_bytes;
    const uint32_t fb = smem_u32(&R.full[s]);
    const bool skip = skip_first && i == 0;
    if (lane == 0 && !skip) mbar_arrive_expect_tx(fb, bytes);
    __syncwarp();
    // One copy per lane: copy o = lane is box (o / 2) % BOXES of K (o even)
    // or V (o odd) of the tile's page o / (2 BOXES); a tile has at most 32
    // (pages x boxes x 2). A single lane issuing a tile's copies one after
    // another paced the ring (about 0.8 us per 32 KB tile with 8 copies).
    const int pi = min(lane / (2 * BOXES), 31);          // the copy's page in the tile
    const int opage = __shfl_sync(0xffffffffu, page, pi);
    const bool ovalid = (vmask >> pi) & 1u && lane < np * 2 * BOXES;
    if (ovalid && !skip) {
      const int c = (lane >> 1) % BOXES, is_v = lane & 1;
      const uint32_t dst = ring_addr(R, s, C::STAGE_BYTES) + uint32_t(is_v) * C::KBYTES +
                           uint32_t(pi) * box_bytes + uint32_t(c) * C::TILE * 128u;  // c = 0 for FP8
      const CUtensorMap* map = is_v ? v_map : k_map;
      if (prm.layout == FI_LAYOUT_NHD)
        tma_load_4d(dst, map, fb, c * 64, item.head, 0, opage);
      else
        tma_load_4d(dst, map, fb, c * 64, 0, item.head, opage);
    }
  }
  return n_tiles;
}

// SIMT consumer warp `cw` (0..NCW-1) for groups of 1 or 2 heads (any g at
// head_dim 256): d/8 lanes per token row, 16 bytes each; a shuffle
// reduction gives each score. The item's tiles are at ring positions r0,
// r0 + 1, ...; every stage is released after use, except the last one when
// `hold_last` (the caller reduces in it and releases it afterwards). Leaves
// the warp's (m, l, lp, O) in the reduction arrays and returns whether any
// consumer aborted (voted, so all agree).
template <int HEAD_DIM, int GROUP, class E, class KV, int NS>
__device__ __forceinline__ bool simt_consumer(const DecodeParams& prm, const WorkItem& item,
                                              int n_tok, int lead, int n_tiles, int r0,
                                              bool hold_last, int cw, const DecRing& R,
                                              int* abort_flag, float* red_o, float* red_m,
                                              float* red_l, float* red_lp) {
  constexpr bool FP8 = std::is_same<KV, E4m3>::value;
  using C = DecodeCfg<HEAD_DIM, GROUP, FP8 ? 1 : 2>;
  const int warp = cw, lane = threadIdx.x & 31;
  const int ch = lane % C::LPT;            // 16-byte chunk of the row this lane owns
  const int ts = lane / C::LPT;            // token slot within a pass
  const int blk = ch >> 3, c8 = ch & 7;
  // score scale in the log2 domain, with the kv head's key scale
  const float qscale =
      prm.sm_scale * kDecLog2e * (prm.k_head_scale ? prm.k_head_scale[item.head] : 1.f);
  float q[GROUP][8];
  {
    const uint16_t* qp = reinterpret_cast<const uint16_t*>(prm.q) +
                         (size_t(item.q_row) * prm.num_qo_heads + item.head * GROUP) * HEAD_DIM +
                         ch * 8;
#pragma unroll
    for (int h = 0; h < GROUP; ++h) {
      const uint4 u = *reinterpret_cast<const uint4*>(qp + h * HEAD_DIM);
      unpack8<E>(u, q[h]);
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
    const int s = ring_stage<NS>(R, r0 + i);
    if (!mbar_wait_warp(smem_u32(&R.full[s]), ring_phase<NS>(R, r0 + i), prm.wait_limit_ns,
                        abort_flag)) {
      if (lane == 0) { *abort_flag = 1; atomicOr(prm.err, kErrTimeout); }
      break;
    }
    const int ntok = min(C::TILE, n_tok - i * C::TILE);
    const int lo = i == 0 ? lead : 0;      // rows below lo are outside the window
    // 16-bit cache: the lane's 16 bytes in its 64-dim slice (swizzled);
    // FP8 cache: its 8 bytes of a HEAD_DIM-byte row (128-byte rows swizzled)
    const uint32_t kbase =
        ring_addr(R, s, C::STAGE_BYTES) + (FP8 ? 0 : blk * C::TILE * 128);
    const uint32_t vbase = kbase + C::KBYTES;
    auto row8 = [&](int r) -> uint32_t {
      return C::SWZ8 ? uint32_t(r * 128 + ((((ch >> 1) ^ (r & 7))) << 4) + (ch & 1) * 8)
                     : uint32_t(r * HEAD_DIM + ch * 8);
    };
#pragma unroll
    for (int p0 = 0; p0 < C::PASSES; p0 += C::SUB) {
      float sc[C::SUB][GROUP];
#pragma unroll
      for (int p = 0; p < C::SUB; ++p) {
        const int r = warp * C::TOK_PER_WARP + (p0 + p) * C::TPP + ts;
        float kf[8];
        if constexpr (FP8) E4m3::unpack8(lds64(kbase + row8(r)), kf);
        else unpack8<E>(lds128(kbase + swz(r, c8)), kf);
#pragma unroll
        for (int h = 0; h < GROUP; ++h) {
          float d0 = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) d0 = fmaf(q[h][j], kf[j], d0);
#pragma unroll
          for (int off = C::LPT / 2; off >= 1; off >>= 1)
            d0 += __shfl_xor_sync(0xffffffffu, d0, off);
          sc[p][h] = (r < ntok && r >= lo) ? d0 : -INFINITY;
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
          if constexpr (FP8) E4m3::unpack8(lds64(vbase + row8(r)), vf);
          else unpack8<E>(lds128(vbase + swz(r, c8)), vf);
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
    if (lane == 0 && !(hold_last && i == n_tiles - 1)) mbar_arrive(smem_u32(&R.empty[s]));
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

  // every consumer thread takes the same decision (abort_flag may still
  // change while warps arrive, so it is voted on at the barrier)
  const bool aborted = named_bar_or(1, C::NCW * 32, *abort_flag != 0);
  if (!aborted && lane < C::LPT) {
#pragma unroll
    for (int h = 0; h < GROUP; ++h) {
      float4* dst = reinterpret_cast<float4*>(red_o + (warp * GROUP + h) * HEAD_DIM + ch * 8);
      dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
      dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
      if (lane == 0) {
        red_m[warp * GROUP + h] = m[h];
        red_l[warp * GROUP + h] = l[h];
        red_lp[warp * GROUP + h] = l[h];
      }
    }
  }
  return aborted;
}

// The consumer warps' end of an item (`ctid` = consumer thread 0..NCW*32-1):
// merge the warps' states from the reduction arrays and write the row (or,
// for a split chunk, its fp32 partial state; the CTA that completes the
// split's last chunk then merges all of its partial states). `merge_last`
// is a shared-memory word. `red_ok` false means the item had no keys and no
// reduction area: every warp's state is empty, and the split merge reads its
// weights from global memory.
template <int HEAD_DIM, int GROUP, class E, class KV, int NCONS = 0>
__device__ __forceinline__ void decode_finish(const DecodeParams& prm, const WorkItem& item,
                                              int ctid, bool red_ok, float* red_o, float* red_m,
                                              float* red_l, float* red_lp, int* merge_last) {
  constexpr bool FP8 = std::is_same<KV, E4m3>::value;
  using C = DecodeCfg<HEAD_DIM, GROUP, FP8 ? 1 : 2>;
  // consumer warps whose states are merged (NCONS, or the configuration's)
  constexpr int NW = NCONS > 0 ? NCONS : C::NCW;
  const int tid = ctid;
  // the value scale of the cache, with the kv head's factor
  const float v_scale =
      prm.v_scale * (prm.v_head_scale ? prm.v_head_scale[item.head] : 1.f);
  named_bar_sync(1, NW * 32);
  for (int idx = tid; idx < GROUP * HEAD_DIM; idx += NW * 32) {
    const int h = idx / HEAD_DIM, dd = idx % HEAD_DIM;
    float rf = 0.f, L = 0.f, LP = 0.f, O = 0.f;
    if (red_ok) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w * GROUP + h]);
      rf = (M == -INFINITY) ? 0.f : M;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float sc = ex2(red_m[w * GROUP + h] - rf);
        L = fmaf(red_l[w * GROUP + h], sc, L);
        LP = fmaf(red_lp[w * GROUP + h], sc, LP);
        O = fmaf(red_o[(w * GROUP + h) * HEAD_DIM + dd], sc, O);
      }
    }
    const float o = (LP > 0.f) ? O * (v_scale / LP) : 0.f;
    const float lse = (L > 0.f) ? (rf + lg2(L)) * kDecLn2 : -INFINITY;
    const int hq = item.head * GROUP + h;
    if (item.slot < 0) {
      reinterpret_cast<uint16_t*>(prm.out)[(size_t(item.q_row) * prm.num_qo_heads + hq) *
                                               HEAD_DIM + dd] = E::one(o);
      if (dd == 0 && prm.lse) prm.lse[size_t(item.q_row) * prm.num_qo_heads + hq] = lse;
    } else {
      prm.partial_o[(size_t(item.slot) * prm.num_qo_heads + hq) * HEAD_DIM + dd] = o;
      if (dd == 0) prm.partial_lse[size_t(item.slot) * prm.num_qo_heads + hq] = lse;
    }
  }
  // Split request: the CTA that writes the last of its chunks' partial
  // states (for this kv head) merges them, so no second launch is needed.
  // Publication: the consumer threads' stores, a barrier of the consumer
  // warps, then one thread's gpu-scope fence and arrival count; the thread
  // that sees the final count fences before the warps read the other CTAs'
  // states (bypassing L1). The merge order is fixed by the slots, so the
  // result does not depend on which CTA comes last.
  if (item.slot >= 0) {
    named_bar_sync(1, NW * 32);
    if (tid == 0) {
      const MergeTask mt = prm.merges[item.merge];
      const int hkv = prm.num_qo_heads / GROUP;
      __threadfence();
      const uint32_t prev = atomicAdd(&prm.merge_counters[item.merge * hkv + item.head], 1u);
      *merge_last = prev == uint32_t(mt.n_states - 1);
      if (*merge_last) __threadfence();
    }
    named_bar_sync(1, NW * 32);
    if (*reinterpret_cast<volatile int*>(merge_last)) {
      const MergeTask mt = prm.merges[item.merge];
      // per head: M = max_i lse_i and w_i = exp(lse_i - M) / sum_j exp(lse_j - M),
      // kept in shared memory (the reduction area is free again) when it fits
      float* wgt = red_o;                       // [n_states][GROUP] when it fits
      float* hm = red_m;                        // [GROUP]: M
      float* hs = red_l;                        // [GROUP]: sum of exp(lse_i - M)
      const bool fits = red_ok && mt.n_states * GROUP <= NW * GROUP * HEAD_DIM;
      __shared__ float hm_g[GROUP], hs_g[GROUP];  // when there is no reduction area
      if (!red_ok) {
        hm = hm_g;
        hs = hs_g;
      }
      // every chunk state's lse of every head, loaded by all the consumer
      // threads at once (a few threads walking the states one L2 round trip
      // after another made the merging CTA the launch's last)
      if (fits) {
        for (int x = tid; x < mt.n_states * GROUP; x += NW * 32)
          wgt[x] = __ldcg(&prm.partial_lse[size_t(mt.slot_base + x / GROUP) * prm.num_qo_heads +
                                           item.head * GROUP + x % GROUP]);
        named_bar_sync(1, NW * 32);
      }
      if (tid < GROUP) {
        const int hq = item.head * GROUP + tid;
        // the chunks' states, and the row's shared-prefix states (if any)
        auto xlse = [&](int e) {
          return __ldcg(&prm.partial_lse[size_t(mt.extra_slot + e * mt.extra_stride) *
                                         prm.num_qo_heads + hq]);
        };
        auto slse = [&](int i) {
          return fits ? wgt[i * GROUP + tid]
                      : __ldcg(&prm.partial_lse[size_t(mt.slot_base + i) * prm.num_qo_heads + hq]);
        };
        float M = -INFINITY;
        for (int e = 0; e < mt.n_extra; ++e) M = fmaxf(M, xlse(e));
        for (int i = 0; i < mt.n_states; ++i) M = fmaxf(M, slse(i));
        float sw = 0.f;
        if (M != -INFINITY) {
          for (int i = 0; i < mt.n_states; ++i) {
            const float w = ex2((slse(i) - M) * kDecLog2e);
            if (fits) wgt[i * GROUP + tid] = w;   // -inf -> 0; this thread's column only
            sw += w;
          }
          for (int e = 0; e < mt.n_extra; ++e) sw += ex2((xlse(e) - M) * kDecLog2e);
        } else if (fits) {
          for (int i = 0; i < mt.n_states; ++i) wgt[i * GROUP + tid] = 0.f;
        }
        hm[tid] = M;
        hs[tid] = sw;
        const size_t orow = size_t(mt.out_row) * prm.num_qo_heads + hq;
        if (prm.lse) prm.lse[orow] = sw > 0.f ? M + lg2(sw) * kDecLn2 : -INFINITY;
      }
      named_bar_sync(1, NW * 32);
      for (int idx = tid; idx < GROUP * HEAD_DIM; idx += NW * 32) {
        const int h = idx / HEAD_DIM, dd = idx % HEAD_DIM;
        const int hq = item.head * GROUP + h;
        const float M = hm[h], sw = hs[h];
        float acc = 0.f;
        if (sw > 0.f) {
#pragma unroll 4
          for (int i = 0; i < mt.n_states; ++i) {
            const size_t row = size_t(mt.slot_base + i) * prm.num_qo_heads + hq;
            const float w = fits ? wgt[i * GROUP + h]
                                 : ex2((__ldcg(&prm.partial_lse[row]) - M) * kDecLog2e);
            acc = fmaf(w, __ldcg(&prm.partial_o[row * HEAD_DIM + dd]), acc);
          }
          for (int e = 0; e < mt.n_extra; ++e) {
            const size_t row = size_t(mt.extra_slot + e * mt.extra_stride) * prm.num_qo_heads + hq;
            const float w = ex2((__ldcg(&prm.partial_lse[row]) - M) * kDecLog2e);
            acc = fmaf(w, __ldcg(&prm.partial_o[row * HEAD_DIM + dd]), acc);
          }
        }
        const size_t orow = size_t(mt.out_row) * prm.num_qo_heads + hq;
        reinterpret_cast<uint16_t*>(prm.out)[orow * HEAD_DIM + dd] =
            E::one(sw > 0.f ? acc / sw : 0.f);
      }
    }
  }
}

}  // namespace
}  // namespace fi
