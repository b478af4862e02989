// merge_states: combine attention states over disjoint key sets by
// log-sum-exp. For each output row and head, with M = max_i lse_i and
// w_i = exp(lse_i - M): o = sum_i w_i o_i / sum_i w_i, lse = M + ln sum_i w_i.
// The split order is fixed (i = 0, 1, ...), so results are deterministic.
// Used both as the ABI call fi_merge_states and after split-KV decode.
#include "elem.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace fi {

namespace {

using namespace dev;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMergeThreads = 128;

template <class E>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(MergeParams p) {
  const int r = blockIdx.x;
  int out_row = r, base = r * p.S, n = p.S;
  if (p.tasks) {
    const MergeTask t = p.tasks[r];
    out_row = t.out_row;
    base = t.slot_base;
    n = t.n_states;
  }
  const int q4 = p.d / 4;
  for (int idx = threadIdx.x; idx < p.H * q4; idx += kMergeThreads) {
    const int h = idx / q4, c = idx % q4;
    float M = -INFINITY;
    for (int i = 0; i < n; ++i) M = fmaxf(M, p.s[size_t(base + i) * p.H + h]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float sw = 0.f;
    if (M != -INFINITY) {
      for (int i = 0; i < n; ++i) {
        const float w = ex2((p.s[size_t(base + i) * p.H + h] - M) * kLog2e);  // -inf -> 0
        if (w == 0.f) continue;
        const float4 v =
            reinterpret_cast<const float4*>(p.v + (size_t(base + i) * p.H + h) * p.d)[c];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
        sw += w;
      }
    }
    const float inv = sw > 0.f ? 1.f / sw : 0.f;
    uint2 packed;
    packed.x = E::pack2(acc.x * inv, acc.y * inv);
    packed.y = E::pack2(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) +
                             (size_t(out_row) * p.H + h) * p.d)[c] = packed;
    if (c == 0 && p.lse)
      p.lse[size_t(out_row) * p.H + h] = sw > 0.f ? M + lg2(sw) * kLn2 : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, int n_rows, cudaStream_t stream) {
  if (n_rows <= 0 || p.H <= 0) return cudaSuccess;
  switch (p.dtype) {
    case FI_DTYPE_BF16: merge_kernel<Bf16><<<n_rows, kMergeThreads, 0, stream>>>(p); break;
    case FI_DTYPE_FP16: merge_kernel<Fp16><<<n_rows, kMergeThreads, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace fi
