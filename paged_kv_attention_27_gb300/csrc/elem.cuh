// Element types of q, K, V and out: bf16 or fp16. Both are 16-bit words;
// the kernels move them untouched (TMA, ldmatrix, tcgen05 operands) and only
// convert where they do arithmetic, so every kernel takes one of these two
// traits structs as a template parameter.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace fi {
namespace dev {

struct Bf16 {
  static constexpr int kDtype = 0;          // FI_DTYPE_BF16
  static constexpr uint32_t kMmaFmt = 1;    // tcgen05 kind::f16 A/B format code
  // the two halves of a packed pair, exactly
  __device__ static __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
  __device__ static __forceinline__ float hi(uint32_t w) {
    return __uint_as_float(w & 0xffff0000u);
  }
  // round-to-nearest-even into a packed pair / one element
  __device__ static __forceinline__ uint32_t pack2(float l, float h) {
    __nv_bfloat162 v = __floats2bfloat162_rn(l, h);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __device__ static __forceinline__ uint16_t one(float x) {
    __nv_bfloat16 v = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&v);
  }
  // D (16x8, fp32) += A (16x16) B (16x8), warp-level
  __device__ static __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                                  uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

struct Fp16 {
  static constexpr int kDtype = 1;          // FI_DTYPE_FP16
  static constexpr uint32_t kMmaFmt = 0;
  __device__ static __forceinline__ float lo(uint32_t w) {
    return __half2float(__ushort_as_half(uint16_t(w & 0xffffu)));
  }
  __device__ static __forceinline__ float hi(uint32_t w) {
    return __half2float(__ushort_as_half(uint16_t(w >> 16)));
  }
  __device__ static __forceinline__ uint32_t pack2(float l, float h) {
    __half2 v = __floats2half2_rn(l, h);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __device__ static __forceinline__ uint16_t one(float x) {
    return __half_as_ushort(__float2half_rn(x));
  }
  __device__ static __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                                  uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

// FP8 E4M3 cache elements (OCP format): converted exactly to fp16 pairs by
// the hardware conversion, then to floats.
struct E4m3 {
  static constexpr int kDtype = 2;          // FI_DTYPE_E4M3
  // four packed e4m3 -> four floats (exact)
  __device__ static __forceinline__ void unpack4(uint32_t w, float* f) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(w & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(w >> 16), __NV_E4M3);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  }
  // eight packed e4m3 (8 bytes) -> eight floats
  __device__ static __forceinline__ void unpack8(const uint2& u, float (&f)[8]) {
    unpack4(u.x, f);
    unpack4(u.y, f + 4);
  }
  // two packed e4m3 (low 16 bits) -> an fp16 pair, first element low (exact)
  __device__ static __forceinline__ uint32_t to_f16x2(uint32_t w) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(w & 0xffffu), __NV_E4M3);
    return uint32_t(h.x) | (uint32_t(h.y) << 16);
  }
  // two floats -> two packed e4m3 in the low 16 bits (a in the low byte),
  // rounded to nearest even, finite values saturated at +-448
  __device__ static __forceinline__ uint32_t from_f32x2(float a, float b) {
    return uint32_t(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
  }
  // D += A B for A 16x32 (row-major) and B 32x8 (column-major) e4m3
  // operands, four elements per register, fp32 accumulators
  __device__ static __forceinline__ void mma16832(float (&d)[4], const uint32_t (&a)[4],
                                                  uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

// Eight packed elements (one 16-byte chunk) -> eight floats.
template <class E>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = E::lo(u.x); f[1] = E::hi(u.x);
  f[2] = E::lo(u.y); f[3] = E::hi(u.y);
  f[4] = E::lo(u.z); f[5] = E::hi(u.z);
  f[6] = E::lo(u.w); f[7] = E::hi(u.w);
}

}  // namespace dev
}  // namespace fi
