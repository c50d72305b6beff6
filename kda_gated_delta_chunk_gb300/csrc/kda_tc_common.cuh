// Device helpers shared by the tcgen05 chunk kernels (fused and k-side):
// fast exp2 / reciprocal, packed bf16 products, shared-memory accessors, the
// SW128 operand descriptors of a K step, and the warp-level tf32 16 x 16
// product used by the blocked unit-lower-triangular inverse.
#pragma once

#include "kda_sm100.cuh"

namespace kda {
namespace tcc {

using namespace sm100;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int NS = 68;   // fp32 row stride (floats) of the 64 x 64 T scratch: 16-byte rows,
                         // column accesses spread over the banks

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcpf(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigm(float x) { return rcpf(1.0f + ex2f(-x * kLog2e)); }
// bf16x2 product, rounded to nearest even
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ void st_u32(unsigned char* base, uint32_t off, uint32_t v) {
  *reinterpret_cast<uint32_t*>(base + off) = v;
}
__device__ __forceinline__ void st_u128(unsigned char* base, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}
__device__ __forceinline__ uint32_t ld_u32(const unsigned char* base, uint32_t off) {
  return *reinterpret_cast<const uint32_t*>(base + off);
}
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// K-step descriptors
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int rows, int ks) {
  return sdesc_sw128(tile + (ks >> 2) * rows * 128 + (ks & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, uint32_t lbo, int ks) {
  return sdesc_sw128(tile + ks * 2048, lbo, 1024);
}

// One warp: D(16 x 16) = -? A(16 x K) B(K x 16), fp32 smem matrices with row stride NS,
// tf32 tensor-core products, K a multiple of 8.  Result written to `dst` (stride NS).
template <int K>
__device__ __forceinline__ void warp_gemm_16x16(const float* A, const float* B, float* dst,
                                                float sign, int lane) {
  const int g = lane >> 2, t = lane & 3;
  float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 8) {
    uint32_t a[4], b0[2], b1[2];
    a[0] = to_tf32(A[g * NS + k0 + t]);
    a[1] = to_tf32(A[(g + 8) * NS + k0 + t]);
    a[2] = to_tf32(A[g * NS + k0 + t + 4]);
    a[3] = to_tf32(A[(g + 8) * NS + k0 + t + 4]);
    b0[0] = to_tf32(B[(k0 + t) * NS + g]);
    b0[1] = to_tf32(B[(k0 + t + 4) * NS + g]);
    b1[0] = to_tf32(B[(k0 + t) * NS + 8 + g]);
    b1[1] = to_tf32(B[(k0 + t + 4) * NS + 8 + g]);
    mma_tf32_16x8x8(d0, a, b0);
    mma_tf32_16x8x8(d1, a, b1);
  }
  *reinterpret_cast<float2*>(dst + g * NS + 2 * t) = make_float2(sign * d0[0], sign * d0[1]);
  *reinterpret_cast<float2*>(dst + (g + 8) * NS + 2 * t) = make_float2(sign * d0[2], sign * d0[3]);
  *reinterpret_cast<float2*>(dst + g * NS + 8 + 2 * t) = make_float2(sign * d1[0], sign * d1[1]);
  *reinterpret_cast<float2*>(dst + (g + 8) * NS + 8 + 2 * t) =
      make_float2(sign * d1[2], sign * d1[3]);
}

}  // namespace tcc
}  // namespace kda
