// Shared pieces of the tensor-core kernels: per-I/O-type constants, the
// 128-byte-swizzled shared-memory layout, and host helpers for the TMA maps
// of the [b, L, heads-or-groups, dim] input tensors.
#pragma once

#include <cuda_bf16.h>

#include <algorithm>

#include "ptx.cuh"
#include "ssd_internal.cuh"
#include "tmap.cuh"

namespace ssd {

// bf16 operands run kind::f16 MMAs (K = 16 per instruction); fp32 operands
// run kind::tf32 (K = 8).  kAE = elements per 128-byte swizzle row.
template <typename IO>
struct IoT;
template <>
struct IoT<__nv_bfloat16> {
  static constexpr int kE = 2, kAE = 64, kKmma = 16;
  static constexpr bool kTf32 = false;
};
template <>
struct IoT<float> {
  static constexpr int kE = 4, kAE = 32, kKmma = 8;
  static constexpr bool kTf32 = true;
};

template <typename IO>
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, bool a_mn, bool b_mn) {
  return IoT<IO>::kTf32 ? ptx::idesc_tf32(M, N, a_mn, b_mn) : ptx::idesc_bf16(M, N, a_mn, b_mn);
}

// Byte offset of byte `cb` (0..127) of row r in a 128-byte-swizzled region
// (rows of 128 bytes, 16-byte chunks permuted by XOR with the row index mod
// 8, as the TMA SWIZZLE_128B mode and the tensor-core descriptors expect).
__device__ __forceinline__ uint32_t sw128(int r, int cb) {
  return (uint32_t)(r * 128 + ((((cb >> 4) ^ r) & 7) << 4) + (cb & 15));
}

// 16 bytes of I/O data from fp32 values: 8 bf16 (round to nearest) or 4 fp32.
__device__ __forceinline__ uint4 pack_io16(const float *v, __nv_bfloat16 *) {
  uint4 o;
  __nv_bfloat162 t;
  t = __floats2bfloat162_rn(v[0], v[1]);
  o.x = *reinterpret_cast<uint32_t *>(&t);
  t = __floats2bfloat162_rn(v[2], v[3]);
  o.y = *reinterpret_cast<uint32_t *>(&t);
  t = __floats2bfloat162_rn(v[4], v[5]);
  o.z = *reinterpret_cast<uint32_t *>(&t);
  t = __floats2bfloat162_rn(v[6], v[7]);
  o.w = *reinterpret_cast<uint32_t *>(&t);
  return o;
}
// fp32 operands of kind::tf32 MMAs: round to nearest tf32 here (the tensor
// core would otherwise drop the low 13 mantissa bits).
__device__ __forceinline__ uint32_t to_tf32(float f) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
  return r;
}
__device__ __forceinline__ uint4 pack_io16(const float *v, float *) {
  return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                    __float_as_uint(v[3]));
}
// 16 bytes of tensor-core operand data: 8 bf16, or 4 fp32 rounded to tf32.
__device__ __forceinline__ uint4 pack_op16(const float *v, __nv_bfloat16 *p) {
  return pack_io16(v, p);
}
__device__ __forceinline__ uint4 pack_op16(const float *v, float *) {
  return make_uint4(to_tf32(v[0]), to_tf32(v[1]), to_tf32(v[2]), to_tf32(v[3]));
}

// Unpack 16 bytes of I/O data into fp32 values (8 for bf16, 4 for fp32).
__device__ __forceinline__ void unpack16(uint4 u, float *v, __nv_bfloat16 *) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 t = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
    const float2 f = __bfloat1622float2(t);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void unpack16(uint4 u, float *v, float *) {
  v[0] = __uint_as_float(u.x);
  v[1] = __uint_as_float(u.y);
  v[2] = __uint_as_float(u.z);
  v[3] = __uint_as_float(u.w);
}

// TMA map of a [b, L, n, dim] tensor (x with n = nheads, B/C with
// n = ngroups) with boxes of (one 128-byte row of `dim`) x 1 x rows x 1.
inline bool make_tmap_bl(CUtensorMap *map, const void *base, bool bf16, int64_t b, int64_t L,
                         int64_t n, int64_t dim, int rows) {
  const uint64_t e = bf16 ? 2 : 4;
  const uint64_t dims[4] = {(uint64_t)dim, (uint64_t)n, (uint64_t)L, (uint64_t)b};
  const uint64_t strides[3] = {dim * e, n * dim * e, L * n * dim * e};
  const uint32_t box[4] = {(uint32_t)(128 / e), 1u, (uint32_t)rows, 1u};
  return make_tmap_sw128(map, base, bf16, 4, dims, strides, box);
}

}  // namespace ssd
