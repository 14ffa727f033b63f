// Shared device helpers of libbpkv (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bpkv.h"

namespace bpkv {

constexpr int kD = BPKV_HEAD_DIM;   // channels per head
constexpr int kBlock = 64;          // tokens per scale block / plane word
constexpr int kPlanes = 4;          // bits per code

// Per-unit (sequence, KV head) base offsets of the cache arrays.
struct Unit {
  int64_t nb_cap;  // words per plane row
  int64_t cap;     // token capacity
  __host__ __device__ int64_t plane_base(int64_t unit) const { return unit * kD * kPlanes * nb_cap; }
  __host__ __device__ int64_t scale_base(int64_t unit) const { return unit * kD * nb_cap; }
  __host__ __device__ int64_t row_base(int64_t unit) const { return unit * cap * kD; }
};

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float fp16_bits_to_float(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}

// Order-preserving map float -> uint32 (larger float -> larger key); -0 and +0
// get the same key, as they compare equal.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

}  // namespace bpkv
