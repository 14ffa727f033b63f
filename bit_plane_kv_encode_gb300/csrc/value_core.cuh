// Device building block of the value-side code (ReadKV page, sections 5.3-5.4):
// the value rows' own 4-bit code with one fp16 scale per row, written as
// token-major bit planes when tokens are appended.  Shared by the append
// kernels; the stage that reads it is in vdepth.cu.
#pragma once

#include "common.cuh"

namespace bpkv {

// Code one value row (128 bf16 values) with a whole warp: lane l holds
// channels l, l + 32, l + 64, l + 96; the plane words come from ballots.
__device__ __forceinline__ void encode_value_row(const uint16_t* __restrict__ v, uint64_t* __restrict__ vp,
                                                 uint16_t* __restrict__ vs) {
  const int lane = threadIdx.x & 31;
  float x[4];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[i] = bf16_bits_to_float(v[lane + 32 * i]);
    amax = fmaxf(amax, fabsf(x[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // a/8 is exact in float32; values past the largest half saturate to it
  const __half hs = __float2half_rn(fminf(amax * 0.125f, 65504.f));
  const uint16_t s16 = __half_as_ushort(hs);
  const float sc = __half2float(hs);
  int c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    c[i] = 8;
    if (s16 != 0) {
      float f = floorf(__fdiv_rn(x[i], sc));
      f = fminf(fmaxf(f, -8.f), 7.f);
      c[i] = static_cast<int>(f) + 8;
    }
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t b0 = __ballot_sync(0xffffffffu, (c[0] >> (3 - p)) & 1);
    const uint32_t b1 = __ballot_sync(0xffffffffu, (c[1] >> (3 - p)) & 1);
    const uint32_t b2 = __ballot_sync(0xffffffffu, (c[2] >> (3 - p)) & 1);
    const uint32_t b3 = __ballot_sync(0xffffffffu, (c[3] >> (3 - p)) & 1);
    if (lane == 2 * p) vp[2 * p] = ((uint64_t)b1 << 32) | b0;
    if (lane == 2 * p + 1) vp[2 * p + 1] = ((uint64_t)b3 << 32) | b2;
  }
  if (lane == 0) *vs = s16;
}

// Value rows of new tokens t0 .. t0 + cnt - 1 that are at or past n_old
// (row r of vnew is token n_old + r), one warp per row; warps w0, w0 + nw, ...
// of the calling CTA take part.
__device__ __forceinline__ void encode_value_rows(const uint16_t* __restrict__ vnew, int64_t n_old, int64_t t0, int cnt,
                                  uint64_t* __restrict__ vplanes, uint16_t* __restrict__ vscales, int w0, int nw) {
  const int warp = threadIdx.x >> 5;
  if (warp < w0) return;
  const int64_t first = max64(t0, n_old);
  for (int64_t tok = first + (warp - w0); tok < t0 + cnt; tok += nw)
    encode_value_row(vnew + (tok - n_old) * kD, vplanes + tok * (kPlanes * kD / 64), vscales + tok);
}

}  // namespace bpkv
