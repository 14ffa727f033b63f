// Device building block of the bit-plane encoder (Fathom page, section 3.2),
// shared by the append kernel and the fused decode kernel.  See encode.cu.
#pragma once

#include "common.cuh"

namespace bpkv {

// Append the tokens of one 64-token block of one unit and re-encode the block,
// for channels c_lo .. c_lo + blockDim.x / PARTS - 1.  Rows t0 .. t0 + cnt - 1
// are the block's tokens; those below n_old come from the stored rows, the
// others from knew/vnew (row r of the new tokens is token n_old + r), which are
// also copied into the row store (these channels of them).  Threads: PARTS per
// channel, 64 / PARTS tokens each.  With a basis R (the unit's [D][D]), the
// codes are those of the keys k R: every channel of the block's rows is staged,
// and channel j of token r is the bf16 rounding of the float32 fused
// multiply-add chain sum_i k_ri R[i][j] in order i = 0 .. D-1.
template <int PARTS>
__device__ void encode_block_cta(uint16_t (*kb)[kD], uint16_t* krow, uint16_t* vrow, const uint16_t* knew,
                                 const uint16_t* vnew, int64_t n_old, int64_t t0, int cnt, uint64_t* pw_base,
                                 uint16_t* scale_base, int64_t nb_cap, int64_t blk, int c_lo = 0,
                                 const float* __restrict__ basis = nullptr) {
  constexpr int TOK = kBlock / PARTS;
  constexpr int kBatch = 4;  // independent 16-byte loads in flight per thread
  const int c_n = (int)(blockDim.x / PARTS);        // this CTA's channels [c_lo, c_lo + c_n)
  const int s_lo = basis ? 0 : c_lo;                // staged channels
  const int n8 = (basis ? kD : c_n) / 8;            // 16-byte pieces of a staged row
  for (int v0 = threadIdx.x; v0 < cnt * n8; v0 += kBatch * blockDim.x) {
    uint4 val[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int v = v0 + b * blockDim.x;
      if (v < cnt * n8) {
        const int r = v / n8, c8 = s_lo + (v % n8) * 8;
        const int64_t tok = t0 + r;
        val[b] = tok < n_old ? *reinterpret_cast<const uint4*>(krow + tok * kD + c8)
                             : *reinterpret_cast<const uint4*>(knew + (tok - n_old) * kD + c8);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int v = v0 + b * blockDim.x;
      if (v < cnt * n8) {
        const int r = v / n8, c8 = s_lo + (v % n8) * 8;
        const int64_t tok = t0 + r;
        if (tok >= n_old && c8 >= c_lo && c8 < c_lo + c_n) {
          const int64_t src = (tok - n_old) * kD + c8;
          *reinterpret_cast<uint4*>(krow + tok * kD + c8) = val[b];
          *reinterpret_cast<uint4*>(vrow + tok * kD + c8) = *reinterpret_cast<const uint4*>(vnew + src);
        }
        *reinterpret_cast<uint4*>(&kb[r][c8]) = val[b];
      }
    }
  }
  __syncthreads();
  // thread = (channel j, part qd): tokens TOK qd .. TOK qd + TOK - 1; the parts
  // of a channel are adjacent lanes.
  const int j = c_lo + threadIdx.x / PARTS, qd = threadIdx.x % PARTS;
  const int r0 = TOK * qd, r1 = min(r0 + TOK, cnt);
  float kv[TOK];  // the coded value of channel j of this thread's tokens
  if (basis) {
#pragma unroll
    for (int t = 0; t < TOK; ++t) kv[t] = 0.f;
    for (int i = 0; i < kD; ++i) {
      const float rv = basis[i * kD + j];
#pragma unroll
      for (int t = 0; t < TOK; ++t)
        if (r0 + t < r1) kv[t] = __fmaf_rn(bf16_bits_to_float(kb[r0 + t][i]), rv, kv[t]);
    }
#pragma unroll
    for (int t = 0; t < TOK; ++t) kv[t] = __bfloat162float(__float2bfloat16_rn(kv[t]));
  } else {
#pragma unroll
    for (int t = 0; t < TOK; ++t) kv[t] = r0 + t < r1 ? bf16_bits_to_float(kb[r0 + t][j]) : 0.f;
  }
  float amax = 0.f;
#pragma unroll
  for (int t = 0; t < TOK; ++t)
    if (r0 + t < r1) amax = fmaxf(amax, fabsf(kv[t]));
#pragma unroll
  for (int o = 1; o < PARTS; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // a/8 is exact in float32; values past the largest half saturate to it.
  const __half hs = __float2half_rn(fminf(amax * 0.125f, 65504.f));
  const uint16_t s16 = __half_as_ushort(hs);
  const float sc = __half2float(hs);
  uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;  // this part's TOK bits of each plane
#pragma unroll
  for (int t = 0; t < TOK; ++t) {
    if (r0 + t >= r1) break;
    int c = 8;
    if (s16 != 0) {
      float f = floorf(__fdiv_rn(kv[t], sc));
      f = fminf(fmaxf(f, -8.f), 7.f);
      c = static_cast<int>(f) + 8;
    }
    const uint32_t bit = 1u << t;
    if (c & 8) w0 |= bit;
    if (c & 4) w1 |= bit;
    if (c & 2) w2 |= bit;
    if (c & 1) w3 |= bit;
  }
  // each part owns TOK / 8 bytes of the little-endian 64-bit word
  uint64_t* pw = pw_base + (int64_t)j * kPlanes * nb_cap + blk;
  if constexpr (PARTS == 4) {
    uint16_t* p = reinterpret_cast<uint16_t*>(pw) + qd;
    p[0] = (uint16_t)w0;
    p[4 * nb_cap] = (uint16_t)w1;
    p[8 * nb_cap] = (uint16_t)w2;
    p[12 * nb_cap] = (uint16_t)w3;
  } else {
    static_assert(PARTS == 2, "2 or 4 parts per channel");
    uint32_t* p = reinterpret_cast<uint32_t*>(pw) + qd;
    p[0] = w0;
    p[2 * nb_cap] = w1;
    p[4 * nb_cap] = w2;
    p[6 * nb_cap] = w3;
  }
  if (qd == 0) scale_base[(int64_t)j * nb_cap + blk] = s16;
}

}  // namespace bpkv
