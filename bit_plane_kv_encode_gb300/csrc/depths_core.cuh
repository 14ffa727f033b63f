// Device building blocks of the depth allocation (Fathom page, section 1,
// observation 1; section 2 "SparQ" for the fixed sets), shared by the
// stand-alone kernels and the fused decode kernel.  See depths.cu.
#pragma once

#include "common.cuh"

namespace bpkv {

constexpr int kItems = kD * 4;  // 512 items (channel, next bit)

struct DepthSmem {
  uint32_t hist[256];  // per radix bin: item count << 16 | summed cost
  int cut_bin, done;
  uint32_t rem;
  unsigned long long top;  // the first non-fitting item's key bits above the level's shift
  int shift;
  float asum[kD];
};

// Water-filling for one (sequence, KV head): qp [G][D], s2 [D], budget B in
// quarter-bits; depths written to out[0..D) and returned to thread j < D (its
// channel's), 0 to the others.  Needs blockDim.x == 256.
//
// The items (j, t) in descending key order (value g_j 4^-t, then the lower
// item index 4 j + t first) are taken until the first one, X, whose running
// cost (5 quarter-bits for a channel's first plane and scale, 4 after) passes
// B, or the first worthless one (value <= 0).  X is found by a radix select
// over the 64-bit keys, 8 bits at a time from the top, with bins weighted by
// cost: at each level the bin where the running cost from the top first
// passes the budget left holds X.  Once X is alone in its bin the taken items
// are exactly those whose key bits above the level's shift exceed the bin's;
// if every positive item fits, all of them are taken.
static __device__ int alloc_depths_cta(DepthSmem& S, const float* __restrict__ qp, const float* __restrict__ s2, int G,
                                        int B, uint8_t* out) {
  const int tid = threadIdx.x, lane = tid & 31;
  unsigned long long key[4] = {0ull, 0ull, 0ull, 0ull};
  if (tid < kD) {
    const float sv = s2[tid];
    float g = 0.f;
    for (int h = 0; h < G; ++h) {
      const float x = qp[h * kD + tid];
      g = __fadd_rn(g, __fmul_rn(__fmul_rn(x, x), sv));
    }
    const float quarter_pow[4] = {1.f, 0.25f, 0.0625f, 0.015625f};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float v = __fmul_rn(g, quarter_pow[t]);
      const uint32_t id = tid * 4 + t;
      key[t] = (v > 0.f) ? ((static_cast<unsigned long long>(__float_as_uint(v)) << 32) | (0xFFFFFFFFu - id)) : 0ull;
    }
  }
  if (tid == 0) {
    S.rem = B < 0 ? 0u : (uint32_t)B;
    S.done = 0;
    S.top = 0ull;
    S.shift = 64;
  }
  unsigned long long pre = 0ull;  // the digits above the current level, in place
  for (int shift = 56; shift >= 0; shift -= 8) {
    S.hist[tid] = 0u;  // blockDim.x == 256 bins
    __syncthreads();
    if (tid < kD) {
      const unsigned long long hi_mask = shift == 56 ? 0ull : (~0ull << (shift + 8));
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (key[t] != 0ull && (key[t] & hi_mask) == pre)
          atomicAdd(&S.hist[(key[t] >> shift) & 0xFF], (1u << 16) | (t == 0 ? 5u : 4u));
    }
    __syncthreads();
    if (tid < 32) {
      // bins from the top, 8 per lane (lane 0: bins 255 .. 248): the bin where
      // the running cost first passes the budget left
      const uint32_t rem = S.rem;
      uint32_t c8[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c8[i] = S.hist[255 - 8 * lane - i] & 0xFFFFu;
        sum += c8[i];
      }
      uint32_t incl = sum;  // inclusive from lane 0
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t before_lane = incl - sum;
      int bin = -1;
      uint32_t before = 0;
      if (before_lane <= rem && incl > rem) {
        uint32_t run = before_lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (bin < 0 && run + c8[i] > rem) {
            bin = 255 - 8 * lane - i;
            before = run;
          }
          run += c8[i];
        }
      }
      const uint32_t hb = __ballot_sync(0xffffffffu, bin >= 0);
      if (lane == 0) S.cut_bin = -1;
      __syncwarp();
      if (hb && lane == __ffs(hb) - 1) {
        S.cut_bin = bin;
        S.rem = rem - before;
      }
      __syncwarp();
      if (lane == 0) {
        const int b = S.cut_bin;
        if (b < 0) {
          S.done = 1;  // every positive item fits
        } else if ((S.hist[b] >> 16) == 1u || shift == 0) {
          S.done = 2;  // X alone in its bin
          S.top = (pre >> shift) | (unsigned long long)b;
          S.shift = shift;
        }
      }
    }
    __syncthreads();
    if (S.done != 0) break;
    pre |= (unsigned long long)S.cut_bin << shift;
  }
  // depth of channel tid: its items taken (keys in descending order per channel)
  int t = 0;
  if (tid < kD) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool taken = key[i] != 0ull && (S.done == 1 || (key[i] >> S.shift) > S.top);
      t += taken ? 1 : 0;
    }
    out[tid] = static_cast<uint8_t>(t);
  }
  __syncthreads();
  return t;
}

// Fixed sets: the n_channels channels with the largest sum_h |q_hj| (ties to
// the lower index) at depth t; returned to thread j < D as for the
// water-filling.  Threads 0..127 take part.
static __device__ int fixed_depths_cta(DepthSmem& S, const float* __restrict__ qp, int G, int n_channels, int t,
                                       uint8_t* out) {
  const int j = threadIdx.x;
  float acc = 0.f;
  if (j < kD) {
    for (int h = 0; h < G; ++h) acc = __fadd_rn(acc, fabsf(qp[h * kD + j]));
    S.asum[j] = acc;
  }
  __syncthreads();
  int d = 0;
  if (j < kD) {
    int rank = 0;
    for (int i = 0; i < kD; ++i) rank += (S.asum[i] > acc) || (S.asum[i] == acc && i < j);
    d = rank < n_channels ? t : 0;
    out[j] = static_cast<uint8_t>(d);
  }
  __syncthreads();
  return d;
}

}  // namespace bpkv
