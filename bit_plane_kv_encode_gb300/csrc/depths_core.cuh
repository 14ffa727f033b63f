// Device building blocks of the depth allocation (Fathom page, section 1,
// observation 1; section 2 "SparQ" for the fixed sets), shared by the
// stand-alone kernels and the fused decode kernel.  See depths.cu.
#pragma once

#include "common.cuh"

namespace bpkv {

constexpr int kItems = kD * 4;  // 512 items (channel, next bit)
constexpr int kNotTaken = 1 << 20;

struct DepthSmem {
  unsigned long long key[kItems];
  int warp_tot[8];
  int cut;
  int cnt[kD];
  float asum[kD];
};

// Water-filling for one (sequence, KV head): qp [G][D], s2 [D], budget B in
// quarter-bits; depths written to out[0..D).  Needs blockDim.x == 256.
static __device__ void alloc_depths_cta(DepthSmem& S, const float* __restrict__ qp, const float* __restrict__ s2, int G,
                                 int B, uint8_t* out) {
  const int tid = threadIdx.x;
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
      S.key[id] = (v > 0.f) ? ((static_cast<unsigned long long>(__float_as_uint(v)) << 32) | (0xFFFFFFFFu - id))
                            : 0ull;
    }
    S.cnt[tid] = 0;
  }
  if (tid == 0) S.cut = kItems;
  __syncthreads();
  // Bitonic sort, descending.
#pragma unroll
  for (int size = 2; size <= kItems; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int i = 2 * tid - (tid & (stride - 1));
      const int j = i + stride;
      const bool desc = (i & size) == 0;
      const unsigned long long x = S.key[i], y = S.key[j];
      if ((x < y) == desc) {
        S.key[i] = y;
        S.key[j] = x;
      }
      __syncthreads();
    }
  }
  // Costs in sorted order; worthless items cost more than any budget.
  const unsigned long long k0 = S.key[2 * tid], k1 = S.key[2 * tid + 1];
  auto cost = [](unsigned long long k) -> int {
    if (k == 0ull) return kNotTaken;
    const uint32_t id = 0xFFFFFFFFu - static_cast<uint32_t>(k);
    return (id & 3u) == 0u ? 5 : 4;
  };
  const int c0 = cost(k0), c1 = cost(k1);
  int x = c0 + c1;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) S.warp_tot[warp] = x;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += S.warp_tot[w];
  const int incl1 = before + x;  // cumulative cost through position 2 tid + 1
  const int incl0 = incl1 - c1;  // through position 2 tid
  // worthless items (key 0) sort last and always stop the allocation
  if (incl0 > B || k0 == 0ull) atomicMin(&S.cut, 2 * tid);
  else if (incl1 > B || k1 == 0ull) atomicMin(&S.cut, 2 * tid + 1);
  __syncthreads();
  if (2 * tid < S.cut) atomicAdd(&S.cnt[(0xFFFFFFFFu - static_cast<uint32_t>(k0)) >> 2], 1);
  if (2 * tid + 1 < S.cut) atomicAdd(&S.cnt[(0xFFFFFFFFu - static_cast<uint32_t>(k1)) >> 2], 1);
  __syncthreads();
  if (tid < kD) out[tid] = static_cast<uint8_t>(S.cnt[tid]);
}

// Fixed sets: the n_channels channels with the largest sum_h |q_hj| (ties to
// the lower index) at depth t.  Threads 0..127 take part.
static __device__ void fixed_depths_cta(DepthSmem& S, const float* __restrict__ qp, int G, int n_channels, int t,
                                 uint8_t* out) {
  const int j = threadIdx.x;
  float acc = 0.f;
  if (j < kD) {
    for (int h = 0; h < G; ++h) acc = __fadd_rn(acc, fabsf(qp[h * kD + j]));
    S.asum[j] = acc;
  }
  __syncthreads();
  if (j < kD) {
    int rank = 0;
    for (int i = 0; i < kD; ++i) rank += (S.asum[i] > acc) || (S.asum[i] == acc && i < j);
    out[j] = static_cast<uint8_t>(rank < n_channels ? t : 0);
  }
  __syncthreads();
}

}  // namespace bpkv
