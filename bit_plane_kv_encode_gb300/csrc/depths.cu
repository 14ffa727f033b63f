// Per-query read depths (Fathom page, section 1, observation 1: "reverse
// water-filling" on marginal value g_j 4^-t_j; section 2, "SparQ": fixed sets).
//
// Water-filling: one CTA per (sequence, KV head).  The 4 D items (j, t) are
// keyed by (value desc, item index asc) with item index 4 j + t, so equal values
// order by channel and, within a channel, by depth.  A bitonic sort in shared
// memory orders the 512 keys, a block scan accumulates their quarter-bit costs
// (5 for a channel's first bit: 4 for the plane + 1 for its fp16 scale; 4 after)
// and the items before the first one that does not fit, or is worthless, are
// taken.  This is the greedy heap's result computed as a single water level.
#include "common.cuh"

namespace bpkv {

struct DepthArgs {
  const float* q;
  const float* sigma2;
  const int32_t* budget_q;
  uint8_t* depths;
  int32_t n_heads;
  int32_t group;
};

constexpr int kItems = kD * 4;  // 512
constexpr int kNotTaken = 1 << 20;

__global__ void __launch_bounds__(256) k_alloc_depths(DepthArgs a) {
  const int unit = blockIdx.x;
  const int s = unit / a.n_heads;
  const int tid = threadIdx.x;
  __shared__ unsigned long long key[kItems];
  __shared__ int warp_tot[8];
  __shared__ int cut;
  __shared__ int cnt[kD];

  if (tid < kD) {
    const float* qp = a.q + (int64_t)unit * a.group * kD;
    const float s2 = a.sigma2[(int64_t)unit * kD + tid];
    float g = 0.f;
    for (int h = 0; h < a.group; ++h) {
      const float x = qp[h * kD + tid];
      g = __fadd_rn(g, __fmul_rn(__fmul_rn(x, x), s2));
    }
    const float quarter_pow[4] = {1.f, 0.25f, 0.0625f, 0.015625f};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float v = __fmul_rn(g, quarter_pow[t]);
      const uint32_t id = tid * 4 + t;
      key[id] = (v > 0.f) ? ((static_cast<unsigned long long>(__float_as_uint(v)) << 32) | (0xFFFFFFFFu - id))
                          : 0ull;
    }
    cnt[tid] = 0;
  }
  if (tid == 0) cut = kItems;
  __syncthreads();

  // Bitonic sort, descending.
  for (int size = 2; size <= kItems; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int i = 2 * tid - (tid & (stride - 1));
      const int j = i + stride;
      const bool desc = (i & size) == 0;
      const unsigned long long x = key[i], y = key[j];
      if ((x < y) == desc) {
        key[i] = y;
        key[j] = x;
      }
      __syncthreads();
    }
  }

  // Costs in sorted order; worthless items cost more than any budget.
  const unsigned long long k0 = key[2 * tid], k1 = key[2 * tid + 1];
  auto cost = [](unsigned long long k) -> int {
    if (k == 0ull) return kNotTaken;
    const uint32_t id = 0xFFFFFFFFu - static_cast<uint32_t>(k);
    return (id & 3u) == 0u ? 5 : 4;
  };
  const int c0 = cost(k0), c1 = cost(k1);
  // Block-wide inclusive scan of (c0 + c1).
  int x = c0 + c1;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  const int incl1 = before + x;      // cumulative cost through position 2 tid + 1
  const int incl0 = incl1 - c1;      // through position 2 tid
  const int B = a.budget_q[s];
  // worthless items (key 0) sort last and always stop the allocation
  if (incl0 > B || k0 == 0ull) atomicMin(&cut, 2 * tid);
  else if (incl1 > B || k1 == 0ull) atomicMin(&cut, 2 * tid + 1);
  __syncthreads();
  if (2 * tid < cut) atomicAdd(&cnt[(0xFFFFFFFFu - static_cast<uint32_t>(k0)) >> 2], 1);
  if (2 * tid + 1 < cut) atomicAdd(&cnt[(0xFFFFFFFFu - static_cast<uint32_t>(k1)) >> 2], 1);
  __syncthreads();
  if (tid < kD) a.depths[(int64_t)unit * kD + tid] = static_cast<uint8_t>(cnt[tid]);
}

// Fixed sets: the n_channels channels with the largest sum_h |q_hj| (ties to
// the lower index) at depth t.
__global__ void __launch_bounds__(128) k_fixed_depths(const float* q, uint8_t* depths, int group, int n_channels,
                                                      int t) {
  const int unit = blockIdx.x;
  const int j = threadIdx.x;
  __shared__ float asum[kD];
  const float* qp = q + (int64_t)unit * group * kD;
  float acc = 0.f;
  for (int h = 0; h < group; ++h) acc = __fadd_rn(acc, fabsf(qp[h * kD + j]));
  asum[j] = acc;
  __syncthreads();
  int rank = 0;
  for (int i = 0; i < kD; ++i) rank += (asum[i] > acc) || (asum[i] == acc && i < j);
  depths[(int64_t)unit * kD + j] = static_cast<uint8_t>(rank < n_channels ? t : 0);
}

cudaError_t launch_alloc_depths(const bpkv_cache& c, const float* q, const float* sigma2, const int32_t* budget_q,
                                uint8_t* depths, cudaStream_t st) {
  DepthArgs a{q, sigma2, budget_q, depths, c.n_kv_heads, c.group};
  k_alloc_depths<<<c.n_seq * c.n_kv_heads, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fixed_depths(const bpkv_cache& c, const float* q, int32_t n_channels, int32_t depth,
                                uint8_t* depths, cudaStream_t st) {
  k_fixed_depths<<<c.n_seq * c.n_kv_heads, 128, 0, st>>>(q, depths, c.group, n_channels, depth);
  return cudaGetLastError();
}

}  // namespace bpkv
