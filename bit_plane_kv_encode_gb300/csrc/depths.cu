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
#include "depths_core.cuh"

namespace bpkv {

struct DepthArgs {
  const float* q;
  const float* sigma2;
  const int32_t* budget_q;
  uint8_t* depths;
  int32_t n_heads;
  int32_t group;
  uint32_t* tickets;  // optional [N][H]: zeroed for the attention of this step
};

__global__ void __launch_bounds__(256) k_alloc_depths(DepthArgs a) {
  pdl_enter();
  __shared__ DepthSmem S;
  const int unit = blockIdx.x;
  const int s = unit / a.n_heads;
  if (a.tickets && threadIdx.x == 0) a.tickets[unit] = 0u;
  alloc_depths_cta(S, a.q + (int64_t)unit * a.group * kD, a.sigma2 + (int64_t)unit * kD, a.group, a.budget_q[s],
                   a.depths + (int64_t)unit * kD);
}

__global__ void __launch_bounds__(128) k_fixed_depths(const float* q, uint8_t* depths, int group, int n_channels,
                                                      int t, uint32_t* tickets) {
  pdl_enter();
  __shared__ DepthSmem S;
  const int unit = blockIdx.x;
  if (tickets && threadIdx.x == 0) tickets[unit] = 0u;
  fixed_depths_cta(S, q + (int64_t)unit * group * kD, group, n_channels, t, depths + (int64_t)unit * kD);
}

cudaError_t launch_alloc_depths(const bpkv_cache& c, const float* q, const float* sigma2, const int32_t* budget_q,
                                uint8_t* depths, cudaStream_t st, uint32_t* tickets) {
  DepthArgs a{q, sigma2, budget_q, depths, c.n_kv_heads, c.group, tickets};
  return launch_pdl(k_alloc_depths, dim3(c.n_seq * c.n_kv_heads), dim3(256), 0, st, a);
}

cudaError_t launch_fixed_depths(const bpkv_cache& c, const float* q, int32_t n_channels, int32_t depth,
                                uint8_t* depths, cudaStream_t st, uint32_t* tickets) {
  return launch_pdl(k_fixed_depths, dim3(c.n_seq * c.n_kv_heads), dim3(128), 0, st, q, depths, (int)c.group,
                    (int)n_channels, (int)depth, tickets);
}

}  // namespace bpkv
