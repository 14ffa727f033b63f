// Per-query read depths (Fathom page, section 1, observation 1: "reverse
// water-filling" on marginal value g_j 4^-t_j; section 2, "SparQ": fixed sets).
//
// Water-filling: one CTA per (sequence, KV head).  The 4 D items (j, t) are
// keyed by (value desc, item index asc) with item index 4 j + t, so equal values
// order by channel and, within a channel, by depth.  The items before the
// first one that does not fit, or is worthless, are taken, with quarter-bit
// costs (5 for a channel's first bit: 4 for the plane + 1 for its fp16 scale;
// 4 after); a cost-weighted radix select over the 512 keys finds that item
// (depths_core.cuh).  This is the greedy heap's result computed as a single
// water level.
//
// In a decode step the same CTA also builds the unit's scan plan (channel
// groups, plane rows, weights q 2^(4-t-pos)) once, so that every scan CTA of
// the unit copies it instead of deriving it again from the depths.
//
// k_front runs a decode step's first work in one launch: per unit, the
// append and re-encode of the new tokens' block(s) (which also clear the
// unit's selection histograms and counters) beside the depth allocation and
// plan; the two do not depend on each other.
#include "depths_core.cuh"
#include "encode_core.cuh"
#include "scan_core.cuh"
#include "value_core.cuh"

#include <type_traits>

namespace bpkv {

struct DepthArgs {
  const float* q;
  const float* sigma2;
  const int32_t* budget_q;
  uint8_t* depths;
  int32_t n_heads;
  int32_t group;
  uint32_t* tickets;  // optional [N][H]: zeroed for the attention of this step
  void* plan;         // optional [N][H] ScanPlan<GP>
  int32_t n_channels; // fixed sets only
  int32_t depth;      // fixed sets only
  uint32_t* hist;     // optional [N][H][G][kTopkBins]: zeroed for the scan of this step
  uint32_t* ctr;      // optional [N][H][G][kSelCounters] selection counters: zeroed with hist
  int32_t* status;    // optional device status word (bounds-checked builds record in it)
};

// Zero this unit's selection histograms (G kTopkBins words).
__device__ __forceinline__ void zero_hist(const DepthArgs& a, int64_t unit) {
  uint4* h = reinterpret_cast<uint4*>(a.hist + unit * a.group * kTopkBins);
  for (int e = threadIdx.x; e < a.group * kTopkBins / 4; e += blockDim.x) h[e] = make_uint4(0u, 0u, 0u, 0u);
  if (a.ctr && (int)threadIdx.x < kSelCounters * a.group) a.ctr[unit * kSelCounters * a.group + threadIdx.x] = 0u;
}

// Build the scan plan of this unit from the depths the CTA just found (thread
// j < D holds its channel's in t) and store it.
template <int GP>
__device__ void emit_plan(const DepthArgs& a, int64_t unit, int t) {
  __shared__ ScanPlan<GP> P;
  __shared__ PlanScratch X;
  const int tid = threadIdx.x;
  float qv[GP];
  if (tid < kD) {
    const float* qp = a.q + unit * a.group * kD;
#pragma unroll
    for (int hh = 0; hh < GP; ++hh) qv[hh] = hh < a.group ? qp[hh * kD + tid] : 0.f;
  }
  scan_setup<GP>(P, X, t, qv, a.status);
  scan_store_plan<GP>(P, reinterpret_cast<ScanPlan<GP>*>(a.plan) + unit);
}

template <int GP>
__global__ void __launch_bounds__(kScanThreads) k_alloc_depths(DepthArgs a) {
  pdl_enter();
  __shared__ DepthSmem S;
  const int unit = blockIdx.x;
  const int s = unit / a.n_heads;
  if (a.tickets && threadIdx.x == 0) a.tickets[unit] = 0u;
  if (a.hist) zero_hist(a, unit);
  uint8_t* dep = a.depths + (int64_t)unit * kD;
  const int t = alloc_depths_cta(S, a.q + (int64_t)unit * a.group * kD, a.sigma2 + (int64_t)unit * kD, a.group,
                                 a.budget_q[s], dep);
  if (a.plan) emit_plan<GP>(a, unit, t);
}

template <int GP>
__global__ void __launch_bounds__(kScanThreads) k_fixed_depths(DepthArgs a) {
  pdl_enter();
  __shared__ DepthSmem S;
  const int unit = blockIdx.x;
  if (a.tickets && threadIdx.x == 0) a.tickets[unit] = 0u;
  if (a.hist) zero_hist(a, unit);
  uint8_t* dep = a.depths + (int64_t)unit * kD;
  const int t = fixed_depths_cta(S, a.q + (int64_t)unit * a.group * kD, a.group, a.n_channels, a.depth, dep);
  if (a.plan) emit_plan<GP>(a, unit, t);
}

template <typename F>
cudaError_t launch_depths_gp(int group, F&& launch) {
  if (group <= 1) return launch(std::integral_constant<int, 1>{});
  if (group <= 2) return launch(std::integral_constant<int, 2>{});
  if (group <= 4) return launch(std::integral_constant<int, 4>{});
  return launch(std::integral_constant<int, 8>{});
}

size_t scan_plan_bytes(int group) {
  if (group <= 1) return sizeof(ScanPlan<1>);
  if (group <= 2) return sizeof(ScanPlan<2>);
  if (group <= 4) return sizeof(ScanPlan<4>);
  return sizeof(ScanPlan<8>);
}

struct FrontArgs {
  DepthArgs d;
  int32_t depth_rule;       // BPKV_DEPTH_WATERFILL, BPKV_DEPTH_FIXED or BPKV_DEPTH_GIVEN
  const uint8_t* depths_in; // BPKV_DEPTH_GIVEN: [N][H][D] the caller's depths
  uint32_t* seq_tick;       // [N]: zeroed for the attention of this step
  uint32_t* hist1;          // optional [N][H][G][kTopkBins]: zeroed with the level-0 histograms
  // append
  uint64_t* planes;
  uint16_t* scales;
  uint16_t* k_rows;
  uint16_t* v_rows;
  const int64_t* seq_len;
  const uint16_t* k_new;
  const uint16_t* v_new;
  int32_t t_new;
  int32_t enc_ctas;         // append CTAs per unit: two (channel halves) per block the new tokens can touch
  int64_t cap;
  const float* basis;       // optional [H][D][D]: keys coded as k R, depths and plan from q R
  float* q_rot;             // with a basis: [N][H][G][D] workspace for q R
  uint64_t* vplanes;        // optional [N][H][cap][4][D/64]: the value rows' own code
  uint16_t* vscales;        // optional [N][H][cap]
};

// Grid (enc_ctas + 1, H, N), kScanThreads threads: x < enc_ctas appends, x ==
// enc_ctas allocates depths and emits the plan.
template <int GP>
__global__ void __launch_bounds__(kScanThreads) k_front(FrontArgs a) {
  pdl_enter();
  const int s = blockIdx.z, h = blockIdx.y, x = blockIdx.x;
  const int64_t unit = (int64_t)s * a.d.n_heads + h;
  const int G = a.d.group;
  if (x < a.enc_ctas) {
    // this CTA's slice of the unit's histograms and counters
    {
      const int n4 = G * kTopkBins / 4;
      uint4* hz = reinterpret_cast<uint4*>(a.d.hist + unit * G * kTopkBins);
      const int e0 = n4 * x / a.enc_ctas, e1 = n4 * (x + 1) / a.enc_ctas;
      for (int e = e0 + threadIdx.x; e < e1; e += blockDim.x) hz[e] = make_uint4(0u, 0u, 0u, 0u);
      if (a.hist1) {
        uint4* hz1 = reinterpret_cast<uint4*>(a.hist1 + unit * G * kTopkBins);
        for (int e = e0 + threadIdx.x; e < e1; e += blockDim.x) hz1[e] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (x == 0 && (int)threadIdx.x < kSelCounters * G) a.d.ctr[unit * kSelCounters * G + threadIdx.x] = 0u;
    }
    // CTA x: block n_old / 64 + x / 2, channels 64 (x % 2) ..
    const int64_t n_old = a.seq_len[s];
    const int64_t n_new = n_old + a.t_new;
    const int64_t blk = n_old / kBlock + x / 2;
    const int64_t t0 = blk * kBlock;
    if (t0 >= n_new || n_new > a.cap) return;
    const int cnt = (int)min64(kBlock, n_new - t0);
    const Unit U{a.cap / kBlock, a.cap};
    __shared__ __align__(16) uint16_t kb[kBlock][kD];
    encode_block_cta<4>(kb, a.k_rows + U.row_base(unit), a.v_rows + U.row_base(unit),
                        a.k_new + unit * a.t_new * kD, a.v_new + unit * a.t_new * kD, n_old, t0, cnt,
                        a.planes + U.plane_base(unit), a.scales + U.scale_base(unit), a.cap / kBlock, blk,
                        (x % 2) * (kD / 2), a.basis ? a.basis + (int64_t)h * kD * kD : nullptr);
    if (a.vplanes && x % 2 == 0)
      encode_value_rows(a.v_new + unit * a.t_new * kD, n_old, t0, cnt, a.vplanes + unit * a.cap * (kPlanes * kD / 64),
                        a.vscales + unit * a.cap, 0, kScanThreads / 32);
    return;
  }
  __shared__ DepthSmem S;
  if (threadIdx.x == 0) {
    a.d.tickets[unit] = 0u;
    if (h == 0) a.seq_tick[s] = 0u;
  }
  uint8_t* dep = a.d.depths + unit * kD;
  // with a basis the depths and the plan come from q R (float32 fused
  // multiply-add chains in channel order, one per output channel)
  DepthArgs d = a.d;
  if (a.basis) {
    const float* R = a.basis + (int64_t)h * kD * kD;
    const float* qs = a.d.q + unit * G * kD;
    float* qr = a.q_rot + unit * G * kD;
    if (threadIdx.x < kD) {
      const int l = threadIdx.x;
      for (int hh = 0; hh < G; ++hh) {
        float acc = 0.f;
        for (int i = 0; i < kD; ++i) acc = __fmaf_rn(qs[hh * kD + i], R[i * kD + l], acc);
        qr[hh * kD + l] = acc;
      }
    }
    __syncthreads();
    d.q = a.q_rot;
  }
  int t = 0;  // thread j < D: channel j's depth
  if (a.depth_rule == BPKV_DEPTH_WATERFILL) {
    t = alloc_depths_cta(S, d.q + unit * G * kD, a.d.sigma2 + unit * kD, G, a.d.budget_q[s], dep);
  } else if (a.depth_rule == BPKV_DEPTH_GIVEN) {
    if (threadIdx.x < kD) {
      t = min((int)a.depths_in[unit * kD + threadIdx.x], 4);
      dep[threadIdx.x] = (uint8_t)t;
    }
  } else {
    t = fixed_depths_cta(S, d.q + unit * G * kD, G, a.d.n_channels, a.d.depth, dep);
  }
  emit_plan<GP>(d, unit, t);
}

cudaError_t launch_front(const bpkv_cache& c, const uint16_t* k_new, const uint16_t* v_new, int32_t t_new,
                         const float* q, const float* sigma2, const int32_t* budget_q, int32_t depth_rule,
                         int32_t n_channels, int32_t depth, uint8_t* depths, void* plan, uint32_t* hist,
                         uint32_t* hist1, uint32_t* ctr, uint32_t* tickets, uint32_t* seq_tick, cudaStream_t st,
                         const uint8_t* depths_in, float* q_rot, int32_t* status) {
  FrontArgs a;
  a.d = DepthArgs{q, sigma2, budget_q, depths, c.n_kv_heads, c.group, tickets, plan, n_channels, depth, hist, ctr,
                  status};
  a.depth_rule = depth_rule;
  a.depths_in = depths_in;
  a.seq_tick = seq_tick;
  a.hist1 = hist1;
  a.planes = c.planes;
  a.scales = c.scales;
  a.k_rows = c.k_rows;
  a.v_rows = c.v_rows;
  a.seq_len = c.seq_len;
  a.k_new = k_new;
  a.v_new = v_new;
  a.t_new = t_new;
  a.enc_ctas = 2 * ((t_new + kBlock - 1) / kBlock + 1);
  a.cap = c.cap_tokens;
  a.basis = c.basis;
  a.q_rot = q_rot;
  a.vplanes = c.vplanes;
  a.vscales = c.vscales;
  const dim3 grid((unsigned)(a.enc_ctas + 1), (unsigned)c.n_kv_heads, (unsigned)c.n_seq);
  return launch_depths_gp(c.group, [&](auto gp) {
    return launch_pdl(k_front<decltype(gp)::value>, grid, dim3(kScanThreads), 0, st, a);
  });
}

cudaError_t launch_alloc_depths(const bpkv_cache& c, const float* q, const float* sigma2, const int32_t* budget_q,
                                uint8_t* depths, cudaStream_t st, uint32_t* tickets, void* plan, uint32_t* hist,
                                uint32_t* ctr) {
  DepthArgs a{q, sigma2, budget_q, depths, c.n_kv_heads, c.group, tickets, plan, 0, 0, hist, ctr, nullptr};
  return launch_depths_gp(c.group, [&](auto gp) {
    return launch_pdl(k_alloc_depths<decltype(gp)::value>, dim3(c.n_seq * c.n_kv_heads), dim3(kScanThreads), 0, st,
                      a);
  });
}

cudaError_t launch_fixed_depths(const bpkv_cache& c, const float* q, int32_t n_channels, int32_t depth,
                                uint8_t* depths, cudaStream_t st, uint32_t* tickets, void* plan, uint32_t* hist,
                                uint32_t* ctr) {
  DepthArgs a{q, nullptr, nullptr, depths, c.n_kv_heads, c.group, tickets, plan, n_channels, depth, hist, ctr,
              nullptr};
  return launch_depths_gp(c.group, [&](auto gp) {
    return launch_pdl(k_fixed_depths<decltype(gp)::value>, dim3(c.n_seq * c.n_kv_heads), dim3(kScanThreads), 0, st,
                      a);
  });
}

}  // namespace bpkv
