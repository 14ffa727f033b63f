// Value-side per-token read depth: the second read stage of ReadKV (the ReadKV
// page, section 5.3 "approximate attention decides value-token depth" and
// section 5.4, the allocator), over the exact key attention of the union rows.
//
// Value rows are coded with the keys' 4-bit mid-rise code, one fp16 scale per
// row (s_i = fp16(max_j |v_ij| / 8)), as token-major bit planes: word (i, p, w)
// bit b is bit (3 - p) of the code of channel 64 w + b, so the first t planes
// of a row are its t-bit quantiser and a row read to depth t costs t x 16
// bytes plus its scale.
//
// Stage 2 for one (sequence, KV head): each query head h attends over its own
// union rows with the exact bf16 keys, p_h(r) = softmax_r(q_h . k_r / sqrt(D));
// each row gets the weight a_r = sum_h p_h(r)^2; items (r, t), t = 0..3, with
// value a_r 4^-t are taken greedily (largest value first, ties to the lower
// row, then the lower t) up to the plane budget B_V, stopping at values <= 0;
// row r is read to depth t_r = its items taken, and o_h = sum_r p_h(r) vhat_r(t_r)
// with vhat = s ((c_t + 1/2) 2^(4-t) - 8) and vhat = 0 at t = 0.
//
// One cluster of kVdCluster CTAs per unit, rows dealt round-robin to the
// CTAs (row r to CTA r mod kVdCluster).  The softmax maxima and sums, the
// radix histograms and the output are reduced across the cluster through
// distributed shared memory at hardware cluster barriers.  The greedy order
// is one total order of 64-bit keys (value bits, then the complemented item
// index), so the taken items are exactly the B_V largest keys: a radix select
// over the key bits finds the B_V-th largest key and every item at or above
// it is taken.
#include "common.cuh"

#include <cooperative_groups.h>

namespace cg = cooperative_groups;

namespace bpkv {

// ---------------------------------------------------------------- stage 2

constexpr int kVdCluster = 8;                          // CTAs per unit (16 measured slower)
constexpr int kVdThreads = 512;
constexpr int kVdWarps = kVdThreads / 32;
constexpr int kVdMaxRows = 2048;                       // union rows of one unit (G k)
constexpr int kVdLocal = kVdMaxRows / kVdCluster;      // rows of one CTA
constexpr int kVdBatch = 4;       // rows a warp loads at once (the value phase: one row per 8 lanes)

struct VdArgs {
  const float* q;          // [N][H][G][D]
  const uint16_t* k_rows;  // [N][H][cap][D]
  const uint64_t* vplanes; // [N][H][cap][4][D/64]
  const uint16_t* vscales; // [N][H][cap]
  const int32_t* uidx;     // [N][H][u_cap]
  const uint8_t* umask;    // [N][H][u_cap]
  const int32_t* ucount;   // [N][H]
  int32_t u_cap;
  int32_t group;
  int32_t budget_v;        // planes per unit
  int64_t cap;
  float* out;              // [N][H][G][D]
  uint8_t* vdepth;         // optional [N][H][u_cap]
  float* weight;           // optional [N][H][u_cap]
};

template <int GP>
struct VdSmem {
  float p[GP][kVdLocal];     // this CTA's rows: logits, then probabilities
  float a[kVdLocal];         // a_r
  uint8_t dep[kVdLocal];
  float q[GP][kD];
  float o[GP][kD];           // this CTA's share of the output
  float red[kVdWarps][GP];
  float cmax[GP], csum[GP];  // this CTA's softmax maximum and sum per head
  uint32_t hist[256];        // this CTA's radix histogram
  uint32_t hsum[256];        // the cluster's
  unsigned long long prefix;
  uint32_t need;
  uint32_t done;             // 0: select on; 1: every positive item taken; 2: the bin at prefix taken whole
};

__device__ __forceinline__ float vd_warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float vd_warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Key of item (r, t): the value a_r 4^-t (a positive float orders like its
// bits), then the complemented item index 4 r + t (lower row, then lower t,
// first).  Items of value <= 0 get key 0 and are never taken.
__device__ __forceinline__ unsigned long long vd_key(float a, int r, int t) {
  const float v = ldexpf(a, -2 * t);
  if (!(v > 0.f)) return 0ull;
  return ((unsigned long long)__float_as_uint(v) << 32) | (0xFFFFFFFFu - (uint32_t)(4 * r + t));
}

template <int GP>
__global__ void __launch_bounds__(kVdThreads) k_attend_vdepth(VdArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char vd_raw[];
  VdSmem<GP>& S = *reinterpret_cast<VdSmem<GP>*>(vd_raw);
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t unit = blockIdx.x / kVdCluster;
  const int G = a.group;
  const int n_u = min(a.ucount[unit], min(a.u_cap, kVdMaxRows));
  const int n_loc = n_u > rank ? (n_u - rank + kVdCluster - 1) / kVdCluster : 0;  // rows rank + kVdCluster i
  auto row_of = [&](int i) { return rank + kVdCluster * i; };
  const int32_t* rows = a.uidx + unit * a.u_cap;
  const uint8_t* masks = a.umask + unit * a.u_cap;
  const uint16_t* kr = a.k_rows + unit * a.cap * kD;
  for (int e = tid; e < GP * kD; e += kVdThreads) {
    const int h = e / kD;
    S.q[h][e % kD] = h < G ? a.q[(unit * G + h) * kD + e % kD] : 0.f;
    S.o[h][e % kD] = 0.f;
  }
  __syncthreads();
  // logits q_h . k_r / sqrt(D) of the heads that selected row r (warp per row,
  // four channels per lane), -inf elsewhere; kVdBatch rows per warp at a
  // time, their loads issued together
  const float scale = rsqrtf((float)kD);
  for (int i0 = warp; i0 < n_loc; i0 += kVdWarps * kVdBatch) {
    uint2 kv[kVdBatch];
#pragma unroll
    for (int u = 0; u < kVdBatch; ++u) {
      const int i = min(i0 + u * kVdWarps, n_loc - 1);
      kv[u] = *reinterpret_cast<const uint2*>(kr + (int64_t)rows[row_of(i)] * kD + 4 * lane);
    }
#pragma unroll
    for (int u = 0; u < kVdBatch; ++u) {
      const int i = i0 + u * kVdWarps;
      if (i >= n_loc) break;  // uniform across the warp
      const float k0 = __uint_as_float(kv[u].x << 16), k1 = __uint_as_float(kv[u].x & 0xFFFF0000u);
      const float k2 = __uint_as_float(kv[u].y << 16), k3 = __uint_as_float(kv[u].y & 0xFFFF0000u);
      const uint32_t m = masks[row_of(i)];
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float* qh = S.q[h] + 4 * lane;
        float d = qh[0] * k0;
        d = fmaf(qh[1], k1, d);
        d = fmaf(qh[2], k2, d);
        d = fmaf(qh[3], k3, d);
        d = vd_warp_sum(d);
        if (lane == 0) S.p[h][i] = (h < G && ((m >> h) & 1)) ? d * scale : -INFINITY;
      }
    }
  }
  __syncthreads();
  // softmax per head over the whole unit: the cluster's maximum, exponentials,
  // the cluster's sum, probabilities
  float mx[GP], z[GP];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    float v = -INFINITY;
    for (int i = tid; i < n_loc; i += kVdThreads) v = fmaxf(v, S.p[h][i]);
    v = vd_warp_max(v);
    if (lane == 0) S.red[warp][h] = v;
  }
  __syncthreads();
  if (tid < GP) {
    float v = -INFINITY;
    for (int w = 0; w < kVdWarps; ++w) v = fmaxf(v, S.red[w][tid]);
    S.cmax[tid] = v;
  }
  cl.sync();
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    mx[h] = -INFINITY;
    for (int c = 0; c < kVdCluster; ++c) mx[h] = fmaxf(mx[h], cl.map_shared_rank(S.cmax, c)[h]);
  }
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    float v = 0.f;
    for (int i = tid; i < n_loc; i += kVdThreads) {
      const float l = S.p[h][i];
      const float e = l == -INFINITY ? 0.f : __expf(l - mx[h]);
      S.p[h][i] = e;
      v += e;
    }
    v = vd_warp_sum(v);
    if (lane == 0) S.red[warp][h] = v;
  }
  __syncthreads();
  if (tid < GP) {
    float v = 0.f;
    for (int w = 0; w < kVdWarps; ++w) v += S.red[w][tid];
    S.csum[tid] = v;
  }
  cl.sync();
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    z[h] = 0.f;
    for (int c = 0; c < kVdCluster; ++c) z[h] += cl.map_shared_rank(S.csum, c)[h];
  }
  // probabilities and row weights a_r = sum_h p_h(r)^2 (heads in order)
  for (int i = tid; i < n_loc; i += kVdThreads) {
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      const float pr = z[h] > 0.f ? S.p[h][i] / z[h] : 0.f;
      S.p[h][i] = pr;
      acc = fmaf(pr, pr, acc);
    }
    S.a[i] = acc;
  }
  if (tid == 0) {
    S.prefix = 0ull;
    S.need = (uint32_t)max(a.budget_v, 0);
    S.done = 0u;
  }
  __syncthreads();
  // radix select, eight bits at a time from the top, of the need-th largest
  // key among the unit's 4 n_u items (the last one taken), each CTA counting
  // its rows' items and every CTA reading the cluster's sum.  It stops early
  // when the bin holding that key is taken whole (the cut is then the bin's
  // lowest key); with fewer positive items than the budget every positive
  // item is taken (the cut falls to key 1).  Every CTA takes the same
  // decisions.
  unsigned long long cut = ~0ull;
  if (S.need > 0) {
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int e = tid; e < 256; e += kVdThreads) S.hist[e] = 0u;
      __syncthreads();
      const unsigned long long pre = S.prefix;
      const unsigned long long hi_mask = shift == 56 ? 0ull : (~0ull << (shift + 8));
      for (int it = tid; it < 4 * n_loc; it += kVdThreads) {
        const unsigned long long k = vd_key(S.a[it >> 2], row_of(it >> 2), it & 3);
        if (k != 0ull && (k & hi_mask) == pre) atomicAdd(&S.hist[(k >> shift) & 0xFF], 1u);
      }
      cl.sync();  // every CTA's histogram is complete
      for (int e = tid; e < 256; e += kVdThreads) {
        uint32_t hv[kVdCluster];
#pragma unroll
        for (int c = 0; c < kVdCluster; ++c) hv[c] = cl.map_shared_rank(S.hist, c)[e];
        uint32_t v = 0u;
#pragma unroll
        for (int c = 0; c < kVdCluster; ++c) v += hv[c];
        S.hsum[e] = v;
      }
      __syncthreads();
      if (warp == 0) {
        // bins from the top: the bin holding the need-th largest key
        uint32_t need = S.need, acc = 0;
        int sel = -1;
        for (int base = 224; base >= 0 && sel < 0; base -= 32) {
          const uint32_t c = S.hsum[base + lane];
          // inclusive sum from the top of this 32-bin slice (lane 31 highest)
          uint32_t incl = c;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
            if (lane + o < 32) incl += y;
          }
          const bool hit = acc + incl >= need && acc + incl - c < need;
          const uint32_t hb = __ballot_sync(0xffffffffu, hit);
          if (hb) {
            const int l = 31 - __clz(hb);  // the one lane where the running count crosses need
            const uint32_t before = __shfl_sync(0xffffffffu, acc + incl - c, l);
            sel = base + l;
            need -= before;
          } else {
            acc += __shfl_sync(0xffffffffu, incl, 0);
          }
        }
        if (lane == 0) {
          if (sel < 0) {
            S.done = 1u;  // fewer positive items than the budget
          } else {
            S.prefix = pre | ((unsigned long long)sel << shift);
            S.need = need;
            if (S.hsum[sel] == need) S.done = 2u;  // the bin is taken whole
          }
        }
      }
      cl.sync();  // every CTA has read the histograms (before they are cleared) and has its decision
      if (S.done != 0u) break;
    }
    cut = S.done == 1u ? 1ull : S.prefix;
  }
  __syncthreads();
  // depth of each row: its items at or above the cut
  for (int i = tid; i < n_loc; i += kVdThreads) {
    const int r = row_of(i);
    int t = 0;
    if (a.budget_v > 0) {
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) t += vd_key(S.a[i], r, tt) >= cut ? 1 : 0;
    }
    S.dep[i] = (uint8_t)t;
    if (a.vdepth) a.vdepth[unit * a.u_cap + r] = (uint8_t)t;
    if (a.weight) a.weight[unit * a.u_cap + r] = S.a[i];
  }
  __syncthreads();
  // o_h = sum_r p_h(r) vhat_r(t_r) over this CTA's rows: warp per row, lane
  // channels l, l + 32, l + 64, l + 96 (word 0 bits l and l + 32, word 1 bits
  // l and l + 32)
  float acc[GP][4];
#pragma unroll
  for (int h = 0; h < GP; ++h)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[h][i] = 0.f;
  const uint64_t* vpu = a.vplanes + unit * a.cap * (kPlanes * kD / 64);
  const uint16_t* vsu = a.vscales + unit * a.cap;
  // kVdBatch rows per warp at a time: each lane loads one of the rows' plane
  // words (row u: words 2 p + w at lanes 8 u + 2 p + w) and their scales, the
  // warp shares them by shuffles
  for (int i0 = warp; i0 < n_loc; i0 += kVdWarps * kVdBatch) {
    uint64_t wl = 0ull;
    uint16_t sl = 0;
    {
      const int u = lane >> 3, i = i0 + u * kVdWarps;
      if (u < kVdBatch && i < n_loc && (lane & 7) < 2 * S.dep[i]) {
        const int64_t tok = rows[row_of(i)];
        wl = vpu[tok * (kPlanes * kD / 64) + (lane & 7)];
        if ((lane & 7) == 0) sl = vsu[tok];
      }
    }
#pragma unroll
    for (int u = 0; u < kVdBatch; ++u) {
      const int i = i0 + u * kVdWarps;
      if (i >= n_loc) break;  // uniform across the warp
      const int t = S.dep[i];
      if (t == 0) continue;
      const float s = fp16_bits_to_float((uint16_t)__shfl_sync(0xffffffffu, (uint32_t)sl, 8 * u));
      uint32_t c[4] = {0u, 0u, 0u, 0u};
      for (int pl = 0; pl < t; ++pl) {
        const uint64_t w0 = __shfl_sync(0xffffffffu, wl, 8 * u + 2 * pl);
        const uint64_t w1 = __shfl_sync(0xffffffffu, wl, 8 * u + 2 * pl + 1);
        c[0] = (c[0] << 1) | (uint32_t)((w0 >> lane) & 1u);
        c[1] = (c[1] << 1) | (uint32_t)((w0 >> (lane + 32)) & 1u);
        c[2] = (c[2] << 1) | (uint32_t)((w1 >> lane) & 1u);
        c[3] = (c[3] << 1) | (uint32_t)((w1 >> (lane + 32)) & 1u);
      }
      const float step = ldexpf(s, 4 - t);  // s 2^(4 - t)
      float vh[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) vh[k] = fmaf((float)c[k] + 0.5f, step, -8.f * s);
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float pr = S.p[h][i];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[h][k] = fmaf(pr, vh[k], acc[h][k]);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < GP; ++h)
#pragma unroll
    for (int k = 0; k < 4; ++k) atomicAdd(&S.o[h][lane + 32 * k], acc[h][k]);
  cl.sync();  // every CTA's share of the output is complete
  // CTA rank adds the cluster's shares of its slice of the G D outputs (CTAs in rank order)
  for (int e = rank * kVdThreads + tid; e < G * kD; e += kVdCluster * kVdThreads) {
    float v = 0.f;
    for (int c = 0; c < kVdCluster; ++c) v += cl.map_shared_rank(&S.o[0][0], c)[e];
    a.out[unit * G * kD + e] = v;
  }
  cl.sync();  // no CTA leaves while another still reads its shared memory
}

size_t vdepth_smem(int group) {
  if (group <= 1) return sizeof(VdSmem<1>);
  if (group <= 2) return sizeof(VdSmem<2>);
  if (group <= 4) return sizeof(VdSmem<4>);
  return sizeof(VdSmem<8>);
}

template <int GP>
cudaError_t launch_vdepth_gp(const VdArgs& a, unsigned units, cudaStream_t st) {
  const int smem = (int)sizeof(VdSmem<GP>);
  cudaError_t e = cudaFuncSetAttribute(k_attend_vdepth<GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (kVdCluster > 8) {
    e = cudaFuncSetAttribute(k_attend_vdepth<GP>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units * kVdCluster);
  cfg.blockDim = dim3(kVdThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kVdCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_attend_vdepth<GP>, a);
}

cudaError_t launch_attend_vdepth(const bpkv_cache& c, const float* q, const int32_t* uidx, const uint8_t* umask,
                                 const int32_t* ucount, int32_t u_cap, int32_t budget_v, float* out,
                                 uint8_t* vdepth, float* weight, cudaStream_t st) {
  VdArgs a{q, c.k_rows, c.vplanes, c.vscales, uidx, umask, ucount, u_cap, c.group, budget_v, c.cap_tokens,
           out, vdepth, weight};
  const unsigned units = (unsigned)(c.n_seq * c.n_kv_heads);
  if (c.group <= 1) return launch_vdepth_gp<1>(a, units, st);
  if (c.group <= 2) return launch_vdepth_gp<2>(a, units, st);
  if (c.group <= 4) return launch_vdepth_gp<4>(a, units, st);
  return launch_vdepth_gp<8>(a, units, st);
}

}  // namespace bpkv
