// Prefix-plane key scan (Fathom page, section 1 observation 2 and section 3.1):
// each key is scored from only the first t_j planes of each channel j and the
// block scales of the channels with t_j > 0; the bytes read are b n / 8.
//
//   khat = s ((c_t + 1/2) 2^(4-t) - 8) = s 2^(4-t) e,   e = c_t - 2^(t-1) + 1/2,
//   score_g = sum_j u_gj e_j   with u_gj = s_j (q_gj 2^(4-t_j))  (one rounding),
// e an exact half-integer, accumulated in float32 with fused multiply-adds.
//
// Work layout.  A CTA per (run of chunks of 8 blocks = 512 tokens, KV head,
// sequence), the run as long as needed for the grid to fit in one wave of
// resident CTAs; the unit's plan is loaded once per CTA.  The active channels are packed into "groups" of 32 plane rows,
// one depth per group (8 channels of depth 4, 10 of depth 3, 16 of depth 2,
// 32 of depth 1), the planes of a channel placed so that, after a 32 x 32 bit
// transpose, each token's code of each channel is a contiguous bit field with
// its most significant bit highest.  The chunk's plane words are staged in
// shared memory with coalesced loads; each warp takes one 64-token block, each
// lane two tokens (i and i + 32).  Per group a lane reads one 32-bit word per
// token half, the warp transposes them with five shuffle / funnel-shift /
// select rounds, and every field becomes a float by OR-ing it under the
// exponent of 2^23 and subtracting a constant (exact).  The products with u
// (staged per block and channel) use packed fp32x2 FMAs over field pairs.
#include "scan_core.cuh"

#include <mutex>
#include <type_traits>

namespace bpkv {

struct ScanArgs {
  const void* plan;          // optional per-unit ScanPlan<GP> built by the depth kernel
  const uint64_t* planes;
  const uint16_t* scales;
  const int64_t* seq_len;
  const float* q;
  const uint8_t* depths;
  float* scores;
  int64_t ld;
  int64_t nb_cap;
  int32_t n_heads;
  int32_t group;
  uint32_t* hist;  // optional [N][H][G][kTopkBins] level-0 selection histogram (zeroed by the caller)
  int32_t n_sink, n_recent;
  int64_t chunks_per_cta;
  int32_t pending;  // tokens appended in this step but not yet in seq_len
  int32_t* status;  // optional device status word (unused by the scan kernels today)
  int64_t chunks;   // chunks per unit (from the host bound on the sequence lengths)
  int64_t units;    // sequences x KV heads
};

template <int GP>
__global__ void __launch_bounds__(kScanThreads, GP >= 8 ? 2 : 4) k_scan(ScanArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ScanSmem<GP>& S = *reinterpret_cast<ScanSmem<GP>*>(smem_raw);
  const int s = blockIdx.z, h = blockIdx.y;
  const int64_t unit = (int64_t)s * a.n_heads + h;
  const int64_t n = a.seq_len[s] + a.pending;
  const int64_t c_begin = (int64_t)blockIdx.x * a.chunks_per_cta;
  if (c_begin * kScanBlocks * kBlock >= n) return;
  const int64_t nb_valid = (n + kBlock - 1) / kBlock;
  const int64_t c_end = min64(c_begin + a.chunks_per_cta, (nb_valid + kScanBlocks - 1) / kScanBlocks);
  const int tid = threadIdx.x;
  const int G = a.group;
  if (a.plan) {
    scan_load_plan<GP>(S.P, reinterpret_cast<const ScanPlan<GP>*>(a.plan) + unit);
  } else {
    int t = 0;
    float qv[GP];
    if (tid < kD) {
      t = min((int)a.depths[unit * kD + tid], 4);  // depth values above 4 read as 4
      const float* qp = a.q + unit * G * kD;
#pragma unroll
      for (int hh = 0; hh < GP; ++hh) qv[hh] = hh < G ? qp[hh * kD + tid] : 0.f;
    }
    scan_setup<GP>(S.P, S.X, t, qv);
  }
  const int64_t lo = min64(a.n_sink, n), hi = max64(n - a.n_recent, lo);
  for (int64_t ch = c_begin; ch < c_end; ++ch) {
    const int64_t b0 = ch * kScanBlocks;
    const int nbl = (int)min64(kScanBlocks, nb_valid - b0);
    float v0[GP], v1[GP];
    const bool act = scan_chunk<GP>(S, a.planes + unit * kD * kPlanes * a.nb_cap + b0,
                                    a.scales + unit * kD * a.nb_cap + b0, a.nb_cap, nbl, G,
                                    a.scores + unit * G * a.ld + b0 * kBlock, a.ld, n - b0 * kBlock, v0, v1);
    if (a.hist && act)
      warp_hist<GP>(G, b0 * kBlock + (threadIdx.x >> 5) * kBlock + (threadIdx.x & 31), lo, hi, v0, v1,
                    a.hist + unit * G * kTopkBins);
  }
}

// Device-resident caches.  The grid is one wave of CTAs over the units'
// chunks laid end to end (unit-major); each CTA takes an equal share of that
// sequence and scores it unit by unit.  Within a unit the steps (chunk, pass)
// go through two stage buffers: once step i has landed and every warp is past
// step i - 1, all threads start the copies of step i + 1 into the other
// buffer, then each warp forms u = s w for its block and scores step i.
template <int GP>
__device__ __forceinline__ void scan_unit_pipe(const ScanArgs& a, PipeSmem<GP>& S, int64_t unit, int64_t c_begin,
                                               int64_t c_want) {
  const int s = (int)(unit / a.n_heads);
  const int64_t n = min64(a.seq_len[s] + a.pending, a.nb_cap * kBlock);
  const int64_t nb_valid = (n + kBlock - 1) / kBlock;
  const int64_t c_end = min64(c_want, (nb_valid + kScanBlocks - 1) / kScanBlocks);
  if (c_begin >= c_end) return;
  const int tid = threadIdx.x, lane = tid & 31, lb = tid >> 5;
  const int G = a.group;
  __syncthreads();  // every warp is done with the previous unit's plan and stage buffers
  if (a.plan) {
    scan_load_plan<GP>(S.P, reinterpret_cast<const ScanPlan<GP>*>(a.plan) + unit);
  } else {
    int t = 0;
    float qv[GP];
    if (tid < kD) {
      t = min((int)a.depths[unit * kD + tid], 4);  // depth values above 4 read as 4
      const float* qp = a.q + unit * G * kD;
#pragma unroll
      for (int hh = 0; hh < GP; ++hh) qv[hh] = hh < G ? qp[hh * kD + tid] : 0.f;
    }
    scan_setup<GP>(S.P, S.X, t, qv);
  }
  const uint64_t* pl = a.planes + unit * kD * kPlanes * a.nb_cap;
  const uint16_t* sp = a.scales + unit * kD * a.nb_cap;
  float* out = a.scores + unit * G * a.ld;
  uint32_t* hist = a.hist ? a.hist + unit * G * kTopkBins : nullptr;
  const int64_t lo = min64(a.n_sink, n), hi = max64(n - a.n_recent, lo);
  const int n_passes = S.P.n_passes;
  const int64_t steps = (c_end - c_begin) * n_passes;
  constexpr bool kSmemHist = pipe_counts_hist<GP>();
  if constexpr (kSmemHist) {
    if (hist) {
      for (int e = tid; e < G * kTopkBins / 2; e += kScanThreads) S.hist[e] = 0u;
      __syncthreads();
    }
  }
  Acc<GP> A;
  acc_zero<GP>(A);
  uint32_t keep[5], rot[5];
  transpose_consts(lane, keep, rot);
  // scores of chunk ch from the accumulators (zeros when no channel is read)
  auto finish_chunk = [&](int64_t ch) {
    const int64_t b0 = ch * kScanBlocks;
    const int nbl = (int)min64(kScanBlocks, nb_valid - b0);
    if (lb < nbl) {
      const int64_t x0 = b0 * kBlock + (int64_t)lb * kBlock + lane;
      float v0[GP], v1[GP];
#pragma unroll
      for (int hh = 0; hh < GP; ++hh) {
        acc_scores<GP>(A, hh, v0[hh], v1[hh]);
        if (hh < G) {
          if (x0 < n) out[hh * a.ld + x0] = v0[hh];
          if (x0 + 32 < n) out[hh * a.ld + x0 + 32] = v1[hh];
          if constexpr (kSmemHist) {
            if (hist) {
              uint32_t* H = S.hist + hh * (kTopkBins / 2);
              if (x0 >= lo && x0 < hi) {
                const uint32_t bin = ordered_key(v0[hh]) >> 20;
                atomicAdd(H + (bin >> 1), 1u << ((bin & 1u) * 16));
              }
              if (x0 + 32 >= lo && x0 + 32 < hi) {
                const uint32_t bin = ordered_key(v1[hh]) >> 20;
                atomicAdd(H + (bin >> 1), 1u << ((bin & 1u) * 16));
              }
            }
          }
        }
      }
      if constexpr (!kSmemHist) {
        if (hist) warp_hist<GP>(G, x0, lo, hi, v0, v1, hist);
      }
    }
    acc_zero<GP>(A);
  };
  // the unit's shared-memory histograms added to its global ones
  auto flush_hist = [&]() {
    if constexpr (kSmemHist) {
      if (hist) {
        __syncthreads();
        for (int e = tid; e < G * kTopkBins / 2; e += kScanThreads) {
          const uint32_t v = S.hist[e];
          if (v == 0u) continue;
          uint32_t* g = hist + (e / (kTopkBins / 2)) * kTopkBins + 2 * (e % (kTopkBins / 2));
          if (v & 0xFFFFu) atomicAdd(g, v & 0xFFFFu);
          if (v >> 16) atomicAdd(g + 1, v >> 16);
        }
      }
    }
  };
  if (steps == 0) {
    for (int64_t ch = c_begin; ch < c_end; ++ch) finish_chunk(ch);
    flush_hist();
    return;
  }
  scan_issue<GP>(S, 0, pl, sp, a.nb_cap, c_begin * kScanBlocks, S.P.pass_g[0], S.P.pass_g[1]);
  int64_t ch = c_begin;  // chunk and pass of step i
  int ps = 0;
  for (int64_t i = 0; i < steps; ++i) {
    const int b = (int)(i & 1);
    cp_async_wait_all();
    __syncthreads();  // step i visible to all; every warp is done with step i - 1 (the other buffer)
    if (i + 1 < steps) {
      const int ps1 = ps + 1 == n_passes ? 0 : ps + 1;
      const int64_t ch1 = ps1 == 0 ? ch + 1 : ch;
      scan_issue<GP>(S, b ^ 1, pl, sp, a.nb_cap, ch1 * kScanBlocks, S.P.pass_g[ps1], S.P.pass_g[ps1 + 1]);
    }
    const int g0 = S.P.pass_g[ps], g1 = S.P.pass_g[ps + 1];
    const int s0 = S.P.grp_base[g0], s1 = g1 < S.P.n_groups ? (int)S.P.grp_base[g1] : S.P.n_slots;
    scan_form_u<GP>(S, b, s0, s1, lb);
    __syncwarp();
    const int nbl = (int)min64(kScanBlocks, nb_valid - ch * kScanBlocks);
    if (lb < nbl) scan_compute_pipe<GP>(S, b, g0, g1, s0, lb, keep, rot, A);
    if (++ps == n_passes) {
      finish_chunk(ch);
      ps = 0;
      ++ch;
    }
  }
  flush_hist();
}

template <int GP>
__global__ void __launch_bounds__(kScanThreads, 2) k_scan_pipe(ScanArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  PipeSmem<GP>& S = *reinterpret_cast<PipeSmem<GP>*>(smem_raw);
  // an equal share of all units' chunks laid end to end, unit by unit
  const int64_t total = a.units * a.chunks;
  const int64_t f1 = total * (blockIdx.x + 1) / gridDim.x;
  for (int64_t f = total * blockIdx.x / gridDim.x; f < f1;) {
    const int64_t unit = f / a.chunks, c0 = f % a.chunks;
    const int64_t c1 = min64(a.chunks, c0 + (f1 - f));
    scan_unit_pipe<GP>(a, S, unit, c0, c1);
    f += c1 - c0;
  }
}

template <int GP, bool Pipe>
cudaError_t launch_scan_gp(ScanArgs a, int64_t chunks, int64_t units, cudaStream_t st) {
  int smem = 0;
  if constexpr (Pipe) smem = (int)sizeof(PipeSmem<GP>);
  else smem = (int)sizeof(ScanSmem<GP>);
  void (*kernel)(ScanArgs) = nullptr;
  if constexpr (Pipe) kernel = k_scan_pipe<GP>;
  else kernel = k_scan<GP>;
  // resident CTAs per device, looked up once per device
  constexpr int kDevs = 64;
  static int slots[kDevs] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kDevs) return cudaErrorInvalidDevice;
  int occ_slots = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (slots[dev] == 0) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      int sms = 0, per_sm = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kScanThreads, smem);
      if (e != cudaSuccess) return e;
      slots[dev] = sms * (per_sm > 0 ? per_sm : 1);
    }
    occ_slots = slots[dev];
  }
  const int64_t total = chunks * units;
  a.chunks = chunks;
  a.units = units;
  if constexpr (Pipe) {
    // one wave; each CTA an equal share of the work (see k_scan_pipe)
    const unsigned ctas = (unsigned)min64(total, (int64_t)occ_slots);
    return launch_pdl(kernel, dim3(ctas), dim3(kScanThreads), (size_t)smem, st, a);
  }
  // enough chunks per CTA for the grid to fit in one wave of resident CTAs
  a.chunks_per_cta = (total + occ_slots - 1) / occ_slots;
  if (a.chunks_per_cta < 1) a.chunks_per_cta = 1;
  const dim3 grid((unsigned)((chunks + a.chunks_per_cta - 1) / a.chunks_per_cta), (unsigned)a.n_heads,
                  (unsigned)(units / a.n_heads));
  return launch_pdl(kernel, grid, dim3(kScanThreads), (size_t)smem, st, a);
}

// Device-resident caches take the pipelined kernel (asynchronous copies into
// shared memory); pinned host caches the direct one (plain loads over the link).
cudaError_t launch_scan(const bpkv_cache& c, const float* q, const uint8_t* depths, float* scores, int64_t ld,
                        cudaStream_t st, const void* plan, uint32_t* hist, int32_t n_sink, int32_t n_recent,
                        int32_t pending, int32_t* status) {
  ScanArgs a{plan,         c.planes, c.scales, c.seq_len, q,        depths, scores,  ld,    c.cap_tokens / kBlock,
             c.n_kv_heads, c.group,  hist,     n_sink,    n_recent, 1,      pending, status, 0, 0};
  const int64_t chunks = (c.n_max + kScanBlocks * kBlock - 1) / (kScanBlocks * kBlock);
  if (chunks == 0) return cudaSuccess;
  const int64_t units = (int64_t)c.n_seq * c.n_kv_heads;
  const bool pipe = c.residency == 0;
  auto go = [&](auto gp) {
    constexpr int GP = decltype(gp)::value;
    return pipe ? launch_scan_gp<GP, true>(a, chunks, units, st) : launch_scan_gp<GP, false>(a, chunks, units, st);
  };
  if (c.group <= 1) return go(std::integral_constant<int, 1>{});
  if (c.group <= 2) return go(std::integral_constant<int, 2>{});
  if (c.group <= 4) return go(std::integral_constant<int, 4>{});
  return go(std::integral_constant<int, 8>{});
}

}  // namespace bpkv
