// Prefix-plane key scan (Fathom page, section 1 observation 2 and section 3.1):
// each key is scored from only the first t_j planes of each channel j and the
// block scales of the channels with t_j > 0; the bytes read are b n / 8.
//
//   khat = s ((c_t + 1/2) 2^(4-t) - 8) = s 2^(4-t) e,   e = c_t - 2^(t-1) + 1/2,
//   score_g = sum_j u_gj e_j   with u_gj = s_j (q_gj 2^(4-t_j))  (one rounding),
// e an exact half-integer, accumulated in float32 with fused multiply-adds.
//
// Work layout.  Chunks are runs of 8 blocks (512 tokens) of one unit
// (sequence, KV head).  One wave of resident CTAs splits all units' chunks,
// laid end to end, into equal shares; a CTA loads the plan of each unit it
// meets.  The active channels are packed into "groups" of 32 plane rows,
// one depth per group (8 channels of depth 4, 10 of depth 3, 16 of depth 2,
// 32 of depth 1), the planes of a channel placed so that, after a 32 x 32 bit
// transpose, each token's code of each channel is a contiguous bit field with
// its most significant bit highest.  The plane words and block scales of each
// step are staged in shared memory by asynchronous copies, double-buffered;
// each warp takes one 64-token block, each lane two tokens (i and i + 32).
// Per group a lane reads one 32-bit word per token half, the warp transposes
// them with five shuffle / funnel-shift / select rounds, and every field
// becomes a float by OR-ing it under the exponent of 2^23 and subtracting a
// constant (exact).  The products with u = s w (formed per block and slot)
// use packed fp32x2 FMAs over head pairs.
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
  int32_t pending;  // tokens appended in this step but not yet in seq_len
  int32_t* status;  // optional device status word (bounds-checked builds record in it)
  int64_t chunks;   // chunks per unit (from the host bound on the sequence lengths)
  int64_t units;    // sequences x KV heads
};

// Device-resident caches.  The grid is one wave of CTAs over the units'
// chunks laid end to end (unit-major); each CTA takes an equal share of that
// sequence and scores it unit by unit.  Within a unit the steps (one pass
// over one chunk, or over kWideSub chunks when the unit's plan allows) go
// through two stage buffers: once step i has landed and every warp is past
// step i - 1, all threads start the copies of step i + 1 into the other
// buffer, then each warp forms u = s w for its block of each chunk of the step
// and scores it.  kHost: the caches are in pinned host memory (wide steps
// allowed, sector-coalesced copies).
template <int GP, bool kHost>
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
    scan_setup<GP>(S.P, S.X, t, qv, a.status);
  }
  const uint64_t* pl = a.planes + unit * kD * kPlanes * a.nb_cap;
  const uint16_t* sp = a.scales + unit * kD * a.nb_cap;
  float* out = a.scores + unit * G * a.ld;
  uint32_t* hist = a.hist ? a.hist + unit * G * kTopkBins : nullptr;
  const int64_t lo = min64(a.n_sink, n), hi = max64(n - a.n_recent, lo);
  const int n_passes = S.P.n_passes;
  // chunks per step: kWideSub for host caches whose plan is one pass that
  // fits a wide step; wide steps start at even chunks (the first one may hold
  // one chunk).  Device memory gains nothing from them (the L2 serves the
  // second half of a scale sector).
  const int sub = (kHost && n_passes == 1 && S.P.n_groups <= kWideGroups) ? kWideSub : 1;
  auto span = [&](int64_t c) -> int {
    return sub == 1 ? 1 : (int)min64((c & 1) ? 1 : kWideSub, c_end - c);
  };
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
  // scores of chunk ch from the accumulators (zeros when no channel is read);
  // positions relative to the chunk in 32-bit arithmetic (a chunk is 512 tokens)
  auto finish_chunk = [&](int64_t ch) {
    const int64_t t0 = ch * (kScanBlocks * kBlock);
    const int r0 = lb * kBlock + lane;  // this lane's first token within the chunk
    const int lim = (int)min64(n - t0, kScanBlocks * kBlock);
    if (lb * kBlock < lim) {  // whole warps (warp_hist needs them)
      const int lo_r = (int)max64(min64(lo - t0, kScanBlocks * kBlock), -1);
      const int hi_r = (int)max64(min64(hi - t0, kScanBlocks * kBlock), -1);
      const bool w0 = r0 < lim, w1 = r0 + 32 < lim;
      const bool in0 = r0 >= lo_r && r0 < hi_r, in1 = r0 + 32 >= lo_r && r0 + 32 < hi_r;
      float* o = out + t0 + r0;
      float v0[GP], v1[GP];
#pragma unroll
      for (int hh = 0; hh < GP; ++hh) {
        acc_scores<GP>(A, hh, v0[hh], v1[hh]);
        if (hh < G) {
          if (w0) o[hh * a.ld] = v0[hh];
          if (w1) o[hh * a.ld + 32] = v1[hh];
          if constexpr (kSmemHist) {
            if (hist) {
              // the order-preserving key straight from the bits (-0 made +0
              // first): bin = key >> 20 counts in word bin / 2 = key >> 21,
              // half (bin & 1) = key bit 20
              uint32_t* H = S.hist + hh * (kTopkBins / 2);
              if (in0) {
                const uint32_t u = __float_as_uint(__fadd_rn(v0[hh], 0.f));
                const uint32_t key = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
                atomicAdd(H + (key >> 21), 1u << ((key >> 16) & 16u));
              }
              if (in1) {
                const uint32_t u = __float_as_uint(__fadd_rn(v1[hh], 0.f));
                const uint32_t key = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
                atomicAdd(H + (key >> 21), 1u << ((key >> 16) & 16u));
              }
            }
          }
        }
      }
      if constexpr (!kSmemHist) {
        if (hist) warp_hist<GP>(G, t0 + r0, lo, hi, v0, v1, hist);
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
  if (n_passes == 0) {
    for (int64_t ch = c_begin; ch < c_end; ++ch) finish_chunk(ch);
    flush_hist();
    return;
  }
  if constexpr (!kHost) {
    // device caches: steps (chunk, pass), one chunk each
    const int64_t steps = (c_end - c_begin) * n_passes;
    scan_issue<GP>(S, 0, pl, sp, a.nb_cap, c_begin * kScanBlocks, S.P.pass_g[0], S.P.pass_g[1], 1, 1, false, a.status);
    int64_t ch = c_begin;  // chunk and pass of step i
    int ps = 0;
    for (int64_t i = 0; i < steps; ++i) {
      const int b = (int)(i & 1);
      cp_async_wait_all();
      __syncthreads();  // step i visible to all; every warp is done with step i - 1 (the other buffer)
      if (i + 1 < steps) {
        const int ps1 = ps + 1 == n_passes ? 0 : ps + 1;
        const int64_t ch1 = ps1 == 0 ? ch + 1 : ch;
        scan_issue<GP>(S, b ^ 1, pl, sp, a.nb_cap, ch1 * kScanBlocks, S.P.pass_g[ps1], S.P.pass_g[ps1 + 1], 1, 1,
                       false, a.status);
      }
      const int g0 = S.P.pass_g[ps], g1 = S.P.pass_g[ps + 1];
      const int s0 = S.P.grp_base[g0], s1 = g1 < S.P.n_groups ? (int)S.P.grp_base[g1] : S.P.n_slots;
      scan_form_u<GP>(S, b, s0, s1, lb, 1, 0, false, a.status);
      __syncwarp();
      const int nbl = (int)min64(kScanBlocks, nb_valid - ch * kScanBlocks);
      if (lb < nbl) scan_compute_pipe<GP>(S, b, g0, g1, s0, lb, 1, 0, false, keep, rot, A, a.status);
      if (++ps == n_passes) {
        finish_chunk(ch);
        ps = 0;
        ++ch;
      }
    }
  } else {
    // host caches: step i covers chunks [ch, ch + n_sub), pass ps
    int64_t ch = c_begin;
    int ps = 0, n_sub = span(c_begin);
    scan_issue<GP>(S, 0, pl, sp, a.nb_cap, ch * kScanBlocks, S.P.pass_g[0], S.P.pass_g[1], sub, n_sub, true, a.status);
    for (int64_t i = 0;; ++i) {
      const int b = (int)(i & 1);
      cp_async_wait_all();
      __syncthreads();  // step i visible to all; every warp is done with step i - 1 (the other buffer)
      const int ps1 = ps + 1 == n_passes ? 0 : ps + 1;
      const int64_t ch1 = ps1 == 0 ? ch + n_sub : ch;
      const int n_sub1 = ch1 < c_end ? span(ch1) : 0;
      if (n_sub1 > 0)
        scan_issue<GP>(S, b ^ 1, pl, sp, a.nb_cap, ch1 * kScanBlocks, S.P.pass_g[ps1], S.P.pass_g[ps1 + 1], sub,
                       n_sub1, true, a.status);
      const int g0 = S.P.pass_g[ps], g1 = S.P.pass_g[ps + 1];
      const int s0 = S.P.grp_base[g0], s1 = g1 < S.P.n_groups ? (int)S.P.grp_base[g1] : S.P.n_slots;
      for (int c = 0; c < n_sub; ++c) {
        if (c > 0) __syncwarp();  // every lane is done reading the previous chunk's u
        scan_form_u<GP>(S, b, s0, s1, lb, sub, c, true, a.status);
        __syncwarp();
        const int nbl = (int)min64(kScanBlocks, nb_valid - (ch + c) * kScanBlocks);
        if (lb < nbl) scan_compute_pipe<GP>(S, b, g0, g1, s0, lb, sub, c, true, keep, rot, A, a.status);
        if (ps + 1 == n_passes) finish_chunk(ch + c);
      }
      if (n_sub1 == 0) break;
      ch = ch1;
      ps = ps1;
      n_sub = n_sub1;
    }
  }
  flush_hist();
}

template <int GP, bool kHost>
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
    scan_unit_pipe<GP, kHost>(a, S, unit, c0, c1);
    f += c1 - c0;
  }
}

template <int GP, bool kHost>
cudaError_t launch_scan_gp(ScanArgs a, int64_t chunks, int64_t units, cudaStream_t st) {
  const int smem = (int)sizeof(PipeSmem<GP>);
  void (*kernel)(ScanArgs) = k_scan_pipe<GP, kHost>;
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
  a.chunks = chunks;
  a.units = units;
  // one wave; each CTA an equal share of the work (see k_scan_pipe)
  const unsigned ctas = (unsigned)min64(chunks * units, (int64_t)occ_slots);
  return launch_pdl(kernel, dim3(ctas), dim3(kScanThreads), (size_t)smem, st, a);
}

// Device-resident and pinned host caches alike: asynchronous copies into
// shared memory; host caches take wide steps.
cudaError_t launch_scan(const bpkv_cache& c, const float* q, const uint8_t* depths, float* scores, int64_t ld,
                        cudaStream_t st, const void* plan, uint32_t* hist, int32_t n_sink, int32_t n_recent,
                        int32_t pending, int32_t* status) {
  ScanArgs a{plan,         c.planes, c.scales, c.seq_len, q,        depths,  scores, ld, c.cap_tokens / kBlock,
             c.n_kv_heads, c.group,  hist,     n_sink,    n_recent, pending, status, 0,  0};
  const int64_t chunks = (c.n_max + kScanBlocks * kBlock - 1) / (kScanBlocks * kBlock);
  if (chunks == 0) return cudaSuccess;
  const int64_t units = (int64_t)c.n_seq * c.n_kv_heads;
  auto go = [&](auto gp) {
    constexpr int GP = decltype(gp)::value;
    return c.residency == 1 ? launch_scan_gp<GP, true>(a, chunks, units, st)
                            : launch_scan_gp<GP, false>(a, chunks, units, st);
  };
  if (c.group <= 1) return go(std::integral_constant<int, 1>{});
  if (c.group <= 2) return go(std::integral_constant<int, 2>{});
  if (c.group <= 4) return go(std::integral_constant<int, 4>{});
  return go(std::integral_constant<int, 8>{});
}

}  // namespace bpkv
