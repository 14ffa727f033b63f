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
      t = a.depths[unit * kD + tid];
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

template <int GP>
cudaError_t launch_scan_gp(ScanArgs a, int64_t chunks, int64_t units, cudaStream_t st) {
  const int smem = (int)sizeof(ScanSmem<GP>);
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
      e = cudaFuncSetAttribute(k_scan<GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      int sms = 0, per_sm = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_scan<GP>, kScanThreads, smem);
      if (e != cudaSuccess) return e;
      slots[dev] = sms * (per_sm > 0 ? per_sm : 1);
    }
    occ_slots = slots[dev];
  }
  // enough chunks per CTA for the grid to fit in one wave of resident CTAs
  const int64_t total = chunks * units;
  a.chunks_per_cta = (total + occ_slots - 1) / occ_slots;
  if (a.chunks_per_cta < 1) a.chunks_per_cta = 1;
  const dim3 grid((unsigned)((chunks + a.chunks_per_cta - 1) / a.chunks_per_cta), (unsigned)a.n_heads,
                  (unsigned)(units / a.n_heads));
  return launch_pdl(k_scan<GP>, grid, dim3(kScanThreads), (size_t)smem, st, a);
}

cudaError_t launch_scan(const bpkv_cache& c, const float* q, const uint8_t* depths, float* scores, int64_t ld,
                        cudaStream_t st, const void* plan, uint32_t* hist, int32_t n_sink, int32_t n_recent,
                        int32_t pending) {
  ScanArgs a{plan,         c.planes, c.scales, c.seq_len, q,        depths, scores, ld, c.cap_tokens / kBlock,
             c.n_kv_heads, c.group,  hist,     n_sink,    n_recent, 1,      pending};
  const int64_t chunks = (c.n_max + kScanBlocks * kBlock - 1) / (kScanBlocks * kBlock);
  if (chunks == 0) return cudaSuccess;
  const int64_t units = (int64_t)c.n_seq * c.n_kv_heads;
  if (c.group <= 1) return launch_scan_gp<1>(a, chunks, units, st);
  if (c.group <= 2) return launch_scan_gp<2>(a, chunks, units, st);
  if (c.group <= 4) return launch_scan_gp<4>(a, chunks, units, st);
  return launch_scan_gp<8>(a, chunks, units, st);
}

}  // namespace bpkv
