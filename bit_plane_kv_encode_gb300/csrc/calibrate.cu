// Offline choices for the scanned channels.
//
// Calibrated channel sets (Fathom page, section 2, "Double Sparsity"):
// per unit, channel j's statistic is mean|q_j| over the calibration queries
// and the unit's query heads times mean|k_j| over the calibration keys, and
// the n_channels largest (ties to the lower index) are read at one depth.
//
// One CTA per unit, one thread per channel: each thread sums its channel's
// column in double in storage order (coalesced across the CTA's threads), so
// the sums, means and product are those of a plain sequential evaluation; the
// ranks come from a comparison against every other channel's statistic.
//
// Bases (Fathom page, contributions: KLT planes; ReadKV page, section 5.1:
// Hadamard-sign transform): bpkv_rotate takes queries into a cache's basis with
// the same float32 fused multiply-add chains the decode step uses.
#include "common.cuh"

namespace bpkv {

struct CalArgs {
  const float* q_cal;     // [units][m_q][group][D]
  const uint16_t* k_cal;  // [units][m_k][D] bf16
  int32_t group;
  int64_t m_q, m_k;
  int32_t n_channels, depth;
  uint8_t* depths;        // [units][D]
};

__global__ void __launch_bounds__(kD) k_calibrate(CalArgs a) {
  pdl_enter();
  __shared__ double st[kD];
  const int j = threadIdx.x;
  const int64_t unit = blockIdx.x;
  const float* q = a.q_cal + unit * a.m_q * a.group * kD + j;
  const uint16_t* k = a.k_cal + unit * a.m_k * kD + j;
  double sq = 0.0, sk = 0.0;
  const int64_t nq = a.m_q * a.group;
  for (int64_t i = 0; i < nq; ++i) sq = __dadd_rn(sq, fabs((double)q[i * kD]));
  for (int64_t i = 0; i < a.m_k; ++i) sk = __dadd_rn(sk, fabs((double)bf16_bits_to_float(k[i * kD])));
  st[j] = __dmul_rn(__ddiv_rn(sq, (double)nq), __ddiv_rn(sk, (double)a.m_k));
  __syncthreads();
  const double mine = st[j];
  int rank = 0;  // channels ordered before j
  for (int i = 0; i < kD; ++i) {
    const double o = st[i];
    rank += (o > mine || (o == mine && i < j)) ? 1 : 0;
  }
  a.depths[unit * kD + j] = (uint8_t)(rank < a.n_channels ? a.depth : 0);
}

// y = x R per KV head: grid (rows, H, N), one thread per output channel.
__global__ void __launch_bounds__(kD) k_rotate(const float* basis, const float* x, float* y, int32_t n_heads,
                                              int64_t rows) {
  pdl_enter();
  const int64_t h = blockIdx.y, row = ((int64_t)blockIdx.z * n_heads + h) * rows + blockIdx.x;
  const float* R = basis + h * kD * kD;
  const float* xr = x + row * kD;
  const int l = threadIdx.x;
  float acc = 0.f;
  for (int i = 0; i < kD; ++i) acc = __fmaf_rn(xr[i], R[i * kD + l], acc);
  y[row * kD + l] = acc;
}

}  // namespace bpkv

extern "C" int bpkv_rotate(const float* basis, int32_t n_seq, int32_t n_kv_heads, int64_t rows, const float* x,
                           float* y, void* stream) {
  using namespace bpkv;
  if (!basis || !x || !y || n_seq < 1 || n_kv_heads < 1 || rows < 1) return BPKV_EINVAL;
  if (n_seq > 65535 || n_kv_heads > 65535 || rows > 0x7FFFFFFF) return BPKV_EUNSUPPORTED;
  const cudaError_t e = launch_pdl(k_rotate, dim3((unsigned)rows, (unsigned)n_kv_heads, (unsigned)n_seq), dim3(kD), 0,
                                   reinterpret_cast<cudaStream_t>(stream), basis, x, y, n_kv_heads, rows);
  return e == cudaSuccess ? BPKV_OK : BPKV_ECUDA;
}

extern "C" int bpkv_calibrate_channels(const float* q_cal, const uint16_t* k_cal, int32_t n_units, int32_t group,
                                       int64_t m_q, int64_t m_k, int32_t n_channels, int32_t depth, uint8_t* depths,
                                       void* stream) {
  using namespace bpkv;
  if (!q_cal || !k_cal || !depths) return BPKV_EINVAL;
  if (n_units < 1 || group < 1 || group > BPKV_MAX_GROUP || m_q < 1 || m_k < 1) return BPKV_EINVAL;
  if (n_channels < 0 || depth < 0 || depth > 4) return BPKV_EINVAL;
  CalArgs a{q_cal, k_cal, group, m_q, m_k, n_channels, depth, depths};
  const cudaError_t e =
      launch_pdl(k_calibrate, dim3((unsigned)n_units), dim3(kD), 0, reinterpret_cast<cudaStream_t>(stream), a);
  return e == cudaSuccess ? BPKV_OK : BPKV_ECUDA;
}
