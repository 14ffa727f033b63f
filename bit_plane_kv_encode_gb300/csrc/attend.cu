// Exact attention over the selected rows (Fathom page, section 2: softmax(q K^T
// / sqrt(D)) V over each query head's selected set) and the dense bf16
// baseline, as split-K flash decoding.
//
// Sparse: one CTA per (chunk of union rows, KV head, sequence).  Every union
// row's K and V are read once and applied to each of the G query heads whose
// mask bit is set, so rows chosen by several heads cost one fetch.  Each warp
// keeps an online softmax (running max m, sum l, output o) per head in the
// log2 domain; the CTA merges its warps and writes (o, m, l) for the chunk; a
// second kernel merges chunks with the usual log-sum-exp rescaling.
// Dense: the same with rows = all stored tokens and every head selected.
#include "common.cuh"

namespace bpkv {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kSparseRows = 64;    // union rows per CTA
constexpr int kDenseRows = 512;    // tokens per CTA (dense)
constexpr int kPartStride = kD + 2;  // o[D], m, l

struct AttnArgs {
  const uint16_t* k_rows;
  const uint16_t* v_rows;
  const int64_t* seq_len;
  const float* q;
  const int32_t* uidx;
  const uint8_t* umask;
  const int32_t* ucount;
  int32_t u_cap;
  float* part;
  int32_t n_chunks;
  int64_t cap;
  int32_t n_heads, group;
  int32_t rows_per_chunk;
  int32_t dense;
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(kAttnThreads) k_attend_partial(AttnArgs a) {
  const int chunk = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int64_t unit = (int64_t)s * a.n_heads + h;
  const int G = a.group;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t rows = a.dense ? min64(a.seq_len[s], a.cap) : min64(a.ucount[unit], a.u_cap);
  const int64_t r0 = (int64_t)chunk * a.rows_per_chunk;
  const int64_t r1 = min64(r0 + a.rows_per_chunk, rows);

  // q scaled by log2(e) / sqrt(D): logits in the log2 domain.
  const float qscale = 0.08838834764831845f * 1.4426950408889634f;
  float qr[BPKV_MAX_GROUP][4];
  const float* qp = a.q + unit * G * kD;
#pragma unroll
  for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
#pragma unroll
    for (int d = 0; d < 4; ++d) qr[g][d] = (g < G) ? qp[g * kD + lane * 4 + d] * qscale : 0.f;
  }
  float m[BPKV_MAX_GROUP], l[BPKV_MAX_GROUP], o[BPKV_MAX_GROUP][4];
#pragma unroll
  for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int d = 0; d < 4; ++d) o[g][d] = 0.f;
  }
  const uint16_t* kb = a.k_rows + unit * a.cap * kD;
  const uint16_t* vb = a.v_rows + unit * a.cap * kD;
  const int32_t* ui = a.uidx + unit * a.u_cap;
  const uint8_t* um = a.umask + unit * a.u_cap;
  for (int64_t r = r0 + warp; r < r1; r += kAttnWarps) {
    const int64_t tok = a.dense ? r : (int64_t)ui[r];
    const uint32_t mask = a.dense ? 0xffu : (uint32_t)um[r];
    const uint2 kw = *reinterpret_cast<const uint2*>(kb + tok * kD + lane * 4);
    const uint2 vw = *reinterpret_cast<const uint2*>(vb + tok * kD + lane * 4);
    const float kf[4] = {__uint_as_float(kw.x << 16), __uint_as_float(kw.x & 0xffff0000u),
                         __uint_as_float(kw.y << 16), __uint_as_float(kw.y & 0xffff0000u)};
    const float vf[4] = {__uint_as_float(vw.x << 16), __uint_as_float(vw.x & 0xffff0000u),
                         __uint_as_float(vw.y << 16), __uint_as_float(vw.y & 0xffff0000u)};
#pragma unroll
    for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
      if (g >= G || !((mask >> g) & 1u)) continue;
      float dot = qr[g][0] * kf[0];
      dot = fmaf(qr[g][1], kf[1], dot);
      dot = fmaf(qr[g][2], kf[2], dot);
      dot = fmaf(qr[g][3], kf[3], dot);
      dot = warp_sum(dot);
      const float mn = fmaxf(m[g], dot);
      const float corr = exp2f(m[g] - mn);
      const float p = exp2f(dot - mn);
      l[g] = l[g] * corr + p;
#pragma unroll
      for (int d = 0; d < 4; ++d) o[g][d] = fmaf(o[g][d], corr, p * vf[d]);
      m[g] = mn;
    }
  }
  // merge the warps of this CTA
  __shared__ float sm_m[kAttnWarps][BPKV_MAX_GROUP], sm_l[kAttnWarps][BPKV_MAX_GROUP];
  __shared__ float sm_o[kAttnWarps][BPKV_MAX_GROUP][kD];
#pragma unroll
  for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
    if (g >= G) break;
    if (lane == 0) {
      sm_m[warp][g] = m[g];
      sm_l[warp][g] = l[g];
    }
#pragma unroll
    for (int d = 0; d < 4; ++d) sm_o[warp][g][lane * 4 + d] = o[g][d];
  }
  __syncthreads();
  float* pp = a.part + (unit * a.n_chunks + chunk) * G * kPartStride;
  const int d = threadIdx.x;  // one output channel per thread
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
    for (int w = 0; w < kAttnWarps; ++w)
      if (sm_l[w][g] > 0.f) M = fmaxf(M, sm_m[w][g]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kAttnWarps; ++w) {
        if (!(sm_l[w][g] > 0.f)) continue;
        const float f = exp2f(sm_m[w][g] - M);
        L += sm_l[w][g] * f;
        O += sm_o[w][g][d] * f;
      }
    }
    pp[g * kPartStride + d] = O;
    if (d == 0) {
      pp[g * kPartStride + kD] = M;
      pp[g * kPartStride + kD + 1] = L;
    }
  }
}

__global__ void __launch_bounds__(kD) k_attend_combine(AttnArgs a, float* out) {
  const int row = blockIdx.x;  // (s * H + h) * G + g
  const int G = a.group;
  const int64_t unit = row / G;
  const int g = row % G;
  const int s = (int)(unit / a.n_heads);
  const int64_t rows = a.dense ? min64(a.seq_len[s], a.cap) : min64(a.ucount[unit], a.u_cap);
  const int nc = (int)min64(a.n_chunks, (rows + a.rows_per_chunk - 1) / a.rows_per_chunk);
  const float* pp = a.part + unit * a.n_chunks * G * kPartStride + g * kPartStride;
  const int d = threadIdx.x;
  float M = -INFINITY;
  for (int c = 0; c < nc; ++c) {
    const float* pc = pp + (int64_t)c * G * kPartStride;
    if (pc[kD + 1] > 0.f) M = fmaxf(M, pc[kD]);
  }
  float L = 0.f, O = 0.f;
  if (M != -INFINITY) {
    for (int c = 0; c < nc; ++c) {
      const float* pc = pp + (int64_t)c * G * kPartStride;
      if (!(pc[kD + 1] > 0.f)) continue;
      const float f = exp2f(pc[kD] - M);
      L += pc[kD + 1] * f;
      O += pc[d] * f;
    }
  }
  out[(int64_t)row * kD + d] = (L > 0.f) ? O / L : 0.f;
}

int attend_chunks(int64_t rows, bool dense) {
  const int rpc = dense ? kDenseRows : kSparseRows;
  return (int)((rows + rpc - 1) / rpc);
}

size_t attend_part_bytes(const bpkv_cache& c, int64_t rows, bool dense) {
  return (size_t)c.n_seq * c.n_kv_heads * attend_chunks(rows, dense) * c.group * kPartStride * sizeof(float);
}

cudaError_t launch_attend(const bpkv_cache& c, const float* q, const int32_t* uidx, const uint8_t* umask,
                          const int32_t* ucount, int32_t u_cap, float* part, float* out, bool dense,
                          cudaStream_t st) {
  const int64_t rows = dense ? c.n_max : (int64_t)u_cap;
  const int n_chunks = attend_chunks(rows, dense);
  AttnArgs a{c.k_rows, c.v_rows, c.seq_len, q, uidx, umask, ucount, u_cap, part, n_chunks, c.cap_tokens,
             c.n_kv_heads, c.group, dense ? kDenseRows : kSparseRows, dense ? 1 : 0};
  if (n_chunks > 0) {
    dim3 grid(n_chunks, c.n_kv_heads, c.n_seq);
    k_attend_partial<<<grid, kAttnThreads, 0, st>>>(a);
  }
  k_attend_combine<<<c.n_seq * c.n_kv_heads * c.group, kD, 0, st>>>(a, out);
  return cudaGetLastError();
}

}  // namespace bpkv
