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

constexpr int kRowBatch = 4;  // rows whose K/V loads a warp issues together

__global__ void __launch_bounds__(kAttnThreads) k_attend_partial(AttnArgs a) {
  pdl_enter();
  const int chunk = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int64_t unit = (int64_t)s * a.n_heads + h;
  const int G = a.group;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t rows = a.dense ? min64(a.seq_len[s], a.cap) : min64(a.ucount[unit], a.u_cap);
  const int64_t r0 = (int64_t)chunk * a.rows_per_chunk;
  const int nrows = (int)max64(0, min64(r0 + a.rows_per_chunk, rows) - r0);

  __shared__ int32_t s_tok[kSparseRows];
  __shared__ uint8_t s_mask[kSparseRows];
  if (!a.dense) {
    const int32_t* ui = a.uidx + unit * a.u_cap + r0;
    const uint8_t* um = a.umask + unit * a.u_cap + r0;
    for (int r = threadIdx.x; r < nrows; r += kAttnThreads) {
      s_tok[r] = ui[r];
      s_mask[r] = um[r];
    }
  }

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
  __syncthreads();
  const uint16_t* kb = a.k_rows + unit * a.cap * kD + lane * 4;
  const uint16_t* vb = a.v_rows + unit * a.cap * kD + lane * 4;
  for (int rb = warp; rb < nrows; rb += kAttnWarps * kRowBatch) {
    uint2 kw[kRowBatch], vw[kRowBatch];
    uint32_t mk[kRowBatch];
#pragma unroll
    for (int b = 0; b < kRowBatch; ++b) {
      const int r = rb + b * kAttnWarps;
      mk[b] = 0;
      if (r < nrows) {
        const int64_t tok = a.dense ? r0 + r : (int64_t)s_tok[r];
        mk[b] = a.dense ? 0xffu : (uint32_t)s_mask[r];
        kw[b] = *reinterpret_cast<const uint2*>(kb + tok * kD);
        vw[b] = *reinterpret_cast<const uint2*>(vb + tok * kD);
      }
    }
#pragma unroll
    for (int b = 0; b < kRowBatch; ++b) {
      if (mk[b] == 0) continue;
      const float kf[4] = {__uint_as_float(kw[b].x << 16), __uint_as_float(kw[b].x & 0xffff0000u),
                           __uint_as_float(kw[b].y << 16), __uint_as_float(kw[b].y & 0xffff0000u)};
      const float vf[4] = {__uint_as_float(vw[b].x << 16), __uint_as_float(vw[b].x & 0xffff0000u),
                           __uint_as_float(vw[b].y << 16), __uint_as_float(vw[b].y & 0xffff0000u)};
#pragma unroll
      for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
        if (g >= G || !((mk[b] >> g) & 1u)) continue;
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

constexpr int kCombineMax = 2048;  // chunk partials merged per pass

__global__ void __launch_bounds__(kD) k_attend_combine(AttnArgs a, float* out) {
  pdl_enter();
  const int row = blockIdx.x;  // (s * H + h) * G + g
  const int G = a.group;
  const int64_t unit = row / G;
  const int g = row % G;
  const int s = (int)(unit / a.n_heads);
  const int64_t rows = a.dense ? min64(a.seq_len[s], a.cap) : min64(a.ucount[unit], a.u_cap);
  const int nc = (int)min64(a.n_chunks, (rows + a.rows_per_chunk - 1) / a.rows_per_chunk);
  const float* pp = a.part + unit * a.n_chunks * G * kPartStride + g * kPartStride;
  const int d = threadIdx.x;
  __shared__ float s_f[kCombineMax];
  __shared__ float s_red[kD / 32];
  // running merge over passes of up to kCombineMax chunks
  float M = -INFINITY, L = 0.f, O = 0.f;
  for (int c0 = 0; c0 < nc; c0 += kCombineMax) {
    const int cn = min(nc - c0, kCombineMax);
    float mloc = -INFINITY;
    for (int c = d; c < cn; c += kD) {
      const float* pc = pp + (int64_t)(c0 + c) * G * kPartStride;
      const float mc = pc[kD], lc = pc[kD + 1];
      s_f[c] = lc > 0.f ? mc : -INFINITY;
      mloc = fmaxf(mloc, s_f[c]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    if ((d & 31) == 0) s_red[d >> 5] = mloc;
    __syncthreads();
    float Mp = s_red[0];
    for (int w = 1; w < kD / 32; ++w) Mp = fmaxf(Mp, s_red[w]);
    const float Mn = fmaxf(M, Mp);
    __syncthreads();
    // weights of this pass's chunks, and the rescale of what came before
    for (int c = d; c < cn; c += kD) s_f[c] = (s_f[c] == -INFINITY) ? 0.f : exp2f(s_f[c] - Mn);
    __syncthreads();
    const float corr = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
    float Lp = 0.f, Op = 0.f;
    int c = 0;
    for (; c + 4 <= cn; c += 4) {
      const float* p0 = pp + (int64_t)(c0 + c) * G * kPartStride;
      const int64_t st = (int64_t)G * kPartStride;
      const float o0 = p0[d], o1 = p0[st + d], o2 = p0[2 * st + d], o3 = p0[3 * st + d];
      const float l0 = p0[kD + 1], l1 = p0[st + kD + 1], l2 = p0[2 * st + kD + 1], l3 = p0[3 * st + kD + 1];
      Op += s_f[c] * o0 + s_f[c + 1] * o1 + s_f[c + 2] * o2 + s_f[c + 3] * o3;
      Lp += s_f[c] * l0 + s_f[c + 1] * l1 + s_f[c + 2] * l2 + s_f[c + 3] * l3;
    }
    for (; c < cn; ++c) {
      const float* pc = pp + (int64_t)(c0 + c) * G * kPartStride;
      Op += s_f[c] * pc[d];
      Lp += s_f[c] * pc[kD + 1];
    }
    O = O * corr + Op;
    L = L * corr + Lp;
    M = Mn;
    __syncthreads();
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
    const cudaError_t e = launch_pdl(k_attend_partial, grid, dim3(kAttnThreads), 0, st, a);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(k_attend_combine, dim3(c.n_seq * c.n_kv_heads * c.group), dim3(kD), 0, st, a, out);
}

}  // namespace bpkv
