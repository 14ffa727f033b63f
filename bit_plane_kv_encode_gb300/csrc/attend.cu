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

// ---------------------------------------------------------------------------
// Decode-step attention straight from the per-head selections.  One CTA per
// (token range, KV head, sequence): it binary-searches each head's ascending
// index list for the tokens of its range, merges those pieces into the range's
// union rows with head masks (ranks by binary search in the other pieces), and
// attends in two phases: logits with one thread per row (a whole 128-channel
// dot product per thread, no shuffles), then V accumulation with one thread per
// channel.  The partial (max, sum, output) of every head goes to the
// workspace; the last CTA of the unit to finish (ticket counter, zeroed by the
// depth kernel earlier in the step) merges them by log-sum-exp and resets it.
constexpr int kRangeThreads = 128;
constexpr int kRangeMaxEnt = 4096;    // selected (token, head) entries in one range (<= G k)
constexpr int kRangeMaxRows = 2048;   // union rows of one range (<= min(range tokens, G k))
constexpr int kRangeMaxRanges = 16;   // ranges per unit

struct RangeArgs {
  const uint16_t* k_rows;
  const uint16_t* v_rows;
  const int64_t* seq_len;
  const float* q;
  const int32_t* idx;     // [N][H][G][k], ascending, -1 padded
  int32_t k;
  int64_t cap;
  int32_t n_heads, group;
  int64_t range_tok;      // tokens per range
  int32_t n_ranges;
  float* part;            // [N][H][n_ranges][G][D + 2]
  uint32_t* tickets;      // [N][H], zero on entry
  float* out;             // [N][H][G][D]
};

struct RangeSmem {
  int32_t sub[kRangeMaxEnt];           // the heads' pieces of their lists, one after another
  int32_t rows[kRangeMaxEnt];
  uint8_t rmask[kRangeMaxEnt];
  float logit[kRangeMaxRows][BPKV_MAX_GROUP];
  float q[BPKV_MAX_GROUP][kD];
  int sa[BPKV_MAX_GROUP], sn[BPKV_MAX_GROUP], soff[BPKV_MAX_GROUP];
  float red[BPKV_MAX_GROUP][kRangeThreads / 32];
  float m[BPKV_MAX_GROUP], l[BPKV_MAX_GROUP];
  uint32_t n_rows, is_last;
};

__device__ __forceinline__ int valid_count(const int32_t* v, int k) {
  int lo = 0, hi = k;  // entries >= 0 come first
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] >= 0) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ int lower_bound_g(const int32_t* v, int n, int64_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)v[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kRangeThreads) k_attend_ranges(RangeArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char range_raw[];
  RangeSmem& S = *reinterpret_cast<RangeSmem*>(range_raw);
  const int rg = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int64_t unit = (int64_t)s * a.n_heads + h;
  const int G = a.group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = a.seq_len[s];
  const int64_t t0 = (int64_t)rg * a.range_tok, t1 = min64(t0 + a.range_tok, n);
  const int32_t* li = a.idx + unit * G * a.k;
  const float qscale = 0.08838834764831845f * 1.4426950408889634f;

  for (int e = tid; e < G * kD; e += kRangeThreads) S.q[e / kD][e % kD] = a.q[unit * G * kD + e] * qscale;
  // the heads' lists, staged with one coalesced pass (rows[] is free until the merge)
  int32_t* lst = S.rows;
  for (int e = tid; e < G * a.k; e += kRangeThreads) lst[e] = li[e];
  __syncthreads();
  if (tid < G) {
    const int32_t* lg = lst + tid * a.k;
    const int cnt = valid_count(lg, a.k);
    const int lo = t0 < t1 ? lower_bound_g(lg, cnt, t0) : 0;
    const int hi = t0 < t1 ? lower_bound_g(lg, cnt, t1) : 0;
    S.sa[tid] = lo;
    S.sn[tid] = hi - lo;
  }
  __syncthreads();
  if (tid == 0) {
    int off = 0;
    for (int g = 0; g < G; ++g) {
      S.soff[g] = off;
      off += S.sn[g];
    }
    S.n_rows = (uint32_t)off;  // entries before merging
  }
  __syncthreads();
  const int n_ent = (int)S.n_rows;
  for (int g = 0; g < G; ++g)
    for (int i = tid; i < S.sn[g]; i += kRangeThreads) S.sub[S.soff[g] + i] = lst[g * a.k + S.sa[g] + i];
  __syncthreads();
  // merge rank of every entry; duplicates (same token, several heads) are ordered by head
  for (int e = tid; e < n_ent; e += kRangeThreads) {
    int g = 0;
    while (g + 1 < G && S.soff[g + 1] <= e) ++g;
    const int32_t x = S.sub[e];
    int pos = e - S.soff[g];
    for (int g2 = 0; g2 < G; ++g2) {
      if (g2 == g) continue;
      const int32_t* v = S.sub + S.soff[g2];
      const int nn = S.sn[g2];
      int lo = 0, hi = nn;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (g2 < g ? v[mid] <= x : v[mid] < x) lo = mid + 1;
        else hi = mid;
      }
      pos += lo;
    }
    S.rows[pos] = x;
    S.rmask[pos] = (uint8_t)g;  // head of the entry for now
  }
  __syncthreads();
  // collapse equal tokens: the first entry of each run keeps the OR of the heads
  uint32_t first = 0, bits = 0;
  int32_t tok = -1;
  if (tid == 0) S.n_rows = 0;
  __syncthreads();
  for (int base = 0; base < n_ent; base += kRangeThreads) {
    const int e = base + tid;
    first = 0;
    if (e < n_ent) {
      tok = S.rows[e];
      first = (e == 0 || S.rows[e - 1] != tok) ? 1u : 0u;
      bits = 0;
      if (first)
        for (int j = e; j < n_ent && S.rows[j] == tok; ++j) bits |= 1u << S.rmask[j];
    }
    __syncthreads();
    const uint32_t bal = __ballot_sync(0xffffffffu, first);
    __shared__ uint32_t wcnt[kRangeThreads / 32];
    if (lane == 0) wcnt[warp] = __popc(bal);
    __syncthreads();
    uint32_t off = S.n_rows;
    for (int w = 0; w < warp; ++w) off += wcnt[w];
    off += __popc(bal & ((1u << lane) - 1u));
    uint32_t tile = 0;
    for (int w = 0; w < kRangeThreads / 32; ++w) tile += wcnt[w];
    __syncthreads();
    if (first) {
      S.rows[off] = tok;  // off <= e: writes land on entries already read
      S.rmask[off] = (uint8_t)bits;
    }
    if (tid == 0) S.n_rows += tile;
    __syncthreads();
  }
  const int nrows = (int)S.n_rows;

  const uint16_t* kb = a.k_rows + unit * a.cap * kD;
  const uint16_t* vb = a.v_rows + unit * a.cap * kD;
  // phase 1: logits, four threads per row (32 channels each).  The loop bound
  // is the same for every thread, so all lanes reach the shuffles.
  const int n_items = nrows * 4;
  for (int t0 = 0; t0 < n_items; t0 += kRangeThreads) {
    const int t = t0 + tid;
    const bool valid = t < n_items;
    const int r = t >> 2, part4 = t & 3;
    uint4 w[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) w[c] = make_uint4(0u, 0u, 0u, 0u);
    if (valid) {
      const uint4* kr = reinterpret_cast<const uint4*>(kb + (int64_t)S.rows[r] * kD + part4 * 32);
#pragma unroll
      for (int c = 0; c < 4; ++c) w[c] = kr[c];
    }
    float acc[BPKV_MAX_GROUP];
#pragma unroll
    for (int g = 0; g < BPKV_MAX_GROUP; ++g) acc[g] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t wv[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(wv[e] << 16), hi = __uint_as_float(wv[e] & 0xffff0000u);
        const int ch = part4 * 32 + c * 8 + 2 * e;
#pragma unroll
        for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
          if (g >= G) break;
          acc[g] = fmaf(S.q[g][ch], lo, acc[g]);
          acc[g] = fmaf(S.q[g][ch + 1], hi, acc[g]);
        }
      }
    }
#pragma unroll
    for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
      acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 1);
      acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 2);
    }
    if (valid && part4 == 0) {
      const uint32_t mk = S.rmask[r];
#pragma unroll
      for (int g = 0; g < BPKV_MAX_GROUP; ++g)
        if (g < G) S.logit[r][g] = ((mk >> g) & 1u) ? acc[g] : -INFINITY;
    }
  }
  __syncthreads();
  // phase 2: per-head max and sum
  for (int g = 0; g < G; ++g) {
    float mx = -INFINITY;
    for (int r = tid; r < nrows; r += kRangeThreads) mx = fmaxf(mx, S.logit[r][g]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) S.red[g][warp] = mx;
  }
  __syncthreads();
  if (tid < G) {
    float mx = S.red[tid][0];
    for (int w = 1; w < kRangeThreads / 32; ++w) mx = fmaxf(mx, S.red[tid][w]);
    S.m[tid] = mx;
  }
  __syncthreads();
  for (int g = 0; g < G; ++g) {
    float sum = 0.f;
    const float mg = S.m[g];
    for (int r = tid; r < nrows; r += kRangeThreads) {
      const float p = (S.logit[r][g] == -INFINITY) ? 0.f : exp2f(S.logit[r][g] - mg);
      S.logit[r][g] = p;
      sum += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) S.red[g][warp] = sum;
  }
  __syncthreads();
  if (tid < G) {
    float sum = 0.f;
    for (int w = 0; w < kRangeThreads / 32; ++w) sum += S.red[tid][w];
    S.l[tid] = sum;
  }
  __syncthreads();
  // phase 3: V accumulation: thread = (row slot rs of 4, channels 4 c4 .. 4 c4 + 3),
  // rows rs, rs + 4, ... with eight 8-byte loads in flight; slots merged in order
  {
    const int rs = tid >> 5, c4 = tid & 31;
    float o[BPKV_MAX_GROUP][4];
#pragma unroll
    for (int g = 0; g < BPKV_MAX_GROUP; ++g)
#pragma unroll
      for (int d = 0; d < 4; ++d) o[g][d] = 0.f;
    for (int r0 = rs; r0 < nrows; r0 += 4 * 8) {
      uint2 vw[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int r = r0 + 4 * b;
        vw[b] = r < nrows ? *reinterpret_cast<const uint2*>(vb + (int64_t)S.rows[r] * kD + 4 * c4)
                          : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int r = r0 + 4 * b;
        if (r >= nrows) break;
        const float vf[4] = {__uint_as_float(vw[b].x << 16), __uint_as_float(vw[b].x & 0xffff0000u),
                             __uint_as_float(vw[b].y << 16), __uint_as_float(vw[b].y & 0xffff0000u)};
#pragma unroll
        for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
          if (g >= G) break;
          const float p = S.logit[r][g];
#pragma unroll
          for (int d = 0; d < 4; ++d) o[g][d] = fmaf(p, vf[d], o[g][d]);
        }
      }
    }
    // merge the four row slots in order through shared memory: the upper half of
    // the logit buffer is free once every weight has been used
    __syncthreads();
    float* acc = &S.logit[kRangeMaxRows / 2][0];  // [slot][head][128]: 4 * 8 * 128 floats
#pragma unroll
    for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
      if (g >= G) break;
#pragma unroll
      for (int d = 0; d < 4; ++d) acc[(rs * BPKV_MAX_GROUP + g) * kD + 4 * c4 + d] = o[g][d];
    }
    __syncthreads();
    const int d = tid;
    float* pp = a.part + ((unit * a.n_ranges + rg) * G) * kPartStride;
    for (int g = 0; g < G; ++g) {
      float v = 0.f;
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) v += acc[(r4 * BPKV_MAX_GROUP + g) * kD + d];
      pp[g * kPartStride + d] = v;
      if (d == 0) {
        pp[g * kPartStride + kD] = S.m[g];
        pp[g * kPartStride + kD + 1] = S.l[g];
      }
    }
  }
  // ticket: the last CTA of the unit merges every range's partial
  __threadfence();
  __syncthreads();
  if (tid == 0) S.is_last = (atomicAdd(&a.tickets[unit], 1u) == (uint32_t)(a.n_ranges - 1)) ? 1u : 0u;
  __syncthreads();
  if (!S.is_last) return;
  __threadfence();
  const float* pu = a.part + unit * a.n_ranges * G * kPartStride;
  // every range's (max, sum) at once, then weights, then the outputs with
  // eight independent loads in flight per thread
  float* wgt = &S.logit[0][0];  // [n_ranges][G] weights (the logits are no longer needed)
  for (int e = tid; e < a.n_ranges * G; e += kRangeThreads) {
    const float lc = __ldcg(pu + e * kPartStride + kD + 1);
    wgt[e] = lc > 0.f ? __ldcg(pu + e * kPartStride + kD) : -INFINITY;
  }
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int c = 0; c < a.n_ranges; ++c) M = fmaxf(M, wgt[c * G + tid]);
    S.m[tid] = M;
  }
  __syncthreads();
  for (int e = tid; e < a.n_ranges * G; e += kRangeThreads) {
    const float mc = wgt[e];
    wgt[e] = (mc == -INFINITY) ? 0.f : exp2f(mc - S.m[e % G]);
  }
  __syncthreads();
  if (tid < G) {
    float L = 0.f;
    for (int c = 0; c < a.n_ranges; ++c) L += wgt[c * G + tid] * __ldcg(pu + (c * G + tid) * kPartStride + kD + 1);
    S.l[tid] = L;
  }
  __syncthreads();
  for (int g = 0; g < G; ++g) {
    float O = 0.f;
    int c = 0;
    for (; c + 8 <= a.n_ranges; c += 8) {
      float ov[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) ov[b] = __ldcg(pu + ((c + b) * G + g) * kPartStride + tid);
#pragma unroll
      for (int b = 0; b < 8; ++b) O = fmaf(wgt[(c + b) * G + g], ov[b], O);
    }
    for (; c < a.n_ranges; ++c) O = fmaf(wgt[c * G + g], __ldcg(pu + (c * G + g) * kPartStride + tid), O);
    a.out[(unit * G + g) * kD + tid] = (S.l[g] > 0.f) ? O / S.l[g] : 0.f;
  }
  if (tid == 0) a.tickets[unit] = 0u;
}

// Tokens per range: at least 512, at most kRangeMaxRanges ranges per unit.
int64_t range_tokens(int64_t n_max) {
  int64_t rt = (n_max + kRangeMaxRanges - 1) / kRangeMaxRanges;
  rt = (rt + 63) / 64 * 64;
  return rt < 512 ? 512 : rt;
}

size_t attend_ranges_part_bytes(const bpkv_cache& c) {
  return (size_t)c.n_seq * c.n_kv_heads * kRangeMaxRanges * c.group * kPartStride * sizeof(float);
}

// The range kernel needs every range's entries and union rows to fit its buffers.
bool attend_ranges_eligible(const bpkv_cache& c, int32_t k) {
  const int64_t ent = (int64_t)c.group * k;
  const int64_t rows = min64(range_tokens(c.n_max), ent);
  return ent <= kRangeMaxEnt && rows <= kRangeMaxRows;
}

cudaError_t launch_attend_ranges(const bpkv_cache& c, const float* q, const int32_t* idx, int32_t k, float* part,
                                 uint32_t* tickets, float* out, cudaStream_t st) {
  const int64_t rt = range_tokens(c.n_max);
  const int32_t nr = (int32_t)((c.n_max + rt - 1) / rt);
  if (nr == 0) return cudaSuccess;
  RangeArgs a{c.k_rows, c.v_rows, c.seq_len, q, idx, k, c.cap_tokens, c.n_kv_heads, c.group, rt, nr, part, tickets,
              out};
  const int smem = (int)sizeof(RangeSmem);
  cudaError_t e = cudaFuncSetAttribute(k_attend_ranges, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_attend_ranges, dim3(nr, c.n_kv_heads, c.n_seq), dim3(kRangeThreads), (size_t)smem, st, a);
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
