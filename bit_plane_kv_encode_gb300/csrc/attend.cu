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

#include <stddef.h>

#include <algorithm>
#include <type_traits>

namespace bpkv {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kSparseRows = 64;    // union rows per CTA
constexpr int kDenseRows = 512;    // tokens per CTA (dense)
constexpr int kPartStride = kD + 4;  // o[D], m, l, 2 pad (rows 16-byte aligned)

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
// Decode-step attention straight from the selection cuts.  One CTA per (token
// range, KV head, sequence).  Every token of the range is marked with the query
// heads that chose it: sinks and recent tokens by all, middle tokens by the
// heads whose cut their (score key, ~index) reaches.  An ordered compaction
// (block scan) lists the range's union rows ascending with their head masks.  Attention then runs in two
// phases: logits with four threads per row, then V accumulation.  The partial
// (max, sum, output) of every head goes to the workspace; the last CTA of the
// unit to finish (ticket counter, zeroed by the depth kernel earlier in the
// step) merges them by log-sum-exp and resets it.
constexpr int kRangeThreads = 256;
constexpr int kRangeMaxRows = 2048;   // union rows of one range (<= min(range tokens, G k))
constexpr int kRangeMaxRanges = 64;   // ranges per unit (long sequences; 24 up to 24 x 4096 tokens)
constexpr int kMergeBlock = 24;       // ranges whose partial outputs the merge holds in registers at once
constexpr int kRangeAlign = 512;      // range sizes are multiples of this
constexpr int kRangeWin = 4096;       // selection window
constexpr int kWinQuads = kRangeWin / 4 / kRangeThreads;  // 4-token quads per thread and window
// quads whose scores a thread loads at once (fewer with more heads: registers)
template <int GP>
__host__ __device__ constexpr int win_batch() { return GP >= 8 ? kWinQuads / 4 : GP >= 4 ? kWinQuads / 2 : kWinQuads; }
constexpr int kQPitch = 36;           // floats per (head, quarter) row of q in shared memory
constexpr int kRcMaxPart = 1024;      // row cache slots of one range

struct RangeArgs {
  const uint16_t* k_rows;
  const uint16_t* v_rows;
  const int64_t* seq_len;
  const float* q;
  const float* scores;             // [N][H][G][ld]
  int64_t ld;
  const unsigned long long* cut;   // [N][H][G]
  int32_t n_sink, n_recent;
  int64_t cap;
  int32_t n_heads, group;
  int64_t range_tok;               // tokens per range, a multiple of kRangeAlign
  int32_t n_ranges;
  float* part;                     // [N][H][n_ranges][G][D + 2]
  uint32_t* tickets;               // [N][H], zero on entry
  float* out;                      // [N][H][G][D]
  int32_t pending;                 // tokens appended in this step but not yet in seq_len
  int64_t* seq_len_out;            // with pending: seq_len, raised by pending once every unit is done
  uint32_t* seq_tick;              // [N], zero on entry (with pending)
  // optional row cache (host-resident caches; see bpkv_cache).  Range rg
  // owns slots [rg part, rg part + part) with part = rc_slots / n_ranges
  // (at most kRcMaxPart), token x of the range lives only in slot
  // rg part + x mod part: a row whose slot holds it is read from there; a row
  // read over the link is written into its slot unless that slot serves a
  // row read from it in this step or a later token of the range claims it
  uint16_t* rc_rows;               // [N][H][rc_slots][2][D]
  int32_t* rc_tok;                 // [N][H][rc_slots]
  int32_t rc_slots;                // 0: no row cache
  int32_t rc_part;                 // slots per range
  uint32_t* rc_stats;              // [N][H][2] rows found, rows (summed over the step's layers)
  // optional: the cut kernel's bits of each head's chosen middle tokens
  // ([N][H][G][map_words], bit x % 32 of word x / 32); without it the
  // selection compares the scores with the cuts
  const uint32_t* selmap;
  int64_t map_words;
};

// Shared memory of a range CTA for up to GP heads (kRc: with the row cache's
// arrays).  The logit buffer later holds the per-slot partial outputs
// [slot][head][D] and the merge's range weights.
template <int GP, bool kRc>
struct RangeSmem {
  static constexpr int kRcRows = kRc ? kRangeMaxRows : 1, kRcPart = kRc ? kRcMaxPart : 1;
  int32_t rows[kRangeMaxRows];
  int32_t rsrc[kRcRows];        // row cache: slot of a row read from it; -2 - slot for a row read over
                                // the link and then written there; -1 otherwise
  int32_t claim[kRcPart];       // row cache: the range's slots (INT32_MAX: serving a row this step)
  uint8_t rmask[kRangeMaxRows];
  __align__(16) float logit[kRangeMaxRows][GP];  // read and written as float4 (slot partials)
  __align__(16) float q[GP * 4 * kQPitch];       // [head][quarter][kQPitch], 32 used; read as float4
  __align__(16) uint8_t wbits[kRangeWin];
  uint32_t ck[BPKV_MAX_GROUP], ci[BPKV_MAX_GROUP];
  float fck[BPKV_MAX_GROUP];              // each head's cut key as a float
  uint32_t mkey[BPKV_MAX_GROUP];          // order-preserving key of each head's largest logit
  uint32_t warp_tot[kRangeThreads / 32];
  float lslot[kRangeThreads / 32][BPKV_MAX_GROUP];
  uint32_t n_rows, is_last;
};

// Bits of the tokens [max(a, x), min(b, x + 32)) in the word of tokens x .. x + 31.
__device__ __forceinline__ uint32_t span_bits(int64_t x, int64_t a, int64_t b) {
  const int64_t s = max64(a - x, 0), e = min64(b - x, 32);
  if (e <= s) return 0u;
  const uint32_t upto = e >= 32 ? 0xFFFFFFFFu : ((1u << e) - 1u);
  return upto & ~((1u << s) - 1u);
}

constexpr int kMapPer = 2;  // map words (32 tokens) per thread and round

// Inverse of ordered_key.
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

template <int GP, bool kRc>
__global__ void __launch_bounds__(kRangeThreads, GP <= 4 ? 3 : 2) k_attend_ranges(RangeArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char range_raw[];
  RangeSmem<GP, kRc>& S = *reinterpret_cast<RangeSmem<GP, kRc>*>(range_raw);
  static_assert(sizeof(S.logit) >= sizeof(float) * (kRangeThreads / 32) * GP * kD, "slot partials fit the logits");
  using SmemT = RangeSmem<GP, kRc>;
  static_assert(offsetof(SmemT, logit) % 16 == 0 && offsetof(SmemT, q) % 16 == 0 && offsetof(SmemT, wbits) % 16 == 0,
                "vector-accessed shared arrays on 16-byte boundaries");
  static_assert(sizeof(S.logit) >= sizeof(float) * kRangeMaxRanges * GP, "merge weights fit the logits");
  const int rg = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int64_t unit = (int64_t)s * a.n_heads + h;
  const int G = a.group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = a.seq_len[s] + a.pending;
  const int64_t t0 = (int64_t)rg * a.range_tok, t1 = min64(t0 + a.range_tok, n);
  const int64_t lo = min64(a.n_sink, n), hi = max64(n - a.n_recent, lo);
  const float qscale = 0.08838834764831845f * 1.4426950408889634f;

  for (int e = tid; e < G * kD; e += kRangeThreads)
    S.q[(e / 32) * kQPitch + e % 32] = a.q[unit * G * kD + e] * qscale;
  if (tid < G) {
    const unsigned long long c = a.cut[unit * G + tid];
    S.ck[tid] = (uint32_t)(c >> 32);
    S.ci[tid] = 0xFFFFFFFFu - (uint32_t)c;
    // key(f) > ck exactly when f > fck, key(f) == ck when f == fck (-0 and +0
    // share a key and compare equal; no score is NaN)
    S.fck[tid] = key_to_float((uint32_t)(c >> 32));
    S.mkey[tid] = 0u;
  }
  __syncthreads();
  uint32_t carry = 0;
  if (a.selmap) {
    // selection from the cut kernel's bits of the chosen middle tokens (a
    // head whose cut is 0 chose every middle token, one whose cut is all ones
    // none); sinks and recent tokens every head.  Each thread takes kMapPer
    // consecutive words of 32 tokens per round and compacts their tokens in
    // order.
    const uint32_t* mp = a.selmap + unit * G * a.map_words;
    const int64_t nw = (t1 - t0 + 31) / 32;  // t0 is a multiple of 32
    for (int64_t i0 = 0; i0 < nw; i0 += (int64_t)kMapPer * kRangeThreads) {
      __syncthreads();  // the previous round is done with warp_tot
      uint32_t hw[kMapPer][GP];
      uint32_t c_sel = 0;
#pragma unroll
      for (int k = 0; k < kMapPer; ++k) {
        const int64_t i = i0 + (int64_t)tid * kMapPer + k;
        const int64_t x = t0 + 32 * i;
        const uint32_t valid = i < nw ? span_bits(x, x, t1) : 0u;
        const uint32_t mid = valid & span_bits(x, lo, hi);
        uint32_t u = 0;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          uint32_t w = 0u;
          if (g < G && valid) {
            const uint32_t ckg = S.ck[g], cig = S.ci[g];
            if (ckg == 0u && cig == 0xFFFFFFFFu) w = 0xFFFFFFFFu;     // cut 0: every middle token
            else if (ckg == 0xFFFFFFFFu && cig == 0u) w = 0u;         // cut all ones: none
            else w = mp[g * a.map_words + (x >> 5)];
            w = (w & mid) | (valid & ~mid);
          }
          hw[k][g] = w;
          u |= w;
        }
        c_sel += __popc(u);
      }
      uint32_t xs = c_sel;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, xs, o);
        if (lane >= o) xs += y;
      }
      if (lane == 31) S.warp_tot[warp] = xs;
      __syncthreads();
      uint32_t pos = carry + xs - c_sel, total = 0;
#pragma unroll
      for (int w = 0; w < kRangeThreads / 32; ++w) {
        const uint32_t t = S.warp_tot[w];
        pos += w < warp ? t : 0u;
        total += t;
      }
#pragma unroll
      for (int k = 0; k < kMapPer; ++k) {
        const int64_t x = t0 + 32 * (i0 + (int64_t)tid * kMapPer + k);
        uint32_t u = 0;
#pragma unroll
        for (int g = 0; g < GP; ++g) u |= hw[k][g];
        while (u) {
          const int b = __ffs(u) - 1;
          u &= u - 1u;
          if (pos < (uint32_t)kRangeMaxRows) {
            uint32_t m = 0;
#pragma unroll
            for (int g = 0; g < GP; ++g) m |= ((hw[k][g] >> b) & 1u) << g;
            S.rows[pos] = (int32_t)(x + b);
            S.rmask[pos] = (uint8_t)m;
          }
          ++pos;
        }
      }
      carry += total;
    }
  } else {
    // selection, in windows of kRangeWin tokens: thread = 4-token quads, all
    // heads' scores of a quad loaded at once (kWinQuads quads in flight); the quads'
    // head masks go to shared memory, then each thread compacts a run of
    // consecutive tokens in order.
    const float* sc = a.scores + unit * G * a.ld;
    const uint32_t all = (1u << G) - 1u;
    for (int64_t w0 = t0; w0 < t1; w0 += kRangeWin) {
      const int wl = (int)min64(kRangeWin, t1 - w0);
      const int wq = (wl + 3) / 4;  // score rows hold whole quads (their length is a multiple of 4)
      // every token of the window is a middle token (no sink, recent or past-the-end checks)
      const bool inner = w0 >= lo && w0 + kRangeWin <= hi && w0 + kRangeWin <= t1;
      __syncthreads();              // the previous window is done
      constexpr int WB = win_batch<GP>();
      for (int q0 = tid; q0 < wq; q0 += WB * kRangeThreads) {
        float4 v[WB][GP];
  #pragma unroll
        for (int u = 0; u < WB; ++u) {
          const int qd = min(q0 + u * kRangeThreads, wq - 1);  // unconditional loads
  #pragma unroll
          for (int g = 0; g < GP; ++g)
            if (g < G) v[u][g] = *reinterpret_cast<const float4*>(sc + g * a.ld + w0 + 4 * qd);
        }
  #pragma unroll
        for (int u = 0; u < WB; ++u) {
          const int qd = q0 + u * kRangeThreads;
          if (qd >= wq) break;
          uint32_t packed = 0;
          const uint32_t xq = (uint32_t)(w0 + 4 * qd);  // the quad's first token
  #pragma unroll
          for (int g = 0; g < GP; ++g) {
            if (g >= G) break;
            const float fc = S.fck[g];
            const uint32_t ci = S.ci[g];
            const float f[4] = {v[u][g].x, v[u][g].y, v[u][g].z, v[u][g].w};
  #pragma unroll
            for (int j = 0; j < 4; ++j)
              if (f[j] > fc || (f[j] == fc && xq + j <= ci)) packed |= 1u << (8 * j + g);
          }
          if (!inner) {
            // tokens past the range's end take nothing; sinks and recent tokens every head
  #pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t x = xq + j;
              if (x >= (uint32_t)t1) packed &= ~(0xFFu << (8 * j));
              else if (x < (uint32_t)lo || x >= (uint32_t)hi) packed |= all << (8 * j);
            }
          }
          reinterpret_cast<uint32_t*>(S.wbits)[qd] = packed;
        }
      }
      __syncthreads();
      const int run = (wl + kRangeThreads - 1) / kRangeThreads, j0 = tid * run;
      uint32_t c_sel = 0;
      for (int j = 0; j < run; ++j) c_sel += (j0 + j < wl && S.wbits[j0 + j] != 0);
      uint32_t x = c_sel;
  #pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) S.warp_tot[warp] = x;
      __syncthreads();
      uint32_t pos = carry + x - c_sel, total = 0;
  #pragma unroll
      for (int w = 0; w < kRangeThreads / 32; ++w) {
        const uint32_t t = S.warp_tot[w];
        pos += w < warp ? t : 0u;
        total += t;
      }
      for (int j = 0; j < run; ++j) {
        if (j0 + j < wl && S.wbits[j0 + j] != 0) {
          if (pos < (uint32_t)kRangeMaxRows) {
            S.rows[pos] = (int32_t)(w0 + j0 + j);
            S.rmask[pos] = S.wbits[j0 + j];
          }
          ++pos;
        }
      }
      carry += total;
    }
  }
  if (tid == 0) S.n_rows = min(carry, (uint32_t)kRangeMaxRows);
  __syncthreads();
  const int nrows = (int)S.n_rows;
  const uint16_t* kb = a.k_rows + unit * a.cap * kD;
  const uint16_t* vb = a.v_rows + unit * a.cap * kD;
  uint16_t* rcu = kRc ? a.rc_rows + unit * a.rc_slots * 2 * kD : nullptr;
  if (kRc) {
    // the range's slots: rows found in the row cache keep theirs; of the rows
    // read over the link, the latest token of each free slot will fill it
    int32_t* tok = a.rc_tok + unit * a.rc_slots;
    const int part = a.rc_part;
    const int32_t sbase = rg * part;
    for (int i = tid; i < part; i += kRangeThreads) S.claim[i] = -1;
    __syncthreads();
    uint32_t hits = 0;
    for (int r = tid; r < nrows; r += kRangeThreads) {
      const int32_t x = S.rows[r];
      const int32_t i = (int32_t)(x % part);
      const bool hit = tok[sbase + i] == x;
      S.rsrc[r] = hit ? sbase + i : -1;
      if (hit) S.claim[i] = INT32_MAX;
      hits += hit ? 1u : 0u;
    }
    __syncthreads();
    for (int r = tid; r < nrows; r += kRangeThreads) {
      const int32_t x = S.rows[r];
      const int32_t i = (int32_t)(x % part);
      if (S.rsrc[r] < 0 && S.claim[i] != INT32_MAX) atomicMax(&S.claim[i], x);
    }
    __syncthreads();
    for (int r = tid; r < nrows; r += kRangeThreads) {
      const int32_t x = S.rows[r];
      const int32_t i = (int32_t)(x % part);
      if (S.rsrc[r] < 0 && S.claim[i] == x) S.rsrc[r] = -2 - (sbase + i);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) hits += __shfl_xor_sync(0xffffffffu, hits, o);
    if (lane == 0) atomicAdd(a.rc_stats + 2 * unit, hits);
    if (tid == 0) atomicAdd(a.rc_stats + 2 * unit + 1, (uint32_t)nrows);
    __syncthreads();
  }
  // the K and V row of union row r: from the row cache or the cache's rows
  auto k_row = [&](int r) -> const uint16_t* {
    const int sl = kRc ? S.rsrc[r] : -1;
    return sl >= 0 ? rcu + (int64_t)sl * 2 * kD : kb + (int64_t)S.rows[r] * kD;
  };
  auto v_row = [&](int r) -> const uint16_t* {
    const int sl = kRc ? S.rsrc[r] : -1;
    return sl >= 0 ? rcu + (int64_t)sl * 2 * kD + kD : vb + (int64_t)S.rows[r] * kD;
  };
  // the row cache slot a row read over the link fills (nullptr: none)
  auto fill_row = [&](int r) -> uint16_t* {
    const int sl = kRc ? S.rsrc[r] : -1;
    return sl <= -2 ? rcu + (int64_t)(-2 - sl) * 2 * kD : nullptr;
  };

  // V rows of this thread's slot, loaded now: they do not depend on the logits.
  // thread = (row slot rs, channels 4 c4 .. 4 c4 + 3); slot rs takes rows
  // rs, rs + kSlots, ...
  constexpr int kSlots = kRangeThreads / 32;
  constexpr int kVPre = 16;
  const int rs = warp, c4 = lane;
  uint2 vpre[kVPre];
  if (nrows > 0) {
#pragma unroll
    for (int b = 0; b < kVPre; ++b) {
      const int r = min(rs + kSlots * b, nrows - 1);
      vpre[b] = *reinterpret_cast<const uint2*>(v_row(r) + 4 * c4);
    }
    if (kRc) {
#pragma unroll
      for (int b = 0; b < kVPre; ++b) {
        const int r = rs + kSlots * b;
        uint16_t* f = r < nrows ? fill_row(r) : nullptr;
        if (f) *reinterpret_cast<uint2*>(f + kD + 4 * c4) = vpre[b];
      }
    }
  }

  // phase 1: logits, four threads per row (32 channels each), two items per
  // thread in flight; the loop bound is the same for every thread, so all
  // lanes reach the shuffles.  q is read as float4 from rows of kQPitch floats
  // per (head, quarter): the four quarters of a warp's rows fall in different
  // banks.  Each head's largest logit goes to S.mkey.
  const int n_items = nrows * 4;
  constexpr int kItemsPer = 1;  // logit items per thread in flight
  float mx[GP];
#pragma unroll
  for (int g = 0; g < GP; ++g) mx[g] = -INFINITY;
  for (int it0 = 0; it0 < n_items; it0 += kItemsPer * kRangeThreads) {
    uint4 w[kItemsPer][4];
#pragma unroll
    for (int u = 0; u < kItemsPer; ++u) {
      const int t = min(it0 + u * kRangeThreads + tid, n_items - 1);
      const uint4* kr = reinterpret_cast<const uint4*>(k_row(t >> 2) + (t & 3) * 32);
#pragma unroll
      for (int c = 0; c < 4; ++c) w[u][c] = kr[c];
      if (kRc && it0 + u * kRangeThreads + tid < n_items) {
        uint16_t* f = fill_row(t >> 2);
        if (f) {
          uint4* fk = reinterpret_cast<uint4*>(f + (t & 3) * 32);
#pragma unroll
          for (int c = 0; c < 4; ++c) fk[c] = w[u][c];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kItemsPer; ++u) {
      const int t = it0 + u * kRangeThreads + tid;
      const bool valid = t < n_items;
      const int r = t >> 2, part4 = t & 3;
      float acc[GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) acc[g] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t wv[4] = {w[u][c].x, w[u][c].y, w[u][c].z, w[u][c].w};
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const float k0 = __uint_as_float(wv[2 * e2] << 16), k1 = __uint_as_float(wv[2 * e2] & 0xffff0000u);
          const float k2 = __uint_as_float(wv[2 * e2 + 1] << 16);
          const float k3 = __uint_as_float(wv[2 * e2 + 1] & 0xffff0000u);
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const float4 qv = *reinterpret_cast<const float4*>(&S.q[(g * 4 + part4) * kQPitch + c * 8 + 4 * e2]);
            acc[g] = fmaf(qv.x, k0, acc[g]);
            acc[g] = fmaf(qv.y, k1, acc[g]);
            acc[g] = fmaf(qv.z, k2, acc[g]);
            acc[g] = fmaf(qv.w, k3, acc[g]);
          }
        }
      }
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 1);
        acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 2);
      }
      if (valid && part4 == 0) {
        const uint32_t mk = S.rmask[r];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          if (g < G) {
            const float lg = ((mk >> g) & 1u) ? acc[g] : -INFINITY;
            S.logit[r][g] = lg;
            mx[g] = fmaxf(mx[g], lg);
          }
        }
      }
    }
  }
#pragma unroll
  for (int g = 0; g < GP; ++g) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], o));
    if (lane == 0 && g < G && mx[g] != -INFINITY) atomicMax(&S.mkey[g], ordered_key(mx[g]));
  }
  __syncthreads();
  float M[GP];
#pragma unroll
  for (int g = 0; g < GP; ++g) M[g] = (g < G && S.mkey[g] != 0u) ? key_to_float(S.mkey[g]) : -INFINITY;

  // phase 2: V accumulation with p = 2^(logit - M) formed on the fly and the
  // sums of p per slot; slots are then added in slot order
  float o[GP][4], lsum[GP];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    lsum[g] = 0.f;
#pragma unroll
    for (int d = 0; d < 4; ++d) o[g][d] = 0.f;
  }
  auto accumulate = [&](uint2 vw, int r) {
    const float vf[4] = {__uint_as_float(vw.x << 16), __uint_as_float(vw.x & 0xffff0000u),
                         __uint_as_float(vw.y << 16), __uint_as_float(vw.y & 0xffff0000u)};
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      if (g >= G) break;
      const float lg = S.logit[r][g];
      const float p = (lg == -INFINITY) ? 0.f : exp2f(lg - M[g]);
      lsum[g] += p;
#pragma unroll
      for (int d = 0; d < 4; ++d) o[g][d] = fmaf(p, vf[d], o[g][d]);
    }
  };
#pragma unroll
  for (int b = 0; b < kVPre; ++b) {
    const int r = rs + kSlots * b;
    if (r < nrows) accumulate(vpre[b], r);
  }
  for (int r0 = rs + kSlots * kVPre; r0 < nrows; r0 += kSlots * 8) {
    uint2 vw[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int r = min(r0 + kSlots * b, nrows - 1);
      vw[b] = *reinterpret_cast<const uint2*>(v_row(r) + 4 * c4);
    }
    if (kRc) {
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int r = r0 + kSlots * b;
        uint16_t* f = r < nrows ? fill_row(r) : nullptr;
        if (f) *reinterpret_cast<uint2*>(f + kD + 4 * c4) = vw[b];
      }
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int r = r0 + kSlots * b;
      if (r < nrows) accumulate(vw[b], r);
    }
  }
  __syncthreads();  // every logit has been read: the logit buffer takes the slot sums
  if (kRc) {
    // the filled slots' rows are written (the barrier above): they now hold their tokens
    int32_t* tok = a.rc_tok + unit * a.rc_slots;
    for (int r = tid; r < nrows; r += kRangeThreads) {
      const int sl = S.rsrc[r];
      if (sl <= -2) tok[-2 - sl] = S.rows[r];
    }
  }
  float* acc = &S.logit[0][0];  // [slot][head][128]
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    if (g >= G) break;
    *reinterpret_cast<float4*>(&acc[(rs * GP + g) * kD + 4 * c4]) = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
    if (lane == 0) S.lslot[rs][g] = lsum[g];
  }
  __syncthreads();
  float* pp = a.part + ((unit * a.n_ranges + rg) * G) * kPartStride;
  for (int e = tid; e < G * kD; e += kRangeThreads) {
    const int g = e / kD, d = e % kD;
    float v = 0.f;
#pragma unroll
    for (int r4 = 0; r4 < kSlots; ++r4) v += acc[(r4 * GP + g) * kD + d];
    pp[g * kPartStride + d] = v;
    if (d == 0) {
      float L = 0.f;
#pragma unroll
      for (int r4 = 0; r4 < kSlots; ++r4) L += S.lslot[r4][g];
      pp[g * kPartStride + kD] = M[g];
      pp[g * kPartStride + kD + 1] = L;
    }
  }
  // ticket: the last CTA of the unit merges every range's partial (the
  // barrier orders the CTA's writes before thread 0's cumulative fence)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    S.is_last = (atomicAdd(&a.tickets[unit], 1u) == (uint32_t)(a.n_ranges - 1)) ? 1u : 0u;
    if (S.is_last) __threadfence();
  }
  __syncthreads();
  if (!S.is_last) return;
  // merge: thread = (head, two channels) with its outputs of kMergeBlock
  // ranges in flight at a time; warp g < G meanwhile reduces head g's (max,
  // sum) pairs across the ranges (lane = range mod 32) into weights
  // 2^(m_c - M) and L (fixed-order sums); the outputs are summed in range order
  const float* pu = a.part + unit * a.n_ranges * G * kPartStride;
  float* pw = &S.logit[0][0];  // [n_ranges][G] weights
  static_assert(kRangeMaxRanges <= 64, "two ranges per lane");
  for (int e0 = 0; e0 < G * (kD / 2); e0 += kRangeThreads) {
    const int e = e0 + tid;
    const int g = min(e, G * (kD / 2) - 1) / (kD / 2), d2 = e % (kD / 2);
    float O0 = 0.f, O1 = 0.f;
    for (int cb = 0; cb < a.n_ranges; cb += kMergeBlock) {
      float2 ov[kMergeBlock];
#pragma unroll
      for (int c = 0; c < kMergeBlock; ++c)  // unconditional loads
        ov[c] = __ldcg(reinterpret_cast<const float2*>(pu + (min(cb + c, a.n_ranges - 1) * G + g) * kPartStride) + d2);
      if (e0 == 0 && cb == 0) {
        if (warp < G) {
          const int gw = warp;
          float mc[2], lc[2];
          bool live[2];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int c = lane + 32 * i;
            const float* pc = pu + (min(c, a.n_ranges - 1) * G + gw) * kPartStride;
            mc[i] = __ldcg(pc + kD);
            lc[i] = __ldcg(pc + kD + 1);
            live[i] = c < a.n_ranges && lc[i] > 0.f;
          }
          float Mx = fmaxf(live[0] ? mc[0] : -INFINITY, live[1] ? mc[1] : -INFINITY);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, o));
          float x = 0.f;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int c = lane + 32 * i;
            const float wc = live[i] ? exp2f(mc[i] - Mx) : 0.f;
            if (live[i]) x += wc * lc[i];
            if (c < a.n_ranges) pw[c * G + gw] = wc;
          }
          // L: inclusive scan over the lanes, the last lane holds the total
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
          }
          if (lane == 31) S.lslot[0][gw] = x;
        }
        __syncthreads();
      }
#pragma unroll
      for (int c = 0; c < kMergeBlock; ++c) {
        if (cb + c < a.n_ranges) {
          const float wc = pw[(cb + c) * G + g];
          O0 = fmaf(wc, ov[c].x, O0);
          O1 = fmaf(wc, ov[c].y, O1);
        }
      }
    }
    const float L = S.lslot[0][g];
    if (e < G * (kD / 2))
      reinterpret_cast<float2*>(a.out + (unit * G + g) * kD)[d2] =
          L > 0.f ? make_float2(O0 / L, O1 / L) : make_float2(0.f, 0.f);
  }
  if (tid == 0) {
    a.tickets[unit] = 0u;
    // every CTA of this unit has read seq_len; the last unit of the sequence
    // to finish raises it by the tokens appended in this step
    if (a.pending && atomicAdd(&a.seq_tick[s], 1u) == (uint32_t)(a.n_heads - 1)) {
      a.seq_len_out[s] += a.pending;
      a.seq_tick[s] = 0u;
    }
  }
}

// Tokens per range: a multiple of kRangeAlign.  Up to kMergeBlock ranges per
// unit while a range stays within one selection window; longer sequences get
// ranges of at least one window, as many as fill the GPU's resident CTAs
// about once over all units (at most kRangeMaxRanges).
int64_t range_tokens(const bpkv_cache& c) {
  const int64_t n_max = c.n_max;
  auto size_for = [&](int64_t ranges) {
    int64_t rt = (n_max + ranges - 1) / ranges;
    rt = (rt + kRangeAlign - 1) / kRangeAlign * kRangeAlign;
    return rt < kRangeAlign ? (int64_t)kRangeAlign : rt;
  };
  const int64_t rt = size_for(kMergeBlock);
  if (rt <= kRangeWin) return rt;
  const int64_t units = std::max<int64_t>(1, (int64_t)c.n_seq * c.n_kv_heads);
  const int64_t per_sm = (c.residency == 1 || c.group > 4) ? 2 : 3;  // resident CTAs per SM
  const int64_t slots = 152 * per_sm;
  const int64_t ranges = std::min<int64_t>(kRangeMaxRanges, std::max<int64_t>(1, slots / units));
  return std::max<int64_t>(kRangeWin, std::max<int64_t>(size_for(ranges), size_for(kRangeMaxRanges)));
}

size_t attend_ranges_part_bytes(const bpkv_cache& c) {
  return (size_t)c.n_seq * c.n_kv_heads * kRangeMaxRanges * c.group * kPartStride * sizeof(float);
}

// A range's union rows (at most its tokens, and at most G k) must fit the row buffers.
bool attend_ranges_eligible(const bpkv_cache& c, int32_t k) {
  const int64_t rows = min64(range_tokens(c), (int64_t)c.group * k);
  return rows <= kRangeMaxRows;
}

cudaError_t launch_attend_ranges(const bpkv_cache& c, const float* q, const float* scores, int64_t ld,
                                 const unsigned long long* cut, int32_t n_sink, int32_t n_recent, float* part,
                                 uint32_t* tickets, float* out, int32_t pending, uint32_t* seq_tick,
                                 cudaStream_t st, uint32_t* rc_stats, const uint32_t* selmap) {
  const int64_t rt = range_tokens(c);
  const int32_t nr = (int32_t)((c.n_max + rt - 1) / rt);
  if (nr == 0) return cudaSuccess;
  const bool rc = c.residency == 1 && c.rc_slots > 0 && rc_stats;
  const int32_t rc_part = rc ? std::min<int32_t>(c.rc_slots / nr, kRcMaxPart) : 0;
  RangeArgs a{c.k_rows, c.v_rows, c.seq_len,     q,       scores, ld,      cut,    n_sink, n_recent,
              c.cap_tokens, c.n_kv_heads, c.group, rt, nr, part, tickets, out, pending, c.seq_len, seq_tick,
              rc && rc_part > 0 ? c.rc_rows : nullptr, rc ? c.rc_tok : nullptr, rc && rc_part > 0 ? c.rc_slots : 0,
              rc_part, rc_stats, selmap, ld / 32};
  auto go = [&](auto kern, auto gp, auto rcv) -> cudaError_t {
    const int smem = (int)sizeof(RangeSmem<decltype(gp)::value, decltype(rcv)::value>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(nr, c.n_kv_heads, c.n_seq), dim3(kRangeThreads), (size_t)smem, st, a);
  };
  using T = std::true_type;
  using F = std::false_type;
  using G1 = std::integral_constant<int, 1>;
  using G2 = std::integral_constant<int, 2>;
  using G4 = std::integral_constant<int, 4>;
  using G8 = std::integral_constant<int, 8>;
  if (a.rc_slots) {
    if (c.group <= 1) return go(k_attend_ranges<1, true>, G1{}, T{});
    if (c.group <= 2) return go(k_attend_ranges<2, true>, G2{}, T{});
    if (c.group <= 4) return go(k_attend_ranges<4, true>, G4{}, T{});
    return go(k_attend_ranges<8, true>, G8{}, T{});
  }
  if (c.group <= 1) return go(k_attend_ranges<1, false>, G1{}, F{});
  if (c.group <= 2) return go(k_attend_ranges<2, false>, G2{}, F{});
  if (c.group <= 4) return go(k_attend_ranges<4, false>, G4{}, F{});
  return go(k_attend_ranges<8, false>, G8{}, F{});
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
