// Device building blocks of the cluster kernels (selection, sorting, block
// reductions, attention over a CTA's rows).  See fused.cu and tail.cu.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace bpkv {

constexpr int kClThreads = 256;
constexpr int kClBins = 2048;
constexpr int kClCand = 2048;            // threshold-bin candidates kept before falling back to a full sort
constexpr int kClSortCap = 8192;         // entries of the full-sort fallback
constexpr int kClMaxTop = 988;           // k - n_sink - n_recent at most (k <= 1024)

struct SelScratch {
  uint32_t hist[kClBins];
  unsigned long long buf[kClSortCap];    // candidates, or every entry for the full sort
  unsigned long long win[kClMaxTop + 4];
  uint32_t warp_red[32];
  uint32_t n_buf, n_win, bin, rem;
};

struct AttScratch {
  float m[8][BPKV_MAX_GROUP], l[8][BPKV_MAX_GROUP];
  float o[8][BPKV_MAX_GROUP][kD];
};

__device__ __forceinline__ unsigned long long sel_entry(uint32_t key, uint32_t tok) {
  return ((unsigned long long)key << 32) | (0xFFFFFFFFu - tok);  // larger = earlier
}
__device__ __forceinline__ uint32_t entry_tok(unsigned long long e) { return 0xFFFFFFFFu - (uint32_t)e; }

__device__ __forceinline__ uint32_t block_sum_u32(uint32_t v, uint32_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  uint32_t s = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
  __syncthreads();
  return s;
}

__device__ __forceinline__ uint32_t block_min_max(uint32_t v, bool is_max, uint32_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t y = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? max(v, y) : min(v, y);
  }
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  uint32_t s = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) s = is_max ? max(s, red[w]) : min(s, red[w]);
  __syncthreads();
  return s;
}

template <typename T>
__device__ void cta_bitonic(T* v, int n2, bool desc) {
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < n2 / 2; t += blockDim.x) {
        const int i = 2 * t - (t & (stride - 1));
        const int j = i + stride;
        const bool d = ((i & size) == 0) == desc;
        const T a = v[i], b = v[j];
        if ((a < b) == d) {
          v[i] = b;
          v[j] = a;
        }
      }
      __syncthreads();
    }
  }
}

__device__ __forceinline__ int pow2_ge(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Exact top-m of cnt entries (u64: key << 32 | ~token; larger first) given by
// get(e).  Winners are handed to emit(entry) (each exactly once).  Scratch S.
template <typename Get, typename Emit>
__device__ void cta_select(SelScratch& S, int cnt, int m, Get get, Emit emit) {
  const int tid = threadIdx.x;
  if (m <= 0 || cnt <= 0) return;
  if (cnt <= m) {
    for (int e = tid; e < cnt; e += blockDim.x) emit(get(e));
    __syncthreads();
    return;
  }
  // Every pass reads kSelBatch entries per thread before using them, so their
  // loads are in flight together.
  constexpr int kSelBatch = 8;
  // key range
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int e0 = tid; e0 < cnt; e0 += blockDim.x * kSelBatch) {
    unsigned long long v[kSelBatch];
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) {
      const int e = e0 + b * (int)blockDim.x;
      v[b] = e < cnt ? get(e) : 0ull;
    }
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) {
      if (e0 + b * (int)blockDim.x >= cnt) continue;
      const uint32_t k = (uint32_t)(v[b] >> 32);
      lo = min(lo, k);
      hi = max(hi, k);
    }
  }
  lo = block_min_max(lo, false, S.warp_red);
  hi = block_min_max(hi, true, S.warp_red);
  // monotone bin map (any non-decreasing map of the key works for selection)
  const float scale = (float)kClBins / ((float)(hi - lo) + 1.f);
  auto bin_of = [&](uint32_t k) -> int { return min((int)((float)(k - lo) * scale), kClBins - 1); };
  for (int b = tid; b < kClBins; b += blockDim.x) S.hist[b] = 0;
  if (tid == 0) S.n_buf = 0;
  __syncthreads();
  for (int e0 = tid; e0 < cnt; e0 += blockDim.x * kSelBatch) {
    unsigned long long v[kSelBatch];
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) {
      const int e = e0 + b * (int)blockDim.x;
      v[b] = e < cnt ? get(e) : 0ull;
    }
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b)
      if (e0 + b * (int)blockDim.x < cnt) atomicAdd(&S.hist[bin_of((uint32_t)(v[b] >> 32))], 1u);
  }
  __syncthreads();
  // threshold bin: the bin holding the m-th largest key, scanned from the top
  if (tid < 32) {
    const int per = kClBins / 32;
    const int top = kClBins - 1 - tid * per;
    uint32_t loc = 0;
    for (int q = 0; q < per; ++q) loc += S.hist[top - q];
    uint32_t incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += y;
    }
    const uint32_t excl = incl - loc;
    if (excl < (uint32_t)m && (uint32_t)m <= incl) {
      uint32_t cum = excl;
      int d = top;
      for (int q = 0; q < per; ++q, --d) {
        if (cum + S.hist[d] >= (uint32_t)m) break;
        cum += S.hist[d];
      }
      S.bin = (uint32_t)d;
      S.rem = (uint32_t)m - cum;
    }
  }
  __syncthreads();
  const int tb = (int)S.bin;
  const uint32_t rem = S.rem;
  const bool crowded = S.hist[tb] > (uint32_t)kClCand;
  __syncthreads();
  if (!crowded) {
    for (int e0 = tid; e0 < cnt; e0 += blockDim.x * kSelBatch) {
      unsigned long long v[kSelBatch];
#pragma unroll
      for (int b = 0; b < kSelBatch; ++b) {
        const int e = e0 + b * (int)blockDim.x;
        v[b] = e < cnt ? get(e) : 0ull;
      }
#pragma unroll
      for (int b = 0; b < kSelBatch; ++b) {
        if (e0 + b * (int)blockDim.x >= cnt) continue;
        const int bb = bin_of((uint32_t)(v[b] >> 32));
        if (bb > tb) {
          emit(v[b]);
        } else if (bb == tb) {
          const uint32_t c = atomicAdd(&S.n_buf, 1u);
          S.buf[c] = v[b];
        }
      }
    }
    __syncthreads();
    const int nb = (int)S.n_buf;
    const int n2 = pow2_ge(max(nb, 2));
    for (int e = nb + tid; e < n2; e += blockDim.x) S.buf[e] = 0ull;
    __syncthreads();
    cta_bitonic(S.buf, n2, true);
    for (int e = tid; e < (int)rem; e += blockDim.x) emit(S.buf[e]);
  } else {
    // many keys in one bin: sort every entry (exact, slower)
    const int n2 = pow2_ge(max(cnt, 2));
    for (int e = tid; e < n2; e += blockDim.x) S.buf[e] = e < cnt ? get(e) : 0ull;
    __syncthreads();
    cta_bitonic(S.buf, n2, true);
    for (int e = tid; e < m; e += blockDim.x) emit(S.buf[e]);
  }
  __syncthreads();
}


// Attention of up to GP query heads over rows given as (token offset, head
// bits) in shared memory: warps take rows in batches whose K/V loads are issued
// together, keep an online softmax per head in the log2 domain, and the CTA
// merges its warps into part[g][0..D) (output), part[g][D] (max), part[g][D+1]
// (sum).  kb / vb point at the first row of the CTA's token range.
template <int GP>
__device__ void attend_rows(AttScratch& A, const int32_t* rows, const uint8_t* rmask, int nrows,
                            const uint16_t* kb, const uint16_t* vb, const float* qp, int G,
                            float (*part)[kD + 2]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_warps = blockDim.x >> 5;
  const float qscale = 0.08838834764831845f * 1.4426950408889634f;
  float qr[GP][4];
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int d = 0; d < 4; ++d) qr[g][d] = (g < G) ? qp[g * kD + lane * 4 + d] * qscale : 0.f;
  float m[GP], l[GP], o[GP][4];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int d = 0; d < 4; ++d) o[g][d] = 0.f;
  }
  kb += lane * 4;
  vb += lane * 4;
  constexpr int RB = 4;
  for (int rb = warp; rb < nrows; rb += n_warps * RB) {
    uint2 kw[RB], vw[RB];
    uint32_t mk[RB];
#pragma unroll
    for (int b = 0; b < RB; ++b) {
      const int r = rb + b * n_warps;
      mk[b] = 0;
      if (r < nrows) {
        const int64_t x = rows[r];
        mk[b] = rmask[r];
        kw[b] = *reinterpret_cast<const uint2*>(kb + x * kD);
        vw[b] = *reinterpret_cast<const uint2*>(vb + x * kD);
      }
    }
#pragma unroll
    for (int b = 0; b < RB; ++b) {
      if (mk[b] == 0) continue;
      const float kf[4] = {__uint_as_float(kw[b].x << 16), __uint_as_float(kw[b].x & 0xffff0000u),
                           __uint_as_float(kw[b].y << 16), __uint_as_float(kw[b].y & 0xffff0000u)};
      const float vf[4] = {__uint_as_float(vw[b].x << 16), __uint_as_float(vw[b].x & 0xffff0000u),
                           __uint_as_float(vw[b].y << 16), __uint_as_float(vw[b].y & 0xffff0000u)};
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        if (g >= G || !((mk[b] >> g) & 1u)) continue;
        float dot = qr[g][0] * kf[0];
        dot = fmaf(qr[g][1], kf[1], dot);
        dot = fmaf(qr[g][2], kf[2], dot);
        dot = fmaf(qr[g][3], kf[3], dot);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
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
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    if (lane == 0) {
      A.m[warp][g] = m[g];
      A.l[warp][g] = l[g];
    }
#pragma unroll
    for (int d = 0; d < 4; ++d) A.o[warp][g][lane * 4 + d] = o[g][d];
  }
  __syncthreads();
  for (int e = tid; e < GP * kD; e += blockDim.x) {
    const int g = e / kD, d = e % kD;
    float M = -INFINITY;
    for (int w = 0; w < n_warps; ++w)
      if (A.l[w][g] > 0.f) M = fmaxf(M, A.m[w][g]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < n_warps; ++w) {
        if (!(A.l[w][g] > 0.f)) continue;
        const float f = exp2f(A.m[w][g] - M);
        L += A.l[w][g] * f;
        O += A.o[w][g][d] * f;
      }
    }
    part[g][d] = O;
    if (d == 0) {
      part[g][kD] = M;
      part[g][kD + 1] = L;
    }
  }
  __syncthreads();
}

// Leader side of the partial merge: output of head g from the partials of
// every CTA of the cluster (log-sum-exp rescaling).  Threads d < D.
template <int CS>
__device__ void merge_partials(cooperative_groups::cluster_group& cluster, float (*part)[kD + 2], int g,
                               float* out) {
  const int d = threadIdx.x;
  if (d >= kD) return;
  float mr[CS], lr[CS];
  float M = -INFINITY;
#pragma unroll
  for (int r = 0; r < CS; ++r) {
    const float* pr = cluster.map_shared_rank(&part[g][0], r);
    mr[r] = pr[kD];
    lr[r] = pr[kD + 1];
    if (lr[r] > 0.f) M = fmaxf(M, mr[r]);
  }
  float L = 0.f, O = 0.f;
  if (M != -INFINITY) {
#pragma unroll
    for (int r = 0; r < CS; ++r) {
      if (!(lr[r] > 0.f)) continue;
      const float* pr = cluster.map_shared_rank(&part[g][0], r);
      const float f = exp2f(mr[r] - M);
      L += lr[r] * f;
      O += pr[d] * f;
    }
  }
  out[d] = (L > 0.f) ? O / L : 0.f;
}

}  // namespace bpkv
