// Selection (Fathom page, section 2, "Top-k decoding") and the GQA union of
// winner rows (section 1 / section 3.1: k_U <= G k distinct rows per KV head).
//
// Top-k: one CTA per query head.  Scores map to order-preserving 32-bit keys
// (staged in shared memory when the row's candidates fit).  A linear histogram
// over the candidates' key range [min, max] locates the bucket holding the
// (k - n_sink - n_recent)-th largest key (bins follow the data, so no bin takes
// most of the atomics); a crowded bucket is refined the same way over its own
// exact key range.  One more pass takes every key above the bucket and gathers
// the bucket's keys, which a shared-memory bitonic sort by (key desc, index
// asc) cuts at the exact count: ties go to the lower index, with an ordered
// scan when more than kCandCap keys equal the threshold key.  Sinks, recent
// tokens and the winners are finally sorted ascending.
//
// Union: one CTA per KV head.  Each sorted list entry's rank in the merge of
// the G lists is its own position plus binary-search counts in the other
// lists (ties ordered by head), duplicates collapse into one row whose mask
// ORs the heads that chose it.
#include "common.cuh"

namespace bpkv {

constexpr int kSelThreads = 1024;

struct TopkArgs {
  const float* scores;
  int64_t ld;
  const int64_t* seq_len;
  int32_t* idx;
  int32_t* status;
  int32_t n_heads, group, k, n_sink, n_recent;
};

// Block-wide exclusive scan of one 32-bit value per thread (blockDim = 1024).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_tot[lane];
    uint32_t incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    warp_tot[lane] = incl - w;
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  const uint32_t r = warp_tot[warp] + x - v;
  __syncthreads();
  return r;
}

constexpr int kHistBins = 2048;
constexpr int kCandCap = 4096;       // keys of the threshold bucket kept for the exact sort
constexpr int kSelCap = 8192;        // selected indices (k <= 8192)
constexpr int kSelBatch = 8;         // independent score loads in flight per thread
constexpr int kStageKeys = 32768;    // candidates staged in shared memory when they fit

struct TopkSmem {
  uint32_t keys[kStageKeys];           // staged order-preserving keys of the candidates
  uint32_t hist[kHistBins];
  unsigned long long cand[kCandCap];   // (key << 32) | ~index: larger = earlier
  int32_t sel[kSelCap];
  uint32_t warp_tot[32];
  uint32_t red[2][32];
  uint32_t n_cand, n_sel, tb, rem, tot, b_lo, b_hi;
};

// Bitonic sort of v[0..n2) (n2 a power of two) by the whole value; descending
// when desc, else ascending.  Called by the whole block.
template <typename T>
__device__ void block_bitonic(T* v, int n2, bool desc) {
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < n2 / 2; t += blockDim.x) {
        const int i = 2 * t - (t & (stride - 1));
        const int j = i + stride;
        const bool d = ((i & size) == 0) == desc;
        const T x = v[i], y = v[j];
        if ((x < y) == d) {
          v[i] = y;
          v[j] = x;
        }
      }
      __syncthreads();
    }
  }
}

__device__ __forceinline__ void sel_push(TopkSmem& S, int32_t i) {
  const uint32_t p = atomicAdd(&S.n_sel, 1u);
  if (p < (uint32_t)kSelCap) S.sel[p] = i;
}

__device__ __forceinline__ int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Block-wide min and max of (lo, hi) pairs.
__device__ __forceinline__ void block_range(uint32_t& lo, uint32_t& hi, TopkSmem& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    S.red[0][warp] = lo;
    S.red[1][warp] = hi;
  }
  __syncthreads();
  lo = S.red[0][0];
  hi = S.red[1][0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
    lo = min(lo, S.red[0][w]);
    hi = max(hi, S.red[1][w]);
  }
  __syncthreads();
}

// Visit the order-preserving keys of candidates [0, cnt) (staged in shared
// memory, or read from the scores kSelBatch at a time): f(index, key).
template <typename F>
__device__ __forceinline__ void for_keys(const TopkSmem& S, bool staged, const float* sc, int64_t lo, int64_t cnt,
                                         F f) {
  if (staged) {
    for (int64_t e = threadIdx.x; e < cnt; e += kSelThreads) f(e, S.keys[e]);
    return;
  }
  for (int64_t e0 = threadIdx.x; e0 < cnt; e0 += (int64_t)kSelBatch * kSelThreads) {
    float v[kSelBatch];
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) {
      const int64_t e = e0 + (int64_t)b * kSelThreads;
      v[b] = e < cnt ? sc[lo + e] : 0.f;
    }
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) {
      const int64_t e = e0 + (int64_t)b * kSelThreads;
      if (e < cnt) f(e, ordered_key(v[b]));
    }
  }
}

__global__ void __launch_bounds__(kSelThreads) k_topk(TopkArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char topk_raw[];
  TopkSmem& S = *reinterpret_cast<TopkSmem*>(topk_raw);
  const int row = blockIdx.x;
  const int s = row / (a.n_heads * a.group);
  const int64_t n = a.seq_len[s];
  const float* sc = a.scores + (int64_t)row * a.ld;
  int32_t* out = a.idx + (int64_t)row * a.k;
  const int64_t lo = min64(a.n_sink, n);
  const int64_t hi = max64(n - a.n_recent, lo);
  const int64_t cnt = hi - lo;
  const int64_t n_top = max(a.k - a.n_sink - a.n_recent, 0);
  const int tid = threadIdx.x;

  if (tid == 0) {
    S.n_cand = 0;
    S.n_sel = 0;
  }
  __syncthreads();
  // fixed tokens
  for (int64_t i = tid; i < lo; i += kSelThreads) sel_push(S, (int32_t)i);
  for (int64_t i = hi + tid; i < n; i += kSelThreads) sel_push(S, (int32_t)i);

  if (cnt <= n_top) {
    for (int64_t i = lo + tid; i < hi; i += kSelThreads) sel_push(S, (int32_t)i);
  } else if (n_top > 0) {
    const bool staged = cnt <= kStageKeys;
    // key range of the candidates (staging them when they fit)
    uint32_t klo = 0xFFFFFFFFu, khi = 0u;
    if (staged) {
      for (int e0 = tid; e0 < cnt; e0 += kSelBatch * kSelThreads) {
        float v[kSelBatch];
#pragma unroll
        for (int b = 0; b < kSelBatch; ++b) {
          const int e = e0 + b * kSelThreads;
          v[b] = e < cnt ? sc[lo + e] : 0.f;
        }
#pragma unroll
        for (int b = 0; b < kSelBatch; ++b) {
          const int e = e0 + b * kSelThreads;
          if (e < cnt) {
            const uint32_t k = ordered_key(v[b]);
            S.keys[e] = k;
            klo = min(klo, k);
            khi = max(khi, k);
          }
        }
      }
    } else {
      for_keys(S, false, sc, lo, cnt, [&](int64_t, uint32_t k) {
        klo = min(klo, k);
        khi = max(khi, k);
      });
    }
    block_range(klo, khi, S);
    // Threshold bucket: a linear histogram over the active key range [klo, khi]
    // locates the bucket holding the rem-th largest active key; a crowded
    // bucket becomes the next active range (its exact min and max keys).
    uint32_t rem = (uint32_t)n_top, b_lo = klo, b_hi = khi, bucket_n = 0;
    int tb_final = -1;
    float scale_final = 0.f;
    for (int lvl = 0; lvl < 3; ++lvl) {
      const float scale = (float)kHistBins / ((float)(khi - klo) + 1.f);
      auto bin_of = [&](uint32_t k) { return min((int)((float)(k - klo) * scale), kHistBins - 1); };
      for (int b = tid; b < kHistBins; b += kSelThreads) S.hist[b] = 0;
      __syncthreads();
      for_keys(S, staged, sc, lo, cnt, [&](int64_t, uint32_t k) {
        if (k >= klo && k <= khi) atomicAdd(&S.hist[bin_of(k)], 1u);
      });
      __syncthreads();
      // thread t owns bins 2047 - 2t and 2046 - 2t (descending); block scan
      const uint32_t h0 = S.hist[kHistBins - 1 - 2 * tid], h1 = S.hist[kHistBins - 2 - 2 * tid];
      const uint32_t ex = block_excl_scan(h0 + h1, S.warp_tot, &S.tot);
      if (ex < rem && rem <= ex + h0) {
        S.tb = kHistBins - 1 - 2 * tid;
        S.rem = rem - ex;
      } else if (ex + h0 < rem && rem <= ex + h0 + h1) {
        S.tb = kHistBins - 2 - 2 * tid;
        S.rem = rem - ex - h0;
      }
      __syncthreads();
      const int tb = (int)S.tb;
      rem = S.rem;
      bucket_n = S.hist[tb];
      if (bucket_n <= (uint32_t)kCandCap) {
        // small bucket: keys are classified by their bin under this level's map
        tb_final = tb;
        scale_final = scale;
        break;
      }
      // crowded bucket: its exact key range becomes the next level's range
      uint32_t blo = 0xFFFFFFFFu, bhi = 0u;
      for_keys(S, staged, sc, lo, cnt, [&](int64_t, uint32_t k) {
        if (k >= klo && k <= khi && bin_of(k) == tb) {
          blo = min(blo, k);
          bhi = max(bhi, k);
        }
      });
      block_range(blo, bhi, S);
      b_lo = blo;
      b_hi = bhi;
      if (b_lo == b_hi) break;
      klo = b_lo;
      khi = b_hi;
    }
    if (tb_final >= 0) {
      // keys in higher bins are selected; the bucket's keys are ranked exactly
      const uint32_t klo_f = klo, khi_f = khi;
      auto bin_f = [&](uint32_t k) { return min((int)((float)(k - klo_f) * scale_final), kHistBins - 1); };
      for_keys(S, staged, sc, lo, cnt, [&](int64_t e, uint32_t k) {
        if (k < klo_f || k > khi_f) {
          if (k > khi_f) sel_push(S, (int32_t)(lo + e));
          return;
        }
        const int b = bin_f(k);
        if (b > tb_final) {
          sel_push(S, (int32_t)(lo + e));
        } else if (b == tb_final) {
          const uint32_t c = atomicAdd(&S.n_cand, 1u);
          if (c < (uint32_t)kCandCap)
            S.cand[c] = ((unsigned long long)k << 32) | (0xFFFFFFFFu - (uint32_t)(lo + e));
        }
      });
      __syncthreads();
      const int nc = (int)min(S.n_cand, (uint32_t)kCandCap);
      if (nc <= kSelThreads) {
        // rank of each candidate among the bucket (distinct entries): no barriers
        if (tid < nc) {
          const unsigned long long mine = S.cand[tid];
          int rank = 0;
          for (int j = 0; j < nc; ++j) rank += S.cand[j] > mine;
          if (rank < (int)rem) sel_push(S, (int32_t)(0xFFFFFFFFu - (uint32_t)mine));
        }
      } else {
        const int nc2 = pow2_at_least(nc);
        for (int e = nc + tid; e < nc2; e += kSelThreads) S.cand[e] = 0ull;
        __syncthreads();
        block_bitonic(S.cand, nc2, true);
        for (int e = tid; e < (int)rem && e < nc; e += kSelThreads)
          sel_push(S, (int32_t)(0xFFFFFFFFu - (uint32_t)S.cand[e]));
      }
    } else {
      // more than kCandCap keys equal the threshold key (b_lo == b_hi): take
      // the rem of them with the lowest indices by an ordered scan
      uint32_t carry = 0;
      for (int64_t base = 0; base < cnt; base += kSelThreads) {
        const int64_t e = base + tid;
        uint32_t tie = 0;
        if (e < cnt) {
          const uint32_t k = staged ? S.keys[e] : ordered_key(sc[lo + e]);
          if (k > b_hi) sel_push(S, (int32_t)(lo + e));
          else if (k == b_lo) tie = 1;
        }
        const uint32_t ex = block_excl_scan(tie, S.warp_tot, &S.tot) + carry;
        if (tie && ex < rem) sel_push(S, (int32_t)(lo + e));
        carry += S.tot;
        __syncthreads();
      }
    }
  }
  __syncthreads();
  const int ns = (int)S.n_sel;
  if (ns > a.k && tid == 0) set_status(a.status, BPKV_DEV_SELECT);
  const int cnt_out = min(ns, a.k);
  if (cnt_out <= kSelThreads) {
    // ascending order by rank (the indices are distinct): no barriers
    if (tid < cnt_out) {
      const int32_t mine = S.sel[tid];
      int rank = 0;
      for (int j = 0; j < cnt_out; ++j) rank += S.sel[j] < mine;
      out[rank] = mine;
    }
    for (int e = cnt_out + tid; e < a.k; e += kSelThreads) out[e] = -1;
    return;
  }
  const int n2 = pow2_at_least(max(cnt_out, 2));
  for (int e = cnt_out + tid; e < n2; e += kSelThreads) S.sel[e] = 0x7FFFFFFF;
  __syncthreads();
  block_bitonic(S.sel, n2, false);
  for (int e = tid; e < a.k; e += kSelThreads) out[e] = e < cnt_out ? S.sel[e] : -1;
}

cudaError_t launch_topk(const bpkv_cache& c, const float* scores, int64_t ld, int32_t k, int32_t n_sink,
                        int32_t n_recent, int32_t* idx, int32_t* status, cudaStream_t st) {
  TopkArgs a{scores, ld, c.seq_len, idx, status, c.n_kv_heads, c.group, k, n_sink, n_recent};
  const int smem = (int)sizeof(TopkSmem);
  cudaError_t e = cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_topk, dim3(c.n_seq * c.n_kv_heads * c.group), dim3(kSelThreads), smem, st, a);
}

// ---------------------------------------------------------------- union

struct UnionArgs {
  const int32_t* idx;
  int32_t* uidx;
  uint8_t* umask;
  int32_t* ucount;
  int32_t group, k;
};

__device__ __forceinline__ int lower_bound_i32(const int32_t* v, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ int upper_bound_i32(const int32_t* v, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] <= x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kSelThreads) k_union(UnionArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) int32_t usm[];
  const int G = a.group, k = a.k;
  int32_t* L = usm;              // [G][k] lists
  int32_t* M = usm + G * k;      // [G k] merged token indices
  uint8_t* MH = reinterpret_cast<uint8_t*>(usm + 2 * G * k);  // [G k] head of each merged entry
  __shared__ int cnt[BPKV_MAX_GROUP];
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t tot;
  const int unit = blockIdx.x;
  const int tid = threadIdx.x;
  const int32_t* src = a.idx + (int64_t)unit * G * k;
  for (int e = tid; e < G * k; e += kSelThreads) L[e] = src[e];
  if (tid < G) cnt[tid] = 0;
  __syncthreads();
  // valid prefix length of each list (entries are ascending, then -1)
  for (int e = tid; e < G * k; e += kSelThreads) {
    const int h = e / k, r = e % k;
    const bool valid = L[e] >= 0;
    const bool next_invalid = (r + 1 == k) || L[e + 1] < 0;
    if (valid && next_invalid) cnt[h] = r + 1;
  }
  __syncthreads();
  int m_total = 0;
  for (int h = 0; h < G; ++h) m_total += cnt[h];
  for (int e = tid; e < G * k; e += kSelThreads) {
    const int h = e / k, r = e % k;
    if (r >= cnt[h]) continue;
    const int32_t x = L[e];
    int pos = r;
    for (int h2 = 0; h2 < G; ++h2) {
      if (h2 == h) continue;
      pos += (h2 < h) ? upper_bound_i32(L + h2 * k, cnt[h2], x) : lower_bound_i32(L + h2 * k, cnt[h2], x);
    }
    M[pos] = x;
    MH[pos] = (uint8_t)h;
  }
  __syncthreads();
  int32_t* uo = a.uidx + (int64_t)unit * G * k;
  uint8_t* mo = a.umask + (int64_t)unit * G * k;
  uint32_t carry = 0;
  for (int base = 0; base < m_total; base += kSelThreads) {
    const int p = base + tid;
    uint32_t first = 0;
    uint8_t mask = 0;
    if (p < m_total) {
      first = (p == 0 || M[p - 1] != M[p]) ? 1u : 0u;
      if (first) {
        for (int q = p; q < m_total && M[q] == M[p]; ++q) mask |= (uint8_t)(1u << MH[q]);
      }
    }
    const uint32_t ex = block_excl_scan(first, warp_tot, &tot) + carry;
    if (first) {
      uo[ex] = M[p];
      mo[ex] = mask;
    }
    carry += tot;
  }
  for (int p = (int)carry + tid; p < G * k; p += kSelThreads) {
    uo[p] = -1;
    mo[p] = 0;
  }
  if (tid == 0) a.ucount[unit] = (int32_t)carry;
}

size_t union_smem_bytes(int G, int k) { return (size_t)G * k * (4 + 4 + 1) + 16; }

cudaError_t launch_union(const bpkv_cache& c, const int32_t* idx, int32_t k, int32_t* uidx, uint8_t* umask,
                         int32_t* ucount, cudaStream_t st) {
  const size_t sm = union_smem_bytes(c.group, k);
  if (sm > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_union, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
  }
  UnionArgs a{idx, uidx, umask, ucount, c.group, k};
  return launch_pdl(k_union, dim3(c.n_seq * c.n_kv_heads), dim3(kSelThreads), sm, st, a);
}

}  // namespace bpkv
