// Selection (Fathom page, section 2, "Top-k decoding") and the GQA union of
// winner rows (section 1 / section 3.1: k_U <= G k distinct rows per KV head).
//
// Top-k: one CTA per query head.  Scores map to order-preserving 32-bit keys.
// A histogram of the top 11 key bits over the candidates (tokens that are
// neither sinks nor recent) locates the bucket holding the
// (k - n_sink - n_recent)-th largest key; if that bucket is crowded the next 11
// bits (then the last 10) refine it.  One more pass takes every key above the
// bucket and gathers the bucket's keys, which a shared-memory bitonic sort by
// (key desc, index asc) cuts at the exact count: ties go to the lower index.
// Sinks, recent tokens and the winners are finally sorted ascending.
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

constexpr int kHistBits = 11;
constexpr int kHistBins = 1 << kHistBits;
constexpr int kCandCap = 4096;       // candidates kept from the threshold bucket
constexpr int kSelCap = 8192;        // selected indices (k <= 8192)
constexpr int kSelBatch = 8;         // independent score loads in flight per thread

struct TopkSmem {
  uint32_t hist[kHistBins];
  unsigned long long cand[kCandCap];   // (key << 32) | ~index: larger = earlier
  int32_t sel[kSelCap];
  uint32_t warp_tot[32];
  uint32_t n_cand, n_sel, digit, rem, tot;
};

// Bitonic sort of v[0..n2) (n2 a power of two) by the whole 64-bit value;
// descending when desc, else ascending.  Called by the whole block.
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

  if (hi - lo <= n_top) {
    for (int64_t i = lo + tid; i < hi; i += kSelThreads) sel_push(S, (int32_t)i);
  } else if (n_top > 0) {
    // Threshold bucket: up to three levels (11, 11, 10 bits), stopping once the
    // bucket holding the n_top-th largest key has at most kCandCap keys.
    uint32_t pref = 0, pmask = 0;
    uint32_t rem = (uint32_t)n_top;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int lvl = 0; lvl < 3; ++lvl) {
      const int shift = shifts[lvl], nb = 1 << widths[lvl];
      for (int b = tid; b < nb; b += kSelThreads) S.hist[b] = 0;
      __syncthreads();
      for (int64_t base = lo; base < hi; base += kSelBatch * kSelThreads) {
        float v[kSelBatch];
#pragma unroll
        for (int b = 0; b < kSelBatch; ++b) {
          const int64_t i = base + b * kSelThreads + tid;
          v[b] = i < hi ? sc[i] : 0.f;
        }
#pragma unroll
        for (int b = 0; b < kSelBatch; ++b) {
          const int64_t i = base + b * kSelThreads + tid;
          const uint32_t u = ordered_key(v[b]);
          if (i < hi && (u & pmask) == pref) atomicAdd(&S.hist[(u >> shift) & (nb - 1)], 1u);
        }
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns bins [nb - (l+1) nb/32, nb - l nb/32), scanned from the top
        const int per = nb / 32;
        const int top = nb - 1 - tid * per;
        uint32_t loc = 0;
        for (int q = 0; q < per; ++q) loc += S.hist[top - q];
        uint32_t incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += y;
        }
        const uint32_t excl = incl - loc;
        if (excl < rem && rem <= incl) {
          uint32_t cum = excl;
          int d = top;
          for (int q = 0; q < per; ++q, --d) {
            if (cum + S.hist[d] >= rem) break;
            cum += S.hist[d];
          }
          S.digit = (uint32_t)d;
          S.rem = rem - cum;
        }
      }
      __syncthreads();
      const uint32_t dgt = S.digit;
      rem = S.rem;
      pref |= dgt << shift;
      pmask |= (uint32_t)(nb - 1) << shift;
      const bool done = S.hist[dgt] <= (uint32_t)kCandCap;
      __syncthreads();
      if (done) break;
    }
    // keys above the bucket are selected; keys in it are candidates
    const uint32_t above = pref | ~pmask;
    const bool exact = pmask == 0xFFFFFFFFu && S.hist[pref & (kHistBins / 2 - 1)] > (uint32_t)kCandCap;
    if (!exact) {
      for (int64_t base = lo; base < hi; base += kSelBatch * kSelThreads) {
        float v[kSelBatch];
#pragma unroll
        for (int b = 0; b < kSelBatch; ++b) {
          const int64_t i = base + b * kSelThreads + tid;
          v[b] = i < hi ? sc[i] : 0.f;
        }
#pragma unroll
        for (int b = 0; b < kSelBatch; ++b) {
          const int64_t i = base + b * kSelThreads + tid;
          if (i >= hi) continue;
          const uint32_t u = ordered_key(v[b]);
          if (u > above) {
            sel_push(S, (int32_t)i);
          } else if ((u & pmask) == pref) {
            const uint32_t c = atomicAdd(&S.n_cand, 1u);
            if (c < (uint32_t)kCandCap)
              S.cand[c] = ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)i);
          }
        }
      }
      __syncthreads();
      const int nc = (int)min(S.n_cand, (uint32_t)kCandCap);
      const int nc2 = pow2_at_least(max(nc, 2));
      for (int e = nc + tid; e < nc2; e += kSelThreads) S.cand[e] = 0ull;
      __syncthreads();
      block_bitonic(S.cand, nc2, true);
      for (int e = tid; e < (int)rem && e < nc; e += kSelThreads)
        sel_push(S, (int32_t)(0xFFFFFFFFu - (uint32_t)S.cand[e]));
    } else {
      // more than kCandCap keys equal the threshold key: take the rem of them
      // with the lowest indices by an ordered scan over the candidates
      uint32_t carry = 0;
      for (int64_t base = lo; base < hi; base += kSelThreads) {
        const int64_t i = base + tid;
        uint32_t tie = 0;
        if (i < hi) {
          const uint32_t u = ordered_key(sc[i]);
          if (u > above) sel_push(S, (int32_t)i);
          else if (u == pref) tie = 1;
        }
        const uint32_t ex = block_excl_scan(tie, S.warp_tot, &S.tot) + carry;
        if (tie && ex < rem) sel_push(S, (int32_t)i);
        carry += S.tot;
        __syncthreads();
      }
    }
  }
  __syncthreads();
  const int ns = (int)S.n_sel;
  if (ns > a.k && tid == 0) set_status(a.status, BPKV_DEV_SELECT);
  const int cnt = min(ns, a.k);
  const int n2 = pow2_at_least(max(cnt, 2));
  for (int e = cnt + tid; e < n2; e += kSelThreads) S.sel[e] = 0x7FFFFFFF;
  __syncthreads();
  block_bitonic(S.sel, n2, false);
  for (int e = tid; e < a.k; e += kSelThreads) out[e] = e < cnt ? S.sel[e] : -1;
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
