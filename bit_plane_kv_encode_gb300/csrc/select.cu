// Selection (Fathom page, section 2, "Top-k decoding") and the GQA union of
// winner rows (section 1 / section 3.1: k_U <= G k distinct rows per KV head).
//
// Top-k: one CTA per query head.  An exact radix select over order-preserving
// 32-bit keys of the candidate scores (8 bits per pass, most significant
// first) finds the key of the (k - n_sink - n_recent)-th largest candidate and
// how many candidates equal to it are still needed; an ordered compaction then
// writes sinks, recent tokens, every candidate above that key and the
// lowest-index candidates equal to it, in ascending token order.
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

__global__ void __launch_bounds__(kSelThreads) k_topk(TopkArgs a) {
  const int row = blockIdx.x;
  const int s = row / (a.n_heads * a.group);
  const int64_t n = a.seq_len[s];
  const float* sc = a.scores + (int64_t)row * a.ld;
  int32_t* out = a.idx + (int64_t)row * a.k;
  const int64_t lo = min64(a.n_sink, n);
  const int64_t hi = max64(n - a.n_recent, lo);
  const int64_t n_top = max(a.k - a.n_sink - a.n_recent, 0);
  const int tid = threadIdx.x;

  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t tot;
  __shared__ uint32_t sh_digit;
  __shared__ int64_t sh_rem;

  const bool select_all = (hi - lo) <= n_top;
  uint32_t thr = 0xFFFFFFFFu;  // with n_top == 0 no candidate passes
  int64_t need = 0;
  if (!select_all && n_top > 0) {
    uint32_t pref = 0, pmask = 0;
    int64_t rem = n_top;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      for (int64_t i = lo + tid; i < hi; i += kSelThreads) {
        const uint32_t u = ordered_key(sc[i]);
        if ((u & pmask) == pref) atomicAdd(&hist[(u >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns digits 255 - 8l ... 248 - 8l (descending)
        uint32_t loc = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) loc += hist[255 - 8 * tid - q];
        uint32_t incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += y;
        }
        const uint32_t excl = incl - loc;
        const bool here = excl < (uint64_t)rem && (uint64_t)rem <= incl;
        if (here) {
          uint32_t cum = excl;
          int d = 255 - 8 * tid;
          for (int q = 0; q < 8; ++q, --d) {
            const uint32_t hcount = hist[d];
            if (cum + hcount >= (uint64_t)rem) break;
            cum += hcount;
          }
          sh_digit = (uint32_t)d;
          sh_rem = rem - cum;
        }
      }
      __syncthreads();
      pref |= sh_digit << shift;
      pmask |= 255u << shift;
      rem = sh_rem;
      __syncthreads();
    }
    thr = pref;
    need = rem;
  }

  // Ordered compaction over all n tokens.
  uint32_t carry_sel = 0, carry_tie = 0;
  for (int64_t base = 0; base < n; base += kSelThreads) {
    const int64_t i = base + tid;
    uint32_t fsel = 0, ftie = 0;
    if (i < n) {
      if (i < lo || i >= hi || select_all) {
        fsel = 1;
      } else {
        const uint32_t u = ordered_key(sc[i]);
        if (u > thr) fsel = 1;
        else if (u == thr) ftie = 1;
      }
    }
    const uint32_t packed = fsel | (ftie << 16);
    const uint32_t ex = block_excl_scan(packed, warp_tot, &tot);
    const uint32_t ex_sel = (ex & 0xffffu) + carry_sel;
    const uint32_t ex_tie = (ex >> 16) + carry_tie;
    const bool take = fsel || (ftie && (int64_t)ex_tie < need);
    if (take) {
      const int64_t pos = (int64_t)ex_sel + min64(ex_tie, need);
      if (pos < a.k) out[pos] = (int32_t)i;
      else set_status(a.status, BPKV_DEV_SELECT);
    }
    carry_sel += tot & 0xffffu;
    carry_tie += tot >> 16;
  }
  const int64_t total = (int64_t)carry_sel + min64(carry_tie, need);
  for (int64_t p = total + tid; p < a.k; p += kSelThreads) out[p] = -1;
}

cudaError_t launch_topk(const bpkv_cache& c, const float* scores, int64_t ld, int32_t k, int32_t n_sink,
                        int32_t n_recent, int32_t* idx, int32_t* status, cudaStream_t st) {
  TopkArgs a{scores, ld, c.seq_len, idx, status, c.n_kv_heads, c.group, k, n_sink, n_recent};
  k_topk<<<c.n_seq * c.n_kv_heads * c.group, kSelThreads, 0, st>>>(a);
  return cudaGetLastError();
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
  k_union<<<c.n_seq * c.n_kv_heads, kSelThreads, sm, st>>>(a);
  return cudaGetLastError();
}

}  // namespace bpkv
