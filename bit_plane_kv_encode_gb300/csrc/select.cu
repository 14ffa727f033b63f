// Selection (Fathom page, section 2, "Top-k decoding") and the GQA union of
// winner rows (section 1 / section 3.1: k_U <= G k distinct rows per KV head).
//
// Top-k, as an exact radix selection over order-preserving 32-bit score keys.
// Each row (query head) keeps its sinks [0, n_sink), its recent tokens
// [n - n_recent, n) and the m = k - n_sink - n_recent largest middle keys,
// ties to the lower index.  Ordering the middle tokens by (key desc, index
// asc), the chosen ones are exactly those whose 64-bit value (key, ~index) is
// at least the m-th largest such value: the row's "cut".
//   1. A 4096-bin histogram of the middle keys' top 12 bits (counted by the
//      scan kernel as it writes the scores, or by k_hist) locates the bucket
//      holding the m-th largest key.
//   2. k_cut: CTAs over 4096-key chunks of the row append the bucket's keys to
//      the row's candidate list; the last CTA to finish ranks them and stores
//      the cut.  A bucket of more than 1024 keys is refined by that CTA on the
//      next 12, then 8, key bits; a bucket that is a single key value repeated
//      more than 1024 times is cut at the right occurrence in index order.
//   3. k_lists (when index lists are wanted): an ordered compaction writes the
//      sinks, the chosen middle tokens and the recent tokens ascending.
// The decode step's attention reads the cuts directly.
//
// Union: one CTA per KV head.  Each sorted list entry's rank in the merge of
// the G lists is its own position plus binary-search counts in the other
// lists (ties ordered by head), duplicates collapse into one row whose mask
// ORs the heads that chose it.
#include "common.cuh"

#include <mutex>

namespace bpkv {

constexpr int kSelThreads = 1024;  // k_lists and k_union
constexpr int kCutThreads = 256;   // k_hist and k_cut
constexpr int kCutChunk = 4096;    // middle keys per k_hist / k_cut CTA
constexpr int kSelBatch = 16;      // independent score loads in flight per thread
constexpr int kTileKeys = 32768;   // keys staged in shared memory per k_lists tile

// Block-wide exclusive scan of one 32-bit value per thread (any block size that
// is a multiple of 32, up to 1024).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = lane < n_warps ? warp_tot[lane] : 0u;
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

// The middle range [lo, hi) of a row and the number m of its keys to choose.
struct RowRange {
  int64_t n, lo, hi, cnt, m;
};

__device__ __forceinline__ RowRange row_range(int64_t n, int32_t k, int32_t n_sink, int32_t n_recent) {
  RowRange r;
  r.n = n;
  r.lo = min64(n_sink, n);
  r.hi = max64(n - n_recent, r.lo);
  r.cnt = r.hi - r.lo;
  r.m = max(k - n_sink - n_recent, 0);
  return r;
}

// f(e, key) for the middle keys e in [e_begin, e_end) of a row (scores sc,
// middle starting at lo), kSelBatch independent loads in flight per thread.
template <typename F>
__device__ __forceinline__ void for_row_keys(const float* __restrict__ sc, int64_t lo, int64_t e_begin,
                                             int64_t e_end, F f) {
  const int nt = blockDim.x;
  for (int64_t e0 = e_begin + threadIdx.x; e0 < e_end; e0 += (int64_t)kSelBatch * nt) {
    float v[kSelBatch];
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) v[b] = sc[lo + min64(e0 + (int64_t)b * nt, e_end - 1)];  // unconditional
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) {
      const int64_t e = e0 + (int64_t)b * nt;
      if (e < e_end) f(e, ordered_key(v[b]));
    }
  }
}

// ------------------------------------------------------------------ k_hist

struct HistArgs {
  const float* scores;
  int64_t ld;
  const int64_t* seq_len;
  uint32_t* hist;  // [rows][kTopkBins], zero on entry
  int32_t rows_per_seq, k, n_sink, n_recent;
  int32_t pending;         // tokens appended in this step but not yet in seq_len
  int32_t chunks_per_cta;  // consecutive chunks of kCutChunk keys per CTA
};

// Level-0 histogram of a run of chunks of one row's middle keys, counted in
// shared memory and added to the row's once.  Grid (runs, rows).
__global__ void __launch_bounds__(kCutThreads) k_hist(HistArgs a) {
  pdl_enter();
  __shared__ uint32_t H[kTopkBins];
  const int row = blockIdx.y;
  const RowRange r = row_range(a.seq_len[row / a.rows_per_seq] + a.pending, a.k, a.n_sink, a.n_recent);
  const int64_t c0 = (int64_t)blockIdx.x * a.chunks_per_cta * kCutChunk;
  const int64_t c1 = min64(c0 + (int64_t)a.chunks_per_cta * kCutChunk, r.cnt);
  if (r.cnt <= r.m || r.m == 0 || c0 >= c1) return;
  for (int b = threadIdx.x; b < kTopkBins; b += kCutThreads) H[b] = 0u;
  __syncthreads();
  for_row_keys(a.scores + (int64_t)row * a.ld, r.lo, c0, c1,
               [&](int64_t, uint32_t key) { atomicAdd(&H[key >> 20], 1u); });
  __syncthreads();
  uint32_t* g = a.hist + (int64_t)row * kTopkBins;
  for (int b = threadIdx.x; b < kTopkBins; b += kCutThreads)
    if (H[b]) atomicAdd(g + b, H[b]);
}

// ------------------------------------------------------------------ k_cut

constexpr int kRankCap = 1024;  // bucket size ranked directly (a multiple of kCutThreads)

struct CutArgs {
  const float* scores;
  int64_t ld;
  const int64_t* seq_len;
  uint32_t* hist;              // [rows][kTopkBins] level-0 histograms of the middle keys
  const uint32_t* hist1;       // optional [rows][kTopkBins] level-1 histograms of the level-0 bucket
  unsigned long long* cand;    // [rows][kRankCap] candidate (key, ~index) values
  uint32_t* ctr;               // [rows][kSelCounters]: zero on entry, left zero
  unsigned long long* cut;     // [rows] out
  int32_t* status;
  int32_t rows_per_seq, k, n_sink, n_recent;
  int32_t build_hist;          // count hist here (zero on entry; cooperative launch) instead of reading it
  int32_t pending;             // tokens appended in this step but not yet in seq_len
  int32_t chunks_per_cta;      // consecutive chunks of kCutChunk keys per CTA (1 when build_hist)
  // optional (k_cut_stream): [rows][map_words] the chosen middle tokens, one
  // bit per token (bit x % 32 of word x / 32); words of tokens past n_max
  // are left as they are
  uint32_t* selmap;
  int64_t map_words;
};

struct __align__(16) CutSmem {
  uint32_t hist[kTopkBins];
  unsigned long long cand[kRankCap + 2];
  uint32_t warp_tot[32];
  uint32_t tot, tb, rem, nb, n_cand, is_last;
  unsigned long long cut;
};

// Radix levels over the 32-bit key: 12, 12 and 8 bits.
__device__ __forceinline__ int level_shift(int l) { return l == 0 ? 20 : (l == 1 ? 8 : 0); }
__device__ __forceinline__ int level_bins(int l) { return l == 2 ? 256 : kTopkBins; }

constexpr int kBinsPerThread = kTopkBins / kCutThreads;  // 16

// Descending bucket search.  Thread t holds the counts of bins top - r,
// r < kBinsPerThread, in h[r] (top = nbins - 1 - kBinsPerThread t; bins below
// 0 hold 0).  Finds the bin holding the rem-th largest key and the rank left
// within it: whole block (kCutThreads); writes S.tb, S.rem, S.nb.
__device__ void find_bucket(CutSmem& S, const uint32_t (&h)[kBinsPerThread], int top, uint32_t rem) {
  __syncthreads();  // every thread has read the previous call's S.tb, S.rem, S.nb
  if (threadIdx.x == 0) {
    S.tb = 0u;
    S.rem = 0u;
    S.nb = 0u;
  }
  uint32_t sum = 0;
#pragma unroll
  for (int r = 0; r < kBinsPerThread; ++r) sum += h[r];
  uint32_t ex = block_excl_scan(sum, S.warp_tot, &S.tot);
#pragma unroll
  for (int r = 0; r < kBinsPerThread; ++r) {
    if (ex < rem && rem <= ex + h[r]) {
      S.tb = (uint32_t)(top - r);
      S.rem = rem - ex;
      S.nb = h[r];
    }
    ex += h[r];
  }
  __syncthreads();
}

// The counts of this thread's bins (descending) from a histogram whose bins
// [0, nbins) are 16-byte aligned words.
__device__ __forceinline__ int bins_of_thread(const uint32_t* hist, int nbins, uint32_t (&h)[kBinsPerThread]) {
  const int top = nbins - 1 - kBinsPerThread * (int)threadIdx.x;
  const int base = top - (kBinsPerThread - 1);
  if (base < 0) {
#pragma unroll
    for (int r = 0; r < kBinsPerThread; ++r) h[r] = 0u;
    return top;
  }
  const uint4* p = reinterpret_cast<const uint4*>(hist + base);
#pragma unroll
  for (int i = 0; i < kBinsPerThread / 4; ++i) {
    const uint4 v = p[i];
    h[kBinsPerThread - 1 - 4 * i] = v.x;
    h[kBinsPerThread - 2 - 4 * i] = v.y;
    h[kBinsPerThread - 3 - 4 * i] = v.z;
    h[kBinsPerThread - 4 - 4 * i] = v.w;
  }
  return top;
}

// Rank S.cand[0..nc) by value and set S.cut to the rem-th largest.  S.cand is
// zero-padded to an even count (0 ranks below every candidate).  Small sets
// are ranked by counting; larger ones by a radix select (S.hist as its
// histogram).
__device__ __forceinline__ void rank_cut(CutSmem& S, int nc, uint32_t rem, int shared_bits) {
  if (nc > 128) {
    // radix select of the rem-th largest (the values are distinct), eight
    // bits at a time from the top below the shared_bits every value shares:
    // descend into the bin holding it until that bin holds it alone
    const int tid = threadIdx.x, lane = tid & 31;
    if (rem < 1 || (int)rem > nc) return;
    int fixed_lo = 64 - shared_bits;  // the bits from fixed_lo up are fixed in pre
    unsigned long long pre = fixed_lo >= 64 ? 0ull : (S.cand[0] & (~0ull << fixed_lo));
    uint32_t need = rem;
    while (true) {
      const int shift = max(fixed_lo - 8, 0);
      const uint32_t dmask = (1u << (fixed_lo - shift)) - 1u;
      for (int b = tid; b < 256; b += blockDim.x) S.hist[b] = 0u;
      __syncthreads();
      const unsigned long long hi_mask = fixed_lo >= 64 ? 0ull : (~0ull << fixed_lo);
      for (int e = tid; e < nc; e += blockDim.x) {
        const unsigned long long x = S.cand[e];
        if ((x & hi_mask) == pre) atomicAdd(&S.hist[(x >> shift) & dmask], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // bins from the top, 32 at a time: the bin where the running count reaches need
        uint32_t acc = 0;
        for (int base = 224; base >= 0; base -= 32) {
          const uint32_t c = S.hist[base + lane];
          uint32_t incl = c;  // keys in bins base + lane .. base + 31
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
            if (lane + o < 32) incl += y;
          }
          const uint32_t hit = __ballot_sync(0xffffffffu, acc + incl >= need && acc + incl - c < need);
          if (hit) {
            const int l = 31 - __clz(hit);
            if (lane == l) {
              S.tb = (uint32_t)(base + l);
              S.rem = need - (acc + incl - c);
              S.nb = c;
            }
            break;
          }
          acc += __shfl_sync(0xffffffffu, incl, 0);
        }
      }
      __syncthreads();
      pre |= (unsigned long long)S.tb << shift;
      need = S.rem;
      fixed_lo = shift;
      if (S.nb == 1u || fixed_lo == 0) break;
    }
    // the one value with the fixed bits
    const unsigned long long mask = ~0ull << fixed_lo;
    for (int e = tid; e < nc; e += blockDim.x)
      if ((S.cand[e] & mask) == pre) S.cut = S.cand[e];
    return;
  }
  const int nc2 = (nc + 1) & ~1;
  for (int e = threadIdx.x; e < nc; e += blockDim.x) {
    const unsigned long long mine = S.cand[e];
    uint32_t r0 = 0, r1 = 0, r2 = 0, r3 = 0;
    int j = 0;
    for (; j + 4 <= nc2; j += 4) {
      const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(&S.cand[j]);
      const ulonglong2 b = *reinterpret_cast<const ulonglong2*>(&S.cand[j + 2]);
      r0 += a.x > mine;
      r1 += a.y > mine;
      r2 += b.x > mine;
      r3 += b.y > mine;
    }
    for (; j < nc2; ++j) r0 += S.cand[j] > mine;
    if (r0 + r1 + r2 + r3 + 1 == rem) S.cut = mine;
  }
}

// The cut of a row whose bucket (key bits prefix at level lvl, S.nb keys)
// holds more than kRankCap keys, by one CTA streaming the row's middle keys.
__device__ void cut_refine(CutSmem& S, const float* __restrict__ sc, int64_t lo, int64_t cnt, uint32_t rem,
                           uint32_t prefix, int lvl) {
  const int tid = threadIdx.x;
  while (lvl < 2 && S.nb > (uint32_t)kRankCap) {
    const int nl = lvl + 1, pre_sh = level_shift(lvl), sh = level_shift(nl);
    const uint32_t bmask = (uint32_t)level_bins(nl) - 1u;
    __syncthreads();  // every thread has read S.nb
    for (int b = tid; b < kTopkBins; b += blockDim.x) S.hist[b] = 0u;
    __syncthreads();
    for_row_keys(sc, lo, 0, cnt, [&](int64_t, uint32_t key) {
      if ((key >> pre_sh) == prefix) atomicAdd(&S.hist[(key >> sh) & bmask], 1u);
    });
    __syncthreads();
    uint32_t h[kBinsPerThread];
    const int top = bins_of_thread(S.hist, level_bins(nl), h);
    find_bucket(S, h, top, rem);
    rem = S.rem;
    prefix = (prefix << (nl == 1 ? 12 : 8)) | S.tb;
    lvl = nl;
  }
  const int sh = level_shift(lvl);
  if (S.nb <= (uint32_t)kRankCap) {
    if (tid == 0) S.n_cand = 0;
    __syncthreads();
    for_row_keys(sc, lo, 0, cnt, [&](int64_t e, uint32_t key) {
      if ((key >> sh) == prefix) {
        const uint32_t c = atomicAdd(&S.n_cand, 1u);
        if (c < (uint32_t)kRankCap)
          S.cand[c] = ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)(lo + e));
      }
    });
    __syncthreads();
    const int nc = (int)min(S.n_cand, (uint32_t)kRankCap);
    if (tid == 0) S.cand[nc] = 0ull;
    __syncthreads();
    rank_cut(S, nc, rem, 32 - level_shift(lvl));
    return;
  }
  // a single key value tk repeated more than kRankCap times: its rem-th
  // occurrence in index order, 16 consecutive keys per thread
  const uint32_t tk = prefix;
  constexpr int kSeg = 16;
  uint32_t carry = 0;
  for (int64_t base = 0; base < cnt && carry < rem; base += (int64_t)kSeg * blockDim.x) {
    const int64_t e0 = base + (int64_t)tid * kSeg;
    uint32_t c = 0;
#pragma unroll
    for (int j = 0; j < kSeg; ++j)
      if (e0 + j < cnt && ordered_key(sc[lo + e0 + j]) == tk) ++c;
    const uint32_t ex = block_excl_scan(c, S.warp_tot, &S.tot) + carry;
    if (ex < rem && rem <= ex + c) {
      uint32_t need = rem - ex;
      for (int j = 0; j < kSeg && e0 + j < cnt; ++j) {
        if (ordered_key(sc[lo + e0 + j]) == tk && --need == 0) {
          S.cut = ((unsigned long long)tk << 32) | (0xFFFFFFFFu - (uint32_t)(lo + e0 + j));
          break;
        }
      }
    }
    carry += S.tot;
  }
}

// Wait until `count` CTAs have arrived at *bar (thread 0 of each CTA arrives
// once); bounded by `limit` rounds of ~100 ns, records BPKV_DEV_TIMEOUT if it
// gives up.  Whole block.
__device__ __forceinline__ void row_barrier(uint32_t* bar, uint32_t count, int32_t* status,
                                            uint32_t limit = kSpinLimit) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    uint32_t it = 0;
    while (*reinterpret_cast<volatile uint32_t*>(bar) < count) {
      if (++it > limit) {
        set_status(status, BPKV_DEV_TIMEOUT);
        break;
      }
      __nanosleep(100);
    }
    __threadfence();
  }
  __syncthreads();
}

// The end of a row's cut, by one CTA once every candidate of the row is
// written: it ranks the candidates, or refines a bucket of more than kRankCap
// keys, stores the cut, adds the bucket's chosen tokens to the selection map
// (when there is one) and clears the row's counters.  Whole block.
__device__ void cut_decide(CutSmem& S, const CutArgs& a, int row, const RowRange& r, const float* __restrict__ sc,
                           uint32_t* ctr, const unsigned long long* cand, uint32_t nb, uint32_t rem, uint32_t prefix,
                           int lvl) {
  const int tid = threadIdx.x;
  if (tid == 0) S.cut = ~0ull;
  uint32_t* mrow = a.selmap ? a.selmap + (int64_t)row * a.map_words : nullptr;
  if (nb <= (uint32_t)kRankCap) {
    // every candidate slot loaded beside the count (slots past it are unused)
    unsigned long long cv[kRankCap / kCutThreads];
#pragma unroll
    for (int i = 0; i < kRankCap / kCutThreads; ++i) cv[i] = __ldcg(cand + tid + kCutThreads * i);
    const int nc = (int)min(__ldcg(ctr), (uint32_t)kRankCap);
#pragma unroll
    for (int i = 0; i < kRankCap / kCutThreads; ++i)
      if (tid + kCutThreads * i < nc) S.cand[tid + kCutThreads * i] = cv[i];
    if (tid == 0) S.cand[nc] = 0ull;
    __syncthreads();
    rank_cut(S, nc, rem, 32 - level_shift(lvl));
    __syncthreads();
    if (mrow && S.cut != ~0ull) {
      // the bucket's chosen keys join the map (the keys above the bucket are in it)
      for (int e = tid; e < nc; e += kCutThreads) {
        const unsigned long long v = S.cand[e];
        if (v >= S.cut) {
          const uint32_t x = 0xFFFFFFFFu - (uint32_t)v;
          atomicOr(mrow + (x >> 5), 1u << (x & 31u));
        }
      }
    }
  } else {
    // refine in the shared histogram buffer
    if (tid == 0) S.nb = nb;
    __syncthreads();
    cut_refine(S, sc, r.lo, r.cnt, rem, prefix, lvl);
    __syncthreads();
    if (mrow && S.cut != ~0ull) {
      // the chosen keys of the streamed bucket join the map
      const int sh = level_shift(lvl);
      const unsigned long long cut = S.cut;
      const int64_t lo = r.lo;
      for_row_keys(sc, lo, 0, r.cnt, [&](int64_t e, uint32_t key) {
        const uint32_t x = (uint32_t)(lo + e);
        if ((key >> sh) == prefix && (((unsigned long long)key << 32) | (0xFFFFFFFFu - x)) >= cut)
          atomicOr(mrow + (x >> 5), 1u << (x & 31u));
      });
    }
  }
  __syncthreads();
  if (tid == 0) {
    a.cut[row] = S.cut;
    if (S.cut == ~0ull) set_status(a.status, BPKV_DEV_SELECT);  // histogram and keys disagree
#pragma unroll
    for (int i = 0; i < kSelCounters; ++i) ctr[i] = 0u;  // every CTA of the row is past its waits
  }
}

// The row's CTAs, after their part: the last one to arrive decides the cut
// (the barrier orders the CTA's candidate writes before thread 0's cumulative
// fence; the ticket is counter 1).
__device__ void cut_finish(CutSmem& S, const CutArgs& a, int row, const RowRange& r, const float* __restrict__ sc,
                           uint32_t* ctr, const unsigned long long* cand, uint32_t nb, uint32_t rem, uint32_t prefix,
                           int lvl) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    S.is_last = (atomicAdd(ctr + 1, 1u) == gridDim.x - 1) ? 1u : 0u;
    if (S.is_last) __threadfence();
  }
  __syncthreads();
  if (!S.is_last) return;
  cut_decide(S, a, row, r, sc, ctr, cand, nb, rem, prefix, lvl);
}

// Append this warp's matching keys (bit b of `match`: key keys[b] of token
// index idx0 + b * stride) to the row's candidate list: one returning atomic
// per warp for the warp's matches.  Whole warps.
__device__ __forceinline__ void append_matches(uint32_t match, const uint32_t (&keys)[kSelBatch], uint32_t idx0,
                                               uint32_t stride, uint32_t* ctr, unsigned long long* cand) {
  const int lane = threadIdx.x & 31;
  const uint32_t cnt = __popc(match);
  uint32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t warp_total = __shfl_sync(0xffffffffu, incl, 31);
  if (warp_total == 0u) return;  // uniform across the warp
  uint32_t base = 0;
  if (lane == 31) base = atomicAdd(ctr, warp_total);
  base = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
#pragma unroll
  for (int b = 0; b < kSelBatch; ++b) {
    if ((match >> b) & 1u) {
      if (base < (uint32_t)kRankCap)
        cand[base] = ((unsigned long long)keys[b] << 32) | (0xFFFFFFFFu - (idx0 + (uint32_t)b * stride));
      ++base;
    }
  }
}

// Cooperative form (the row's CTAs count the level-0 histogram themselves):
// grid (chunks of kCutChunk middle keys, rows), launched so that every CTA is
// resident; each thread holds kCutChunk / kCutThreads keys of its CTA's chunk.
__global__ void __launch_bounds__(kCutThreads, 2) k_cut(CutArgs a) {
  pdl_enter();
  __shared__ CutSmem S;
  const int row = blockIdx.y, tid = threadIdx.x;
  static_assert(kCutChunk == kSelBatch * kCutThreads, "one batch of loads per thread");
  const RowRange r = row_range(a.seq_len[row / a.rows_per_seq] + a.pending, a.k, a.n_sink, a.n_recent);
  if (r.cnt <= r.m || r.m == 0) {
    // every middle key, or none
    if (blockIdx.x == 0 && tid == 0) a.cut[row] = r.cnt <= r.m ? 0ull : ~0ull;
    return;
  }
  const float* sc = a.scores + (int64_t)row * a.ld;
  uint32_t* ctr = a.ctr + (int64_t)kSelCounters * row;
  unsigned long long* cand = a.cand + (int64_t)row * kRankCap;
  // this CTA's chunk; all loads in flight
  const int64_t c0 = (int64_t)blockIdx.x * kCutChunk, c1 = min64(c0 + kCutChunk, r.cnt);
  uint32_t keys[kSelBatch], valid = 0;
  {
    float v[kSelBatch];
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) v[b] = sc[r.lo + min64(c0 + tid + (int64_t)b * kCutThreads, c1 - 1)];
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b) {
      keys[b] = ordered_key(v[b]);
      if (c0 + tid + (int64_t)b * kCutThreads < c1) valid |= 1u << b;
    }
  }
  // level-0 histogram counted per CTA in shared memory, added to the row's
  // with one atomic per non-empty bin, then every CTA of the row waits for
  // the others (the grid is launched cooperatively)
  for (int b = tid; b < kTopkBins; b += kCutThreads) S.hist[b] = 0u;
  __syncthreads();
#pragma unroll
  for (int b = 0; b < kSelBatch; ++b)
    if ((valid >> b) & 1u) atomicAdd(&S.hist[keys[b] >> 20], 1u);
  __syncthreads();
  uint32_t* gh = a.hist + (int64_t)row * kTopkBins;
  for (int b = tid; b < kTopkBins; b += kCutThreads)
    if (S.hist[b]) atomicAdd(gh + b, S.hist[b]);
  row_barrier(ctr + 2, gridDim.x, a.status);
  uint32_t h[kBinsPerThread];
  const int top = bins_of_thread(reinterpret_cast<const uint32_t*>(gh), kTopkBins, h);
  find_bucket(S, h, top, (uint32_t)r.m);
  const uint32_t prefix = S.tb, nb = S.nb, rem = S.rem;
  if (nb <= (uint32_t)kRankCap) {
    uint32_t match = 0;
#pragma unroll
    for (int b = 0; b < kSelBatch; ++b)
      if (((valid >> b) & 1u) && (keys[b] >> 20) == prefix) match |= 1u << b;
    append_matches(match, keys, (uint32_t)(r.lo + c0 + tid), kCutThreads, ctr, cand);
  }
  cut_finish(S, a, row, r, sc, ctr, cand, nb, rem, prefix, 0);
}

// Streaming form (the row's bucket found by k_bucket, narrowed by the
// level-1 histogram on long rows): grid (chunks of kStreamChunk tokens in
// absolute position, rows); each thread loads kStreamVec 16-byte groups of
// scores (tokens 4 (t + 256 j) .. + 3 of the chunk) at once, then keeps the
// middle tokens whose key is in the bucket and appends them.  k_rank then
// decides each row's cut.
constexpr int kStreamVec = 8;                              // float4 loads per thread
constexpr int kStreamChunk = 4 * kStreamVec * kCutThreads;  // 8192 tokens per CTA
static_assert(kStreamVec == 8, "a thread's 32 tokens are eight nibbles of the selection map");

__global__ void __launch_bounds__(kCutThreads, 4) k_cut_stream(CutArgs a) {
  pdl_enter();
  const int row = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
  const float* sc = a.scores + (int64_t)row * a.ld;
  uint32_t* ctr = a.ctr + (int64_t)kSelCounters * row;
  unsigned long long* cand = a.cand + (int64_t)row * kRankCap;
  // the chunk's scores, the row's length and its bucket (k_bucket) read
  // together: none of the loads waits for another
  const uint32_t x0 = (uint32_t)blockIdx.x * kStreamChunk;  // the chunk's first token
  const uint32_t ld = (uint32_t)a.ld;
  const float4* p = reinterpret_cast<const float4*>(sc + x0);
  float4 v[kStreamVec];
#pragma unroll
  for (int j = 0; j < kStreamVec; ++j) {
    const uint32_t x = x0 + 4 * (tid + kCutThreads * j);
    v[j] = x < ld ? p[tid + kCutThreads * j] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int64_t n_row = a.seq_len[row / a.rows_per_seq];
  const uint32_t prefix = ctr[4], nb = ctr[6];
  const int lvl = (int)ctr[7];
  const RowRange r = row_range(n_row + a.pending, a.k, a.n_sink, a.n_recent);
  if (r.cnt <= r.m || r.m == 0) {
    if (blockIdx.x == 0 && tid == 0) a.cut[row] = r.cnt <= r.m ? 0ull : ~0ull;
    return;
  }
  // the bucket as an interval of floats: key(f) in [klo, khi] exactly when
  // flo <= f <= fhi, and key(f) > khi exactly when f > fhi (the
  // order-preserving key is monotone; -0 and +0 share a key, so a bucket
  // ending just below +0's key ends at the negative float nearest 0)
  const int sh = level_shift(lvl);
  const uint32_t klo = prefix << sh, khi = klo | ((1u << sh) - 1u);
  auto key_float = [](uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
  };
  const float flo = key_float(klo);
  const float fhi = khi == 0x7FFFFFFFu ? __uint_as_float(0x80000001u) : key_float(khi);
  const uint32_t lo = (uint32_t)r.lo, hi = (uint32_t)r.hi;
  // bit 4 j + e: token x0 + 4 (tid + 256 j) + e is a middle token in the
  // bucket (match) or above it (above: every such token is chosen)
  uint32_t match = 0, above = 0;
#pragma unroll
  for (int j = 0; j < kStreamVec; ++j) {
    const float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (f[e] > fhi) above |= 1u << (4 * j + e);
      else if (f[e] >= flo) match |= 1u << (4 * j + e);
    }
  }
  if (!(x0 >= lo && x0 + kStreamChunk <= hi)) {  // not every token of the chunk is a middle token
    uint32_t mid = 0;
#pragma unroll
    for (int j = 0; j < kStreamVec; ++j) {
      const uint32_t x = x0 + 4 * (tid + kCutThreads * j);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (x + e >= lo && x + e < hi) mid |= 1u << (4 * j + e);
    }
    match &= mid;
    above &= mid;
  }
  if (a.selmap) {
    // the map's words of this chunk (the last CTA adds the bucket's chosen
    // tokens): word (x0 + 1024 j) / 32 + tid / 8 is nibble j of lanes
    // 8 (lane / 8) .. + 7, so an 8 x 8 nibble transpose within each group of
    // eight lanes leaves word j = lane % 8 in each lane
    uint32_t w = above;
    const int l8 = lane & 7;
    {
      const uint32_t p = __shfl_xor_sync(0xffffffffu, w, 4);
      w = (l8 & 4) ? ((w & 0xFFFF0000u) | (p >> 16)) : ((w & 0x0000FFFFu) | (p << 16));
    }
    {
      const uint32_t p = __shfl_xor_sync(0xffffffffu, w, 2);
      w = (l8 & 2) ? ((w & 0xFF00FF00u) | ((p >> 8) & 0x00FF00FFu)) : ((w & 0x00FF00FFu) | ((p << 8) & 0xFF00FF00u));
    }
    {
      const uint32_t p = __shfl_xor_sync(0xffffffffu, w, 1);
      w = (l8 & 1) ? ((w & 0xF0F0F0F0u) | ((p >> 4) & 0x0F0F0F0Fu)) : ((w & 0x0F0F0F0Fu) | ((p << 4) & 0xF0F0F0F0u));
    }
    const uint32_t xw = x0 + 1024u * (uint32_t)l8 + 32u * (uint32_t)(tid >> 3);  // the word's first token
    if (xw < ld) a.selmap[(int64_t)row * a.map_words + (xw >> 5)] = w;
  }
  if (nb <= (uint32_t)kRankCap) {
    const uint32_t cnt = __popc(match);
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t warp_total = __shfl_sync(0xffffffffu, incl, 31);
    if (warp_total != 0u) {  // uniform across the warp
      uint32_t base = 0;
      if (lane == 31) base = atomicAdd(ctr, warp_total);
      base = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
      // the few matches, their scores read again (cached)
      while (match) {
        const int b = __ffs(match) - 1;
        match &= match - 1u;
        const uint32_t x = x0 + 4 * (tid + kCutThreads * (b >> 2)) + (b & 3);
        if (base < (uint32_t)kRankCap) cand[base] = ((unsigned long long)ordered_key(sc[x]) << 32) | (0xFFFFFFFFu - x);
        ++base;
      }
    }
  }
}

// After k_cut_stream, one CTA per row: the row's cut (cut_decide).
__global__ void __launch_bounds__(kCutThreads) k_rank(CutArgs a) {
  pdl_enter();
  __shared__ CutSmem S;
  const int row = blockIdx.x;
  const RowRange r = row_range(a.seq_len[row / a.rows_per_seq] + a.pending, a.k, a.n_sink, a.n_recent);
  if (r.cnt <= r.m || r.m == 0) return;  // k_cut_stream stored these rows' cuts
  uint32_t* ctr = a.ctr + (int64_t)kSelCounters * row;
  const uint32_t prefix = ctr[4], rem = ctr[5], nb = ctr[6];
  const int lvl = (int)ctr[7];
  cut_decide(S, a, row, r, a.scores + (int64_t)row * a.ld, ctr, a.cand + (int64_t)row * kRankCap, nb, rem, prefix, lvl);
}

// ------------------------------------------------------------------ k_bucket

// Per row (one CTA each), kLevel 0: the level-0 bucket holding the m-th
// largest middle key, from the row's counted histogram, stored in the row's
// counters [4 .. 7] (key prefix, rank left in the bucket, keys in the bucket,
// level) for k_hist1 and k_cut_stream, so that their many CTAs need not each
// read and scan the 4096 bins.  kLevel 1 (long rows, after k_hist1): a bucket
// of more than kRankCap keys narrowed by its level-1 histogram.
template <int kLevel>
__global__ void __launch_bounds__(kCutThreads) k_bucket(CutArgs a) {
  pdl_enter();
  __shared__ CutSmem S;
  const int row = blockIdx.x;
  uint32_t* ctr = a.ctr + (int64_t)kSelCounters * row;
  if (kLevel == 1 && ctr[6] <= (uint32_t)kRankCap) return;  // small enough to rank (or no bucket)
  uint32_t h[kBinsPerThread];
  const int top = bins_of_thread((kLevel == 1 ? a.hist1 : a.hist) + (int64_t)row * kTopkBins, kTopkBins, h);
  const RowRange r = row_range(a.seq_len[row / a.rows_per_seq] + a.pending, a.k, a.n_sink, a.n_recent);
  if (r.cnt <= r.m || r.m == 0) return;  // k_cut_stream decides these rows without a bucket
  find_bucket(S, h, top, kLevel == 1 ? ctr[5] : (uint32_t)r.m);
  if (threadIdx.x == 0) {
    ctr[4] = kLevel == 1 ? (ctr[4] << 12) | S.tb : S.tb;
    ctr[5] = S.rem;
    ctr[6] = S.nb;
    ctr[7] = (uint32_t)kLevel;
  }
}

// ------------------------------------------------------------------ k_hist1

// Level-1 histogram (key bits 19..8) of the keys in each long row's level-0
// bucket, counted by all CTAs of the row over their runs of chunks.  Grid
// (runs, rows); rows whose bucket needs no refinement return at once.
__global__ void __launch_bounds__(kCutThreads, 2) k_hist1(CutArgs a) {
  pdl_enter();
  __shared__ CutSmem S;
  const int row = blockIdx.y, tid = threadIdx.x;
  const RowRange r = row_range(a.seq_len[row / a.rows_per_seq] + a.pending, a.k, a.n_sink, a.n_recent);
  const int64_t e0 = (int64_t)blockIdx.x * a.chunks_per_cta * kCutChunk;
  const int64_t e1 = min64(e0 + (int64_t)a.chunks_per_cta * kCutChunk, r.cnt);
  if (r.cnt <= r.m || r.m == 0 || e0 >= e1) return;
  const uint32_t* ctr = a.ctr + (int64_t)kSelCounters * row;  // the row's bucket (k_bucket)
  const uint32_t tb = ctr[4];
  if (ctr[6] <= (uint32_t)kRankCap) return;
  for (int b = tid; b < kTopkBins; b += kCutThreads) S.hist[b] = 0u;
  __syncthreads();
  for_row_keys(a.scores + (int64_t)row * a.ld, r.lo, e0, e1, [&](int64_t, uint32_t key) {
    if ((key >> 20) == tb) atomicAdd(&S.hist[(key >> 8) & 0xFFFu], 1u);
  });
  __syncthreads();
  uint32_t* g1 = const_cast<uint32_t*>(a.hist1) + (int64_t)row * kTopkBins;
  for (int b = tid; b < kTopkBins; b += kCutThreads)
    if (S.hist[b]) atomicAdd(g1 + b, S.hist[b]);
}

// ------------------------------------------------------------------ k_lists

struct ListArgs {
  const float* scores;
  int64_t ld;
  const int64_t* seq_len;
  const unsigned long long* cut;
  int32_t* idx;  // [rows][k]
  int32_t* status;
  int32_t rows_per_seq, k, n_sink, n_recent;
  int32_t pending;  // tokens appended in this step but not yet in seq_len
};

struct ListSmem {
  uint32_t keys[kTileKeys];
  uint32_t warp_tot[32];
  uint32_t tot;
};

// Index lists from the cuts: sinks, the chosen middle tokens, the recent
// tokens, ascending, -1 padded.  One CTA (kSelThreads) per row.
__global__ void __launch_bounds__(kSelThreads) k_lists(ListArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char list_raw[];
  ListSmem& S = *reinterpret_cast<ListSmem*>(list_raw);
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const RowRange r = row_range(a.seq_len[row / a.rows_per_seq] + a.pending, a.k, a.n_sink, a.n_recent);
  const float* sc = a.scores + (int64_t)row * a.ld;
  int32_t* out = a.idx + (int64_t)row * a.k;
  const int64_t n_mid = r.cnt <= r.m ? r.cnt : r.m;
  for (int64_t i = tid; i < r.lo; i += kSelThreads) out[i] = (int32_t)i;
  for (int64_t e = tid; e < r.n - r.hi; e += kSelThreads) out[r.lo + n_mid + e] = (int32_t)(r.hi + e);
  for (int64_t e = r.lo + n_mid + (r.n - r.hi) + tid; e < a.k; e += kSelThreads) out[e] = -1;
  if (r.cnt <= r.m) {
    for (int64_t e = tid; e < r.cnt; e += kSelThreads) out[r.lo + e] = (int32_t)(r.lo + e);
    return;
  }
  if (r.m == 0) return;
  const unsigned long long cut = a.cut[row];
  const uint32_t ck = (uint32_t)(cut >> 32), ci = 0xFFFFFFFFu - (uint32_t)cut;
  uint32_t carry = 0;
  for (int64_t t0 = 0; t0 < r.cnt; t0 += kTileKeys) {
    const int len = (int)min64(kTileKeys, r.cnt - t0);
    __syncthreads();  // the previous tile's readers are done
    for_row_keys(sc, r.lo + t0, 0, len, [&](int64_t e, uint32_t key) { S.keys[e] = key; });
    __syncthreads();
    // thread = segment of seg consecutive keys, read rotated by lane (no bank conflicts)
    const int seg = (len + kSelThreads - 1) / kSelThreads, start = tid * seg;
    uint32_t mask = 0;
    for (int j = 0; j < seg; ++j) {
      int jj = j + lane % seg;
      if (jj >= seg) jj -= seg;
      const int e = start + jj;
      if (e < len) {
        const uint32_t key = S.keys[e];
        const uint32_t i = (uint32_t)(r.lo + t0 + e);
        if (key > ck || (key == ck && i <= ci)) mask |= 1u << jj;
      }
    }
    const uint32_t ex = block_excl_scan((uint32_t)__popc(mask), S.warp_tot, &S.tot) + carry;
    int32_t* o = out + r.lo + ex;
    int64_t room = n_mid - ex;
    while (mask && room-- > 0) {
      const int b = __ffs(mask) - 1;
      mask &= mask - 1u;
      *o++ = (int32_t)(r.lo + t0 + start + b);
    }
    carry += S.tot;
  }
  if (carry != (uint32_t)n_mid) {
    if (tid == 0) set_status(a.status, BPKV_DEV_SELECT);
    for (int64_t e = min64(carry, n_mid) + tid; e < n_mid; e += kSelThreads) out[r.lo + e] = -1;
  }
}

// ------------------------------------------------------------------ launchers

int64_t cut_chunks(const bpkv_cache& c) {
  const int64_t ch = (c.n_max + kCutChunk - 1) / kCutChunk;
  return ch < 1 ? 1 : ch;
}

size_t cut_scratch_bytes(const bpkv_cache& c) {
  const size_t rows = (size_t)c.n_seq * c.n_kv_heads * c.group;
  return rows * ((size_t)kRankCap * 8 + kSelCounters * 4 + 8);
}

// Resident CTAs of k_cut on the current device (looked up once per device); 0 if unknown.
int cut_slots() {
  constexpr int kDevs = 64;
  static int slots[kDevs] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (slots[dev] == 0) {
    int sms = 0, per_sm = 0, coop = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_cut, kCutThreads, 0) != cudaSuccess) return 0;
    slots[dev] = (coop && sms * per_sm > 0) ? sms * per_sm : -1;
  }
  return slots[dev] > 0 ? slots[dev] : 0;
}

// Resident CTAs of a histogram kernel (k_hist: which 0, k_hist1: which 1) on
// the current device (looked up once per device); 4 per SM of 152 if unknown.
int64_t hist_slots(int which) {
  constexpr int kDevs = 64;
  static int slots[2][kDevs] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return 4 * 152;
  std::lock_guard<std::mutex> lock(mu);
  if (slots[which][dev] == 0) {
    int sms = 0, per_sm = 0;
    const cudaError_t e = which == 0
                              ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_hist, kCutThreads, 0)
                              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_hist1, kCutThreads, 0);
    if (e != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 4 * 152;
    slots[which][dev] = sms * per_sm > 0 ? sms * per_sm : 4 * 152;
  }
  return slots[which][dev];
}

// Chunks per CTA of a histogram kernel: about two waves of its resident
// CTAs, so that each CTA streams few chunks (one dependent round of loads
// each) and flushes its bins once.
int32_t hist_chunks_per_cta(const bpkv_cache& c, int which) {
  const int64_t rows = (int64_t)c.n_seq * c.n_kv_heads * c.group, chunks = cut_chunks(c);
  const int64_t slots = 2 * hist_slots(which);
  const int64_t cpc = (chunks * rows + slots - 1) / slots;
  return (int32_t)(cpc < 1 ? 1 : cpc);
}

dim3 run_grid(const bpkv_cache& c, int32_t cpc) {
  return dim3((unsigned)((cut_chunks(c) + cpc - 1) / cpc), (unsigned)(c.n_seq * c.n_kv_heads * c.group));
}

cudaError_t launch_hist(const bpkv_cache& c, const float* scores, int64_t ld, int32_t k, int32_t n_sink,
                        int32_t n_recent, uint32_t* hist, int32_t pending, cudaStream_t st) {
  const int32_t cpc = hist_chunks_per_cta(c, 0);
  HistArgs a{scores, ld, c.seq_len, hist, c.n_kv_heads * c.group, k, n_sink, n_recent, pending, cpc};
  return launch_pdl(k_hist, run_grid(c, cpc), dim3(kCutThreads), 0, st, a);
}

// Whether the cut kernel can count the level-0 histograms itself: its grid
// (one CTA per chunk and row) must be resident at once (cooperative launch).
bool cut_counts_hist(const bpkv_cache& c) {
  const int n = cut_slots();
  const int64_t grid = cut_chunks(c) * (int64_t)c.n_seq * c.n_kv_heads * c.group;
  return n > 0 && grid <= n;
}

// Whether the scan kernel should count the level-0 histograms as it writes
// the scores (when the cut cannot): the pinned-host scan (its link-bound loop
// hides the atomics) and the device-side scan for groups of up to 4 query
// heads (in shared memory); otherwise k_hist counts them from the scores.
bool scan_counts_hist(const bpkv_cache& c) { return !cut_counts_hist(c) && (c.residency == 1 || c.group <= 4); }

// Rows long enough that the level-0 bucket usually exceeds kRankCap keys get
// a parallel level-1 histogram (k_hist1) before the cut.
bool long_rows(const bpkv_cache& c) { return c.n_max >= kLongRowTokens; }

// selmap (optional, streaming form only): the chosen middle tokens' bits,
// [rows][ld / 32] words (ld a multiple of 32).
cudaError_t launch_cut(const bpkv_cache& c, const float* scores, int64_t ld, int32_t k, int32_t n_sink,
                       int32_t n_recent, const SelBufs& b, bool build_hist, int32_t pending, int32_t* status,
                       cudaStream_t st, uint32_t* selmap) {
  const bool l1 = !build_hist && long_rows(c);
  const int32_t cpc = build_hist ? 1 : hist_chunks_per_cta(c, 1);  // k_hist1's runs
  CutArgs a{scores,   ld,           c.seq_len, b.hist, l1 ? b.hist1 : nullptr, b.cand, b.ctr, b.cut, status,
            c.n_kv_heads * c.group, k, n_sink, n_recent, build_hist ? 1 : 0, pending, cpc,
            build_hist ? nullptr : selmap, ld / 32};
  if (build_hist) return launch_coop_pdl(k_cut, run_grid(c, 1), dim3(kCutThreads), 0, st, a);
  // each row's bucket once, then (long rows) the level-1 histogram and the
  // bucket narrowed by it, then the streaming filter and each row's rank
  const dim3 rows((unsigned)(c.n_seq * c.n_kv_heads * c.group));
  cudaError_t e = launch_pdl(k_bucket<0>, rows, dim3(kCutThreads), 0, st, a);
  if (e != cudaSuccess) return e;
  if (l1) {
    e = launch_pdl(k_hist1, run_grid(c, cpc), dim3(kCutThreads), 0, st, a);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k_bucket<1>, rows, dim3(kCutThreads), 0, st, a);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid((unsigned)((c.n_max + kStreamChunk - 1) / kStreamChunk), rows.x);
  e = launch_pdl(k_cut_stream, grid, dim3(kCutThreads), 0, st, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_rank, rows, dim3(kCutThreads), 0, st, a);
}

cudaError_t launch_lists(const bpkv_cache& c, const float* scores, int64_t ld, int32_t k, int32_t n_sink,
                         int32_t n_recent, const unsigned long long* cut, int32_t* idx, int32_t* status,
                         int32_t pending, cudaStream_t st) {
  ListArgs a{scores, ld, c.seq_len, cut, idx, status, c.n_kv_heads * c.group, k, n_sink, n_recent, pending};
  const int smem = (int)sizeof(ListSmem);
  cudaError_t e = cudaFuncSetAttribute(k_lists, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_lists, dim3(c.n_seq * c.n_kv_heads * c.group), dim3(kSelThreads), smem, st, a);
}

// Top-k of every row: the cuts into b.cut and, when idx is given, the index
// lists.  Histograms still to be counted are counted by the cut kernel itself
// (cooperative launch) or, when its grid cannot be resident at once, by k_hist
// first.  selmap: see launch_cut (written when the cut is not the cooperative
// one, i.e. when !cut_counts_hist(c) or the histograms come counted).
cudaError_t launch_topk(const bpkv_cache& c, const float* scores, int64_t ld, int32_t k, int32_t n_sink,
                        int32_t n_recent, const SelBufs& b, HistState hs, int32_t* idx, int32_t* status,
                        cudaStream_t st, int32_t pending, uint32_t* selmap) {
  cudaError_t e;
  bool build = false;
  if (hs == HistState::kDirty) {
    const size_t rows = (size_t)c.n_seq * c.n_kv_heads * c.group;
    e = cudaMemsetAsync(b.hist, 0, rows * (2 * kTopkBins + kSelCounters) * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
  }
  if (hs != HistState::kCounted) {
    build = cut_counts_hist(c);
    if (!build) {
      e = launch_hist(c, scores, ld, k, n_sink, n_recent, b.hist, pending, st);
      if (e != cudaSuccess) return e;
    }
  }
  e = launch_cut(c, scores, ld, k, n_sink, n_recent, b, build, pending, status, st, selmap);
  if (e != cudaSuccess || !idx) return e;
  return launch_lists(c, scores, ld, k, n_sink, n_recent, b.cut, idx, status, pending, st);
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


// Self-test of the bounded wait: one CTA arrives at a fresh barrier that
// expects `count` arrivals and waits there as the cut's CTAs do (nothing else
// arrives when count > 1, so the wait runs out after `limit` rounds and
// records BPKV_DEV_TIMEOUT).
__global__ void k_selftest_wait(uint32_t* bar, uint32_t count, uint32_t limit, int32_t* status) {
  if (threadIdx.x == 0) *bar = 0u;
  row_barrier(bar, count, status, limit);
}

cudaError_t launch_selftest_wait(uint32_t* bar, uint32_t count, uint32_t limit, int32_t* status, cudaStream_t st) {
  k_selftest_wait<<<1, 32, 0, st>>>(bar, count, limit, status);
  return cudaGetLastError();
}

}  // namespace bpkv
