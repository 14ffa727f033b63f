// Selection, GQA union and sparse attention of one decode pass in a single
// cluster kernel per (sequence, KV head), after the scan has written the scores
// (Fathom page, section 2: sinks + recent + per-head top (k - 36), exact
// attention over each head's selection; sections 1 and 3.1: the union of the
// G heads' winners is fetched once).
//
// CTA r of the cluster owns tokens [r T, (r + 1) T).  Steps:
//   1. sinks and recent tokens of its range go to its entry list with every head
//      bit;                                                  -- cluster barrier
//   2. per query head it selects its local top-(k - 36) candidates (exact: key
//      desc, index asc) and copies them to the head's leader (CTA g);
//                                                            -- cluster barrier
//   3. each leader selects the global winners among the merged local winners
//      (the global top set lies in their union) and appends (token, head bit)
//      to the owner CTA's entry list;                        -- cluster barrier
//   4. each CTA sorts its entries by token and merges equal tokens: its share
//      of the union, ascending, with head masks; per-head counts are published;
//                                                            -- cluster barrier
//   5. the ascending index list of every head is written at prefix offsets,
//      each CTA attends over its union rows (each row read once for all heads)
//      and publishes per-head (max, sum, output) partials;   -- cluster barrier
//   6. each leader merges its head's partials by log-sum-exp. -- final barrier
// Entries hold the token offset in the CTA's range in bits 8..31 and the head
// bits in bits 0..7, so sorting them as integers orders them by token.
#include "cluster_core.cuh"

namespace cg = cooperative_groups;

namespace bpkv {

constexpr int kTailCS = 8;
constexpr int kTailMaxList = 8192;

struct TailArgs {
  const float* scores;
  int64_t ld;
  const uint16_t* k_rows;
  const uint16_t* v_rows;
  const int64_t* seq_len;
  int64_t cap;
  int32_t n_heads, group;
  const float* q;
  int32_t k, n_sink, n_recent;
  float* out;          // [N][H][G][D]
  int32_t* idx_out;    // optional [N][H][G][k]
  int32_t tpc;         // tokens per CTA (multiple of 64)
  int32_t list_cap;    // entries of each CTA's list (power of two)
  int32_t merge_cap;   // entries of each leader's merge buffer
};

template <int GP>
struct TailSmem {
  float part[GP][kD + 2];
  uint32_t head_cnt[BPKV_MAX_GROUP];
  uint32_t merge_n[BPKV_MAX_GROUP];
  uint32_t n_list, n_rows;
  uint32_t tile_cnt[kClThreads / 32][BPKV_MAX_GROUP];
  union {
    SelScratch sel;
    struct {
      int32_t rows[kTailMaxList];
      uint8_t rmask[kTailMaxList];
      AttScratch a;
    } att;
  } x;
  // followed by: list[list_cap] (uint32), merge[merge_cap] (uint64)
};

template <int GP>
__global__ void __launch_bounds__(kClThreads) k_select_attend(TailArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char tail_raw[];
  TailSmem<GP>& S = *reinterpret_cast<TailSmem<GP>*>(tail_raw);
  uint32_t* list = reinterpret_cast<uint32_t*>(tail_raw + sizeof(TailSmem<GP>));
  unsigned long long* merge = reinterpret_cast<unsigned long long*>(list + a.list_cap);
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int h = blockIdx.y, s = blockIdx.z;
  const int64_t unit = (int64_t)s * a.n_heads + h;
  const int G = a.group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = a.seq_len[s];
  const int T = a.tpc;
  const int64_t t_begin = (int64_t)rank * T;
  const int n_own = (int)max64(0, min64(t_begin + T, n) - t_begin);
  const int64_t lo = min64(a.n_sink, n);
  const int64_t hi = max64(n - a.n_recent, lo);
  const int n_top = max(a.k - a.n_sink - a.n_recent, 0);
  const bool take_all = (hi - lo) <= n_top;
  const int ca = (int)min64(max64(lo - t_begin, 0), n_own);
  const int cb = (int)min64(max64(hi - t_begin, 0), n_own);
  const uint32_t all_bits = (1u << G) - 1u;

  if (tid < BPKV_MAX_GROUP) {
    S.head_cnt[tid] = 0;
    S.merge_n[tid] = 0;
  }
  if (tid == 0) S.n_list = 0;
  __syncthreads();
  // ---- 1. fixed tokens (every token when all are kept)
  if (take_all) {
    for (int x = tid; x < n_own; x += kClThreads) {
      const uint32_t p = atomicAdd(&S.n_list, 1u);
      if (p < (uint32_t)a.list_cap) list[p] = ((uint32_t)x << 8) | all_bits;
    }
  } else {
    for (int x = tid; x < ca; x += kClThreads) {
      const uint32_t p = atomicAdd(&S.n_list, 1u);
      if (p < (uint32_t)a.list_cap) list[p] = ((uint32_t)x << 8) | all_bits;
    }
    for (int x = cb + tid; x < n_own; x += kClThreads) {
      const uint32_t p = atomicAdd(&S.n_list, 1u);
      if (p < (uint32_t)a.list_cap) list[p] = ((uint32_t)x << 8) | all_bits;
    }
  }
  cluster.sync();

  // ---- 2. local candidates per head, copied to the head's leader
  if (!take_all && n_top > 0) {
    for (int g = 0; g < G; ++g) {
      const float* sg = a.scores + (unit * G + g) * a.ld + t_begin;
      if (tid == 0) S.x.sel.n_win = 0;
      __syncthreads();
      cta_select(
          S.x.sel, cb - ca, n_top,
          [&](int e) -> unsigned long long {
            return sel_entry(ordered_key(sg[ca + e]), (uint32_t)(t_begin + ca + e));
          },
          [&](unsigned long long v) { S.x.sel.win[atomicAdd(&S.x.sel.n_win, 1u)] = v; });
      __syncthreads();
      const int nw = (int)S.x.sel.n_win;
      __shared__ uint32_t base_sh;
      if (tid == 0) base_sh = atomicAdd(cluster.map_shared_rank(&S.merge_n[g], g), (unsigned int)nw);
      __syncthreads();
      unsigned long long* rbuf = cluster.map_shared_rank(merge, g);
      for (int e = tid; e < nw; e += kClThreads)
        if (base_sh + e < (uint32_t)a.merge_cap) rbuf[base_sh + e] = S.x.sel.win[e];
      __syncthreads();
    }
  }
  cluster.sync();

  // ---- 3. leaders pick the global winners of their head
  if (!take_all && n_top > 0 && rank < G) {
    const int g = rank;
    const int cnt = (int)min(S.merge_n[g], (uint32_t)a.merge_cap);
    cta_select(
        S.x.sel, cnt, n_top, [&](int e) -> unsigned long long { return merge[e]; },
        [&](unsigned long long v) {
          const uint32_t tok = entry_tok(v);
          const int owner = (int)(tok / (uint32_t)T);
          const uint32_t x = tok - (uint32_t)owner * (uint32_t)T;
          const uint32_t p = atomicAdd(cluster.map_shared_rank(&S.n_list, owner), 1u);
          if (p < (uint32_t)a.list_cap) cluster.map_shared_rank(list, owner)[p] = (x << 8) | (1u << g);
        });
  }
  cluster.sync();

  // ---- 4. sort the entries by token and merge equal tokens into union rows
  const int nl = (int)min(S.n_list, (uint32_t)a.list_cap);
  {
    const int n2 = pow2_ge(max(nl, 2));
    for (int e = nl + tid; e < n2; e += kClThreads) list[e] = 0xFFFFFFFFu;
    __syncthreads();
    cta_bitonic(list, n2, false);
    if (tid == 0) S.n_rows = 0;
    __syncthreads();
    uint32_t carry = 0;
    for (int base = 0; base < nl; base += kClThreads) {
      const int i = base + tid;
      uint32_t first = 0, bits = 0;
      if (i < nl) {
        const uint32_t tok = list[i] >> 8;
        first = (i == 0 || (list[i - 1] >> 8) != tok) ? 1u : 0u;
        if (first)
          for (int j = i; j < nl && (list[j] >> 8) == tok; ++j) bits |= list[j] & 0xffu;
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, first);
      if (lane == 0) S.tile_cnt[warp][0] = __popc(bal);
      __syncthreads();
      uint32_t off = carry;
      for (int w = 0; w < warp; ++w) off += S.tile_cnt[w][0];
      off += __popc(bal & ((1u << lane) - 1u));
      if (first) {
        S.x.att.rows[off] = (int32_t)(list[i] >> 8);
        S.x.att.rmask[off] = (uint8_t)bits;
      }
      uint32_t tile = 0;
      for (int w = 0; w < kClThreads / 32; ++w) tile += S.tile_cnt[w][0];
      carry += tile;
      __syncthreads();
    }
    if (tid == 0) S.n_rows = carry;
    // per-head counts of this CTA's rows
    uint32_t c[BPKV_MAX_GROUP];
#pragma unroll
    for (int g = 0; g < BPKV_MAX_GROUP; ++g) c[g] = 0;
    for (int r = tid; r < (int)carry; r += kClThreads) {
      const uint32_t mk = S.x.att.rmask[r];
#pragma unroll
      for (int g = 0; g < BPKV_MAX_GROUP; ++g) c[g] += (mk >> g) & 1u;
    }
#pragma unroll
    for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
      uint32_t v = c[g];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && g < G && v) atomicAdd(&S.head_cnt[g], v);
    }
  }
  cluster.sync();
  const int nrows = (int)S.n_rows;

  // ---- 5. ordered index lists, then attention over this CTA's rows
  if (a.idx_out) {
    uint32_t before[BPKV_MAX_GROUP], total[BPKV_MAX_GROUP];
    for (int g = 0; g < G; ++g) {
      before[g] = 0;
      total[g] = 0;
      for (int r = 0; r < kTailCS; ++r) {
        const uint32_t v = *cluster.map_shared_rank(&S.head_cnt[g], r);
        if (r < rank) before[g] += v;
        total[g] += v;
      }
    }
    for (int base = 0; base < nrows; base += kClThreads) {
      const int r = base + tid;
      const uint32_t mk = r < nrows ? S.x.att.rmask[r] : 0u;
      uint32_t bal[BPKV_MAX_GROUP];
#pragma unroll
      for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
        bal[g] = __ballot_sync(0xffffffffu, (mk >> g) & 1u);
        if (lane == 0) S.tile_cnt[warp][g] = __popc(bal[g]);
      }
      __syncthreads();
      for (int g = 0; g < G; ++g) {
        uint32_t off = before[g];
        for (int w = 0; w < warp; ++w) off += S.tile_cnt[w][g];
        off += __popc(bal[g] & ((1u << lane) - 1u));
        if (((mk >> g) & 1u) && off < (uint32_t)a.k)
          a.idx_out[(unit * G + g) * a.k + off] = (int32_t)(t_begin + S.x.att.rows[r]);
        uint32_t tile = 0;
        for (int w = 0; w < kClThreads / 32; ++w) tile += S.tile_cnt[w][g];
        before[g] += tile;
      }
      __syncthreads();
    }
    if (rank == kTailCS - 1)
      for (int g = 0; g < G; ++g)
        for (int p = (int)total[g] + tid; p < a.k; p += kClThreads) a.idx_out[(unit * G + g) * a.k + p] = -1;
  }
  {
    const int64_t rb = unit * a.cap * kD + t_begin * kD;
    attend_rows<GP>(S.x.att.a, S.x.att.rows, S.x.att.rmask, nrows, a.k_rows + rb, a.v_rows + rb,
                    a.q + unit * G * kD, G, S.part);
  }
  cluster.sync();

  // ---- 6. leaders merge their head's partials
  if (rank < G) merge_partials<kTailCS>(cluster, S.part, rank, a.out + (unit * G + rank) * kD);
  cluster.sync();
}

namespace {

int tail_tpc(const bpkv_cache& c) {
  const int64_t nb = (c.n_max + kBlock - 1) / kBlock;
  return (int)((nb + kTailCS - 1) / kTailCS) * kBlock;
}

int tail_gp(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8; }

template <int GP>
size_t tail_smem(int list_cap, int merge_cap) {
  return sizeof(TailSmem<GP>) + (size_t)list_cap * 4 + (size_t)merge_cap * 8;
}

size_t tail_smem_any(int gp, int list_cap, int merge_cap) {
  return gp == 1 ? tail_smem<1>(list_cap, merge_cap) : gp == 2 ? tail_smem<2>(list_cap, merge_cap)
       : gp == 4 ? tail_smem<4>(list_cap, merge_cap) : tail_smem<8>(list_cap, merge_cap);
}

void tail_caps(const bpkv_cache& c, int32_t k, int32_t n_sink, int32_t n_recent, int* list_cap, int* merge_cap) {
  const int n_top = max(k - n_sink - n_recent, 0);
  int need = c.group * n_top + n_sink + n_recent + 64;
  if (need < k + 64) need = k + 64;
  int p = 2;
  while (p < need) p <<= 1;
  *list_cap = p;
  *merge_cap = kTailCS * max(n_top, 1);
}

template <int GP>
cudaError_t launch_tail_gp(const TailArgs& a, dim3 grid, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(k_select_attend<GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kTailCS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_select_attend<GP>, a);
}

}  // namespace

// Whether the cluster tail can run this pass: G fits the cluster, the tokens
// per CTA fit the 24-bit entry offsets, k fits the merge buffers and the lists
// fit shared memory.
bool tail_eligible(const bpkv_cache& c, int32_t k, int32_t n_sink, int32_t n_recent) {
  if (c.group > kTailCS) return false;
  if (k - n_sink - n_recent > kClMaxTop) return false;
  if (tail_tpc(c) >= (1 << 24)) return false;
  int list_cap = 0, merge_cap = 0;
  tail_caps(c, k, n_sink, n_recent, &list_cap, &merge_cap);
  if (list_cap > kTailMaxList) return false;
  int dev = 0, max_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
  return tail_smem_any(tail_gp(c.group), list_cap, merge_cap) <= (size_t)max_smem;
}

cudaError_t launch_select_attend(const bpkv_cache& c, const float* scores, int64_t ld, const float* q, int32_t k,
                                 int32_t n_sink, int32_t n_recent, float* out, int32_t* idx_out, cudaStream_t st) {
  int list_cap = 0, merge_cap = 0;
  tail_caps(c, k, n_sink, n_recent, &list_cap, &merge_cap);
  TailArgs a{scores, ld, c.k_rows, c.v_rows, c.seq_len, c.cap_tokens, c.n_kv_heads, c.group, q, k, n_sink,
             n_recent, out, idx_out, tail_tpc(c), list_cap, merge_cap};
  const int gp = tail_gp(c.group);
  const size_t smem = tail_smem_any(gp, list_cap, merge_cap);
  dim3 grid(kTailCS, c.n_kv_heads, c.n_seq);
  if (gp == 1) return launch_tail_gp<1>(a, grid, smem, st);
  if (gp == 2) return launch_tail_gp<2>(a, grid, smem, st);
  if (gp == 4) return launch_tail_gp<4>(a, grid, smem, st);
  return launch_tail_gp<8>(a, grid, smem, st);
}

}  // namespace bpkv
