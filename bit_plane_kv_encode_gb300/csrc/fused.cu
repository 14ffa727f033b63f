// One decode pass of one (sequence, KV head) unit in a single kernel: append
// the new token, allocate depths, scan, select, form the union and attend
// (Fathom page: section 3.2 encoder, section 1 depth rule and prefix scan,
// section 2 top-k protocol and exact attention over each head's selection).
//
// A thread-block cluster of kFuseCS CTAs serves one unit; CTA r owns the
// tokens [r T, (r + 1) T), T = bpc * 64, and keeps their scores in shared
// memory.  Cross-CTA steps use distributed shared memory (DSMEM):
//   1. the CTA holding the new token appends it and re-encodes its block; every
//      CTA computes the (identical) depth vector;
//   2. each CTA scans its tokens;                            -- cluster barrier
//      then selects, per query head, its local
//      top-(k - n_sink - n_recent) candidates (exact: key desc, index asc) and
//      copies them into the merge buffer of that head's leader CTA (CTA g for
//      head g);                                              -- cluster barrier
//   3. each leader selects the head's global winners among the merged local
//      winners (the global top set is contained in their union) and sets bit g
//      of the winners' entries in the owners' per-token head masks; sinks and
//      recent tokens are set by their owners;                -- cluster barrier
//   4. per-head counts are published and each CTA writes its selected tokens
//      to the ascending index list at its prefix offset;     -- cluster barrier
//   5. each CTA attends over its own rows with a non-zero mask (its share of the
//      union, every row read once for all heads) and publishes per-head
//      (max, sum, output) partials;                          -- cluster barrier
//   6. each leader merges its head's partials by log-sum-exp.  -- final barrier
// The sequence length is advanced by a separate kernel afterwards.
#include <cooperative_groups.h>

#include "cluster_core.cuh"
#include "depths_core.cuh"
#include "encode_core.cuh"
#include "scan_core.cuh"

namespace cg = cooperative_groups;

namespace bpkv {

constexpr int kFuseCS = 8;                 // CTAs per cluster
constexpr int kFuseThreads = kScanThreads; // 256
constexpr int kFuseMaxBlocks = 80;         // blocks per CTA (5120 tokens)
constexpr int kFuseMaxTok = kFuseMaxBlocks * kBlock;
constexpr int kFuseMaxTop = kClMaxTop;

struct FusedArgs {
  uint64_t* planes;
  uint16_t* scales;
  uint16_t* k_rows;
  uint16_t* v_rows;
  const int64_t* seq_len;
  int64_t cap, nb_cap;
  int32_t n_heads, group;
  const uint16_t* k_new;  // [N][H][D]
  const uint16_t* v_new;
  const float* q;         // [N][H][G][D]
  const float* sigma2;    // [N][H][D]
  const int32_t* budget_q;
  int32_t depth_rule, fixed_channels, fixed_depth;
  int32_t k, n_sink, n_recent;
  float* out;             // [N][H][G][D]
  uint8_t* depths_out;    // optional [N][H][D]
  int32_t* idx_out;       // optional [N][H][G][k]
  int32_t bpc;            // blocks per CTA
  int32_t merge_cap;      // entries of each leader's merge buffer
};

// Scratch reused by the phases of the kernel (never live at the same time).
template <int GP>
union FusedScratch {
  uint16_t kb[kBlock][kD];
  DepthSmem dep;
  ScanSmem<GP> scan;
  SelScratch sel;
  struct {
    int32_t rows[kFuseMaxTok];
    uint8_t rmask[kFuseMaxTok];
    AttScratch a;
    uint32_t warp_red[32];
    uint32_t n_rows;
  } att;
};

template <int GP>
struct FusedSmem {
  float scores[GP * kFuseMaxTok];
  uint32_t mask[kFuseMaxTok / 4];           // 8 head bits per token, 4 tokens per word
  float part[GP][kD + 2];                   // this CTA's attention partial per head
  uint32_t head_cnt[BPKV_MAX_GROUP];        // selected tokens per head in this CTA
  uint32_t merge_n[BPKV_MAX_GROUP];         // leader: entries in its merge buffer
  uint8_t depth[kD];
  FusedScratch<GP> x;
  // followed by the merge buffer of merge_cap 64-bit entries
};

template <int GP>
__global__ void __launch_bounds__(kFuseThreads) k_decode_fused(FusedArgs a) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char fused_raw[];
  FusedSmem<GP>& S = *reinterpret_cast<FusedSmem<GP>*>(fused_raw);
  unsigned long long* merge = reinterpret_cast<unsigned long long*>(fused_raw + sizeof(FusedSmem<GP>));
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int h = blockIdx.y, s = blockIdx.z;
  const int64_t unit = (int64_t)s * a.n_heads + h;
  const int G = a.group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n_old = a.seq_len[s];
  const int64_t n = n_old + 1;
  const int T = a.bpc * kBlock;
  const int64_t t_begin = (int64_t)rank * T;
  const int64_t t_end = min64(t_begin + T, n);
  const int n_own = (int)max64(0, t_end - t_begin);
  const Unit U{a.nb_cap, a.cap};

  for (int e = tid; e < kFuseMaxTok / 4; e += kFuseThreads) S.mask[e] = 0u;
  if (tid < BPKV_MAX_GROUP) {
    S.head_cnt[tid] = 0;
    S.merge_n[tid] = 0;
  }

  // ---- 1. append the new token (its block is re-encoded by the CTA holding it)
  if (n_old / T == rank && n <= a.cap) {
    const int64_t blk = n_old / kBlock;
    encode_block_cta<2>(S.x.kb, a.k_rows + U.row_base(unit), a.v_rows + U.row_base(unit), a.k_new + unit * kD,
                        a.v_new + unit * kD, n_old, blk * kBlock, (int)(n - blk * kBlock),
                        a.planes + U.plane_base(unit), a.scales + U.scale_base(unit), a.nb_cap, blk);
  }
  __syncthreads();
  // ---- depths
  const float* qp = a.q + unit * G * kD;
  if (a.depth_rule == BPKV_DEPTH_WATERFILL)
    alloc_depths_cta(S.x.dep, qp, a.sigma2 + unit * kD, G, a.budget_q[s], S.depth);
  else
    fixed_depths_cta(S.x.dep, qp, G, a.fixed_channels, a.fixed_depth, S.depth);
  __syncthreads();
  if (rank == 0 && a.depths_out && tid < kD) a.depths_out[unit * kD + tid] = S.depth[tid];

  // ---- 2. scan own tokens into shared memory
  {
    int t = 0;
    float qv[GP];
    if (tid < kD) {
      t = S.depth[tid];
#pragma unroll
      for (int hh = 0; hh < GP; ++hh) qv[hh] = hh < G ? qp[hh * kD + tid] : 0.f;
    }
    scan_setup<GP>(S.x.scan.P, S.x.scan.X, t, qv);
    const int64_t b_begin = t_begin / kBlock;
    for (int c0 = 0; c0 * kBlock < n_own; c0 += kScanBlocks) {
      const int nbl = (int)min64(kScanBlocks, (n_own - (int64_t)c0 * kBlock + kBlock - 1) / kBlock);
      float v0[GP], v1[GP];
      scan_chunk<GP>(S.x.scan, a.planes + U.plane_base(unit) + b_begin + c0,
                     a.scales + U.scale_base(unit) + b_begin + c0, a.nb_cap, nbl, G, S.scores + c0 * kBlock, T,
                     n_own - (int64_t)c0 * kBlock, v0, v1);
    }
    __syncthreads();
  }

  // ---- local selection per head, pushed to the head's leader
  const int64_t lo = min64(a.n_sink, n);
  const int64_t hi = max64(n - a.n_recent, lo);
  const int n_top = max(a.k - a.n_sink - a.n_recent, 0);
  const bool take_all = (hi - lo) <= n_top;
  // own candidate range [ca, cb) (local token offsets)
  const int ca = (int)min64(max64(lo - t_begin, 0), n_own);
  const int cb = (int)min64(max64(hi - t_begin, 0), n_own);
  // fixed tokens (and every token when all are kept) get all head bits
  const uint32_t all_bits = (1u << G) - 1u;
  for (int x = tid; x < n_own; x += kFuseThreads) {
    const int64_t tok = t_begin + x;
    if (take_all || tok < lo || tok >= hi) atomicOr(&S.mask[x >> 2], all_bits << (8 * (x & 3)));
  }
  // every CTA of the cluster is running and has initialised its masks and
  // merge counters before any distributed shared memory access
  cluster.sync();
  if (!take_all && n_top > 0) {
    for (int g = 0; g < G; ++g) {
      const float* sg = S.scores + g * T;
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
      unsigned int* rcnt = cluster.map_shared_rank(&S.merge_n[g], g);
      __shared__ uint32_t base_sh;
      if (tid == 0) base_sh = atomicAdd(rcnt, (unsigned int)nw);
      __syncthreads();
      unsigned long long* rbuf = cluster.map_shared_rank(merge, g);
      for (int e = tid; e < nw; e += kFuseThreads)
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
          const int x = (int)(tok - (uint32_t)owner * (uint32_t)T);
          uint32_t* rm = cluster.map_shared_rank(&S.mask[x >> 2], owner);
          atomicOr(rm, 1u << (8 * (x & 3) + g));
        });
  }
  cluster.sync();

  // ---- 4. ordered index output
  if (a.idx_out) {
    uint32_t c[BPKV_MAX_GROUP];
#pragma unroll
    for (int g = 0; g < BPKV_MAX_GROUP; ++g) c[g] = 0;
    for (int x = tid; x < n_own; x += kFuseThreads) {
      const uint32_t mk = (S.mask[x >> 2] >> (8 * (x & 3))) & 0xffu;
#pragma unroll
      for (int g = 0; g < BPKV_MAX_GROUP; ++g) c[g] += (mk >> g) & 1u;
    }
    if (tid < BPKV_MAX_GROUP) S.head_cnt[tid] = 0;
    __syncthreads();
#pragma unroll
    for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
      uint32_t v = c[g];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && g < G && v) atomicAdd(&S.head_cnt[g], v);
    }
  }
  cluster.sync();
  if (a.idx_out) {
    uint32_t before[BPKV_MAX_GROUP], total[BPKV_MAX_GROUP];
    for (int g = 0; g < G; ++g) {
      before[g] = 0;
      total[g] = 0;
      for (int r = 0; r < kFuseCS; ++r) {
        const uint32_t v = *cluster.map_shared_rank(&S.head_cnt[g], r);
        if (r < rank) before[g] += v;
        total[g] += v;
      }
    }
    // ordered compaction of this CTA's selected tokens, all heads per 256-token tile
    __shared__ uint32_t tile_cnt[8][BPKV_MAX_GROUP];
    for (int x0 = 0; x0 < n_own; x0 += kFuseThreads) {
      const int x = x0 + tid;
      const uint32_t mk = (x < n_own) ? (S.mask[x >> 2] >> (8 * (x & 3))) & 0xffu : 0u;
      uint32_t bal[BPKV_MAX_GROUP];
#pragma unroll
      for (int g = 0; g < BPKV_MAX_GROUP; ++g) {
        bal[g] = __ballot_sync(0xffffffffu, (mk >> g) & 1u);
        if (lane == 0) tile_cnt[warp][g] = __popc(bal[g]);
      }
      __syncthreads();
      for (int g = 0; g < G; ++g) {
        uint32_t off = before[g];
        for (int w = 0; w < warp; ++w) off += tile_cnt[w][g];
        off += __popc(bal[g] & ((1u << lane) - 1u));
        if ((mk >> g) & 1u && off < (uint32_t)a.k) a.idx_out[(unit * G + g) * a.k + off] = (int32_t)(t_begin + x);
        uint32_t tile = 0;
        for (int w = 0; w < kFuseThreads / 32; ++w) tile += tile_cnt[w][g];
        before[g] += tile;
      }
      __syncthreads();
    }
    if (rank == kFuseCS - 1)
      for (int g = 0; g < G; ++g)
        for (int p = (int)total[g] + tid; p < a.k; p += kFuseThreads) a.idx_out[(unit * G + g) * a.k + p] = -1;
  }

  // ---- 5. attention over this CTA's union rows
  {
    auto& A = S.x.att;
    if (tid == 0) A.n_rows = 0;
    __syncthreads();
    for (int x0 = 0; x0 < n_own; x0 += kFuseThreads) {
      const int x = x0 + tid;
      const uint32_t mk = (x < n_own) ? ((S.mask[x >> 2] >> (8 * (x & 3))) & 0xffu) : 0u;
      const uint32_t bal = __ballot_sync(0xffffffffu, mk != 0u);
      uint32_t wbase = 0;
      if (lane == 0 && bal) wbase = atomicAdd(&A.n_rows, (uint32_t)__popc(bal));
      wbase = __shfl_sync(0xffffffffu, wbase, 0);
      if (mk) {
        const uint32_t r = wbase + __popc(bal & ((1u << lane) - 1u));
        A.rows[r] = x;
        A.rmask[r] = (uint8_t)mk;
      }
    }
    __syncthreads();
    attend_rows<GP>(A.a, A.rows, A.rmask, (int)A.n_rows, a.k_rows + U.row_base(unit) + t_begin * kD,
                    a.v_rows + U.row_base(unit) + t_begin * kD, qp, G, S.part);
  }
  cluster.sync();

  // ---- 6. leaders merge their head's partials
  if (rank < G) merge_partials<kFuseCS>(cluster, S.part, rank, a.out + (unit * G + rank) * kD);
  cluster.sync();
}

template <int GP>
size_t fused_smem_bytes(int merge_cap) {
  return sizeof(FusedSmem<GP>) + (size_t)merge_cap * sizeof(unsigned long long);
}

template <int GP>
cudaError_t launch_fused_gp(const FusedArgs& a, dim3 grid, cudaStream_t st) {
  const size_t smem = fused_smem_bytes<GP>(a.merge_cap);
  cudaError_t e = cudaFuncSetAttribute(k_decode_fused<GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kFuseThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kFuseCS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_decode_fused<GP>, a);
}

// Whether one decode pass of this cache fits the fused kernel: the group fits
// the cluster, each CTA's share of the tokens and its scores fit shared
// memory, and k is small enough for the leaders' merge buffers.
bool fused_eligible(const bpkv_cache& c, int32_t k, int32_t n_sink, int32_t n_recent, int32_t depth_rule) {
  if (depth_rule == BPKV_DEPTH_DENSE || depth_rule == BPKV_DEPTH_GIVEN || c.basis || c.group > kFuseCS) return false;
  const int64_t nb = (c.n_max + 1 + kBlock - 1) / kBlock;
  const int64_t bpc = (nb + kFuseCS - 1) / kFuseCS;
  if (bpc < 1 || bpc > kFuseMaxBlocks) return false;
  const int n_top = k - n_sink - n_recent;
  if (n_top > kFuseMaxTop) return false;
  const int gp = c.group <= 1 ? 1 : c.group <= 2 ? 2 : c.group <= 4 ? 4 : 8;
  const int merge_cap = kFuseCS * max(n_top, 1);
  const size_t smem = gp == 1 ? fused_smem_bytes<1>(merge_cap) : gp == 2 ? fused_smem_bytes<2>(merge_cap)
                    : gp == 4 ? fused_smem_bytes<4>(merge_cap) : fused_smem_bytes<8>(merge_cap);
  int dev = 0, max_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
  return smem <= (size_t)max_smem;
}

cudaError_t launch_decode_fused(const bpkv_cache& c, const uint16_t* k_new, const uint16_t* v_new, const float* q,
                                const float* sigma2, const int32_t* budget_q, int32_t depth_rule,
                                int32_t fixed_channels, int32_t fixed_depth, int32_t k, int32_t n_sink,
                                int32_t n_recent, float* out, uint8_t* depths_out, int32_t* idx_out,
                                cudaStream_t st) {
  const int64_t nb = (c.n_max + 1 + kBlock - 1) / kBlock;
  const int32_t bpc = (int32_t)((nb + kFuseCS - 1) / kFuseCS);
  const int n_top = k - n_sink - n_recent;
  FusedArgs a{c.planes, c.scales, c.k_rows, c.v_rows, c.seq_len, c.cap_tokens, c.cap_tokens / kBlock,
              c.n_kv_heads, c.group, k_new, v_new, q, sigma2, budget_q, depth_rule, fixed_channels, fixed_depth,
              k, n_sink, n_recent, out, depths_out, idx_out, bpc, kFuseCS * max(n_top, 1)};
  dim3 grid(kFuseCS, c.n_kv_heads, c.n_seq);
  cudaError_t e;
  if (c.group <= 1) e = launch_fused_gp<1>(a, grid, st);
  else if (c.group <= 2) e = launch_fused_gp<2>(a, grid, st);
  else if (c.group <= 4) e = launch_fused_gp<4>(a, grid, st);
  else e = launch_fused_gp<8>(a, grid, st);
  return e;
}

}  // namespace bpkv
