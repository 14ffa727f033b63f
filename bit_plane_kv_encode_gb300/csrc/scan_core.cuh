// Device building blocks of the prefix-plane scan (the scan kernel and the
// plan builder of the depth kernel).  See scan.cu for the method.
#pragma once

#include "common.cuh"

namespace bpkv {

constexpr int kScanBlocks = 8;                  // 64-token blocks per chunk
constexpr int kScanThreads = 32 * kScanBlocks;  // one warp per block
constexpr int kMaxGroups = 20;                  // 16 depth-4 groups + one partial group per other depth
constexpr int kMaxSlots = 288;                  // padded channel slots over all groups
// Groups are staged and scored in passes of at most kPassGroups groups and
// kPassSlots slots (one pass for every budget up to about 300 bits per token).
constexpr int kPassGroups = 10;
constexpr int kPassSlots = 144;
constexpr int kMaxPasses = 8;

template <int T>
struct Depth {
  static constexpr int cap = 32 / T;                  // channels per group
  static constexpr int pitch = (cap + 3) / 4 * 4;     // slots per group, multiple of 4
};

__host__ __device__ constexpr int slot_pitch(int t) {
  return t == 4 ? 8 : t == 3 ? 12 : t == 2 ? 16 : 32;
}
__host__ __device__ constexpr int group_cap(int t) { return 32 / t; }

// Bit position of field m of a depth-t group inside the shifted word it is read
// from (x << 1 when the field ends at or below bit 21, x >> 9 otherwise), so
// that the field sits in [1, 23) under the exponent of 2^23.
__host__ __device__ constexpr int field_pos(int t, int m) {
  return (m * t + t <= 22) ? m * t + 1 : m * t - 9;
}

// What a CTA needs to scan one unit, derived from its depth vector and query:
// the channel groups, the plane row of every (group, lane), the channel and
// group of every slot, and the weights w = q 2^(4 - t - pos).
template <int GP>
struct __align__(16) ScanPlan {
  float w[kMaxSlots * GP];                          // [slot][head]
  int16_t row_of_lane[kMaxGroups * 32];             // j * 4 + p, or -1
  int16_t slot_ch[kMaxSlots];                       // channel of each slot, or -1
  int8_t slot_grp[kMaxSlots];                       // group of each slot
  int8_t grp_t[kMaxGroups];
  int16_t grp_base[kMaxGroups];                     // first slot of each group
  int8_t grp_cnt[kMaxGroups];                       // channels in each group
  int8_t pass_g[kMaxPasses + 1];                    // first group of each pass, then n_groups
  int n_groups, n_slots, n_passes;
};

struct PlanScratch {
  int cnt_t[5];
  int warp_cnt[4][5];
};

// 32 x 32 bit transpose across the warp: on return bit r of lane l's word is
// bit l of lane r's input word.  Five exchange rounds with the lane at
// distance 16, 8, 4, 2, 1; the byte-level rounds (16, 8) merge with one byte
// permute (sel[0], sel[1] per lane), the others with a rotate and a select.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, const uint32_t (&keep)[5],
                                                     const uint32_t (&rot)[5]) {
  x = __byte_perm(x, __shfl_xor_sync(0xffffffffu, x, 16), keep[0]);
  x = __byte_perm(x, __shfl_xor_sync(0xffffffffu, x, 8), keep[1]);
#pragma unroll
  for (int s = 2; s < 5; ++s) {
    const int j = 16 >> s;
    const uint32_t p = __shfl_xor_sync(0xffffffffu, x, j);
    const uint32_t r = __funnelshift_l(p, p, rot[s]);
    x = (x & keep[s]) | (r & ~keep[s]);
  }
  return x;
}

__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ void unpack2(unsigned long long v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Transpose constants of this lane (see warp_transpose32): byte selectors of
// the rounds at distance 16 and 8 (keep[0], keep[1]; rot unused), kept bits and
// rotation of the others.
__device__ __forceinline__ void transpose_consts(int lane, uint32_t (&keep)[5], uint32_t (&rot)[5]) {
  keep[0] = (lane & 16) ? 0x3276u : 0x5410u;
  keep[1] = (lane & 8) ? 0x3715u : 0x6240u;
  rot[0] = rot[1] = 0u;
#pragma unroll
  for (int st = 2; st < 5; ++st) {
    const int j = 16 >> st;
    const uint32_t M = st == 2 ? 0x0F0F0F0Fu : st == 3 ? 0x33333333u : 0x55555555u;
    const bool hi = (lane & j) != 0;
    keep[st] = hi ? ~M : M;
    rot[st] = hi ? (uint32_t)(32 - j) : (uint32_t)j;
  }
}

// Channel groups and per-query weights.  Threads 0..127 pass their channel's
// depth t and q values; blockDim.x must be kScanThreads.  The groups of depth
// 4 come first, then 3, 2, 1; within a depth, groups of group_cap(t) channels
// in channel order.  Every layout figure follows in closed form from the four
// per-depth channel counts.
template <int GP>
__device__ void scan_setup(ScanPlan<GP>& S, PlanScratch& X, int t, const float (&qv)[GP],
                           int32_t* status = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int rank = 0;
  if (tid < kD) {
#pragma unroll
    for (int d = 1; d <= 4; ++d) {
      const uint32_t b = __ballot_sync(0xffffffffu, t == d);
      if (t == d) rank = __popc(b & ((1u << lane) - 1u));
      if (lane == 0) X.warp_cnt[warp][d] = __popc(b);
    }
  }
  // defaults of every entry, before any thread writes its channel's entries
  for (int e = tid; e < kMaxGroups * 32; e += kScanThreads) S.row_of_lane[e] = -1;
  for (int e = tid; e < kMaxSlots * GP; e += kScanThreads) S.w[e] = 0.f;
  for (int e = tid; e < kMaxSlots; e += kScanThreads) S.slot_ch[e] = -1;
  __syncthreads();
  // per depth d: channels, groups, first group and first slot
  int cnt[5], ng[5], goff[5], soff[5];
  int n_groups = 0, n_slots = 0;
#pragma unroll
  for (int d = 4; d >= 1; --d) {
    cnt[d] = X.warp_cnt[0][d] + X.warp_cnt[1][d] + X.warp_cnt[2][d] + X.warp_cnt[3][d];
    ng[d] = (cnt[d] + group_cap(d) - 1) / group_cap(d);
    goff[d] = n_groups;
    soff[d] = n_slots;
    n_groups += ng[d];
    n_slots += ng[d] * slot_pitch(d);
  }
  if (tid < n_groups) {
    const int gi = (int)BPKV_CHK(tid, kMaxGroups, status);
#pragma unroll
    for (int d = 4; d >= 1; --d) {
      if (tid >= goff[d] && tid < goff[d] + ng[d]) {
        const int i = tid - goff[d];
        S.grp_t[gi] = (int8_t)d;
        S.grp_base[gi] = (int16_t)(soff[d] + i * slot_pitch(d));
        S.grp_cnt[gi] = (int8_t)min(group_cap(d), cnt[d] - i * group_cap(d));
      }
    }
  }
  for (int e = tid; e < kMaxSlots; e += kScanThreads) {
    int g = 0;
#pragma unroll
    for (int d = 4; d >= 1; --d)
      if (e >= soff[d] && e < soff[d] + ng[d] * slot_pitch(d)) g = goff[d] + (e - soff[d]) / slot_pitch(d);
    S.slot_grp[e] = (int8_t)g;
  }
  if (tid == 0) {
    S.n_groups = n_groups;
    S.n_slots = n_slots;
    // passes: greedy runs of groups within kPassGroups groups and kPassSlots
    // slots (at most 4 runs for any depth vector: the slots total <= 288)
    int np = 0, run_g = 0, run_s = 0;
    for (int d = 4; d >= 1; --d) {
      for (int i = 0; i < ng[d]; ++i) {
        const int pt = slot_pitch(d);
        if (run_g == 0 || run_g == kPassGroups || run_s + pt > kPassSlots) {
          if (np < kMaxPasses) S.pass_g[np] = (int8_t)(goff[d] + i);
          ++np;
          run_g = 0;
          run_s = 0;
        }
        ++run_g;
        run_s += pt;
      }
    }
    np = min(np, kMaxPasses);
    S.pass_g[np] = (int8_t)n_groups;
    S.n_passes = np;
  }
  if (tid < kD && t > 0) {
    for (int w = 0; w < warp; ++w) rank += X.warp_cnt[w][t];
    int goff_t = 0, soff_t = 0;  // selected without dynamic indexing (keeps the arrays in registers)
#pragma unroll
    for (int d = 1; d <= 4; ++d) {
      if (d == t) {
        goff_t = goff[d];
        soff_t = soff[d];
      }
    }
    const int gi = rank / group_cap(t), m = rank % group_cap(t);
    const int g = goff_t + gi, base = soff_t + gi * slot_pitch(t), P = slot_pitch(t);
    S.slot_ch[BPKV_CHK(base + m, kMaxSlots, status)] = (int16_t)tid;
    for (int p = 0; p < t; ++p)
      S.row_of_lane[BPKV_CHK(g * 32 + m * t + (t - 1 - p), kMaxGroups * 32, status)] = (int16_t)(tid * 4 + p);
    // w = q 2^(4 - t - pos) per head, laid out [group][head][slot]; other slots stay 0
#pragma unroll
    for (int hh = 0; hh < GP; ++hh)
      S.w[BPKV_CHK((base + m) * GP + hh, kMaxSlots * GP, status)] = ldexpf(qv[hh], 4 - t - field_pos(t, m));
  }
  __syncthreads();
}

// Copy a plan built by scan_setup elsewhere (global memory) into shared memory.
template <int GP>
__device__ void scan_load_plan(ScanPlan<GP>& S, const ScanPlan<GP>* __restrict__ src) {
  static_assert(sizeof(ScanPlan<GP>) % 16 == 0, "plan copied in 16-byte pieces");
  const uint4* g = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(&S);
  for (int e = threadIdx.x; e < (int)(sizeof(ScanPlan<GP>) / 16); e += blockDim.x) d[e] = g[e];
  __syncthreads();
}

// Store the plan (shared memory) to global memory.
template <int GP>
__device__ void scan_store_plan(const ScanPlan<GP>& S, ScanPlan<GP>* __restrict__ dst) {
  const uint4* s = reinterpret_cast<const uint4*>(&S);
  uint4* g = reinterpret_cast<uint4*>(dst);
  for (int e = threadIdx.x; e < (int)(sizeof(ScanPlan<GP>) / 16); e += blockDim.x) g[e] = s[e];
}

// ---------------------------------------------------------------------------
// Pipelined form: the plane words and raw block scales of one step are
// fetched by asynchronous 16-byte copies into one of two stage buffers while
// the warps score the other.  A step is one pass over one chunk, or, for a
// unit whose plan is a single pass of at most kWideGroups groups, one pass
// over kWideSub consecutive chunks starting at an even chunk: each slot's
// block scales then come as one whole 32-byte sector instead of two halves
// fetched in different steps (device memory serves the second half from L2;
// reads of pinned host memory by these copies are not kept in L2, so there
// every half sector crosses the link in full).
//
// Staged plane rows.  Device caches: one-chunk steps, each row's 16 words
// followed by 4 words of padding (row pitch 20 words: the 8-byte reads of one
// block column by rows r .. r + 7 fall in eight different 16-byte bank
// groups).  Host caches: no padding; a row of a step of `sub` chunks is 2 sub
// 32-byte pieces (4 blocks each), piece k of row r at piece slot
// k ^ swz_piece(r) of the row with its two 16-byte halves swapped when
// swz_half(r) is 1, which gives the reads the same eight bank groups while
// every 32-byte sector read from memory lands in one aligned 32-byte slot (a
// copy whose sector halves land in different slots is split and fetches the
// sector twice; the L2 absorbs that for device memory, but over the host link
// it costs the bytes in full).

constexpr int kStageRows = kPassGroups * 32;
constexpr int kRowPitch = 2 * kScanBlocks + 4;              // device caches
constexpr int kStageWords = kStageRows * kRowPitch;         // device caches
constexpr int kHostStageWords = kStageRows * 2 * kScanBlocks;
constexpr int kWideSub = 2;                                 // chunks per step of a wide unit
constexpr int kWideGroups = kHostStageWords / (32 * 2 * kScanBlocks * kWideSub);
constexpr int kStageU32 = kStageWords + kPassSlots * kScanBlocks / 2 > kHostStageWords + kPassSlots * kScanBlocks * kWideSub / 2
                              ? kStageWords + kPassSlots * kScanBlocks / 2
                              : kHostStageWords + kPassSlots * kScanBlocks * kWideSub / 2;
static_assert(kWideGroups >= 5, "a wide step must hold the single-pass plans of usual budgets");

// u32 words per staged plane row for steps of `sub` chunks.
__host__ __device__ constexpr int row_pitch(int sub, bool host) { return host ? 2 * kScanBlocks * sub : kRowPitch; }
// Placement of the pieces of staged row r of a host cache (see above).
__host__ __device__ __forceinline__ int swz_piece(int r, int sub) { return sub == 1 ? (r >> 1) & 1 : r & 3; }
__host__ __device__ __forceinline__ int swz_half(int r) { return (r >> 2) & 1; }
// u32 word of 16-byte part q (0 .. 4 sub - 1) of staged row r
__host__ __device__ __forceinline__ int staged_word(int r, int q, int sub, bool host) {
  if (!host) return r * kRowPitch + 4 * q;
  return r * row_pitch(sub, true) + ((4 * q) ^ (8 * swz_piece(r, sub) + 4 * swz_half(r)));
}

// One stage buffer: the plane words (row (g - g0) * 32 + lane at
// u32[row * row_pitch]), then the raw block scales, [slot - s0][sub chunks x
// 8 blocks], from word kStageWords (device caches) or kHostStageWords.
struct __align__(16) ScanStage {
  uint32_t u32[kStageU32];
};
__device__ __forceinline__ uint16_t* stage_sc(ScanStage& st, bool host) {
  return reinterpret_cast<uint16_t*>(st.u32 + (host ? kHostStageWords : kStageWords));
}
__device__ __forceinline__ const uint16_t* stage_sc(const ScanStage& st, bool host) {
  return reinterpret_cast<const uint16_t*>(st.u32 + (host ? kHostStageWords : kStageWords));
}

template <int GP>
struct __align__(16) PipeSmem {
  ScanStage st[2];
  float u[kScanBlocks][kPassSlots * GP];      // per warp (block): u = s w, [slot - s0][head]
  ScanPlan<GP> P;
  PlanScratch X;
  // level-0 selection histograms of the unit being scored, two 16-bit counts
  // per word (bins 2i and 2i + 1 of head h at word h * kTopkBins / 2 + i)
  uint32_t hist[GP <= 4 ? GP * kTopkBins / 2 : 1];
};

// Whether the pipelined scan counts the level-0 histograms in shared memory.
template <int GP>
__host__ __device__ constexpr bool pipe_counts_hist() { return GP <= 4; }

__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Packed accumulators of one lane: for each of its two tokens, the heads in
// pairs (one head, the two tokens, when GP = 1); even and odd fields apart.
template <int GP>
struct Acc {
  static constexpr int HP = GP == 1 ? 1 : GP / 2;
  unsigned long long t0[2][HP];  // [field parity][head pair]: token lane (GP = 1: both tokens)
  unsigned long long t1[2][HP];  // token lane + 32 (unused when GP = 1)
};

// Field M of a depth-T group for this lane's two tokens.  xa / xb are the
// transposed words shifted (see field_pos) with the exponent of 2^23 already
// in bits 23..30, so one AND keeps the field and the exponent: the float is
// 2^23 + c 2^pos, and one packed subtraction of the offset gives both tokens'
// e 2^pos (exact).  Each pair of heads then takes one packed FMA per token
// with e broadcast.
template <int T, int M, int GP>
__device__ __forceinline__ void field_heads(uint32_t xa0, uint32_t xb0, uint32_t xa1, uint32_t xb1,
                                            const float* __restrict__ ud, Acc<GP>& A) {
  constexpr int pos = field_pos(T, M);
  constexpr uint32_t keep = (((1u << T) - 1u) << pos) | 0xFF800000u;
  constexpr float K = 8388608.f + ((float)(1 << (T - 1)) - 0.5f) * (float)(1u << pos);
  constexpr bool use_a = (M * T + T <= 22);
  constexpr int par = M & 1;
  const uint32_t s0 = use_a ? xa0 : xb0, s1 = use_a ? xa1 : xb1;
  const unsigned long long E = fadd2(pack2(__uint_as_float(s0 & keep), __uint_as_float(s1 & keep)), pack2(-K, -K));
  const float* up = ud + M * GP;
  if constexpr (GP == 1) {
    A.t0[par][0] = ffma2(pack2(up[0], up[0]), E, A.t0[par][0]);
  } else {
    float e0, e1;
    unpack2(E, e0, e1);
    const unsigned long long E0 = pack2(e0, e0), E1 = pack2(e1, e1);
    if constexpr (GP == 2) {
      const float2 uu = *reinterpret_cast<const float2*>(up);
      const unsigned long long U = pack2(uu.x, uu.y);
      A.t0[par][0] = ffma2(U, E0, A.t0[par][0]);
      A.t1[par][0] = ffma2(U, E1, A.t1[par][0]);
    } else {
#pragma unroll
      for (int q = 0; q < GP / 4; ++q) {
        const float4 uu = *reinterpret_cast<const float4*>(up + 4 * q);
        const unsigned long long Ua = pack2(uu.x, uu.y), Ub = pack2(uu.z, uu.w);
        A.t0[par][2 * q] = ffma2(Ua, E0, A.t0[par][2 * q]);
        A.t0[par][2 * q + 1] = ffma2(Ub, E0, A.t0[par][2 * q + 1]);
        A.t1[par][2 * q] = ffma2(Ua, E1, A.t1[par][2 * q]);
        A.t1[par][2 * q + 1] = ffma2(Ub, E1, A.t1[par][2 * q + 1]);
      }
    }
  }
}

// Fields 4 B .. 4 B + 3 of a depth-T group (those below the group's capacity).
// Slots past the group's channel count have u = 0, so their fields add 0.
template <int T, int B, int GP>
__device__ __forceinline__ void field_block(uint32_t xa0, uint32_t xb0, uint32_t xa1, uint32_t xb1,
                                            const float* __restrict__ ud, Acc<GP>& A) {
  constexpr int C = Depth<T>::cap;
  if constexpr (4 * B < C) field_heads<T, 4 * B, GP>(xa0, xb0, xa1, xb1, ud, A);
  if constexpr (4 * B + 1 < C) field_heads<T, 4 * B + 1, GP>(xa0, xb0, xa1, xb1, ud, A);
  if constexpr (4 * B + 2 < C) field_heads<T, 4 * B + 2, GP>(xa0, xb0, xa1, xb1, ud, A);
  if constexpr (4 * B + 3 < C) field_heads<T, 4 * B + 3, GP>(xa0, xb0, xa1, xb1, ud, A);
}

// The fields of one group in blocks of four: one jump to the group's last
// block, then straight-line code down to block 0 (no test per field).
template <int T, int GP>
__device__ __forceinline__ void group_fields_heads(int cnt, uint32_t xa0, uint32_t xb0, uint32_t xa1, uint32_t xb1,
                                                   const float* __restrict__ ud, Acc<GP>& A) {
  constexpr int NB = (Depth<T>::cap + 3) / 4;
  static_assert(NB <= 8, "at most 32 fields per group");
#define BPKV_FIELD_BLOCK(b)                                                                    \
  case (b) + 1:                                                                                \
    if constexpr ((b) < NB) field_block<T, (b), GP>(xa0, xb0, xa1, xb1, ud, A); \
    [[fallthrough]];
  switch ((cnt + 3) >> 2) {
    BPKV_FIELD_BLOCK(7)
    BPKV_FIELD_BLOCK(6)
    BPKV_FIELD_BLOCK(5)
    BPKV_FIELD_BLOCK(4)
    BPKV_FIELD_BLOCK(3)
    BPKV_FIELD_BLOCK(2)
    BPKV_FIELD_BLOCK(1)
    case 1:
      field_block<T, 0, GP>(xa0, xb0, xa1, xb1, ud, A);
      [[fallthrough]];
    default:
      break;
  }
#undef BPKV_FIELD_BLOCK
}

// This lane's scores of head hh for its two tokens.
template <int GP>
__device__ __forceinline__ void acc_scores(const Acc<GP>& A, int hh, float& v0, float& v1) {
  float a, b, c, d;
  if constexpr (GP == 1) {
    unpack2(A.t0[0][0], a, b);
    unpack2(A.t0[1][0], c, d);
    v0 = a + c;
    v1 = b + d;
  } else {
    unpack2(A.t0[0][hh >> 1], a, b);
    unpack2(A.t0[1][hh >> 1], c, d);
    v0 = (hh & 1) ? b + d : a + c;
    unpack2(A.t1[0][hh >> 1], a, b);
    unpack2(A.t1[1][hh >> 1], c, d);
    v1 = (hh & 1) ? b + d : a + c;
  }
}

template <int GP>
__device__ __forceinline__ void acc_zero(Acc<GP>& A) {
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int i = 0; i < Acc<GP>::HP; ++i) A.t0[p][i] = A.t1[p][i] = 0ull;
}

// All threads: start the copies of step (n_sub chunks from block b0, groups
// [g0, g1)) into stage buffer b, laid out for steps of `sub` chunks: per used
// plane row its n_sub x 8 words (16-byte pieces), per used slot its n_sub x 8
// block scales (one piece per chunk); then commit them as this thread's newest
// group.  Host caches (`host`): consecutive pieces of a row are taken by
// consecutive threads, so that each warp instruction copies whole sectors
// (the halves of a sector copied by different instructions would each fetch
// it over the link); device caches: each thread takes whole rows (fewer
// instructions; the L2 serves the second half).  pl / sp are the unit's
// planes and scales; b0 + 8 n_sub <= nb_cap.
template <int GP>
__device__ __forceinline__ void scan_issue(PipeSmem<GP>& S, int b, const uint64_t* pl, const uint16_t* sp,
                                           int64_t nb_cap, int64_t b0, int g0, int g1, int sub, int n_sub,
                                           bool host, int32_t* status = nullptr) {
  const ScanPlan<GP>& P = S.P;
  const int sc_pitch = kScanBlocks * sub;
  const int n_row = (g1 - g0) * 32;
  const int s0 = P.grp_base[g0], s1 = g1 < P.n_groups ? (int)P.grp_base[g1] : P.n_slots;
  const int sh = n_sub - 1;  // n_sub is 1 or 2
  const int n_sc = (s1 - s0) << sh;
  if (host) {
    const int n_piece = n_row << (2 + sh);
    for (int e = threadIdx.x; e < n_piece + n_sc; e += kScanThreads) {
      if (e < n_piece) {
        const int r = e >> (2 + sh), piece = e & ((4 << sh) - 1);
        const int row = P.row_of_lane[BPKV_CHK(g0 * 32 + r, kMaxGroups * 32, status)];
        if (row >= 0)
          cp_async16(&S.st[b].u32[BPKV_CHK(staged_word(r, piece, sub, true), kHostStageWords - 3, status)],
                     pl + BPKV_CHK((int64_t)row * nb_cap + b0 + 2 * piece, kD * kPlanes * nb_cap - 1, status));
      } else {
        const int f = e - n_piece, rel = f >> sh, c = f & sh;
        const int ch = P.slot_ch[BPKV_CHK(s0 + rel, kMaxSlots, status)];
        uint16_t* dst = stage_sc(S.st[b], host) +
                        BPKV_CHK(rel * sc_pitch + kScanBlocks * c, 2 * (kStageU32 - kHostStageWords) - 7, status);
        if (ch >= 0) cp_async16(dst, sp + BPKV_CHK((int64_t)ch * nb_cap + b0 + kScanBlocks * c, kD * nb_cap - 7, status));
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);  // unused slot: scale 0
      }
    }
  } else {
    for (int e = threadIdx.x; e < n_row + n_sc; e += kScanThreads) {
      if (e < n_row) {
        const int row = P.row_of_lane[BPKV_CHK(g0 * 32 + e, kMaxGroups * 32, status)];
        if (row >= 0) {
          const uint64_t* src = pl + BPKV_CHK((int64_t)row * nb_cap + b0, kD * kPlanes * nb_cap - 8 * (1 << sh) + 1, status);
#pragma unroll 4
          for (int piece = 0; piece < (4 << sh); ++piece)
            cp_async16(&S.st[b].u32[BPKV_CHK(staged_word(e, piece, sub, false), kStageWords - 3, status)],
                       src + 2 * piece);
        }
      } else {
        const int f = e - n_row, rel = f >> sh, c = f & sh;
        const int ch = P.slot_ch[BPKV_CHK(s0 + rel, kMaxSlots, status)];
        uint16_t* dst = stage_sc(S.st[b], host) +
                        BPKV_CHK(rel * sc_pitch + kScanBlocks * c, 2 * (kStageU32 - kStageWords) - 7, status);
        if (ch >= 0) cp_async16(dst, sp + BPKV_CHK((int64_t)ch * nb_cap + b0 + kScanBlocks * c, kD * nb_cap - 7, status));
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);  // unused slot: scale 0
      }
    }
  }
  cp_async_commit();
}

// s w.  A slot that no channel uses has w = 0 and a staged scale of 0 (its
// copy writes zeros), so stale stage contents never reach a score; the
// scales of blocks past the end of a unit's cache are whatever the cache
// holds there, but they only reach tokens past the end, which are not written.
__device__ __forceinline__ float sw(float s, float w) { return s * w; }

// This warp's u = s w for the slots [s0, s1) of a landed stage (block lb of
// chunk c of a step of `sub` chunks; `host`: the host-cache layout): one slot
// per lane at a time, all heads with vector loads and stores.
template <int GP>
__device__ __forceinline__ void scan_form_u(PipeSmem<GP>& S, int b, int s0, int s1, int lb, int sub, int c,
                                            bool host, int32_t* status = nullptr) {
  const int lane = threadIdx.x & 31;
  const int sc_pitch = kScanBlocks * sub;
  const uint16_t* sc = stage_sc(S.st[b], host) + kScanBlocks * c + lb;
  const float* w = S.P.w + s0 * GP;
  float* ud = S.u[lb];
#ifdef BPKV_CHECKS
  if (lane == 0 && (s0 < 0 || s1 > kMaxSlots || s1 - s0 > kPassSlots)) set_status(status, BPKV_DEV_BOUNDS);
#endif
  for (int rel = lane; rel < s1 - s0; rel += 32) {
    const float sv = fp16_bits_to_float(sc[rel * sc_pitch]);
    if constexpr (GP == 1) {
      ud[rel] = sw(sv, w[rel]);
    } else if constexpr (GP == 2) {
      const float2 wv = *reinterpret_cast<const float2*>(w + 2 * rel);
      *reinterpret_cast<float2*>(ud + 2 * rel) = make_float2(sw(sv, wv.x), sw(sv, wv.y));
    } else {
#pragma unroll
      for (int q = 0; q < GP / 4; ++q) {
        const float4 wv = *reinterpret_cast<const float4*>(w + GP * rel + 4 * q);
        *reinterpret_cast<float4*>(ud + GP * rel + 4 * q) =
            make_float4(sw(sv, wv.x), sw(sv, wv.y), sw(sv, wv.z), sw(sv, wv.w));
      }
    }
  }
}

// Add groups [g0, g1) of a landed stage to this lane's accumulators (warp lb:
// block lb of chunk c of a step of `sub` chunks, tokens lane and lane + 32;
// `host`: the host-cache layout).  u must be formed.
template <int GP>
__device__ __forceinline__ void scan_compute_pipe(const PipeSmem<GP>& S, int b, int g0, int g1, int s0, int lb,
                                                  int sub, int c, bool host, const uint32_t (&keep)[5],
                                                  const uint32_t (&rot)[5], Acc<GP>& A, int32_t* status = nullptr) {
  const int lane = threadIdx.x & 31;
  const ScanPlan<GP>& P = S.P;
  // block lb of chunk c is word 2 (lb % 2) of 16-byte part 4 c + lb / 2 of
  // row (g - g0) * 32 + lane (placed as row lane: 32 is a multiple of 8)
  const uint32_t* wl = S.st[b].u32 + staged_word(lane, 4 * c + (lb >> 1), sub, host) + 2 * (lb & 1);
  const int g_stride = 32 * row_pitch(sub, host);
  for (int g = g0; g < g1; ++g) {
    const int d = P.grp_t[g], cnt = P.grp_cnt[g];
#ifdef BPKV_CHECKS
    // the group's rows inside the stage, its slots inside the pass's u
    if (lane == 0 && ((g - g0 + 1) * g_stride > (host ? kHostStageWords : kStageWords) || d < 1 || d > 4 ||
                      (P.grp_base[g] - s0 + slot_pitch(d)) > kPassSlots || P.grp_base[g] < s0))
      set_status(status, BPKV_DEV_BOUNDS);
#endif
    const uint2 wv = *reinterpret_cast<const uint2*>(wl + (g - g0) * g_stride);
    const uint32_t x0 = warp_transpose32(wv.x, keep, rot);
    const uint32_t x1 = warp_transpose32(wv.y, keep, rot);
    // the exponent of 2^23 over bits 23..30 of both shifted forms
    const uint32_t xa0 = ((x0 << 1) & 0x007FFFFFu) | 0x4B000000u, xb0 = (x0 >> 9) | 0x4B000000u;
    const uint32_t xa1 = ((x1 << 1) & 0x007FFFFFu) | 0x4B000000u, xb1 = (x1 >> 9) | 0x4B000000u;
    const float* ud = S.u[lb] + (P.grp_base[g] - s0) * GP;
    switch (d) {
      case 4: group_fields_heads<4, GP>(cnt, xa0, xb0, xa1, xb1, ud, A); break;
      case 3: group_fields_heads<3, GP>(cnt, xa0, xb0, xa1, xb1, ud, A); break;
      case 2: group_fields_heads<2, GP>(cnt, xa0, xb0, xa1, xb1, ud, A); break;
      default: group_fields_heads<1, GP>(cnt, xa0, xb0, xa1, xb1, ud, A); break;
    }
  }
}

// Level-0 selection histogram of one warp's block (top 12 bits of the
// order-preserving key), for tokens x0 + lane and x0 + lane + 32 in [lo, hi),
// added to hist [G][kTopkBins]: lanes with equal (head, bin) are counted by
// one atomic of their leader.  Called by whole warps.
template <int GP>
__device__ __forceinline__ void warp_hist(int G, int64_t x0, int64_t lo, int64_t hi, const float (&v0)[GP],
                                          const float (&v1)[GP], uint32_t* __restrict__ hist) {
  const int lane = threadIdx.x & 31;
  const bool in0 = x0 >= lo && x0 < hi, in1 = x0 + 32 >= lo && x0 + 32 < hi;
#pragma unroll
  for (int hh = 0; hh < GP; ++hh) {
    if (hh >= G) break;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const bool in = half ? in1 : in0;
      const uint32_t b = in ? (ordered_key(half ? v1[hh] : v0[hh]) >> 20) : 0xFFFFu;
      const uint32_t peers = __match_any_sync(0xffffffffu, b);
      if (in && lane == __ffs(peers) - 1) atomicAdd(hist + hh * kTopkBins + b, (uint32_t)__popc(peers));
    }
  }
}

}  // namespace bpkv
