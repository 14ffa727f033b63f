// Prefix-plane key scan (Fathom page, section 1 observation 2 and section 3.1):
// each key is scored from only the first t_j planes of each channel j and the
// block scales of the channels with t_j > 0; the bytes read are b n / 8.
//
// khat = s ((c_t + 1/2) 2^(4-t) - 8) = (s q 2^(4-t)) (c_t - 2^(t-1) + 1/2) / q,
// so each (block, channel, head) contributes u * e with u = s * q_gj * 2^(4-t)
// (one rounding) and the exact half-integer e = c_t - 2^(t-1) + 1/2.
//
// Launch: one CTA per (chunk of kChunkBlocks blocks, KV head, sequence).  The
// CTA builds the list of active channels, stages their plane words and scales
// for the chunk in shared memory with coalesced loads, then each thread scores
// tokens (lane = token, so the words a warp reads are shared broadcasts).
#include "common.cuh"

namespace bpkv {

constexpr int kChunkBlocks = 16;               // 1024 tokens per CTA
constexpr int kScanThreads = 256;
constexpr int kMaxPlaneRows = kD * kPlanes;    // 512

struct ScanArgs {
  const uint64_t* planes;
  const uint16_t* scales;
  const int64_t* seq_len;
  const float* q;
  const uint8_t* depths;
  float* scores;
  int64_t ld;
  int64_t nb_cap;
  int32_t n_heads;
  int32_t group;
};

struct ScanSmem {
  uint64_t words[kMaxPlaneRows * kChunkBlocks];  // 64 KB
  float scale[kD * kChunkBlocks];                // 8 KB
  float w[kD * BPKV_MAX_GROUP];                  // q * 2^(4-t), per active channel
  float off[kD];                                 // 2^(t-1) - 1/2
  int16_t row_of_plane[kMaxPlaneRows];           // j * 4 + p of each staged plane row
  int16_t ch[kD];                                // active channel -> j
  int16_t t[kD];                                 // active channel -> depth
  int16_t pofs[kD];                              // active channel -> first staged row
  int n_act, n_rows;
};

__global__ void __launch_bounds__(kScanThreads) k_scan(ScanArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ScanSmem& S = *reinterpret_cast<ScanSmem*>(smem_raw);
  const int s = blockIdx.z, h = blockIdx.y;
  const int64_t unit = (int64_t)s * a.n_heads + h;
  const int64_t n = a.seq_len[s];
  const int64_t b0 = (int64_t)blockIdx.x * kChunkBlocks;
  if (b0 * kBlock >= n) return;
  const int64_t nb_valid = (n + kBlock - 1) / kBlock;
  const int nbl = (int)min64(kChunkBlocks, nb_valid - b0);
  const int tid = threadIdx.x;
  const int G = a.group;

  if (tid == 0) {
    int na = 0, nr = 0;
    for (int j = 0; j < kD; ++j) {
      const int t = a.depths[unit * kD + j];
      if (t == 0) continue;
      S.ch[na] = (int16_t)j;
      S.t[na] = (int16_t)t;
      S.pofs[na] = (int16_t)nr;
      for (int p = 0; p < t; ++p) S.row_of_plane[nr + p] = (int16_t)(j * 4 + p);
      nr += t;
      ++na;
    }
    S.n_act = na;
    S.n_rows = nr;
  }
  __syncthreads();
  const int n_act = S.n_act, n_rows = S.n_rows;
  const float* qp = a.q + unit * G * kD;
  for (int e = tid; e < n_act * G; e += kScanThreads) {
    const int ai = e / G, g = e % G;
    const int t = S.t[ai];
    S.w[ai * G + g] = ldexpf(qp[g * kD + S.ch[ai]], 4 - t);
  }
  for (int ai = tid; ai < n_act; ai += kScanThreads) S.off[ai] = ldexpf(1.f, S.t[ai] - 1) - 0.5f;
  const uint64_t* pl = a.planes + unit * kD * kPlanes * a.nb_cap;
  for (int e = tid; e < n_rows * kChunkBlocks; e += kScanThreads) {
    const int r = e / kChunkBlocks, lb = e % kChunkBlocks;
    if (lb < nbl) S.words[r * kChunkBlocks + lb] = pl[(int64_t)S.row_of_plane[r] * a.nb_cap + b0 + lb];
  }
  const uint16_t* sp = a.scales + unit * kD * a.nb_cap;
  for (int e = tid; e < n_act * kChunkBlocks; e += kScanThreads) {
    const int ai = e / kChunkBlocks, lb = e % kChunkBlocks;
    if (lb < nbl) S.scale[ai * kChunkBlocks + lb] = fp16_bits_to_float(sp[(int64_t)S.ch[ai] * a.nb_cap + b0 + lb]);
  }
  __syncthreads();

  float* out = a.scores + unit * G * a.ld;
  for (int x = tid; x < nbl * kBlock; x += kScanThreads) {
    const int64_t tok = b0 * kBlock + x;
    if (tok >= n) break;
    const int lb = x / kBlock, bit = x % kBlock;
    float acc[BPKV_MAX_GROUP];
#pragma unroll
    for (int g = 0; g < BPKV_MAX_GROUP; ++g) acc[g] = 0.f;
    for (int ai = 0; ai < n_act; ++ai) {
      const int t = S.t[ai];
      const int r0 = S.pofs[ai];
      int c = 0;
      for (int p = 0; p < t; ++p) c = (c << 1) | (int)((S.words[(r0 + p) * kChunkBlocks + lb] >> bit) & 1ull);
      const float e = (float)c - S.off[ai];
      const float sc = S.scale[ai * kChunkBlocks + lb];
#pragma unroll
      for (int g = 0; g < BPKV_MAX_GROUP; ++g)
        if (g < G) acc[g] = fmaf(sc * S.w[ai * G + g], e, acc[g]);
    }
#pragma unroll
    for (int g = 0; g < BPKV_MAX_GROUP; ++g)
      if (g < G) out[g * a.ld + tok] = acc[g];
  }
}

size_t scan_smem_bytes() { return sizeof(ScanSmem); }

cudaError_t launch_scan(const bpkv_cache& c, const float* q, const uint8_t* depths, float* scores, int64_t ld,
                        cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_scan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(ScanSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  ScanArgs a{c.planes, c.scales, c.seq_len, q, depths, scores, ld, c.cap_tokens / kBlock, c.n_kv_heads, c.group};
  const int64_t chunks = (c.n_max + kChunkBlocks * kBlock - 1) / (kChunkBlocks * kBlock);
  if (chunks == 0) return cudaSuccess;
  dim3 grid((unsigned)chunks, c.n_kv_heads, c.n_seq);
  k_scan<<<grid, kScanThreads, sizeof(ScanSmem), st>>>(a);
  return cudaGetLastError();
}

}  // namespace bpkv
