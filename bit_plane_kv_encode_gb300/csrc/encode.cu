// Bit-plane encoder / appender (Fathom page, section 3.2: "bit-plane K cache").
//
// One CTA per (touched 64-token block, KV head, sequence), one thread per
// channel.  The CTA stages the block's bf16 keys in shared memory (old tokens
// from the stored rows, new ones from the caller's buffer, which it also copies
// into the row store), takes a = max |k| per channel, rounds s = a/8 to fp16,
// computes c = clip(floor(k / s), -8, 7) + 8 with IEEE float32 division and
// packs bit (3 - p) of the 64 codes into plane word p (token i -> bit i).
#include "common.cuh"

namespace bpkv {

struct EncodeArgs {
  uint64_t* planes;
  uint16_t* scales;
  uint16_t* k_rows;
  uint16_t* v_rows;
  const int64_t* seq_len;
  const uint16_t* k_new;
  const uint16_t* v_new;
  int32_t n_heads;
  int32_t t_new;
  int64_t cap;
  int64_t nb_cap;
};

__global__ void __launch_bounds__(128) k_encode_append(EncodeArgs a) {
  const int s = blockIdx.z, h = blockIdx.y;
  const int64_t unit = (int64_t)s * a.n_heads + h;
  const int64_t n_old = a.seq_len[s];
  const int64_t n_new = n_old + a.t_new;
  const int64_t blk = n_old / kBlock + blockIdx.x;
  const int64_t t0 = blk * kBlock;
  if (t0 >= n_new || n_new > a.cap) return;
  const int cnt = (int)min64(kBlock, n_new - t0);
  const Unit U{a.nb_cap, a.cap};
  uint16_t* krow = a.k_rows + U.row_base(unit);
  uint16_t* vrow = a.v_rows + U.row_base(unit);

  __shared__ __align__(16) uint16_t kb[kBlock][kD];
  // 16-byte vectors: 16 per 256-byte row.
  for (int v = threadIdx.x; v < cnt * 16; v += blockDim.x) {
    const int r = v >> 4, c8 = (v & 15) * 8;
    const int64_t tok = t0 + r;
    uint4 val;
    if (tok < n_old) {
      val = *reinterpret_cast<const uint4*>(krow + tok * kD + c8);
    } else {
      const int64_t src = (unit * a.t_new + (tok - n_old)) * kD + c8;
      val = *reinterpret_cast<const uint4*>(a.k_new + src);
      *reinterpret_cast<uint4*>(krow + tok * kD + c8) = val;
      *reinterpret_cast<uint4*>(vrow + tok * kD + c8) = *reinterpret_cast<const uint4*>(a.v_new + src);
    }
    *reinterpret_cast<uint4*>(&kb[r][c8]) = val;
  }
  __syncthreads();

  const int j = threadIdx.x;
  float amax = 0.f;
  for (int r = 0; r < cnt; ++r) amax = fmaxf(amax, fabsf(bf16_bits_to_float(kb[r][j])));
  // a/8 is exact in float32; values past the largest half saturate to it.
  const __half hs = __float2half_rn(fminf(amax * 0.125f, 65504.f));
  const uint16_t s16 = __half_as_ushort(hs);
  const float sc = __half2float(hs);

  uint64_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
  for (int r = 0; r < cnt; ++r) {
    int c = 8;
    if (s16 != 0) {
      float f = floorf(__fdiv_rn(bf16_bits_to_float(kb[r][j]), sc));
      f = fminf(fmaxf(f, -8.f), 7.f);
      c = static_cast<int>(f) + 8;
    }
    const uint64_t bit = 1ull << r;
    if (c & 8) w0 |= bit;
    if (c & 4) w1 |= bit;
    if (c & 2) w2 |= bit;
    if (c & 1) w3 |= bit;
  }
  uint64_t* pw = a.planes + U.plane_base(unit) + (int64_t)j * kPlanes * a.nb_cap + blk;
  pw[0] = w0;
  pw[a.nb_cap] = w1;
  pw[2 * a.nb_cap] = w2;
  pw[3 * a.nb_cap] = w3;
  a.scales[U.scale_base(unit) + (int64_t)j * a.nb_cap + blk] = s16;
}

__global__ void k_bump_len(int64_t* seq_len, int n_seq, int32_t t_new) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < n_seq) seq_len[s] += t_new;
}

cudaError_t launch_encode_append(const bpkv_cache& c, const uint16_t* k_new, const uint16_t* v_new,
                                 int32_t t_new, cudaStream_t st) {
  EncodeArgs a;
  a.planes = c.planes;
  a.scales = c.scales;
  a.k_rows = c.k_rows;
  a.v_rows = c.v_rows;
  a.seq_len = c.seq_len;
  a.k_new = k_new;
  a.v_new = v_new;
  a.n_heads = c.n_kv_heads;
  a.t_new = t_new;
  a.cap = c.cap_tokens;
  a.nb_cap = c.cap_tokens / kBlock;
  dim3 grid((t_new + kBlock - 1) / kBlock + 1, c.n_kv_heads, c.n_seq);
  k_encode_append<<<grid, 128, 0, st>>>(a);
  k_bump_len<<<(c.n_seq + 127) / 128, 128, 0, st>>>(c.seq_len, c.n_seq, t_new);
  return cudaGetLastError();
}

}  // namespace bpkv
