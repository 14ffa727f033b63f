// Bit-plane encoder / appender (Fathom page, section 3.2: "bit-plane K cache").
//
// One CTA per (touched 64-token block, KV head, sequence), four threads per
// channel (16 tokens each).  The CTA stages the block's bf16 keys in shared memory (old tokens
// from the stored rows, new ones from the caller's buffer, which it also copies
// into the row store), takes a = max |k| per channel, rounds s = a/8 to fp16,
// computes c = clip(floor(k / s), -8, 7) + 8 with IEEE float32 division and
// packs bit (3 - p) of the 64 codes into plane word p (token i -> bit i).
#include "encode_core.cuh"
#include "value_core.cuh"

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
  const float* basis;  // optional [H][D][D]: code the keys k R
  uint64_t* vplanes;   // optional [N][H][cap][4][D/64]: the value rows' own code
  uint16_t* vscales;   // optional [N][H][cap]
};

constexpr int kEncThreads = 4 * kD;  // four threads per channel, 16 tokens each

__global__ void __launch_bounds__(kEncThreads) k_encode_append(EncodeArgs a) {
  pdl_enter();
  const int s = blockIdx.z, h = blockIdx.y;
  const int64_t unit = (int64_t)s * a.n_heads + h;
  const int64_t n_old = a.seq_len[s];
  const int64_t n_new = n_old + a.t_new;
  const int64_t blk = n_old / kBlock + blockIdx.x;
  const int64_t t0 = blk * kBlock;
  if (t0 >= n_new || n_new > a.cap) return;
  const int cnt = (int)min64(kBlock, n_new - t0);
  const Unit U{a.nb_cap, a.cap};
  __shared__ __align__(16) uint16_t kb[kBlock][kD];
  encode_block_cta<4>(kb, a.k_rows + U.row_base(unit), a.v_rows + U.row_base(unit),
                      a.k_new + unit * a.t_new * kD, a.v_new + unit * a.t_new * kD, n_old, t0, cnt,
                      a.planes + U.plane_base(unit), a.scales + U.scale_base(unit), a.nb_cap, blk, 0,
                      a.basis ? a.basis + (int64_t)h * kD * kD : nullptr);
  if (a.vplanes)
    encode_value_rows(a.v_new + unit * a.t_new * kD, n_old, t0, cnt, a.vplanes + unit * a.cap * (kPlanes * kD / 64),
                      a.vscales + unit * a.cap, 0, kEncThreads / 32);
}

__global__ void k_bump_len(int64_t* seq_len, int n_seq, int32_t t_new) {
  pdl_enter();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < n_seq) seq_len[s] += t_new;
}

cudaError_t launch_bump_len(const bpkv_cache& c, int32_t t_new, cudaStream_t st) {
  return launch_pdl(k_bump_len, dim3((c.n_seq + 127) / 128), dim3(128), 0, st, c.seq_len, (int)c.n_seq, t_new);
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
  a.basis = c.basis;
  a.vplanes = c.vplanes;
  a.vscales = c.vscales;
  dim3 grid((t_new + kBlock - 1) / kBlock + 1, c.n_kv_heads, c.n_seq);
  cudaError_t e = launch_pdl(k_encode_append, grid, dim3(kEncThreads), 0, st, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_bump_len, dim3((c.n_seq + 127) / 128), dim3(128), 0, st, c.seq_len, (int)c.n_seq, t_new);
}

}  // namespace bpkv
