// Shared device helpers of libbpkv (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bpkv.h"

namespace bpkv {

constexpr int kD = BPKV_HEAD_DIM;   // channels per head
constexpr int kBlock = 64;          // tokens per scale block / plane word
constexpr int kPlanes = 4;          // bits per code
constexpr int32_t kMaxK = 8192;     // largest per-head selection size

// Host-side argument checks shared by the entry points (abi.cu): BPKV_OK or
// the status an entry point returns before enqueueing anything.
int check_cache(const bpkv_cache* c);
int check_k(int32_t k, int32_t n_sink, int32_t n_recent);

// Per-unit (sequence, KV head) base offsets of the cache arrays.
struct Unit {
  int64_t nb_cap;  // words per plane row
  int64_t cap;     // token capacity
  __host__ __device__ int64_t plane_base(int64_t unit) const { return unit * kD * kPlanes * nb_cap; }
  __host__ __device__ int64_t scale_base(int64_t unit) const { return unit * kD * nb_cap; }
  __host__ __device__ int64_t row_base(int64_t unit) const { return unit * cap * kD; }
};

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float fp16_bits_to_float(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}

// Order-preserving map float -> uint32 (larger float -> larger key); -0 and +0
// get the same key, as they compare equal.
constexpr int kTopkBins = 4096;  // level-0 histogram: top 12 bits of the ordered key

// per row: candidates gathered, CTAs done, CTAs at the barrier, spare, then
// the row's bucket as k_bucket found it (key prefix, rank left in it, keys in
// it, level of the prefix: 0, or 1 once narrowed by the level-1 histogram)
constexpr int kSelCounters = 8;
constexpr int64_t kLongRowTokens = 262144;  // rows this long get a parallel level-1 histogram

// Selection scratch for rows = N H G query heads.  hist, hist1 and ctr must
// be zero when the selection starts (ctr is left zero by it); they are
// contiguous, so one memset clears all three.
// State of SelBufs::hist and ::ctr when a selection starts.
enum class HistState {
  kCounted,  // histograms counted (by the scan), counters zero
  kZero,     // histograms and counters zero
  kDirty,    // anything: cleared by the selection
};

struct SelBufs {
  uint32_t* hist;            // [rows][kTopkBins] level 0: top 12 key bits
  uint32_t* hist1;           // [rows][kTopkBins] level 1 (next 12 bits) of long rows' bucket keys
  uint32_t* ctr;             // [rows][kSelCounters]
  unsigned long long* cand;  // [rows][1024]
  unsigned long long* cut;   // [rows]
};

__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

// Bounds-checked builds (compiled with -DBPKV_CHECKS=1, a separate library):
// indices the kernels compute into shared and global arrays are checked;
// one outside [0, n) is recorded as BPKV_DEV_BOUNDS in the status word (when
// the call has one) and replaced by 0, so the access stays inside the array.
// Regular builds compile the checks away.
#ifdef BPKV_CHECKS
__device__ __forceinline__ int64_t bpkv_checked(int64_t i, int64_t n, int32_t* status) {
  if (i < 0 || i >= n) {
    set_status(status, BPKV_DEV_BOUNDS);
    return 0;
  }
  return i;
}
#define BPKV_CHK(i, n, st) bpkv_checked((int64_t)(i), (int64_t)(n), (st))
#else
#define BPKV_CHK(i, n, st) (i)
#endif

// Programmatic dependent launch: every kernel of the library lets the next
// kernel on its stream start launching at once, then waits until the kernel
// before it has completed and its writes are visible.  Launches without the
// programmatic attribute make both instructions no-ops in effect.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch with the programmatic-stream-serialization attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Cooperative launch (every CTA of the grid resident at once, so that CTAs
// may wait for one another) with programmatic dependent launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_coop_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Spin limit of in-kernel waits for other CTAs (each round sleeps ~100 ns):
// well above any real wait, then the waiter records BPKV_DEV_TIMEOUT and goes on.
constexpr uint32_t kSpinLimit = 1u << 21;

// ---- asynchronous 16-byte copies global -> shared (this thread's groups) ----

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Both addresses 16-byte aligned; cached in L2 only.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until every copy this thread committed has landed.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

}  // namespace bpkv
