// bpkv_scan_topk_noalloc: scan + top-k with the score scratch in a fixed
// device array that is part of the library image, for callers that cannot
// allocate device memory (see include/bpkv.h).
//
// The array below is a file-scope __device__ symbol.  In host code its name
// stands for a host-side shadow, not a device address, so it is never passed
// to a kernel directly: every call asks the runtime for the symbol's device
// address on the current device and passes that.  (The address is looked up
// again on every call rather than kept: after a device reset the module is
// loaded again and the array may sit elsewhere.)  Every call on a device
// shares the same array and it keeps whatever the previous call left in it.
// The array holds a status word, the scores, then the selection's histograms
// and counters (cleared by an enqueued memset on every call, which allocates
// nothing), candidates and cuts.  Everything else is written before it is
// read.
#include "common.cuh"

namespace bpkv {
cudaError_t launch_scan(const bpkv_cache& c, const float* q, const uint8_t* depths, float* scores, int64_t ld,
                        cudaStream_t st, const void* plan = nullptr, uint32_t* hist = nullptr,
                        int32_t n_sink = 0, int32_t n_recent = 0, int32_t pending = 0,
                        int32_t* status = nullptr);
cudaError_t launch_topk(const bpkv_cache& c, const float* scores, int64_t ld, int32_t k, int32_t n_sink,
                        int32_t n_recent, const SelBufs& b, HistState hs, int32_t* idx, int32_t* status,
                        cudaStream_t st, int32_t pending = 0, uint32_t* selmap = nullptr);
bool scan_counts_hist(const bpkv_cache& c);
}  // namespace bpkv

namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;  // 16 MiB per device, held until exit
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" int bpkv_scan_topk_noalloc(const bpkv_cache* c, const float* q, const uint8_t* depths, int32_t k,
                                      int32_t n_sink, int32_t n_recent, int32_t* idx, void* stream) {
  using namespace bpkv;
  int rc = check_cache(c);
  if (rc != BPKV_OK) return rc;
  rc = check_k(k, n_sink, n_recent);
  if (rc != BPKV_OK) return rc;
  if (!q || !depths || !idx) return BPKV_EINVAL;
  // a 256-byte status word; scores [rows][ld] with ld = n_max rounded up to 64
  // floats; then per row a level-0 and level-1 histogram and its counters,
  // 1024 candidates and the cut
  const size_t rows = (size_t)c->n_seq * c->n_kv_heads * c->group;
  const int64_t ld = (c->n_max + 63) / 64 * 64;
  const size_t off_scores = 256;
  const size_t off_hist = round256(off_scores + rows * (size_t)ld * sizeof(float));
  const size_t off_cand = round256(off_hist + rows * (2 * kTopkBins + kSelCounters) * sizeof(uint32_t));
  const size_t off_cut = round256(off_cand + rows * 1024 * sizeof(unsigned long long));
  const size_t need = off_cut + rows * sizeof(unsigned long long);
  if (need > kNoallocScratchBytes) return BPKV_ENOWORKSPACE;
  // the array's device address on the current device (not its host-side name)
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || scratch == nullptr) return BPKV_ECUDA;
  unsigned char* base = static_cast<unsigned char*>(scratch);
  int32_t* status = reinterpret_cast<int32_t*>(base);
  float* scores = reinterpret_cast<float*>(base + off_scores);
  SelBufs b{reinterpret_cast<uint32_t*>(base + off_hist),
            reinterpret_cast<uint32_t*>(base + off_hist + rows * kTopkBins * sizeof(uint32_t)),
            reinterpret_cast<uint32_t*>(base + off_hist + 2 * rows * kTopkBins * sizeof(uint32_t)),
            reinterpret_cast<unsigned long long*>(base + off_cand), reinterpret_cast<unsigned long long*>(base + off_cut)};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return BPKV_ECUDA;
  if (cudaMemsetAsync(b.hist, 0, rows * (2 * kTopkBins + kSelCounters) * sizeof(uint32_t), st) != cudaSuccess)
    return BPKV_ECUDA;
  const bool scan_counts = scan_counts_hist(*c);
  if (ld > 0 && launch_scan(*c, q, depths, scores, ld, st, nullptr, scan_counts ? b.hist : nullptr, n_sink, n_recent,
                            0, status) != cudaSuccess)
    return BPKV_ECUDA;
  if (launch_topk(*c, scores, ld > 0 ? ld : 1, k, n_sink, n_recent, b,
                  scan_counts ? HistState::kCounted : HistState::kZero, idx, status, st) != cudaSuccess)
    return BPKV_ECUDA;
  return BPKV_OK;
}
