// bpkv_scan_topk_noalloc: scan + top-k with the score scratch in a fixed
// device array that is part of the library image, for callers that cannot
// allocate device memory (see include/bpkv.h).
//
// The array below is a file-scope __device__ symbol.  In host code its name
// stands for a host-side shadow, not a device address, so it is never passed
// to a kernel directly: the first call on each device (with that device
// current) asks the runtime for the symbol's device address once and caches
// it.  Every call on a device shares the same array and it keeps whatever the
// previous call left in it.  The array holds the scores, then the selection's
// histograms and counters (cleared by an enqueued memset on every call, which
// allocates nothing), candidates and cuts.  Everything else is written before
// it is read.
#include <mutex>

#include "common.cuh"

namespace bpkv {
cudaError_t launch_scan(const bpkv_cache& c, const float* q, const uint8_t* depths, float* scores, int64_t ld,
                        cudaStream_t st, const void* plan = nullptr, uint32_t* hist = nullptr,
                        int32_t n_sink = 0, int32_t n_recent = 0, int32_t pending = 0,
                        int32_t* status = nullptr);
cudaError_t launch_topk(const bpkv_cache& c, const float* scores, int64_t ld, int32_t k, int32_t n_sink,
                        int32_t n_recent, const SelBufs& b, HistState hs, int32_t* idx, int32_t* status,
                        cudaStream_t st, int32_t pending = 0);
bool scan_counts_hist(const bpkv_cache& c);
}  // namespace bpkv

namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;  // 16 MiB per device, held until exit
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BPKV_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return BPKV_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return BPKV_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return BPKV_OK;
}

bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" int bpkv_scan_topk_noalloc(const bpkv_cache* c, const float* q, const uint8_t* depths, int32_t k,
                                      int32_t n_sink, int32_t n_recent, int32_t* idx, void* stream) {
  using namespace bpkv;
  if (!c || !q || !depths || !idx) return BPKV_EINVAL;
  if (c->head_dim != kD) return BPKV_EUNSUPPORTED;
  if (c->n_seq < 1 || c->n_kv_heads < 1 || c->group < 1 || c->group > BPKV_MAX_GROUP) return BPKV_EINVAL;
  if (c->n_seq > 65535 || c->n_kv_heads > 65535) return BPKV_EUNSUPPORTED;
  if (c->cap_tokens < 512 || c->cap_tokens % 512 != 0 || c->n_max < 0 || c->n_max > c->cap_tokens)
    return BPKV_EINVAL;
  if (c->residency != 0 && c->residency != 1) return BPKV_EINVAL;
  if (!c->planes || !c->scales || !c->k_rows || !c->v_rows || !c->seq_len) return BPKV_EINVAL;
  if (!is_aligned(c->planes, 16) || !is_aligned(c->scales, 16) || !is_aligned(c->seq_len, 8)) return BPKV_EINVAL;
  if (n_sink < 0 || n_recent < 0 || k < 1 || k > 8192 || (int64_t)n_sink + n_recent > k) return BPKV_EINVAL;
  // scores [rows][ld] with ld = n_max rounded up to 64 floats, then per row a
  // level-0 and level-1 histogram and its counters, 1024 candidates and the cut
  const size_t rows = (size_t)c->n_seq * c->n_kv_heads * c->group;
  const int64_t ld = (c->n_max + 63) / 64 * 64;
  const size_t off_hist = round256(rows * (size_t)ld * sizeof(float));
  const size_t off_cand = round256(off_hist + rows * (2 * kTopkBins + kSelCounters) * sizeof(uint32_t));
  const size_t off_cut = round256(off_cand + rows * 1024 * sizeof(unsigned long long));
  const size_t need = off_cut + rows * sizeof(unsigned long long);
  if (need > kNoallocScratchBytes) return BPKV_ENOWORKSPACE;
  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != BPKV_OK) return rc;
  unsigned char* base = static_cast<unsigned char*>(scratch);
  float* scores = reinterpret_cast<float*>(base);
  SelBufs b{reinterpret_cast<uint32_t*>(base + off_hist),
            reinterpret_cast<uint32_t*>(base + off_hist + rows * kTopkBins * sizeof(uint32_t)),
            reinterpret_cast<uint32_t*>(base + off_hist + 2 * rows * kTopkBins * sizeof(uint32_t)),
            reinterpret_cast<unsigned long long*>(base + off_cand), reinterpret_cast<unsigned long long*>(base + off_cut)};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(b.hist, 0, rows * (2 * kTopkBins + kSelCounters) * sizeof(uint32_t), st) != cudaSuccess)
    return BPKV_ECUDA;
  const bool scan_counts = scan_counts_hist(*c);
  if (ld > 0 &&
      launch_scan(*c, q, depths, scores, ld, st, nullptr, scan_counts ? b.hist : nullptr, n_sink, n_recent) !=
          cudaSuccess)
    return BPKV_ECUDA;
  if (launch_topk(*c, scores, ld > 0 ? ld : 1, k, n_sink, n_recent, b,
                  scan_counts ? HistState::kCounted : HistState::kZero, idx, nullptr, st) != cudaSuccess)
    return BPKV_ECUDA;
  return BPKV_OK;
}
