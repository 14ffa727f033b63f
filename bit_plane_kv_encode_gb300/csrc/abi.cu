// extern "C" entry points of libbpkv (declared in include/bpkv.h): argument
// checks, workspace layout and launch sequencing.  No allocation happens here.
#include <stdio.h>

#include "common.cuh"

namespace bpkv {
cudaError_t launch_encode_append(const bpkv_cache& c, const uint16_t* k_new, const uint16_t* v_new, int32_t t_new,
                                 cudaStream_t st);
cudaError_t launch_alloc_depths(const bpkv_cache& c, const float* q, const float* sigma2, const int32_t* budget_q,
                                uint8_t* depths, cudaStream_t st, uint32_t* tickets = nullptr,
                                void* plan = nullptr, uint32_t* hist = nullptr, uint32_t* ctr = nullptr);
cudaError_t launch_fixed_depths(const bpkv_cache& c, const float* q, int32_t n_channels, int32_t depth,
                                uint8_t* depths, cudaStream_t st, uint32_t* tickets = nullptr, void* plan = nullptr,
                                uint32_t* hist = nullptr, uint32_t* ctr = nullptr);
size_t scan_plan_bytes(int group);
size_t attend_ranges_part_bytes(const bpkv_cache& c);
bool attend_ranges_eligible(const bpkv_cache& c, int32_t k);
cudaError_t launch_attend_ranges(const bpkv_cache& c, const float* q, const float* scores, int64_t ld,
                                 const unsigned long long* cut, int32_t n_sink, int32_t n_recent, float* part,
                                 uint32_t* tickets, float* out, int32_t pending, uint32_t* seq_tick,
                                 cudaStream_t st, uint32_t* rc_stats = nullptr, const uint32_t* selmap = nullptr);
cudaError_t launch_scan(const bpkv_cache& c, const float* q, const uint8_t* depths, float* scores, int64_t ld,
                        cudaStream_t st, const void* plan = nullptr, uint32_t* hist = nullptr,
                        int32_t n_sink = 0, int32_t n_recent = 0, int32_t pending = 0,
                        int32_t* status = nullptr);
cudaError_t launch_topk(const bpkv_cache& c, const float* scores, int64_t ld, int32_t k, int32_t n_sink,
                        int32_t n_recent, const SelBufs& b, HistState hs, int32_t* idx, int32_t* status,
                        cudaStream_t st, int32_t pending = 0, uint32_t* selmap = nullptr);
cudaError_t launch_front(const bpkv_cache& c, const uint16_t* k_new, const uint16_t* v_new, int32_t t_new,
                         const float* q, const float* sigma2, const int32_t* budget_q, int32_t depth_rule,
                         int32_t n_channels, int32_t depth, uint8_t* depths, void* plan, uint32_t* hist,
                         uint32_t* hist1, uint32_t* ctr, uint32_t* tickets, uint32_t* seq_tick, cudaStream_t st,
                         const uint8_t* depths_in, float* q_rot, int32_t* status = nullptr);
bool scan_counts_hist(const bpkv_cache& c);
bool cut_counts_hist(const bpkv_cache& c);
cudaError_t launch_union(const bpkv_cache& c, const int32_t* idx, int32_t k, int32_t* uidx, uint8_t* umask,
                         int32_t* ucount, cudaStream_t st);
cudaError_t launch_attend(const bpkv_cache& c, const float* q, const int32_t* uidx, const uint8_t* umask,
                          const int32_t* ucount, int32_t u_cap, float* part, float* out, bool dense,
                          cudaStream_t st);
size_t attend_part_bytes(const bpkv_cache& c, int64_t rows, bool dense);
cudaError_t launch_bump_len(const bpkv_cache& c, int32_t t_new, cudaStream_t st);
cudaError_t launch_selftest_wait(uint32_t* bar, uint32_t count, uint32_t limit, int32_t* status, cudaStream_t st);
cudaError_t launch_attend_vdepth(const bpkv_cache& c, const float* q, const int32_t* uidx, const uint8_t* umask,
                                 const int32_t* ucount, int32_t u_cap, int32_t budget_v, float* out,
                                 uint8_t* vdepth, float* weight, cudaStream_t st);

namespace {
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

int check_cache(const bpkv_cache* c) {
  if (!c) return BPKV_EINVAL;
  if (c->head_dim != kD) return BPKV_EUNSUPPORTED;
  if (c->n_seq < 1 || c->n_kv_heads < 1 || c->group < 1 || c->group > BPKV_MAX_GROUP) return BPKV_EINVAL;
  if (c->n_seq > 65535 || c->n_kv_heads > 65535) return BPKV_EUNSUPPORTED;
  if (c->cap_tokens < 512 || c->cap_tokens % 512 != 0) return BPKV_EINVAL;
  if (c->n_max < 0 || c->n_max > c->cap_tokens) return BPKV_EINVAL;
  if (c->residency != 0 && c->residency != 1) return BPKV_EINVAL;
  if (!c->planes || !c->scales || !c->k_rows || !c->v_rows || !c->seq_len) return BPKV_EINVAL;
  if (!aligned(c->planes, 16) || !aligned(c->scales, 16) || !aligned(c->k_rows, 16) || !aligned(c->v_rows, 16) ||
      !aligned(c->seq_len, 8))
    return BPKV_EINVAL;
  if ((c->vplanes == nullptr) != (c->vscales == nullptr)) return BPKV_EINVAL;
  if (c->rc_slots != 0) {
    if (c->rc_slots < 64 || c->rc_slots > (1 << 20) || (c->rc_slots & (c->rc_slots - 1)) != 0) return BPKV_EINVAL;
    if (!c->rc_rows || !c->rc_tok || !aligned(c->rc_rows, 16) || !aligned(c->rc_tok, 4)) return BPKV_EINVAL;
  }
  if (c->vplanes && (!aligned(c->vplanes, 16) || !aligned(c->vscales, 16))) return BPKV_EINVAL;
  return BPKV_OK;
}

int check_k(int32_t k, int32_t n_sink, int32_t n_recent) {
  if (n_sink < 0 || n_recent < 0 || k < 1 || k > kMaxK) return BPKV_EINVAL;
  if ((int64_t)n_sink + n_recent > k) return BPKV_EINVAL;
  return BPKV_OK;
}

}  // namespace bpkv

using namespace bpkv;

namespace {

constexpr size_t kAlign = 256;
constexpr int32_t kMaxUnion = 16384;
constexpr int32_t kMaxVdepthRows = 2048;  // union rows the value-depth stage holds per unit

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Workspace layout: status word, then the buffers each call family needs.
struct Layout {
  size_t scores = 0, hist = 0, hist1 = 0, ctr = 0, cand = 0, cut = 0, part = 0, depths = 0, idx = 0, uidx = 0, umask = 0,
         ucount = 0, tickets = 0, seq_tick = 0, plan = 0, q_rot = 0, rc_stats = 0, selmap = 0, total = 0;
};

Layout layout(const bpkv_cache& c, int32_t k, int32_t what) {
  Layout L;
  size_t off = kAlign;  // status word
  const size_t NH = (size_t)c.n_seq * c.n_kv_heads;
  if (what & (BPKV_WS_SCAN_TOPK | BPKV_WS_STEP)) {
    L.scores = off;
    off = align_up(off + NH * c.group * (size_t)c.cap_tokens * sizeof(float));
    // selection scratch; ctr directly follows hist (one memset clears both)
    const size_t rows = NH * c.group;
    L.hist = off;
    L.hist1 = L.hist + rows * kTopkBins * sizeof(uint32_t);
    L.ctr = L.hist1 + rows * kTopkBins * sizeof(uint32_t);
    off = align_up(L.ctr + rows * kSelCounters * sizeof(uint32_t));
    L.cand = off;
    off = align_up(off + rows * 1024 * sizeof(unsigned long long));
    L.cut = off;
    off = align_up(off + rows * sizeof(unsigned long long));
  }
  size_t part = 0;
  if (what & (BPKV_WS_ATTEND | BPKV_WS_STEP)) part = attend_part_bytes(c, (int64_t)c.group * k, false);
  if (what & (BPKV_WS_DENSE | BPKV_WS_STEP)) {
    const size_t pd = attend_part_bytes(c, c.cap_tokens, true);
    if (pd > part) part = pd;
  }
  if (what & BPKV_WS_STEP) {
    const size_t pr = attend_ranges_part_bytes(c);
    if (pr > part) part = pr;
  }
  if (part) {
    L.part = off;
    off = align_up(off + part);
  }
  if (what & BPKV_WS_STEP) {
    L.depths = off;
    off = align_up(off + NH * kD);
    L.idx = off;
    off = align_up(off + NH * c.group * (size_t)k * sizeof(int32_t));
    L.uidx = off;
    off = align_up(off + NH * c.group * (size_t)k * sizeof(int32_t));
    L.umask = off;
    off = align_up(off + NH * c.group * (size_t)k);
    L.ucount = off;
    off = align_up(off + NH * sizeof(int32_t));
    L.tickets = off;
    off = align_up(off + NH * sizeof(uint32_t));
    L.seq_tick = off;
    off = align_up(off + (size_t)c.n_seq * sizeof(uint32_t));
    L.plan = off;
    off = align_up(off + NH * scan_plan_bytes(c.group));
    L.q_rot = off;  // q R when the cache has a basis
    off = align_up(off + NH * c.group * kD * sizeof(float));
    // the row cache's counts of the step: rows found in it, rows
    L.rc_stats = off;
    off = align_up(off + 2 * NH * sizeof(uint32_t));
    // the cut's bits of each head's chosen middle tokens, for the attention
    L.selmap = off;
    off = align_up(off + NH * c.group * (size_t)(c.cap_tokens / 32) * sizeof(uint32_t));
  }
  L.total = off;
  return L;
}

SelBufs sel_bufs(void* ws, const Layout& L) {
  unsigned char* w = static_cast<unsigned char*>(ws);
  return SelBufs{reinterpret_cast<uint32_t*>(w + L.hist), reinterpret_cast<uint32_t*>(w + L.hist1),
                 reinterpret_cast<uint32_t*>(w + L.ctr), reinterpret_cast<unsigned long long*>(w + L.cand),
                 reinterpret_cast<unsigned long long*>(w + L.cut)};
}

int check_ws(const bpkv_cache& c, int32_t k, int32_t what, void* ws, size_t ws_bytes) {
  if (!ws || !aligned(ws, kAlign)) return BPKV_ENOWORKSPACE;
  if (ws_bytes < layout(c, k, what).total) return BPKV_ENOWORKSPACE;
  return BPKV_OK;
}

unsigned char* at(void* ws, size_t off) { return static_cast<unsigned char*>(ws) + off; }

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return BPKV_OK;
  fprintf(stderr, "libbpkv: %s\n", cudaGetErrorString(e));
  return BPKV_ECUDA;
}

}  // namespace

#define BPKV_TRY(x)              \
  do {                           \
    const int rc_ = (x);         \
    if (rc_ != BPKV_OK) return rc_; \
  } while (0)

extern "C" {

int32_t bpkv_version(void) { return 2; }

const char* bpkv_status_string(int status) {
  switch (status) {
    case BPKV_OK: return "ok";
    case BPKV_EINVAL: return "invalid argument";
    case BPKV_ENOWORKSPACE: return "workspace missing or too small";
    case BPKV_ECUDA: return "CUDA error";
    case BPKV_EUNSUPPORTED: return "unsupported shape";
    case BPKV_EDEVICE: return "device-side error flagged";
    default: return "unknown status";
  }
}

size_t bpkv_workspace_size(const bpkv_cache* c, int32_t k, int32_t what) {
  if (check_cache(c) != BPKV_OK || k < 1 || k > kMaxK) return 0;
  return layout(*c, k, what).total;
}

int bpkv_clear_status(void* ws, void* stream) {
  if (!ws) return BPKV_ENOWORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, sizeof(int32_t), as_stream(stream)));
}

int bpkv_read_status(const void* ws, int32_t* status, void* stream) {
  if (!ws || !status) return BPKV_EINVAL;
  BPKV_TRY(cuda_status(cudaStreamSynchronize(as_stream(stream))));
  BPKV_TRY(cuda_status(cudaMemcpy(status, ws, sizeof(int32_t), cudaMemcpyDeviceToHost)));
  return *status ? BPKV_EDEVICE : BPKV_OK;
}

int bpkv_selftest_wait(void* ws, int32_t arrivals, int32_t spin_limit, void* stream) {
  if (!ws || !aligned(ws, kAlign)) return BPKV_ENOWORKSPACE;
  if (arrivals < 1 || arrivals > 1024 || spin_limit < 1 || (uint32_t)spin_limit > kSpinLimit) return BPKV_EINVAL;
  // the barrier counter lives in the workspace's first 256 bytes, after the status word
  uint32_t* bar = reinterpret_cast<uint32_t*>(at(ws, 64));
  return cuda_status(launch_selftest_wait(bar, (uint32_t)arrivals, (uint32_t)spin_limit, static_cast<int32_t*>(ws),
                                          as_stream(stream)));
}

int bpkv_row_cache_stats(const bpkv_cache* c, int32_t k, const void* ws, uint32_t* out, void* stream) {
  BPKV_TRY(check_cache(c));
  if (!ws || !out || k < 1 || k > kMaxK) return BPKV_EINVAL;
  const Layout L = layout(*c, k, BPKV_WS_STEP);
  const size_t NH = (size_t)c->n_seq * c->n_kv_heads;
  BPKV_TRY(cuda_status(cudaStreamSynchronize(as_stream(stream))));
  BPKV_TRY(cuda_status(cudaMemcpy(out, static_cast<const unsigned char*>(ws) + L.rc_stats, 2 * NH * sizeof(uint32_t),
                                  cudaMemcpyDeviceToHost)));
  for (size_t u = 0; u < NH; ++u) out[2 * u + 1] -= out[2 * u];  // rows - hits
  return BPKV_OK;
}

int bpkv_selection_map(const bpkv_cache* c, int32_t k, const void* ws, uint32_t* out, void* stream) {
  BPKV_TRY(check_cache(c));
  if (!ws || !out || k < 1 || k > kMaxK) return BPKV_EINVAL;
  if (cut_counts_hist(*c)) return BPKV_EUNSUPPORTED;  // the cooperative cut writes no map
  const Layout L = layout(*c, k, BPKV_WS_STEP);
  const size_t words = (size_t)c->n_seq * c->n_kv_heads * c->group * (size_t)(c->cap_tokens / 32);
  BPKV_TRY(cuda_status(cudaStreamSynchronize(as_stream(stream))));
  return cuda_status(cudaMemcpy(out, static_cast<const unsigned char*>(ws) + L.selmap, words * sizeof(uint32_t),
                                cudaMemcpyDeviceToHost));
}

int bpkv_encode_append(bpkv_cache* c, const uint16_t* k_new, const uint16_t* v_new, int32_t t_new, void* stream) {
  BPKV_TRY(check_cache(c));
  if (t_new < 1 || !k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)) return BPKV_EINVAL;
  if (c->n_max + t_new > c->cap_tokens) return BPKV_EINVAL;
  BPKV_TRY(cuda_status(launch_encode_append(*c, k_new, v_new, t_new, as_stream(stream))));
  c->n_max += t_new;
  return BPKV_OK;
}

int bpkv_alloc_depths(const bpkv_cache* c, const float* q, const float* sigma2, const int32_t* budget_q,
                      uint8_t* depths, void* stream) {
  BPKV_TRY(check_cache(c));
  if (!q || !sigma2 || !budget_q || !depths) return BPKV_EINVAL;
  return cuda_status(launch_alloc_depths(*c, q, sigma2, budget_q, depths, as_stream(stream)));
}

int bpkv_fixed_depths(const bpkv_cache* c, const float* q, int32_t n_channels, int32_t depth, uint8_t* depths,
                      void* stream) {
  BPKV_TRY(check_cache(c));
  if (!q || !depths || n_channels < 0 || depth < 0 || depth > 4) return BPKV_EINVAL;
  return cuda_status(launch_fixed_depths(*c, q, n_channels, depth, depths, as_stream(stream)));
}

int bpkv_scan(const bpkv_cache* c, const float* q, const uint8_t* depths, float* scores, int64_t ld_scores,
              void* stream) {
  BPKV_TRY(check_cache(c));
  if (!q || !depths || !scores || ld_scores < c->n_max) return BPKV_EINVAL;
  return cuda_status(launch_scan(*c, q, depths, scores, ld_scores, as_stream(stream)));
}

int bpkv_topk(const bpkv_cache* c, const float* scores, int64_t ld_scores, int32_t k, int32_t n_sink,
              int32_t n_recent, int32_t* idx, void* ws, size_t ws_bytes, void* stream) {
  BPKV_TRY(check_cache(c));
  BPKV_TRY(check_k(k, n_sink, n_recent));
  if (!scores || !idx || ld_scores < c->n_max) return BPKV_EINVAL;
  BPKV_TRY(check_ws(*c, k, BPKV_WS_SCAN_TOPK, ws, ws_bytes));
  const Layout L = layout(*c, k, BPKV_WS_SCAN_TOPK);
  return cuda_status(launch_topk(*c, scores, ld_scores, k, n_sink, n_recent, sel_bufs(ws, L), HistState::kDirty, idx,
                                 static_cast<int32_t*>(ws), as_stream(stream)));
}

int bpkv_scan_topk(const bpkv_cache* c, const float* q, const uint8_t* depths, int32_t k, int32_t n_sink,
                   int32_t n_recent, int32_t* idx, void* ws, size_t ws_bytes, void* stream) {
  BPKV_TRY(check_cache(c));
  BPKV_TRY(check_k(k, n_sink, n_recent));
  if (!q || !depths || !idx) return BPKV_EINVAL;
  BPKV_TRY(check_ws(*c, k, BPKV_WS_SCAN_TOPK, ws, ws_bytes));
  const Layout L = layout(*c, k, BPKV_WS_SCAN_TOPK);
  float* scores = reinterpret_cast<float*>(at(ws, L.scores));
  const SelBufs b = sel_bufs(ws, L);
  cudaStream_t st = as_stream(stream);
  const size_t rows = (size_t)c->n_seq * c->n_kv_heads * c->group;
  BPKV_TRY(cuda_status(cudaMemsetAsync(b.hist, 0, rows * (2 * kTopkBins + kSelCounters) * sizeof(uint32_t), st)));
  // the level-0 histograms: counted by the cut kernel when it can, else by the scan
  const bool scan_counts = scan_counts_hist(*c);
  BPKV_TRY(cuda_status(launch_scan(*c, q, depths, scores, c->cap_tokens, st, nullptr, scan_counts ? b.hist : nullptr,
                                   n_sink, n_recent, 0, static_cast<int32_t*>(ws))));
  return cuda_status(launch_topk(*c, scores, c->cap_tokens, k, n_sink, n_recent, b,
                                 scan_counts ? HistState::kCounted : HistState::kZero, idx, static_cast<int32_t*>(ws),
                                 st));
}

int bpkv_union(const bpkv_cache* c, const int32_t* idx, int32_t k, int32_t* uidx, uint8_t* umask, int32_t* ucount,
               void* stream) {
  BPKV_TRY(check_cache(c));
  if (!idx || !uidx || !umask || !ucount || k < 1 || (int64_t)k * c->group > kMaxUnion) return BPKV_EINVAL;
  return cuda_status(launch_union(*c, idx, k, uidx, umask, ucount, as_stream(stream)));
}

int bpkv_sparse_attend(const bpkv_cache* c, const float* q, const int32_t* uidx, const uint8_t* umask,
                       const int32_t* ucount, int32_t u_cap, float* out, void* ws, size_t ws_bytes, void* stream) {
  BPKV_TRY(check_cache(c));
  if (!q || !uidx || !umask || !ucount || !out || u_cap < 1 || u_cap > kMaxUnion) return BPKV_EINVAL;
  if (!ws || !aligned(ws, kAlign)) return BPKV_ENOWORKSPACE;
  const size_t need = kAlign + attend_part_bytes(*c, u_cap, false);
  if (ws_bytes < need) return BPKV_ENOWORKSPACE;
  return cuda_status(launch_attend(*c, q, uidx, umask, ucount, u_cap, reinterpret_cast<float*>(at(ws, kAlign)), out,
                                   false, as_stream(stream)));
}

int bpkv_sparse_attend_vdepth(const bpkv_cache* c, const float* q, const int32_t* uidx, const uint8_t* umask,
                              const int32_t* ucount, int32_t u_cap, int32_t budget_v, float* out, uint8_t* vdepth,
                              float* weight, void* stream) {
  BPKV_TRY(check_cache(c));
  if (!c->vplanes || !q || !uidx || !umask || !ucount || !out) return BPKV_EINVAL;
  if (u_cap < 1 || u_cap > kMaxVdepthRows || budget_v < 0) return BPKV_EINVAL;
  return cuda_status(
      launch_attend_vdepth(*c, q, uidx, umask, ucount, u_cap, budget_v, out, vdepth, weight, as_stream(stream)));
}

int bpkv_dense_attend(const bpkv_cache* c, const float* q, float* out, void* ws, size_t ws_bytes, void* stream) {
  BPKV_TRY(check_cache(c));
  if (!q || !out) return BPKV_EINVAL;
  BPKV_TRY(check_ws(*c, 1, BPKV_WS_DENSE, ws, ws_bytes));
  const Layout L = layout(*c, 1, BPKV_WS_DENSE);
  return cuda_status(launch_attend(*c, q, nullptr, nullptr, nullptr, 1, reinterpret_cast<float*>(at(ws, L.part)),
                                   out, true, as_stream(stream)));
}

int bpkv_decode_step(bpkv_cache* layers, int32_t n_layers, const bpkv_step_args* a, void* ws, size_t ws_bytes,
                     void* stream) {
  if (!layers || n_layers < 1 || !a) return BPKV_EINVAL;
  for (int32_t l = 0; l < n_layers; ++l) {
    BPKV_TRY(check_cache(&layers[l]));
    const bpkv_cache& x = layers[l];
    const bpkv_cache& y = layers[0];
    if (x.n_seq != y.n_seq || x.n_kv_heads != y.n_kv_heads || x.group != y.group || x.cap_tokens != y.cap_tokens)
      return BPKV_EINVAL;
    if (x.n_max + 1 > x.cap_tokens) return BPKV_EINVAL;
  }
  if (!a->k_new || !a->v_new || !a->q || !a->out || (a->flags & ~BPKV_STEP_VDEPTH) != 0) return BPKV_EINVAL;
  const bool vdepth = (a->flags & BPKV_STEP_VDEPTH) != 0;
  if (!aligned(a->k_new, 16) || !aligned(a->v_new, 16)) return BPKV_EINVAL;
  const bool dense = a->depth_rule == BPKV_DEPTH_DENSE;
  if (a->depth_rule == BPKV_DEPTH_WATERFILL && (!a->sigma2 || !a->budget_q)) return BPKV_EINVAL;
  if (a->depth_rule == BPKV_DEPTH_FIXED && (a->fixed_channels < 0 || a->fixed_depth < 0 || a->fixed_depth > 4))
    return BPKV_EINVAL;
  if (a->depth_rule < 0 || a->depth_rule > 3) return BPKV_EINVAL;
  if (a->depth_rule == BPKV_DEPTH_GIVEN && !a->depths_in) return BPKV_EINVAL;
  if (!dense) {
    BPKV_TRY(check_k(a->k, a->n_sink, a->n_recent));
    if ((int64_t)a->k * layers[0].group > kMaxUnion) return BPKV_EINVAL;
  }
  if (vdepth) {
    if (dense || a->budget_v < 0 || (int64_t)a->k * layers[0].group > kMaxVdepthRows) return BPKV_EINVAL;
    for (int32_t l = 0; l < n_layers; ++l)
      if (!layers[l].vplanes) return BPKV_EINVAL;
  }
  const int32_t k = dense ? 1 : a->k;
  BPKV_TRY(check_ws(layers[0], k, BPKV_WS_STEP, ws, ws_bytes));
  const Layout L = layout(layers[0], k, BPKV_WS_STEP);
  cudaStream_t st = as_stream(stream);
  const bpkv_cache& c0 = layers[0];
  const size_t NH = (size_t)c0.n_seq * c0.n_kv_heads;
  const size_t G = c0.group;
  float* scores = reinterpret_cast<float*>(at(ws, L.scores));
  float* part = reinterpret_cast<float*>(at(ws, L.part));
  int32_t* status = static_cast<int32_t*>(ws);
  auto mark = [&](int32_t l, int e) -> int {
    if (!a->stage_events) return BPKV_OK;
    cudaEvent_t ev = static_cast<cudaEvent_t>(a->stage_events[(size_t)l * BPKV_STAGE_EVENTS + e]);
    return cuda_status(cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal));
  };
  BPKV_TRY(cuda_status(cudaMemsetAsync(at(ws, L.rc_stats), 0, 2 * NH * sizeof(uint32_t), st)));
  for (int32_t l = 0; l < n_layers; ++l) {
    bpkv_cache& c = layers[l];
    const uint16_t* kn = a->k_new + (size_t)l * NH * kD;
    const uint16_t* vn = a->v_new + (size_t)l * NH * kD;
    const float* q = a->q + (size_t)l * NH * G * kD;
    float* out = a->out + (size_t)l * NH * G * kD;
    BPKV_TRY(mark(l, 0));
    uint8_t* depths = a->depths_out ? a->depths_out + (size_t)l * NH * kD : at(ws, L.depths);
    int32_t* idx = a->idx_out ? a->idx_out + (size_t)l * NH * G * a->k : reinterpret_cast<int32_t*>(at(ws, L.idx));
    int32_t* uidx = reinterpret_cast<int32_t*>(at(ws, L.uidx));
    uint8_t* umask = at(ws, L.umask);
    int32_t* ucount = reinterpret_cast<int32_t*>(at(ws, L.ucount));
    uint32_t* tickets = reinterpret_cast<uint32_t*>(at(ws, L.tickets));
    uint32_t* seq_tick = reinterpret_cast<uint32_t*>(at(ws, L.seq_tick));
    void* plan = at(ws, L.plan);
    const SelBufs sb = sel_bufs(ws, L);
    const float* s2 = a->sigma2 ? a->sigma2 + (size_t)l * NH * kD : nullptr;
    if (dense) {
      // append (and length update) first, then attention over every row
      BPKV_TRY(cuda_status(launch_encode_append(c, kn, vn, 1, st)));
      c.n_max += 1;
      for (int e = 1; e <= 5; ++e) BPKV_TRY(mark(l, e));
      BPKV_TRY(cuda_status(launch_attend(c, q, nullptr, nullptr, nullptr, 1, part, out, true, st)));
      BPKV_TRY(mark(l, 6));
      continue;
    }
    // append beside depths and plan in one launch; the new token counts in
    // seq_len only from the end of the layer (pending = 1 until then)
    // long rows (as the cut will see them, with the new token) use the level-1 histograms too
    const bool l1 = c.n_max + 1 >= kLongRowTokens;
    BPKV_TRY(cuda_status(launch_front(c, kn, vn, 1, q, s2, a->budget_q, a->depth_rule, a->fixed_channels,
                                      a->fixed_depth, depths, plan, sb.hist, l1 ? sb.hist1 : nullptr, sb.ctr,
                                      tickets, seq_tick, st, a->depths_in,
                                      reinterpret_cast<float*>(at(ws, L.q_rot)), status)));
    c.n_max += 1;
    BPKV_TRY(mark(l, 1));
    BPKV_TRY(mark(l, 2));
    // the level-0 histograms (zeroed by the front kernel): counted by the cut kernel when it can, else by the scan
    const bool scan_counts = scan_counts_hist(c);
    const HistState hs = scan_counts ? HistState::kCounted : HistState::kZero;
    BPKV_TRY(cuda_status(launch_scan(c, q, depths, scores, c.cap_tokens, st, plan, scan_counts ? sb.hist : nullptr,
                                     a->n_sink, a->n_recent, 1, status)));
    BPKV_TRY(mark(l, 3));
    if (vdepth) {
      // index lists, the union, then the value-side depth stage over it
      BPKV_TRY(
          cuda_status(launch_topk(c, scores, c.cap_tokens, a->k, a->n_sink, a->n_recent, sb, hs, idx, status, st, 1)));
      BPKV_TRY(mark(l, 4));
      BPKV_TRY(cuda_status(launch_union(c, idx, a->k, uidx, umask, ucount, st)));
      BPKV_TRY(mark(l, 5));
      BPKV_TRY(cuda_status(launch_bump_len(c, 1, st)));  // the union's rows are final: count the new token
      uint8_t* vd = a->vdepth_out ? a->vdepth_out + (size_t)l * NH * G * a->k : nullptr;
      BPKV_TRY(cuda_status(launch_attend_vdepth(c, q, uidx, umask, ucount, (int32_t)(G * a->k), a->budget_v, out, vd,
                                                nullptr, st)));
      BPKV_TRY(mark(l, 6));
      continue;
    }
    if (attend_ranges_eligible(c, a->k)) {
      // cuts only (lists when asked for); the attention selects by cut, forms
      // the union per token range and finally raises seq_len
      int32_t* iout = a->idx_out ? a->idx_out + (size_t)l * NH * G * a->k : nullptr;
      // the streaming cut also marks the chosen tokens for the attention
      uint32_t* selmap = cut_counts_hist(c) ? nullptr : reinterpret_cast<uint32_t*>(at(ws, L.selmap));
      BPKV_TRY(cuda_status(
          launch_topk(c, scores, c.cap_tokens, a->k, a->n_sink, a->n_recent, sb, hs, iout, status, st, 1, selmap)));
      BPKV_TRY(mark(l, 4));
      BPKV_TRY(mark(l, 5));
      BPKV_TRY(cuda_status(launch_attend_ranges(c, q, scores, c.cap_tokens, sb.cut, a->n_sink, a->n_recent, part,
                                                tickets, out, 1, seq_tick, st,
                                                reinterpret_cast<uint32_t*>(at(ws, L.rc_stats)), selmap)));
      BPKV_TRY(mark(l, 6));
      continue;
    }
    BPKV_TRY(
        cuda_status(launch_topk(c, scores, c.cap_tokens, a->k, a->n_sink, a->n_recent, sb, hs, idx, status, st, 1)));
    BPKV_TRY(mark(l, 4));
    BPKV_TRY(cuda_status(launch_union(c, idx, a->k, uidx, umask, ucount, st)));
    BPKV_TRY(mark(l, 5));
    BPKV_TRY(cuda_status(launch_bump_len(c, 1, st)));  // the union's rows are final: count the new token
    BPKV_TRY(cuda_status(launch_attend(c, q, uidx, umask, ucount, (int32_t)(G * a->k), part, out, false, st)));
    BPKV_TRY(mark(l, 6));
  }
  return BPKV_OK;
}

}  // extern "C"
