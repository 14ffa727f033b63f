/*
 * bpkv.h - C ABI of libbpkv: query-dependent prefix reads of a bit-plane K
 * cache during decode, on one GB300 (sm_103a).
 *
 * The method is the one of "Fathom: per-query read depth for sparse decoding
 * over an offloaded KV cache" (the Fathom page):
 *   section 3.2   keys as 4-bit per-channel uniform symmetric codes, one fp16
 *                 scale per 64-token block, stored as channel-major bit planes;
 *   section 1     (observation 1) per-query depth per channel by reverse
 *                 water-filling on g_j 4^-t_j; (observation 2) the first t planes
 *                 of a channel are its t-bit mid-rise quantiser;
 *   section 3.1   Eq. 1: the scan reads b n / 8 bytes per (sequence, layer, KV
 *                 head), the winner rows k_U R;
 *   section 2     ("Top-k decoding") 4 sink and 32 recent tokens always kept,
 *                 the other k - 36 are each query head's top scores, exact
 *                 attention over the selected set; ("SparQ") fixed channel sets
 *                 ranked by the group's summed |q|.
 *
 * Conventions for every call:
 *   - All pointers are caller-owned.  Device pointers unless stated otherwise.
 *     The library allocates nothing: scratch comes from the caller's workspace
 *     (size from bpkv_workspace_size).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work on it and return; results are ready when the stream is.
 *   - Return value: BPKV_OK or a negative status.  Argument errors are detected
 *     on the host before anything is enqueued.  BPKV_ECUDA reports a failed
 *     launch (cudaGetLastError after enqueueing).  Errors found by kernels while
 *     running are written to the workspace's status word; read it with
 *     bpkv_read_status.
 *   - Head dimension D = 128; group G in 1..8; cap_tokens a multiple of 512.
 *   - Integer/bit outputs (planes, scales, depths, indices, union) are exact.
 *     Scores are float32 sums; attention is float32 with float32 softmax.
 */
#ifndef BPKV_H
#define BPKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------- status codes */
#define BPKV_OK 0
#define BPKV_EINVAL (-1)       /* invalid argument; nothing was enqueued */
#define BPKV_ENOWORKSPACE (-2) /* workspace NULL or smaller than bpkv_workspace_size */
#define BPKV_ECUDA (-3)        /* a CUDA launch or API call failed */
#define BPKV_EUNSUPPORTED (-4) /* valid but unsupported shape (e.g. D != 128) */
#define BPKV_EDEVICE (-5)      /* a kernel flagged an error in the status word */

/* device status word bits (bpkv_read_status) */
#define BPKV_DEV_OVERFLOW 1    /* append would pass cap_tokens; nothing written */
#define BPKV_DEV_SELECT 2      /* a selection produced more rows than its output holds */
#define BPKV_DEV_TIMEOUT 4     /* a wait inside a kernel for the other CTAs of its grid gave up */
#define BPKV_DEV_BOUNDS 8      /* bounds-checked builds only: a computed index was outside its array
                                  (the access was redirected to element 0) */

#define BPKV_MAX_GROUP 8
#define BPKV_HEAD_DIM 128

/* ------------------------------------------------------------- the cache */
/*
 * One layer's cache for N sequences x H KV heads.  Layouts (row-major, last
 * index fastest), NB = cap_tokens / 64:
 *   planes  uint64 [N][H][D][4][NB]  word (j, p, b): bit i is bit (3 - p) of the
 *                                    code of token 64 b + i (p = 0: most
 *                                    significant bit = sign), so the first t
 *                                    planes of channel j are t NB contiguous words
 *   scales  uint16 [N][H][D][NB]     fp16 bit pattern of s = blockmax / 8
 *                                    (round to nearest even, saturated at 65504)
 *   k_rows  uint16 [N][H][cap][D]    bf16 keys as appended
 *   v_rows  uint16 [N][H][cap][D]    bf16 values as appended
 *   seq_len int64  [N]               device memory: tokens stored per sequence
 * residency 0: planes, scales and rows are in device memory.  residency 1: they
 * are in host memory the GPU can read (pinned with cudaHostAlloc/cudaHostRegister,
 * or any memory on a system with address translation); kernels read them in
 * place over the host link.  seq_len is always device memory.
 * planes, scales and the rows must start on 16-byte boundaries (BPKV_EINVAL
 * otherwise); with cap_tokens a multiple of 1024 and the four arrays on 256-byte
 * boundaries every plane row segment, scale segment and row a kernel reads
 * starts on a 32-byte sector, which matters for host memory, whose reads L2 does
 * not keep (a segment that starts inside a sector moves one more sector over the
 * link).
 * n_max is host state: an upper bound of every seq_len[i], used to size
 * launches; bpkv_encode_append raises it.
 * basis (optional, NULL: the raw channels) float [H][D][D] in device memory: an
 * orthogonal basis per KV head for the coded keys (Fathom page, contributions:
 * the keys' KLT planes for models without QK norm; ReadKV page, section 5.1:
 * a Hadamard-sign transform).  The planes and scales then code the keys k R
 * (channel l = sum_j k_j R[j][l], one float32 fused multiply-add chain in order
 * j = 0 .. D-1, rounded to bf16); bpkv_decode_step allocates depths and scores
 * with q R (sigma2 is then the variance in the basis), and the rows and the
 * exact attention stay in the original channels.  The stand-alone depth, scan
 * and top-k calls take q already in the basis (bpkv_rotate).  Set the basis
 * before the first append.
 * vplanes, vscales (optional, NULL: no value planes; both or neither) hold the
 * values' own 4-bit code for the value-side read depth (ReadKV page,
 * sections 5.3-5.4): one fp16 scale per row, token-major planes
 *   vplanes uint64 [N][H][cap][4][D/64]  word (x, p, w): bit b is bit (3 - p) of
 *                                        the code of channel 64 w + b of token x
 *   vscales uint16 [N][H][cap]           fp16 bit pattern of s = max_j |v_xj| / 8
 * with the keys' code, c = clip(floor(v / s), -8, 7) + 8 (all 8 when s rounds
 * to 0), so the first t planes of a row are its t-bit mid-rise quantiser.
 * bpkv_encode_append and bpkv_decode_step write them for every appended token
 * when present (same residency as the rows; 16-byte aligned).
 * rc_rows, rc_tok, rc_slots (optional, rc_slots = 0: none; host-resident
 * caches only) are a device-memory cache of recently selected rows, so that
 * rows selected again in later steps are read from HBM instead of over the
 * host link (the KVDrive page's reuse of critical KV across steps; Fathom
 * page, section 1: the winner rows' k_U R term):
 *   rc_rows uint16 [N][H][rc_slots][2][D]  the bf16 K row, then the V row, held in each slot
 *   rc_tok  int32  [N][H][rc_slots]        token held by each slot, -1 for none (the caller
 *                                          fills it with -1 before the first step)
 * rc_slots is a power of two from 64 to 2^20.  bpkv_decode_step splits a
 * sequence's tokens into ranges (one attention CTA each) and gives range r
 * the slots [r P, r P + P), P = min(rc_slots / ranges, 1024); token x of the
 * range can sit only in slot r P + x mod P.  A selected row is read from its
 * slot when the slot holds that token; a row read over the link is written
 * into its slot by the same kernel, unless the slot serves another selected
 * row in that step (of several with one free slot, the latest token wins).
 * Rows never change once appended, so a cached row is always the current
 * one; results are identical with or without the row cache.
 */
typedef struct bpkv_cache {
  int32_t n_seq;
  int32_t n_kv_heads;
  int32_t group;
  int32_t head_dim;
  int64_t cap_tokens;
  int64_t n_max;
  int32_t residency;
  int32_t reserved;
  uint64_t *planes;
  uint16_t *scales;
  uint16_t *k_rows;
  uint16_t *v_rows;
  int64_t *seq_len;
  const float *basis;
  uint64_t *vplanes;
  uint16_t *vscales;
  uint16_t *rc_rows;
  int32_t *rc_tok;
  int32_t rc_slots;
  int32_t rc_reserved;
} bpkv_cache;

/* ------------------------------------------------------------- workspace */
#define BPKV_WS_SCAN_TOPK 1   /* bpkv_topk / bpkv_scan_topk */
#define BPKV_WS_ATTEND 2      /* bpkv_sparse_attend */
#define BPKV_WS_DENSE 4       /* bpkv_dense_attend */
#define BPKV_WS_STEP 8        /* bpkv_decode_step (includes everything it needs) */

/* Bytes of workspace the calls named in `what` (OR of BPKV_WS_*) need for this
 * cache and selection size k.  0 on invalid arguments.  The workspace must be
 * device memory aligned to 256 bytes; its first 256 bytes hold the status word. */
size_t bpkv_workspace_size(const bpkv_cache *c, int32_t k, int32_t what);

/* Clear the status word (enqueued on `stream`). */
int bpkv_clear_status(void *ws, void *stream);

/* Synchronise `stream`, then copy the status word to *status (0 = no error).
 * Returns BPKV_EDEVICE when it is non-zero. */
int bpkv_read_status(const void *ws, int32_t *status, void *stream);

const char *bpkv_status_string(int status);

/*
 * Self-test of failure detection (the pages have no counterpart: this checks
 * the library's own bounded waits).  One CTA waits, as the selection's CTAs
 * do for one another, at a barrier that expects `arrivals` CTAs; only it
 * arrives, so for arrivals > 1 the wait gives up after spin_limit rounds of
 * about 100 ns (1 .. 2^21), records BPKV_DEV_TIMEOUT in the status word of
 * `ws` (device memory, 256-byte aligned, at least 256 bytes; the barrier
 * counter uses bytes 64..67) and returns, leaving the context usable.
 * arrivals = 1 completes at once.  BPKV_EINVAL for arrivals outside 1..1024
 * or spin_limit outside 1 .. 2^21.
 */
int bpkv_selftest_wait(void *ws, int32_t arrivals, int32_t spin_limit, void *stream);
int32_t bpkv_version(void);

/* ------------------------------------------------------------- encode (F1, F2) */
/*
 * Fathom page section 3.2.  Append t_new tokens to every sequence: rows
 * k_new/v_new [N][H][t_new][D] bf16 (device) are written at positions
 * seq_len[i] .. seq_len[i]+t_new-1, every 64-token block they touch is
 * (re)encoded from the stored rows (the open tail block is re-encoded because
 * its blockmax, hence its scale, may grow), then seq_len[i] += t_new and
 * c->n_max += t_new.  Per block and channel: a = max |k| over the tokens present,
 * s = fp16(a / 8), c = clip(floor(k / s), -8, 7) + 8 (float32 IEEE division), all
 * codes 8 when s rounds to 0; bits of absent tokens are 0.
 * Errors: EINVAL when n_max + t_new > cap_tokens or t_new < 1.
 */
int bpkv_encode_append(bpkv_cache *c, const uint16_t *k_new, const uint16_t *v_new, int32_t t_new,
                       void *stream);

/* ------------------------------------------------------------- depths (F4, F5) */
/*
 * Fathom page section 1, observation 1.  For each (sequence, KV head):
 * g_j = sum_h q_hj^2 sigma2_j over its G query heads (float32, heads in order,
 * no fused multiply-add); items (j, t) for t = 0..3 with value g_j 4^-t; each
 * costs 4 quarter-bits per token, plus 1 (the fp16 scale) for t = 0.  Items are
 * taken in order of value (ties: lower channel first) until one has value <= 0
 * or does not fit budget_q[i] quarter-bits.  depths[i][h][j] = bits taken.
 *   q        float [N][H][G][D]
 *   sigma2   float [N][H][D]   channel variances of the keys
 *   budget_q int32 [N]         per-sequence budget in quarter-bits per token (4 b)
 *   depths   uint8 [N][H][D]   out, values 0..4
 */
int bpkv_alloc_depths(const bpkv_cache *c, const float *q, const float *sigma2, const int32_t *budget_q,
                      uint8_t *depths, void *stream);

/*
 * Fathom page section 2 ("SparQ", "thumbnail"): fixed-depth channel sets.  The
 * n_channels channels with the largest sum_h |q_hj| (float32, heads in order,
 * ties to the lower index) get depth `depth`, the others 0.  n_channels >= D
 * reads all channels (the 2-bit thumbnail: n_channels = 128, depth = 2; the
 * 136-bit SparQ r = 32 set: 32, 4).
 */
int bpkv_fixed_depths(const bpkv_cache *c, const float *q, int32_t n_channels, int32_t depth,
                      uint8_t *depths, void *stream);

/*
 * Fathom page section 2 ("Double Sparsity"): a channel set chosen offline from
 * calibration statistics.  For each of n_units units (e.g. every (layer, KV
 * head), or every (sequence, KV head) of one layer), the statistic of channel j
 * is mean|q_j| over the unit's calibration queries and its `group` query heads
 * times mean|k_j| over its calibration keys; the n_channels channels with the
 * largest statistic (ties to the lower index) get depth `depth`, the others 0
 * (32 channels at depth 4 read 136 bits per token).  Sums run in double in
 * storage order (queries, then heads; keys in order), each mean divides its sum
 * once and the product is one double multiplication, so the choice matches a
 * plain CPU evaluation exactly.  Inputs must be finite.
 *   q_cal   float [n_units][m_q][group][D]   calibration queries (device)
 *   k_cal   bf16  [n_units][m_k][D]          calibration keys (device)
 *   depths  uint8 [n_units][D]               out (device); pass to bpkv_decode_step
 *                                             with BPKV_DEPTH_GIVEN or to the scans
 * BPKV_EINVAL for n_units, group, m_q or m_k below 1, group above
 * BPKV_MAX_GROUP, n_channels below 0 or depth outside 0..4.
 */
int bpkv_calibrate_channels(const float *q_cal, const uint16_t *k_cal, int32_t n_units, int32_t group, int64_t m_q,
                            int64_t m_k, int32_t n_channels, int32_t depth, uint8_t *depths, void *stream);

/*
 * y = x R per KV head: x, y float [n_seq][H][rows][D] (device), basis R float
 * [H][D][D]; channel l of a row is one float32 fused multiply-add chain
 * sum_j x_j R[j][l] in order j = 0 .. D-1 (the same arithmetic as the decode
 * step's q R).  x and y may not overlap.
 */
int bpkv_rotate(const float *basis, int32_t n_seq, int32_t n_kv_heads, int64_t rows, const float *x, float *y,
                void *stream);

/* ------------------------------------------------------------- scan (F3, F7) */
/*
 * Fathom page sections 1 and 3.1.  score[i][h][g][x] = sum_j q_gj khat_xj(t_j)
 * for every token x < seq_len[i], where for t = depths[i][h][j] > 0
 * khat = s ((c_t + 1/2) 2^(4-t) - 8), c_t the first t planes of the code and
 * s the block scale; channels with t = 0 are not read (depth values above 4
 * are read as 4).  No 1/sqrt(D) factor.
 *   scores float [N][H][G][ld_scores], ld_scores >= n_max; entries past
 *   seq_len[i] are not written.
 */
int bpkv_scan(const bpkv_cache *c, const float *q, const uint8_t *depths, float *scores, int64_t ld_scores,
              void *stream);

/* ------------------------------------------------------------- select (F8, F9) */
/*
 * Fathom page section 2 ("Top-k decoding").  For each query head, tokens
 * [0, n_sink) and [n - n_recent, n) plus the k - n_sink - n_recent highest
 * scores among the rest (ties: lower token index); all n tokens when those are
 * at most k.  idx [N][H][G][k] int32 out: ascending token indices, -1 padded.
 * Needs workspace BPKV_WS_SCAN_TOPK.  k >= n_sink + n_recent, k <= 8192.
 */
int bpkv_topk(const bpkv_cache *c, const float *scores, int64_t ld_scores, int32_t k, int32_t n_sink,
              int32_t n_recent, int32_t *idx, void *ws, size_t ws_bytes, void *stream);

/* bpkv_scan into the workspace followed by bpkv_topk.  The scan also counts
 * each row's first-level selection histogram into the workspace (cleared by an
 * enqueued memset first), which the top-k then reads instead of counting it. */
int bpkv_scan_topk(const bpkv_cache *c, const float *q, const uint8_t *depths, int32_t k, int32_t n_sink,
                   int32_t n_recent, int32_t *idx, void *ws, size_t ws_bytes, void *stream);

/*
 * bpkv_scan_topk without a workspace, for callers that cannot allocate device
 * memory: for example a host program whose own pool already holds all of the
 * GPU's memory, or a loop that must not pay the device-wide synchronisation a
 * cudaMalloc/cudaFree can cause.  The Fathom page has no counterpart of this
 * call; its results are identical to bpkv_scan_topk's.
 * The scratch (a status word, scores and selection buffers) is a fixed 16 MiB
 * array built into the library, held on every GPU that loads the library
 * until the process exits; requests needing more (rows = N * H * G; 256 +
 * rows * (4 * round_up(n_max, 64) + 40984) bytes plus under 1 KiB of
 * alignment > 16 MiB) return BPKV_ENOWORKSPACE.  The call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine); it enqueues
 * memsets of the status word and the selection counters.  Every call looks
 * up the array's device address on the current device; the first call on a
 * device also loads the library's kernels there, so make it before any
 * stream capture.  After a device reset the next call finds the array again.
 * All calls on a device share the one array, so calls whose work overlaps on
 * the GPU (other streams, other threads) race and must be serialised by the
 * caller.  No device status word is reported: if the selection's bounded wait
 * for its other CTAs gives up (BPKV_DEV_TIMEOUT on the workspace call), idx
 * can be wrong without any error returned.
 */
int bpkv_scan_topk_noalloc(const bpkv_cache *c, const float *q, const uint8_t *depths, int32_t k,
                           int32_t n_sink, int32_t n_recent, int32_t *idx, void *stream);

/*
 * GQA union of one KV head's G selections (Fathom page sections 1 and 3.1:
 * k_U <= G k distinct winner rows per KV head, fetched once).
 *   idx   int32 [N][H][G][k] ascending, -1 padded (as bpkv_topk writes it)
 *   uidx  int32 [N][H][G*k]  out: distinct rows ascending, -1 padded
 *   umask uint8 [N][H][G*k]  out: bit g set when query head g selected the row
 *   ucount int32 [N][H]      out: union size
 * G * k <= 16384.
 */
int bpkv_union(const bpkv_cache *c, const int32_t *idx, int32_t k, int32_t *uidx, uint8_t *umask,
               int32_t *ucount, void *stream);

/* ------------------------------------------------------------- attention (F10) */
/*
 * Fathom page section 2: exact attention of each query head over its own
 * selected rows, o_g = sum_x softmax_x(q_g . k_x / sqrt(D)) v_x with the stored
 * bf16 rows, read once per union row for all G heads (split over row chunks,
 * combined with log-sum-exp).  A head with no selected row gets zeros.
 *   uidx/umask/ucount as bpkv_union writes them, u_cap = their row stride (G k)
 *   out float [N][H][G][D]
 * Needs workspace BPKV_WS_ATTEND.
 */
int bpkv_sparse_attend(const bpkv_cache *c, const float *q, const int32_t *uidx, const uint8_t *umask,
                       const int32_t *ucount, int32_t u_cap, float *out, void *ws, size_t ws_bytes,
                       void *stream);

/*
 * Value-side read depth (ReadKV page, section 5.3: the approximate attention
 * decides each value row's depth; section 5.4: the allocator), over the union
 * of each KV head's selections: head h's probabilities p_h(r) = softmax over
 * its own rows of q_h . k_r / sqrt(D) with the exact bf16 keys; row weights
 * a_r = sum_h p_h(r)^2 (float32); depths t_r by greedy on a_r 4^-t_r, one
 * plane per item, largest first (ties to the lower row), at most budget_v
 * planes per (sequence, KV head), items worth <= 0 never taken; then
 * o_h = sum_r p_h(r) vhat_r(t_r) with each value row read to its depth from
 * the cache's vplanes / vscales: vhat = s ((c_t + 1/2) 2^(4-t) - 8), the zero
 * row at t = 0.  The depths are those of the float32 weights: where two
 * weights are within float32 rounding the order may differ from an exact
 * evaluation's.
 *   uidx/umask/ucount, u_cap as bpkv_union writes them (u_cap <= 2048)
 *   out    float [N][H][G][D]
 *   vdepth uint8 [N][H][u_cap] (optional, NULL to skip): depth of each union row
 *   weight float [N][H][u_cap] (optional, NULL to skip): a_r
 * BPKV_EINVAL when the cache has no value planes, u_cap is outside 1..2048 or
 * budget_v < 0.  No workspace.
 */
int bpkv_sparse_attend_vdepth(const bpkv_cache *c, const float *q, const int32_t *uidx, const uint8_t *umask,
                              const int32_t *ucount, int32_t u_cap, int32_t budget_v, float *out, uint8_t *vdepth,
                              float *weight, void *stream);

/* Dense bf16 attention over every stored row (the dense baseline), same output
 * layout.  Needs workspace BPKV_WS_DENSE. */
int bpkv_dense_attend(const bpkv_cache *c, const float *q, float *out, void *ws, size_t ws_bytes,
                      void *stream);

/* ------------------------------------------------------------- decode step */
#define BPKV_DEPTH_WATERFILL 0  /* bpkv_alloc_depths with sigma2 and budget_q */
#define BPKV_DEPTH_FIXED 1      /* bpkv_fixed_depths(fixed_channels, fixed_depth) */
#define BPKV_DEPTH_DENSE 2      /* no scan: dense attention over all rows */
#define BPKV_DEPTH_GIVEN 3      /* the caller's depths_in (e.g. from bpkv_calibrate_channels) */

typedef struct bpkv_step_args {
  const uint16_t *k_new;    /* [L][N][H][D] bf16: the one new token per sequence and layer */
  const uint16_t *v_new;    /* [L][N][H][D] bf16 */
  const float *q;           /* [L][N][H][G][D] */
  const float *sigma2;      /* [L][N][H][D] (water-filling only) */
  const int32_t *budget_q;  /* [N] quarter-bits per token (water-filling only) */
  int32_t depth_rule;       /* BPKV_DEPTH_* */
  int32_t fixed_channels;   /* BPKV_DEPTH_FIXED */
  int32_t fixed_depth;      /* BPKV_DEPTH_FIXED */
  int32_t k, n_sink, n_recent;
  float *out;               /* [L][N][H][G][D] */
  uint8_t *depths_out;      /* optional [L][N][H][D], NULL to skip */
  int32_t *idx_out;         /* optional [L][N][H][G][k], NULL to skip */
  void *const *stage_events;/* optional [L][BPKV_STAGE_EVENTS] cudaEvent_t, NULL to skip:
                               recorded on `stream` (as external events, so they also
                               time graph replays) before encode, depths, scan, top-k,
                               union, attention and after attention */
  int32_t flags;            /* BPKV_STEP_* (0: keys only) */
  const uint8_t *depths_in; /* [L][N][H][D] BPKV_DEPTH_GIVEN: depth of every channel (values above
                               4 read as 4; depths_out, if given, receives them as read) */
  int32_t budget_v;         /* BPKV_STEP_VDEPTH: value planes per (sequence, KV head) */
  uint8_t *vdepth_out;      /* BPKV_STEP_VDEPTH, optional [L][N][H][G k]: depth of each union row */
} bpkv_step_args;

/*
 * Hits and misses of the row cache in the last bpkv_decode_step that used
 * this workspace (summed over its layers): synchronises `stream`, then
 * out[2 (seq H + h)] = selected rows read from the row cache and out[... + 1]
 * = rows read over the host link, for every (sequence, KV head) (host array
 * of 2 N H).  The workspace must be the step's (same cache shape and k).
 */
int bpkv_row_cache_stats(const bpkv_cache *c, int32_t k, const void *ws, uint32_t *out, void *stream);

/*
 * The selection the range attention read in the last layer of the last
 * bpkv_decode_step that used this workspace (Fathom page, section 2 "Top-k
 * decoding": each query head's top (k - 36) middle tokens): synchronises
 * `stream`, then copies the map to the host array out of N H G (cap_tokens /
 * 32) words, row (seq, h, g) at ((seq H + h) G + g) (cap_tokens / 32).  Bit
 * x % 32 of word x / 32 is set when middle token x (n_sink <= x < n -
 * n_recent) was chosen by query head g; sinks and recent tokens are not in
 * the map, and neither are the rows of a head that chose every middle token
 * or none (their words are left as they were).  The streaming cut writes the
 * map; the cooperative cut of small problems (whole grid resident) does not,
 * and then BPKV_EUNSUPPORTED is returned.  The workspace must be the step's
 * (same cache shape and k).
 */
int bpkv_selection_map(const bpkv_cache *c, int32_t k, const void *ws, uint32_t *out, void *stream);

#define BPKV_STAGE_EVENTS 7
#define BPKV_STEP_VDEPTH 1      /* read the value rows to per-row depths (bpkv_sparse_attend_vdepth)
                                   instead of in full; the cache needs value planes */

/*
 * One decode step over n_layers layers (each its own bpkv_cache, same shapes):
 * append the new token (encode), choose depths, scan + top-k, union, sparse
 * attention (or dense attention for BPKV_DEPTH_DENSE).  Every layer's n_max is
 * raised by one.  Needs workspace BPKV_WS_STEP.  With BPKV_STEP_VDEPTH the
 * step forms each KV head's union list and attends with value-side depths
 * (bpkv_sparse_attend_vdepth, budget_v planes per sequence and KV head).
 * BPKV_EINVAL for other flags, or BPKV_STEP_VDEPTH on a cache without value
 * planes, with budget_v < 0 or with G k > 2048.
 */
int bpkv_decode_step(bpkv_cache *layers, int32_t n_layers, const bpkv_step_args *a, void *ws,
                     size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BPKV_H */
