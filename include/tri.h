/*
 * tri.h — C ABI of libtri: the TriAttention periodic KV-cache compression step
 * on one B300 GPU (sm_103a).
 *
 * Source of the method (no code exists; the operations below restate it):
 *   "实现单卡4090跑通OpenClaw!英伟达&浙大等提出长上下文推理KV压缩新方法TriAttention"
 *   (yeyulingfeng.com), section 主要方法 (main method):
 *     - concentration paragraph: per-head, per-band pre-RoPE Q centers and the
 *       mean resultant length R;
 *     - trig-series paragraph: the RoPE logit is a sum over frequency bands of a
 *       function of the query-key distance, a trigonometric series once Q is
 *       replaced by its center;
 *     - two-part score paragraph: trig-series score + norm score whose weight
 *       falls with concentration, fused into one key importance;
 *     - pruning paragraph: scores averaged over a geometric set of future
 *       offsets; every 128 generated tokens, when the cache exceeds budget B,
 *       every key is scored and the top B are kept; GQA query heads are z-scored
 *       per head and max-aggregated per KV head.
 *
 * Notation.  d = head dim (64 or 128), F = d/2 RoPE bands, omega_f = theta^(-2f/d).
 * Band f of a vector x is x_f = x[f] + i*x[f+F] (TRI_PAIR_HALF, rotate-half) or
 * x[2f] + i*x[2f+1] (TRI_PAIR_INTERLEAVED).  Caches hold post-RoPE keys k~.
 * G = Hq/Hkv (1, 2, 4 or 8); query head h belongs to KV head h/G.
 * A unit is one (sequence s, layer l, KV head g); its index is
 * u = (l*S + s)*Hkv + g and it holds N = seq_len[s] keys in slots 0..N-1.
 *
 * For one unit and each of its query heads h (statistics of query head g*G+h):
 *   A_{h,f} = c_{h,f} * e^{i*omega_f*t_s} * Phi_f,  Phi_f = mean_{o in O} e^{i*omega_f*o}
 *   W_{h,f} = (1 - R_{h,f}) * m_{h,f}
 *   s_{h,i} = sum_f Re[A_{h,f} * conj(k~_{i,f})] + sum_f W_{h,f} * |k~_{i,f}|
 *   z_{h,i} = (s_{h,i} - mean_i s_h) / std_i s_h    (population std; 0 if std = 0)
 *   a_i     = max_h z_{h,i}
 *   kept    = the B slots with largest a (ties: lower slot; NaN lowest), ascending
 *   K[j] <- K[kept_j], V[j] <- V[kept_j] for j < B, in place.
 * The phase omega_f*t_s is reduced modulo 2*pi in fp64; everything per key is fp32.
 *
 * Conventions for every entry point.
 *   - All pointers are DEVICE pointers unless marked (host).  The caller owns
 *     every buffer; the library allocates nothing.  Scratch comes from the
 *     caller's workspace, sized by tri_workspace_bytes() and 16-byte aligned
 *     (cudaMalloc alignment satisfies this).
 *   - Work is enqueued asynchronously on `stream`; nothing synchronises.
 *   - Arguments are validated on the host first: a bad argument returns
 *     TRI_ERR_INVALID, a valid but unsupported shape TRI_ERR_UNSUPPORTED, a too
 *     small workspace TRI_ERR_WORKSPACE, and nothing is launched.  A failed
 *     launch returns TRI_ERR_CUDA.
 *   - Conditions only visible on the device (seq_len[s] > cap, a block id out of
 *     range, an idx list that is not strictly increasing inside [0, N)) skip the
 *     affected unit and record the first error code in a device status word read
 *     by tri_get_device_status().  A sequence skipped for a bad block id gets
 *     new_len = N (nothing compressed); with seq_len > cap new_len is not
 *     written.  Device waits are bounded; a wait that gives
 *     up records TRI_ERR_TIMEOUT (in the status word unless an earlier error
 *     holds it) and sets a timeout flag, after which the kernels of this and
 *     later calls return without work until tri_clear_device_status(); the
 *     outputs (cache rows, idx, lengths) of the call in which a wait gave up
 *     are then unspecified for the units it had not finished.
 *   - No C++ exception crosses this ABI.
 */
#ifndef TRI_H
#define TRI_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define TRI_API __attribute__((visibility("default")))
#else
#define TRI_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TRI_OK = 0,
  TRI_ERR_INVALID = 1,      /* bad argument (host) or bad device-side data      */
  TRI_ERR_CUDA = 2,         /* a CUDA runtime call failed                       */
  TRI_ERR_UNSUPPORTED = 3,  /* valid but not implemented (d, G, sizes)          */
  TRI_ERR_WORKSPACE = 4,    /* workspace missing, too small or misaligned       */
  TRI_ERR_TIMEOUT = 5,      /* a bounded device wait gave up                    */
  TRI_ERR_BOUNDS = 6        /* device-side index check failed (block id, N>cap) */
} tri_status;

typedef enum { TRI_F32 = 0, TRI_BF16 = 1 } tri_dtype;
typedef enum { TRI_PAIR_HALF = 0, TRI_PAIR_INTERLEAVED = 1 } tri_pairing;
/* Layout of the B kept rows after compaction (both keep the same set):
 *   TRI_COMPACT_ORDERED : slot j holds the j-th kept slot in ascending order
 *                         (moves the kept rows past the first evicted slot);
 *   TRI_COMPACT_HOLEFILL: kept slots below B stay where they are; the evicted
 *                         slots below B, ascending, receive the kept slots at or
 *                         above B, ascending (moves at most min(B, N - B) rows).
 *                         Valid because a post-RoPE key carries its position in
 *                         its phase and V rows move with their K rows; a caller
 *                         that needs positions tracks them through idx_out. */
typedef enum { TRI_COMPACT_ORDERED = 0, TRI_COMPACT_HOLEFILL = 1 } tri_compact_mode;

/* KV cache description.
 * Dense (block_table == NULL): k and v are each [L][S][Hkv][cap][d] contiguous,
 *   elements of `dtype`; unit u's slot i is row u*cap + i.
 * Paged (block_table != NULL): k and v are pools [L][nblocks][block][Hkv][d];
 *   block_table is [S][max_blocks] int32 (device); logical slot i of sequence s
 *   lives in physical block block_table[s*max_blocks + i/block], row i%block,
 *   for every layer.  cap must equal max_blocks*block.  Physical blocks must not
 *   be shared between sequences (compaction writes in place).
 * seq_len is [S] int32 (device): N of every unit of sequence s, N <= cap.
 * k, v must be 16-byte aligned. */
typedef struct {
  void *k;
  void *v;
  tri_dtype dtype;
  int L, S, Hkv, d;
  int64_t cap;
  const int32_t *seq_len;
  const int32_t *block_table;
  int max_blocks;
  int block;
  int64_t nblocks;
} tri_cache;

/* Offline statistics, fp32, per layer and query head:
 * center [L][Hq][F][2] (re, im), R [L][Hq][F], mag [L][Hq][F]. */
typedef struct {
  const float *center;
  const float *R;
  const float *mag;
  int Hq;
} tri_stats;

/* Per-step parameters.  t is [S] int32 (device): the position of the next
 * query of each sequence; offsets (host) are the future offsets o >= 0 averaged
 * over (the pages use 2^0..2^K); budget is B >= 1. */
typedef struct {
  double theta;
  tri_pairing pairing;
  const int32_t *t;
  const int32_t *offsets;
  int n_offsets;
  int budget;
} tri_params;

/* Offline calibration (concentration paragraph; pipeline summary "offline
 * Q/K centers, norms and concentration").
 * q_pre: [L][n][Hq][d] pre-RoPE queries (f32 or bf16).  Writes, per (l, h, f):
 *   center = mean_i q_f,  mag = mean_i |q_f|,
 *   R = |mean over samples with |q_f| > 0 of q_f/|q_f||  (0 if none).
 * Returns TRI_ERR_INVALID for n < 1, L < 1, Hq < 1, d not in {64, 128}. */
TRI_API tri_status tri_calibrate_stats(const void *q_pre, tri_dtype dtype, int64_t n, int L, int Hq,
                               int d, tri_pairing pairing, float *center, float *R, float *mag,
                               cudaStream_t stream);

/* Streamed calibration (concentration paragraph; pipeline summary: the
 * centers, norms and concentration are offline statistics).  The statistics
 * of tri_calibrate_stats are means over the samples, so they are carried as
 * sums that chunks of samples add to in any order, on any number of streams
 * or devices, and are divided out at the end.
 *
 * acc: [L][H][F][TRI_CALIB_ACC_DOUBLES] fp64 (device, 8-byte aligned), per
 * (layer, head, band): sum re q_f, sum im q_f, sum |q_f|, sum re q_f/|q_f| and
 * sum im q_f/|q_f| over samples with |q_f| > 0, the count of those samples, the
 * count of all samples, and one unused slot.  The caller owns it
 * (L*H*(d/2)*TRI_CALIB_ACC_DOUBLES*8 bytes).
 *
 * tri_calib_reset     zeroes acc.
 * tri_calib_accumulate adds n samples: element e of head h of sample i of layer l
 *                     is q[l*layer_stride + i*sample_stride + h*d + e] (elements
 *                     of dtype; sample_stride 0 means H*d, layer_stride 0 means
 *                     n*sample_stride), e.g. the query slice of a fused QKV
 *                     activation.  q 16-byte aligned; strides multiples of 4
 *                     elements; sample_stride >= H*d.  n = 0 adds nothing
 *                     (q may then be NULL).
 *                     Accumulation is fp32 over at most 512 samples per thread
 *                     group, then fp64 atomics: the low bits of the sums depend
 *                     on the order in which CTAs finish.
 * tri_calib_merge     acc += other (element-wise; e.g. partial accumulators of
 *                     several streams or devices, copied to one device).
 * tri_calib_finalize  writes center = sum q / count, mag = sum |q| / count,
 *                     R = |sum q/|q|| / nonzero count (0 if none); a band with
 *                     no samples gets 0 everywhere.  Same layouts as
 *                     tri_calibrate_stats.
 * All return TRI_ERR_INVALID for L < 1, H < 1, d not in {64, 128}, or bad
 * pointers, strides or alignment. */
#define TRI_CALIB_ACC_DOUBLES 8
TRI_API tri_status tri_calib_reset(double *acc, int L, int H, int d, cudaStream_t stream);
TRI_API tri_status tri_calib_accumulate(const void *q, tri_dtype dtype, int64_t n, int L, int H, int d,
                                        tri_pairing pairing, int64_t sample_stride, int64_t layer_stride,
                                        double *acc, cudaStream_t stream);
TRI_API tri_status tri_calib_merge(double *acc, const double *other, int L, int H, int d,
                                   cudaStream_t stream);
TRI_API tri_status tri_calib_finalize(const double *acc, int L, int H, int d, float *center, float *R,
                                      float *mag, cudaStream_t stream);

/* Distance-preference curves (trig-series paragraph: with Q/K replaced by
 * their calibrated centers the RoPE logit becomes a trigonometric series in the
 * query-key distance, the head's distance-preference curve, reported to track
 * the attention's distance preference with high correlation).  For query head h
 * of layer l, KV head g = h / (Hq/Hkv), distance delta = 0..n_delta-1:
 *   center_curve[l][h][delta] = sum_f Re[cq_{h,f} conj(ck_{g,f}) e^{i omega_f delta}]
 *   logit_curve[l][h][delta]  = mean over i in [0, n - delta) of the RoPE logit of
 *       query sample i + delta (position i + delta) against key sample i
 *       (position i): sum_f Re[q_{i+delta,f} conj(k_{i,f}) e^{i omega_f delta}]
 *   corr[l][h] = Pearson correlation of the two curves over delta (0 when
 *       either curve is constant).
 * q_center: [L][Hq][F][2], k_center: [L][Hkv][F][2] fp32 (e.g. tri_calibrate_stats
 * of pre-RoPE queries and of pre-RoPE keys).  q_seq: [L][n][Hq][d], k_seq:
 * [L][n][Hkv][d] pre-RoPE samples of one sequence (dtype, 4-byte aligned).
 * Outputs fp32 [L][Hq][n_delta] and [L][Hq].  logit_curve and corr may be NULL
 * (then q_seq, k_seq are not read; corr needs logit_curve).  The phase
 * omega_f*delta is reduced modulo 2*pi in fp64.  Requires n_delta >= 1, and
 * n_delta <= n when the logit curve is asked for. */
TRI_API tri_status tri_distance_curves(const float *q_center, const float *k_center, const void *q_seq,
                                       const void *k_seq, tri_dtype dtype, int64_t n, int L, int Hq, int Hkv,
                                       int d, double theta, tri_pairing pairing, int n_delta,
                                       float *center_curve, float *logit_curve, float *corr,
                                       cudaStream_t stream);

/* Workspace bytes that tri_score / tri_compress_step need for these arguments
 * (0 when every unit fits one CTA's shared memory).  `bytes` is a host pointer. */
TRI_API tri_status tri_workspace_bytes(const tri_cache *cache, const tri_stats *stats,
                               const tri_params *params, size_t *bytes);

/* Scores every key of every unit (two-part score paragraph; pruning paragraph).
 * agg: [L][S][Hkv][cap] fp32, a_i for i < N (slots >= N untouched).
 * raw: NULL or [L][S][Hq][cap] fp32, s_{h,i} of query head h for i < N.
 * Units with N = 0 are skipped.  ws/ws_bytes: workspace (may be NULL/0 when
 * tri_workspace_bytes reports 0). */
TRI_API tri_status tri_score(const tri_cache *cache, const tri_stats *stats, const tri_params *params,
                     float *agg, float *raw, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Top-B per unit from aggregated scores (pruning paragraph).
 * agg: [L][S][Hkv][cap] fp32.  idx: [L][S][Hkv][budget] int32, the kept slots in
 * ascending order; a unit with N <= budget gets 0..N-1 followed by -1.
 * Ties keep the lower slot; NaN ranks lowest.  Only cache->L, S, Hkv, cap,
 * seq_len are read (k, v may be NULL).  ws is unused (pass NULL, 0). */
TRI_API tri_status tri_select_topb(const tri_cache *cache, const float *agg, int budget, int32_t *idx,
                           void *ws, size_t ws_bytes, cudaStream_t stream);

/* In-place compaction (pruning paragraph: the top B keys are kept, the rest
 * of the unit's keys are dropped from the cache) of every unit with N > budget
 * to its kept slots
 * idx[u][0..budget) (as tri_select_topb writes them: strictly increasing in
 * [0, N), checked on the device: a bad row skips its unit and records
 * TRI_ERR_INVALID).  ORDERED: row j of K and V becomes row idx[u][j];
 * HOLEFILL: the hole-fill layout of those slots (see tri_compact_mode).
 * new_len: NULL or [S] int32 receiving min(N, budget); it must not alias
 * seq_len. */
TRI_API tri_status tri_compact_kv(const tri_cache *cache, const int32_t *idx, int budget,
                          tri_compact_mode mode, int32_t *new_len, cudaStream_t stream);

/* The fused step (pruning paragraph: every 128 generated tokens, when the
 * cache exceeds the budget, score every key, z-score per query head and take
 * the max per KV head, keep the top B): score -> GQA z/max -> top-B -> in-place
 * compaction for every unit with N > budget (units with N <= budget untouched).
 * The caller makes the call at its 128-token boundaries.
 * idx_out: NULL or [L][S][Hkv][budget] int32: the original slot of the row now
 * at each slot j < budget (ORDERED: the kept slots ascending, as
 * tri_select_topb writes them; HOLEFILL: j for kept slots below B, the mover
 * for each hole).
 * new_len: NULL or [S] int32 (min(N, budget)); must not alias seq_len. */
TRI_API tri_status tri_compress_step(const tri_cache *cache, const tri_stats *stats,
                             const tri_params *params, tri_compact_mode mode, int32_t *idx_out,
                             int32_t *new_len, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Size in bytes of the scratch array built into the library for
 * tri_compress_step_static_scratch (32 MiB). */
#define TRI_STATIC_SCRATCH_BYTES (32u << 20)

/* tri_compress_step for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a library convenience, not part of
 * the method.  Some callers cannot call cudaMalloc: for example, a serving
 * engine that gives nearly all device memory to its KV-cache pool at start-up
 * and forbids later allocations, or code running in a plugin that has no
 * access to the process's allocator.  Such a caller still owns the cache and
 * the outputs but cannot supply the workspace that long units need.
 *
 * Same arguments and results as tri_compress_step, without ws/ws_bytes.  When
 * the step needs scratch (tri_workspace_bytes > 0), it uses a file-scope
 * device array of TRI_STATIC_SCRATCH_BYTES bytes that every GPU loading the
 * library holds until the process exits.  A step that needs more than that
 * returns TRI_ERR_WORKSPACE and launches nothing (no other limit differs).
 * Nothing is allocated: no cudaMalloc, no cudaFree.
 *
 * Set-up: the first call on each device looks up that device's address of the
 * array (with that device current), so make that first call before any stream
 * capture begins.  A failed lookup returns TRI_ERR_CUDA.  The address is kept
 * per device together with the CUDA context that was current at the lookup; a
 * call under another context (after cudaDeviceReset, or with a context the
 * caller made current) looks the address up again, so again make such a call
 * outside any stream capture.
 *
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents; the step writes each scratch entry before reading it, so
 * nothing needs clearing.  Calls whose work overlaps on the GPU (two streams,
 * or two host threads) race on the array and give wrong results: order them
 * on one stream or with events. */
TRI_API tri_status tri_compress_step_static_scratch(const tri_cache *cache, const tri_stats *stats,
                                            const tri_params *params, tri_compact_mode mode,
                                            int32_t *idx_out, int32_t *new_len,
                                            cudaStream_t stream);

/* Decode loop around the compression step (pruning paragraph: during online
 * decoding the step runs once every 128 generated tokens when the cache exceeds
 * the budget).  These calls are the decode side of that loop: they are not part
 * of the compression method, they let it run inside a decode loop on the same
 * cache.  A loop appends a token to every unit, attends, and every 128 tokens
 * calls tri_compress_step with t = the next query position.
 *
 * tri_append_kv: k_new, v_new [L][S][Hkv][d] (cache dtype, 16-byte aligned):
 *   the new token's pre-RoPE key and its value for every unit.  The key is
 *   rotated to position pos[s] (band f times e^{i omega_f pos[s]}, the phase
 *   reduced modulo 2 pi in fp64, rounded to the cache dtype) and written with
 *   the value into slot N = seq_len[s] of unit (l, s, g) (paged: block
 *   block_table[s][N / block], row N % block).  seq_len_out[s] receives N + 1 and
 *   pos_out[s] (NULL: not written) pos[s] + 1.  Neither may alias seq_len or
 *   pos.  A sequence whose slot N is not available (N >= cap, or its block id
 *   out of range) is skipped with TRI_ERR_BOUNDS in the device status and
 *   seq_len_out[s] = N, pos_out[s] = pos[s].
 * tri_decode_workspace_bytes: scratch that tri_decode_attention needs (0 when
 *   one CTA per unit suffices; otherwise per-slice partial results).
 * tri_decode_attention: q [L][S][Hq][d] bf16 pre-RoPE queries (one per
 *   sequence and query head), rotated to pos[s] inside; for query head h of
 *   unit (l, s, g = h / (Hq/Hkv)):
 *     out[l][s][h] = sum_{i < N} w_i v_i,  w = softmax_i(scale * q~_h . k~_i)
 *   over the unit's N = seq_len[s] slots, out fp32 [L][S][Hq][d].  The slot
 *   order does not matter (ordered or hole-fill compaction give the same
 *   output).  bf16 caches only (TRI_ERR_UNSUPPORTED otherwise), G in {1, 2, 4,
 *   8}.  Both products run on the tensor cores with the query and the
 *   probabilities split into bf16 hi + lo parts and fp32 accumulation.  A unit
 *   with N = 0 gets out = 0. */
TRI_API tri_status tri_append_kv(const tri_cache *cache, const void *k_new, const void *v_new,
                                 const int32_t *pos, double theta, tri_pairing pairing,
                                 int32_t *seq_len_out, int32_t *pos_out, cudaStream_t stream);
TRI_API tri_status tri_decode_workspace_bytes(const tri_cache *cache, int Hq, size_t *bytes);
TRI_API tri_status tri_decode_attention(const tri_cache *cache, const void *q, int Hq, const int32_t *pos,
                                        double theta, tri_pairing pairing, float scale, float *out,
                                        void *ws, size_t ws_bytes, cudaStream_t stream);

/* Health check of the bounded-wait path: launches one warp whose thread 0
 * waits on a shared-memory barrier that nothing arrives at, with a limit of
 * limit_us microseconds (1..1000000); nothing else is in flight.  The wait
 * gives up, records TRI_ERR_TIMEOUT in the device status word and the kernel
 * returns, after which the kernels of later calls return without work until
 * tri_clear_device_status() (exactly as after a wait that gave up inside a
 * step).  Lets a caller confirm that a stuck wait ends with a status, not a
 * hang.  Not part of the method. */
TRI_API tri_status tri_check_bounded_wait(uint32_t limit_us, cudaStream_t stream);

/* Reads (and synchronises `stream` for) the device status word; *out (host)
 * receives TRI_OK or the first device-side error recorded since the last clear. */
TRI_API tri_status tri_get_device_status(cudaStream_t stream, int32_t *out);

/* Resets the device status word to TRI_OK and clears the timeout flag
 * (asynchronous on `stream`). */
TRI_API tri_status tri_clear_device_status(cudaStream_t stream);

/* Static description of a status code. */
TRI_API const char *tri_status_string(tri_status status);

/* ABI version of this header (major*100 + minor). */
TRI_API int tri_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TRI_H */
