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
 *     up records TRI_ERR_TIMEOUT, after which the kernels of this and later calls
 *     return without work until tri_clear_device_status().
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

/* In-place compaction of every unit with N > budget to its kept slots
 * idx[u][0..budget) (as tri_select_topb writes them: strictly increasing in
 * [0, N), checked on the device: a bad row skips its unit and records
 * TRI_ERR_INVALID).  ORDERED: row j of K and V becomes row idx[u][j];
 * HOLEFILL: the hole-fill layout of those slots (see tri_compact_mode).
 * new_len: NULL or [S] int32 receiving min(N, budget); it must not alias
 * seq_len. */
TRI_API tri_status tri_compact_kv(const tri_cache *cache, const int32_t *idx, int budget,
                          tri_compact_mode mode, int32_t *new_len, cudaStream_t stream);

/* The fused step: score -> GQA z/max -> top-B -> in-place compaction for every
 * unit with N > budget (units with N <= budget untouched).
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
 * capture begins.  A failed lookup returns TRI_ERR_CUDA.
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

/* Reads (and synchronises `stream` for) the device status word; *out (host)
 * receives TRI_OK or the first device-side error recorded since the last clear. */
TRI_API tri_status tri_get_device_status(cudaStream_t stream, int32_t *out);

/* Resets the device status word to TRI_OK (asynchronous on `stream`). */
TRI_API tri_status tri_clear_device_status(cudaStream_t stream);

/* Static description of a status code. */
TRI_API const char *tri_status_string(tri_status status);

/* ABI version of this header (major*100 + minor). */
TRI_API int tri_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TRI_H */
