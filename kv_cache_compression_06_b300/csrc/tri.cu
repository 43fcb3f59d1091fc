// libtri: kernels and C ABI of the TriAttention periodic KV-cache compression step.
//
// Method source: "实现单卡4090跑通OpenClaw!英伟达&浙大等提出长上下文推理KV压缩新方法TriAttention"
// (yeyulingfeng.com), section 主要方法 (concentration / trig-series / two-part
// score / pruning paragraphs).  The operations are restated in include/tri.h.
//
// Kernels
//   calib_kernel         a0: per (layer, query head): center, mean |q_f|, R.
//   fused_kernel         a1..a5 for units whose scores fit one CTA's shared
//                        memory: weights -> TMA-streamed scoring (producer warp +
//                        8 consumer warps) -> z/max -> radix top-B -> in-place
//                        bulk-copy compaction.  Also the score-only variant
//                        behind tri_score.
//   score_tiles_kernel   a1+a2 for long units, 2048 keys per CTA (same pipeline):
//                        raw scores and per-tile (mean, M2) to the workspace
//                        (tri_score; the compress step with fp32 or interleaved
//                        caches).  score_tiles_mma_kernel: its tensor-core form.
//   score_keys_mma_kernel a1+a2 of the compress step for long bf16 units:
//                        key-major raw scores straight from the MMA fragments,
//                        moments in registers, one (mean, M2) per CTA.
//   score_heads_mma_kernel the same for paged caches whose block holds 128
//                        head-rows: every KV head of a block from one copy.
//   select_only_kernel   a3+a4 of the compress step for long units: kept slots
//                        (one pass over the raw scores, or the full passes).
//   compact_only_kernel  a5 of the compress step for long units.
//   holefill_apply_kernel a5 in the hole-fill layout after a selection that
//                        wrote kept lists or bitmasks: layout + independent row moves.
//   zmax_kernel          a3 for long units (tri_score): Chan-merged moments -> agg.
//   select_compact_kernel a3..a5 for long units whose kept list or hole-fill
//                        bookkeeping does not fit compact_only_kernel,
//                        tri_select_topb (from agg) and tri_compact_kv (from idx).
//   calib_*_kernel       streamed calibration: sums per (layer, head, band) that
//                        chunks of samples add to, merged, then finalised.
//   *_curve_kernel       distance-preference curves (centers vs exact logits).
//   wait_check_kernel    a bounded wait that gives up (health check of the
//                        timeout path).
//   append_kv_kernel     decode loop: one token's K (rotated to its position)
//                        and V into slot N of every unit.
//   decode_attn_kernel   decode loop: single-query attention over the cache
//                        (split-K, tensor cores), decode_merge_kernel merges splits.
#include <cmath>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <mutex>

#include "tri_mma.cuh"
#include "tri_calib.cuh"
#include "tri_curve.cuh"
#include "tri_decode.cuh"

namespace tri {

constexpr int kMaxSmem = 232448;   // 227 KB opt-in dynamic shared memory per CTA (sm_103a)

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- a0 calibration
__global__ void __launch_bounds__(256) calib_kernel(const void *q, int bf16, long long n, int Hq,
                                                    int d, int inter, float *center, float *R,
                                                    float *mag) {
  __shared__ double acc[6][256];
  const int h = blockIdx.x, l = blockIdx.y, F = d / 2;
  const int parts = blockDim.x / F;
  const int f = threadIdx.x % F, part = threadIdx.x / F;
  float sr = 0, si = 0, sm = 0, ur = 0, ui = 0;
  int cnt = 0;
  if (part < parts) {
    const int ire = inter ? 2 * f : f, iim = inter ? 2 * f + 1 : f + F;
    for (long long i = part; i < n; i += parts) {
      const long long base = (((long long)l * n + i) * Hq + h) * d;
      float re, im;
      if (bf16) {
        const unsigned short *p = static_cast<const unsigned short *>(q);
        re = __uint_as_float((uint32_t)p[base + ire] << 16);
        im = __uint_as_float((uint32_t)p[base + iim] << 16);
      } else {
        const float *p = static_cast<const float *>(q);
        re = p[base + ire];
        im = p[base + iim];
      }
      const float m = sqrtf(re * re + im * im);
      sr += re;
      si += im;
      sm += m;
      if (m > 0.f) {
        ur += re / m;
        ui += im / m;
        ++cnt;
      }
    }
  }
  acc[0][threadIdx.x] = sr;
  acc[1][threadIdx.x] = si;
  acc[2][threadIdx.x] = sm;
  acc[3][threadIdx.x] = ur;
  acc[4][threadIdx.x] = ui;
  acc[5][threadIdx.x] = cnt;
  __syncthreads();
  if (threadIdx.x < F) {
    double t[6] = {0, 0, 0, 0, 0, 0};
    for (int p = 0; p < parts; ++p)
      for (int k = 0; k < 6; ++k) t[k] += acc[k][p * F + threadIdx.x];
    const long long o = ((long long)l * Hq + h) * F + threadIdx.x;
    center[2 * o] = (float)(t[0] / (double)n);
    center[2 * o + 1] = (float)(t[1] / (double)n);
    mag[o] = (float)(t[2] / (double)n);
    R[o] = t[5] > 0 ? (float)(sqrt(t[3] * t[3] + t[4] * t[4]) / t[5]) : 0.0f;
  }
}

// ---------------------------------------------------------------- fused short-unit kernel
// One CTA of kFusedThreads per unit: score (every warp; warp 0 refills the
// ring), z/max, select, compact.  Two CTAs per SM for G <= 4.
struct FusedArgs {
  CacheView c;
  const float *center, *R, *mag;
  int Hq;
  const int *t;
  int budget, mode, inter, capp;   // mode 0: compress, 1: score only
  int holefill;                    // compaction layout: 0 ordered, 1 hole-fill
  int defer;                       // hole-fill: write the kept set to idx_out as a bitmask
                                   // and leave the layout and rows to holefill_apply_kernel
  int mma_ok;                      // host only: try the tensor-core variant
  const tri_cache *cache;          // host only: for that variant's tensor map
  const tri_params *params;
  float *agg, *raw;
  int *idx_out, *new_len;
  StepConst sc;
};

// Shared-memory layout of the fused kernel.  Scores of head h live at
// scores[h * sstride + i]; sstride = capp + 4 (= 4 mod 32) keeps the per-row
// score writes of the different heads in different banks.
struct FusedLayout {
  int bars, wts, red, hist, sm, scores, idx, sstride, total;
  __host__ __device__ FusedLayout(int G, int F, int capp) {
    sstride = capp + 4;
    int o = kRingBytes;
    bars = o;   o += 256;                 // score barriers, 2 x kStages compaction barriers, flags
    wts = o;    o += align_up(G * 3 * F * 4, 128);
    red = o;    o += 1024;                // block sums; per-warp moment states, then the merged moments
    hist = o;   o += 1024;
    sm = o;     o += 256;
    scores = o; o += align_up(G * sstride * 4, 128);
    if (G >= 2) {
      idx = scores + sstride * 4;   // overlays head 1's scores (dead after z/max)
    } else {
      idx = o;
      o += align_up(capp * 4, 128);
    }
    total = o;
  }
};

template <int D, int G, bool BF16>
__global__ void __launch_bounds__(kFusedThreads, (G <= 4 ? 2 : 1)) fused_kernel(const FusedArgs a) {
  constexpr int F = D / 2;
  extern __shared__ __align__(1024) char smem[];
  const FusedLayout lay(G, F, a.capp);
  char *ring = smem;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bars);
  float *wts = reinterpret_cast<float *>(smem + lay.wts);
  float *red = reinterpret_cast<float *>(smem + lay.red);
  uint32_t *hist = reinterpret_cast<uint32_t *>(smem + lay.hist);
  int *sm = reinterpret_cast<int *>(smem + lay.sm);
  float *scores = reinterpret_cast<float *>(smem + lay.scores);
  int *idxs = reinterpret_cast<int *>(smem + lay.idx);

  const CacheView &c = a.c;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int u = blockIdx.x;
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  if (timed_out()) return;
  const int N = c.seq_len[s];
  const int B = a.budget;
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  const bool len_writer = a.mode == 0 && tid == 0 && a.new_len != nullptr && l == 0 && g == 0;
  if (a.mode == 0 && N <= B) {
    if (len_writer) a.new_len[s] = N;
    if (a.idx_out != nullptr)
      for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = j < N ? j : -1;
    return;
  }
  if (N == 0) return;
  if (!c.blocks_ok(s, N)) {   // the sequence is skipped: its length stays N
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    if (len_writer) a.new_len[s] = N;
    return;
  }
  if (len_writer) a.new_len[s] = B;
  const int ss = lay.sstride;
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 32);
    for (int st = 0; st < kStages; ++st) mbar_init(&bars[kStages + st], 1);
    fence_mbar_init();
  }
  build_weights<G, F>(wts, a.center, a.R, a.mag, a.Hq, l, g, a.t[s], a.sc);
  __syncthreads();
  LaneWeights<G> lw;
  load_lane_weights<G, F>(lw, wts, (tid & 31) % RowGeom<D, BF16>::LPR);
  if (!score_unit_rows<D, G, BF16>(c, l, s, g, 0, N, ring, bars, scores, ss, lw, a.inter != 0))
    return;

  float mu[G], inv[G];
  head_moments<G>(scores, ss, N, red, mu, inv);
  uint32_t *keys = reinterpret_cast<uint32_t *>(scores);   // overlays head 0's scores
  for (int i = tid; i < N; i += nt) {
    float sv[G];
#pragma unroll
    for (int h = 0; h < G; ++h) sv[h] = scores[h * ss + i];
    float z = (sv[0] - mu[0]) * inv[0];
#pragma unroll
    for (int h = 1; h < G; ++h) z = fmaxf(z, (sv[h] - mu[h]) * inv[h]);
    if (a.mode == 1) {
      a.agg[(long long)u * c.cap + i] = z;
      if (a.raw != nullptr) {
#pragma unroll
        for (int h = 0; h < G; ++h) a.raw[((long long)u * G + h) * c.cap + i] = sv[h];
      }
    } else {
      keys[i] = score_key(z);
    }
  }
  if (a.mode == 1) return;
  __syncthreads();
  int ntie;
  const uint32_t T = radix_select_atomic(keys, N, B, hist, sm, &ntie);
  if (a.defer) {   // hole-fill: the kept set as a bitmask in idx_out; holefill_apply_kernel does the rest
    kept_bits(keys, N, T, ntie, reinterpret_cast<uint32_t *>(a.idx_out + (long long)u * B), sm);
    return;
  }
  const int e0 = build_kept_chunked(keys, N, B, T, ntie, idxs, sm);
  if (a.holefill) {   // keys are dead: their 4N bytes hold the hole-fill bookkeeping
    holefill_unit(c, l, s, g, idxs, B, N, reinterpret_cast<char *>(keys), ring, kRingBytes, sm,
                  a.idx_out != nullptr ? a.idx_out + (long long)u * B : nullptr);
    return;
  }
  if (a.idx_out != nullptr)
    for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = idxs[j];
  // The ring was last read by generic loads (scoring); TMA writes it next.
  fence_proxy_async_smem();
  __syncthreads();
  if ((tid >> 5) == 0) compact_unit_runs(c, l, s, g, idxs, e0, B, N, ring, bars + kStages);
}

// Pipe over the barrier block of a layout (256 bytes): full[4] | empty[4] |
// compaction[2][4] | fail, issued.
__device__ __forceinline__ Pipe make_pipe(char *smem, int bars) {
  uint64_t *b = reinterpret_cast<uint64_t *>(smem + bars);
  Pipe p;
  p.ring = smem;
  p.full = b;
  p.empty = b + kStages;
  p.fail = reinterpret_cast<volatile int *>(b + 4 * kStages);
  p.issued = p.fail + 1;
  return p;
}

// ---------------------------------------------------------------- long units: step phases
// E[s][f] = e^{i*omega_f*t_s} * Phi_f for every sequence and band, once per call
// (the tile CTAs of a unit all need it; computing it per tile cost ~20
// instructions per key at G = 8).
// Sum over the block (64 threads) of v; every thread gets it.
__device__ __forceinline__ int sum64(int v, int *part) {
  v = warp_sum_int(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
  __syncthreads();
  return part[0] + part[1];
}

// Also, when `order` is given, the sequences ranked by length, longest first
// (ties by index): order[rank] = s.  The long-unit selection takes its units
// in that order, so that the longest ones do not start in the last wave.
// When `plan` is given, the chunk plan of the head-grouped score kernel
// (chunks of `ck` keys of the sequences with budget < N <= cap): plan[0] = full
// chunks per layer, plan[1] = sequences with a partial last chunk,
// plan[2 + s] = full chunks of the sequences before s, plan[2 + S + r] = the
// sequence with the r-th largest partial chunk (ties by index).  The score
// kernel runs the full chunks first and the partial ones last, largest first,
// so that the last wave holds the smallest CTAs.
__global__ void __launch_bounds__(64) phase_kernel(const int *t, int F, float2 *phase, const StepConst sc,
                                                   const int *seq_len, int S, int *order, int *plan, int budget,
                                                   long long cap, int ck) {
  __shared__ int part[2];
  const int s = blockIdx.x;
  for (int f = threadIdx.x; f < F; f += blockDim.x) phase[(long long)s * F + f] = step_phase(sc, f, t[s]);
  if (order != nullptr) {
    const int n = seq_len[s];
    int r = 0;
    for (int x = threadIdx.x; x < S; x += blockDim.x) {
      const int m = seq_len[x];
      r += (m > n) || (m == n && x < s);
    }
    r = sum64(r, part);
    if (threadIdx.x == 0) order[r] = s;
  }
  if (plan != nullptr) {
    auto live = [&](int m) { return m > budget && (long long)m <= cap; };
    const int n = seq_len[s], rem = live(n) ? n % ck : 0;
    int before = 0, tot_full = 0, tot_part = 0, rank = 0;
    for (int x = threadIdx.x; x < S; x += blockDim.x) {
      const int m = seq_len[x];
      const int fx = live(m) ? m / ck : 0, rx = live(m) ? m % ck : 0;
      if (x < s) before += fx;
      tot_full += fx;
      tot_part += rx > 0;
      rank += rx > 0 && (rx > rem || (rx == rem && x < s));
    }
    before = sum64(before, part);
    if (s == 0) {
      tot_full = sum64(tot_full, part);
      tot_part = sum64(tot_part, part);
    }
    rank = sum64(rank, part);
    if (threadIdx.x == 0) {
      plan[2 + s] = before;
      if (rem > 0) plan[2 + S + rank] = s;
      if (s == 0) {
        plan[0] = tot_full;
        plan[1] = tot_part;
      }
    }
  }
}

// ---------------------------------------------------------------- long units: tiles
struct TileArgs {
  TmaMaps maps;      // k4 (CUDA-core variant)
  CUtensorMap ks;    // tensor-core variant: 128B-swizzled K map (dense 2-D, paged 4-D), boxes of 64 elements
  CacheView c;
  const float *center, *R, *mag;
  int Hq;
  const int *t;
  int budget, skip_small, inter, ntiles, mma_ok;
  int hg;            // ks boxes every KV head of a block: score_heads_mma_kernel
  long long raw_stride;
  const float2 *phase;   // [S][F] step phases (phase_kernel); raw_stride: floats between the raw rows of two heads (cap, or capp in the workspace)
  int *order;            // [S] sequences by length, longest first (phase_kernel), or null
  int *plan;             // [2 S + 2] chunk plan of score_heads_mma_kernel (phase_kernel), or null
  float *raw;      // [(u*G + h)*raw_stride + i]
  float2 *part;    // [(u*ntiles + tile)*G + h] = (mean, M2) of the tile
  StepConst sc;
};

// per-head score stride of a tile (= 4 mod 32: no bank conflicts)
__host__ __device__ constexpr int tile_stride_for(int G) { return tile_keys_for(G) + 4; }

struct TileLayout {
  int bars, wts, red, scores, total;
  __host__ __device__ TileLayout(int G, int F) {
    int o = kRingBytes;
    bars = o;   o += 256;
    wts = o;    o += align_up(G * 3 * F * 4, 128);
    red = o;    o += 512;
    scores = o; o += G * tile_stride_for(G) * 4;
    total = o;
  }
};

// Mean and M2 (sum of squared deviations) per head over one tile's scores,
// two passes, on the scores minus the tile's first score (as head_moments): a
// constant tile gets M2 = 0 exactly and its mean equals the constant.
template <int G>
__device__ __forceinline__ void head_mean_m2(const float *scores, int stride, int n, float *red,
                                             float (&mu)[G], float (&m2)[G]) {
  float v[G], sh[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    v[h] = 0.f;
    sh[h] = scores[h * stride];
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
#pragma unroll
    for (int h = 0; h < G; ++h) v[h] += scores[h * stride + i] - sh[h];
  }
  block_sum<G>(v, red);
  float md[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    md[h] = v[h] / (float)n;
    mu[h] = sh[h] + md[h];
    v[h] = 0.f;
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float dl = (scores[h * stride + i] - sh[h]) - md[h];
      v[h] = fmaf(dl, dl, v[h]);
    }
  }
  block_sum<G>(v, red);
#pragma unroll
  for (int h = 0; h < G; ++h) m2[h] = v[h];
}

template <int D, int G, bool BF16>
__global__ void __launch_bounds__(kThreads, (G <= 4 ? 2 : 1))
    score_tiles_kernel(const __grid_constant__ TileArgs a) {
  constexpr int F = D / 2;
  extern __shared__ __align__(1024) char smem[];
  const TileLayout lay(G, F);
  const Pipe pipe = make_pipe(smem, lay.bars);
  float *wts = reinterpret_cast<float *>(smem + lay.wts);
  float *red = reinterpret_cast<float *>(smem + lay.red);
  float *scores = reinterpret_cast<float *>(smem + lay.scores);
  const CacheView &c = a.c;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int tile = blockIdx.x, u = blockIdx.y;
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  if (timed_out()) return;
  const int N = c.seq_len[s];
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (a.skip_small && N <= a.budget) return;
  constexpr int TK = tile_keys_for(G), TS = tile_stride_for(G);
  const int i0 = tile * TK;
  if (i0 >= N) return;
  const int n = min(TK, N - i0);
  if (!c.blocks_ok(s, n, i0)) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (tid == 0) pipe_init(pipe);
  build_weights<G, F>(wts, a.center, a.R, a.mag, a.Hq, l, g, a.t[s], a.sc, a.phase + (long long)s * F);
  __syncthreads();
  LaneWeights<G> lw;
  load_lane_weights<G, F>(lw, wts, (tid & 31) % RowGeom<D, BF16>::LPR);
  if (!stream_and_score<D, G, BF16>(c, &a.maps.k4, l, s, g, i0, n, pipe, scores, TS, lw,
                                    a.inter != 0))
    return;
  for (int i = tid; i < n; i += nt) {
#pragma unroll
    for (int h = 0; h < G; ++h) a.raw[((long long)u * G + h) * a.raw_stride + i0 + i] = scores[h * TS + i];
  }
  float mu[G], m2[G];
  head_mean_m2<G>(scores, TS, n, red, mu, m2);
  if (tid == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h)
      a.part[((long long)u * a.ntiles + tile) * G + h] = make_float2(mu[h], m2[h]);
  }
}

// Writes one tile's raw scores (G rows of tn floats, head h at raw + h *
// rstride) and returns their (mean, M2) per head, taken on the scores minus the
// tile's first score (a constant head gets M2 = 0 exactly); one pass stores and sums, a second
// sums the squared deviations.  vec: 16-byte loads and stores (raw rows
// 16-byte aligned); else 4-byte ones.
template <int G>
__device__ __forceinline__ void tile_flush(const float *scores, int stride, int tn, float *raw, long long rstride,
                                           bool vec, float *red, int nthreads, float (&mu)[G], float (&m2)[G]) {
  const int tid = threadIdx.x;
  float v[G], sh[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    v[h] = 0.f;
    sh[h] = scores[h * stride];
  }
  const int n4 = vec ? tn >> 2 : 0;
  for (int q = tid; q < n4; q += nthreads) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float4 x = reinterpret_cast<const float4 *>(scores + h * stride)[q];
      reinterpret_cast<float4 *>(raw + h * rstride)[q] = x;
      v[h] += ((x.x - sh[h]) + (x.y - sh[h])) + ((x.z - sh[h]) + (x.w - sh[h]));
    }
  }
  for (int i = 4 * n4 + tid; i < tn; i += nthreads) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float x = scores[h * stride + i];
      raw[h * rstride + i] = x;
      v[h] += x - sh[h];
    }
  }
  group_sum<G>(v, red, nthreads);
  float md[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    md[h] = v[h] / (float)tn;
    mu[h] = sh[h] + md[h];
    v[h] = 0.f;
  }
  const int m4 = tn >> 2;
  for (int q = tid; q < m4; q += nthreads) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float4 x = reinterpret_cast<const float4 *>(scores + h * stride)[q];
      const float d0 = (x.x - sh[h]) - md[h], d1 = (x.y - sh[h]) - md[h];
      const float d2 = (x.z - sh[h]) - md[h], d3 = (x.w - sh[h]) - md[h];
      v[h] = fmaf(d0, d0, fmaf(d1, d1, fmaf(d2, d2, fmaf(d3, d3, v[h]))));
    }
  }
  for (int i = 4 * m4 + tid; i < tn; i += nthreads) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float dl = (scores[h * stride + i] - sh[h]) - md[h];
      v[h] = fmaf(dl, dl, v[h]);
    }
  }
  group_sum<G>(v, red, nthreads);
#pragma unroll
  for (int h = 0; h < G; ++h) m2[h] = v[h];
}

// Tensor-core variant of score_tiles_kernel for bf16 caches with rotate-half
// bands.  A CTA covers kTilesPerCta consecutive tiles of one unit: the weights
// are built once, the producer warp streams the CTA's whole row range through
// the ring, and the 8 consumer warps score 16-key tiles of each stage with
// score_tile_mma (for d = 128 two groups of 4 warps take alternate stages; the
// empty barrier then counts the 4 warps of a group).  At the end of each tile
// the consumer warps alone (named barrier) write its raw scores and (mean, M2)
// while the producer keeps loading the next tile.
template <int D, int G>
__global__ void __launch_bounds__(kThreads, 2) score_tiles_mma_kernel(const __grid_constant__ TileArgs a) {
  constexpr int F = D / 2;
  constexpr int TR = kStageBytes / (2 * D);
  constexpr int SPS = TR / 16;                    // key tiles per stage
  constexpr int GROUPS = kConsumerWarps / SPS;    // warp groups taking alternate stages
  constexpr int TK = tile_keys_for(G), TS = tile_stride_for(G);
  constexpr int SPT = TK / TR;                    // stages per tile
  constexpr int NC = kConsumerWarps * 32;
  extern __shared__ __align__(1024) char smem[];
  const TileLayout lay(G, F);
  const Pipe pipe = make_pipe(smem, lay.bars);
  float *wts = reinterpret_cast<float *>(smem + lay.wts);
  float *red = reinterpret_cast<float *>(smem + lay.red);
  float *scores = reinterpret_cast<float *>(smem + lay.scores);
  const CacheView &c = a.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.y;
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  if (timed_out()) return;
  const int N = c.seq_len[s];
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (a.skip_small && N <= a.budget) return;
  const int tile0 = blockIdx.x * kTilesPerCta;
  const int i0 = tile0 * TK;
  if (i0 >= N) return;
  const int n = min(kTilesPerCta * TK, N - i0);   // rows of this CTA
  if (!c.blocks_ok(s, n, i0)) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&pipe.full[st], 1);
      mbar_init(&pipe.empty[st], SPS);
    }
    *pipe.fail = 0;
    *pipe.issued = 0;
    fence_mbar_init();
  }
  build_weights<G, F>(wts, a.center, a.R, a.mag, a.Hq, l, g, a.t[s], a.sc, a.phase + (long long)s * F);
  __syncthreads();
  const int nst = (n + TR - 1) / TR;   // stages of this CTA
  const long long urow0 = (long long)u * c.cap;   // dense: row of slot 0 in the 2-D view
  if (warp == kProducerWarp) {
    int t = 0;
    for (; t < nst; ++t) {
      const int st = t % kStages;
      if (*pipe.fail || (t >= kStages && !mbar_wait(&pipe.empty[st], (uint32_t)(((t / kStages) - 1) & 1)))) {
        *pipe.fail = 1;
        break;
      }
      produce_stage_sw<D>(c, &a.ks, l, s, g, urow0, i0 + t * TR, min(TR, n - t * TR),
                          pipe.ring + st * kStageBytes, &pipe.full[st], lane);
    }
    if (lane == 0) *pipe.issued = t;
  } else {
    MmaWeights<D, G> w;
    load_mma_weights<D, G>(w, wts, kConsumerWarps * 32, warp == 0);
    const int grp = warp / SPS, sub = warp % SPS;
    const uint32_t ring = smem_u32(pipe.ring);
    // tiles start at multiples of 64 keys: 16-byte raw stores when the rows are aligned
    const bool raw_vec = (a.raw_stride & 3) == 0 && (reinterpret_cast<uintptr_t>(a.raw) & 15) == 0;
    for (int tt = 0; tt * SPT < nst; ++tt) {   // tiles of this CTA
      const int tbeg = tt * SPT, tend = min(nst, tbeg + SPT);
      for (int t = tbeg + (grp - tbeg % GROUPS + GROUPS) % GROUPS; t < tend; t += GROUPS) {
        const int st = t % kStages;
        if (!*pipe.fail && !mbar_wait(&pipe.full[st], (uint32_t)((t / kStages) & 1))) *pipe.fail = 1;
        score_tile_mma<D, G, TR>(ring + st * kStageBytes, 16 * sub, min(TR, n - t * TR), (t - tbeg) * TR,
                                 scores, TS, w, c.paged() ? c.block : 0);
        __syncwarp();
        if (lane == 0) mbar_arrive(&pipe.empty[st]);
      }
      named_sync(1, NC);   // the tile's scores are in shared memory
      const int tn = min(TK, n - tbeg * TR);
      const int ti0 = i0 + tbeg * TR;
      if (!*pipe.fail) {
        float mu[G], m2[G];
        tile_flush<G>(scores, TS, tn, a.raw + (long long)u * G * a.raw_stride + ti0, a.raw_stride, raw_vec, red, NC,
                      mu, m2);
        if (tid == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h)
            a.part[((long long)u * a.ntiles + tile0 + tt) * G + h] = make_float2(mu[h], m2[h]);
        }
      }
      named_sync(1, NC);   // scores may be overwritten by the next tile
    }
  }
  __syncthreads();
  if (*pipe.fail) {
    if (tid == 0) {
      const int issued = *pipe.issued;
      for (int st = 0; st < kStages && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / kStages) * kStages;
        mbar_wait(&pipe.full[st], (uint32_t)((last / kStages) & 1));
      }
    }
    __syncthreads();
  }
}

// Chan's combination of (count, mean, M2) summaries: (n, mean, M2) absorbs (nb, mb, Mb).
__device__ __forceinline__ void chan_merge(float &n, float &mean, float &M2, float nb, float mb, float Mb) {
  if (nb <= 0.f) return;
  if (n <= 0.f) {
    n = nb;
    mean = mb;
    M2 = Mb;
    return;
  }
  const float tot = n + nb, dl = mb - mean;
  mean = fmaf(dl, nb / tot, mean);
  M2 = M2 + Mb + dl * dl * (n * nb / tot);
  n = tot;
}

// ---------------------------------------------------------------- moments from MMA fragments
// Per-lane shifted sums of the scores of the two heads n0, n0 + 1 (n0 = 2 (lane
// % 4)) that a lane holds in the m16n8 fragments: the shift is the first score
// the lane sees, so a constant head has exactly zero deviation.
struct LaneMoments {
  float cnt = 0.f, sh[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f}, s2[2] = {0.f, 0.f};
  __device__ __forceinline__ void add(float x0, float x1) {
    if (cnt == 0.f) {
      sh[0] = x0;
      sh[1] = x1;
    }
    const float d0 = x0 - sh[0], d1 = x1 - sh[1];
    s1[0] += d0;
    s1[1] += d1;
    s2[0] = fmaf(d0, d0, s2[0]);
    s2[1] = fmaf(d1, d1, s2[1]);
    cnt += 1.f;
  }
  // (count, mean, M2) of the warp's lanes of this lane's class, merged (Chan)
  // over lane bits 2..4; lanes 0..3 write theirs to red[(warp * 4 + lane) * 5 ..].
  __device__ __forceinline__ void to_shared(float *red, int warp) const {
    const int lane = threadIdx.x & 31;
    float n = cnt, mean[2], m2[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      mean[j] = n > 0.f ? sh[j] + s1[j] / n : 0.f;
      m2[j] = n > 0.f ? fmaxf(s2[j] - s1[j] * s1[j] / n, 0.f) : 0.f;
    }
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
      const float nb = __shfl_xor_sync(0xffffffffu, n, off);
      float mb[2], qb[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        mb[j] = __shfl_xor_sync(0xffffffffu, mean[j], off);
        qb[j] = __shfl_xor_sync(0xffffffffu, m2[j], off);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float nn = n;
        chan_merge(nn, mean[j], m2[j], nb, mb[j], qb[j]);
      }
      n += nb;
    }
    if (lane < 4) {
      float *rw = red + (warp * 4 + lane) * 5;
      rw[0] = n;
      rw[1] = mean[0];
      rw[2] = mean[1];
      rw[3] = m2[0];
      rw[4] = m2[1];
    }
  }
};

// Merges the nwarps warps' states in red for head h: (count, mean, M2).
__device__ __forceinline__ void merge_warp_moments(const float *red, int nwarps, int h, float &n, float &mean,
                                                   float &m2) {
  const int cls = h / 2, j = h & 1;
  n = mean = m2 = 0.f;
  for (int wp = 0; wp < nwarps; ++wp) {
    const float *rw = red + (wp * 4 + cls) * 5;
    chan_merge(n, mean, m2, rw[0], rw[1 + j], rw[3 + j]);
  }
}

// ---------------------------------------------------------------- fused short-unit kernel, tensor cores
// fused_kernel with the tensor-core score of score_tiles_mma_kernel (bf16
// caches, rotate-half bands): a producer warp streams the unit's K through the
// ring with 128B-swizzled tensor copies, 8 consumer warps score 16-key tiles
// with score_tile_mma into the unit's shared-memory scores; then every thread
// runs the same z/max, select and compaction as fused_kernel.
struct FusedMmaArgs {
  CUtensorMap ks;   // 128B-swizzled K map (as TileArgs::ks)
  TmaMaps maps;     // paged caches: block maps for the compaction's tensor stores
  FusedArgs f;
};

// PB: paged cache with block maps (two-warp compaction with row gathers and
// block stores); otherwise warp 0's run copies.
template <int D, int G, bool PB>
__global__ void __launch_bounds__(kThreads, (G <= 4 ? 2 : 1))
    fused_mma_kernel(const __grid_constant__ FusedMmaArgs A) {
  const FusedArgs &a = A.f;
  constexpr int F = D / 2;
  constexpr int TR = kStageBytes / (2 * D);
  constexpr int SPS = TR / 16;
  constexpr int GROUPS = kConsumerWarps / SPS;
  extern __shared__ __align__(1024) char smem[];
  const FusedLayout lay(G, F, a.capp);
  char *ring = smem;
  const Pipe pipe = make_pipe(smem, lay.bars);
  uint64_t *cbars = pipe.full + 2 * kStages;
  float *wts = reinterpret_cast<float *>(smem + lay.wts);
  float *red = reinterpret_cast<float *>(smem + lay.red);
  uint32_t *hist = reinterpret_cast<uint32_t *>(smem + lay.hist);
  int *sm = reinterpret_cast<int *>(smem + lay.sm);
  float *scores = reinterpret_cast<float *>(smem + lay.scores);
  int *idxs = reinterpret_cast<int *>(smem + lay.idx);

  const CacheView &c = a.c;
  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.x;
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  if (timed_out()) return;
  const int N = c.seq_len[s];
  const int B = a.budget;
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  const bool len_writer = a.mode == 0 && tid == 0 && a.new_len != nullptr && l == 0 && g == 0;
  if (a.mode == 0 && N <= B) {
    if (len_writer) a.new_len[s] = N;
    if (a.idx_out != nullptr)
      for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = j < N ? j : -1;
    return;
  }
  if (N == 0) return;
  if (!c.blocks_ok(s, N)) {   // the sequence is skipped: its length stays N
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    if (len_writer) a.new_len[s] = N;
    return;
  }
  if (len_writer) a.new_len[s] = B;
  const int ss = lay.sstride;
  // paged caches compact with two warps (K and V), row gathers and block
  // stores; dense ones with warp 0's run copies
  constexpr bool blk_compact = PB;
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&pipe.full[st], 1);
      mbar_init(&pipe.empty[st], SPS);
      mbar_init(&cbars[st], blk_compact ? kCompactArrivals : 1);
      mbar_init(&cbars[kStages + st], kCompactArrivals);
    }
    *pipe.fail = 0;
    *pipe.issued = 0;
    fence_mbar_init();
  }
  build_weights<G, F>(wts, a.center, a.R, a.mag, a.Hq, l, g, a.t[s], a.sc);
  __syncthreads();
  const int nst = (N + TR - 1) / TR;
  if (warp == kProducerWarp) {
    int t = 0;
    for (; t < nst; ++t) {
      const int st = t % kStages;
      if (*pipe.fail || (t >= kStages && !mbar_wait(&pipe.empty[st], (uint32_t)(((t / kStages) - 1) & 1)))) {
        *pipe.fail = 1;
        break;
      }
      produce_stage_sw<D>(c, &A.ks, l, s, g, (long long)u * c.cap, t * TR, min(TR, N - t * TR),
                          ring + st * kStageBytes, &pipe.full[st], lane);
    }
    if (lane == 0) *pipe.issued = t;
  } else {
    MmaWeights<D, G> w;
    load_mma_weights<D, G>(w, wts, kConsumerWarps * 32, warp == 0);
    const int grp = warp / SPS, sub = warp % SPS;
    const uint32_t ring_a = smem_u32(ring);
    // fragment geometry: this lane holds keys r, r + 8 of a tile for heads n0, n0 + 1
    const int r = lane >> 2, n0 = 2 * (lane & 3);
    const bool holds = G == 8 || n0 < G;
    LaneMoments lm;
    for (int t = grp; t < nst; t += GROUPS) {
      const int st = t % kStages;
      if (!*pipe.fail && !mbar_wait(&pipe.full[st], (uint32_t)((t / kStages) & 1))) *pipe.fail = 1;
      float o[4];
      score_tile_mma_frag<D, G, TR>(ring_a + st * kStageBytes, 16 * sub, w, c.paged() ? c.block : 0, o);
      __syncwarp();
      if (lane == 0) mbar_arrive(&pipe.empty[st]);
      const int nrows = min(TR, N - t * TR), row0 = t * TR;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int row = 16 * sub + r + 8 * hh;
        if (holds && row < nrows) {
          scores[n0 * ss + row0 + row] = o[2 * hh];
          if (G > 1) scores[(n0 + 1) * ss + row0 + row] = o[2 * hh + 1];
          lm.add(o[2 * hh], o[2 * hh + 1]);
        }
      }
    }
    lm.to_shared(red, warp);
  }
  __syncthreads();
  if (*pipe.fail) {
    if (tid == 0) {
      const int issued = *pipe.issued;
      for (int st = 0; st < kStages && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / kStages) * kStages;
        mbar_wait(&pipe.full[st], (uint32_t)((last / kStages) & 1));
      }
    }
    return;
  }

  // the heads' moments from the consumer warps' states
  float *mom = red + kConsumerWarps * 4 * 5;
  if (tid < G) {
    float n, mean, m2;
    merge_warp_moments(red, kConsumerWarps, tid, n, mean, m2);
    const float sd = sqrtf(m2 / (float)N);
    mom[tid] = mean;
    mom[8 + tid] = sd > 0.f ? 1.0f / sd : 0.0f;
  }
  __syncthreads();
  float mu[G], inv[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mu[h] = mom[h];
    inv[h] = mom[8 + h];
  }
  uint32_t *keys = reinterpret_cast<uint32_t *>(scores);   // overlays head 0's scores
  for (int i = tid; i < N; i += nt) {
    float sv[G];
#pragma unroll
    for (int h = 0; h < G; ++h) sv[h] = scores[h * ss + i];
    float z = (sv[0] - mu[0]) * inv[0];
#pragma unroll
    for (int h = 1; h < G; ++h) z = fmaxf(z, (sv[h] - mu[h]) * inv[h]);
    if (a.mode == 1) {
      a.agg[(long long)u * c.cap + i] = z;
      if (a.raw != nullptr) {
#pragma unroll
        for (int h = 0; h < G; ++h) a.raw[((long long)u * G + h) * c.cap + i] = sv[h];
      }
    } else {
      keys[i] = score_key(z);
    }
  }
  if (a.mode == 1) return;
  __syncthreads();
  int ntie;
  const uint32_t T = radix_select_atomic(keys, N, B, hist, sm, &ntie);
  if (a.defer) {   // hole-fill: the kept set as a bitmask in idx_out; holefill_apply_kernel does the rest
    kept_bits(keys, N, T, ntie, reinterpret_cast<uint32_t *>(a.idx_out + (long long)u * B), sm);
    return;
  }
  const int e0 = build_kept_chunked(keys, N, B, T, ntie, idxs, sm);
  if (a.holefill) {
    holefill_unit(c, l, s, g, idxs, B, N, reinterpret_cast<char *>(keys), ring, kRingBytes, sm,
                  a.idx_out != nullptr ? a.idx_out + (long long)u * B : nullptr);
    return;
  }
  if (a.idx_out != nullptr)
    for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = idxs[j];
  // The ring was last read by ldmatrix (generic proxy); TMA writes it next.
  fence_proxy_async_smem();
  __syncthreads();
  if constexpr (PB) {
    if (warp < 2) compact_unit_tma(c, &A.maps, warp, l, s, g, idxs, e0, B, N, ring, kStages, cbars + warp * kStages);
  } else {
    if (warp == 0) compact_unit_runs(c, l, s, g, idxs, e0, B, N, ring, cbars);
  }
}

// Merges the per-tile (mean, M2) of a unit's N keys; warp h < G handles head h
// (lanes take tiles lane, lane + 32, ..., then a butterfly of Chan merges) and
// writes mean and 1/std (0 if std = 0) to mom[h], mom[8 + h].  Needs blockDim
// >= 32 * G; the caller synchronises before reading mom.
__device__ __forceinline__ void merge_tile_moments(const float2 *part, long long u, int ntiles, int G,
                                                   int N, float *mom, int part_keys) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= G) return;
  const int h = warp;
  const int TK = part_keys;
  const int used = (N + TK - 1) / TK;
  float n = 0.f, mean = 0.f, M2 = 0.f;
  for (int t = lane; t < used; t += 32) {
    const float2 p = part[(u * ntiles + t) * G + h];
    chan_merge(n, mean, M2, (float)min(TK, N - t * TK), p.x, p.y);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float n2 = __shfl_xor_sync(0xffffffffu, n, o);
    const float m2 = __shfl_xor_sync(0xffffffffu, mean, o);
    const float q2 = __shfl_xor_sync(0xffffffffu, M2, o);
    if (lane & o)
      chan_merge(n, mean, M2, n2, m2, q2);   // both partners merge in the same order
    else {
      float a = n2, b = m2, cq = q2;
      chan_merge(a, b, cq, n, mean, M2);
      n = a;
      mean = b;
      M2 = cq;
    }
  }
  if (lane == 0) {
    const float sd = sqrtf(M2 / n);
    mom[h] = mean;
    mom[8 + h] = sd > 0.f ? 1.0f / sd : 0.0f;
  }
}

// a3 from key-major raw scores: key i's G scores are raw_u[i*G .. i*G + G)
// (16-byte aligned rows of 4 keys); each thread takes quads of keys (G 16-byte
// loads, contiguous across threads) and writes their order-preserving keys.
// Key slots in [N, round4(N)) receive don't-care values.
template <int G>
__device__ void zmax_from_raw_km(const float *raw_u, int N, const float *mom, uint32_t *keys) {
  const int tid = threadIdx.x, nt = blockDim.x;
  float mu[G], iv[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mu[h] = mom[h];
    iv[h] = mom[8 + h];
  }
  const int n4 = (N + 3) / 4;
  const float4 *rows = reinterpret_cast<const float4 *>(raw_u);
  for (int q = tid; q < n4; q += nt) {
    float x[4 * G];
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const float4 v = __ldg(rows + (long long)q * G + k);
      x[4 * k] = v.x;
      x[4 * k + 1] = v.y;
      x[4 * k + 2] = v.z;
      x[4 * k + 3] = v.w;
    }
    uint32_t kk[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float z = (x[j * G] - mu[0]) * iv[0];
#pragma unroll
      for (int h = 1; h < G; ++h) z = fmaxf(z, (x[j * G + h] - mu[h]) * iv[h]);
      kk[j] = score_key(z);
    }
    reinterpret_cast<uint4 *>(keys)[q] = make_uint4(kk[0], kk[1], kk[2], kk[3]);
  }
}

// ---------------------------------------------------------------- long units: key-major scores
// The compress step's long-unit score kernel (bf16 caches, rotate-half bands).
// As score_tiles_mma_kernel, but each 16-key tile's scores go straight from the
// MMA fragments to the workspace in key-major order (key i's G scores at
// raw[(u*capp + i)*G + h]: a quad of lanes holds one key's heads, so the warp
// writes whole 256-byte (G = 8) or 128-byte (G = 4) runs), and every lane keeps
// shifted sums of its heads' scores in registers.  There is no per-tile
// epilogue: the consumers never stop streaming.  At the end the lanes' (count,
// mean, M2) merge (Chan) into one entry per CTA and head in `part`.
constexpr int kKmCtaKeys = 8192;   // keys per CTA (one part entry)
constexpr int kKmStages = 6;       // ring stages (the score tile buffer is gone)

struct KmLayout {
  int bars, wts, red, total;
  __host__ __device__ KmLayout(int G, int F) {
    int o = kKmStages * kStageBytes;
    bars = o;  o += 256;                       // full[6], empty[6], fail, issued
    wts = o;   o += align_up(G * 3 * F * 4, 128);
    red = o;   o += kConsumerWarps * 4 * 5 * 4;   // per warp and lane class: n, mean[2], M2[2]
    total = o;
  }
};

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 2) score_keys_mma_kernel(const __grid_constant__ TileArgs a) {
  constexpr int F = D / 2;
  constexpr int TR = kStageBytes / (2 * D);
  constexpr int SPS = TR / 16;
  constexpr int GROUPS = kConsumerWarps / SPS;
  constexpr int NC = kConsumerWarps * 32;
  extern __shared__ __align__(1024) char smem[];
  const KmLayout lay(G, F);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint64_t *empty = full + kKmStages;
  volatile int *fail = reinterpret_cast<volatile int *>(empty + kKmStages);
  volatile int *issued = fail + 1;
  float *wts = reinterpret_cast<float *>(smem + lay.wts);
  float *red = reinterpret_cast<float *>(smem + lay.red);
  const CacheView &c = a.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.y;
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  if (timed_out()) return;
  const int N = c.seq_len[s];
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (a.skip_small && N <= a.budget) return;
  const int i0 = blockIdx.x * kKmCtaKeys;
  if (i0 >= N) return;
  const int n = min(kKmCtaKeys, N - i0);
  if (!c.blocks_ok(s, n, i0)) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (tid == 0) {
    for (int st = 0; st < kKmStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], SPS);
    }
    *fail = 0;
    *issued = 0;
    fence_mbar_init();
  }
  build_weights<G, F>(wts, a.center, a.R, a.mag, a.Hq, l, g, a.t[s], a.sc, a.phase + (long long)s * F);
  __syncthreads();
  const int nst = (n + TR - 1) / TR;
  const long long urow0 = (long long)u * c.cap;
  // lane state: shifted sums of the two heads n0, n0 + 1 of this lane
  const int r = lane >> 2, n0 = 2 * (lane & 3);
  const bool holds = G == 8 || n0 < G;
  LaneMoments lm;
  if (warp == kProducerWarp) {
    int t = 0;
    for (; t < nst; ++t) {
      const int st = t % kKmStages;
      if (*fail || (t >= kKmStages && !mbar_wait(&empty[st], (uint32_t)(((t / kKmStages) - 1) & 1)))) {
        *fail = 1;
        break;
      }
      produce_stage_sw<D>(c, &a.ks, l, s, g, urow0, i0 + t * TR, min(TR, n - t * TR), smem + st * kStageBytes,
                          &full[st], lane);
    }
    if (lane == 0) *issued = t;
  } else {
    MmaWeights<D, G> w;
    load_mma_weights<D, G>(w, wts, NC, warp == 0);
    const int grp = warp / SPS, sub = warp % SPS;
    const uint32_t ring = smem_u32(smem);
    float *raw_c = a.raw + ((long long)u * a.raw_stride + i0) * G;   // this CTA's first key
    const int blk = c.paged() ? c.block : 0;
    for (int t = grp; t < nst; t += GROUPS) {
      const int st = t % kKmStages;
      if (!*fail && !mbar_wait(&full[st], (uint32_t)((t / kKmStages) & 1))) *fail = 1;
      float o[4];
      score_tile_mma_frag<D, G, TR>(ring + st * kStageBytes, 16 * sub, w, blk, o);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);   // the stage's rows are in registers
      if (*fail) continue;
      const int kb = t * TR + 16 * sub;         // CTA-local key of this tile's row 0
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int key = kb + r + 8 * hh;
        if (holds && key < n) {
          const float x0 = o[2 * hh], x1 = o[2 * hh + 1];
          if constexpr (G == 1)
            raw_c[key] = x0;
          else
            *reinterpret_cast<float2 *>(raw_c + (long long)key * G + n0) = make_float2(x0, x1);
          lm.add(x0, x1);
        }
      }
    }
    lm.to_shared(red, warp);
  }
  __syncthreads();
  if (*fail) {
    if (tid == 0) {
      const int iss = *issued;
      for (int st = 0; st < kKmStages && st < iss; ++st) {
        const int last = st + ((iss - 1 - st) / kKmStages) * kKmStages;
        mbar_wait(&full[st], (uint32_t)((last / kKmStages) & 1));
      }
    }
    return;
  }
  if (tid < G) {
    float nn, mm, qq;
    merge_warp_moments(red, kConsumerWarps, tid, nn, mm, qq);
    a.part[((long long)u * a.ntiles + blockIdx.x) * G + tid] = make_float2(mm, qq);
  }
}

// ---------------------------------------------------------------- long units, paged: every KV head of a block
// score_keys_mma_kernel for paged bf16 caches (d = 128, rotate-half bands)
// whose block holds 128 head-rows (Hkv x block = 128: 8 heads of 16 rows, or 4
// of 32): a CTA scores all KV heads of one (layer, sequence) over kHgKeys
// keys, and each stage is one whole block, 32 KB contiguous in HBM, brought in
// by one tensor copy (box: 64 elements x block rows x 2 halves x Hkv heads),
// instead of one 4 KB copy per block and head with the rows 2 KB apart.  In
// shared memory the stage is [head][half][block rows][128 B], each head's part
// laid out as a one-block stage of the per-head kernel.  16 consumer warps:
// warp w takes tile w % 8 of the stages with parity w / 8 (a stage holds 8
// 16-row tiles, Hkv x block / 16), i.e. the rows 16 (tile % TPH) .. of head
// tile / TPH (TPH = block / 16 tiles per head).  Raw scores and the lanes'
// moments as score_keys_mma_kernel, one (mean, M2) entry per CTA and head.
// One CTA per SM (17 warps) with a 6 x 32 KB ring.  The consumers build the
// fp32 weights of all the CTA's heads in ring slots 4 and 5 and take their
// fragments (G = 8: lo fragments to a region of their own) while the producer
// fills slots 0 to 3; it issues slot 4 only once every consumer has passed
// named barrier 2.  The stage count is even so that every ring slot is only
// ever read by the warps of one parity: a warp then waits on each phase of its
// slots' full barriers in turn, and a parity wait cannot match a phase two
// back (a slot shared by both parities would let a warp that ran a cycle
// ahead see the previous use's completed phase as its own).
constexpr int kHgKeys = 8192;       // keys per CTA and head (one part entry)
constexpr int kHgStages = 6;
constexpr int kHgEarly = 4;         // stages issued before the weights are taken
static_assert(kHgStages % 2 == 0, "ring slots must belong to one consumer parity");
constexpr int kHgStageBytes = 32768;
constexpr int kHgConsumers = 16;
constexpr int kHgThreads = (kHgConsumers + 1) * 32;

struct HgLayout {
  int bars, wts, lo, red, total;
  __host__ __device__ HgLayout(int G, int F, int Hkv) {
    int o = kHgStages * kHgStageBytes;
    wts = kHgEarly * kHgStageBytes;                    // [Hkv][G][3][F] fp32, in ring slots 4 and 5
    bars = o;  o += 256;                               // full[6], empty[6], fail, issued
    lo = o;    o += G == 8 ? Hkv * (3 * F / 16) * 32 * 8 : 0;   // G = 8: [Hkv][12 k-steps][32 lanes] lo fragments
    red = o;   o += kHgConsumers * 4 * 5 * 4;
    total = o;
  }
};

template <int G>
__global__ void __launch_bounds__(kHgThreads, 1) score_heads_mma_kernel(const __grid_constant__ TileArgs a) {
  constexpr int D = 128, F = 64, NC = kHgConsumers * 32;
  extern __shared__ __align__(1024) char smem[];
  const CacheView &c = a.c;
  const HgLayout lay(G, F, c.Hkv);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint64_t *empty = full + kHgStages;
  volatile int *fail = reinterpret_cast<volatile int *>(empty + kHgStages);
  volatile int *issued = fail + 1;
  float *wts = reinterpret_cast<float *>(smem + lay.wts);
  float *lo = reinterpret_cast<float *>(smem + lay.lo);
  float *red = reinterpret_cast<float *>(smem + lay.red);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int ls, chunk;
  if (a.plan != nullptr) {   // 1-D grid over the chunk plan: full chunks, then partial ones, largest first
    const int nfull = a.plan[0], npart = a.plan[1];
    const long long i = blockIdx.x, nf = (long long)c.L * nfull;
    int ll, sq;
    if (i < nf) {
      ll = (int)(i / nfull);
      const int k = (int)(i % nfull);
      int lo = 0, hi = c.S - 1;   // the last sequence whose full chunks start at or before k
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.plan[2 + mid] <= k) lo = mid; else hi = mid - 1;
      }
      sq = lo;
      chunk = k - a.plan[2 + lo];
    } else if (i < nf + (long long)c.L * npart) {
      const long long j = i - nf;
      ll = (int)(j % c.L);
      sq = a.plan[2 + c.S + (int)(j / c.L)];
      chunk = c.seq_len[sq] / kHgKeys;
    } else {
      return;
    }
    ls = ll * c.S + sq;
  } else {
    ls = blockIdx.y;
    chunk = blockIdx.x;
  }
  const int s = ls % c.S, l = ls / c.S;
  if (timed_out()) return;
  const int N = c.seq_len[s];
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (a.skip_small && N <= a.budget) return;
  const int i0 = chunk * kHgKeys;
  if (i0 >= N) return;
  const int n = min(kHgKeys, N - i0);
  if (!c.blocks_ok(s, n, i0)) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  const int blk = c.block, TPH = blk / 16;
  const int nst = (n + blk - 1) / blk;
  if (tid == 0) {
    for (int st = 0; st < kHgStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 8);   // the 8 consumer warps of the stage's parity
    }
    *fail = 0;
    *issued = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kHgConsumers) {   // producer: one copy per block, all heads
    int t = 0;
    bool taken = false;   // the consumers hold their weights: slots kHgEarly.. are free
    for (; t < nst; ++t) {
      if (t == kHgEarly) {
        named_sync(2, kHgThreads);
        taken = true;
      }
      const int st = t % kHgStages;
      if (*fail || (t >= kHgStages && !mbar_wait(&empty[st], (uint32_t)(((t / kHgStages) - 1) & 1)))) {
        *fail = 1;
        break;
      }
      if (lane == 0) {
        const int b = c.bt[(long long)s * c.max_blocks + i0 / blk + t];
        mbar_arrive_expect_tx(&full[st], (uint32_t)(c.Hkv * blk * 256));
        tma_load_5d(smem + st * kHgStageBytes, &a.ks, 0, 0, 0, 0, (int)((long long)l * c.nblocks + b), &full[st]);
      }
      __syncwarp();
    }
    if (lane == 0) *issued = t;
    if (!taken) named_sync(2, kHgThreads);
  } else {
    for (int hh = 0; hh < c.Hkv; ++hh)
      build_weights<G, F>(wts + hh * G * 3 * F, a.center, a.R, a.mag, a.Hq, l, hh, a.t[s], a.sc,
                          a.phase + (long long)s * F, NC);
    named_sync(1, NC);
    const int tile = warp & 7, par = warp >> 3;
    const int h = tile / TPH, sub = tile - h * TPH;
    MmaWeights<D, G> w;
    load_mma_weights<D, G>(w, wts + h * G * 3 * F, NC, par == 0 && sub == 0, lo + h * (3 * F / 16) * 32 * 2);
    fence_proxy_async_smem();    // slots 4 and 5 were written by plain stores; tensor copies refill them
    named_sync(2, kHgThreads);   // the weights there are dead: the producer may refill them
    const uint32_t ring = smem_u32(smem);
    const long long u = (long long)ls * c.Hkv + h;
    float *raw_c = a.raw + ((long long)u * a.raw_stride + i0) * G;   // this CTA's first key of head h
    const int r = lane >> 2, n0 = 2 * (lane & 3);
    const bool holds = G == 8 || n0 < G;
    LaneMoments lm;
    for (int t = par; t < nst; t += 2) {
      const int st = t % kHgStages;
      if (!*fail && !mbar_wait(&full[st], (uint32_t)((t / kHgStages) & 1))) *fail = 1;
      float o[4];
      score_tile_mma_frag<D, G, 64>(ring + st * kHgStageBytes + h * (2 * blk * 128), 16 * sub, w, blk, o);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);   // the stage's rows are in registers
      if (*fail) continue;
      const int kb = t * blk + 16 * sub;        // CTA-local key of this tile's row 0
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int key = kb + r + 8 * hh;
        if (holds && key < n) {
          const float x0 = o[2 * hh], x1 = o[2 * hh + 1];
          if constexpr (G == 1)
            raw_c[key] = x0;
          else
            *reinterpret_cast<float2 *>(raw_c + (long long)key * G + n0) = make_float2(x0, x1);
          lm.add(x0, x1);
        }
      }
    }
    lm.to_shared(red, warp);
  }
  __syncthreads();
  if (*fail) {
    if (tid == 0) {
      const int iss = *issued;
      for (int st = 0; st < kHgStages && st < iss; ++st) {
        const int last = st + ((iss - 1 - st) / kHgStages) * kHgStages;
        mbar_wait(&full[st], (uint32_t)((last / kHgStages) & 1));
      }
    }
    return;
  }
  if (tid < c.Hkv * G) {   // (KV head, query head of its group): merge the warps of that KV head
    const int h = tid / G, qh = tid - h * G, cls = qh / 2, j = qh & 1;
    float nn = 0.f, mm = 0.f, qq = 0.f;
    for (int wp = 0; wp < kHgConsumers; ++wp) {
      if ((wp & 7) / TPH != h) continue;
      const float *rw = red + (wp * 4 + cls) * 5;
      chan_merge(nn, mm, qq, rw[0], rw[1 + j], rw[3 + j]);
    }
    const long long u = (long long)ls * c.Hkv + h;
    a.part[((long long)u * a.ntiles + chunk) * G + qh] = make_float2(mm, qq);
  }
}

struct ZArgs {
  int S, Hkv, G, ntiles;
  long long cap, raw_stride;
  const int *seq_len;
  const float *raw;
  const float2 *part;
  float *agg;
};

__global__ void __launch_bounds__(256) zmax_kernel(const ZArgs a) {
  __shared__ float mom[16];
  const int tile = blockIdx.x, u = blockIdx.y;
  const int s = (u / a.Hkv) % a.S;
  const int N = a.seq_len[s];
  if (N < 0 || N > a.cap) return;
  const int i0 = tile * tile_keys_for(a.G);
  if (i0 >= N) return;
  merge_tile_moments(a.part, u, a.ntiles, a.G, N, mom, tile_keys_for(a.G));
  __syncthreads();
  const int i1 = min(N, i0 + tile_keys_for(a.G));
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    float z = -INFINITY;
    for (int h = 0; h < a.G; ++h) {
      const float zh = (a.raw[((long long)u * a.G + h) * a.raw_stride + i] - mom[h]) * mom[8 + h];
      z = h == 0 ? zh : fmaxf(z, zh);
    }
    a.agg[(long long)u * a.cap + i] = z;
  }
}

// ---------------------------------------------------------------- select / compact
struct SCArgs {
  TmaMaps maps;
  CacheView c;
  int G, budget, mode, ntiles, capp, bcap;   // mode 0: from raw (+compact), 1: from agg, 2: compact idx
  int holefill;                              // compaction layout (modes 0, 2): 0 ordered, 1 hole-fill
  const float *raw;     // mode 0: workspace [(u*G + h)*capp + i], rows 16-byte aligned
  const float2 *part;
  const float *agg;
  const int *idx_in;
  int *idx_out, *new_len;
  uint32_t *keys;   // select_only_kernel: workspace [units][capp] (16-byte aligned rows)
  int raw_km;       // mode 0: raw is key-major [(u*capp + i)*G + h] (else head-major)
  int part_keys;    // mode 0: keys covered by one (mean, M2) entry of part
  int *kept;        // select_only / compact_only: kept slots [units][budget] (idx_out or workspace)
  int *e0s;         // select_only / compact_only: first dropped slot per unit (workspace)
  const int *order; // select_only: sequences longest first (its CTAs take units in that order), or null
};

// The keys (one u32 per slot) and the compaction ring share one region at the
// start of shared memory: the keys are dead once the kept list is built, and
// the ring is first used after that.  The region holds at least kCompactStages
// stages (more when the keys need it, up to kMaxCompactStages).
struct SCLayout {
  int keys, bars, hist, sm, mom, idx, nstages, total;
  __host__ __device__ SCLayout(int capp, int bcap) {
    int o = 0;
    keys = o;
    const int kb = align_up(capp * 4 > kCompactStages * kStageBytes ? capp * 4 : kCompactStages * kStageBytes,
                            kStageBytes);
    o += kb;
    nstages = min(kMaxCompactStages, kb / kStageBytes);
    bars = o; o += 2 * kMaxCompactStages * 8;
    hist = o; o += 1024;
    sm = o;   o += kSelInts * 4;
    mom = o;  o += 128;
    idx = o;  o += align_up(bcap * 4, 128);
    total = o;
  }
};



// a3 for one long unit from its raw scores: the G rows raw[h][0..N) (stride
// capp floats, 16-byte aligned) are read with 16-byte loads, U*G of them per
// thread and batch, the next batch's loads issued before the current batch is
// used; every thread turns its keys into z = max_h (s_h - mean_h) / std_h and
// writes the order-preserving keys (4 per store).  Key slots in
// [N, round4(N)) receive don't-care values.
template <int G, bool PF = true>
__device__ void zmax_from_raw(const float *raw_u, int capp, int N, const float *mom, uint32_t *keys) {
  constexpr int U = G >= 8 ? 1 : 8 / G;
  const int tid = threadIdx.x, nt = blockDim.x;
  float mu[G], iv[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mu[h] = mom[h];
    iv[h] = mom[8 + h];
  }
  const int n4 = (N + 3) / 4;
  const float4 *rows = reinterpret_cast<const float4 *>(raw_u);
  const int hs = capp / 4;   // float4 stride between heads
  float4 cur[U][G], nxt[PF ? U : 1][PF ? G : 1];
  auto load = [&](float4 (&v)[U][G], int base) {
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int q = base + k * nt;
#pragma unroll
      for (int h = 0; h < G; ++h) v[k][h] = q < n4 ? __ldg(rows + (long long)h * hs + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  if constexpr (PF) load(cur, tid);
  for (int base = tid; base < n4; base += nt * U) {
    if constexpr (PF)
      load(nxt, base + nt * U);
    else
      load(cur, base);
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int q = base + k * nt;
      float z[4];
      z[0] = (cur[k][0].x - mu[0]) * iv[0];
      z[1] = (cur[k][0].y - mu[0]) * iv[0];
      z[2] = (cur[k][0].z - mu[0]) * iv[0];
      z[3] = (cur[k][0].w - mu[0]) * iv[0];
#pragma unroll
      for (int h = 1; h < G; ++h) {
        z[0] = fmaxf(z[0], (cur[k][h].x - mu[h]) * iv[h]);
        z[1] = fmaxf(z[1], (cur[k][h].y - mu[h]) * iv[h]);
        z[2] = fmaxf(z[2], (cur[k][h].z - mu[h]) * iv[h]);
        z[3] = fmaxf(z[3], (cur[k][h].w - mu[h]) * iv[h]);
      }
      if (q < n4)
        reinterpret_cast<uint4 *>(keys)[q] = make_uint4(score_key(z[0]), score_key(z[1]), score_key(z[2]),
                                                        score_key(z[3]));
    }
    if constexpr (PF) {
#pragma unroll
      for (int k = 0; k < U; ++k)
#pragma unroll
        for (int h = 0; h < G; ++h) cur[k][h] = nxt[k][h];
    }
  }
}

// zmax_from_raw or zmax_from_raw_km for the unit's G.
template <bool PF>
__device__ __forceinline__ void zmax_dispatch(const SCArgs &a, long long u, int N, const float *mom,
                                              uint32_t *keys) {
  const float *raw_u = a.raw + u * a.G * a.capp;
  if (a.raw_km) {
    switch (a.G) {
      case 1: zmax_from_raw_km<1>(raw_u, N, mom, keys); break;
      case 2: zmax_from_raw_km<2>(raw_u, N, mom, keys); break;
      case 4: zmax_from_raw_km<4>(raw_u, N, mom, keys); break;
      default: zmax_from_raw_km<8>(raw_u, N, mom, keys); break;
    }
    return;
  }
  switch (a.G) {
    case 1: zmax_from_raw<1, PF>(raw_u, a.capp, N, mom, keys); break;
    case 2: zmax_from_raw<2, PF>(raw_u, a.capp, N, mom, keys); break;
    case 4: zmax_from_raw<4, PF>(raw_u, a.capp, N, mom, keys); break;
    default: zmax_from_raw<8, PF>(raw_u, a.capp, N, mom, keys); break;
  }
}

__global__ void __launch_bounds__(kSelThreads, 1) select_compact_kernel(const __grid_constant__ SCArgs a) {
  extern __shared__ __align__(1024) char smem[];
  const SCLayout lay(a.capp, a.bcap);
  char *ring = smem;
  uint64_t *cbars = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint32_t *hist = reinterpret_cast<uint32_t *>(smem + lay.hist);
  int *sm = reinterpret_cast<int *>(smem + lay.sm);
  float *mom = reinterpret_cast<float *>(smem + lay.mom);
  uint32_t *keys = reinterpret_cast<uint32_t *>(smem + lay.keys);
  int *idxs = reinterpret_cast<int *>(smem + lay.idx);
  const CacheView &c = a.c;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int u = blockIdx.x;
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  if (timed_out()) return;
  const int N = c.seq_len[s];
  const int B = a.budget;
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  const bool len_writer = a.mode != 1 && tid == 0 && a.new_len != nullptr && l == 0 && g == 0;
  if (N <= B) {
    if (len_writer) a.new_len[s] = N;
    if (a.mode != 2 && a.idx_out != nullptr)
      for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = j < N ? j : -1;
    return;
  }
  if (a.mode != 1 && !c.blocks_ok(s, N)) {   // the sequence is skipped: its length stays N
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    if (len_writer) a.new_len[s] = N;
    return;
  }
  if (len_writer) a.new_len[s] = B;
  if (tid == 0) {
    for (int st = 0; st < lay.nstages; ++st) {
      mbar_init(&cbars[st], kCompactArrivals);                       // K warp
      mbar_init(&cbars[kMaxCompactStages + st], kCompactArrivals);   // V warp
    }
    fence_mbar_init();
  }
  if (a.mode == 2) {
    const int *src = a.idx_in + (long long)u * B;
    int bad = 0;
    for (int j = tid; j < B; j += nt) {
      const int v = src[j];
      idxs[j] = v;
      bad |= (v < 0) | (v >= N) | (j > 0 && v <= src[j - 1]);
    }
    if (tid == 0) sm[56] = B;
    if (__syncthreads_or(bad)) {
      if (tid == 0) set_status(TRI_ERR_INVALID);
      return;
    }
    if (a.holefill) {
      const int wb = align_up(holefill_work_bytes(B, N), 128);
      holefill_unit(c, l, s, g, idxs, B, N, reinterpret_cast<char *>(keys) + lay.bars - wb, reinterpret_cast<char *>(keys),
                    lay.bars - wb, sm, nullptr);
      return;
    }
    for (int j = tid; j < B; j += nt)
      if (idxs[j] != j) atomicMin(&sm[56], j);
    __syncthreads();
    const int e0 = sm[56];
    __syncthreads();
    if ((tid >> 5) < 2)
      compact_unit_tma(c, &a.maps, tid >> 5, l, s, g, idxs, e0, B, N, ring, lay.nstages,
                       cbars + (tid >> 5) * kMaxCompactStages);
    return;
  }
  if (a.mode == 0) {
    merge_tile_moments(a.part, u, a.ntiles, a.G, N, mom, a.part_keys);
    __syncthreads();
    zmax_dispatch<true>(a, u, N, mom, keys);
  } else {
    for (int i = tid; i < N; i += nt) keys[i] = score_key(a.agg[(long long)u * c.cap + i]);
  }
  __syncthreads();
  int ntie;
  const uint32_t T = radix_select_atomic(keys, N, B, hist, sm, &ntie);
  const int e0 = build_kept(keys, N, B, T, ntie, idxs, sm);
  if (a.mode == 0 && a.holefill) {   // keys are dead: their region holds the hole-fill bookkeeping
    const int wb = align_up(holefill_work_bytes(B, N), 128);
    holefill_unit(c, l, s, g, idxs, B, N, reinterpret_cast<char *>(keys) + lay.bars - wb, reinterpret_cast<char *>(keys),
                  lay.bars - wb, sm, a.idx_out != nullptr ? a.idx_out + (long long)u * B : nullptr);
    return;
  }
  if (a.idx_out != nullptr)
    for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = idxs[j];
  if (a.mode == 0) {
    // The ring extends over the keys, last accessed by generic loads and
    // stores; TMA writes them next.
    fence_proxy_async_smem();
    __syncthreads();
    if ((tid >> 5) < 2)
      compact_unit_tma(c, &a.maps, tid >> 5, l, s, g, idxs, e0, B, N, ring, lay.nstages,
                       cbars + (tid >> 5) * kMaxCompactStages);
  }
}

// ---------------------------------------------------------------- long units: select, then compact
// The compress step's long-unit selection and compaction as two kernels.  The
// selection's passes over a unit's keys (z/max from the raw scores, four radix
// passes, two kept-list passes; keys in the workspace, L2-resident) are bound
// by L2 latency, not bandwidth, so select_only_kernel keeps almost nothing in
// shared memory and many units share an SM; it writes each unit's kept slots
// and first dropped slot.  compact_only_kernel then only moves rows: two CTAs
// per SM, each with a K warp and a V warp on 6-stage rings, so the bytes in
// flight per SM stay high for the whole kernel.
constexpr int kSelOnlyThreads = 256;
constexpr int kCoThreads = 256;
constexpr int kCoStages = 6;

// Digit step of a radix select: hist[256] counts the current digit over the
// keys still in play, and k of them are to be taken from the top.  Every
// thread gets the digit d with S[d] >= k > S[d + 1] (S[x] = keys whose digit is
// >= x) and the number to take among the keys with digit d.  The caller
// synchronises between building hist and this call.  blockDim >= 256; sm: the
// selection's shared ints ([0..1] and [8..15] here).
__device__ __forceinline__ void radix_pick(const uint32_t *hist, int k, int *sm, uint32_t &dgt, int &k_in) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int P = 0;
  if (tid < 256) {   // thread t scans the reversed histogram: its prefix is S[255 - t]
    P = (int)hist[255 - tid];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, P, o);
      if (lane >= o) P += y;
    }
    if (lane == 31) sm[8 + warp] = P;
  }
  __syncthreads();
  if (tid < 256) {
    int wsum = 0;
    for (int w = 0; w < warp; ++w) wsum += sm[8 + w];
    P += wsum;
    int Pprev = __shfl_up_sync(0xffffffffu, P, 1);
    if (lane == 0) Pprev = wsum;
    if (P >= k && Pprev < k) {
      sm[0] = 255 - tid;
      sm[1] = k - Pprev;
    }
  }
  __syncthreads();
  dgt = (uint32_t)sm[0];
  k_in = sm[1];
  __syncthreads();
}

// a3 from key-major raw scores (as zmax_from_raw_km) plus the histogram of the
// keys' top digit (the radix select's first pass).  Each thread loads U quads
// of keys (8 16-byte loads) before using any of them.
template <int G>
__device__ __noinline__ void zmax_km_hist(const float *raw_u, int N, const float *mom, uint32_t *keys, uint32_t *hist) {
  constexpr int U = G >= 8 ? 1 : 8 / G;
  const int tid = threadIdx.x, nt = blockDim.x;
  float mu[G], iv[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mu[h] = mom[h];
    iv[h] = mom[8 + h];
  }
  const int n4 = (N + 3) / 4;
  const float4 *rows = reinterpret_cast<const float4 *>(raw_u);
  for (int q0 = tid; q0 < n4; q0 += nt * U) {
    float4 v[U][G];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int q = q0 + k * nt;
#pragma unroll
      for (int h = 0; h < G; ++h) v[k][h] = q < n4 ? __ldg(rows + (long long)q * G + h) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int q = q0 + k * nt;
      if (q >= n4) break;
      float x[4 * G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        x[4 * h] = v[k][h].x;
        x[4 * h + 1] = v[k][h].y;
        x[4 * h + 2] = v[k][h].z;
        x[4 * h + 3] = v[k][h].w;
      }
      uint32_t kk[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float z = (x[j * G] - mu[0]) * iv[0];
#pragma unroll
        for (int h = 1; h < G; ++h) z = fmaxf(z, (x[j * G + h] - mu[h]) * iv[h]);
        kk[j] = score_key(z);
        if (4 * q + j < N) atomicAdd(&hist[kk[j] >> 24], 1u);
      }
      reinterpret_cast<uint4 *>(keys)[q] = make_uint4(kk[0], kk[1], kk[2], kk[3]);
    }
  }
}

__device__ __forceinline__ void zmax_km_hist_dispatch(const SCArgs &a, long long u, int N, const float *mom,
                                                      uint32_t *keys, uint32_t *hist) {
  const float *raw_u = a.raw + u * a.G * a.capp;
  switch (a.G) {
    case 1: zmax_km_hist<1>(raw_u, N, mom, keys, hist); break;
    case 2: zmax_km_hist<2>(raw_u, N, mom, keys, hist); break;
    case 4: zmax_km_hist<4>(raw_u, N, mom, keys, hist); break;
    default: zmax_km_hist<8>(raw_u, N, mom, keys, hist); break;
  }
}

// The rest of a long unit's top-K after the first digit (d1, with k to take
// among the keys whose top digit is d1; hist holds nothing needed).  One pass
// over the keys (each warp its contiguous segment, as the kept list's) counts
// per warp the keys whose top digit exceeds d1, which are kept whatever their
// other digits, and appends the keys whose top digit is d1 to cand as (key,
// slot) pairs, histogramming their second digit.  The last three digits are
// then resolved over the candidates alone, which also give each warp's count
// of keys above and equal to the threshold T; a last pass writes the kept
// slots in ascending order (those > T, then the first ntie equal to T in slot
// order), as build_kept_gmem.  cand: room for every key of digit d1.  wc:
// 3 nw + 1 shared ints.  Returns the first dropped slot.
__device__ __noinline__ int select_rest_candidates(const uint32_t *keys, int n, uint32_t d1, int k, uint2 *cand,
                                                   uint32_t *hist, int *sm, int *wc, int *idx, int K) {
  constexpr int PF = 16;  // steps of 32 keys loaded together (the passes are bound by L2 latency)
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  int *cgt = wc, *gtc = wc + nw, *eqc = wc + 2 * nw, *ncand = wc + 3 * nw;
  for (int b = tid; b < 256; b += nt) hist[b] = 0;
  if (tid < nw) {
    gtc[tid] = 0;
    eqc[tid] = 0;
  }
  if (tid == 0) *ncand = 0;
  __syncthreads();
  const int seg = (((n + nw - 1) / nw) + 31) / 32 * 32;
  const int lo = min(n, warp * seg), hi = min(n, lo + seg);
  const unsigned lt = lanemask_lt();
  int ngt = 0;
  for (int base = lo; base < hi; base += 32 * PF) {
    uint32_t u[PF];
#pragma unroll
    for (int e = 0; e < PF; ++e) {
      const int i = base + 32 * e + lane;
      u[e] = i < hi ? keys[i] : 0u;
    }
#pragma unroll
    for (int e = 0; e < PF; ++e) {
      const int i = base + 32 * e + lane;
      const bool in = i < hi;
      const uint32_t top = u[e] >> 24;
      ngt += __popc(__ballot_sync(0xffffffffu, in && top > d1));
      const unsigned m = __ballot_sync(0xffffffffu, in && top == d1);
      if (m != 0u) {
        int b0 = 0;
        if (lane == 0) b0 = atomicAdd(ncand, __popc(m));
        b0 = __shfl_sync(0xffffffffu, b0, 0);
        if (in && top == d1) {
          cand[b0 + __popc(m & lt)] = make_uint2(u[e], (uint32_t)i);
          atomicAdd(&hist[(u[e] >> 16) & 255u], 1u);
        }
      }
    }
  }
  if (lane == 0) cgt[warp] = ngt;
  __syncthreads();   // candidates (global) and their histogram are complete
  const int c1 = *ncand;
  uint32_t dg;
  radix_pick(hist, k, sm, dg, k);
  uint32_t prefix = (d1 << 24) | (dg << 16), mask = 0xffff0000u;
  for (int shift = 8; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += nt) hist[b] = 0;
    __syncthreads();
    for (int x = tid; x < c1; x += nt) {
      const uint32_t key = cand[x].x;
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    radix_pick(hist, k, sm, dg, k);
    prefix |= dg << shift;
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;
  const int ntie = k;
  for (int x = tid; x < c1; x += nt) {
    const uint2 p = cand[x];
    const int w = (int)p.y / seg;
    if (p.x > T) atomicAdd(&gtc[w], 1);
    else if (p.x == T) atomicAdd(&eqc[w], 1);
  }
  if (tid == 0) sm[56] = n;
  __syncthreads();
  int eq_before = 0, kept_before = 0;
  for (int w = 0; w < warp; ++w) {
    const int e = eqc[w];
    kept_before += cgt[w] + gtc[w] + max(0, min(e, ntie - eq_before));
    eq_before += e;
  }
  int eq_run = eq_before, pos_run = kept_before, first_drop = n;
  for (int base = lo; base < hi; base += 32 * PF) {
    uint32_t u[PF];
#pragma unroll
    for (int e = 0; e < PF; ++e) {
      const int i = base + 32 * e + lane;
      u[e] = i < hi ? keys[i] : 0u;
    }
#pragma unroll
    for (int e = 0; e < PF; ++e) {
      const int i = base + 32 * e + lane;
      const bool valid = i < hi;
      const unsigned eqm = __ballot_sync(0xffffffffu, valid && u[e] == T);
      const bool keep = valid && (u[e] > T || (u[e] == T && eq_run + __popc(eqm & lt) < ntie));
      const unsigned km = __ballot_sync(0xffffffffu, keep);
      const unsigned dm = __ballot_sync(0xffffffffu, valid && !keep);
      const int pos = pos_run + __popc(km & lt);
      if (keep && pos < K) idx[pos] = i;
      if (dm != 0u && first_drop == n) first_drop = base + 32 * e + __ffs(dm) - 1;
      eq_run += __popc(eqm);
      pos_run += __popc(km);
    }
  }
  if (lane == 0 && first_drop < n) atomicMin(&sm[56], first_drop);
  __syncthreads();
  const int e0 = sm[56];
  __syncthreads();
  return e0;
}

// ---- long-unit selection in one pass over the raw scores
// A sample of kSampleKeys keys (every (N / kSampleKeys)-th slot) locates the
// B-th largest key to a range of 12-bit digits [d_lo, d_hi] (the sample ranks
// p ns -/+ (4 sqrt(ns p (1 - p)) + 4), p = B / N).  One pass over the raw
// scores then turns every key into its z/max key and sorts it three ways
// without storing it: digit > d_hi sets the key's bit in a kept bitmask in
// shared memory (8 lanes assemble a 32-slot word from their quads' nibbles);
// d_lo <= digit <= d_hi appends (key, slot) to a candidate list in the unit's
// (dead) key region; below d_lo nothing.  If the count above d_hi is below B
// and the candidates reach B, the threshold T is the (B - above)-th largest
// candidate (a 4 x 8-bit radix select over the candidates only); candidates
// above T set their bits, those equal to T mark a second bitmask, of which the
// first ntie in slot order join the kept set; a scan over the words writes
// the kept slots in ascending order.  Same result as the full passes (kept =
// keys > T, then the first ntie keys equal to T in slot order); the raw scores
// are read once and no key array is written.  Returns false, with no output
// written (only shared memory and the unit's key region touched), when the
// sample's range missed T or the candidates overflow: the caller then runs the
// full passes.
constexpr int kSampleKeys = 1024;
constexpr int kBmMaxKeys = 65536;   // bitmask words in shared memory: 2 x 8 KB

// Key i's G raw scores (key-major rows, 16-byte aligned for G >= 4).
template <int G>
__device__ __forceinline__ void load_key_scores(const float *raw_u, int i, float (&x)[G]) {
  const float *p = raw_u + (long long)i * G;
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int q = 0; q < G / 4; ++q) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(p) + q);
      x[4 * q] = v.x;
      x[4 * q + 1] = v.y;
      x[4 * q + 2] = v.z;
      x[4 * q + 3] = v.w;
    }
  } else if constexpr (G == 2) {
    const float2 v = __ldg(reinterpret_cast<const float2 *>(p));
    x[0] = v.x;
    x[1] = v.y;
  } else {
    x[0] = __ldg(p);
  }
}

template <int G>
__device__ __forceinline__ uint32_t zkey_from(const float (&x)[G], const float *mu, const float *iv) {
  float z = (x[0] - mu[0]) * iv[0];
#pragma unroll
  for (int h = 1; h < G; ++h) z = fmaxf(z, (x[h] - mu[h]) * iv[h]);
  return score_key(z);
}

// Digits of the (r0 + 1)-th and (r1 + 1)-th largest keys counted in hist[4096]
// (12-bit digits): thread t (blockDim 256) owns bins [4080 - 16 t, 4096 - 16 t).
__device__ __forceinline__ void pick12(const uint32_t *hist, int r0, int r1, int *sm, uint32_t &d0, uint32_t &d1) {
  const int tid = threadIdx.x;
  const int top = 4095 - 16 * tid;
  int cnt = 0;
#pragma unroll 4
  for (int b = 0; b < 16; ++b) cnt += (int)hist[top - b];
  int tot;
  const int before = block_excl_scan(cnt, sm, &tot);
  if (tid == 0) {
    sm[40] = 0;
    sm[41] = 0;
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int r = q == 0 ? r0 : r1;
    if (r >= before && r < before + cnt) {
      int run = before;
      for (int b = 0; b < 16; ++b) {
        run += (int)hist[top - b];
        if (run > r) {
          sm[40 + q] = top - b;
          break;
        }
      }
    }
  }
  __syncthreads();
  d0 = (uint32_t)sm[40];
  d1 = (uint32_t)sm[41];
  __syncthreads();
}

template <int G>
__device__ __noinline__ bool select_one_pass(const float *raw_u, int N, int B, const float *mom, uint32_t *hist,
                                             uint32_t *bm, uint32_t *eqm, int *sm, uint2 *cand, int cand_cap,
                                             int *idx, int *e0_out) {
  constexpr int U = G >= 8 ? 1 : 8 / G;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31;
  float mu[G], iv[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mu[h] = mom[h];
    iv[h] = mom[8 + h];
  }
  const int W = (N + 31) / 32, n4 = (N + 3) / 4;
  for (int b = tid; b < 4096; b += nt) hist[b] = 0;
  for (int w = tid; w < W; w += nt) {
    bm[w] = 0;
    eqm[w] = 0;
  }
  if (tid == 0) {
    sm[48] = 0;   // keys above d_hi
    sm[49] = 0;   // candidates
    sm[50] = 0;   // candidate overflow
  }
  __syncthreads();
  // the sample: every thread's keys loaded before any is used
  const int ns = min(kSampleKeys, N);
  {
    constexpr int SPT = kSampleKeys / kSelOnlyThreads;
    float x[SPT][G];
#pragma unroll
    for (int k = 0; k < SPT; ++k) {
      const int j = tid + k * nt;
      if (j < ns) load_key_scores<G>(raw_u, (int)(((long long)j * N) / ns), x[k]);
    }
#pragma unroll
    for (int k = 0; k < SPT; ++k)
      if (tid + k * nt < ns) atomicAdd(&hist[zkey_from<G>(x[k], mu, iv) >> 20], 1u);
  }
  __syncthreads();
  const float p = (float)B / (float)N;
  const float m = 4.0f * sqrtf((float)ns * p * (1.0f - p)) + 4.0f;
  const int r_hi = max(0, (int)floorf(p * ns - m)), r_lo = min(ns - 1, (int)ceilf(p * ns + m));
  uint32_t d_hi, d_lo;
  pick12(hist, r_hi, r_lo, sm, d_hi, d_lo);
  // the pass: warp-uniform loop over rounds of U quads per lane
  const float4 *rows = reinterpret_cast<const float4 *>(raw_u);
  for (int q0 = tid - lane; q0 < n4; q0 += nt * U) {
    float4 v[U][G];   // quads q = q0 + lane + k nt: the 4 G key-major scores of keys 4q .. 4q + 3
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int q = q0 + lane + k * nt;
#pragma unroll
      for (int h = 0; h < G; ++h)
        v[k][h] = q < n4 ? __ldg(rows + (long long)q * G + h) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int q = q0 + lane + k * nt;
      float x[4 * G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        x[4 * h] = v[k][h].x;
        x[4 * h + 1] = v[k][h].y;
        x[4 * h + 2] = v[k][h].z;
        x[4 * h + 3] = v[k][h].w;
      }
      uint32_t nib = 0, ck[4];
      int cc = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float z = (x[j * G] - mu[0]) * iv[0];
#pragma unroll
        for (int h = 1; h < G; ++h) z = fmaxf(z, (x[j * G + h] - mu[h]) * iv[h]);
        const uint32_t key = score_key(z), dg = key >> 20;
        const bool in = q < n4 && 4 * q + j < N;
        ck[j] = key;
        if (in && dg > d_hi) nib |= 1u << j;
        else if (in && dg >= d_lo) cc |= 1 << j;   // candidate mask
      }
      // the word of slots 32 (q >> 3) .. : 8 consecutive lanes' nibbles
      uint32_t word = nib << (4 * (lane & 7));
      word |= __shfl_xor_sync(0xffffffffu, word, 1);
      word |= __shfl_xor_sync(0xffffffffu, word, 2);
      word |= __shfl_xor_sync(0xffffffffu, word, 4);
      if ((lane & 7) == 0 && q < n4) bm[q >> 3] = word;
      const int na = __reduce_add_sync(0xffffffffu, __popc(nib));
      // candidates: one atomic per warp, positions by an inclusive scan of the lanes' counts
      const int nc = __popc((unsigned)cc);
      int incl = nc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int base = 0;
      if (lane == 31) {
        if (na) atomicAdd(&sm[48], na);
        base = incl > 0 ? atomicAdd(&sm[49], incl) : 0;
      }
      base = __shfl_sync(0xffffffffu, base, 31) + incl - nc;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (cc & (1 << j)) {
          if (base < cand_cap) cand[base] = make_uint2(ck[j], (uint32_t)(4 * q + j));
          else sm[50] = 1;
          ++base;
        }
    }
  }
  __syncthreads();
  const int above = sm[48], c = sm[49];
  const int k_in = B - above;
  if (sm[50] != 0 || k_in < 1 || k_in > c) {
    __syncthreads();
    return false;
  }
  // T: the k_in-th largest candidate (its top 8 bits are known when the
  // range's digits share them)
  const bool top_known = (d_lo >> 4) == (d_hi >> 4);
  uint32_t prefix = top_known ? (d_lo >> 4) << 24 : 0u, mask = top_known ? 0xff000000u : 0u;
  int k = k_in;
  for (int shift = top_known ? 16 : 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += nt) hist[b] = 0;
    __syncthreads();
    for (int x = tid; x < c; x += nt) {
      const uint32_t key = cand[x].x;
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    uint32_t dg;
    radix_pick(hist, k, sm, dg, k);
    prefix |= dg << shift;
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;
  const int ntie = k;
  for (int x = tid; x < c; x += nt) {
    const uint2 pr = cand[x];
    if (pr.x > T) atomicOr(&bm[pr.y >> 5], 1u << (pr.y & 31));
    else if (pr.x == T) atomicOr(&eqm[pr.y >> 5], 1u << (pr.y & 31));
  }
  if (tid == 0) sm[56] = N;
  __syncthreads();
  // the first ntie keys equal to T in slot order, then the kept slots in order;
  // thread t owns words [t wpt, (t + 1) wpt)
  const int wpt = (W + nt - 1) / nt, w0 = min(W, tid * wpt), w1 = min(W, w0 + wpt);
  int ce = 0;
  for (int w = w0; w < w1; ++w) ce += __popc(eqm[w]);
  int tot;
  int eb = block_excl_scan(ce, sm, &tot);
  int ck = 0, first_drop = N;
  for (int w = w0; w < w1; ++w) {
    uint32_t e = eqm[w], sel = 0;
    int allow = ntie - eb;
    eb += __popc(e);
    while (allow > 0 && e != 0u) {
      const uint32_t b = e & (0u - e);
      sel |= b;
      e ^= b;
      --allow;
    }
    const uint32_t kw = bm[w] | sel;
    bm[w] = kw;
    ck += __popc(kw);
    const uint32_t valid = (w == W - 1 && (N & 31)) ? ((1u << (N & 31)) - 1u) : 0xffffffffu;
    const uint32_t dropped = ~kw & valid;
    if (dropped != 0u && first_drop == N) first_drop = 32 * w + __ffs(dropped) - 1;
  }
  int kb = block_excl_scan(ck, sm, &tot);
  if (first_drop < N) atomicMin(&sm[56], first_drop);
  for (int w = w0; w < w1; ++w) {
    uint32_t kw = bm[w];
    while (kw != 0u) {
      const int b = __ffs(kw) - 1;
      kw &= kw - 1u;
      if (kb < B) idx[kb] = 32 * w + b;
      ++kb;
    }
  }
  __syncthreads();
  *e0_out = sm[56];
  __syncthreads();
  return true;
}

__device__ __forceinline__ bool select_one_pass_dispatch(const SCArgs &a, long long u, int N, const float *mom,
                                                         uint32_t *hist, uint32_t *bm, uint32_t *eqm, int *sm,
                                                         int *kept, int *e0) {
  const float *raw_u = a.raw + u * a.G * a.capp;
  uint2 *cand = reinterpret_cast<uint2 *>(a.keys + u * a.capp);   // the unit's key region, unused by this route
  const int cap = a.capp / 2;
  switch (a.G) {
    case 1: return select_one_pass<1>(raw_u, N, a.budget, mom, hist, bm, eqm, sm, cand, cap, kept, e0);
    case 2: return select_one_pass<2>(raw_u, N, a.budget, mom, hist, bm, eqm, sm, cand, cap, kept, e0);
    case 4: return select_one_pass<4>(raw_u, N, a.budget, mom, hist, bm, eqm, sm, cand, cap, kept, e0);
    default: return select_one_pass<8>(raw_u, N, a.budget, mom, hist, bm, eqm, sm, cand, cap, kept, e0);
  }
}

__global__ void __launch_bounds__(kSelOnlyThreads, 4) select_only_kernel(const __grid_constant__ SCArgs a) {
  __shared__ uint32_t hist[4096];
  __shared__ uint32_t bm[kBmMaxKeys / 32], eqm[kBmMaxKeys / 32];
  __shared__ int sm[kSelInts];
  __shared__ float mom[32];
  __shared__ int wc[3 * (kSelOnlyThreads / 32) + 1];
  const CacheView &c = a.c;
  const int tid = threadIdx.x, nt = blockDim.x;
  int u = blockIdx.x;
  if (a.order != nullptr) {   // CTA i takes the units of the (i / (L Hkv))-th longest sequence
    const int per = c.L * c.Hkv, rem = u % per;
    u = ((rem / c.Hkv) * c.S + a.order[u / per]) * c.Hkv + rem % c.Hkv;
  }
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  if (timed_out()) return;
  const int N = c.seq_len[s];
  const int B = a.budget;
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (N <= B) return;            // compact_only_kernel writes its outputs
  if (!c.blocks_ok(s, N)) {      // the sequence is skipped (status recorded by compact_only_kernel)
    return;
  }
  merge_tile_moments(a.part, u, a.ntiles, a.G, N, mom, a.part_keys);
  uint32_t *keys = a.keys + (long long)u * a.capp;
  int *kept = a.kept + (long long)u * B;
  if (!a.raw_km) {   // head-major raw scores (CUDA-core score kernel)
    __syncthreads();
    zmax_dispatch<false>(a, u, N, mom, keys);
    __syncthreads();   // the keys (global) are visible to the whole CTA
    int ntie;
    const uint32_t T = radix_select_gmem(keys, N, B, hist, sm, &ntie);
    const int e0 = build_kept_gmem(keys, N, B, T, ntie, kept, sm);
    if (tid == 0) a.e0s[u] = e0;
    return;
  }
  if (N <= kBmMaxKeys) {
    __syncthreads();
    int e0 = N;
    if (select_one_pass_dispatch(a, u, N, mom, hist, bm, eqm, sm, kept, &e0)) {
      if (tid == 0) a.e0s[u] = e0;
      return;
    }
  }
  for (int b = tid; b < 256; b += nt) hist[b] = 0;
  __syncthreads();
  zmax_km_hist_dispatch(a, u, N, mom, keys, hist);
  __syncthreads();   // the keys (global) and the first digit's histogram are complete
  uint32_t d1;
  int k1;
  radix_pick(hist, B, sm, d1, k1);
  const int c1 = (int)hist[d1];
  __syncthreads();
  // the unit's raw scores are dead: their G * capp floats hold the candidates
  uint2 *cand = reinterpret_cast<uint2 *>(const_cast<float *>(a.raw) + (long long)u * a.G * a.capp);
  int e0;
  if (8ll * c1 <= 4ll * a.G * a.capp) {
    e0 = select_rest_candidates(keys, N, d1, k1, cand, hist, sm, wc, kept, B);
  } else {
    int ntie;
    const uint32_t T = radix_select_gmem(keys, N, B, hist, sm, &ntie);
    e0 = build_kept_gmem(keys, N, B, T, ntie, kept, sm);
  }
  if (tid == 0) a.e0s[u] = e0;
}

struct CoLayout {
  int bars, sm, idx, total;
  __host__ __device__ explicit CoLayout(int bcap) {
    int o = kCoStages * kStageBytes;   // ring (also the hole-fill bookkeeping)
    bars = o; o += 2 * kCoStages * 8;
    sm = o;   o += kSelInts * 4;
    idx = o;  o += align_up(bcap * 4, 128);
    total = o;
  }
};

__global__ void __launch_bounds__(kCoThreads, 2) compact_only_kernel(const __grid_constant__ SCArgs a) {
  extern __shared__ __align__(1024) char smem[];
  const CoLayout lay(a.bcap);
  char *ring = smem;
  uint64_t *cbars = reinterpret_cast<uint64_t *>(smem + lay.bars);
  int *sm = reinterpret_cast<int *>(smem + lay.sm);
  int *idxs = reinterpret_cast<int *>(smem + lay.idx);
  const CacheView &c = a.c;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int u = blockIdx.x;
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  if (timed_out()) return;
  const int N = c.seq_len[s];
  const int B = a.budget;
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  // the new lengths and, for units with N <= B, the identity indices
  const bool len_writer = tid == 0 && a.new_len != nullptr && l == 0 && g == 0;
  if (N <= B) {
    if (len_writer) a.new_len[s] = N;
    if (a.idx_out != nullptr)
      for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = j < N ? j : -1;
    return;
  }
  if (!c.blocks_ok(s, N)) {   // the sequence is skipped: its length stays N
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    if (len_writer) a.new_len[s] = N;
    return;
  }
  if (len_writer) a.new_len[s] = B;
  if (tid == 0) {
    for (int st = 0; st < kCoStages; ++st) {
      mbar_init(&cbars[st], kCompactArrivals);               // K warp
      mbar_init(&cbars[kCoStages + st], kCompactArrivals);   // V warp
    }
    fence_mbar_init();
  }
  const int *kept = a.kept + (long long)u * B;
  for (int j = tid; j < B; j += nt) idxs[j] = kept[j];
  const int e0 = a.e0s[u];
  __syncthreads();
  if (a.holefill) {
    const int wb = align_up(holefill_work_bytes(B, N), 128);
    holefill_unit(c, l, s, g, idxs, B, N, ring + kCoStages * kStageBytes - wb, ring, kCoStages * kStageBytes - wb, sm,
                  a.idx_out != nullptr ? a.idx_out + (long long)u * B : nullptr);
    return;
  }
  if ((tid >> 5) < 2)
    compact_unit_tma(c, &a.maps, tid >> 5, l, s, g, idxs, e0, B, N, ring, kCoStages,
                     cbars + (tid >> 5) * kCoStages);
}

// ---------------------------------------------------------------- hole-fill moves
// Hole-fill compaction of every unit from its kept set, written by the
// selection earlier in the step: as the ascending kept list (select_only_kernel)
// or as a bitmask (the fused kernel), from which a scan of the words' counts
// builds the list in shared memory.  Layout: the kept slots below B stay; the r-th evicted slot below B (hole r)
// receives the r-th kept slot at or above B (mover r).  A slot finds its
// source without a scan: with P kept slots below B and kb of them below j
// (binary search in the list's head), slot j is kept iff list[kb] == j, else it
// is hole j - kb and receives list[P + j - kb].  Sources (>= B) and
// destinations (< B) are disjoint, so the row copies are independent: after
// the holes are ranked, each warp copies whole rows (lanes on the K pieces,
// then the V pieces), kHfBatch movers per lane batch with every load of the
// batch issued before its stores, and several CTAs share an SM.  Moving the
// rows here instead of at the end of the selecting CTA keeps that CTA's tail
// (a few row gathers at full latency) off the streaming kernel.
constexpr int kHfThreads = 256;
constexpr int kHfBatch = 4;

struct HfArgs {
  CacheView c;
  int budget;
  const int *kept;   // [units][B] ascending kept slots, or (from_bits) the kept bitmask in
                     // the first ceil(N / 32) words of the unit's row; may alias idx_out
  int from_bits;
  int *idx_out;      // [units][B] or null: the layout (original slot now at j)
  int *new_len;      // [S] or null
  int outputs;       // 1: also the lengths and the identity idx of units with N <= B
};

// Dynamic shared memory of holefill_apply_kernel: the list, then the holes.
__host__ __device__ __forceinline__ int hf_apply_smem(int B) { return 8 * B; }

__global__ void __launch_bounds__(kHfThreads, 4) holefill_apply_kernel(const __grid_constant__ HfArgs a) {
  extern __shared__ __align__(16) int hsm[];
  const CacheView &c = a.c;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int u = blockIdx.x;
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  if (timed_out()) return;   // a selection may have stopped before writing its list
  const int N = c.seq_len[s];
  const int B = a.budget;
  if (N < 0 || N > c.cap) {
    if (a.outputs && tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  const bool len_writer = a.outputs && tid == 0 && a.new_len != nullptr && l == 0 && g == 0;
  if (N <= B) {
    if (a.outputs) {
      if (len_writer) a.new_len[s] = N;
      if (a.idx_out != nullptr)
        for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = j < N ? j : -1;
    }
    return;
  }
  if (!c.blocks_ok(s, N)) {   // the sequence is skipped: its length stays N
    if (a.outputs) {
      if (tid == 0) set_status(TRI_ERR_BOUNDS);
      if (len_writer) a.new_len[s] = N;
    }
    return;
  }
  int *list = hsm, *holes = hsm + B;
  const int *src = a.kept + (long long)u * B;
  int bad = 0;
  if (a.from_bits) {   // the kept slots are the set bits, in order: a scan of the words' counts
    __shared__ int scan[32];
    const uint32_t *bits = reinterpret_cast<const uint32_t *>(src);
    const int W = (N + 31) / 32, wpt = (W + nt - 1) / nt;
    const int w0 = min(W, tid * wpt), w1 = min(W, w0 + wpt);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) {
      const uint32_t b = bits[w];
      cnt += __popc(b);
      if (w == W - 1 && (N & 31) != 0) bad |= (b >> (N & 31)) != 0u;   // no bit at or past N
    }
    int tot;
    int pos = block_excl_scan(cnt, scan, &tot);
    bad |= tot != B;
    for (int w = w0; w < w1; ++w) {
      uint32_t b = bits[w];
      while (b != 0u) {
        const int i = __ffs(b) - 1;
        b &= b - 1u;
        if (pos < B) list[pos] = 32 * w + i;
        ++pos;
      }
    }
  } else {
    for (int j = tid; j < B; j += nt) list[j] = src[j];
  }
  __syncthreads();
  for (int j = tid; j < B; j += nt) bad |= (list[j] < 0) | (list[j] >= N) | (j > 0 && list[j] <= list[j - 1]);
  if (__syncthreads_or(bad)) {   // every read of the list in global memory is done
    if (tid == 0) set_status(TRI_ERR_INVALID);
    if (len_writer) a.new_len[s] = N;
    return;
  }
  if (len_writer) a.new_len[s] = B;
  int lo = 0, hi = B;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (list[mid] < B) lo = mid + 1; else hi = mid;
  }
  const int P = lo, M = B - P;
  for (int j = tid; j < B; j += nt) {
    int kl = 0, kh = P;
    while (kl < kh) {
      const int mid = (kl + kh) >> 1;
      if (list[mid] < j) kl = mid + 1; else kh = mid;
    }
    const bool stays = kl < P && list[kl] == j;
    if (!stays) holes[j - kl] = j;
    if (a.idx_out != nullptr) a.idx_out[(long long)u * B + j] = stays ? j : list[P + j - kl];
  }
  __syncthreads();
  // mover r: row list[P + r] -> row holes[r], K then V; 16-byte pieces, lane
  // q (and q + 32) of the warp on piece q of the K and V rows together
  const int ppr = c.rb >> 4, pp = 2 * ppr;
  for (int r0 = warp * kHfBatch; r0 < M; r0 += nw * kHfBatch) {
    long long so[kHfBatch], dof[kHfBatch];
#pragma unroll
    for (int b = 0; b < kHfBatch; ++b) {
      const int r = r0 + b;
      so[b] = r < M ? c.row_off(l, s, g, list[P + r]) : -1;
      dof[b] = r < M ? c.row_off(l, s, g, holes[r]) : -1;
      if (dof[b] < 0) so[b] = -1;
    }
    for (int e = 0; 32 * e < pp; ++e) {   // one or two rounds of 16-byte pieces
      const int q = lane + 32 * e;
      const bool kq = q < ppr;
      const int col = (kq ? q : q - ppr) * 16;
      const bool in = q < pp;
      uint4 v[kHfBatch];
#pragma unroll
      for (int b = 0; b < kHfBatch; ++b)
        if (in && so[b] >= 0) v[b] = *reinterpret_cast<const uint4 *>((kq ? c.k : c.v) + so[b] + col);
#pragma unroll
      for (int b = 0; b < kHfBatch; ++b)
        if (in && so[b] >= 0) *reinterpret_cast<uint4 *>((kq ? c.k : c.v) + dof[b] + col) = v[b];
    }
  }
}

// ================================================================ host side
static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static tri_status check_cache(const tri_cache *c, bool need_k, bool need_v) {
  if (c == nullptr) return TRI_ERR_INVALID;
  if (c->L < 1 || c->S < 1 || c->Hkv < 1 || c->cap < 1 || c->seq_len == nullptr)
    return TRI_ERR_INVALID;
  if (c->d < 2 || (c->d & 1)) return TRI_ERR_INVALID;
  if (c->dtype != TRI_F32 && c->dtype != TRI_BF16) return TRI_ERR_INVALID;
  if (c->d != 64 && c->d != 128) return TRI_ERR_UNSUPPORTED;
  if (c->cap > (1ll << 30)) return TRI_ERR_UNSUPPORTED;
  if (need_k && (c->k == nullptr || !aligned16(c->k))) return TRI_ERR_INVALID;
  if (need_v && (c->v == nullptr || !aligned16(c->v))) return TRI_ERR_INVALID;
  if (c->block_table != nullptr) {
    if (c->block < 1 || c->max_blocks < 1 || c->nblocks < 1) return TRI_ERR_INVALID;
    if ((int64_t)c->max_blocks * c->block != c->cap) return TRI_ERR_INVALID;
  }
  return TRI_OK;
}

static tri_status check_stats(const tri_cache *c, const tri_stats *st) {
  if (st == nullptr || st->center == nullptr || st->R == nullptr || st->mag == nullptr)
    return TRI_ERR_INVALID;
  if (st->Hq < 1 || st->Hq % c->Hkv != 0) return TRI_ERR_INVALID;
  const int G = st->Hq / c->Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return TRI_ERR_UNSUPPORTED;
  return TRI_OK;
}

static tri_status check_params(const tri_params *p) {
  if (p == nullptr || p->t == nullptr || p->offsets == nullptr || p->n_offsets < 1) return TRI_ERR_INVALID;
  if (!(p->theta > 0.0) || !std::isfinite(p->theta)) return TRI_ERR_INVALID;
  if (p->pairing != TRI_PAIR_HALF && p->pairing != TRI_PAIR_INTERLEAVED) return TRI_ERR_INVALID;
  if (p->budget < 1) return TRI_ERR_INVALID;
  for (int i = 0; i < p->n_offsets; ++i)
    if (p->offsets[i] < 0) return TRI_ERR_INVALID;
  return TRI_OK;
}

static CacheView make_view(const tri_cache *c) {
  CacheView v;
  v.k = static_cast<char *>(c->k);
  v.v = static_cast<char *>(c->v);
  v.L = c->L;
  v.S = c->S;
  v.Hkv = c->Hkv;
  v.d = c->d;
  v.rb = c->d * (c->dtype == TRI_BF16 ? 2 : 4);
  v.cap = c->cap;
  v.seq_len = c->seq_len;
  v.bt = c->block_table;
  v.max_blocks = c->block_table ? c->max_blocks : 0;
  v.block = c->block_table ? c->block : 1;
  v.nblocks = c->block_table ? c->nblocks : 0;
  v.tm_ok = 0;
  v.g4_ok = 0;
  return v;
}

// cuTensorMapEncodeTiled from the driver, looked up once (no link against libcuda).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Tensor map over a paged pool [L][nblocks][block][Hkv][d] whose box is one
// block of one head ({d, 1, block, 1}), for the per-stage K loads and the
// per-block compaction stores.  Used only when a score stage holds a whole
// number of blocks (at most 32 of them); returns false otherwise or if encoding
// fails (per-row copies are used instead).
static bool make_block_map(const tri_cache *c, void *base, CUtensorMap *map) {
  if (c->block_table == nullptr) return false;
  const int es = c->dtype == TRI_BF16 ? 2 : 4;
  const int rb = c->d * es;
  const int tr = kStageBytes / rb;
  if (c->block > 256 || tr % c->block != 0 || tr / c->block > 32) return false;
  if ((int64_t)c->L * c->nblocks >= (1ll << 31)) return false;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)c->d, (cuuint64_t)c->Hkv, (cuuint64_t)c->block,
                              (cuuint64_t)c->L * (cuuint64_t)c->nblocks};
  const cuuint64_t strides[3] = {(cuuint64_t)rb, (cuuint64_t)c->Hkv * rb, (cuuint64_t)c->block * c->Hkv * rb};
  const cuuint32_t box[4] = {(cuuint32_t)c->d, 1u, (cuuint32_t)c->block, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = enc(map, c->dtype == TRI_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                         4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map viewing the K or V storage as rows [rows][d] (dense: L*S*Hkv*cap
// rows; paged: L*nblocks*block*Hkv pool rows) with a box of one row, for the
// tile::gather4 loads of the compaction.  Row coordinates are int32, so the
// view must have fewer than 2^31 rows; returns false otherwise or on failure.
static bool make_row_map(const tri_cache *c, void *base, CUtensorMap *map) {
  const int es = c->dtype == TRI_BF16 ? 2 : 4;
  const int rb = c->d * es;
  const int64_t rows = c->block_table == nullptr ? (int64_t)c->L * c->S * c->Hkv * c->cap
                                                 : (int64_t)c->L * c->nblocks * c->block * c->Hkv;
  if (rows < 1 || rows >= (1ll << 31)) return false;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)c->d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)rb};
  const cuuint32_t box[2] = {(cuuint32_t)c->d, 1u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(map, c->dtype == TRI_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                         2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 128B-swizzled map of K or V (`base`) for the tensor-core kernels (bf16, d in
// {64, 128}): dense, a 2-D view [rows][d] with boxes of 64 elements x one
// stage of rows; paged, the 4-D pool view with boxes of 64 elements x one block
// of one head (a stage must hold a whole number of blocks, at most 32).
// heads: KV heads per box (paged d = 128 only): 1, or every head of a block.
static bool make_sw_map(const tri_cache *c, void *base, CUtensorMap *map, int heads = 1) {
  if (c->dtype != TRI_BF16 || (c->d != 64 && c->d != 128)) return false;
  const int rb = c->d * 2, tr = kStageBytes / rb;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr || base == nullptr) return false;
  CUresult r;
  if (c->block_table == nullptr) {
    if (heads != 1) return false;
    const int64_t rows = (int64_t)c->L * c->S * c->Hkv * c->cap;
    if (rows >= (1ll << 31)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)c->d, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)rb};
    const cuuint32_t box[2] = {64u, (cuuint32_t)tr};
    const cuuint32_t estr[2] = {1u, 1u};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else if (c->d == 128) {
    // 5-D view (64 elements, block rows, halves, heads, blocks) with a box of
    // one block of `heads` heads, both halves: smem [head][half][block rows][128 B]
    if (c->block > 256 || c->block % 8 != 0 || tr % c->block != 0 || tr / c->block > 32) return false;
    if (heads != 1 && heads != c->Hkv) return false;
    if ((int64_t)c->L * c->nblocks >= (1ll << 31)) return false;
    const cuuint64_t dims[5] = {64u, (cuuint64_t)c->block, 2u, (cuuint64_t)c->Hkv,
                                (cuuint64_t)c->L * (cuuint64_t)c->nblocks};
    const cuuint64_t strides[4] = {(cuuint64_t)c->Hkv * rb, 128u, (cuuint64_t)rb,
                                   (cuuint64_t)c->block * c->Hkv * rb};
    const cuuint32_t box[5] = {64u, (cuuint32_t)c->block, 2u, (cuuint32_t)heads, 1u};
    const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    if (heads != 1) return false;
    if (c->block > 256 || tr % c->block != 0 || tr / c->block > 32) return false;
    if ((int64_t)c->L * c->nblocks >= (1ll << 31)) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)c->d, (cuuint64_t)c->Hkv, (cuuint64_t)c->block,
                                (cuuint64_t)c->L * (cuuint64_t)c->nblocks};
    const cuuint64_t strides[3] = {(cuuint64_t)rb, (cuuint64_t)c->Hkv * rb, (cuuint64_t)c->block * c->Hkv * rb};
    const cuuint32_t box[4] = {64u, 1u, (cuuint32_t)c->block, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS;
}

// The score kernels' K map: bf16 caches with rotate-half bands only.
static bool make_swizzled_map(const tri_cache *c, const tri_params *p, CUtensorMap *map) {
  return p->pairing == TRI_PAIR_HALF && make_sw_map(c, c->k, map);
}

// Builds the tensor maps of a call and sets the view's flags.  K and V maps
// are made together; a V map is needed only when V is given (compaction).
static void make_maps(const tri_cache *c, CacheView *v, TmaMaps *m) {
  std::memset(m, 0, sizeof(*m));
  v->tm_ok = make_block_map(c, c->k, &m->k4) && (c->v == nullptr || make_block_map(c, c->v, &m->v4));
  v->g4_ok = c->k != nullptr && c->v != nullptr && make_row_map(c, c->k, &m->k2) && make_row_map(c, c->v, &m->v2);
}

static StepConst make_const(const tri_params *p, int d) {
  StepConst sc;
  std::memset(&sc, 0, sizeof(sc));
  const int F = d / 2;
  for (int f = 0; f < F; ++f) {
    const double om = std::pow(p->theta, -2.0 * f / (double)d);
    double re = 0, im = 0;
    for (int i = 0; i < p->n_offsets; ++i) {
      re += std::cos(om * (double)p->offsets[i]);
      im += std::sin(om * (double)p->offsets[i]);
    }
    sc.omega[f] = om;
    sc.phi[f] = make_float2((float)(re / p->n_offsets), (float)(im / p->n_offsets));
  }
  return sc;
}

static int round32(int64_t x) { return (int)((x + 31) / 32 * 32); }
static int64_t units_of(const tri_cache *c) { return (int64_t)c->L * c->S * c->Hkv; }
static int ntiles_of(const tri_cache *c, int G) {
  return (int)((c->cap + tile_keys_for(G) - 1) / tile_keys_for(G));
}
static bool fused_fits(const tri_cache *c, int G) {
  return FusedLayout(G, c->d / 2, round32(c->cap)).total <= kMaxSmem;
}

struct SplitWs {
  size_t raw_off, part_off, phase_off, keys_off, kept_off, e0_off, order_off, plan_off, total;
};
static SplitWs split_ws(const tri_cache *c, int G, int budget) {
  SplitWs w;
  // raw rows padded to round32(cap) floats: 16-byte aligned for bulk copies
  const size_t raw = (size_t)units_of(c) * G * (size_t)round32(c->cap) * sizeof(float);
  const size_t part = (size_t)units_of(c) * ntiles_of(c, G) * G * sizeof(float2);
  const size_t phase = (size_t)c->S * (c->d / 2) * sizeof(float2);
  w.raw_off = 0;
  w.part_off = (raw + 255) / 256 * 256;
  const size_t keys = (size_t)units_of(c) * (size_t)round32(c->cap) * sizeof(uint32_t);
  w.phase_off = w.part_off + (part + 255) / 256 * 256;
  w.keys_off = w.phase_off + (phase + 255) / 256 * 256;
  // kept slots and first dropped slot per unit (select_only -> compact_only)
  const size_t kept = (size_t)units_of(c) * (size_t)std::max(budget, 1) * sizeof(int);
  const size_t e0 = (size_t)units_of(c) * sizeof(int);
  w.kept_off = w.keys_off + (keys + 255) / 256 * 256;
  w.e0_off = w.kept_off + (kept + 255) / 256 * 256;
  w.order_off = w.e0_off + (e0 + 255) / 256 * 256;   // sequences by length (S ints)
  w.plan_off = w.order_off + ((size_t)c->S * sizeof(int) + 255) / 256 * 256;   // chunk plan (2 S + 2 ints)
  w.total = w.plan_off + ((size_t)(2 * c->S + 2) * sizeof(int) + 255) / 256 * 256;
  return w;
}

static tri_status launch_result() {
  return cudaGetLastError() == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

// Fills the workspace's step phases (before the tile kernels).
static tri_status run_phases(const tri_cache *c, const TileArgs &ta, cudaStream_t st) {
  phase_kernel<<<(unsigned)c->S, 64, 0, st>>>(ta.t, c->d / 2, const_cast<float2 *>(ta.phase), ta.sc, c->seq_len,
                                               (int)c->S, ta.order, ta.plan, ta.budget, (long long)c->cap, kHgKeys);
  return launch_result();
}

template <typename K>
static tri_status set_smem(K kernel, int bytes) {
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return TRI_ERR_CUDA;
  return TRI_OK;
}

// Hole-fill rows are moved after the selection, by holefill_apply_kernel, when
// a unit's list and holes (8 B bytes) fit 56 KB of shared memory (four CTAs
// per SM at least); else the selecting kernel moves them itself.
constexpr int kHfMaxSmem = 57344;
static bool hf_apply_ok(int B) { return hf_apply_smem(B) <= kHfMaxSmem; }

static tri_status run_holefill_apply(const CacheView &view, int B, const int *kept, int from_bits, int32_t *idx_out,
                                     int32_t *new_len, int outputs, int64_t units, cudaStream_t st) {
  HfArgs h;
  std::memset(&h, 0, sizeof(h));
  h.c = view;
  h.budget = B;
  h.kept = kept;
  h.from_bits = from_bits;
  h.idx_out = idx_out;
  h.new_len = new_len;
  h.outputs = outputs;
  const int bytes = hf_apply_smem(B);
  if (set_smem(holefill_apply_kernel, bytes) != TRI_OK) return TRI_ERR_CUDA;
  holefill_apply_kernel<<<(unsigned)units, kHfThreads, bytes, st>>>(h);
  return launch_result();
}

template <int D, int G, bool BF16>
static tri_status run_fused(const FusedArgs &a, int64_t units, cudaStream_t st) {
  const FusedLayout lay(G, D / 2, a.capp);
  if constexpr (BF16) {
    if (a.mma_ok) {
      FusedMmaArgs m;
      std::memset(&m, 0, sizeof(m));
      m.f = a;
      if (a.cache->block_table != nullptr && a.mode == 0) make_maps(a.cache, &m.f.c, &m.maps);
      if (make_swizzled_map(a.cache, a.params, &m.ks)) {
        auto k = m.f.c.bt != nullptr && m.f.c.tm_ok ? fused_mma_kernel<D, G, true> : fused_mma_kernel<D, G, false>;
        if (set_smem(k, lay.total) != TRI_OK) return TRI_ERR_CUDA;
        k<<<(unsigned)units, kThreads, lay.total, st>>>(m);
        return launch_result();
      }
    }
  }
  auto k = fused_kernel<D, G, BF16>;
  if (set_smem(k, lay.total) != TRI_OK) return TRI_ERR_CUDA;
  k<<<(unsigned)units, kFusedThreads, lay.total, st>>>(a);
  return launch_result();
}

template <int D, int G, bool BF16>
static tri_status run_tiles(const TileArgs &a, int64_t units, cudaStream_t st) {
  const TileLayout lay(G, D / 2);
  if constexpr (BF16) {
    if (a.mma_ok) {
      auto k = score_tiles_mma_kernel<D, G>;
      if (set_smem(k, lay.total) != TRI_OK) return TRI_ERR_CUDA;
      const unsigned ctas = (unsigned)((a.ntiles + kTilesPerCta - 1) / kTilesPerCta);
      k<<<dim3(ctas, (unsigned)units), kThreads, lay.total, st>>>(a);
      return launch_result();
    }
  }
  auto k = score_tiles_kernel<D, G, BF16>;
  if (set_smem(k, lay.total) != TRI_OK) return TRI_ERR_CUDA;
  k<<<dim3((unsigned)a.ntiles, (unsigned)units), kThreads, lay.total, st>>>(a);
  return launch_result();
}

// The compress step's long-unit scores: the key-major tensor-core kernel for
// bf16 rotate-half caches (one part entry per CTA of kKmCtaKeys keys), else
// the CUDA-core tile kernel (head-major, one entry per tile).
template <int D, int G, bool BF16>
static tri_status run_keys(const TileArgs &a, int64_t units, cudaStream_t st) {
  if constexpr (BF16 && D == 128) {
    if (a.mma_ok && a.hg) {
      const HgLayout lay(G, D / 2, a.c.Hkv);
      auto k = score_heads_mma_kernel<G>;
      if (set_smem(k, lay.total) != TRI_OK) return TRI_ERR_CUDA;
      const dim3 grid = a.plan != nullptr ? dim3((unsigned)((long long)a.c.L * a.c.S * a.ntiles))
                                          : dim3((unsigned)a.ntiles, (unsigned)(a.c.L * a.c.S));
      k<<<grid, kHgThreads, lay.total, st>>>(a);
      return launch_result();
    }
  }
  if constexpr (BF16) {
    if (a.mma_ok) {
      const KmLayout lay(G, D / 2);
      auto k = score_keys_mma_kernel<D, G>;
      if (set_smem(k, lay.total) != TRI_OK) return TRI_ERR_CUDA;
      k<<<dim3((unsigned)a.ntiles, (unsigned)units), kThreads, lay.total, st>>>(a);
      return launch_result();
    }
  }
  TileArgs b = a;
  b.mma_ok = 0;
  return run_tiles<D, G, BF16>(b, units, st);
}

// Expands a call over the supported (head dim, group size, dtype) instantiations.
#define TRI_DISPATCH(FN, D, G, BF16, ...)                                   \
  [&]() -> tri_status {                                                     \
    switch ((D) * 100 + (G) * 10 + ((BF16) ? 1 : 0)) {                      \
      case 6410: return FN<64, 1, false>(__VA_ARGS__);                      \
      case 6411: return FN<64, 1, true>(__VA_ARGS__);                       \
      case 6420: return FN<64, 2, false>(__VA_ARGS__);                      \
      case 6421: return FN<64, 2, true>(__VA_ARGS__);                       \
      case 6440: return FN<64, 4, false>(__VA_ARGS__);                      \
      case 6441: return FN<64, 4, true>(__VA_ARGS__);                       \
      case 6480: return FN<64, 8, false>(__VA_ARGS__);                      \
      case 6481: return FN<64, 8, true>(__VA_ARGS__);                       \
      case 12810: return FN<128, 1, false>(__VA_ARGS__);                    \
      case 12811: return FN<128, 1, true>(__VA_ARGS__);                     \
      case 12820: return FN<128, 2, false>(__VA_ARGS__);                    \
      case 12821: return FN<128, 2, true>(__VA_ARGS__);                     \
      case 12840: return FN<128, 4, false>(__VA_ARGS__);                    \
      case 12841: return FN<128, 4, true>(__VA_ARGS__);                     \
      case 12880: return FN<128, 8, false>(__VA_ARGS__);                    \
      case 12881: return FN<128, 8, true>(__VA_ARGS__);                     \
      default: return TRI_ERR_UNSUPPORTED;                                  \
    }                                                                       \
  }()

static tri_status run_select_compact(const SCArgs &a, int64_t units, cudaStream_t st) {
  const SCLayout lay(a.capp, a.bcap);
  if (lay.total > kMaxSmem) return TRI_ERR_UNSUPPORTED;
  if (set_smem(select_compact_kernel, lay.total) != TRI_OK) return TRI_ERR_CUDA;
  select_compact_kernel<<<(unsigned)units, kSelThreads, lay.total, st>>>(a);
  return launch_result();
}

static FusedArgs fused_args(const tri_cache *c, const tri_stats *stt, const tri_params *p) {
  FusedArgs a;
  std::memset(&a, 0, sizeof(a));
  a.c = make_view(c);
  a.center = stt->center;
  a.R = stt->R;
  a.mag = stt->mag;
  a.Hq = stt->Hq;
  a.t = p->t;
  a.budget = p->budget;
  a.inter = p->pairing == TRI_PAIR_INTERLEAVED;
  a.capp = round32(c->cap);
  a.sc = make_const(p, c->d);
  a.mma_ok = kFusedMma;
  a.cache = c;
  a.params = p;
  return a;
}

static TileArgs tile_args(const tri_cache *c, const tri_stats *stt, const tri_params *p) {
  TileArgs a;
  std::memset(&a, 0, sizeof(a));
  a.c = make_view(c);
  a.center = stt->center;
  a.R = stt->R;
  a.mag = stt->mag;
  a.Hq = stt->Hq;
  a.t = p->t;
  a.budget = p->budget;
  a.inter = p->pairing == TRI_PAIR_INTERLEAVED;
  a.ntiles = ntiles_of(c, stt->Hq / c->Hkv);
  a.sc = make_const(p, c->d);
  make_maps(c, &a.c, &a.maps);
  a.mma_ok = make_swizzled_map(c, p, &a.ks) ? 1 : 0;
  return a;
}

static int bcap_of(const tri_cache *c, int budget) {
  return round32(budget < c->cap ? budget : c->cap);
}

// ---------------------------------------------------------------- calibration streaming, curves
template <int D, bool BF16, bool INTER>
static tri_status run_calib_acc(const char *q, long long n, long long ss, long long ls, int L, int H,
                                double *acc, cudaStream_t st) {
  constexpr long long kMaxZ = 65535;
  const int es = BF16 ? 2 : 4;
  for (long long i0 = 0; i0 < n; i0 += kMaxZ * kCalibChunk) {
    const long long m = std::min(n - i0, kMaxZ * kCalibChunk);
    const unsigned z = (unsigned)((m + kCalibChunk - 1) / kCalibChunk);
    calib_accumulate_kernel<D, BF16, INTER><<<dim3((unsigned)H, (unsigned)L, z), kCalibThreads, 0, st>>>(
        q + i0 * ss * es, m, ss, ls, H, acc);
    if (cudaGetLastError() != cudaSuccess) return TRI_ERR_CUDA;
  }
  return TRI_OK;
}

template <int D, bool BF16, bool INTER>
static tri_status run_logit_curve(const void *q, const void *k, long long n, int L, int Hq, int Hkv, int n_delta,
                                  const StepConst &sc, float *curve, cudaStream_t st) {
  const unsigned gx = (unsigned)((n_delta + kCurveDeltas - 1) / kCurveDeltas);
  logit_curve_kernel<D, BF16, INTER><<<dim3(gx, (unsigned)Hq, (unsigned)L), kCurveThreads, 0, st>>>(
      q, k, n, Hq, Hkv, n_delta, sc, curve);
  return launch_result();
}

// Phase-only constants (omega_f; Phi unused) for the curve kernels.
static StepConst omega_const(double theta, int d) {
  StepConst sc;
  std::memset(&sc, 0, sizeof(sc));
  for (int f = 0; f < d / 2; ++f) sc.omega[f] = std::pow(theta, -2.0 * f / (double)d);
  return sc;
}

__global__ void __launch_bounds__(32) wait_check_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  // nothing arrives on the barrier: its phase 0 never completes and the wait
  // gives up after limit_ns (nothing is in flight)
  if (threadIdx.x == 0) mbar_wait_for(&bar, 0, limit_ns);
}

// ---------------------------------------------------------------- decode loop
// Slices per unit for the decode attention: enough CTAs for two waves of two
// per SM, slices of at most 8192 keys, at least one stage of rows each.
static int decode_splits(const tri_cache *c) {
  const int tr = kStageBytes / (2 * c->d);
  const int64_t units = units_of(c);
  int64_t n = std::max<int64_t>((2 * 148 * 2 + units - 1) / units, (c->cap + 8191) / 8192);
  n = std::min<int64_t>(n, (c->cap + tr - 1) / tr);
  return (int)std::max<int64_t>(1, std::min<int64_t>(n, 65535));
}

template <int D, int G>
static tri_status run_decode(const DecodeArgs &a, int64_t units, cudaStream_t st) {
  const DecLayout lay(G, D);
  auto k = decode_attn_kernel<D, G>;
  if (set_smem(k, lay.total) != TRI_OK) return TRI_ERR_CUDA;
  k<<<dim3((unsigned)a.nsplit, (unsigned)units), kDecThreads, lay.total, st>>>(a);
  tri_status e = launch_result();
  if (e != TRI_OK || a.nsplit == 1) return e;
  decode_merge_kernel<<<(unsigned)units, 256, 0, st>>>(a.part, a.nsplit, G, D, a.c.S, a.c.Hkv, a.Hq, a.out);
  return launch_result();
}

// ---------------------------------------------------------------- built-in scratch
// Scratch of tri_compress_step_static_scratch, for callers that cannot
// allocate.  In host code `g_static_scratch` names a host-side stand-in, not
// the device array: its device address is looked up per device below.
static __device__ __align__(256) unsigned char g_static_scratch[TRI_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
static std::mutex g_static_mu;
static void *g_static_addr[kMaxDevices];
static CUcontext g_static_ctx[kMaxDevices];

// cuCtxGetCurrent from the driver, looked up once (no link against libcuda).
static PFN_cuCtxGetCurrent_v4000 ctx_getter() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  return fn;
}

// Device address of g_static_scratch on the current device, looked up with
// that device current and cached together with the context that was current
// then.  A call under another context (after a device reset, or a context the
// caller made current) looks the address up again: a cached address belongs to
// the context it was taken in.
static tri_status static_scratch_addr(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TRI_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TRI_ERR_UNSUPPORTED;
  PFN_cuCtxGetCurrent_v4000 get = ctx_getter();
  if (get == nullptr) return TRI_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return TRI_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (ctx == nullptr || g_static_addr[dev] == nullptr || g_static_ctx[dev] != ctx) {
    // the lookup also binds the runtime's context for this device when none
    // is current yet; the context is read again after it
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return TRI_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return TRI_ERR_CUDA;
    g_static_addr[dev] = p;
    g_static_ctx[dev] = ctx;
  }
  *out = g_static_addr[dev];
  return TRI_OK;
}

}  // namespace tri

using namespace tri;

// ================================================================ C ABI
extern "C" {

int tri_version(void) { return 100; }

const char *tri_status_string(tri_status s) {
  switch (s) {
    case TRI_OK: return "ok";
    case TRI_ERR_INVALID: return "invalid argument";
    case TRI_ERR_CUDA: return "CUDA runtime error";
    case TRI_ERR_UNSUPPORTED: return "unsupported shape or option";
    case TRI_ERR_WORKSPACE: return "workspace missing or too small";
    case TRI_ERR_TIMEOUT: return "device wait timed out";
    case TRI_ERR_BOUNDS: return "device-side index check failed";
  }
  return "unknown status";
}

tri_status tri_calibrate_stats(const void *q_pre, tri_dtype dtype, int64_t n, int L, int Hq, int d,
                               tri_pairing pairing, float *center, float *R, float *mag,
                               cudaStream_t stream) {
  if (q_pre == nullptr || center == nullptr || R == nullptr || mag == nullptr) return TRI_ERR_INVALID;
  if (n < 1 || L < 1 || Hq < 1) return TRI_ERR_INVALID;
  if (dtype != TRI_F32 && dtype != TRI_BF16) return TRI_ERR_INVALID;
  if (pairing != TRI_PAIR_HALF && pairing != TRI_PAIR_INTERLEAVED) return TRI_ERR_INVALID;
  if (d != 64 && d != 128) return TRI_ERR_INVALID;
  calib_kernel<<<dim3((unsigned)Hq, (unsigned)L), 256, 0, stream>>>(
      q_pre, dtype == TRI_BF16, n, Hq, d, pairing == TRI_PAIR_INTERLEAVED, center, R, mag);
  return launch_result();
}

tri_status tri_workspace_bytes(const tri_cache *cache, const tri_stats *stats,
                               const tri_params *params, size_t *bytes) {
  if (bytes == nullptr) return TRI_ERR_INVALID;
  tri_status e;
  if ((e = check_cache(cache, false, false)) != TRI_OK) return e;
  if ((e = check_stats(cache, stats)) != TRI_OK) return e;
  if ((e = check_params(params)) != TRI_OK) return e;
  const int G = stats->Hq / cache->Hkv;
  *bytes = fused_fits(cache, G) ? 0 : split_ws(cache, G, params->budget).total;
  return TRI_OK;
}

tri_status tri_score(const tri_cache *cache, const tri_stats *stats, const tri_params *params,
                     float *agg, float *raw, void *ws, size_t ws_bytes, cudaStream_t stream) {
  tri_status e;
  if ((e = check_cache(cache, true, false)) != TRI_OK) return e;
  if ((e = check_stats(cache, stats)) != TRI_OK) return e;
  if ((e = check_params(params)) != TRI_OK) return e;
  if (agg == nullptr) return TRI_ERR_INVALID;
  const int G = stats->Hq / cache->Hkv;
  const bool bf16 = cache->dtype == TRI_BF16;
  const int64_t units = units_of(cache);
  if (fused_fits(cache, G)) {
    FusedArgs a = fused_args(cache, stats, params);
    a.mode = 1;
    a.agg = agg;
    a.raw = raw;
    return TRI_DISPATCH(run_fused, cache->d, G, bf16, a, units, stream);
  }
  const SplitWs w = split_ws(cache, G, params->budget);
  if (ws == nullptr || ws_bytes < w.total || !aligned16(ws)) return TRI_ERR_WORKSPACE;
  TileArgs ta = tile_args(cache, stats, params);
  ta.skip_small = 0;
  ta.raw = raw != nullptr ? raw : reinterpret_cast<float *>(static_cast<char *>(ws) + w.raw_off);
  ta.raw_stride = raw != nullptr ? cache->cap : round32(cache->cap);
  ta.part = reinterpret_cast<float2 *>(static_cast<char *>(ws) + w.part_off);
  ta.phase = reinterpret_cast<const float2 *>(static_cast<char *>(ws) + w.phase_off);
  if ((e = run_phases(cache, ta, stream)) != TRI_OK) return e;
  if ((e = TRI_DISPATCH(run_tiles, cache->d, G, bf16, ta, units, stream)) != TRI_OK) return e;
  ZArgs z;
  z.S = cache->S;
  z.Hkv = cache->Hkv;
  z.G = G;
  z.ntiles = ta.ntiles;
  z.cap = cache->cap;
  z.raw_stride = ta.raw_stride;
  z.seq_len = cache->seq_len;
  z.raw = ta.raw;
  z.part = ta.part;
  z.agg = agg;
  zmax_kernel<<<dim3((unsigned)ta.ntiles, (unsigned)units), 256, 0, stream>>>(z);
  return launch_result();
}

tri_status tri_select_topb(const tri_cache *cache, const float *agg, int budget, int32_t *idx,
                           void *ws, size_t ws_bytes, cudaStream_t stream) {
  (void)ws;
  (void)ws_bytes;
  tri_status e;
  if ((e = check_cache(cache, false, false)) != TRI_OK) return e;
  if (agg == nullptr || idx == nullptr || budget < 1) return TRI_ERR_INVALID;
  SCArgs a;
  std::memset(&a, 0, sizeof(a));
  a.c = make_view(cache);
  a.budget = budget;
  a.mode = 1;
  a.capp = round32(cache->cap);
  a.bcap = bcap_of(cache, budget);
  a.agg = agg;
  a.idx_out = idx;
  return run_select_compact(a, units_of(cache), stream);
}

tri_status tri_compact_kv(const tri_cache *cache, const int32_t *idx, int budget,
                          tri_compact_mode mode, int32_t *new_len, cudaStream_t stream) {
  tri_status e;
  if ((e = check_cache(cache, true, true)) != TRI_OK) return e;
  if (idx == nullptr || budget < 1) return TRI_ERR_INVALID;
  if (mode != TRI_COMPACT_ORDERED && mode != TRI_COMPACT_HOLEFILL) return TRI_ERR_UNSUPPORTED;
  if (new_len != nullptr && new_len == cache->seq_len) return TRI_ERR_INVALID;
  SCArgs a;
  std::memset(&a, 0, sizeof(a));
  a.c = make_view(cache);
  make_maps(cache, &a.c, &a.maps);
  a.budget = budget;
  a.mode = 2;
  a.holefill = mode == TRI_COMPACT_HOLEFILL;
  a.capp = a.holefill ? round32(cache->cap) : 0;   // hole-fill bookkeeping: < 4 N bytes in the keys region
  a.bcap = bcap_of(cache, budget);
  a.idx_in = idx;
  a.new_len = new_len;
  return run_select_compact(a, units_of(cache), stream);
}

tri_status tri_compress_step(const tri_cache *cache, const tri_stats *stats,
                             const tri_params *params, tri_compact_mode mode, int32_t *idx_out,
                             int32_t *new_len, void *ws, size_t ws_bytes, cudaStream_t stream) {
  tri_status e;
  if ((e = check_cache(cache, true, true)) != TRI_OK) return e;
  if ((e = check_stats(cache, stats)) != TRI_OK) return e;
  if ((e = check_params(params)) != TRI_OK) return e;
  if (mode != TRI_COMPACT_ORDERED && mode != TRI_COMPACT_HOLEFILL) return TRI_ERR_UNSUPPORTED;
  if (new_len != nullptr && new_len == cache->seq_len) return TRI_ERR_INVALID;
  const int G = stats->Hq / cache->Hkv;
  const bool bf16 = cache->dtype == TRI_BF16;
  const int64_t units = units_of(cache);
  if (fused_fits(cache, G)) {
    FusedArgs a = fused_args(cache, stats, params);
    a.mode = 0;
    a.holefill = mode == TRI_COMPACT_HOLEFILL;
    // hole-fill: the fused kernel selects and writes the kept set to idx_out as a
    // bitmask (ceil(cap / 32) <= B words), holefill_apply_kernel turns it into
    // the layout and moves the rows
    a.defer = a.holefill && idx_out != nullptr && hf_apply_ok(params->budget) &&
              (cache->cap + 31) / 32 <= params->budget;
    a.idx_out = idx_out;
    a.new_len = new_len;
    if ((e = TRI_DISPATCH(run_fused, cache->d, G, bf16, a, units, stream)) != TRI_OK || !a.defer) return e;
    return run_holefill_apply(a.c, params->budget, idx_out, 1, idx_out, new_len, 0, units, stream);
  }
  const SplitWs w = split_ws(cache, G, params->budget);
  if (ws == nullptr || ws_bytes < w.total || !aligned16(ws)) return TRI_ERR_WORKSPACE;
  SCArgs sa;
  std::memset(&sa, 0, sizeof(sa));
  sa.c = make_view(cache);
  make_maps(cache, &sa.c, &sa.maps);
  sa.G = G;
  sa.budget = params->budget;
  sa.mode = 0;
  sa.holefill = mode == TRI_COMPACT_HOLEFILL;
  sa.ntiles = ntiles_of(cache, G);
  sa.capp = round32(cache->cap);
  sa.bcap = bcap_of(cache, params->budget);
  if (SCLayout(sa.capp, sa.bcap).total > kMaxSmem) return TRI_ERR_UNSUPPORTED;
  TileArgs ta = tile_args(cache, stats, params);
  ta.skip_small = 1;
  ta.raw = reinterpret_cast<float *>(static_cast<char *>(ws) + w.raw_off);
  ta.raw_stride = sa.capp;
  ta.part = reinterpret_cast<float2 *>(static_cast<char *>(ws) + w.part_off);
  ta.phase = reinterpret_cast<const float2 *>(static_cast<char *>(ws) + w.phase_off);
  // paged d = 128 caches whose block holds 128 head-rows: every KV head of a
  // block in one copy (score_heads_mma_kernel)
  ta.hg = ta.mma_ok && cache->block_table != nullptr && cache->d == 128 && cache->Hkv * cache->block == 128 &&
          cache->block % 16 == 0 && (int64_t)cache->L * cache->S <= 65535 &&
          HgLayout(G, cache->d / 2, cache->Hkv).total <= kMaxSmem && make_sw_map(cache, cache->k, &ta.ks, cache->Hkv);
  if (ta.mma_ok && !ta.hg) ta.mma_ok = make_swizzled_map(cache, params, &ta.ks) ? 1 : 0;   // (the per-head map again)
  if (ta.hg) {
    ta.ntiles = (int)((cache->cap + kHgKeys - 1) / kHgKeys);
    sa.raw_km = 1;
    sa.part_keys = kHgKeys;
  } else if (ta.mma_ok) {   // key-major raw scores, one moment entry per CTA
    ta.ntiles = (int)((cache->cap + kKmCtaKeys - 1) / kKmCtaKeys);
    sa.raw_km = 1;
    sa.part_keys = kKmCtaKeys;
  } else {
    sa.raw_km = 0;
    sa.part_keys = tile_keys_for(G);
  }
  sa.ntiles = ta.ntiles;
  sa.raw = ta.raw;
  sa.part = ta.part;
  sa.idx_out = idx_out;
  sa.new_len = new_len;
  char *wsb = static_cast<char *>(ws);
  sa.keys = reinterpret_cast<uint32_t *>(wsb + w.keys_off);
  // selection, then compaction (two kernels), when the compaction's ring holds
  // the hole-fill bookkeeping (B bytes + 4 min(B, N - B)) with room to stage
  // rows and its shared memory the kept list; else the one-per-SM kernel with
  // keys in shared memory.
  const CoLayout co(sa.bcap);
  const int64_t movers = std::min<int64_t>(params->budget, cache->cap - params->budget);
  // hole-fill: the bookkeeping sits at the end of the ring, and at least 16 KB
  // stays for staging the moved rows
  const bool hf_fits = !sa.holefill || align_up(params->budget + 16 + 4 * (int)std::max<int64_t>(movers, 0), 128) +
                                               16384 <= kCoStages * kStageBytes;
  // hole-fill with holefill_apply_kernel after the selection: the kept list
  // goes to idx_out (rewritten there as the layout) or the workspace
  const bool apply = sa.holefill && hf_apply_ok(params->budget);
  const bool split = co.total <= kMaxSmem && (apply || hf_fits);
  if (split) {
    sa.kept = ((!sa.holefill || apply) && idx_out != nullptr) ? idx_out : reinterpret_cast<int *>(wsb + w.kept_off);
    sa.e0s = reinterpret_cast<int *>(wsb + w.e0_off);
    // longest sequences first in the selection (ranked by phase_kernel; the
    // ranking costs S per sequence, so only for S up to 4096)
    if (cache->S <= 4096) {
      ta.order = reinterpret_cast<int *>(wsb + w.order_off);
      sa.order = ta.order;
      if (ta.hg && (long long)cache->L * cache->S * ta.ntiles < (1ll << 31))
        ta.plan = reinterpret_cast<int *>(wsb + w.plan_off);
    }
  }
  if ((e = run_phases(cache, ta, stream)) != TRI_OK) return e;
  if ((e = TRI_DISPATCH(run_keys, cache->d, G, bf16, ta, units, stream)) != TRI_OK) return e;
  if (!split) return run_select_compact(sa, units, stream);
  select_only_kernel<<<(unsigned)units, kSelOnlyThreads, 0, stream>>>(sa);
  if ((e = launch_result()) != TRI_OK) return e;
  if (apply) return run_holefill_apply(sa.c, params->budget, sa.kept, 0, idx_out, new_len, 1, units, stream);
  if (set_smem(compact_only_kernel, co.total) != TRI_OK) return TRI_ERR_CUDA;
  compact_only_kernel<<<(unsigned)units, kCoThreads, co.total, stream>>>(sa);
  return launch_result();
}

tri_status tri_compress_step_static_scratch(const tri_cache *cache, const tri_stats *stats,
                                            const tri_params *params, tri_compact_mode mode,
                                            int32_t *idx_out, int32_t *new_len,
                                            cudaStream_t stream) {
  tri_status e;
  if ((e = check_cache(cache, true, true)) != TRI_OK) return e;
  if (mode != TRI_COMPACT_ORDERED && mode != TRI_COMPACT_HOLEFILL) return TRI_ERR_UNSUPPORTED;
  size_t need = 0;
  if ((e = tri_workspace_bytes(cache, stats, params, &need)) != TRI_OK) return e;
  if (need == 0) return tri_compress_step(cache, stats, params, mode, idx_out, new_len, nullptr, 0, stream);
  if (need > (size_t)TRI_STATIC_SCRATCH_BYTES) return TRI_ERR_WORKSPACE;
  void *ws = nullptr;
  if ((e = static_scratch_addr(&ws)) != TRI_OK) return e;
  return tri_compress_step(cache, stats, params, mode, idx_out, new_len, ws,
                           (size_t)TRI_STATIC_SCRATCH_BYTES, stream);
}

static tri_status check_calib_shape(int L, int H, int d) {
  if (L < 1 || H < 1) return TRI_ERR_INVALID;
  if (d != 64 && d != 128) return TRI_ERR_INVALID;
  return TRI_OK;
}
static long long calib_doubles(int L, int H, int d) { return (long long)L * H * (d / 2) * kCalibAcc; }
static unsigned grid_for(long long count) {
  return (unsigned)std::max<long long>(1, std::min<long long>((count + 255) / 256, 148 * 8));
}

tri_status tri_calib_reset(double *acc, int L, int H, int d, cudaStream_t stream) {
  tri_status e;
  if ((e = check_calib_shape(L, H, d)) != TRI_OK) return e;
  if (acc == nullptr || (reinterpret_cast<uintptr_t>(acc) & 7u)) return TRI_ERR_INVALID;
  const long long cnt = calib_doubles(L, H, d);
  calib_zero_kernel<<<grid_for(cnt), 256, 0, stream>>>(acc, cnt);
  return launch_result();
}

tri_status tri_calib_accumulate(const void *q, tri_dtype dtype, int64_t n, int L, int H, int d,
                                tri_pairing pairing, int64_t sample_stride, int64_t layer_stride, double *acc,
                                cudaStream_t stream) {
  tri_status e;
  if ((e = check_calib_shape(L, H, d)) != TRI_OK) return e;
  if (acc == nullptr || (reinterpret_cast<uintptr_t>(acc) & 7u)) return TRI_ERR_INVALID;
  if (n < 0 || sample_stride < 0 || layer_stride < 0) return TRI_ERR_INVALID;
  if (dtype != TRI_F32 && dtype != TRI_BF16) return TRI_ERR_INVALID;
  if (pairing != TRI_PAIR_HALF && pairing != TRI_PAIR_INTERLEAVED) return TRI_ERR_INVALID;
  const long long ss = sample_stride ? sample_stride : (long long)H * d;
  const long long ls = layer_stride ? layer_stride : n * ss;
  if (ss < (long long)H * d || (ss & 3) || (ls & 3)) return TRI_ERR_INVALID;
  if (H > 65535 || L > 65535) return TRI_ERR_UNSUPPORTED;
  if (n == 0) return TRI_OK;   // nothing is read (q may be NULL)
  if (q == nullptr || !aligned16(q)) return TRI_ERR_INVALID;
  const char *qc = static_cast<const char *>(q);
  const bool bf = dtype == TRI_BF16, in = pairing == TRI_PAIR_INTERLEAVED;
  switch ((d == 128 ? 4 : 0) + (bf ? 2 : 0) + (in ? 1 : 0)) {
    case 0: return run_calib_acc<64, false, false>(qc, n, ss, ls, L, H, acc, stream);
    case 1: return run_calib_acc<64, false, true>(qc, n, ss, ls, L, H, acc, stream);
    case 2: return run_calib_acc<64, true, false>(qc, n, ss, ls, L, H, acc, stream);
    case 3: return run_calib_acc<64, true, true>(qc, n, ss, ls, L, H, acc, stream);
    case 4: return run_calib_acc<128, false, false>(qc, n, ss, ls, L, H, acc, stream);
    case 5: return run_calib_acc<128, false, true>(qc, n, ss, ls, L, H, acc, stream);
    case 6: return run_calib_acc<128, true, false>(qc, n, ss, ls, L, H, acc, stream);
    default: return run_calib_acc<128, true, true>(qc, n, ss, ls, L, H, acc, stream);
  }
}

tri_status tri_calib_merge(double *acc, const double *other, int L, int H, int d, cudaStream_t stream) {
  tri_status e;
  if ((e = check_calib_shape(L, H, d)) != TRI_OK) return e;
  if (acc == nullptr || other == nullptr || acc == other) return TRI_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(acc) & 7u) || (reinterpret_cast<uintptr_t>(other) & 7u)) return TRI_ERR_INVALID;
  const long long cnt = calib_doubles(L, H, d);
  calib_add_kernel<<<grid_for(cnt), 256, 0, stream>>>(acc, other, cnt);
  return launch_result();
}

tri_status tri_calib_finalize(const double *acc, int L, int H, int d, float *center, float *R, float *mag,
                              cudaStream_t stream) {
  tri_status e;
  if ((e = check_calib_shape(L, H, d)) != TRI_OK) return e;
  if (acc == nullptr || center == nullptr || R == nullptr || mag == nullptr) return TRI_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(acc) & 7u) return TRI_ERR_INVALID;
  const long long bands = (long long)L * H * (d / 2);
  calib_finalize_kernel<<<grid_for(bands), 256, 0, stream>>>(acc, bands, center, R, mag);
  return launch_result();
}

tri_status tri_distance_curves(const float *q_center, const float *k_center, const void *q_seq, const void *k_seq,
                               tri_dtype dtype, int64_t n, int L, int Hq, int Hkv, int d, double theta,
                               tri_pairing pairing, int n_delta, float *center_curve, float *logit_curve,
                               float *corr, cudaStream_t stream) {
  if (L < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return TRI_ERR_INVALID;
  if (d != 64 && d != 128) return TRI_ERR_INVALID;
  if (!(theta > 0.0) || !std::isfinite(theta)) return TRI_ERR_INVALID;
  if (dtype != TRI_F32 && dtype != TRI_BF16) return TRI_ERR_INVALID;
  if (pairing != TRI_PAIR_HALF && pairing != TRI_PAIR_INTERLEAVED) return TRI_ERR_INVALID;
  if (n_delta < 1 || q_center == nullptr || k_center == nullptr || center_curve == nullptr) return TRI_ERR_INVALID;
  const bool want_logit = logit_curve != nullptr || corr != nullptr;
  if (want_logit && (q_seq == nullptr || k_seq == nullptr || logit_curve == nullptr)) return TRI_ERR_INVALID;
  if (want_logit && (n < 1 || n_delta > n)) return TRI_ERR_INVALID;
  if (Hq > 65535 || L > 65535) return TRI_ERR_UNSUPPORTED;
  const StepConst sc = omega_const(theta, d);
  center_curve_kernel<<<dim3((unsigned)Hq, (unsigned)L), 256, 0, stream>>>(q_center, k_center, Hq, Hkv, d / 2,
                                                                            n_delta, sc, center_curve);
  tri_status e;
  if ((e = launch_result()) != TRI_OK) return e;
  if (!want_logit) return TRI_OK;
  const bool bf = dtype == TRI_BF16, in = pairing == TRI_PAIR_INTERLEAVED;
  switch ((d == 128 ? 4 : 0) + (bf ? 2 : 0) + (in ? 1 : 0)) {
    case 0: e = run_logit_curve<64, false, false>(q_seq, k_seq, n, L, Hq, Hkv, n_delta, sc, logit_curve, stream); break;
    case 1: e = run_logit_curve<64, false, true>(q_seq, k_seq, n, L, Hq, Hkv, n_delta, sc, logit_curve, stream); break;
    case 2: e = run_logit_curve<64, true, false>(q_seq, k_seq, n, L, Hq, Hkv, n_delta, sc, logit_curve, stream); break;
    case 3: e = run_logit_curve<64, true, true>(q_seq, k_seq, n, L, Hq, Hkv, n_delta, sc, logit_curve, stream); break;
    case 4: e = run_logit_curve<128, false, false>(q_seq, k_seq, n, L, Hq, Hkv, n_delta, sc, logit_curve, stream); break;
    case 5: e = run_logit_curve<128, false, true>(q_seq, k_seq, n, L, Hq, Hkv, n_delta, sc, logit_curve, stream); break;
    case 6: e = run_logit_curve<128, true, false>(q_seq, k_seq, n, L, Hq, Hkv, n_delta, sc, logit_curve, stream); break;
    default: e = run_logit_curve<128, true, true>(q_seq, k_seq, n, L, Hq, Hkv, n_delta, sc, logit_curve, stream); break;
  }
  if (e != TRI_OK || corr == nullptr) return e;
  curve_corr_kernel<<<(unsigned)((long long)L * Hq), 256, 0, stream>>>(center_curve, logit_curve, n_delta, corr);
  return launch_result();
}

tri_status tri_append_kv(const tri_cache *cache, const void *k_new, const void *v_new, const int32_t *pos,
                         double theta, tri_pairing pairing, int32_t *seq_len_out, int32_t *pos_out,
                         cudaStream_t stream) {
  tri_status e;
  if ((e = check_cache(cache, true, true)) != TRI_OK) return e;
  if (k_new == nullptr || v_new == nullptr || pos == nullptr || seq_len_out == nullptr) return TRI_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new)) return TRI_ERR_INVALID;
  if (seq_len_out == cache->seq_len || pos_out == pos || (pos_out != nullptr && pos_out == cache->seq_len) ||
      reinterpret_cast<const void *>(seq_len_out) == reinterpret_cast<const void *>(pos))
    return TRI_ERR_INVALID;
  if (!(theta > 0.0) || !std::isfinite(theta)) return TRI_ERR_INVALID;
  if (pairing != TRI_PAIR_HALF && pairing != TRI_PAIR_INTERLEAVED) return TRI_ERR_INVALID;
  AppendArgs a;
  std::memset(&a, 0, sizeof(a));
  a.c = make_view(cache);
  a.k_new = k_new;
  a.v_new = v_new;
  a.pos = pos;
  a.seq_len_out = seq_len_out;
  a.pos_out = pos_out;
  a.inter = pairing == TRI_PAIR_INTERLEAVED;
  a.sc = omega_const(theta, cache->d);
  const unsigned units = (unsigned)units_of(cache);
  if (cache->dtype == TRI_BF16)
    append_kv_kernel<true><<<units, 32, 0, stream>>>(a);
  else
    append_kv_kernel<false><<<units, 32, 0, stream>>>(a);
  return launch_result();
}

tri_status tri_decode_workspace_bytes(const tri_cache *cache, int Hq, size_t *bytes) {
  if (bytes == nullptr) return TRI_ERR_INVALID;
  tri_status e;
  if ((e = check_cache(cache, false, false)) != TRI_OK) return e;
  if (Hq < 1 || Hq % cache->Hkv != 0) return TRI_ERR_INVALID;
  const int G = Hq / cache->Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return TRI_ERR_UNSUPPORTED;
  const int ns = decode_splits(cache);
  *bytes = ns == 1 ? 0 : (size_t)units_of(cache) * ns * G * (cache->d + 2) * sizeof(float);
  return TRI_OK;
}

tri_status tri_decode_attention(const tri_cache *cache, const void *q, int Hq, const int32_t *pos, double theta,
                                tri_pairing pairing, float scale, float *out, void *ws, size_t ws_bytes,
                                cudaStream_t stream) {
  tri_status e;
  if ((e = check_cache(cache, true, true)) != TRI_OK) return e;
  if (q == nullptr || pos == nullptr || out == nullptr) return TRI_ERR_INVALID;
  if (!(theta > 0.0) || !std::isfinite(theta) || !(scale > 0.f) || !std::isfinite(scale)) return TRI_ERR_INVALID;
  if (pairing != TRI_PAIR_HALF && pairing != TRI_PAIR_INTERLEAVED) return TRI_ERR_INVALID;
  size_t need = 0;
  if ((e = tri_decode_workspace_bytes(cache, Hq, &need)) != TRI_OK) return e;
  if (cache->dtype != TRI_BF16) return TRI_ERR_UNSUPPORTED;
  if (need > 0 && (ws == nullptr || ws_bytes < need || !aligned16(ws))) return TRI_ERR_WORKSPACE;
  DecodeArgs a;
  std::memset(&a, 0, sizeof(a));
  a.c = make_view(cache);
  if (!make_sw_map(cache, cache->k, &a.kmap) || !make_sw_map(cache, cache->v, &a.vmap)) return TRI_ERR_UNSUPPORTED;
  a.q = q;
  a.pos = pos;
  a.Hq = Hq;
  a.nsplit = decode_splits(cache);
  a.inter = pairing == TRI_PAIR_INTERLEAVED;
  a.qscale = scale * 1.4426950408889634f;
  a.out = out;
  a.part = static_cast<float *>(ws);
  a.sc = omega_const(theta, cache->d);
  const int G = Hq / cache->Hkv;
  const int64_t units = units_of(cache);
  switch (cache->d * 10 + G) {
    case 641: return run_decode<64, 1>(a, units, stream);
    case 642: return run_decode<64, 2>(a, units, stream);
    case 644: return run_decode<64, 4>(a, units, stream);
    case 648: return run_decode<64, 8>(a, units, stream);
    case 1281: return run_decode<128, 1>(a, units, stream);
    case 1282: return run_decode<128, 2>(a, units, stream);
    case 1284: return run_decode<128, 4>(a, units, stream);
    default: return run_decode<128, 8>(a, units, stream);
  }
}

tri_status tri_check_bounded_wait(uint32_t limit_us, cudaStream_t stream) {
  if (limit_us < 1 || limit_us > 1000000u) return TRI_ERR_INVALID;
  wait_check_kernel<<<1, 32, 0, stream>>>((unsigned long long)limit_us * 1000ull);
  return launch_result();
}

tri_status tri_get_device_status(cudaStream_t stream, int32_t *out) {
  if (out == nullptr) return TRI_ERR_INVALID;
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_tri_status, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return TRI_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return TRI_ERR_CUDA;
  *out = v;
  return TRI_OK;
}

tri_status tri_clear_device_status(cudaStream_t stream) {
  static const int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_tri_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) !=
          cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_tri_timeout, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) !=
          cudaSuccess)
    return TRI_ERR_CUDA;
  return TRI_OK;
}

}  // extern "C"
