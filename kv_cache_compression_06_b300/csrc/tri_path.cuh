// Device building blocks of the compression step: cache addressing, per-unit
// weight preparation, key scoring from a shared-memory tile, GQA z/max, radix
// top-B selection, and in-place ordered compaction.
//
// Method source: "实现单卡4090跑通OpenClaw!英伟达&浙大等提出长上下文推理KV压缩新方法TriAttention"
// (yeyulingfeng.com), section 主要方法 — trig-series paragraph (RoPE logit as a
// sum over bands of a function of the distance), two-part score paragraph (trig
// score + concentration-weighted norm score), pruning paragraph (geometric future
// offsets averaged; top-B every 128 tokens; GQA per-head z-score then max).
#pragma once

#include "tri_device.cuh"

namespace tri {

// Per-call constants: omega_f = theta^(-2f/d) (fp64) and
// Phi_f = mean_{o in O} e^{i*omega_f*o} (computed in fp64 on the host, stored fp32).
struct StepConst {
  double omega[64];
  float2 phi[64];
};

// Tensor maps of one call (kernel parameters, valid per the CacheView flags):
// k4/v4 view a paged pool as [L*nblocks][block][Hkv][d] with a box of one block
// of one head; k2/v2 view the K/V storage as rows [rows][d] with a box of one row
// (for tile::gather4).
struct TmaMaps {
  CUtensorMap k4, v4, k2, v2;
};

// Dense [L][S][Hkv][cap][d] or paged [L][nblocks][block][Hkv][d] addressing.
struct CacheView {
  char *k;
  char *v;
  int L, S, Hkv, d, rb;   // rb = bytes per row
  long long cap;
  const int *seq_len;
  const int *bt;          // block table [S][max_blocks] or nullptr
  int max_blocks, block;
  long long nblocks;
  int tm_ok;              // paged, and the block maps (box = one block of one head) are valid
  int g4_ok;              // the row maps (2-D [rows][d], box one row) are valid

  __host__ __device__ __forceinline__ bool paged() const { return bt != nullptr; }
  // Byte offset of slot i of unit (l, s, g); -1 if the block id is out of range.
  __device__ __forceinline__ long long row_off(int l, int s, int g, int i) const {
    if (bt == nullptr) return ((((long long)l * S + s) * Hkv + g) * cap + i) * (long long)rb;
    const int b = bt[(long long)s * max_blocks + i / block];
    if (b < 0 || b >= nblocks) return -1;
    return ((((long long)l * nblocks + b) * block + (i % block)) * Hkv + g) * (long long)rb;
  }
  // Row of slot i of unit (l, s, g) in the 2-D row view [rows][d] of the K/V
  // storage (dense: u*cap + i; paged: pool row); -1 if the block id is out of range.
  __device__ __forceinline__ long long row2d(int l, int s, int g, int i) const {
    if (bt == nullptr) return (((long long)l * S + s) * Hkv + g) * cap + i;
    const int b = bt[(long long)s * max_blocks + i / block];
    if (b < 0 || b >= nblocks) return -1;
    return (((long long)l * nblocks + b) * block + (i % block)) * Hkv + g;
  }
  // Checks every block id that rows [row0, row0 + n) of sequence s touch
  // (CTA-wide; every thread gets the answer).
  __device__ bool blocks_ok(int s, int n, int row0 = 0) const {
    if (bt == nullptr) return true;
    const int b0 = row0 / block, nb = (row0 + n + block - 1) / block;
    int bad = 0;
    for (int b = b0 + threadIdx.x; b < nb; b += blockDim.x) {
      const int id = bt[(long long)s * max_blocks + b];
      bad |= (id < 0 || id >= nblocks);
    }
    return __syncthreads_or(bad) == 0;
  }
};

// ---------------------------------------------------------------- weights (a1)
// Phase factor of band f for a step at position t: e^{i*omega_f*t} * Phi_f.
// The phase omega_f*t is reduced modulo 2*pi in fp64 (two-term 2*pi split)
// before an fp32 sincos: omega_0*t reaches ~3e4 rad, far beyond fp32 phase
// accuracy.
// e^{i*ph} for a phase given in fp64: ph is reduced modulo 2*pi in fp64 (two-term
// 2*pi split) before an fp32 sincos.  Returns (cos, sin).
__device__ __forceinline__ float2 reduced_cis(double ph) {
  constexpr double kTwoPiHi = 6.283185307179586232;
  constexpr double kTwoPiLo = 2.449293598294706e-16;
  constexpr double kInvTwoPi = 0.15915494309189535;
  const double q = rint(ph * kInvTwoPi);
  double r = fma(-q, kTwoPiHi, ph);
  r = fma(-q, kTwoPiLo, r);
  float sn, cs;
  sincosf((float)r, &sn, &cs);
  return make_float2(cs, sn);
}

__device__ __forceinline__ float2 step_phase(const StepConst &sc, int f, int t) {
  const float2 e = reduced_cis(sc.omega[f] * (double)t);
  const float2 p = sc.phi[f];
  return make_float2(e.x * p.x - e.y * p.y, e.x * p.y + e.y * p.x);
}

// wts layout [G][3][F]: Re A, Im A, W for the G query heads of KV head g.
// A_{h,f} = c_{h,f} * E_f with E_f the step phase of band f (computed here, or
// taken from `phase` [F] when given); W_{h,f} = (1 - R_{h,f}) * m_{h,f}.
// Threads [0, nthr) of the block take part (default: all).
template <int G, int F>
__device__ __forceinline__ void build_weights(float *wts, const float *center, const float *R,
                                              const float *mag, int Hq, int l, int g, int t,
                                              const StepConst &sc, const float2 *phase = nullptr,
                                              int nthr = 0) {
  const int n = nthr > 0 ? nthr : (int)blockDim.x;
  if ((int)threadIdx.x >= n) return;
  for (int x = threadIdx.x; x < G * F; x += n) {
    const int h = x / F, f = x - h * F;
    const long long o = ((long long)l * Hq + (long long)g * G + h) * F + f;
    const float2 e = phase != nullptr ? phase[f] : step_phase(sc, f, t);
    const float cr = center[2 * o], ci = center[2 * o + 1];
    wts[(h * 3 + 0) * F + f] = cr * e.x - ci * e.y;
    wts[(h * 3 + 1) * F + f] = cr * e.y + ci * e.x;
    wts[(h * 3 + 2) * F + f] = (1.0f - R[o]) * mag[o];
  }
}

// ---------------------------------------------------------------- scoring (a2)
// One row (key) is handled by LPR = F/4 lanes, each owning 4 consecutive bands.
template <int D, bool BF16>
struct RowGeom {
  static constexpr int F = D / 2;
  static constexpr int LPR = F / 4;
  static constexpr int RPW = 32 / LPR;
  static constexpr int ES = BF16 ? 2 : 4;
  static constexpr int RB = D * ES;
};

// The 4 bands a lane owns, as packed pairs: re01 = (re_0, re_1), re23, im01, im23.
struct LaneBands {
  uint64_t re01, re23, im01, im23;
};

// Loads the 4 bands of this lane (bands 4j..4j+3) from a row in shared memory.
template <int D, bool BF16>
__device__ __forceinline__ LaneBands load_bands(const char *row, int j, bool inter) {
  constexpr int F = D / 2;
  LaneBands x;
  if constexpr (BF16) {
    if (!inter) {
      // rotate-half: re = elements 4j..4j+3, im = elements F+4j..F+4j+3
      const uint2 lo = *reinterpret_cast<const uint2 *>(row + 2 * (4 * j));
      const uint2 hi = *reinterpret_cast<const uint2 *>(row + 2 * (F + 4 * j));
      x.re01 = pk(bf16lo(lo.x), bf16hi(lo.x));
      x.re23 = pk(bf16lo(lo.y), bf16hi(lo.y));
      x.im01 = pk(bf16lo(hi.x), bf16hi(hi.x));
      x.im23 = pk(bf16lo(hi.y), bf16hi(hi.y));
    } else {
      // interleaved: band b = elements (2b, 2b+1) -> one 32-bit word per band
      const uint4 w = *reinterpret_cast<const uint4 *>(row + 2 * (8 * j));
      x.re01 = pk(bf16lo(w.x), bf16lo(w.y));
      x.re23 = pk(bf16lo(w.z), bf16lo(w.w));
      x.im01 = pk(bf16hi(w.x), bf16hi(w.y));
      x.im23 = pk(bf16hi(w.z), bf16hi(w.w));
    }
  } else {
    if (!inter) {
      const float4 lo = *reinterpret_cast<const float4 *>(row + 4 * (4 * j));
      const float4 hi = *reinterpret_cast<const float4 *>(row + 4 * (F + 4 * j));
      x.re01 = pk(lo.x, lo.y);
      x.re23 = pk(lo.z, lo.w);
      x.im01 = pk(hi.x, hi.y);
      x.im23 = pk(hi.z, hi.w);
    } else {
      const float4 a = *reinterpret_cast<const float4 *>(row + 4 * (8 * j));
      const float4 b = *reinterpret_cast<const float4 *>(row + 4 * (8 * j + 4));
      x.re01 = pk(a.x, a.z);
      x.re23 = pk(b.x, b.z);
      x.im01 = pk(a.y, a.w);
      x.im23 = pk(b.y, b.w);
    }
  }
  return x;
}

// Sums v[0..G) across the LPR lanes of a row group.  The first log2(G) levels
// reduce-scatter (each level halves the values a lane keeps), the rest
// all-reduce; lane j of the group ends with the full sum of head j / (LPR/G).
template <int G, int LPR>
__device__ __forceinline__ float group_reduce(float (&v)[G], int lane) {
  int m = LPR / 2;
#pragma unroll
  for (int n = G; n > 1; n >>= 1) {
    const int half = n / 2;
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = up ? v[k] : v[k + half];
      const float keep = up ? v[k + half] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
    m >>= 1;
  }
  float x = v[0];
#pragma unroll
  for (; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

// Lane-private weights of the 4 bands a lane owns, for each of the G heads, as
// packed pairs over bands (4j, 4j+1) and (4j+2, 4j+3).
template <int G>
struct LaneWeights {
  uint64_t ar01[G], ar23[G], ai01[G], ai23[G], w01[G], w23[G];
};

template <int G, int F>
__device__ __forceinline__ void load_lane_weights(LaneWeights<G> &lw, const float *wts, int j) {
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float4 ar = *reinterpret_cast<const float4 *>(wts + (h * 3 + 0) * F + 4 * j);
    const float4 ai = *reinterpret_cast<const float4 *>(wts + (h * 3 + 1) * F + 4 * j);
    const float4 w = *reinterpret_cast<const float4 *>(wts + (h * 3 + 2) * F + 4 * j);
    lw.ar01[h] = pk(ar.x, ar.y);
    lw.ar23[h] = pk(ar.z, ar.w);
    lw.ai01[h] = pk(ai.x, ai.y);
    lw.ai23[h] = pk(ai.z, ai.w);
    lw.w01[h] = pk(w.x, w.y);
    lw.w23[h] = pk(w.z, w.w);
  }
}

// Scores the rows [0, nrows) of a tile in shared memory; s_{h, row0 + r} goes to
// scores[h * sstride + row0 + r].  Per lane and head: 6 paired FMAs over its 4
// bands (Re A * Re k~ + Im A * Im k~ + W * |k~|), then a cross-lane sum.  Called
// by the `nw` consumer warps; `warp` is this warp's index among them.
template <int D, int G, bool BF16>
__device__ __forceinline__ void score_tile(const char *tile, int nrows, int row0, float *scores,
                                           int sstride, const LaneWeights<G> &lw, bool inter, int warp,
                                           int nw) {
  using RG = RowGeom<D, BF16>;
  constexpr int LPR = RG::LPR, RPW = RG::RPW, RB = RG::RB;
  const int lane = threadIdx.x & 31;
  const int j = lane % LPR;
  const int rsub = lane / LPR;
  const int head = j / (LPR / G);
  const bool writer = (j % (LPR / G)) == 0;
  for (int rb = 0; rb < nrows; rb += nw * RPW) {
    const int r = rb + warp * RPW + rsub;
    const bool valid = r < nrows;
    LaneBands x;
    if (valid) {
      x = load_bands<D, BF16>(tile + (long long)r * RB, j, inter);
    } else {
      x.re01 = x.re23 = x.im01 = x.im23 = 0ull;
    }
    uint64_t mg01, mg23;
    {
      float a, b, c, e;
      upk(ffma2(x.im01, x.im01, fmul2(x.re01, x.re01)), a, b);
      upk(ffma2(x.im23, x.im23, fmul2(x.re23, x.re23)), c, e);
      mg01 = pk(sqrt_approx(a), sqrt_approx(b));
      mg23 = pk(sqrt_approx(c), sqrt_approx(e));
    }
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      uint64_t t = fmul2(lw.ar01[h], x.re01);
      t = ffma2(lw.ar23[h], x.re23, t);
      t = ffma2(lw.ai01[h], x.im01, t);
      t = ffma2(lw.ai23[h], x.im23, t);
      t = ffma2(lw.w01[h], mg01, t);
      t = ffma2(lw.w23[h], mg23, t);
      float lo, hi;
      upk(t, lo, hi);
      acc[h] = lo + hi;
    }
    const float s = group_reduce<G, LPR>(acc, lane);
    if (valid && writer) scores[head * sstride + row0 + r] = s;
  }
}

// ---------------------------------------------------------------- K streaming (short units)
// Issues the copy of rows [row0, row0 + nrows) of one unit's K into `dst` on
// `bar` (arrival count 32: every lane of the calling warp arrives once).
// Dense: one bulk copy of the contiguous rows.  Paged: one bulk copy per row.
__device__ __forceinline__ void issue_rows(const CacheView &c, int l, int s, int g, int row0,
                                           int nrows, char *dst, uint64_t *bar, int lane) {
  if (!c.paged()) {
    if (lane == 0) {
      const uint32_t bytes = (uint32_t)nrows * (uint32_t)c.rb;
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(dst, c.k + c.row_off(l, s, g, row0), bytes, bar);
    } else {
      mbar_arrive(bar);
    }
    return;
  }
  uint32_t bytes = 0;
  for (int r = lane; r < nrows; r += 32) bytes += (c.row_off(l, s, g, row0 + r) >= 0) ? c.rb : 0;
  if (bytes > 0)
    mbar_arrive_expect_tx(bar, bytes);
  else
    mbar_arrive(bar);
  for (int r = lane; r < nrows; r += 32) {
    const long long off = c.row_off(l, s, g, row0 + r);
    if (off >= 0) bulk_g2s(dst + (long long)r * c.rb, c.k + off, c.rb, bar);
  }
}

// Short-unit variant of the K streaming (the fused kernel's): every warp scores,
// warp 0 refills a stage right after the CTA barrier that ends it.  With two
// CTAs per SM this measured faster than the producer-warp pipeline below.
// Streams rows [0, n) of unit (l, s, g) through the ring and scores them into
// scores[h * sstride + i].  Returns false (CTA-uniform) if a wait timed out.
// The caller has initialised bars[0..kStages) with count 32 and synchronised.
template <int D, int G, bool BF16>
__device__ bool score_unit_rows(const CacheView &c, int l, int s, int g, int row_begin, int n,
                                char *ring, uint64_t *bars, float *scores, int sstride,
                                const LaneWeights<G> &lw, bool inter) {
  constexpr int TR = kStageBytes / RowGeom<D, BF16>::RB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int ntiles = (n + TR - 1) / TR;
  if (warp == 0) {
    for (int t = 0; t < ntiles && t < kStages; ++t)
      issue_rows(c, l, s, g, row_begin + t * TR, min(TR, n - t * TR), ring + t * kStageBytes,
                 &bars[t], lane);
  }
  for (int t = 0; t < ntiles; ++t) {
    const int st = t % kStages;
    const bool ok = mbar_wait(&bars[st], (uint32_t)((t / kStages) & 1));
    score_tile<D, G, BF16>(ring + st * kStageBytes, min(TR, n - t * TR), t * TR, scores, sstride,
                           lw, inter, warp, nw);
    if (__syncthreads_or(!ok)) return false;
    if (warp == 0 && t + kStages < ntiles) {
      const int tn = t + kStages;
      issue_rows(c, l, s, g, row_begin + tn * TR, min(TR, n - tn * TR), ring + st * kStageBytes,
                 &bars[st], lane);
    }
  }
  return true;
}

// ---------------------------------------------------------------- K streaming pipeline
// The score phase of a CTA is a producer/consumer pipeline over a ring of
// kStages shared-memory stages of kStageBytes:
//   - the producer warp (kProducerWarp) loads stage after stage of K rows with
//     bulk / tensor copies (TMA), completing on full[st] (arrival count 1 plus the
//     transaction bytes);
//   - the kConsumerWarps consumer warps score each stage, then each arrives once
//     on empty[st] (arrival count kConsumerWarps), which lets the producer
//     refill it.
// No block-wide barrier is taken per stage.  Every wait is bounded: a wait that
// gives up records TRI_ERR_TIMEOUT and sets *fail (shared), the pipeline runs to
// its end without waiting further on that stage, and the CTA drains its copies
// in flight (bounded again) before it leaves.
struct Pipe {
  char *ring;
  uint64_t *full;    // [kStages]
  uint64_t *empty;   // [kStages]
  volatile int *fail;     // shared flag
  volatile int *issued;   // shared: stages the producer issued
};

// Initialises the pipeline barriers (thread 0; caller synchronises).
__device__ __forceinline__ void pipe_init(const Pipe &p) {
  for (int st = 0; st < kStages; ++st) {
    mbar_init(&p.full[st], 1);
    mbar_init(&p.empty[st], kConsumerWarps);
  }
  *p.fail = 0;
  *p.issued = 0;
  fence_mbar_init();
}

// Producer side: loads rows [row0, row0 + nrows) of unit (l, s, g)'s K into dst,
// completing on `full`.  Dense: one bulk copy of the contiguous rows.  Paged with
// a tensor map: one 4-D tensor copy per block (box = one block of one head; rows
// of the last block past nrows are loaded too, they exist).  Paged without: one
// bulk copy per row.  Called by all 32 lanes of the producer warp.
template <int RB>
__device__ __forceinline__ void produce_stage(const CacheView &c, const CUtensorMap *tmk, int l, int s,
                                              int g, int row0, int nrows, char *dst, uint64_t *full,
                                              int lane) {
  if (!c.paged()) {
    if (lane == 0) {
      const uint32_t bytes = (uint32_t)nrows * (uint32_t)RB;
      mbar_arrive_expect_tx(full, bytes);
      bulk_g2s(dst, c.k + c.row_off(l, s, g, row0), bytes, full);
    }
    return;
  }
  if (c.tm_ok) {
    const int blk = c.block, nblk = (nrows + blk - 1) / blk;
    if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(nblk * blk * RB));
    __syncwarp();
    if (lane < nblk) {
      const int b = c.bt[(long long)s * c.max_blocks + row0 / blk + lane];
      tma_load_4d(dst + lane * blk * RB, tmk, 0, g, 0, (int)((long long)l * c.nblocks + b), full);
    }
    return;
  }
  int bytes = 0;
  for (int r = lane; r < nrows; r += 32) bytes += (c.row_off(l, s, g, row0 + r) >= 0) ? RB : 0;
  bytes = warp_sum_int(bytes);
  if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)bytes);
  __syncwarp();
  for (int r = lane; r < nrows; r += 32) {
    const long long off = c.row_off(l, s, g, row0 + r);
    if (off >= 0) bulk_g2s(dst + (long long)r * RB, c.k + off, (uint32_t)RB, full);
  }
}

// Streams rows [row_begin, row_begin + n) of unit (l, s, g) through the ring and
// scores them into scores[h * sstride + i] (i relative to row_begin).  Called by
// every thread of the CTA (kThreads); returns false (CTA-uniform, after a
// barrier) if a wait gave up.  The caller initialised the pipe and synchronised.
template <int D, int G, bool BF16>
__device__ bool stream_and_score(const CacheView &c, const CUtensorMap *tmk, int l, int s, int g,
                                 int row_begin, int n, const Pipe &p, float *scores, int sstride,
                                 const LaneWeights<G> &lw, bool inter) {
  using RG = RowGeom<D, BF16>;
  constexpr int TR = kStageBytes / RG::RB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = (n + TR - 1) / TR;
  if (warp == kProducerWarp) {
    int t = 0;
    for (; t < ntiles; ++t) {
      const int st = t % kStages;
      if (*p.fail || (t >= kStages && !mbar_wait(&p.empty[st], (uint32_t)(((t / kStages) - 1) & 1)))) {
        *p.fail = 1;
        break;
      }
      produce_stage<RG::RB>(c, tmk, l, s, g, row_begin + t * TR, min(TR, n - t * TR),
                            p.ring + st * kStageBytes, &p.full[st], lane);
    }
    if (lane == 0) *p.issued = t;
  } else {
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % kStages;
      if (!*p.fail && !mbar_wait(&p.full[st], (uint32_t)((t / kStages) & 1))) *p.fail = 1;
      score_tile<D, G, BF16>(p.ring + st * kStageBytes, min(TR, n - t * TR), t * TR, scores, sstride, lw,
                             inter, warp, kConsumerWarps);
      __syncwarp();
      if (lane == 0) mbar_arrive(&p.empty[st]);
    }
  }
  __syncthreads();
  if (*p.fail == 0) return true;
  // Drain: wait (bounded) for the last phase issued on every stage.
  if (threadIdx.x == 0) {
    const int issued = *p.issued;
    for (int st = 0; st < kStages && st < issued; ++st) {
      const int last = st + ((issued - 1 - st) / kStages) * kStages;
      mbar_wait(&p.full[st], (uint32_t)((last / kStages) & 1));
    }
  }
  __syncthreads();
  return false;
}

// ---------------------------------------------------------------- GQA moments (a3)
// Population mean and 1/std per head over scores[h * sstride + i], i < n (two
// passes over shared memory).  inv = 0 when std = 0 (z = 0).  The sums are
// taken of the scores minus the head's first score (z does not depend on a
// shift): a head whose scores are all equal then has exactly zero deviation,
// and cancellation stays small when the mean is large against the spread.
template <int G>
__device__ __forceinline__ void head_moments(const float *scores, int sstride, int n, float *red,
                                             float (&mu)[G], float (&inv)[G]) {
  float v[G], sh[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    v[h] = 0.f;
    sh[h] = scores[h * sstride];
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
#pragma unroll
    for (int h = 0; h < G; ++h) v[h] += scores[h * sstride + i] - sh[h];
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
      const float dlt = (scores[h * sstride + i] - sh[h]) - md[h];
      v[h] = fmaf(dlt, dlt, v[h]);
    }
  }
  block_sum<G>(v, red);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float sd = sqrtf(v[h] / (float)n);
    inv[h] = sd > 0.f ? 1.0f / sd : 0.0f;
  }
}

// ---------------------------------------------------------------- top-B (a4)
// Shared scratch of the selection (ints): [0..1] radix result, [8..23] per-warp
// partial sums of the histogram scan, [24..39] per-warp tie counts, [40..55]
// per-warp kept counts, [56] first dropped slot.  kSelInts ints.
constexpr int kSelInts = 64;

// Short-unit variant of the selection (the fused kernel's; measured faster there
// than the variants below, whose extra passes only pay off for long units).
// Radix select (8-bit digits, most significant first) of the K-th largest key
// among keys[0..n).  Returns the threshold key T and, in *ntie, how many keys
// equal to T are kept (the lowest slots).  Needs blockDim >= 256.
// hist: 256 u32; sm: 4 ints.
__device__ __noinline__ uint32_t radix_select_atomic(const uint32_t *keys, int n, int K, uint32_t *hist,
                                              int *sm, int *ntie) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, mask = 0;
  int k = K;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
      const uint32_t u = keys[i];
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    // Suffix counts S[x] = #{digit >= x}: thread t < 256 scans the reversed
    // histogram, so its inclusive prefix P_t equals S[255 - t] and P_{t-1}
    // equals S[256 - t].  The digit x is the one with S[x] >= k > S[x + 1].
    int P = 0, wsum = 0;
    if (tid < 256) {
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
    const uint32_t dgt = (uint32_t)sm[0];
    k = sm[1];
    prefix |= dgt << shift;
    mask |= 255u << shift;
    __syncthreads();
  }
  *ntie = k;
  return prefix;
}

// Writes the kept slots of keys[0..n) (those > T, plus the first ntie equal to
// T in slot order) to idx[0..K) in ascending order; returns the first dropped
// slot (n if none).  Never writes past idx[K-1].  Each thread walks a
// contiguous chunk of slots.  sm: 40 ints.
__device__ __noinline__ int build_kept_chunked(const uint32_t *keys, int n, int K, uint32_t T, int ntie,
                                       int *idx, int *sm) {
  const int tid = threadIdx.x;
  const int chunk = (n + blockDim.x - 1) / blockDim.x;
  const int i0 = min(n, tid * chunk), i1 = min(n, i0 + chunk);
  int ceq = 0;
  for (int i = i0; i < i1; ++i) ceq += (keys[i] == T);
  int tot;
  const int eq_before = block_excl_scan(ceq, sm, &tot);
  int ck = 0, e = eq_before, first_drop = n;
  for (int i = i0; i < i1; ++i) {
    const uint32_t u = keys[i];
    bool keep = u > T;
    if (u == T) {
      keep = e < ntie;
      ++e;
    }
    ck += keep;
    if (!keep && first_drop == n) first_drop = i;
  }
  if (tid == 0) sm[36] = n;
  __syncthreads();
  const int kb = block_excl_scan(ck, sm, &tot);
  if (first_drop < n) atomicMin(&sm[36], first_drop);
  e = eq_before;
  int o = kb;
  for (int i = i0; i < i1; ++i) {
    const uint32_t u = keys[i];
    bool keep = u > T;
    if (u == T) {
      keep = e < ntie;
      ++e;
    }
    if (keep && o < K) idx[o++] = i;
  }
  __syncthreads();
  const int e0 = sm[36];
  __syncthreads();
  return e0;
}

// Writes the kept slots of keys[0..n) (those > T, plus the first ntie equal to
// T in slot order) to idx[0..K) in ascending order; returns the first dropped
// slot (n if none).  Never writes past idx[K-1].  Each warp owns one contiguous
// segment of slots and walks it 32 consecutive slots at a time (ballot + popc
// for the in-order positions), so lanes read consecutive words.
__device__ __noinline__ int build_kept(const uint32_t *keys, int n, int K, uint32_t T, int ntie,
                                       int *idx, int *sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int seg = (((n + nw - 1) / nw) + 31) / 32 * 32;
  const int lo = min(n, warp * seg), hi = min(n, lo + seg);
  int cgt = 0, ceq = 0;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const uint32_t u = i < hi ? keys[i] : 0u;
    cgt += __popc(__ballot_sync(0xffffffffu, i < hi && u > T));
    ceq += __popc(__ballot_sync(0xffffffffu, i < hi && u == T));
  }
  if (lane == 0) {
    sm[24 + warp] = ceq;
    sm[40 + warp] = cgt;
  }
  if (tid == 0) sm[56] = n;
  __syncthreads();
  int eq_before = 0, kept_before = 0;
  for (int w = 0; w < warp; ++w) {
    const int e = sm[24 + w];
    const int tw = max(0, min(e, ntie - eq_before));
    kept_before += sm[40 + w] + tw;
    eq_before += e;
  }
  const unsigned lt = lanemask_lt();
  int eq_run = eq_before, pos_run = kept_before, first_drop = n;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const bool valid = i < hi;
    const uint32_t u = valid ? keys[i] : 0u;
    const unsigned eqm = __ballot_sync(0xffffffffu, valid && u == T);
    const bool keep = valid && (u > T || (u == T && eq_run + __popc(eqm & lt) < ntie));
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    const unsigned dm = __ballot_sync(0xffffffffu, valid && !keep);
    const int pos = pos_run + __popc(km & lt);
    if (keep && pos < K) idx[pos] = i;
    if (dm != 0u && first_drop == n) first_drop = base + __ffs(dm) - 1;
    eq_run += __popc(eqm);
    pos_run += __popc(km);
  }
  if (lane == 0 && first_drop < n) atomicMin(&sm[56], first_drop);
  __syncthreads();
  const int e0 = sm[56];
  __syncthreads();
  return e0;
}

// Writes the kept set of keys[0..n) (those > T, plus the first ntie equal to
// T in slot order) as a bitmask: bit i % 32 of out[i / 32] (bits of slots at or
// past n are 0).  Each warp owns a contiguous run of 32-slot words; a block
// scan of the warps' counts of keys equal to T allots the ties in slot order.
// sm: 32 ints for the scan.
__device__ __noinline__ void kept_bits(const uint32_t *keys, int n, uint32_t T, int ntie, uint32_t *out, int *sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int W = (n + 31) / 32, wpw = (W + nw - 1) / nw;
  const int w0 = min(W, warp * wpw), w1 = min(W, w0 + wpw);
  int ceq = 0;
  for (int w = w0; w < w1; ++w) {
    const int i = 32 * w + lane;
    ceq += __popc(__ballot_sync(0xffffffffu, i < n && keys[i] == T));
  }
  int tot;
  int before = block_excl_scan(lane == 0 ? ceq : 0, sm, &tot);
  before = __shfl_sync(0xffffffffu, before, 0);
  int allow = ntie - before;   // ties this warp may still keep (warp-uniform)
  for (int w = w0; w < w1; ++w) {
    const int i = 32 * w + lane;
    const bool in = i < n;
    const uint32_t k = in ? keys[i] : 0u;
    const uint32_t gt = __ballot_sync(0xffffffffu, in && k > T);
    uint32_t eq = __ballot_sync(0xffffffffu, in && k == T), sel = 0;
    while (allow > 0 && eq != 0u) {
      const uint32_t b = eq & (0u - eq);
      sel |= b;
      eq ^= b;
      --allow;
    }
    if (lane == 0) out[w] = gt | sel;
  }
}

// ---------------------------------------------------------------- top-B over keys in global memory
// Variants of radix_select_atomic / build_kept for keys stored in global memory
// (L2-resident: one unit's keys are 4 N bytes), used by the long-unit select
// kernel so that its shared memory fits two CTAs per SM.  Rows of keys are
// 16-byte aligned; the reads are 16-byte vectors (radix) or 8 steps of 32
// consecutive keys per warp issued together (kept list).

// Radix select as radix_select_atomic, reading keys4[0..ceil(n/4)).
__device__ __noinline__ uint32_t radix_select_gmem(const uint32_t *keys, int n, int K, uint32_t *hist, int *sm,
                                                   int *ntie) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
  const uint4 *keys4 = reinterpret_cast<const uint4 *>(keys);
  const int n4 = (n + 3) / 4;
  uint32_t prefix = 0, mask = 0;
  int k = K;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += nt) hist[b] = 0;
    __syncthreads();
#pragma unroll 4
    for (int q = tid; q < n4; q += nt) {
      const uint4 v = keys4[q];
      const uint32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (4 * q + j < n && (e[j] & mask) == prefix) atomicAdd(&hist[(e[j] >> shift) & 255u], 1u);
    }
    __syncthreads();
    int P = 0, wsum = 0;
    if (tid < 256) {
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
    const uint32_t dgt = (uint32_t)sm[0];
    k = sm[1];
    prefix |= dgt << shift;
    mask |= 255u << shift;
    __syncthreads();
  }
  *ntie = k;
  return prefix;
}

// build_kept over keys in global memory (same result and shared scratch).
__device__ __noinline__ int build_kept_gmem(const uint32_t *keys, int n, int K, uint32_t T, int ntie, int *idx,
                                            int *sm) {
  constexpr int PF = 8;   // steps of 32 keys loaded together
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int seg = (((n + nw - 1) / nw) + 31) / 32 * 32;
  const int lo = min(n, warp * seg), hi = min(n, lo + seg);
  int cgt = 0, ceq = 0;
  for (int base = lo; base < hi; base += 32 * PF) {
    uint32_t u[PF];
#pragma unroll
    for (int e = 0; e < PF; ++e) {
      const int i = base + 32 * e + lane;
      u[e] = i < hi ? keys[i] : 0u;
    }
#pragma unroll
    for (int e = 0; e < PF; ++e) {
      const bool in = base + 32 * e + lane < hi;
      cgt += __popc(__ballot_sync(0xffffffffu, in && u[e] > T));
      ceq += __popc(__ballot_sync(0xffffffffu, in && u[e] == T));
    }
  }
  if (lane == 0) {
    sm[24 + warp] = ceq;
    sm[40 + warp] = cgt;
  }
  if (tid == 0) sm[56] = n;
  __syncthreads();
  int eq_before = 0, kept_before = 0;
  for (int w = 0; w < warp; ++w) {
    const int e = sm[24 + w];
    const int tw = max(0, min(e, ntie - eq_before));
    kept_before += sm[40 + w] + tw;
    eq_before += e;
  }
  const unsigned lt = lanemask_lt();
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

// ---------------------------------------------------------------- compaction (a5)
// Short-unit variant of the compaction (the fused kernel's): warp 0 alone, bulk
// copies only, a fixed ring of kStages stages.  Its per-chunk issue path is the
// shortest dependency chain, which is what bounds a single warp moving ~2000
// mostly contiguous rows.  In-place ordered gather of K and V rows of unit
// (l, s, g): row j <- row idx[j] for j in [e0, B) (rows below e0 are kept in
// place); the other warps may leave.
//
// Destination chunks of up to 32 rows (K and V, one ring stage) are processed in
// ascending order.  Lane r of warp 0 owns destination row j0 + r of a chunk.
// Loads: dense caches copy each run of consecutive source slots with one bulk
// copy per tensor; paged caches copy row by row.  Stores: one bulk store per
// tensor for a dense chunk (its destination rows are contiguous), row by row for
// paged.  In-place safety: a chunk is stored only after its loads completed,
// and every load of a later chunk reads slots >= that chunk's first destination,
// which no earlier store touches, since idx is strictly increasing (idx_j >= j).
// A ring stage is refilled only after the bulk stores that read it finished
// reading (per-lane bulk async-groups, one group per chunk per lane).
//
// cbars: kStages mbarriers initialised with arrival count 1.  Returns false if a
// wait timed out (status recorded).
__device__ __noinline__ bool compact_unit_runs(const CacheView &c, int l, int s, int g,
                                              const int *idx, int e0, int B, int N, char *ring,
                                              uint64_t *cbars) {
  const int lane = threadIdx.x & 31;
  const int rb = c.rb;
  const int ch = min(32, kStageBytes / (2 * rb));   // rows per chunk
  const int M = B - e0;
  if (M <= 0) return true;
  const int nch = (M + ch - 1) / ch;
  const bool paged = c.paged();

  auto issue_loads = [&](int cidx) {
    const int st = cidx % kStages;
    char *sk = ring + st * kStageBytes;   // K rows [0, ch), then V rows [ch, 2ch)
    const int j0 = e0 + cidx * ch;
    const int rows = min(ch, B - j0);
    int src = -1;
    bool valid = lane < rows;
    if (valid) {
      src = idx[j0 + lane];
      if (src < 0 || src >= N) {
        set_status(TRI_ERR_BOUNDS);
        valid = false;
      }
    }
    long long off = valid ? c.row_off(l, s, g, src) : -1;
    if (off < 0) valid = false;
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    if (lane == 0) mbar_arrive_expect_tx(&cbars[st], (uint32_t)__popc(vmask) * 2u * (uint32_t)rb);
    __syncwarp();
    if (!paged) {
      const int prev = __shfl_up_sync(0xffffffffu, src, 1);
      const bool boundary = !valid || lane == 0 || prev + 1 != src;
      const unsigned bmask = __ballot_sync(0xffffffffu, boundary);
      if (valid && boundary) {
        const unsigned later = (lane == 31) ? 0u : (bmask & (0xffffffffu << (lane + 1)));
        const int end = later ? (__ffs(later) - 1) : rows;
        const uint32_t bytes = (uint32_t)(end - lane) * (uint32_t)rb;
        bulk_g2s(sk + (long long)lane * rb, c.k + off, bytes, &cbars[st]);
        bulk_g2s(sk + (long long)(ch + lane) * rb, c.v + off, bytes, &cbars[st]);
      }
    } else if (valid) {
      bulk_g2s(sk + (long long)lane * rb, c.k + off, (uint32_t)rb, &cbars[st]);
      bulk_g2s(sk + (long long)(ch + lane) * rb, c.v + off, (uint32_t)rb, &cbars[st]);
    }
  };

  for (int x = 0; x < kStages - 1 && x < nch; ++x) issue_loads(x);
  bool ok = true;
  for (int cidx = 0; cidx < nch; ++cidx) {
    const int st = cidx % kStages;
    const char *sk = ring + st * kStageBytes;
    const int j0 = e0 + cidx * ch;
    const int rows = min(ch, B - j0);
    if (!mbar_wait(&cbars[st], (uint32_t)((cidx / kStages) & 1))) {
      ok = false;
      break;
    }
    if (!paged) {
      if (lane == 0) {
        const long long off = c.row_off(l, s, g, j0);
        bulk_s2g(c.k + off, sk, (uint32_t)(rows * rb));
        bulk_s2g(c.v + off, sk + (long long)ch * rb, (uint32_t)(rows * rb));
      }
    } else if (lane < rows) {
      const long long off = c.row_off(l, s, g, j0 + lane);
      if (off >= 0) {
        bulk_s2g(c.k + off, sk + (long long)lane * rb, (uint32_t)rb);
        bulk_s2g(c.v + off, sk + (long long)(ch + lane) * rb, (uint32_t)rb);
      }
    }
    bulk_commit();
    bulk_wait_read<1>();   // the stores of chunk cidx-1 no longer read their stage
    __syncwarp();
    if (cidx + kStages - 1 < nch) issue_loads(cidx + kStages - 1);   // refills that stage
  }
  bulk_wait<0>();
  return ok;
}

// In-place ordered gather of K and V rows of unit (l, s, g): row j <- row idx[j]
// for j in [e0, B) (rows below e0 are kept in place), issued by warp 0 alone
// with TMA copies; the other warps may leave.
//
// Destination chunks of ch rows (K rows then V rows fill one ring stage; lane r
// owns destination row j0 + r) are processed in ascending order.
// Loads, per chunk and tensor (a TMA op costs tens of ns to issue, so the
// number of ops per chunk is what is minimised):
//   - dense caches whose chunk has at most kRunLimit runs of consecutive source
//     slots: one bulk copy per run;
//   - otherwise (scattered sources, and every chunk of a paged cache): one
//     tile::gather4 of 4 source rows per quad of destination rows through the
//     row map (or, with kCompactLsu = 1, the warp's own 16-byte cp.async
//     copies, whole rows per instruction).
// Stores: dense, one bulk store per tensor (the destination rows are
// contiguous); paged with block maps, one tensor store per destination block
// (chunks then start at a block boundary: rows below e0 in the first block are
// reloaded from themselves and rewritten unchanged; rows at or past B in the
// last block receive don't-care values); otherwise one bulk store per row.
// In-place safety: a chunk is stored only after its loads completed, and every
// load of a later chunk reads slots >= that chunk's first destination, which no
// earlier store touches, since idx is strictly increasing (idx_j >= j).  A ring
// stage is refilled only after the bulk stores that read it finished reading.
//
// ring: nstages (2..kMaxCompactStages) stages of kStageBytes; cbars: nstages
// mbarriers initialised with arrival count kCompactArrivals.  Returns false if a wait timed out
// (status recorded; loads already issued are waited for, bounded).
constexpr int kRunLimit = 8;   // runs per chunk up to which bulk copies beat row gathers
#ifndef TRI_COMPACT_LSU
#define TRI_COMPACT_LSU 0
#endif
// Scattered rows are gathered by tile::gather4 tensor copies (0) or by the
// warp's own 16-byte cp.async copies (1).  Measured on the long and the paged
// workloads, the tensor gathers were 2-3 % faster, so they are the default.
constexpr int kCompactLsu = TRI_COMPACT_LSU;
// Arrivals per phase of a compaction ring barrier: lane 0's byte-count arrival
// plus one cp.async-completion arrival from each of the warp's 32 lanes.
constexpr int kCompactArrivals = 33;

// Compacts one tensor (which = 0: K, 1: V) of unit (l, s, g); the calling warp
// owns it alone (the two tensors are independent arrays, so a K warp and a V
// warp run side by side, each with its own barriers and bulk groups).  Stage st
// holds the chunk's K rows at [0, ch) and V rows at [ch, 2ch).
__device__ __noinline__ bool compact_unit_tma(const CacheView &c, const TmaMaps *maps, int which, int l, int s,
                                              int g, const int *idx, int e0, int B, int N, char *ring,
                                              int nstages, uint64_t *cbars) {
  const int lane = threadIdx.x & 31;
  const int rb = c.rb;
  const int ch = min(32, kStageBytes / (2 * rb));   // rows per chunk (a multiple of 4)
  if (B - e0 <= 0) return true;
  char *base = which ? c.v : c.k;
  const CUtensorMap *map2 = which ? &maps->v2 : &maps->k2;
  const CUtensorMap *map4 = which ? &maps->v4 : &maps->k4;
  const long long toff = (long long)which * ch * rb;   // this tensor's rows within a stage
  const bool paged = c.paged();
  const bool blkst = paged && c.tm_ok && ch % c.block == 0;
  const int jb = blkst ? (e0 / c.block) * c.block : e0;
  const int nch = (B - jb + ch - 1) / ch;

  auto issue_loads = [&](int cidx) {
    const int st = cidx % nstages;
    char *sk = ring + st * kStageBytes + toff;
    const int j0 = jb + cidx * ch;
    const int rows = min(ch, B - j0);
    int src = -1;
    bool valid = lane < rows;
    if (valid) {
      src = idx[j0 + lane];
      if (src < 0 || src >= N) {
        set_status(TRI_ERR_BOUNDS);
        valid = false;
      }
    }
    const long long r2 = valid ? c.row2d(l, s, g, src) : -1;
    if (r2 < 0) valid = false;
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    // runs of consecutive source slots (dense caches only: paged rows of one
    // head are not adjacent in memory)
    const int prev = __shfl_up_sync(0xffffffffu, src, 1);
    const bool boundary = valid && (paged || lane == 0 || !((vmask >> (lane - 1)) & 1u) || prev + 1 != src);
    const unsigned bmask = __ballot_sync(0xffffffffu, boundary);
    const bool use_runs = !paged && (__popc(bmask) <= kRunLimit || (!kCompactLsu && c.g4_ok == 0));
    if (use_runs) {
      // one bulk copy per run [lane, next boundary or invalid lane)
      int end = lane;
      if (boundary) {
        const unsigned stop = (bmask | ~vmask) & (lane == 31 ? 0u : (0xffffffffu << (lane + 1)));
        end = stop ? (__ffs(stop) - 1) : 32;
      }
      const int bytes = warp_sum_int((end - lane) * rb);
      if (lane == 0) mbar_arrive_expect_tx(&cbars[st], (uint32_t)bytes);
      __syncwarp();
      if (boundary)
        bulk_g2s(sk + (long long)lane * rb, base + r2 * rb, (uint32_t)((end - lane) * rb), &cbars[st]);
    } else if (kCompactLsu) {
      // 16-byte cp.async pieces, ppr lanes per row and 32 / ppr rows per
      // instruction, so each instruction reads whole rows (coalesced); the
      // rows land at their destination positions of the stage
      if (lane == 0) mbar_arrive_expect_tx(&cbars[st], 0u);
      const int ppr = rb >> 4, rpi = 32 / ppr;
      const int sub = lane / ppr, piece = lane - sub * ppr;
      for (int r0 = 0; r0 < rows; r0 += rpi) {
        const int row = r0 + sub;
        const long long rr = __shfl_sync(0xffffffffu, r2, row & 31);
        if (row < rows && ((vmask >> row) & 1u))
          cp_async16(sk + (long long)row * rb + piece * 16, base + rr * rb + piece * 16);
      }
    } else if (c.g4_ok) {
      // one tile::gather4 per quad of destination rows (lanes past `rows`
      // repeat the quad's first valid row; those smem rows are never stored)
      const int q0 = lane & ~3;
      const unsigned qmask = 0xfu << q0;
      const int firstv = __ffs(vmask & qmask) - 1;
      const long long rfill = __shfl_sync(0xffffffffu, r2, firstv < 0 ? lane : firstv);
      const int rc = (int)(valid ? r2 : rfill);
      const int c0 = __shfl_sync(0xffffffffu, rc, q0);
      const int c1 = __shfl_sync(0xffffffffu, rc, q0 + 1);
      const int c2 = __shfl_sync(0xffffffffu, rc, q0 + 2);
      const int c3 = __shfl_sync(0xffffffffu, rc, q0 + 3);
      const bool gath = lane == q0 && (vmask & qmask) != 0u;
      const unsigned gmask = __ballot_sync(0xffffffffu, gath);
      if (lane == 0) mbar_arrive_expect_tx(&cbars[st], (uint32_t)(__popc(gmask) * 4 * rb));
      __syncwarp();
      if (gath) tma_gather4(sk + (long long)q0 * rb, map2, 0, c0, c1, c2, c3, &cbars[st]);
    } else {
      // paged without row maps: one bulk copy per row
      if (lane == 0) mbar_arrive_expect_tx(&cbars[st], (uint32_t)(__popc(vmask) * rb));
      __syncwarp();
      if (valid) bulk_g2s(sk + (long long)lane * rb, base + r2 * rb, (uint32_t)rb, &cbars[st]);
    }
    // every lane arrives once its cp.async copies (if any) have landed
    cp_async_arrive_noinc(&cbars[st]);
  };

  for (int x = 0; x < nstages - 1 && x < nch; ++x) issue_loads(x);
  bool ok = true;
  int cidx = 0;
  for (; cidx < nch; ++cidx) {
    const int st = cidx % nstages;
    const char *sk = ring + st * kStageBytes + toff;
    const int j0 = jb + cidx * ch;
    const int rows = min(ch, B - j0);
    if (!mbar_wait(&cbars[st], (uint32_t)((cidx / nstages) & 1))) {
      ok = false;
      break;
    }
    // rows written by cp.async (generic proxy) are read next by TMA stores
    fence_proxy_async_smem();
    if (!paged) {
      if (lane == 0) bulk_s2g(base + c.row_off(l, s, g, j0), sk, (uint32_t)(rows * rb));
    } else if (blkst) {
      const int nb = (rows + c.block - 1) / c.block;
      if (lane < nb) {
        const int b = c.bt[(long long)s * c.max_blocks + j0 / c.block + lane];
        tma_store_4d(map4, 0, g, 0, (int)((long long)l * c.nblocks + b), sk + (long long)lane * c.block * rb);
      }
    } else if (lane < rows) {
      const long long off = c.row_off(l, s, g, j0 + lane);
      if (off >= 0) bulk_s2g(base + off, sk + (long long)lane * rb, (uint32_t)rb);
    }
    bulk_commit();
    bulk_wait_read<1>();   // the stores of chunk cidx-1 no longer read their stage
    __syncwarp();
    if (cidx + nstages - 1 < nch) issue_loads(cidx + nstages - 1);   // refills that stage
  }
  if (!ok) {
    // loads of chunks [cidx, cidx + nstages - 1) may still be in flight
    for (int x = cidx; x < nch && x < cidx + nstages - 1; ++x)
      if (!mbar_wait(&cbars[x % nstages], (uint32_t)((x / nstages) & 1))) break;
  }
  cp_async_wait_all();   // this lane's gathers (global reads: they always complete)
  bulk_wait<0>();
  return ok;
}

// ---------------------------------------------------------------- hole-fill compaction (a5, alternative)
// Bytes of holefill_unit's bookkeeping for a unit of N keys: one flag byte per
// slot below B (rounded to 16), then the hole list (at most min(B, N - B) ints).
__host__ __device__ __forceinline__ int holefill_work_bytes(int B, int N) {
  const int movers = N - B < B ? N - B : B;
  return ((B + 15) & ~15) + 4 * (movers > 0 ? movers : 0);
}

// Hole-fill layout of unit (l, s, g) from its ascending kept list idx[0..B):
// kept slots below B stay; the evicted slots below B (holes, ascending) receive
// the kept slots at or above B (movers, ascending), the k-th hole the k-th
// mover.  Sources (>= B) and destinations (< B) are disjoint, so every row copy
// is independent.  The movers are the tail of the ascending kept list, so
// their K and V rows are gathered first, with 16-byte cp.async copies (a warp
// per row, its lanes on the row's pieces) into `stage`, while the holes are
// ranked; then stored from shared memory to their holes.  All at once when
// they fit the stage, else in batches of a quarter of it, three in flight
// while the oldest is stored.  `work` (shared,
// holefill_work_bytes(B, N), 16-byte aligned, dead by now, disjoint from
// `stage`) holds one flag byte per slot below B, then the hole list.  stage:
// 16-byte aligned; with less than 4 row sizes the rows are copied directly.  out (global, may be null)
// receives the layout: out[j] = original slot now at j.  sm: 40 ints for the
// scan.  Ends with a CTA barrier.
__device__ __noinline__ void holefill_unit(const CacheView &c, int l, int s, int g, const int *idx, int B,
                                           int N, char *work, char *stage, int stage_bytes, int *sm, int *out) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int rb = c.rb, ppr = rb >> 4, pp = 2 * ppr;
  // the movers (kept slots >= B) are the tail idx[P..B) of the ascending kept
  // list: their gathers start now, ahead of the bookkeeping
  int lo = 0, hi = B;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (idx[mid] < B) lo = mid + 1; else hi = mid;
  }
  const int P = lo, total = B - P;
  // every mover fits the stage at once, or batches of a quarter of it cycle
  // through 4 buffers with 3 batches in flight
  constexpr int kBufs = 4;
  const int rows_full = stage_bytes / (2 * rb);
  const bool single = total <= rows_full;
  const int rh = single ? rows_full : stage_bytes / (kBufs * 2 * rb);
  const int half = rh * 2 * rb;   // bytes of one buffer
  const int nbat = rh > 0 ? (total + rh - 1) / rh : 0;
  auto issue = [&](int b) {       // always commits a group (empty past the last batch)
    char *st = stage + (b % kBufs) * half;
    const int k0 = b * rh, nr = b < nbat ? min(rh, total - k0) : 0;
    for (int k = warp; k < nr; k += nw) {
      const long long so = c.row_off(l, s, g, idx[P + k0 + k]);
      if (so < 0) continue;
      for (int q = lane; q < pp; q += 32) {
        const char *base = q < ppr ? c.k : c.v;
        const int col = (q < ppr ? q : q - ppr) * 16;
        cp_async16(st + (long long)k * 2 * rb + (q < ppr ? 0 : rb) + col, base + so + col);
      }
    }
    cp_async_commit();
  };
  if (rh > 0) {
    if (single) {
      if (nbat > 0) issue(0);
    } else {
      for (int b = 0; b < kBufs - 1; ++b) issue(b);
    }
  }
  unsigned char *kept = reinterpret_cast<unsigned char *>(work);
  int *holes = reinterpret_cast<int *>(work + ((B + 15) & ~15));
  for (int j = tid; j < B; j += nt) kept[j] = 0;
  __syncthreads();
  for (int j = tid; j < P; j += nt) kept[idx[j]] = 1;
  __syncthreads();
  // holes in slot order: each thread scans a contiguous chunk of slots
  const int chunk = (B + nt - 1) / nt;
  const int j0 = min(B, tid * chunk), j1 = min(B, j0 + chunk);
  int nh = 0;
  for (int j = j0; j < j1; ++j) nh += kept[j] == 0;
  int nholes;
  int r = block_excl_scan(nh, sm, &nholes);   // nholes == total
  for (int j = j0; j < j1; ++j) {
    if (kept[j]) {
      if (out != nullptr) out[j] = j;
    } else {
      holes[r] = j;
      if (out != nullptr) out[j] = idx[P + r];
      ++r;
    }
  }
  __syncthreads();
  // copy mover k's K and V rows into hole k: a warp owns a row at a time, its
  // lanes take the row's 2 ppr 16-byte pieces (K pieces, then V pieces)
  if (rh < 1) {
    // no room to stage: 16-byte copies straight from the movers to the holes
    for (int k = warp; k < total; k += nw) {
      const long long so = c.row_off(l, s, g, idx[P + k]), dof = c.row_off(l, s, g, holes[k]);
      if (so < 0 || dof < 0) continue;
      for (int q = lane; q < pp; q += 32) {
        char *base = q < ppr ? c.k : c.v;
        const int col = (q < ppr ? q : q - ppr) * 16;
        *reinterpret_cast<uint4 *>(base + dof + col) = *reinterpret_cast<const uint4 *>(base + so + col);
      }
    }
    __syncthreads();
    return;
  }
  auto store = [&](int b) {
    const char *st = stage + (b % kBufs) * half;
    const int k0 = b * rh, nr = min(rh, total - k0);
    for (int k = warp; k < nr; k += nw) {
      const long long so = c.row_off(l, s, g, idx[P + k0 + k]), dof = c.row_off(l, s, g, holes[k0 + k]);
      if (so < 0 || dof < 0) continue;
      for (int q = lane; q < pp; q += 32) {
        char *base = q < ppr ? c.k : c.v;
        const int col = (q < ppr ? q : q - ppr) * 16;
        *reinterpret_cast<uint4 *>(base + dof + col) =
            *reinterpret_cast<const uint4 *>(st + (long long)k * 2 * rb + (q < ppr ? 0 : rb) + col);
      }
    }
  };
  if (single) {
    cp_async_wait<0>();
    __syncthreads();          // every mover has landed
    if (nbat > 0) store(0);
  } else {
    for (int b = 0; b < nbat; ++b) {
      issue(b + kBufs - 1);   // its buffer was freed by the barrier that ended batch b - 1
      cp_async_wait<kBufs - 1>();
      __syncthreads();        // batch b has landed for every thread
      store(b);
      __syncthreads();        // batch b's buffer may be refilled
    }
    cp_async_wait<0>();
  }
  __syncthreads();
}

}  // namespace tri
