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

  __device__ __forceinline__ bool paged() const { return bt != nullptr; }
  // Byte offset of slot i of unit (l, s, g); -1 if the block id is out of range.
  __device__ __forceinline__ long long row_off(int l, int s, int g, int i) const {
    if (bt == nullptr) return ((((long long)l * S + s) * Hkv + g) * cap + i) * (long long)rb;
    const int b = bt[(long long)s * max_blocks + i / block];
    if (b < 0 || b >= nblocks) return -1;
    return ((((long long)l * nblocks + b) * block + (i % block)) * Hkv + g) * (long long)rb;
  }
  // Checks every block id a unit of sequence s with n keys will touch.
  __device__ bool blocks_ok(int s, int n) const {
    if (bt == nullptr) return true;
    const int nb = (n + block - 1) / block;
    int bad = 0;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
      const int id = bt[(long long)s * max_blocks + b];
      bad |= (id < 0 || id >= nblocks);
    }
    return __syncthreads_or(bad) == 0;
  }
};

// ---------------------------------------------------------------- weights (a1)
// wts layout [G][3][F]: Re A, Im A, W for the G query heads of KV head g.
// A_{h,f} = c_{h,f} * e^{i*omega_f*t} * Phi_f; W_{h,f} = (1 - R_{h,f}) * m_{h,f}.
// The phase omega_f*t is reduced modulo 2*pi in fp64 (two-term 2*pi split) before
// an fp32 sincos: omega_0*t reaches ~3e4 rad, far beyond fp32 phase accuracy.
template <int G, int F>
__device__ __forceinline__ void build_weights(float *wts, const float *center, const float *R,
                                              const float *mag, int Hq, int l, int g, int t,
                                              const StepConst &sc) {
  constexpr double kTwoPiHi = 6.283185307179586232;
  constexpr double kTwoPiLo = 2.449293598294706e-16;
  constexpr double kInvTwoPi = 0.15915494309189535;
  for (int x = threadIdx.x; x < G * F; x += blockDim.x) {
    const int h = x / F, f = x - h * F;
    const long long o = ((long long)l * Hq + (long long)g * G + h) * F + f;
    const double ph = sc.omega[f] * (double)t;
    const double q = rint(ph * kInvTwoPi);
    double r = fma(-q, kTwoPiHi, ph);
    r = fma(-q, kTwoPiLo, r);
    float sn, cs;
    sincosf((float)r, &sn, &cs);
    const float2 p = sc.phi[f];
    const float er = cs * p.x - sn * p.y;
    const float ei = cs * p.y + sn * p.x;
    const float cr = center[2 * o], ci = center[2 * o + 1];
    wts[(h * 3 + 0) * F + f] = cr * er - ci * ei;
    wts[(h * 3 + 1) * F + f] = cr * ei + ci * er;
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
// bands (Re A * Re k~ + Im A * Im k~ + W * |k~|), then a cross-lane sum.
template <int D, int G, bool BF16>
__device__ __forceinline__ void score_tile(const char *tile, int nrows, int row0, float *scores,
                                           int sstride, const LaneWeights<G> &lw, bool inter) {
  using RG = RowGeom<D, BF16>;
  constexpr int LPR = RG::LPR, RPW = RG::RPW, RB = RG::RB;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
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

// Streams rows [0, n) of unit (l, s, g) through the ring and scores them into
// scores[h * sstride + i].  Returns false (CTA-uniform) if a wait timed out.
// The caller has initialised bars[0..kStages) with count 32 and synchronised.
template <int D, int G, bool BF16>
__device__ bool score_unit_rows(const CacheView &c, int l, int s, int g, int row_begin, int n,
                                char *ring, uint64_t *bars, float *scores, int sstride,
                                const LaneWeights<G> &lw, bool inter) {
  constexpr int TR = kStageBytes / RowGeom<D, BF16>::RB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
                           lw, inter);
    if (__syncthreads_or(!ok)) return false;
    if (warp == 0 && t + kStages < ntiles) {
      const int tn = t + kStages;
      issue_rows(c, l, s, g, row_begin + tn * TR, min(TR, n - tn * TR), ring + st * kStageBytes,
                 &bars[st], lane);
    }
  }
  return true;
}

// ---------------------------------------------------------------- GQA moments (a3)
// Population mean and 1/std per head over scores[h * sstride + i], i < n (two
// passes over shared memory).  inv = 0 when std = 0 (z = 0).
template <int G>
__device__ __forceinline__ void head_moments(const float *scores, int sstride, int n, float *red,
                                             float (&mu)[G], float (&inv)[G]) {
  float v[G];
#pragma unroll
  for (int h = 0; h < G; ++h) v[h] = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
#pragma unroll
    for (int h = 0; h < G; ++h) v[h] += scores[h * sstride + i];
  }
  block_sum<G>(v, red);
#pragma unroll
  for (int h = 0; h < G; ++h) mu[h] = v[h] / (float)n;
#pragma unroll
  for (int h = 0; h < G; ++h) v[h] = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float dlt = scores[h * sstride + i] - mu[h];
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
// Radix select (8-bit digits, most significant first) of the K-th largest key
// among keys[0..n).  Returns the threshold key T and, in *ntie, how many keys
// equal to T are kept (the lowest slots).  Needs blockDim >= 256.
// hist: 256 u32; sm: 4 ints.
__device__ __noinline__ uint32_t radix_select(const uint32_t *keys, int n, int K, uint32_t *hist,
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
// slot (n if none).  Never writes past idx[K-1].  sm: 40 ints.
__device__ __noinline__ int build_kept(const uint32_t *keys, int n, int K, uint32_t T, int ntie,
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

// ---------------------------------------------------------------- compaction (a5)
// In-place ordered gather of K and V rows of unit (l, s, g): row j <- row idx[j]
// for j in [e0, B) (rows below e0 are kept in place), executed by warp 0 alone
// with bulk (TMA) copies; the other warps may leave.
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
__device__ __noinline__ bool compact_unit_tma(const CacheView &c, int l, int s, int g,
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

}  // namespace tri
