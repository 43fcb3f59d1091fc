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

// Loads the 4 bands (re, im) of this lane from a row in shared memory.
template <int D, bool BF16>
__device__ __forceinline__ void load_bands(const char *row, int j, bool inter, float (&re)[4],
                                           float (&im)[4]) {
  constexpr int F = D / 2;
  if constexpr (BF16) {
    if (!inter) {
      const uint2 lo = *reinterpret_cast<const uint2 *>(row + 2 * (4 * j));
      const uint2 hi = *reinterpret_cast<const uint2 *>(row + 2 * (F + 4 * j));
      re[0] = bf16lo(lo.x); re[1] = bf16hi(lo.x); re[2] = bf16lo(lo.y); re[3] = bf16hi(lo.y);
      im[0] = bf16lo(hi.x); im[1] = bf16hi(hi.x); im[2] = bf16lo(hi.y); im[3] = bf16hi(hi.y);
    } else {
      const uint4 w = *reinterpret_cast<const uint4 *>(row + 2 * (8 * j));
      re[0] = bf16lo(w.x); im[0] = bf16hi(w.x); re[1] = bf16lo(w.y); im[1] = bf16hi(w.y);
      re[2] = bf16lo(w.z); im[2] = bf16hi(w.z); re[3] = bf16lo(w.w); im[3] = bf16hi(w.w);
    }
  } else {
    if (!inter) {
      const float4 lo = *reinterpret_cast<const float4 *>(row + 4 * (4 * j));
      const float4 hi = *reinterpret_cast<const float4 *>(row + 4 * (F + 4 * j));
      re[0] = lo.x; re[1] = lo.y; re[2] = lo.z; re[3] = lo.w;
      im[0] = hi.x; im[1] = hi.y; im[2] = hi.z; im[3] = hi.w;
    } else {
      const float4 a = *reinterpret_cast<const float4 *>(row + 4 * (8 * j));
      const float4 b = *reinterpret_cast<const float4 *>(row + 4 * (8 * j + 4));
      re[0] = a.x; im[0] = a.y; re[1] = a.z; im[1] = a.w;
      re[2] = b.x; im[2] = b.y; re[3] = b.z; im[3] = b.w;
    }
  }
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

// Lane-private weights of the 4 bands a lane owns, for each of the G heads.
template <int G>
struct LaneWeights {
  float4 ar[G], ai[G], w[G];
};

template <int G, int F>
__device__ __forceinline__ void load_lane_weights(LaneWeights<G> &lw, const float *wts, int j) {
#pragma unroll
  for (int h = 0; h < G; ++h) {
    lw.ar[h] = *reinterpret_cast<const float4 *>(wts + (h * 3 + 0) * F + 4 * j);
    lw.ai[h] = *reinterpret_cast<const float4 *>(wts + (h * 3 + 1) * F + 4 * j);
    lw.w[h] = *reinterpret_cast<const float4 *>(wts + (h * 3 + 2) * F + 4 * j);
  }
}

// Scores the rows [0, nrows) of a tile in shared memory; s_{h, row0 + r} goes to
// scores[h * sstride + row0 + r].
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
    float re[4], im[4];
    if (valid) {
      load_bands<D, BF16>(tile + (long long)r * RB, j, inter, re, im);
    } else {
#pragma unroll
      for (int b = 0; b < 4; ++b) re[b] = im[b] = 0.f;
    }
    float mg[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) mg[b] = sqrt_approx(fmaf(re[b], re[b], im[b] * im[b]));
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float x = lw.ar[h].x * re[0];
      x = fmaf(lw.ar[h].y, re[1], x);
      x = fmaf(lw.ar[h].z, re[2], x);
      x = fmaf(lw.ar[h].w, re[3], x);
      x = fmaf(lw.ai[h].x, im[0], x);
      x = fmaf(lw.ai[h].y, im[1], x);
      x = fmaf(lw.ai[h].z, im[2], x);
      x = fmaf(lw.ai[h].w, im[3], x);
      x = fmaf(lw.w[h].x, mg[0], x);
      x = fmaf(lw.w[h].y, mg[1], x);
      x = fmaf(lw.w[h].z, mg[2], x);
      x = fmaf(lw.w[h].w, mg[3], x);
      acc[h] = x;
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
// for j in [e0, B) (rows below e0 are kept in place).  Destination chunks are
// processed in ascending order through a cp.async ring; every load of a chunk
// completes (wait_group + barrier) before any store of that chunk, and a load of
// a later chunk only reads slots >= that chunk's first destination, which no
// earlier store touches, because idx is strictly increasing (idx_j >= j).
__device__ __noinline__ void compact_unit(const CacheView &c, int l, int s, int g, const int *idx,
                                          int e0, int B, int N, char *ring) {
  const int rb = c.rb;
  const int pr = rb >> 4;                          // 16-byte pieces per row
  const int ch = kStageBytes / (2 * rb);           // rows per chunk (K and V)
  const int per = ch * pr;                         // pieces per tensor per chunk
  const int M = B - e0;
  if (M <= 0) return;
  const int nch = (M + ch - 1) / ch;
  const int tid = threadIdx.x, nt = blockDim.x;
  auto issue = [&](int cidx) {
    if (cidx < nch) {
      char *st = ring + (cidx % kStages) * kStageBytes;
      const int j0 = e0 + cidx * ch;
      for (int q = tid; q < 2 * per; q += nt) {
        const int tsr = q >= per;
        const int rem = q - tsr * per;
        const int r = rem / pr, p = rem - r * pr;
        const int j = j0 + r;
        if (j < B) {
          const int src = idx[j];
          const long long off = (src >= 0 && src < N) ? c.row_off(l, s, g, src) : -1;
          if (off >= 0) cp_async16(st + (long long)q * 16, (tsr ? c.v : c.k) + off + p * 16);
        }
      }
    }
    cp_async_commit();
  };
#pragma unroll 1
  for (int x = 0; x < kStages - 1; ++x) issue(x);
#pragma unroll 1
  for (int cidx = 0; cidx < nch; ++cidx) {
    issue(cidx + kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncthreads();
    const char *st = ring + (cidx % kStages) * kStageBytes;
    const int j0 = e0 + cidx * ch;
    for (int q = tid; q < 2 * per; q += nt) {
      const int tsr = q >= per;
      const int rem = q - tsr * per;
      const int r = rem / pr, p = rem - r * pr;
      const int j = j0 + r;
      if (j < B) {
        const long long off = c.row_off(l, s, g, j);
        if (off >= 0)
          *reinterpret_cast<uint4 *>((tsr ? c.v : c.k) + off + p * 16) =
              *reinterpret_cast<const uint4 *>(st + (long long)q * 16);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();
}

}  // namespace tri
