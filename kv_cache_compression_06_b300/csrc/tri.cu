// libtri: kernels and C ABI of the TriAttention periodic KV-cache compression step.
//
// Method source: "实现单卡4090跑通OpenClaw!英伟达&浙大等提出长上下文推理KV压缩新方法TriAttention"
// (yeyulingfeng.com), section 主要方法 (concentration / trig-series / two-part
// score / pruning paragraphs).  The operations are restated in include/tri.h.
//
// Kernels
//   calib_kernel         a0: per (layer, query head): center, mean |q_f|, R.
//   fused_kernel         a1..a5 for units whose scores fit one CTA's shared
//                        memory: weights -> TMA-streamed scoring -> z/max ->
//                        radix top-B -> in-place cp.async compaction.  Also the
//                        score-only variant behind tri_score.
//   score_tiles_kernel   a1+a2 for long units, 2048 keys per CTA: raw scores and
//                        per-tile (mean, M2) to the workspace.
//   zmax_kernel          a3 for long units (tri_score): Chan-merged moments -> agg.
//   select_compact_kernel a3..a5 for long units (from raw scores), tri_select_topb
//                        (from agg) and tri_compact_kv (from idx).
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "tri_path.cuh"

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
struct FusedArgs {
  CacheView c;
  const float *center, *R, *mag;
  int Hq;
  const int *t;
  int budget, mode, inter, capp;   // mode 0: compress, 1: score only
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
    bars = o;   o += 128;                 // kStages score barriers + kStages compaction barriers
    wts = o;    o += align_up(G * 3 * F * 4, 128);
    red = o;    o += 256;
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
__global__ void __launch_bounds__(kThreads, (G <= 4 ? 2 : 1)) fused_kernel(const FusedArgs a) {
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
  const int N = c.seq_len[s];
  const int B = a.budget;
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (a.mode == 0) {
    if (tid == 0 && a.new_len != nullptr && l == 0 && g == 0) a.new_len[s] = min(N, B);
    if (N <= B) {
      if (a.idx_out != nullptr)
        for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = j < N ? j : -1;
      return;
    }
  }
  if (N == 0) return;
  if (!c.blocks_ok(s, N)) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
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
  const uint32_t T = radix_select(keys, N, B, hist, sm, &ntie);
  const int e0 = build_kept(keys, N, B, T, ntie, idxs, sm);
  if (a.idx_out != nullptr)
    for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = idxs[j];
  // The ring was last read by generic loads (scoring); TMA writes it next.
  fence_proxy_async_smem();
  __syncthreads();
  if ((tid >> 5) == 0) compact_unit_tma(c, l, s, g, idxs, e0, B, N, ring, bars + kStages);
}

// ---------------------------------------------------------------- long units: tiles
struct TileArgs {
  CacheView c;
  const float *center, *R, *mag;
  int Hq;
  const int *t;
  int budget, skip_small, inter, ntiles;
  float *raw;      // [(u*G + h)*cap + i]
  float2 *part;    // [(u*ntiles + tile)*G + h] = (mean, M2) of the tile
  StepConst sc;
};

constexpr int kTileStride = kTileKeys + 4;   // per-head score stride (= 4 mod 32: no bank conflicts)

struct TileLayout {
  int bars, wts, red, scores, total;
  __host__ __device__ TileLayout(int G, int F) {
    int o = kRingBytes;
    bars = o;   o += 128;
    wts = o;    o += align_up(G * 3 * F * 4, 128);
    red = o;    o += 256;
    scores = o; o += G * kTileStride * 4;
    total = o;
  }
};

template <int G>
__device__ __forceinline__ void head_mean_m2(const float *scores, int stride, int n, float *red,
                                             float (&mu)[G], float (&m2)[G]) {
  float v[G];
#pragma unroll
  for (int h = 0; h < G; ++h) v[h] = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
#pragma unroll
    for (int h = 0; h < G; ++h) v[h] += scores[h * stride + i];
  }
  block_sum<G>(v, red);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mu[h] = v[h] / (float)n;
    v[h] = 0.f;
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float dl = scores[h * stride + i] - mu[h];
      v[h] = fmaf(dl, dl, v[h]);
    }
  }
  block_sum<G>(v, red);
#pragma unroll
  for (int h = 0; h < G; ++h) m2[h] = v[h];
}

template <int D, int G, bool BF16>
__global__ void __launch_bounds__(kThreads, (G <= 4 ? 2 : 1)) score_tiles_kernel(const TileArgs a) {
  constexpr int F = D / 2;
  extern __shared__ __align__(1024) char smem[];
  const TileLayout lay(G, F);
  char *ring = smem;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bars);
  float *wts = reinterpret_cast<float *>(smem + lay.wts);
  float *red = reinterpret_cast<float *>(smem + lay.red);
  float *scores = reinterpret_cast<float *>(smem + lay.scores);
  const CacheView &c = a.c;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int tile = blockIdx.x, u = blockIdx.y;
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  const int N = c.seq_len[s];
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (a.skip_small && N <= a.budget) return;
  const int i0 = tile * kTileKeys;
  if (i0 >= N) return;
  const int n = min(kTileKeys, N - i0);
  if (!c.blocks_ok(s, N)) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 32);
    fence_mbar_init();
  }
  build_weights<G, F>(wts, a.center, a.R, a.mag, a.Hq, l, g, a.t[s], a.sc);
  __syncthreads();
  LaneWeights<G> lw;
  load_lane_weights<G, F>(lw, wts, (tid & 31) % RowGeom<D, BF16>::LPR);
  if (!score_unit_rows<D, G, BF16>(c, l, s, g, i0, n, ring, bars, scores, kTileStride, lw,
                                   a.inter != 0))
    return;
  for (int i = tid; i < n; i += nt) {
#pragma unroll
    for (int h = 0; h < G; ++h) a.raw[((long long)u * G + h) * c.cap + i0 + i] = scores[h * kTileStride + i];
  }
  float mu[G], m2[G];
  head_mean_m2<G>(scores, kTileStride, n, red, mu, m2);
  if (tid == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h)
      a.part[((long long)u * a.ntiles + tile) * G + h] = make_float2(mu[h], m2[h]);
  }
}

// Chan's parallel combination of per-tile (count, mean, M2), in fp64; thread h < G
// writes mean and 1/std (0 if std = 0) of head h to mom[h], mom[8 + h].
__device__ __forceinline__ void merge_tile_moments(const float2 *part, long long u, int ntiles,
                                                   int G, int N, float *mom) {
  const int h = threadIdx.x;
  if (h < G) {
    double n = 0, mean = 0, M2 = 0;
    const int nt = (N + kTileKeys - 1) / kTileKeys;
    for (int t = 0; t < nt; ++t) {
      const double nb = (double)min(kTileKeys, N - t * kTileKeys);
      const float2 p = part[(u * ntiles + t) * G + h];
      if (n == 0) {
        n = nb;
        mean = p.x;
        M2 = p.y;
      } else {
        const double tot = n + nb, dl = (double)p.x - mean;
        mean += dl * nb / tot;
        M2 += (double)p.y + dl * dl * n * nb / tot;
        n = tot;
      }
    }
    const double sd = sqrt(M2 / n);
    mom[h] = (float)mean;
    mom[8 + h] = sd > 0 ? (float)(1.0 / sd) : 0.0f;
  }
}

struct ZArgs {
  int S, Hkv, G, ntiles;
  long long cap;
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
  const int i0 = tile * kTileKeys;
  if (i0 >= N) return;
  merge_tile_moments(a.part, u, a.ntiles, a.G, N, mom);
  __syncthreads();
  const int i1 = min(N, i0 + kTileKeys);
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    float z = -INFINITY;
    for (int h = 0; h < a.G; ++h) {
      const float zh = (a.raw[((long long)u * a.G + h) * a.cap + i] - mom[h]) * mom[8 + h];
      z = h == 0 ? zh : fmaxf(z, zh);
    }
    a.agg[(long long)u * a.cap + i] = z;
  }
}

// ---------------------------------------------------------------- select / compact
struct SCArgs {
  CacheView c;
  int G, budget, mode, ntiles, capp, bcap;   // mode 0: from raw (+compact), 1: from agg, 2: compact idx
  const float *raw;
  const float2 *part;
  const float *agg;
  const int *idx_in;
  int *idx_out, *new_len;
};

struct SCLayout {
  int bars, hist, sm, mom, keys, idx, total;
  __host__ __device__ SCLayout(int capp, int bcap) {
    int o = kRingBytes;
    bars = o; o += 128;
    hist = o; o += 1024;
    sm = o;   o += 256;
    mom = o;  o += 128;
    keys = o; o += align_up(capp * 4, 128);
    idx = o;  o += align_up(bcap * 4, 128);
    total = o;
  }
};

__global__ void __launch_bounds__(kSelThreads, 1) select_compact_kernel(const SCArgs a) {
  extern __shared__ __align__(1024) char smem[];
  const SCLayout lay(a.mode == 2 ? 0 : a.capp, a.bcap);
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
  const int N = c.seq_len[s];
  const int B = a.budget;
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (a.mode != 1 && tid == 0 && a.new_len != nullptr && l == 0 && g == 0) a.new_len[s] = min(N, B);
  if (N <= B) {
    if (a.mode != 2 && a.idx_out != nullptr)
      for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = j < N ? j : -1;
    return;
  }
  if (a.mode != 1 && !c.blocks_ok(s, N)) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&cbars[st], 1);
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
    if (tid == 0) sm[36] = B;
    if (__syncthreads_or(bad)) {
      if (tid == 0) set_status(TRI_ERR_INVALID);
      return;
    }
    for (int j = tid; j < B; j += nt)
      if (idxs[j] != j) atomicMin(&sm[36], j);
    __syncthreads();
    const int e0 = sm[36];
    __syncthreads();
    if ((tid >> 5) == 0) compact_unit_tma(c, l, s, g, idxs, e0, B, N, ring, cbars);
    return;
  }
  if (a.mode == 0) {
    merge_tile_moments(a.part, u, a.ntiles, a.G, N, mom);
    __syncthreads();
    for (int i = tid; i < N; i += nt) {
      float z = 0.f;
      for (int h = 0; h < a.G; ++h) {
        const float zh = (a.raw[((long long)u * a.G + h) * c.cap + i] - mom[h]) * mom[8 + h];
        z = h == 0 ? zh : fmaxf(z, zh);
      }
      keys[i] = score_key(z);
    }
  } else {
    for (int i = tid; i < N; i += nt) keys[i] = score_key(a.agg[(long long)u * c.cap + i]);
  }
  __syncthreads();
  int ntie;
  const uint32_t T = radix_select(keys, N, B, hist, sm, &ntie);
  const int e0 = build_kept(keys, N, B, T, ntie, idxs, sm);
  if (a.idx_out != nullptr)
    for (int j = tid; j < B; j += nt) a.idx_out[(long long)u * B + j] = idxs[j];
  if (a.mode == 0) {
    __syncthreads();
    if ((tid >> 5) == 0) compact_unit_tma(c, l, s, g, idxs, e0, B, N, ring, cbars);
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
  return v;
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
static int ntiles_of(const tri_cache *c) { return (int)((c->cap + kTileKeys - 1) / kTileKeys); }
static bool fused_fits(const tri_cache *c, int G) {
  return FusedLayout(G, c->d / 2, round32(c->cap)).total <= kMaxSmem;
}

struct SplitWs {
  size_t raw_off, part_off, total;
};
static SplitWs split_ws(const tri_cache *c, int G) {
  SplitWs w;
  const size_t raw = (size_t)units_of(c) * G * (size_t)c->cap * sizeof(float);
  const size_t part = (size_t)units_of(c) * ntiles_of(c) * G * sizeof(float2);
  w.raw_off = 0;
  w.part_off = (raw + 255) / 256 * 256;
  w.total = w.part_off + (part + 255) / 256 * 256;
  return w;
}

static tri_status launch_result() {
  return cudaGetLastError() == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

template <typename K>
static tri_status set_smem(K kernel, int bytes) {
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return TRI_ERR_CUDA;
  return TRI_OK;
}

template <int D, int G, bool BF16>
static tri_status run_fused(const FusedArgs &a, int64_t units, cudaStream_t st) {
  const FusedLayout lay(G, D / 2, a.capp);
  auto k = fused_kernel<D, G, BF16>;
  if (set_smem(k, lay.total) != TRI_OK) return TRI_ERR_CUDA;
  k<<<(unsigned)units, kThreads, lay.total, st>>>(a);
  return launch_result();
}

template <int D, int G, bool BF16>
static tri_status run_tiles(const TileArgs &a, int64_t units, cudaStream_t st) {
  const TileLayout lay(G, D / 2);
  auto k = score_tiles_kernel<D, G, BF16>;
  if (set_smem(k, lay.total) != TRI_OK) return TRI_ERR_CUDA;
  k<<<dim3((unsigned)a.ntiles, (unsigned)units), kThreads, lay.total, st>>>(a);
  return launch_result();
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
  const SCLayout lay(a.mode == 2 ? 0 : a.capp, a.bcap);
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
  a.ntiles = ntiles_of(c);
  a.sc = make_const(p, c->d);
  return a;
}

static int bcap_of(const tri_cache *c, int budget) {
  return round32(budget < c->cap ? budget : c->cap);
}

// ---------------------------------------------------------------- built-in scratch
// Scratch of tri_compress_step_static_scratch, for callers that cannot
// allocate.  In host code `g_static_scratch` names a host-side stand-in, not
// the device array: its device address is looked up per device below.
static __device__ __align__(256) unsigned char g_static_scratch[TRI_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
static std::mutex g_static_mu;
static void *g_static_addr[kMaxDevices];

// Device address of g_static_scratch on the current device, looked up once per
// device (with that device current) and cached.
static tri_status static_scratch_addr(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TRI_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TRI_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return TRI_ERR_CUDA;
    g_static_addr[dev] = p;
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
  *bytes = fused_fits(cache, G) ? 0 : split_ws(cache, G).total;
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
  const SplitWs w = split_ws(cache, G);
  if (ws == nullptr || ws_bytes < w.total) return TRI_ERR_WORKSPACE;
  TileArgs ta = tile_args(cache, stats, params);
  ta.skip_small = 0;
  ta.raw = raw != nullptr ? raw : reinterpret_cast<float *>(static_cast<char *>(ws) + w.raw_off);
  ta.part = reinterpret_cast<float2 *>(static_cast<char *>(ws) + w.part_off);
  if ((e = TRI_DISPATCH(run_tiles, cache->d, G, bf16, ta, units, stream)) != TRI_OK) return e;
  ZArgs z;
  z.S = cache->S;
  z.Hkv = cache->Hkv;
  z.G = G;
  z.ntiles = ta.ntiles;
  z.cap = cache->cap;
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
  if (mode != TRI_COMPACT_ORDERED) return TRI_ERR_UNSUPPORTED;
  if (new_len != nullptr && new_len == cache->seq_len) return TRI_ERR_INVALID;
  SCArgs a;
  std::memset(&a, 0, sizeof(a));
  a.c = make_view(cache);
  a.budget = budget;
  a.mode = 2;
  a.capp = 0;
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
  if (mode != TRI_COMPACT_ORDERED) return TRI_ERR_UNSUPPORTED;
  if (new_len != nullptr && new_len == cache->seq_len) return TRI_ERR_INVALID;
  const int G = stats->Hq / cache->Hkv;
  const bool bf16 = cache->dtype == TRI_BF16;
  const int64_t units = units_of(cache);
  if (fused_fits(cache, G)) {
    FusedArgs a = fused_args(cache, stats, params);
    a.mode = 0;
    a.idx_out = idx_out;
    a.new_len = new_len;
    return TRI_DISPATCH(run_fused, cache->d, G, bf16, a, units, stream);
  }
  const SplitWs w = split_ws(cache, G);
  if (ws == nullptr || ws_bytes < w.total) return TRI_ERR_WORKSPACE;
  SCArgs sa;
  std::memset(&sa, 0, sizeof(sa));
  sa.c = make_view(cache);
  sa.G = G;
  sa.budget = params->budget;
  sa.mode = 0;
  sa.ntiles = ntiles_of(cache);
  sa.capp = round32(cache->cap);
  sa.bcap = bcap_of(cache, params->budget);
  if (SCLayout(sa.capp, sa.bcap).total > kMaxSmem) return TRI_ERR_UNSUPPORTED;
  TileArgs ta = tile_args(cache, stats, params);
  ta.skip_small = 1;
  ta.raw = reinterpret_cast<float *>(static_cast<char *>(ws) + w.raw_off);
  ta.part = reinterpret_cast<float2 *>(static_cast<char *>(ws) + w.part_off);
  if ((e = TRI_DISPATCH(run_tiles, cache->d, G, bf16, ta, units, stream)) != TRI_OK) return e;
  sa.raw = ta.raw;
  sa.part = ta.part;
  sa.idx_out = idx_out;
  sa.new_len = new_len;
  return run_select_compact(sa, units, stream);
}

tri_status tri_compress_step_static_scratch(const tri_cache *cache, const tri_stats *stats,
                                            const tri_params *params, tri_compact_mode mode,
                                            int32_t *idx_out, int32_t *new_len,
                                            cudaStream_t stream) {
  tri_status e;
  if ((e = check_cache(cache, true, true)) != TRI_OK) return e;
  if (mode != TRI_COMPACT_ORDERED) return TRI_ERR_UNSUPPORTED;
  size_t need = 0;
  if ((e = tri_workspace_bytes(cache, stats, params, &need)) != TRI_OK) return e;
  if (need == 0) return tri_compress_step(cache, stats, params, mode, idx_out, new_len, nullptr, 0, stream);
  if (need > (size_t)TRI_STATIC_SCRATCH_BYTES) return TRI_ERR_WORKSPACE;
  void *ws = nullptr;
  if ((e = static_scratch_addr(&ws)) != TRI_OK) return e;
  return tri_compress_step(cache, stats, params, mode, idx_out, new_len, ws,
                           (size_t)TRI_STATIC_SCRATCH_BYTES, stream);
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
      cudaSuccess)
    return TRI_ERR_CUDA;
  return TRI_OK;
}

}  // extern "C"
