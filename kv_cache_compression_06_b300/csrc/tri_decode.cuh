// Decode-loop kernels around the compression step: appending one token's K/V
// to the cache and single-query attention over the cache.
//
// Method source: "实现单卡4090跑通OpenClaw!英伟达&浙大等提出长上下文推理KV压缩新方法TriAttention"
// (yeyulingfeng.com), section 主要方法: pruning paragraph (during online decoding
// the compression runs once every 128 generated tokens when the cache exceeds
// the budget) and trig-series paragraph (the RoPE attention logit).  These
// kernels are the decode side of that loop; the attention itself is the
// standard softmax attention over post-RoPE keys.
//
// Append: for every unit (l, s, g) the new token's pre-RoPE key is rotated to
// its position p_s (band f times e^{i*omega_f*p_s}, phase reduced modulo 2*pi in
// fp64) and written with its value into slot N_s = seq_len[s].
//
// Attention: out[l][s][h] = sum_i w_i v_i, w_i = softmax_i(scale * q~_h . k~_i) over
// the unit's N slots, q~ = the query rotated to p_s.  Split-K over the keys: a
// CTA takes one slice of one unit; each consumer warp keeps a running max, sum
// and output per head (online softmax) over its 16-key tiles; the CTA merges
// its warps, and a second kernel merges the slices.  Both products run on the
// tensor cores (m16n8k16, fp32 accumulation) with the 16 rows of the A operand
// = [hi parts of the G heads | lo parts], so the query and the probabilities
// enter as hi + lo bf16 pairs (about 2^-16 relative) against the exact bf16
// keys and values:
//   S = [q~hi; q~lo] K^T   (keys as the N dimension, ldmatrix of K rows)
//   O = [p hi; p lo] V     (keys as the K dimension; the S accumulators of two
//                           8-key tiles are the A fragment; ldmatrix.trans of V)
// and the hi and lo rows of one head sit in the same lane (rows r and r + 8).
#pragma once

#include "tri_mma.cuh"

namespace tri {

// ---------------------------------------------------------------- append
struct AppendArgs {
  CacheView c;
  const void *k_new, *v_new;   // [L][S][Hkv][d], cache dtype
  const int *pos;              // [S]
  int *seq_len_out;            // [S]
  int *pos_out;                // [S] or null
  int inter;
  StepConst sc;
};

// One warp per unit.  Lane j owns bands j, j + 32 (F = 64) or j (F = 32).
template <bool BF16>
__global__ void __launch_bounds__(32) append_kv_kernel(const AppendArgs a) {
  const CacheView &c = a.c;
  const int u = blockIdx.x, lane = threadIdx.x;
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  const bool writer = lane == 0 && l == 0 && g == 0;
  const int N = c.seq_len[s];
  const long long off = (N >= 0 && N < c.cap) ? c.row_off(l, s, g, N) : -1;
  if (off < 0) {   // full, or its block id is out of range: nothing is appended
    if (lane == 0) set_status(TRI_ERR_BOUNDS);
    if (writer) {
      a.seq_len_out[s] = N;
      if (a.pos_out != nullptr) a.pos_out[s] = a.pos[s];
    }
    return;
  }
  const int F = c.d / 2;
  const int p = a.pos[s];
  const long long src = (long long)u * c.d;
  for (int f = lane; f < F; f += 32) {
    const int ire = a.inter ? 2 * f : f, iim = a.inter ? 2 * f + 1 : f + F;
    const float2 e = reduced_cis(a.sc.omega[f] * (double)p);
    float re, im;
    if constexpr (BF16) {
      const uint16_t *kp = static_cast<const uint16_t *>(a.k_new) + src;
      re = __uint_as_float((uint32_t)kp[ire] << 16);
      im = __uint_as_float((uint32_t)kp[iim] << 16);
      uint16_t *dst = reinterpret_cast<uint16_t *>(c.k + off);
      const uint32_t pr = pack_bf16x2(re * e.x - im * e.y, re * e.y + im * e.x);
      dst[ire] = (uint16_t)(pr & 0xffffu);
      dst[iim] = (uint16_t)(pr >> 16);
    } else {
      const float *kp = static_cast<const float *>(a.k_new) + src;
      re = kp[ire];
      im = kp[iim];
      float *dst = reinterpret_cast<float *>(c.k + off);
      dst[ire] = re * e.x - im * e.y;
      dst[iim] = re * e.y + im * e.x;
    }
  }
  const int es = BF16 ? 2 : 4;
  const char *vs = static_cast<const char *>(a.v_new) + src * es;
  for (int x = lane; x < c.rb / 4; x += 32)
    reinterpret_cast<uint32_t *>(c.v + off)[x] = reinterpret_cast<const uint32_t *>(vs)[x];
  if (writer) {
    a.seq_len_out[s] = N + 1;
    if (a.pos_out != nullptr) a.pos_out[s] = p + 1;
  }
}

// ---------------------------------------------------------------- attention
constexpr int kDecConsumers = 4;                              // consumer warps
constexpr int kDecThreads = (kDecConsumers + 1) * 32;         // + one producer warp
constexpr int kDecStages = 3;                                 // ring of K+V stages
constexpr int kDecStageBytes = 2 * kStageBytes;               // K (16 KB) then V (16 KB)

struct DecodeArgs {
  CUtensorMap kmap, vmap;   // 128B-swizzled maps of K and V (as the score kernel's K map)
  CacheView c;
  const void *q;            // [L][S][Hq][d] pre-RoPE queries, bf16
  const int *pos;           // [S]
  int Hq, nsplit, inter;
  float qscale;             // softmax scale * log2(e)
  float *out;               // [L][S][Hq][d] fp32
  float *part;              // [units][nsplit][G][d + 2]: O (unnormalised), max, sum (base-2 logits)
  StepConst sc;
};

// The warps' final states ([consumer][G][D + 2] floats) overlay the ring once
// every stage has been consumed.
struct DecLayout {
  int bars, q, total;
  __host__ __device__ DecLayout(int G, int D) {
    int o = kDecStages * kDecStageBytes;
    bars = o;  o += 128;
    q = o;     o += G * D * 4;
    total = o;
  }
};

// Keys [k0, k1) of this split for a unit of N keys: slices of a multiple of the
// stage's rows.
template <int TR>
__device__ __forceinline__ void dec_slice(int N, int nsplit, int sp, int &k0, int &k1) {
  const int per = ((N + nsplit - 1) / nsplit + TR - 1) / TR * TR;
  k0 = min(N, sp * per);
  k1 = min(N, k0 + per);
}

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, 2) decode_attn_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int F = D / 2, TR = kStageBytes / (2 * D), TPS = TR / 16;   // rows and 16-key tiles per stage
  constexpr int KS = D / 16, NT = D / 8;
  extern __shared__ __align__(1024) char smem[];
  const DecLayout lay(G, D);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint64_t *empty = full + kDecStages;
  volatile int *fail = reinterpret_cast<volatile int *>(empty + kDecStages);
  volatile int *issued = fail + 1;
  float *qs = reinterpret_cast<float *>(smem + lay.q);
  float *mrg = reinterpret_cast<float *>(smem);   // after the pipeline: overlays the ring
  const CacheView &c = a.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sp = blockIdx.x, u = blockIdx.y;
  const int g = u % c.Hkv, s = (u / c.Hkv) % c.S, l = u / (c.Hkv * c.S);
  if (timed_out()) return;
  const int N = c.seq_len[s];
  if (N < 0 || N > c.cap) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  int k0, k1;
  dec_slice<TR>(N, a.nsplit, sp, k0, k1);
  if (k1 > k0 && !c.blocks_ok(s, k1 - k0, k0)) {
    if (tid == 0) set_status(TRI_ERR_BOUNDS);
    return;
  }
  if (tid == 0) {
    for (int st = 0; st < kDecStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kDecConsumers);
    }
    *fail = 0;
    *issued = 0;
    fence_mbar_init();
  }
  // the G queries of this KV head, rotated to p_s and scaled, fp32
  {
    const int p = a.pos[s];
    const uint16_t *qb = static_cast<const uint16_t *>(a.q) + (((long long)l * c.S + s) * a.Hq + (long long)g * G) * D;
    for (int x = tid; x < G * F; x += kDecThreads) {
      const int h = x / F, f = x - h * F;
      const int ire = a.inter ? 2 * f : f, iim = a.inter ? 2 * f + 1 : f + F;
      const float re = __uint_as_float((uint32_t)qb[h * D + ire] << 16);
      const float im = __uint_as_float((uint32_t)qb[h * D + iim] << 16);
      const float2 e = reduced_cis(a.sc.omega[f] * (double)p);
      qs[h * D + ire] = (re * e.x - im * e.y) * a.qscale;
      qs[h * D + iim] = (re * e.y + im * e.x) * a.qscale;
    }
  }
  __syncthreads();
  const int nst = (k1 - k0 + TR - 1) / TR;
  const long long urow0 = (long long)u * c.cap;
  // consumer state: output accumulators of [hi; lo] rows, running max and sum of head hr
  const int hr = lane >> 2, kq = 2 * (lane & 3);
  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  if (warp == kDecConsumers) {
    // producer: K and V rows of one stage under one barrier arrival
    int t = 0;
    for (; t < nst; ++t) {
      const int st = t % kDecStages;
      if (*fail || (t >= kDecStages && !mbar_wait(&empty[st], (uint32_t)(((t / kDecStages) - 1) & 1)))) {
        *fail = 1;
        break;
      }
      const int row0 = k0 + t * TR, nrows = min(TR, k1 - row0);
      char *dst = smem + st * kDecStageBytes;
      if (lane == 0) mbar_arrive_expect_tx(&full[st], 2u * stage_sw_bytes<D>(c, nrows));
      __syncwarp();
      issue_stage_sw<D>(c, &a.kmap, l, s, g, urow0, row0, nrows, dst, &full[st], lane);
      issue_stage_sw<D>(c, &a.vmap, l, s, g, urow0, row0, nrows, dst + kStageBytes, &full[st], lane);
    }
    if (lane == 0) *issued = t;
  } else {
    // A fragments of [q~ hi; q~ lo]: rows r = lane/4 (hi of head r) and r + 8 (lo of head r)
    uint32_t qa[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
      if (hr < G) {
        const float *qr = qs + hr * D + 16 * ks + kq;
        v0 = qr[0];
        v1 = qr[1];
        v2 = qr[8];
        v3 = qr[9];
      }
      split_bf16x2(v0, v1, qa[ks][0], qa[ks][1]);
      split_bf16x2(v2, v3, qa[ks][2], qa[ks][3]);
    }
    const uint32_t ring = smem_u32(smem);
    const int blk = c.paged() && D == 128 ? c.block : 0;
    for (int t = 0; t < nst; ++t) {
      const int st = t % kDecStages;
      if (!*fail && !mbar_wait(&full[st], (uint32_t)((t / kDecStages) & 1))) *fail = 1;
      const uint32_t kst = ring + st * kDecStageBytes, vst = kst + kStageBytes;
      const int row_base = k0 + t * TR;
      for (int tile = warp; tile < TPS && !*fail; tile += kDecConsumers) {
        const int r0 = 16 * tile;                     // stage row of this tile's first key
        const int nvalid = min(16, k1 - row_base - r0);
        if (nvalid <= 0) break;
        if (nvalid < 16) {
          // rows past the slice may hold stale, non-finite values: clear their V
          // rows (their logits are masked below)
          char *vrow = smem + st * kDecStageBytes + kStageBytes;
          for (int x = lane; x < (16 - nvalid) * (D / 8); x += 32) {
            const int rr = r0 + nvalid + x / (D / 8), col = (x % (D / 8)) * 8;
            const SwRow sr = sw_row<TR>(rr, blk);
            *reinterpret_cast<uint4 *>(vrow + (sw_addr(0, sr, col))) = make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
        // S tiles of keys r0..r0+7 and r0+8..r0+15: lanes address K rows
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int mtx = lane >> 3;
          const SwRow sr = sw_row<TR>(r0 + (lane & 7) + (mtx >> 1) * 8, blk);
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(b0, b1, b2, b3, sw_addr(kst, sr, 16 * ks + (mtx & 1) * 8));
            mma_bf16(sc[0], qa[ks], b0, b1);
            mma_bf16(sc[1], qa[ks], b2, b3);
          }
        }
        // logits of head hr at keys r0 + 8 j + kq + {0, 1}: hi row + lo row
        float sv[2][2];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = 8 * j + kq + e;
            sv[j][e] = key < nvalid ? sc[j][e] + sc[j][2 + e] : -INFINITY;
          }
        float mx = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run, mx);            // finite: key r0 is valid
        const float corr = exp2f(m_run - m_new);          // 0 on the first tile
        float pv[2][2], ps = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            pv[j][e] = exp2f(sv[j][e] - m_new);
            ps += pv[j][e];
          }
        ps += __shfl_xor_sync(0xffffffffu, ps, 1);
        ps += __shfl_xor_sync(0xffffffffu, ps, 2);
        l_run = l_run * corr + ps;
        m_run = m_new;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          o[nt][0] *= corr;
          o[nt][1] *= corr;
          o[nt][2] *= corr;
          o[nt][3] *= corr;
        }
        uint32_t pa[4];
        split_bf16x2(pv[0][0], pv[0][1], pa[0], pa[1]);
        split_bf16x2(pv[1][0], pv[1][1], pa[2], pa[3]);
        // O += P V: ldmatrix.trans of V rows; lanes address key rows
        {
          const int mtx = lane >> 3;
          const SwRow sr = sw_row<TR>(r0 + (lane & 7) + (mtx & 1) * 8, blk);
#pragma unroll
          for (int dt = 0; dt < D / 16; ++dt) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(b0, b1, b2, b3, sw_addr(vst, sr, 16 * dt + (mtx >> 1) * 8));
            mma_bf16(o[2 * dt], pa, b0, b1);
            mma_bf16(o[2 * dt + 1], pa, b2, b3);
          }
        }
      }
      // the stage may be refilled by TMA (V rows cleared above were written by
      // generic stores)
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }
  __syncthreads();   // every warp is done with the ring (no copy is in flight unless a wait failed)
  if (warp < kDecConsumers && !*fail && hr < G) {
    // this warp's state: per head hr, O = hi rows + lo rows
    float *mw = mrg + warp * G * (D + 2);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mw[hr * (D + 2) + 8 * nt + kq] = o[nt][0] + o[nt][2];
      mw[hr * (D + 2) + 8 * nt + kq + 1] = o[nt][1] + o[nt][3];
    }
    if ((lane & 3) == 0) {
      mw[hr * (D + 2) + D] = m_run;
      mw[hr * (D + 2) + D + 1] = l_run;
    }
  }
  if (*fail) {
    if (tid == 0) {
      const int iss = *issued;
      for (int st = 0; st < kDecStages && st < iss; ++st) {
        const int last = st + ((iss - 1 - st) / kDecStages) * kDecStages;
        mbar_wait(&full[st], (uint32_t)((last / kDecStages) & 1));
      }
    }
    return;
  }
  __syncthreads();   // the warps' states are in shared memory
  // merge the warps: per (head, element)
  const int Gq = g * G;
  for (int x = tid; x < G * D; x += kDecThreads) {
    const int h = x / D, e = x - h * D;
    float mstar = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecConsumers; ++w) mstar = fmaxf(mstar, mrg[(w * G + h) * (D + 2) + D]);
    float ov = 0.f, lv = 0.f;
    if (mstar > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecConsumers; ++w) {
        const float *mw = mrg + (w * G + h) * (D + 2);
        const float mw_ = mw[D];
        if (mw_ > -INFINITY) {
          const float f = exp2f(mw_ - mstar);
          ov += mw[e] * f;
          lv += mw[D + 1] * f;
        }
      }
    }
    if (a.nsplit == 1) {
      a.out[(((long long)l * c.S + s) * a.Hq + Gq + h) * D + e] = lv > 0.f ? ov / lv : 0.f;
    } else {
      float *pp = a.part + (((long long)u * a.nsplit + sp) * G + h) * (D + 2);
      pp[e] = ov;
      if (e == 0) {
        pp[D] = mstar;
        pp[D + 1] = lv;
      }
    }
  }
}

// Merges the slices of each unit: grid units, threads over (head, element).
__global__ void __launch_bounds__(256) decode_merge_kernel(const float *part, int nsplit, int G, int D, int S,
                                                           int Hkv, int Hq, float *out) {
  const int u = blockIdx.x;
  const int g = u % Hkv, s = (u / Hkv) % S, l = u / (Hkv * S);
  for (int x = threadIdx.x; x < G * D; x += blockDim.x) {
    const int h = x / D, e = x - h * D;
    float mstar = -INFINITY;
    for (int sp = 0; sp < nsplit; ++sp) mstar = fmaxf(mstar, part[(((long long)u * nsplit + sp) * G + h) * (D + 2) + D]);
    float ov = 0.f, lv = 0.f;
    if (mstar > -INFINITY) {
      for (int sp = 0; sp < nsplit; ++sp) {
        const float *pp = part + (((long long)u * nsplit + sp) * G + h) * (D + 2);
        if (pp[D] > -INFINITY) {
          const float f = exp2f(pp[D] - mstar);
          ov += pp[e] * f;
          lv += pp[D + 1] * f;
        }
      }
    }
    out[(((long long)l * S + s) * Hq + g * G + h) * D + e] = lv > 0.f ? ov / lv : 0.f;
  }
}

}  // namespace tri
