// Distance-preference curves of the trig-series paragraph.
//
// Method source: "实现单卡4090跑通OpenClaw!英伟达&浙大等提出长上下文推理KV压缩新方法TriAttention"
// (yeyulingfeng.com), section 主要方法, trig-series paragraph: under RoPE the
// attention logit is a sum over frequency bands of a function of the query-key
// distance; with Q/K replaced by their calibrated centers it becomes a
// trigonometric series in that distance, the head's distance-preference curve,
// which the write-up reports to reconstruct the attention's distance preference
// with high correlation.
//
// For query head h of layer l (KV head g = h / G) and distance delta >= 0:
//   center curve C(delta) = sum_f Re[cq_{h,f} * conj(ck_{g,f}) * e^{i*omega_f*delta}]
//   logit curve  E(delta) = mean over i in [0, n - delta) of the RoPE logit of the
//                query sample at position i + delta against the key sample at
//                position i of one sequence
//                = (1/(n - delta)) sum_f Re[X_f(delta) * e^{i*omega_f*delta}],
//                X_f(delta) = sum_i q_{i+delta,f} * conj(k_{i,f})   (pre-RoPE bands)
//   corr = Pearson correlation of C and E over delta = 0..n_delta-1.
#pragma once

#include "tri_path.cuh"

namespace tri {

constexpr int kCurveDeltas = 32;      // distances per CTA of the logit-curve kernel
constexpr int kCurveRows = 16;        // samples per shared-memory pass (static smem < 48 KB)
constexpr int kCurveThreads = 256;    // 32 distances x 8 band groups

// Band f of row `row` (elements of `dtype`) as (re, im) floats.
template <bool BF16, bool INTER>
__device__ __forceinline__ float2 load_band(const void *rowp, int f, int F) {
  const int ire = INTER ? 2 * f : f, iim = INTER ? 2 * f + 1 : f + F;
  if constexpr (BF16) {
    const uint16_t *p = static_cast<const uint16_t *>(rowp);
    return make_float2(__uint_as_float((uint32_t)p[ire] << 16), __uint_as_float((uint32_t)p[iim] << 16));
  } else {
    const float *p = static_cast<const float *>(rowp);
    return make_float2(p[ire], p[iim]);
  }
}

// Logit curve.  Grid (ceil(n_delta / 32), Hq, L).  Thread (dl = tid % 32,
// fg = tid / 32) accumulates X_f(delta0 + dl) for the F/8 bands of group fg over
// passes of kCurveRows samples staged in shared memory as fp32 bands (query rows
// [i + delta0, i + delta0 + 48), key rows [i, i + 16)); the bands are then rotated by
// e^{i*omega_f*delta} (fp64 phase reduction), summed over the groups and divided
// by n - delta.  q: [L][n][Hq][d], k: [L][n][Hkv][d].
template <int D, bool BF16, bool INTER>
__global__ void __launch_bounds__(kCurveThreads) logit_curve_kernel(const void *q, const void *k, long long n,
                                                                    int Hq, int Hkv, int n_delta,
                                                                    const StepConst sc, float *curve) {
  constexpr int F = D / 2, BPT = F / 8, QR = kCurveRows + kCurveDeltas, PAD = F + 1;
  constexpr int ES = BF16 ? 2 : 4;
  __shared__ float2 qs[QR * PAD];
  __shared__ float2 ks[kCurveRows * PAD];
  __shared__ float red[8][kCurveDeltas];
  const int h = blockIdx.y, l = blockIdx.z, g = h / (Hq / Hkv);
  const int tid = threadIdx.x, dl = tid % kCurveDeltas, fg = tid / kCurveDeltas;
  const int d0 = blockIdx.x * kCurveDeltas;
  const int delta = d0 + dl;
  const char *qb = static_cast<const char *>(q) + ((long long)l * n * Hq + h) * D * ES;
  const char *kb = static_cast<const char *>(k) + ((long long)l * n * Hkv + g) * D * ES;
  const long long qrow = (long long)Hq * D * ES, krow = (long long)Hkv * D * ES;
  float xr[BPT], xi[BPT];
#pragma unroll
  for (int b = 0; b < BPT; ++b) xr[b] = xi[b] = 0.f;
  // keys i < n - d0 can pair with a query of some distance in this CTA
  for (long long i0 = 0; i0 < n - d0; i0 += kCurveRows) {
    __syncthreads();
    for (int x = tid; x < QR * F; x += kCurveThreads) {
      const int r = x / F, f = x - r * F;
      const long long qi = i0 + d0 + r;
      qs[r * PAD + f] = qi < n ? load_band<BF16, INTER>(qb + qi * qrow, f, F) : make_float2(0.f, 0.f);
    }
    for (int x = tid; x < kCurveRows * F; x += kCurveThreads) {
      const int r = x / F, f = x - r * F;
      const long long ki = i0 + r;
      ks[r * PAD + f] = ki < n ? load_band<BF16, INTER>(kb + ki * krow, f, F) : make_float2(0.f, 0.f);
    }
    __syncthreads();
    if (delta < n_delta) {
      // pairs (query i + delta, key i) with i + delta < n; rows past n are zero
      const int rmax = (int)min((long long)kCurveRows, n - delta - i0);
      for (int r = 0; r < rmax; ++r) {
        const float2 *qrow_s = qs + (r + dl) * PAD + fg * BPT;
        const float2 *krow_s = ks + r * PAD + fg * BPT;
#pragma unroll
        for (int b = 0; b < BPT; ++b) {
          const float2 a = qrow_s[b], c = krow_s[b];
          xr[b] = fmaf(a.x, c.x, fmaf(a.y, c.y, xr[b]));
          xi[b] = fmaf(a.y, c.x, fmaf(-a.x, c.y, xi[b]));
        }
      }
    }
  }
  float part = 0.f;
  if (delta < n_delta) {
#pragma unroll
    for (int b = 0; b < BPT; ++b) {
      const float2 e = reduced_cis(sc.omega[fg * BPT + b] * (double)delta);
      part += xr[b] * e.x - xi[b] * e.y;
    }
  }
  red[fg][dl] = part;
  __syncthreads();
  if (tid < kCurveDeltas && d0 + tid < n_delta) {
    float t = 0.f;
#pragma unroll
    for (int x = 0; x < 8; ++x) t += red[x][tid];
    const long long pairs = n - (d0 + tid);
    curve[((long long)l * Hq + h) * n_delta + d0 + tid] = pairs > 0 ? t / (float)pairs : 0.f;
  }
}

// Center curve.  Grid (Hq, L); threads over delta.  cq: [L][Hq][F][2],
// ck: [L][Hkv][F][2].  The products cq * conj(ck) are formed once per CTA.
__global__ void __launch_bounds__(256) center_curve_kernel(const float *cq, const float *ck, int Hq, int Hkv,
                                                           int F, int n_delta, const StepConst sc, float *curve) {
  __shared__ float2 prod[64];
  const int h = blockIdx.x, l = blockIdx.y, g = h / (Hq / Hkv);
  for (int f = threadIdx.x; f < F; f += blockDim.x) {
    const long long oq = ((long long)l * Hq + h) * F + f, ok = ((long long)l * Hkv + g) * F + f;
    const float ar = cq[2 * oq], ai = cq[2 * oq + 1], br = ck[2 * ok], bi = ck[2 * ok + 1];
    prod[f] = make_float2(ar * br + ai * bi, ai * br - ar * bi);
  }
  __syncthreads();
  for (int dlt = threadIdx.x; dlt < n_delta; dlt += blockDim.x) {
    float t = 0.f;
    for (int f = 0; f < F; ++f) {
      const float2 e = reduced_cis(sc.omega[f] * (double)dlt);
      t += prod[f].x * e.x - prod[f].y * e.y;
    }
    curve[((long long)l * Hq + h) * n_delta + dlt] = t;
  }
}

// Pearson correlation of two curves per head, in fp64, two passes (means, then
// centered sums).  Grid (Hq * L); 256 threads.  A curve with zero variance gives 0.
__global__ void __launch_bounds__(256) curve_corr_kernel(const float *a, const float *b, int n_delta, float *corr) {
  __shared__ double red[3][256];
  const long long base = (long long)blockIdx.x * n_delta;
  const int tid = threadIdx.x;
  auto reduce = [&](double (&s)[3]) {
#pragma unroll
    for (int k = 0; k < 3; ++k) red[k][tid] = s[k];
    __syncthreads();
    for (int w = 128; w >= 1; w >>= 1) {
      if (tid < w)
#pragma unroll
        for (int k = 0; k < 3; ++k) red[k][tid] += red[k][tid + w];
      __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) s[k] = red[k][0];
    __syncthreads();
  };
  double s[3] = {0, 0, 0};
  for (int x = tid; x < n_delta; x += blockDim.x) {
    s[0] += a[base + x];
    s[1] += b[base + x];
  }
  reduce(s);
  const double ma = s[0] / n_delta, mb = s[1] / n_delta;
  s[0] = s[1] = s[2] = 0;
  for (int x = tid; x < n_delta; x += blockDim.x) {
    const double u = a[base + x] - ma, v = b[base + x] - mb;
    s[0] += u * u;
    s[1] += v * v;
    s[2] += u * v;
  }
  reduce(s);
  if (tid == 0) corr[blockIdx.x] = (s[0] > 0 && s[1] > 0) ? (float)(s[2] / sqrt(s[0] * s[1])) : 0.f;
}

}  // namespace tri
