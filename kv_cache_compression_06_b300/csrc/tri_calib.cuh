// Streamed calibration of the per-band statistics (a0 at scale).
//
// Method source: "实现单卡4090跑通OpenClaw!英伟达&浙大等提出长上下文推理KV压缩新方法TriAttention"
// (yeyulingfeng.com), section 主要方法: concentration paragraph (pre-RoPE Q/K
// cluster around fixed non-zero centers; concentration measured by the mean
// resultant length R) and the pipeline summary (the centers, norms and
// concentration are offline statistics).
//
// The statistics are means over the calibration samples, so they are carried
// as sums that chunks of samples add to in any order:
//   acc[l][h][f][0..7] = (sum re q_f, sum im q_f, sum |q_f|,
//                         sum re q_f/|q_f|, sum im q_f/|q_f|  (samples with |q_f| > 0),
//                         count of samples with |q_f| > 0, count of samples, 0)
// in fp64.  Finalising divides: center = sum q / n, mag = sum |q| / n,
// R = |sum q/|q|| / count_nonzero (0 when that count is 0).
#pragma once

#include "tri_device.cuh"

namespace tri {

constexpr int kCalibAcc = 8;          // doubles per (layer, head, band)
constexpr int kCalibThreads = 256;
constexpr int kCalibChunk = 512;      // samples per CTA of the accumulate kernel

// One chunk of samples into the accumulator.  Grid (H, L, ceil(n / kCalibChunk)).
// A row (one sample of one head) is read by TPR = F/2 threads, each owning two
// adjacent bands, with 4-byte (bf16) or 8-byte (fp32) loads per half, so a warp
// reads whole rows in coalesced segments.  Per-thread sums are fp32 over at most
// kCalibChunk / (rows per CTA) samples, then fp64 across the CTA and one fp64
// atomic add per (band, quantity).
template <int D, bool BF16, bool INTER>
__global__ void __launch_bounds__(kCalibThreads) calib_accumulate_kernel(const void *q, long long n,
                                                                         long long sample_stride,
                                                                         long long layer_stride, int H,
                                                                         double *acc) {
  constexpr int F = D / 2, TPR = F / 2, RPC = kCalibThreads / TPR;   // threads per row, rows per CTA pass
  __shared__ double red[6][kCalibThreads];
  const int h = blockIdx.x, l = blockIdx.y;
  const int tid = threadIdx.x, j = tid % TPR, r = tid / TPR;
  const long long i0 = (long long)blockIdx.z * kCalibChunk;
  const long long i1 = min(n, i0 + kCalibChunk);
  float s[2][5] = {{0.f, 0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f, 0.f}};
  int cnt[2] = {0, 0};
  for (long long i = i0 + r; i < i1; i += RPC) {
    const long long base = (long long)l * layer_stride + i * sample_stride + (long long)h * D;
    float re[2], im[2];
    if constexpr (BF16) {
      const uint16_t *p = static_cast<const uint16_t *>(q) + base;
      if constexpr (!INTER) {
        const uint32_t a = *reinterpret_cast<const uint32_t *>(p + 2 * j);
        const uint32_t b = *reinterpret_cast<const uint32_t *>(p + F + 2 * j);
        re[0] = bf16lo(a); re[1] = bf16hi(a);
        im[0] = bf16lo(b); im[1] = bf16hi(b);
      } else {
        const uint2 a = *reinterpret_cast<const uint2 *>(p + 4 * j);
        re[0] = bf16lo(a.x); im[0] = bf16hi(a.x);
        re[1] = bf16lo(a.y); im[1] = bf16hi(a.y);
      }
    } else {
      const float *p = static_cast<const float *>(q) + base;
      if constexpr (!INTER) {
        const float2 a = *reinterpret_cast<const float2 *>(p + 2 * j);
        const float2 b = *reinterpret_cast<const float2 *>(p + F + 2 * j);
        re[0] = a.x; re[1] = a.y;
        im[0] = b.x; im[1] = b.y;
      } else {
        const float4 a = *reinterpret_cast<const float4 *>(p + 4 * j);
        re[0] = a.x; im[0] = a.y;
        re[1] = a.z; im[1] = a.w;
      }
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float m = sqrtf(re[e] * re[e] + im[e] * im[e]);
      s[e][0] += re[e];
      s[e][1] += im[e];
      s[e][2] += m;
      if (m > 0.f) {
        s[e][3] += re[e] / m;
        s[e][4] += im[e] / m;
        ++cnt[e];
      }
    }
  }
  // CTA reduction per band: the RPC threads of band pair j add up in fp64
  for (int e = 0; e < 2; ++e) {
#pragma unroll
    for (int k = 0; k < 5; ++k) red[k][tid] = (double)s[e][k];
    red[5][tid] = (double)cnt[e];
    __syncthreads();
    if (tid < TPR) {
      double t[6] = {0, 0, 0, 0, 0, 0};
      for (int rr = 0; rr < RPC; ++rr)
#pragma unroll
        for (int k = 0; k < 6; ++k) t[k] += red[k][rr * TPR + tid];
      const int f = 2 * tid + e;
      double *a = acc + (((long long)l * H + h) * F + f) * kCalibAcc;
#pragma unroll
      for (int k = 0; k < 6; ++k)
        if (t[k] != 0.0) atomicAdd(a + k, t[k]);
      atomicAdd(a + 6, (double)(i1 - i0));
    }
    __syncthreads();
  }
}

__global__ void calib_add_kernel(double *acc, const double *other, long long count) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += (long long)gridDim.x * blockDim.x)
    acc[i] += other[i];
}

__global__ void calib_zero_kernel(double *acc, long long count) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += (long long)gridDim.x * blockDim.x)
    acc[i] = 0.0;
}

// Statistics from the sums; one thread per (layer, head, band).  Bands that saw
// no sample (count 0) get center 0, mag 0, R 0.
__global__ void calib_finalize_kernel(const double *acc, long long bands, float *center, float *R, float *mag) {
  for (long long o = (long long)blockIdx.x * blockDim.x + threadIdx.x; o < bands; o += (long long)gridDim.x * blockDim.x) {
    const double *a = acc + o * kCalibAcc;
    const double n = a[6], nz = a[5];
    center[2 * o] = n > 0 ? (float)(a[0] / n) : 0.f;
    center[2 * o + 1] = n > 0 ? (float)(a[1] / n) : 0.f;
    mag[o] = n > 0 ? (float)(a[2] / n) : 0.f;
    R[o] = nz > 0 ? (float)(sqrt(a[3] * a[3] + a[4] * a[4]) / nz) : 0.f;
  }
}

}  // namespace tri
