// Device helpers shared by every libtri kernel: inline-PTX wrappers for
// mbarriers, bulk (TMA) copies and cp.async, bounded waits, the device status
// word, block-wide reductions and scans, and the order-preserving float key.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/tri.h"

namespace tri {

constexpr int kFusedThreads = 256;             // CTA size of the fused short-unit kernel
#ifndef TRI_FUSED_MMA
#define TRI_FUSED_MMA 1
#endif
constexpr int kFusedMma = TRI_FUSED_MMA;       // short units of bf16 rotate-half caches on the tensor cores
constexpr int kConsumerWarps = 8;              // warps that score keys (long-unit tiles)
constexpr int kProducerWarp = kConsumerWarps;   // the warp that issues the K loads
constexpr int kThreads = (kConsumerWarps + 1) * 32;   // CTA size of the long-unit score kernel
constexpr int kStageBytes = 16384;              // one pipeline stage (K tile or K+V chunk)
constexpr int kStages = 4;                      // stages of the score ring
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kCompactStages = 12;              // stages of the long-unit compaction ring, at least
constexpr int kMaxCompactStages = 13;           // and at most (bounded by shared memory)
// Keys per CTA in the split (long-unit) path: the tile's G rows of fp32 scores
// sit in shared memory next to the 64 KB ring; 1024 keys for G = 8 keep two CTAs
// per SM.
__host__ __device__ constexpr int tile_keys_for(int G) { return G >= 8 ? 1024 : 2048; }
constexpr int kTilesPerCta = 4;   // tiles of one unit per CTA in the tensor-core score kernel
constexpr int kSelThreads = 512;                // CTA size of the select/compact kernel
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // bounded device waits: 2 s

// First device-side error since the last clear (0 = TRI_OK).
__device__ int g_tri_status = 0;
// Nonzero once some wait has given up since the last clear, whichever error
// the status word holds (an earlier error keeps its place there).
__device__ int g_tri_timeout = 0;

__device__ __forceinline__ void set_status(int code) { atomicCAS(&g_tri_status, 0, code); }

// True once some wait has given up (and the flags are not yet cleared):
// kernels that wait on copies then leave at once instead of waiting out their
// own limits one CTA after another, and kernels that consume a list an earlier
// kernel of the step wrote do not trust lists that kernel may have left
// unwritten.
__device__ __forceinline__ bool timed_out() {
  return *reinterpret_cast<volatile int *>(&g_tri_timeout) != 0;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with `parity` to complete.  Gives up after limit_ns,
// records TRI_ERR_TIMEOUT and returns false (the caller then leaves the CTA).
__device__ __noinline__ bool mbar_wait_for(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int k = 0; k < 64; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      set_status(TRI_ERR_TIMEOUT);
      atomicExch(&g_tri_timeout, 1);
      return false;
    }
  }
}
// The kernels' wait: mbar_wait_for with the library's limit (kWaitLimitNs).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// ---------------------------------------------------------------- bulk copy (TMA, untiled)
// global -> shared, completion counted in bytes on `bar`.  Both addresses 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Tiled 4-D tensor load (TMA) of the box at coordinates (c0, c1, c2, c3) of the
// tensor map `map` (a kernel parameter) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// Tiled 2-D tensor load (TMA) of the box at (c0, c1) into shared memory.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// Tiled 5-D tensor load (TMA) of the box at (c0, .., c4) into shared memory.
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            int c4, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar))
      : "memory");
}

// Tiled 2-D gather (TMA tile::gather4): loads rows r0..r3 (box one row high,
// `col` the first element) of the 2-D tensor map `map` into four consecutive
// rows at dst, completing on `bar`.
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *map, int col, int r0, int r1,
                                            int r2, int r3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

// Tiled 4-D tensor store (TMA) of the box at (c0, c1, c2, c3) from shared memory,
// tracked by the issuing thread's bulk async-groups.  Coordinates must be >= 0.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                             const void *src) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
               : "memory");
}

// shared -> global bulk store, tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until at most N of this thread's bulk groups are still incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- cp.async (16 B)
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Arrives on `bar` once all of this thread's earlier cp.async copies have landed;
// the arrival counts toward the barrier's expected count (noinc).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- arithmetic
__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed pairs of fp32 in one 64-bit register (low word = first element) and
// the sm_100-family paired fp32 arithmetic on them.
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Order-preserving map of an fp32 score to u32 (larger float -> larger key);
// NaN maps to 0 (ranks lowest), -0 and +0 map to the same key.
__device__ __forceinline__ uint32_t score_key(float f) {
  if (f != f) return 0u;
  uint32_t u = __float_as_uint(f);
  if (f == 0.0f) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ---------------------------------------------------------------- block reductions
template <int G>
__device__ __forceinline__ void block_sum(float (&v)[G], float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float x = v[h];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    v[h] = x;
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) red[warp * G + h] = v[h];
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float t = 0.f;
    for (int w = 0; w < nw; ++w) t += red[w * G + h];
    v[h] = t;
  }
  __syncthreads();
}

// Barrier over the first n threads of the CTA (n a multiple of 32) on named
// barrier `id` (1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// block_sum over the first nthreads threads only, synchronised on named barrier 1.
template <int G>
__device__ __forceinline__ void group_sum(float (&v)[G], float *red, int nthreads) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = nthreads >> 5;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float x = v[h];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    v[h] = x;
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) red[warp * G + h] = v[h];
  }
  named_sync(1, nthreads);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float t = 0.f;
    for (int w = 0; w < nw; ++w) t += red[w * G + h];
    v[h] = t;
  }
  named_sync(1, nthreads);
}

// Exclusive prefix sum of one int per thread across the CTA; *total receives
// the CTA-wide sum.  sm needs 32 ints.
__device__ __forceinline__ int block_excl_scan(int v, int *sm, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? sm[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sm[lane] = w;
  }
  __syncthreads();
  const int base = warp ? sm[warp - 1] : 0;
  *total = sm[nw - 1];
  __syncthreads();
  return base + x - v;
}

}  // namespace tri
