// Key scoring on the tensor cores (bf16 caches, rotate-half bands).
//
// The two-part score of a key is a dot product of a per-key feature vector
// with a per-head weight vector (trig-series paragraph and two-part score
// paragraph of the method's write-up):
//   s_{h,i} = sum_f Re A_{h,f} * Re k~_{i,f} + Im A_{h,f} * Im k~_{i,f} + W_{h,f} * |k~_{i,f}|
// i.e. S = X Y with X_i = (Re k~_i, Im k~_i, |k~_i|) (3F features) and
// Y = (Re A; Im A; W) (3F x G).  Per 16 keys it runs as m16n8k16 bf16 MMAs with
// fp32 accumulation:
//   - Re/Im k~ are the cache's own bf16 values (exact operands);
//   - every weight is split into hi = bf16(w) and lo = bf16(w - hi), and the
//     MMA sees both (G <= 4: N = 8 columns = [hi of the G heads | lo of the G
//     heads], summed after; G = 8: two MMAs);
//   - |k~| is computed in fp32 from the A fragments themselves (the Re and Im
//     fragments of a band block hold the same (key, band) positions) and split
//     into hi + lo as well; the lo x lo product is dropped.
// The split keeps every product to about 2^-16 relative; accumulation is fp32.
//
// K arrives in shared memory through 128B-swizzled tensor copies: a stage is
// [half][TR rows][128 B] (d = 128: half 0 = Re (elements 0..63), half 1 = Im;
// d = 64: one half holding both), the 16-byte chunk c of row r stored at chunk
// c ^ (r & 7), which makes the ldmatrix row reads conflict-free.  A paged
// d = 128 stage is one such [half][blk rows][128 B] group per cache block (one
// tensor copy per block carries both halves).
#pragma once

#include "tri_path.cuh"

namespace tri {

__device__ __forceinline__ void ldmatrix_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                            uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// ldmatrix_x4 with each 8x8 matrix transposed on the way to the registers.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                                  uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A * B for one m16n8k16 tile (A 16x16 row-major bf16, B 16x8 bf16, fp32 D).
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 -> one bf16x2 register (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Splits two fp32 values into bf16x2 hi and lo parts (hi + lo ~ v to 2^-16).
__device__ __forceinline__ void split_bf16x2(float v0, float v1, uint32_t &hi, uint32_t &lo) {
  hi = pack_bf16x2(v0, v1);
  lo = pack_bf16x2(v0 - bf16lo(hi), v1 - bf16hi(hi));
}

// B fragments (weights) of one warp, for D / 16 trig k-steps (Re then Im
// blocks of 16 bands) and F / 16 magnitude k-steps.
//   G <= 4: bt[ks] = [hi | lo] columns; bm[ks] = [hi | lo]; bm2[ks] = [hi | 0]
//   G == 8: bt/bm = hi; the lo fragments stay in shared memory ([KT + KM][32
//           lanes] pairs at `lo`: trig k-steps, then magnitude k-steps; `lo`
//           addresses this lane's pair of k-step 0), read back per k-step,
//           which keeps the kernel within 96 registers
template <int D, int G>
struct MmaWeights {
  static constexpr int KT = D / 16, KM = D / 32;
  uint32_t bt[KT][2], bm[KM][2], bm2[G == 8 ? 1 : KM][2];
  uint32_t lo;
};

__device__ __forceinline__ void lds_v2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}

// Builds this lane's B fragments from wts [G][3][F] (Re A, Im A, W).  Lane l
// holds column n = l / 4 and rows k = 2 (l % 4) + {0, 1, 8, 9} of each k-step.
// Called by all nc consumer threads (named barrier 1); for G == 8 the first
// consumer warp (`writer`) then overwrites the start of wts with the lo trig
// fragments (wts is dead once every consumer holds its fragments).
// lo_dst (G == 8): where the lo fragments go instead of the start of wts
// (12 x 32 lanes x 8 bytes), for callers whose wts region is reused after.
template <int D, int G>
__device__ __forceinline__ void load_mma_weights(MmaWeights<D, G> &w, float *wts, int nc, bool writer,
                                                 float *lo_dst = nullptr) {
  constexpr int F = D / 2;
  const int lane = threadIdx.x & 31, n = lane >> 2, k0 = 2 * (lane & 3);
  const int kk[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
  // column n of the split weights: head h, part (0 = hi, 1 = lo), or none
  const int h = G == 8 ? n : (n & 3);
  const bool live = G == 8 || h < G;
  const int part = G == 8 ? 0 : (n >> 2);
  uint32_t lo[G == 8 ? MmaWeights<D, G>::KT + MmaWeights<D, G>::KM : 1][2];
#pragma unroll
  for (int ks = 0; ks < MmaWeights<D, G>::KT; ++ks) {
    // features 16 ks + k: Re A for bands < F, Im A after
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int f = 16 * ks + kk[e];
      v[e] = live ? (f < F ? wts[(h * 3 + 0) * F + f] : wts[(h * 3 + 1) * F + f - F]) : 0.f;
    }
    uint32_t h01, l01, h23, l23;
    split_bf16x2(v[0], v[1], h01, l01);
    split_bf16x2(v[2], v[3], h23, l23);
    w.bt[ks][0] = part ? l01 : h01;
    w.bt[ks][1] = part ? l23 : h23;
    if constexpr (G == 8) {
      lo[ks][0] = l01;
      lo[ks][1] = l23;
    }
  }
#pragma unroll
  for (int ks = 0; ks < MmaWeights<D, G>::KM; ++ks) {
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = live ? wts[(h * 3 + 2) * F + 16 * ks + kk[e]] : 0.f;
    uint32_t h01, l01, h23, l23;
    split_bf16x2(v[0], v[1], h01, l01);
    split_bf16x2(v[2], v[3], h23, l23);
    if constexpr (G == 8) {
      w.bm[ks][0] = h01;
      w.bm[ks][1] = h23;
      lo[MmaWeights<D, G>::KT + ks][0] = l01;
      lo[MmaWeights<D, G>::KT + ks][1] = l23;
    } else {
      w.bm[ks][0] = part ? l01 : h01;
      w.bm[ks][1] = part ? l23 : h23;
      w.bm2[ks][0] = part ? 0u : h01;
      w.bm2[ks][1] = part ? 0u : h23;
    }
  }
  w.lo = 0;
  if constexpr (G == 8) {
    uint2 *dst = reinterpret_cast<uint2 *>(lo_dst != nullptr ? lo_dst : wts);
    named_sync(1, nc);   // every consumer has read wts
    if (writer) {
#pragma unroll
      for (int ks = 0; ks < MmaWeights<D, G>::KT + MmaWeights<D, G>::KM; ++ks)
        dst[ks * 32 + lane] = make_uint2(lo[ks][0], lo[ks][1]);
    }
    named_sync(1, nc);
    w.lo = smem_u32(dst) + lane * 8;
  }
}

// Position of one row in a swizzled stage: byte offset of its 128-byte segment
// in half 0, the stride between halves, and its swizzle key.  blk = 0: the
// stage is [half][TR rows]; blk > 0 (paged, d = 128): [block][half][blk rows].
struct SwRow {
  int off, hstride, key;
};
template <int TR>
__device__ __forceinline__ SwRow sw_row(int row, int blk) {
  SwRow r;
  if (blk > 0) {
    const int b = row / blk, rr = row - b * blk;
    r.off = b * blk * 256 + rr * 128;
    r.hstride = blk * 128;
    r.key = rr & 7;
  } else {
    r.off = row * 128;
    r.hstride = TR * 128;
    r.key = row & 7;
  }
  return r;
}
// Byte address of element column `col` (a multiple of 8) of that row.
__device__ __forceinline__ uint32_t sw_addr(uint32_t stage, const SwRow &r, int col) {
  return stage + (uint32_t)(r.off + (col >> 6) * r.hstride + ((((col & 63) >> 3) ^ r.key) << 4));
}

// Bytes that issue_stage_sw's copies of rows [row0, row0 + nrows) deliver (a
// dense stage always carries its whole box; rows past the tensor read as zero).
template <int D>
__device__ __forceinline__ uint32_t stage_sw_bytes(const CacheView &c, int nrows) {
  constexpr int NH = D / 64;
  if (!c.paged()) return (uint32_t)kStageBytes;
  const int blk = c.block, nblk = (nrows + blk - 1) / blk;
  return (uint32_t)(nblk * blk * 128 * NH);
}

// Issues the tensor copies of rows [row0, row0 + nrows) of unit (l, s, g) of
// the tensor behind `map` into a swizzled stage of kStageBytes (two boxes of
// 64 elements per row for d = 128, one for d = 64), completing on `full`; the
// caller has announced the bytes.  Dense: the unit's slot 0 is row urow0 of the
// 2-D view; rows past the unit are loaded too, rows past the tensor read as
// zero.  Paged: one copy per block carrying both halves.  All lanes of the
// calling warp take part.
template <int D>
__device__ __forceinline__ void issue_stage_sw(const CacheView &c, const CUtensorMap *map, int l, int s, int g,
                                               long long urow0, int row0, int nrows, char *dst, uint64_t *full,
                                               int lane) {
  constexpr int TR = kStageBytes / (2 * D), NH = D / 64;   // rows per stage, halves per row
  if (!c.paged()) {
    if (lane == 0) {
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) tma_load_2d(dst + hh * TR * 128, map, 64 * hh, (int)(urow0 + row0), full);
    }
    return;
  }
  const int blk = c.block, nblk = (nrows + blk - 1) / blk;
  if (lane < nblk) {
    const int b = c.bt[(long long)s * c.max_blocks + row0 / blk + lane];
    const int z = (int)((long long)l * c.nblocks + b);
    if constexpr (NH == 2)
      tma_load_5d(dst + lane * blk * 256, map, 0, 0, 0, g, z, full);   // [half][blk rows] of one block
    else
      tma_load_4d(dst + lane * blk * 128, map, 0, g, 0, z, full);
  }
}

// One stage of K for the score kernels: the arrival with its byte count, then
// the copies.  Called by all lanes of the producer warp.
template <int D>
__device__ __forceinline__ void produce_stage_sw(const CacheView &c, const CUtensorMap *map, int l, int s,
                                                 int g, long long urow0, int row0, int nrows, char *dst,
                                                 uint64_t *full, int lane) {
  if (lane == 0) mbar_arrive_expect_tx(full, stage_sw_bytes<D>(c, nrows));
  __syncwarp();
  issue_stage_sw<D>(c, map, l, s, g, urow0, row0, nrows, dst, full, lane);
}

// Scores the 16 keys at stage rows [r0, r0 + 16) into this lane's fragment
// values: o[e] is the score of key r0 + lane/4 + 8 (e >> 1) for head
// n + (e & 1), n = 2 (lane % 4).  G = 8: every lane's n is a head; G <= 4: the
// lo columns are folded into the hi ones, and lanes with n >= G hold nothing
// meaningful.
template <int D, int G, int TR>
__device__ __forceinline__ void score_tile_mma_frag(uint32_t stage, int r0, const MmaWeights<D, G> &w, int blk,
                                                    float (&o)[4]) {
  constexpr int F = D / 2;
  const int lane = threadIdx.x & 31;
  const int lrow = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;   // ldmatrix row of this lane
  const int lcol = (lane >> 4) * 8;                           // and column offset
  const SwRow sr = sw_row<TR>(lrow, D == 128 ? blk : 0);
  // two accumulators (trig, magnitude): two shorter dependent MMA chains
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, accm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < F / 16; ++ks) {
    uint32_t re[4], im[4];
    ldmatrix_x4(re[0], re[1], re[2], re[3], sw_addr(stage, sr, 16 * ks + lcol));
    ldmatrix_x4(im[0], im[1], im[2], im[3], sw_addr(stage, sr, F + 16 * ks + lcol));
    mma_bf16(acc, re, w.bt[ks][0], w.bt[ks][1]);
    mma_bf16(acc, im, w.bt[F / 16 + ks][0], w.bt[F / 16 + ks][1]);
    if constexpr (G == 8) {
      uint32_t lr[2], li[2];
      lds_v2(lr, w.lo + ks * 256);
      lds_v2(li, w.lo + (F / 16 + ks) * 256);
      mma_bf16(acc, re, lr[0], lr[1]);
      mma_bf16(acc, im, li[0], li[1]);
    }
    // |k~| at the same fragment positions, split into hi + lo
    uint32_t mh[4], ml[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float a, b;
      upk(ffma2(pk(bf16lo(im[e]), bf16hi(im[e])), pk(bf16lo(im[e]), bf16hi(im[e])),
                fmul2(pk(bf16lo(re[e]), bf16hi(re[e])), pk(bf16lo(re[e]), bf16hi(re[e])))),
          a, b);
      split_bf16x2(sqrt_approx(a), sqrt_approx(b), mh[e], ml[e]);
    }
    mma_bf16(accm, mh, w.bm[ks][0], w.bm[ks][1]);
    if constexpr (G == 8) {
      uint32_t lm[2];
      lds_v2(lm, w.lo + (D / 16 + ks) * 256);
      mma_bf16(accm, mh, lm[0], lm[1]);                 // hi x lo
      mma_bf16(accm, ml, w.bm[ks][0], w.bm[ks][1]);     // lo x hi
    } else {
      mma_bf16(accm, ml, w.bm2[ks][0], w.bm2[ks][1]);   // lo x hi (lo columns get 0)
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) acc[e] += accm[e];
  if constexpr (G == 8) {
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = acc[e];
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = acc[e] + __shfl_xor_sync(0xffffffffu, acc[e], 2);   // hi + lo
  }
}

// Scores the 16 keys at stage rows [r0, r0 + 16) (row0 + r0 + i is the key's
// index in the caller's score rows); rows at or past nrows are not stored.
template <int D, int G, int TR>
__device__ __forceinline__ void score_tile_mma(uint32_t stage, int r0, int nrows, int row0, float *scores,
                                               int sstride, const MmaWeights<D, G> &w, int blk) {
  const int lane = threadIdx.x & 31;
  float o[4];
  score_tile_mma_frag<D, G, TR>(stage, r0, w, blk, o);
  // D fragment: o[0..1] row r, columns n, n + 1; o[2..3] row r + 8.
  const int r = lane >> 2, n = 2 * (lane & 3);
  if (G == 8 || n < 4) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = r0 + r + (e >> 1) * 8, h = n + (e & 1);
      if (h < G && row < nrows) scores[h * sstride + row0 + row] = o[e];
    }
  }
}

}  // namespace tri
