// Warp-level attention step shared by the decode kernels: one 16-key tile
// (or BS keys) of K and V staged by TMA with the 128-byte swizzle, the GQA
// query group as the MMA N dimension, online softmax in fp32 with exp2.
//
// Math: softmax(scale * q K^T) V (x321.org "The serving bottleneck is not just
// FLOPs", section "First understand what the KV cache is storing"), computed
// block by block with a running max and sum so that every K/V byte is read
// once.
#pragma once

#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "ptx.cuh"

namespace pkv {
namespace attend {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleSlack = 8.f;  // log2 units: weights stay below 256

// Shared-memory address of the 16-byte chunk `dchunk` of tile row `row`.  The
// tile is staged as boxes of R rows, each [64-column half][R rows][128 bytes]
// (HALVES halves), with the TMA 128-byte swizzle: chunk index XOR row mod 8
// inside each 1024-byte atom; every box starts 1024-byte aligned.
template <int R, int HALVES>
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int dchunk) {
  return base + (row / R) * (HALVES * R * 128) + (dchunk >> 3) * (R * 128) + (row % R) * 128 +
         ((((dchunk & 7) ^ (row & 7))) << 4);
}

template <int D, int NT>
struct WarpAcc {
  float m[NT][2];  // running max of the thread's two columns per n-tile (log2 units)
  float l[NT][2];  // thread-partial running sum
  float o[D / 16][NT][4];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int md = 0; md < D / 16; ++md) o[md][nt][0] = o[md][nt][1] = o[md][nt][2] = o[md][nt][3] = 0.f;
    }
  }
};

// Running-max update shared by the block steps.  The reference max moves only
// when a column's block max exceeds it by more than kRescaleSlack (log2 units),
// so most blocks skip rescaling the accumulators.  Exact: numerator and
// denominator use the same reference, and every weight stays below
// 2^kRescaleSlack.  bmax holds the thread's column maxima (reduced here over
// the lanes sharing a column); msub receives the reference to subtract.
template <int D, int NT>
__device__ __forceinline__ void online_max_update(WarpAcc<D, NT> &acc, float (&bmax)[NT][2],
                                                  float (&msub)[NT][2]) {
  float alpha[NT][2];
  bool rescale = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float b = bmax[nt][e];
      b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, 4));
      b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, 8));
      b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, 16));
      const float m = acc.m[nt][e];
      alpha[nt][e] = 1.f;
      if (b > m + kRescaleSlack) {  // also true while m is -inf and b finite
        alpha[nt][e] = m == -INFINITY ? 0.f : exp2f(m - b);
        acc.m[nt][e] = b;
        rescale = true;
      }
      msub[nt][e] = acc.m[nt][e] == -INFINITY ? 0.f : acc.m[nt][e];
    }
  if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        acc.l[nt][e] *= alpha[nt][e];
#pragma unroll
        for (int md = 0; md < D / 16; ++md) {
          acc.o[md][nt][e] *= alpha[nt][e];
          acc.o[md][nt][e + 2] *= alpha[nt][e];
        }
      }
  }
}

// One staged unit of BS keys (boxes of R rows, see swz) for one warp's columns.
//   qf:    B fragments of Q^T (column = query row) per n-tile and 16-wide d step
//   valid: keys of this unit that hold tokens (1..BS)
//   vis:   keys of this unit visible to each of the thread's columns
template <int D, int BS, int NT, int R = BS>
__device__ __forceinline__ void attend_block(WarpAcc<D, NT> &acc,
                                             const uint32_t (&qf)[NT][D / 16][2], uint32_t kbase,
                                             uint32_t vbase, int valid, const int (&vis)[NT][2],
                                             float scale_log2, int lane) {
  constexpr int MT = BS / 16;
  const int r8 = lane & 7, mi = lane >> 3;
  const int g4 = lane >> 2, c4 = lane & 3;

  // S^T[key][col] = K[key][:] . Q[col][:]; even and odd d-steps accumulate in
  // separate registers so the two MMA chains overlap
  float sc[MT][NT][4], sc2[MT][NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[mt][nt][i] = sc2[mt][nt][i] = 0.f;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t a[4];
      ldsm_x4(swz<R, D / 64>(kbase, mt * 16 + r8 + (mi & 1) * 8, ks * 2 + (mi >> 1)), a);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (ks & 1) mma_bf16_16816(sc2[mt][nt], a, qf[nt][ks][0], qf[nt][ks][1]);
        else mma_bf16_16816(sc[mt][nt], a, qf[nt][ks][0], qf[nt][ks][1]);
      }
    }
  }

  // scale, mask, block max per column
  float bmax[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) bmax[nt][0] = bmax[nt][1] = -INFINITY;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int key = mt * 16 + g4 + (i >> 1) * 8;
        const float s = key < vis[nt][i & 1] ? (sc[mt][nt][i] + sc2[mt][nt][i]) * scale_log2 : -INFINITY;
        sc[mt][nt][i] = s;
        bmax[nt][i & 1] = fmaxf(bmax[nt][i & 1], s);
      }
  float msub[NT][2];
  online_max_update<D, NT>(acc, bmax, msub);

  // probabilities -> bf16 -> B fragments of P^T (movmatrix transposes the
  // accumulator layout into the operand layout)
  uint32_t pb[MT][NT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint32_t lo = pack_bf16x2(exp2f(sc[mt][nt][0] - msub[nt][0]), exp2f(sc[mt][nt][1] - msub[nt][1]));
      const uint32_t hi = pack_bf16x2(exp2f(sc[mt][nt][2] - msub[nt][0]), exp2f(sc[mt][nt][3] - msub[nt][1]));
      // the running sum uses the same rounded weights as the P V product
      const float2 flo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&lo));
      const float2 fhi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi));
      acc.l[nt][0] += flo.x + fhi.x;
      acc.l[nt][1] += flo.y + fhi.y;
      pb[mt][nt][0] = movmatrix_trans(lo);
      pb[mt][nt][1] = movmatrix_trans(hi);
    }

  // O^T[d][col] += V^T[d][key] P^T[key][col]
#pragma unroll
  for (int kt = 0; kt < MT; ++kt) {
    const bool tail = valid < (kt + 1) * 16;  // warp-uniform
    const int k0 = kt * 16 + 2 * c4;
    const uint32_t m0 = (k0 < valid ? 0x0000FFFFu : 0u) | (k0 + 1 < valid ? 0xFFFF0000u : 0u);
    const uint32_t m1 = (k0 + 8 < valid ? 0x0000FFFFu : 0u) | (k0 + 9 < valid ? 0xFFFF0000u : 0u);
#pragma unroll
    for (int md = 0; md < D / 16; ++md) {
      uint32_t a[4];
      ldsm_x4_trans(swz<R, D / 64>(vbase, kt * 16 + r8 + (mi >> 1) * 8, md * 2 + (mi & 1)), a);
      if (tail) {  // slots past the sequence end were never written: keep NaNs out
        a[0] &= m0;
        a[1] &= m0;
        a[2] &= m1;
        a[3] &= m1;
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc.o[md][nt], a, pb[kt][nt][0], pb[kt][nt][1]);
    }
  }
}

}  // namespace attend
}  // namespace pkv
