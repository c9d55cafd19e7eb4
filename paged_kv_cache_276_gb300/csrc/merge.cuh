// Exact merge of split-K partials (one warp per output row):
//   out = sum_p O_p 2^(m_p - M) / sum_p l_p 2^(m_p - M),  M = max_p m_p,
// the log-sum-exp combination of partial softmax results over disjoint key
// ranges (the partials carry their running max in log2 units).  The lanes read
// the partitions' (max, sum) pairs in parallel, then each lane keeps eight
// partitions' slices of O in flight, so a merge costs a few memory round trips
// instead of two per partition.  An empty partition (max -inf) weighs 0 and its
// O is never read.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace pkv {

template <int D>
__device__ __forceinline__ void merge_partials(const float2 *ml, const float *o_row, int nparts, __nv_bfloat16 *dst,
                                               int lane) {
  constexpr int PER = D / 32;
  const float *o = o_row + lane * PER;
  float M = -INFINITY;
  for (int i = lane; i < nparts; i += 32) M = fmaxf(M, ml[i].x);
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float den = 0.f, accv[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) accv[k] = 0.f;
  for (int base = 0; base < nparts; base += 32) {
    // lane i holds the weight of partition base + i (0 for an empty slot)
    const int i = base + lane;
    float f = 0.f;
    if (i < nparts) {
      const float2 v = ml[i];
      f = v.x == -INFINITY ? 0.f : exp2f(v.x - M);
      den += v.y * f;
    }
    const int cnt = min(32, nparts - base);
    for (int j0 = 0; j0 < cnt; j0 += 8) {
      float w[8];
      float x[8][PER];
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // eight independent loads in flight
        w[j] = __shfl_sync(0xffffffffu, f, (j0 + j) & 31);
        const bool use = j0 + j < cnt && w[j] != 0.f;
#pragma unroll
        for (int k = 0; k < PER; ++k) x[j][k] = 0.f;
        if (use) {
          const float *src = o + static_cast<size_t>(base + j0 + j) * D;
          if constexpr (PER == 4) {
            const float4 t = *reinterpret_cast<const float4 *>(src);
            x[j][0] = t.x; x[j][1] = t.y; x[j][2] = t.z; x[j][3] = t.w;
          } else {
            const float2 t = *reinterpret_cast<const float2 *>(src);
            x[j][0] = t.x; x[j][1] = t.y;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int k = 0; k < PER; ++k) accv[k] += w[j] * x[j][k];
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
  for (int k = 0; k < PER; ++k) dst[lane * PER + k] = __float2bfloat16_rn(accv[k] * inv);
}

}  // namespace pkv
