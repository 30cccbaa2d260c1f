// Merge of the per-unit partials of decode attention (split attention over the work list).
//
// Every warp that worked on a unit left, per query head, an unnormalised partial: the running
// maximum m (log2 units), l = sum_t 2^(s_t - m) and acc[c] = sum_t 2^(s_t - m) v_tc over its
// tokens.  The output is sum_w 2^(m_w - M) acc_w / sum_w 2^(m_w - M) l_w with M = max_w m_w
// (log-sum-exp combination), written as fp16.
#pragma once

#include <cuda_fp16.h>

#include "kvq_internal.h"

namespace kvq {

// One warp merges the n partial slots of HG query heads bh0 .. bh0+HG-1.  Slots are taken in
// rounds of 32: one slot's (m, l) per lane, a running maximum across rounds, then every lane's
// four channels of each slot with the slot's weight (sixteen loads in flight).
template <int HG>
__device__ __forceinline__ void merge_partials(const DecodeParams& p, int64_t bh0, int n, int lane) {
  constexpr int D = kHeadDim;
  constexpr unsigned all = 0xffffffffu;
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    const float* ml = p.part_ml + (bh0 + h) * p.max_slots * 2;
    const float* pacc = p.part_acc + (bh0 + h) * p.max_slots * D + 4 * lane;
    float Mrun = -INFINITY, L = 0.0f, a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
    for (int base = 0; base < n; base += 32) {
      const int nb = min(32, n - base);
      float2 mine = make_float2(-INFINITY, 0.0f);
      if (lane < nb) mine = __ldcg(reinterpret_cast<const float2*>(ml + 2 * (base + lane)));
      float Mr = mine.x;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) Mr = fmaxf(Mr, __shfl_xor_sync(all, Mr, off));
      const float Mnew = fmaxf(Mrun, Mr);
      if (Mrun != -INFINITY && Mnew != Mrun) {
        const float so = exp2f(Mrun - Mnew);
        L *= so;
        a0 *= so;
        a1 *= so;
        a2 *= so;
        a3 *= so;
      }
      Mrun = Mnew;
      const float f = mine.x == -INFINITY ? 0.0f : exp2f(mine.x - Mnew);
      L = fmaf(f, mine.y, L);
#pragma unroll 16
      for (int sp = 0; sp < nb; ++sp) {
        const float fs = __shfl_sync(all, f, sp);
        const float4 v = __ldcg(reinterpret_cast<const float4*>(pacc + (int64_t)(base + sp) * D));
        a0 = fmaf(fs, v.x, a0);
        a1 = fmaf(fs, v.y, a1);
        a2 = fmaf(fs, v.z, a2);
        a3 = fmaf(fs, v.w, a3);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(all, L, off);
    const float inv = 1.0f / L;
    const __half2 o01 = __floats2half2_rn(a0 * inv, a1 * inv), o23 = __floats2half2_rn(a2 * inv, a3 * inv);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&o01);
    packed.y = *reinterpret_cast<const uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(p.out + (bh0 + h) * D + 4 * lane) = packed;
  }
}

}  // namespace kvq
