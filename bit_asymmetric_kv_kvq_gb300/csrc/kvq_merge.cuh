// Merge of the per-unit partials of decode attention (split attention over the work list), run by
// merge_kernel right after each decode launch.
//
// Every warp that worked on a unit left, per query head, an unnormalised partial: the running
// maximum m (log2 units), l = sum_t 2^(s_t - m) and acc[c] = sum_t 2^(s_t - m) v_tc over its
// tokens.  The output is sum_w 2^(m_w - M) acc_w / sum_w 2^(m_w - M) l_w with M = max_w m_w
// (log-sum-exp combination), written as fp16.
#pragma once

#include <cuda_fp16.h>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

constexpr int kMergeWarpsPerHead = 4;

// One CTA per unit, kMergeWarpsPerHead warps per query head.  The partials sit in L2, so the
// merge is a latency problem: every (m, l) of the head is loaded at once to fix M and the weights,
// then the head's warps split the slots and keep all their acc loads in flight, and shared memory
// sums the warps.  Two L2 round trips per unit.  Dynamic shared memory: HG * max_slots floats.
template <int HG>
__global__ void __launch_bounds__(HG * kMergeWarpsPerHead * 32) merge_kernel(const DecodeParams p) {
  constexpr int D = kHeadDim;
  constexpr int WH = kMergeWarpsPerHead;
  constexpr unsigned all = 0xffffffffu;
  extern __shared__ float wts[];  // [HG][max_slots]
  __shared__ float red[HG][WH][D];
  __shared__ float hmax[HG][WH], hsum[HG][WH];
  __shared__ int n_s;
  const int64_t unit = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = warp / WH, wh = warp % WH, ht = tid - h * WH * 32;  // head, warp and thread within it
  pdl_allow_next();
  pdl_wait();  // the decode launch's partials
  if (tid == 0) n_s = min(p.nslot[unit], p.max_slots);
  __syncthreads();
  const int n = n_s;
  const int64_t b = unit / p.Hkv, kvh = unit - b * p.Hkv;
  const int64_t bh = b * p.Hq + kvh * HG + h;
  const float* ml = p.part_ml + bh * p.max_slots * 2;
  const float* pacc = p.part_acc + bh * p.max_slots * D + 4 * lane;
  float* w = wts + h * p.max_slots;

  // the head's maximum, the slot weights and the weighted sum of l
  float mx = -INFINITY;
  for (int s = ht; s < n; s += WH * 32) mx = fmaxf(mx, __ldcg(ml + 2 * s));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(all, mx, off));
  if (lane == 0) hmax[h][wh] = mx;
  __syncthreads();
  float M = hmax[h][0];
#pragma unroll
  for (int i = 1; i < WH; ++i) M = fmaxf(M, hmax[h][i]);
  float lsum = 0.0f;
  for (int s = ht; s < n; s += WH * 32) {
    const float2 v = __ldcg(reinterpret_cast<const float2*>(ml + 2 * s));
    const float f = v.x == -INFINITY ? 0.0f : exp2f(v.x - M);
    w[s] = f;
    lsum = fmaf(f, v.y, lsum);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(all, lsum, off);
  if (lane == 0) hsum[h][wh] = lsum;
  __syncthreads();

  // this warp's slots wh, wh + WH, ...: lane l owns channels 4l .. 4l+3
  float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll 8
  for (int s = wh; s < n; s += WH) {
    const float f = w[s];
    const float4 v = __ldcg(reinterpret_cast<const float4*>(pacc + (int64_t)s * D));
    a0 = fmaf(f, v.x, a0);
    a1 = fmaf(f, v.y, a1);
    a2 = fmaf(f, v.z, a2);
    a3 = fmaf(f, v.w, a3);
  }
  *reinterpret_cast<float4*>(&red[h][wh][4 * lane]) = make_float4(a0, a1, a2, a3);
  __syncthreads();
  if (wh == 0) {
    float L = 0.0f;
#pragma unroll
    for (int i = 0; i < WH; ++i) L += hsum[h][i];
    float4 o = *reinterpret_cast<const float4*>(&red[h][0][4 * lane]);
#pragma unroll
    for (int i = 1; i < WH; ++i) {
      const float4 v = *reinterpret_cast<const float4*>(&red[h][i][4 * lane]);
      o.x += v.x;
      o.y += v.y;
      o.z += v.z;
      o.w += v.w;
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    const __half2 o01 = __floats2half2_rn(o.x * inv, o.y * inv), o23 = __floats2half2_rn(o.z * inv, o.w * inv);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&o01);
    packed.y = *reinterpret_cast<const uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(p.out + bh * D + 4 * lane) = packed;
  }
  if (tid == 0) p.nslot[unit] = 0;  // every thread has read n_s (barriers above)
}

}  // namespace kvq
