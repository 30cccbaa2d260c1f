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
constexpr int kMergeChunk = 16;  // slots a warp loads at once

// One CTA per unit, kMergeWarpsPerHead warps per query head.  The partials sit in L2, so the
// merge is a latency problem: each warp takes every kMergeWarpsPerHead-th slot and loads the
// (m, l) and acc of sixteen of them together, merging them into a running (M, L, acc) of its own;
// shared memory then merges the head's warps.  For up to 64 slots per head that is one L2 round
// trip after the slot count.
template <int HG>
__global__ void __launch_bounds__(HG * kMergeWarpsPerHead * 32) merge_kernel(const DecodeParams p) {
  constexpr int D = kHeadDim;
  constexpr int WH = kMergeWarpsPerHead, CH = kMergeChunk;
  constexpr unsigned all = 0xffffffffu;
  __shared__ float4 red[HG][WH][32];
  __shared__ float wm[HG][WH], wl[HG][WH];
  __shared__ int n_s;
  const int64_t unit = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = warp / WH, wh = warp % WH;  // head and warp within it
  pdl_allow_next();
  pdl_wait();  // the decode launch's partials
  if (tid == 0) n_s = min(p.nslot[unit], p.max_slots);
  __syncthreads();
  const int n = n_s;
  const int64_t b = unit / p.Hkv, kvh = unit - b * p.Hkv;
  const int64_t bh = b * p.Hq + kvh * HG + h;
  const float* ml = p.part_ml + bh * p.max_slots * 2;
  const float* pacc = p.part_acc + bh * p.max_slots * D + 4 * lane;

  float M = -INFINITY, L = 0.0f;
  float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int base = wh; base < n; base += WH * CH) {
    // this chunk's slots base + WH*k, k < CH: lane k < CH loads slot k's (m, l); every lane loads
    // its four channels of every slot's acc -- all in flight together
    const int sl = base + WH * lane;
    const float2 mlv = lane < CH && sl < n ? __ldcg(reinterpret_cast<const float2*>(ml + 2 * sl))
                                            : make_float2(-INFINITY, 0.0f);
    float4 v[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int sk = base + WH * k;
      v[k] = sk < n ? __ldcg(reinterpret_cast<const float4*>(pacc + (int64_t)sk * D)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float cm = mlv.x;
#pragma unroll
    for (int off = 1; off < CH; off <<= 1) cm = fmaxf(cm, __shfl_xor_sync(all, cm, off));
    cm = __shfl_sync(all, cm, 0);
    const float Mn = fmaxf(M, cm);
    const float fo = M == -INFINITY ? 0.0f : exp2f(M - Mn);
    const float wk = mlv.x == -INFINITY ? 0.0f : exp2f(mlv.x - Mn);
    float lp = wk * mlv.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lp += __shfl_xor_sync(all, lp, off);
    L = fmaf(L, fo, lp);
    a.x *= fo;
    a.y *= fo;
    a.z *= fo;
    a.w *= fo;
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const float f = __shfl_sync(all, wk, k);
      a.x = fmaf(f, v[k].x, a.x);
      a.y = fmaf(f, v[k].y, a.y);
      a.z = fmaf(f, v[k].z, a.z);
      a.w = fmaf(f, v[k].w, a.w);
    }
    M = Mn;
  }
  red[h][wh][lane] = a;
  if (lane == 0) {
    wm[h][wh] = M;
    wl[h][wh] = L;
  }
  __syncthreads();
  if (wh == 0) {
    float Mh = wm[h][0];
#pragma unroll
    for (int i = 1; i < WH; ++i) Mh = fmaxf(Mh, wm[h][i]);
    float Lh = 0.0f;
    float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < WH; ++i) {
      const float f = wm[h][i] == -INFINITY ? 0.0f : exp2f(wm[h][i] - Mh);
      Lh = fmaf(f, wl[h][i], Lh);
      const float4 r = red[h][i][lane];
      o.x = fmaf(f, r.x, o.x);
      o.y = fmaf(f, r.y, o.y);
      o.z = fmaf(f, r.z, o.z);
      o.w = fmaf(f, r.w, o.w);
    }
    const float inv = Lh > 0.0f ? 1.0f / Lh : 0.0f;
    const __half2 o01 = __floats2half2_rn(o.x * inv, o.y * inv), o23 = __floats2half2_rn(o.z * inv, o.w * inv);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&o01);
    packed.y = *reinterpret_cast<const uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(p.out + bh * D + 4 * lane) = packed;
  }
  if (tid == 0) p.nslot[unit] = 0;  // every thread has read n_s (barriers above)
}

}  // namespace kvq
