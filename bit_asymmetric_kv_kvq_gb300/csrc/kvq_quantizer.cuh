// The uniform asymmetric group quantizer on the GPU, shared by the page kernel (kvq_quant.cu) and
// the axis-ablation kernels (kvq_ablation.cu).
//
// Zero point = group minimum, step = range/(2^B - 1), round to the nearest step ("KV cache has a
// geometry problem, not a bit problem", section "Quantization error in practice"), in fp32 with
// every rounding fixed:
//   range = mx - mn (RN), s32 = range / L (RN, true division),
//   z = fp16(mn), s = fp16_rn(s32), code = clamp(rint((x - z) / s), 0, L)
// with z and s the stored fp16 values.  A zero minimum is stored as +0 and a zero range gives
// s = +0 and codes 0.  The quotient is formed as (x - z) * (1/s) and replaced by the IEEE quotient
// within 2^-14 of a half-integer, where the two could round differently (kvq_quant.cu explains
// the bound), so every code equals the one the true division gives.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace kvq {
namespace {

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ uint16_t f2h(float f) { return __half_as_ushort(__float2half_rn(f)); }

// Per-group quantizer: the reciprocal of the scale and the two fp16 bit patterns (zero point low,
// scale high); the zero point and scale as stored are widened from the bits where they are used.
struct __align__(8) GroupQ {
  float inv;
  uint32_t bits;
  __device__ __forceinline__ float zf() const { return h2f((uint16_t)(bits & 0xFFFFu)); }
  __device__ __forceinline__ float sf() const { return h2f((uint16_t)(bits >> 16)); }
};

// Zero point and scale of a group from its exact min and max.
__device__ __forceinline__ GroupQ group_params(float mn, float mx, int L) {
  GroupQ g;
  mn = __fadd_rn(mn, 0.0f);  // -0 -> +0
  float range = __fsub_rn(mx, mn);
  if (!(range > 0.0f)) range = 0.0f;
  const float s32 = __fdiv_rn(range, (float)L);
  const uint16_t zb = f2h(mn), sb = f2h(s32);
  const float sf = h2f(sb);
  g.inv = sf > 0.0f ? __frcp_rn(sf) : 0.0f;
  g.bits = (uint32_t)zb | ((uint32_t)sb << 16);
  return g;
}

// Branch-free in the common case: a zero step has inv = 0, so r = 0 and the code is 0; the exact
// quotient is taken only when some lane of the warp is within 2^-14 of a half-integer (about one
// warp step in 300), so the warp pays one vote instead of a divergent branch per code.  "Within
// 2^-14 of a half-integer" is |r - rint(r)| >= 1/2 - 2^-14; the difference is exact (r and its
// rounding are within a factor of two of each other, or the rounding is 0).
__device__ __forceinline__ uint32_t quant_code(float x, const GroupQ& g, int L) {
  const float d = __fsub_rn(x, g.zf());
  const float r = __fmul_rn(d, g.inv);
  float q = rintf(r);
  const bool near = fabsf(__fsub_rn(r, q)) >= 0.5f - 0x1.0p-14f;
  if (__any_sync(__activemask(), near)) {
    if (near) q = rintf(__fdiv_rn(d, g.sf()));  // near a rounding tie: the exact quotient (s > 0 here)
  }
  q = fminf(fmaxf(q, 0.0f), (float)L);
  return (uint32_t)q;
}

// Codebook quantizer (non-uniform levels, "nuqX" without its calibration): the same zero point and
// step, then the nearest of the caller's levels lev[0..L] (in steps, 0 = lev[0] < ... < lev[L] = L).
// y = (x - z) / s is the IEEE quotient and the code is the number of decision thresholds
// thr[j] = fp32((lev[j] + lev[j+1]) * 0.5) that y exceeds, so a value on a threshold takes the lower
// level.  thr == nullptr selects the uniform quantizer.
__device__ __forceinline__ uint32_t code_of(float x, const GroupQ& g, int L, const float* thr) {
  if (!thr) return quant_code(x, g, L);
  const float sf = g.sf();
  if (sf == 0.0f) return 0;
  const float y = __fdiv_rn(__fsub_rn(x, g.zf()), sf);
  uint32_t c = 0;
  for (int j = 0; j < L; ++j) c += y > thr[j] ? 1u : 0u;
  return c;
}

}  // namespace
}  // namespace kvq
