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

// ---------------------------------------------------------------------------------------------
// Decision thresholds of the uniform quantizer, for comparing fp16 inputs directly.
//
// For a group with stored zero point z and step s > 0 (fp16 values widened to fp32), the code of an
// fp16 value x is clamp(rint(q), 0, L) with q = fl(fl(x - z) / s), both roundings to nearest even.
// It is non-decreasing in x, so for every k < L there is a smallest fp16 value t_k whose code is
// at least k + 1, and code(x) = #{k : x >= t_k} for every x of the group.  t_k is found by testing
// "code(x) >= k + 1" exactly, without a division:
//
//   with h = k + 1/2 and d = fl(x - z) >= 0, rint(q) >= k + 1 means q > h, or q == h when k + 1 is
//   even (ties go to even).  h has at most five significant bits, so it is even as an fp32 value
//   and the fp32 numbers next to it are h -/+ ulp(h) (h is not a power of two for k >= 1; for
//   k = 0, h = 1/2 and only the number above it matters).  Rounding to nearest then gives
//     k odd :  q >= h       <=>  d / s >= h - ulp(h)/2   (a tie rounds to h, which is even)
//     k even:  q >= h + ulp <=>  d / s >  h + ulp(h)/2   (a tie rounds to h, not above it)
//   With A = h*s and B = -/+ s*ulp(h)/2 (both exact in fp32: 5 + 11 significant bits, and a power
//   of two times s), that is d - A >= B (k odd) or d - A > B (k even).  fl(d - A) decides it
//   exactly: within a factor of two of A the subtraction is exact (Sterbenz), and outside it
//   |d - A| >= A/2 is far larger than |B| <= A * 2^-24, so the rounded difference has the same
//   order against B as the exact one.
//
// The candidate t_k is the fp16 rounding of z + A + B; the exact test at it and at its neighbour
// confirms it (or its neighbour) almost always, and a bisection over the fp16 values between the
// group's minimum (code 0) and maximum settles the rest.  A threshold no value of the group reaches
// is +inf (0x7C00), which no finite input passes.
namespace kvq {
namespace qthr {

__host__ __device__ __forceinline__ float sub_rn(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fsub_rn(a, b);
#else
  volatile float r = a - b;
  return r;
#endif
}
__host__ __device__ __forceinline__ float add_rn(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fadd_rn(a, b);
#else
  volatile float r = a + b;
  return r;
#endif
}
__host__ __device__ __forceinline__ float mul_rn(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fmul_rn(a, b);
#else
  volatile float r = a * b;
  return r;
#endif
}
__host__ __device__ __forceinline__ float div_rn(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fdiv_rn(a, b);
#else
  volatile float r = a / b;
  return r;
#endif
}
__host__ __device__ __forceinline__ float fma_rn(float a, float b, float c) {
#ifdef __CUDA_ARCH__
  return __fmaf_rn(a, b, c);
#else
  return fmaf(a, b, c);
#endif
}
// a / L correctly rounded for a >= 0 (L = 3, 7, 15): the product with the rounded reciprocal,
// corrected once with the exact remainder a - q*L.  Every step scales exactly with a power of two
// of a, so one binade of significands and the range of subnormal quotients cover every a; both
// are checked exhaustively against the IEEE division on the host (tests/host/threshold_check.cu).
template <int L>
__host__ __device__ __forceinline__ float div_const(float a) {
  constexpr float inv = 1.0f / (float)L;
  const float q = mul_rn(a, inv);
  return fma_rn(fma_rn(-q, (float)L, a), inv, q);
}
__host__ __device__ __forceinline__ float half_to_float(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__host__ __device__ __forceinline__ uint16_t float_to_half(float f) { return __half_as_ushort(__float2half_rn(f)); }
__host__ __device__ __forceinline__ uint16_t half_rd(float f) { return __half_as_ushort(__float2half_rd(f)); }
__host__ __device__ __forceinline__ uint16_t half_ru(float f) { return __half_as_ushort(__float2half_ru(f)); }

// fp16 bit patterns in value order (-0 and +0 both 0), and back
__host__ __device__ __forceinline__ int ord(uint32_t b) { return (b & 0x8000u) ? -(int)(b & 0x7FFFu) : (int)b; }
__host__ __device__ __forceinline__ uint32_t bits_of(int o) { return o >= 0 ? (uint32_t)o : (0x8000u | (uint32_t)(-o)); }

// 2^e as an fp32 constant (-40 < e < 40)
__host__ __device__ constexpr float pow2(int e) { return e == 0 ? 1.0f : e > 0 ? 2.0f * pow2(e - 1) : 0.5f * pow2(e + 1); }

// h = k + 1/2 and the signed half-ulp factor of the test above (B = s * bfac)
__host__ __device__ constexpr int half_exp(int k) { return k == 0 ? -1 : k < 2 ? 0 : k < 4 ? 1 : k < 8 ? 2 : 3; }
__host__ __device__ constexpr float bfac(int k) { return ((k & 1) ? -1.0f : 1.0f) * pow2(half_exp(k) - 24); }

// code(x) >= k + 1, exactly (z, A = (k+1/2)*s, B = s*bfac(k))
template <int K>
__host__ __device__ __forceinline__ bool above(float x, float z, float A, float B) {
  const float e = sub_rn(sub_rn(x, z), A);
  return (K & 1) ? e >= B : e > B;
}

// t_k of a group with zero point z and step s > 0 (+inf when no finite fp16 value reaches code
// k + 1).
//
// Fast path: the test switches at a real X* with |X* - (z + A + B)| <= 1.5 ulp(A + B) (where
// fl(x - z) crosses A + B), and y = fl(fl(z + A) + B) is within 2^-24 (|z + A| + |y|) of
// z + A + B, so |y - X*| < 2^-21 (|z| + |A| + |y|) = eps/2.  Let a be the smallest and b the
// largest fp16 value in [y - eps, y + eps] (the ends rounded in fp32 stay well inside the margin).
// No fp16 value there (a > b): X* lies strictly between b and a, the next value up from b, and a
// is t_k.  Exactly one, a == b: every value below a fails, every value above passes, and one test
// at a decides between a and the next value up.  Two or more (an fp16 spacing below eps: values
// far smaller than the group's range, rare): X* is still inside the window, so the value below a
// fails and the value above b passes, and a bisection over the window's values finds t_k (a few
// halvings: the window holds about eps / spacing values).
template <int K>
__host__ __device__ __forceinline__ uint32_t threshold(float z, float s) {
  const float A = mul_rn(s, (float)K + 0.5f), B = mul_rn(s, bfac(K));
  const float y = add_rn(add_rn(z, A), B);
  const float eps = mul_rn(add_rn(add_rn(fabsf(z), A), fabsf(y)), 0x1.0p-20f);
  const uint16_t a = half_ru(sub_rn(y, eps)), b = half_rd(add_rn(y, eps));
  const float fa = half_to_float(a), fb = half_to_float(b);
  if (fa > fb) return a;
  if (fa == fb) return above<K>(fa, z, A, B) ? a : bits_of(ord(a) + 1);
  int lo = ord(a) - 1, hi = ord(b) + 1;  // above() is false at lo and true at hi
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (above<K>(half_to_float((uint16_t)bits_of(mid)), z, A, B)) hi = mid;
    else lo = mid;
  }
  return bits_of(hi);
}

// Zero point and step of a group from its exact fp16 minimum and maximum (as in group_params):
// returns the stored pair (zero point low, step high) and the widened values.
template <int L>
__host__ __device__ __forceinline__ uint32_t zero_step(float mn, float mx, float* z, float* s) {
  mn = add_rn(mn, 0.0f);  // -0 -> +0
  float range = sub_rn(mx, mn);
  if (!(range > 0.0f)) range = 0.0f;
  const uint16_t zb = float_to_half(mn), sb = float_to_half(div_const<L>(range));
  *z = half_to_float(zb);
  *s = half_to_float(sb);
  return (uint32_t)zb | ((uint32_t)sb << 16);
}

// The three thresholds of a 2-bit group (t[0] <= t[1] <= t[2]); all +inf for a zero step.
__host__ __device__ __forceinline__ uint32_t thresholds2(float mn, float mx, uint32_t t[3]) {
  float z, s;
  const uint32_t zs = zero_step<3>(mn, mx, &z, &s);
  if (!(s > 0.0f)) {
    t[0] = t[1] = t[2] = 0x7C00u;
    return zs;
  }
  t[0] = threshold<0>(z, s);
  t[1] = threshold<1>(z, s);
  t[2] = threshold<2>(z, s);
  return zs;
}

}  // namespace qthr
}  // namespace kvq
