// Axis ablation: the group quantizer applied along either axis of a key or value tensor, its
// dequantization, and exact fp32 decode attention over the result.
//
// The pages' central comparison ("KV cache has a geometry problem, not a bit problem", sections
// "Keys" and "Values"): keys have a few outlier channels, so a group that runs along the tokens of
// one channel (per-channel quantization) keeps each channel's own range, while a group that runs
// across the channels of one token takes the outlier's range for every channel in it; values have
// no such channels and are read as weighted sums over tokens, which favours per-token groups.
// These kernels let either tensor be quantized along either axis on the GPU, so that the score and
// output errors of the four combinations can be measured on the same inputs.  They are an analysis
// path beside the cache, not part of it.
//
//   axis KVQ_AXIS_TOKENS   : groups of G tokens of one channel; zero/scale [units][T/G][D]
//   axis KVQ_AXIS_CHANNELS : groups of G channels of one token; zero/scale [units][T][D/G]
//
// The quantizer is the cache's (kvq_quantizer.cuh), so codes, zero points and scales are those of
// the scalar IEEE definition bit for bit.  Dequantization is z + s*code with one rounding (fma).
#include <cuda_fp16.h>

#include "kvq.h"
#include "kvq_internal.h"
#include "kvq_quantizer.cuh"

namespace kvq {
namespace {

constexpr int kD = kHeadDim;
constexpr unsigned kAll = 0xffffffffu;

// Groups along tokens: one CTA of D threads per (unit, group), thread c owns channel c.  Each
// step of the two passes reads one whole token row (coalesced); the second pass hits in cache.
__global__ void __launch_bounds__(kD) axis_tokens_kernel(const uint16_t* __restrict__ x, int64_t T, int G, int L,
                                                          uint8_t* __restrict__ codes, uint16_t* __restrict__ zo,
                                                          uint16_t* __restrict__ so) {
  const int c = threadIdx.x;
  const int64_t unit = blockIdx.y, g = blockIdx.x;
  const int64_t row0 = unit * T + g * G;
  const uint16_t* src = x + row0 * kD + c;
  float mn = INFINITY, mx = -INFINITY;
  for (int t = 0; t < G; ++t) {
    const float v = h2f(src[(int64_t)t * kD]);
    mn = fminf(mn, v);
    mx = fmaxf(mx, v);
  }
  const GroupQ q = group_params(mn, mx, L);
  for (int t = 0; t < G; ++t) codes[(row0 + t) * kD + c] = (uint8_t)quant_code(h2f(src[(int64_t)t * kD]), q, L);
  const int64_t mo = (unit * (T / G) + g) * kD + c;
  zo[mo] = (uint16_t)(q.bits & 0xFFFFu);
  so[mo] = (uint16_t)(q.bits >> 16);
}

// Groups along channels: one warp per token row, lane l owns channels 4l .. 4l+3; a group is
// G/4 consecutive lanes.
constexpr int kRowsPerCta = 8;

__global__ void __launch_bounds__(kRowsPerCta * 32) axis_channels_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                          int G, int L, uint8_t* __restrict__ codes,
                                                                          uint16_t* __restrict__ zo,
                                                                          uint16_t* __restrict__ so) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (row >= rows) return;  // whole warps leave together
  const uint2 w = *reinterpret_cast<const uint2*>(x + row * kD + 4 * lane);
  const float v[4] = {h2f((uint16_t)(w.x & 0xFFFFu)), h2f((uint16_t)(w.x >> 16)), h2f((uint16_t)(w.y & 0xFFFFu)),
                      h2f((uint16_t)(w.y >> 16))};
  float mn = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
  float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
  const int lanes = G / 4;
  for (int off = 1; off < lanes; off <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(kAll, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, off));
  }
  const GroupQ q = group_params(mn, mx, L);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) packed |= quant_code(v[i], q, L) << (8 * i);
  *reinterpret_cast<uint32_t*>(codes + row * kD + 4 * lane) = packed;
  if (lane % lanes == 0) {
    const int64_t mo = row * (kD / G) + (4 * lane) / G;
    zo[mo] = (uint16_t)(q.bits & 0xFFFFu);
    so[mo] = (uint16_t)(q.bits >> 16);
  }
}

// z + s*code, four elements per thread.
__global__ void __launch_bounds__(256) axis_dequant_kernel(const uint8_t* __restrict__ codes,
                                                            const uint16_t* __restrict__ zi,
                                                            const uint16_t* __restrict__ si, int64_t rows, int64_t T,
                                                            int G, int axis, float* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t e0 = 4 * i;
  if (e0 >= rows * kD) return;
  const int64_t row = e0 / kD;
  const int c0 = (int)(e0 - row * kD);
  const uint32_t cw = *reinterpret_cast<const uint32_t*>(codes + e0);
  float r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = c0 + j;
    int64_t mo;
    if (axis == KVQ_AXIS_TOKENS) {
      const int64_t unit = row / T, t = row - unit * T;
      mo = (unit * (T / G) + t / G) * kD + c;
    } else {
      mo = row * (kD / G) + c / G;
    }
    r[j] = fmaf(h2f(si[mo]), (float)((cw >> (8 * j)) & 0xFFu), h2f(zi[mo]));
  }
  *reinterpret_cast<float4*>(out + e0) = make_float4(r[0], r[1], r[2], r[3]);
}

// Exact decode attention of HG query heads per unit over T rows of K and V (fp32, or fp16 when
// F32 is false): one CTA of 8 warps per unit; the warps split the tokens, lane l owns channels
// 4l .. 4l+3, each warp keeps an online softmax per head (base 2), shared memory merges the warps.
// scores (optional) receives scale * q.k per (unit, head, token).
constexpr int kAttnWarps = 8;

template <bool F32>
__device__ __forceinline__ float4 load_row4(const void* base, int64_t row, int lane) {
  if constexpr (F32) {
    return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + row * kD) + lane);
  } else {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + row * kD) + lane);
    return make_float4(h2f((uint16_t)(w.x & 0xFFFFu)), h2f((uint16_t)(w.x >> 16)), h2f((uint16_t)(w.y & 0xFFFFu)),
                       h2f((uint16_t)(w.y >> 16)));
  }
}

template <int HG, bool F32>
__global__ void __launch_bounds__(kAttnWarps * 32) axis_attention_kernel(const void* k, const void* v,
                                                                          const uint16_t* __restrict__ q, int64_t T,
                                                                          float scale, float* __restrict__ scores,
                                                                          float* __restrict__ out) {
  __shared__ float m_s[kAttnWarps][HG], l_s[kAttnWarps][HG];
  __shared__ float4 acc_s[kAttnWarps][HG][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t unit = blockIdx.x;
  const float scale_log2 = scale * 1.4426950408889634f;
  float qv[HG][4];
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    const uint2 w = *reinterpret_cast<const uint2*>(q + ((unit * HG + h) * kD) + 4 * lane);
    qv[h][0] = h2f((uint16_t)(w.x & 0xFFFFu));
    qv[h][1] = h2f((uint16_t)(w.x >> 16));
    qv[h][2] = h2f((uint16_t)(w.y & 0xFFFFu));
    qv[h][3] = h2f((uint16_t)(w.y >> 16));
  }
  float m[HG], l[HG];
  float4 acc[HG];
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
    acc[h] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  for (int64_t t = warp; t < T; t += kAttnWarps) {
    const float4 kr = load_row4<F32>(k, unit * T + t, lane);
    const float4 vr = load_row4<F32>(v, unit * T + t, lane);
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      float d = fmaf(qv[h][0], kr.x, fmaf(qv[h][1], kr.y, fmaf(qv[h][2], kr.z, qv[h][3] * kr.w)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(kAll, d, off);
      if (scores && lane == 0) scores[(unit * HG + h) * T + t] = d * scale;
      const float s2 = d * scale_log2;
      const float mn = fmaxf(m[h], s2);
      const float f = exp2f(m[h] - mn);  // 0 while m is -inf
      const float p = exp2f(s2 - mn);
      l[h] = fmaf(l[h], f, p);
      acc[h].x = fmaf(acc[h].x, f, p * vr.x);
      acc[h].y = fmaf(acc[h].y, f, p * vr.y);
      acc[h].z = fmaf(acc[h].z, f, p * vr.z);
      acc[h].w = fmaf(acc[h].w, f, p * vr.w);
      m[h] = mn;
    }
  }
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    if (lane == 0) {
      m_s[warp][h] = m[h];
      l_s[warp][h] = l[h];
    }
    acc_s[warp][h][lane] = acc[h];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, m_s[w][h]);
      float L = 0.0f;
      float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        const float f = m_s[w][h] == -INFINITY ? 0.0f : exp2f(m_s[w][h] - M);
        L = fmaf(f, l_s[w][h], L);
        const float4 a = acc_s[w][h][lane];
        o.x = fmaf(f, a.x, o.x);
        o.y = fmaf(f, a.y, o.y);
        o.z = fmaf(f, a.z, o.z);
        o.w = fmaf(f, a.w, o.w);
      }
      const float inv = 1.0f / L;
      reinterpret_cast<float4*>(out + (unit * HG + h) * kD)[lane] = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
    }
  }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace kvq

extern "C" {

kvq_status kvq_axis_quantize(const void* x_f16, int64_t n_units, int64_t n_tokens, int32_t head_dim, int32_t bits,
                             int32_t group_size, int32_t axis, void* codes_u8, void* zero_f16, void* scale_f16,
                             void* cuda_stream) {
  using namespace kvq;
  if (!x_f16 || !codes_u8 || !zero_f16 || !scale_f16) return KVQ_ERR_INVALID_ARG;
  if (n_units < 1 || n_tokens < 1 || bits < 2 || bits > 4) return KVQ_ERR_INVALID_ARG;
  if (axis != KVQ_AXIS_TOKENS && axis != KVQ_AXIS_CHANNELS) return KVQ_ERR_INVALID_ARG;
  if (head_dim != kD || (group_size != 32 && group_size != 64)) return KVQ_ERR_UNSUPPORTED;
  if (axis == KVQ_AXIS_TOKENS && (n_tokens % group_size || n_units > 65535)) return KVQ_ERR_INVALID_ARG;
  if (!aligned(x_f16, 8) || !aligned(codes_u8, 4) || !aligned(zero_f16, 2) || !aligned(scale_f16, 2))
    return KVQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const int L = (1 << bits) - 1;
  const uint16_t* x = static_cast<const uint16_t*>(x_f16);
  uint8_t* codes = static_cast<uint8_t*>(codes_u8);
  uint16_t* z = static_cast<uint16_t*>(zero_f16);
  uint16_t* sc = static_cast<uint16_t*>(scale_f16);
  if (axis == KVQ_AXIS_TOKENS) {
    const int64_t groups = n_tokens / group_size;
    if (groups > 0x7fffffff) return KVQ_ERR_UNSUPPORTED;
    axis_tokens_kernel<<<dim3((unsigned)groups, (unsigned)n_units), kD, 0, s>>>(x, n_tokens, group_size, L, codes, z,
                                                                               sc);
  } else {
    const int64_t rows = n_units * n_tokens;
    const int64_t ctas = (rows + kRowsPerCta - 1) / kRowsPerCta;
    if (ctas > 0x7fffffff) return KVQ_ERR_UNSUPPORTED;
    axis_channels_kernel<<<(unsigned)ctas, kRowsPerCta * 32, 0, s>>>(x, rows, group_size, L, codes, z, sc);
  }
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_axis_dequantize(const void* codes_u8, const void* zero_f16, const void* scale_f16, int64_t n_units,
                               int64_t n_tokens, int32_t head_dim, int32_t group_size, int32_t axis, void* out_f32,
                               void* cuda_stream) {
  using namespace kvq;
  if (!codes_u8 || !zero_f16 || !scale_f16 || !out_f32) return KVQ_ERR_INVALID_ARG;
  if (n_units < 1 || n_tokens < 1) return KVQ_ERR_INVALID_ARG;
  if (axis != KVQ_AXIS_TOKENS && axis != KVQ_AXIS_CHANNELS) return KVQ_ERR_INVALID_ARG;
  if (head_dim != kD || (group_size != 32 && group_size != 64)) return KVQ_ERR_UNSUPPORTED;
  if (axis == KVQ_AXIS_TOKENS && n_tokens % group_size) return KVQ_ERR_INVALID_ARG;
  if (!aligned(codes_u8, 4) || !aligned(out_f32, 16)) return KVQ_ERR_INVALID_ARG;
  const int64_t rows = n_units * n_tokens;
  const int64_t ctas = (rows * kD / 4 + 255) / 256;
  if (ctas > 0x7fffffff) return KVQ_ERR_UNSUPPORTED;
  axis_dequant_kernel<<<(unsigned)ctas, 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      static_cast<const uint8_t*>(codes_u8), static_cast<const uint16_t*>(zero_f16),
      static_cast<const uint16_t*>(scale_f16), rows, n_tokens, group_size, axis, static_cast<float*>(out_f32));
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_axis_attention(const void* k, const void* v, int32_t kv_f32, const void* q_f16, int64_t n_units,
                              int32_t heads_per_unit, int64_t n_tokens, int32_t head_dim, float softmax_scale,
                              void* scores_f32, void* out_f32, void* cuda_stream) {
  using namespace kvq;
  if (!k || !v || !q_f16 || !out_f32) return KVQ_ERR_INVALID_ARG;
  if (n_units < 1 || n_tokens < 1 || (kv_f32 != 0 && kv_f32 != 1)) return KVQ_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f)) return KVQ_ERR_INVALID_ARG;
  if (head_dim != kD) return KVQ_ERR_UNSUPPORTED;
  if (heads_per_unit != 1 && heads_per_unit != 2 && heads_per_unit != 4) return KVQ_ERR_UNSUPPORTED;
  if (n_units > 0x7fffffff) return KVQ_ERR_UNSUPPORTED;
  if (!aligned(k, kv_f32 ? 16 : 8) || !aligned(v, kv_f32 ? 16 : 8) || !aligned(q_f16, 8) || !aligned(out_f32, 16) ||
      !aligned(scores_f32, 4))
    return KVQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const uint16_t* q = static_cast<const uint16_t*>(q_f16);
  float* sc = static_cast<float*>(scores_f32);
  float* o = static_cast<float*>(out_f32);
  const unsigned grid = (unsigned)n_units;
  constexpr unsigned threads = kAttnWarps * 32;
#define KVQ_ATTN(HGV)                                                                                        \
  if (heads_per_unit == HGV) {                                                                               \
    if (kv_f32) axis_attention_kernel<HGV, true><<<grid, threads, 0, s>>>(k, v, q, n_tokens, softmax_scale, sc, o); \
    else axis_attention_kernel<HGV, false><<<grid, threads, 0, s>>>(k, v, q, n_tokens, softmax_scale, sc, o);       \
  }
  KVQ_ATTN(1) KVQ_ATTN(2) KVQ_ATTN(4)
#undef KVQ_ATTN
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // extern "C"
