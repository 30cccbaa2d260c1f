// Quantize-and-pack kernel (prefill and residual flush) and the token copy
// kernel (prefill tail, append).
//
// One CTA turns R fp16 tokens of one (batch, kv-head) unit into one packed
// page.  Keys are quantized per channel over G-token groups, values per token
// over G-channel groups ("KV cache has a geometry problem, not a bit problem",
// sections "Keys" and "Values"), each group with the uniform asymmetric
// quantizer of section "Quantization error in practice": zero point = group
// minimum, step = range/(2^B - 1), round to the nearest step.  With sparse
// keys the largest-|x| entries of each key vector are kept in fp16 and left
// out of the channel ranges (KVQuant review, "Proposed method").
//
// The fp32 arithmetic is fixed step by step so that codes, zero points and
// scales are bit-identical to a scalar IEEE implementation:
//   range = mx - mn (RN), s32 = range / L (RN, true division),
//   z = fp16(mn), s = fp16_rn(s32), code = clamp(rint((x - z) / s), 0, L)
// with z and s the stored fp16 values.  A zero minimum is stored as +0 and a
// zero range gives s = +0 and codes 0.
//
// Data movement: the two fp16 input tiles (R x D each) arrive by bulk copy
// into shared memory, the page is assembled in shared memory and leaves by
// one bulk copy, so all global traffic is 16-byte granular and contiguous.
#include <cuda_fp16.h>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

namespace {

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ uint16_t f2h(float f) { return __half_as_ushort(__float2half_rn(f)); }

struct GroupQuant {
  uint16_t zb, sb;
  float zf, sf;
};

// Zero point and scale of a group from its exact min and max.
__device__ __forceinline__ GroupQuant group_params(float mn, float mx, int L) {
  GroupQuant g;
  mn = __fadd_rn(mn, 0.0f);  // -0 -> +0
  float range = __fsub_rn(mx, mn);
  if (!(range > 0.0f)) range = 0.0f;
  const float s32 = __fdiv_rn(range, (float)L);
  g.zb = f2h(mn);
  g.sb = f2h(s32);
  g.zf = h2f(g.zb);
  g.sf = h2f(g.sb);
  return g;
}

__device__ __forceinline__ uint8_t quant_code(float x, float zf, float sf, int L) {
  if (sf == 0.0f) return 0;
  const float d = __fsub_rn(x, zf);
  float q = rintf(__fdiv_rn(d, sf));
  q = fminf(fmaxf(q, 0.0f), (float)L);
  return (uint8_t)q;
}

// Pack one bitstream word: bits [32w, 32w+32) of a row of byte codes.
template <int BITS>
__device__ __forceinline__ uint32_t pack_word(const uint8_t* row, int w) {
  const int first = (32 * w) / BITS;
  const int last = (32 * w + 31) / BITS;
  uint32_t word = 0;
  for (int i = first; i <= last; ++i) {
    const int b = i * BITS - 32 * w;
    const uint32_t c = row[i];
    word |= b >= 0 ? (c << b) : (c >> (-b));
  }
  return word;
}

constexpr int kQuantThreads = 256;
constexpr int kMaxSparse = 4;

template <int BK, int BV>
__global__ void __launch_bounds__(kQuantThreads) quantize_pages_kernel(const QuantizeParams p) {
  const int page = blockIdx.x;
  const int unit = blockIdx.y;
  const int D = p.D, R = p.R, G = p.G, nsp = p.nsp;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int LK = (1 << BK) - 1, LV = (1 << BV) - 1;

  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* kt = reinterpret_cast<uint16_t*>(smem);              // [R][D]
  uint16_t* vt = kt + R * D;                                      // [R][D]
  uint8_t* kc8 = reinterpret_cast<uint8_t*>(vt + R * D);          // [R][D]
  uint8_t* vc8 = kc8 + R * D;                                     // [R][D]
  float* kzs = reinterpret_cast<float*>(vc8 + R * D);             // [R/G][D][2]
  uint8_t* sidx = reinterpret_cast<uint8_t*>(kzs + 2 * (R / G) * D);  // [R][kMaxSparse]
  uint8_t* pg = sidx + R * kMaxSparse;                            // page image (16-byte aligned: see smem size)
  __shared__ __align__(8) uint64_t bar;
  __shared__ int failed;

  const int64_t tok0 = p.src_tok0 + (int64_t)page * R;
  const uint16_t* ksrc = p.k_src + (int64_t)unit * p.src_unit_stride + tok0 * D;
  const uint16_t* vsrc = p.v_src + (int64_t)unit * p.src_unit_stride + tok0 * D;
  uint8_t* dst = p.pages + (int64_t)unit * p.unit_page_stride + (p.page0 + page) * (int64_t)p.lay.bytes;

  if (tid == 0) {
    failed = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t tile_bytes = (uint32_t)(R * D * 2);
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, 2 * tile_bytes);
    bulk_g2s(kt, ksrc, tile_bytes, &bar);
    bulk_g2s(vt, vsrc, tile_bytes, &bar);
  }
  if (!mbar_wait(&bar, 0)) {
    report_error(p.err, kDevWaitTimeout);
    mbar_wait(&bar, 0);  // give the copies in flight one more bounded chance to land
    return;
  }

  // ---- sparse outliers of each key vector: the nsp largest |x|, ties to the lower channel
  if (nsp > 0) {
    for (int t = warp; t < R; t += kQuantThreads / 32) {
      const uint16_t* row = kt + t * D;
      float a[kHeadDim / 32];
#pragma unroll
      for (int j = 0; j < kHeadDim / 32; ++j) a[j] = fabsf(h2f(row[lane + 32 * j]));
      int chosen[kMaxSparse];
      for (int k = 0; k < nsp; ++k) {
        float bv = -1.0f;
        int bc = 1 << 30;
#pragma unroll
        for (int j = 0; j < kHeadDim / 32; ++j) {
          if (a[j] > bv) {  // channels visited in increasing order: ties keep the lower one
            bv = a[j];
            bc = lane + 32 * j;
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
          const int oc = __shfl_xor_sync(0xffffffffu, bc, off);
          if (ov > bv || (ov == bv && oc < bc)) {
            bv = ov;
            bc = oc;
          }
        }
        chosen[k] = bc;
#pragma unroll
        for (int j = 0; j < kHeadDim / 32; ++j)
          if (lane + 32 * j == bc) a[j] = -2.0f;  // taken
      }
      if (lane == 0) {
        for (int i = 1; i < nsp; ++i) {  // ascending channel order
          const int v = chosen[i];
          int j = i - 1;
          while (j >= 0 && chosen[j] > v) {
            chosen[j + 1] = chosen[j];
            --j;
          }
          chosen[j + 1] = v;
        }
        uint8_t* si = pg + p.lay.off_si + t * nsp;
        uint16_t* sv = reinterpret_cast<uint16_t*>(pg + p.lay.off_sv) + t * nsp;
        for (int k = 0; k < kMaxSparse; ++k) sidx[t * kMaxSparse + k] = k < nsp ? (uint8_t)chosen[k] : 0xFF;
        for (int k = 0; k < nsp; ++k) {
          si[k] = (uint8_t)chosen[k];
          sv[k] = row[chosen[k]];
        }
      }
    }
    // zero the padding of the sparse sections
    const int si_used = R * nsp, sv_used = R * nsp * 2;
    for (int i = si_used + tid; i < p.lay.off_sv - p.lay.off_si; i += kQuantThreads) pg[p.lay.off_si + i] = 0;
    for (int i = sv_used + tid; i < p.lay.bytes - p.lay.off_sv; i += kQuantThreads) pg[p.lay.off_sv + i] = 0;
    __syncthreads();
  }

  // ---- keys: one (zero point, scale) per (G-token group, channel)
  const int ngk = R / G;
  for (int idx = tid; idx < ngk * D; idx += kQuantThreads) {
    const int g = idx / D, c = idx - g * D;
    bool any = false;
    float mn = 0.0f, mx = 0.0f;
    for (int t = g * G; t < g * G + G; ++t) {
      if (nsp > 0) {
        bool ex = false;
        for (int k = 0; k < nsp; ++k) ex |= sidx[t * kMaxSparse + k] == c;
        if (ex) continue;
      }
      const float v = h2f(kt[t * D + c]);
      if (!any) {
        mn = v;
        mx = v;
        any = true;
      } else {
        mn = v < mn ? v : mn;
        mx = v > mx ? v : mx;
      }
    }
    const GroupQuant q = group_params(mn, mx, LK);
    reinterpret_cast<uint32_t*>(pg + p.lay.off_km)[g * D + c] = (uint32_t)q.zb | ((uint32_t)q.sb << 16);
    kzs[2 * idx] = q.zf;
    kzs[2 * idx + 1] = q.sf;
  }
  __syncthreads();
  for (int idx = tid; idx < R * D; idx += kQuantThreads) {
    const int t = idx / D, c = idx - t * D;
    const int gi = (t / G) * D + c;
    bool ex = false;
    if (nsp > 0)
      for (int k = 0; k < nsp; ++k) ex |= sidx[t * kMaxSparse + k] == c;
    kc8[idx] = ex ? 0 : quant_code(h2f(kt[idx]), kzs[2 * gi], kzs[2 * gi + 1], LK);
  }

  // ---- values: one (zero point, scale) per (token, G-channel group); a warp per token,
  //      4 consecutive channels per lane, G/4 lanes per group
  {
    const int lanes_per_group = G / 4;
    const int c0 = lane * 4;
    for (int t = warp; t < R; t += kQuantThreads / 32) {
      float x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = h2f(vt[t * D + c0 + i]);
      float mn = x[0], mx = x[0];
#pragma unroll
      for (int i = 1; i < 4; ++i) {
        mn = x[i] < mn ? x[i] : mn;
        mx = x[i] > mx ? x[i] : mx;
      }
      for (int off = 1; off < lanes_per_group; off <<= 1) {
        const float omn = __shfl_xor_sync(0xffffffffu, mn, off);
        const float omx = __shfl_xor_sync(0xffffffffu, mx, off);
        mn = omn < mn ? omn : mn;
        mx = omx > mx ? omx : mx;
      }
      const GroupQuant q = group_params(mn, mx, LV);
      if ((lane & (lanes_per_group - 1)) == 0) {
        const int g = c0 / G;
        reinterpret_cast<uint32_t*>(pg + p.lay.off_vm)[t * (D / G) + g] = (uint32_t)q.zb | ((uint32_t)q.sb << 16);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) vc8[t * D + c0 + i] = quant_code(x[i], q.zf, q.sf, LV);
    }
  }
  __syncthreads();

  // ---- pack both code planes into their bitstreams
  {
    constexpr int WKW = kHeadDim * BK / 32, WVW = kHeadDim * BV / 32;
    uint32_t* kc = reinterpret_cast<uint32_t*>(pg + p.lay.off_kc);
    uint32_t* vc = reinterpret_cast<uint32_t*>(pg + p.lay.off_vc);
    for (int idx = tid; idx < R * WKW; idx += kQuantThreads) {
      const int t = idx / WKW, w = idx - t * WKW;
      kc[idx] = pack_word<BK>(kc8 + t * D, w);
    }
    for (int idx = tid; idx < R * WVW; idx += kQuantThreads) {
      const int t = idx / WVW, w = idx - t * WVW;
      vc[idx] = pack_word<BV>(vc8 + t * D, w);
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {
    bulk_s2g(dst, pg, (uint32_t)p.lay.bytes);
    bulk_commit();
    bulk_wait_all();
  }
}

__global__ void copy_tokens_kernel(const CopyTokensParams p) {
  const int unit = blockIdx.x;
  const int64_t n16 = (int64_t)p.n_tok * p.D / 8;  // 16-byte vectors per tensor
  const uint4* ks = reinterpret_cast<const uint4*>(p.k_src + unit * p.src_unit_stride + p.src_tok0 * p.D);
  const uint4* vs = reinterpret_cast<const uint4*>(p.v_src + unit * p.src_unit_stride + p.src_tok0 * p.D);
  uint4* kd = reinterpret_cast<uint4*>(p.k_dst + unit * p.dst_unit_stride + p.dst_tok0 * p.D);
  uint4* vd = reinterpret_cast<uint4*>(p.v_dst + unit * p.dst_unit_stride + p.dst_tok0 * p.D);
  for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

template <int BK, int BV>
cudaError_t launch_quantize_t(const QuantizeParams& p, int n_pages, cudaStream_t s) {
  const size_t smem = quantize_smem_bytes(p.R, p.D, p.lay);
  auto kern = quantize_pages_kernel<BK, BV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)n_pages, (unsigned)p.n_units);
  kern<<<grid, kQuantThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t quantize_smem_bytes(int R, int D, const PageLayout& lay) {
  // fp16 tiles, byte codes, per-group (z, s) floats, sparse index table, page image
  size_t b = (size_t)R * D * 2 * 2 + (size_t)R * D * 2 + (size_t)2 * R * D * 4 / 32 + (size_t)R * kMaxSparse;
  b = (b + 15) & ~(size_t)15;
  return b + (size_t)lay.bytes;
}

bool quantize_supported(int bk, int bv) { return bk >= 2 && bk <= 4 && bv >= 2 && bv <= 4; }

cudaError_t launch_quantize(const QuantizeParams& p, int bk, int bv, int n_pages, cudaStream_t s) {
  if (n_pages <= 0 || p.n_units <= 0) return cudaSuccess;
#define KVQ_Q(BKV, BVV) \
  if (bk == BKV && bv == BVV) return launch_quantize_t<BKV, BVV>(p, n_pages, s);
  KVQ_Q(2, 2) KVQ_Q(2, 3) KVQ_Q(2, 4) KVQ_Q(3, 2) KVQ_Q(3, 3) KVQ_Q(3, 4) KVQ_Q(4, 2) KVQ_Q(4, 3) KVQ_Q(4, 4)
#undef KVQ_Q
  return cudaErrorInvalidValue;
}

cudaError_t launch_copy_tokens(const CopyTokensParams& p, cudaStream_t s) {
  if (p.n_tok <= 0 || p.n_units <= 0) return cudaSuccess;
  copy_tokens_kernel<<<p.n_units, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
