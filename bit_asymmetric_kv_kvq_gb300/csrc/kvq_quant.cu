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
// The quotient (x - z) / s only matters through rint, so it is formed as
// (x - z) * (1/s) with a per-group reciprocal.  That product is within 2^-18
// of the correctly rounded quotient (|quotient| <= 16, two roundings of at
// most 2^-24 relative each); when it lies within 2^-14 of a half-integer --
// the only place where the two could round differently, ties included -- the
// code takes the IEEE quotient instead.  So every code equals the one the
// true division gives, at the cost of one multiply for all but ~1e-4 of the
// elements.
//
// Data movement: the two fp16 input tiles (R x D each) arrive by bulk copy
// into shared memory, each thread computes and packs whole 32-bit code words
// straight from the tile, the page is assembled in shared memory and leaves
// by one bulk copy, so all global traffic is 16-byte granular and contiguous.
#include <cuda_fp16.h>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"
#include "kvq_quantizer.cuh"

namespace kvq {

namespace {

constexpr int kQuantThreads = 256;
constexpr int kMaxSparse = 4;

// Shared-memory plan of one CTA (bytes, all 16-byte aligned).
struct QuantSmem {
  size_t kt, vt, kq, vq, sidx, pg, total;
};

// page_bytes = 0: the page is written straight to global memory (no image in shared memory).
__host__ __device__ inline QuantSmem quant_smem(int R, int D, int G, int page_bytes) {
  QuantSmem m;
  m.kt = 0;
  m.vt = m.kt + (size_t)R * D * 2;
  m.kq = m.vt + (size_t)R * D * 2;
  m.vq = m.kq + (size_t)(R / G) * D * sizeof(GroupQ);
  m.sidx = m.vq + (size_t)R * (D / G) * sizeof(GroupQ);
  m.pg = m.sidx + (((size_t)R * kMaxSparse + 15) / 16) * 16;
  m.total = m.pg + (size_t)page_bytes;
  return m;
}

// Key quantizers are stored interleaved by 32-channel chunk: channel c = 32*ch + i
// lives at slot i*NCH + ch, so the threads of a warp, which take consecutive
// chunks, read consecutive slots.
constexpr int kChunk = 32;
__device__ __forceinline__ int kq_slot(int c) { return (c % kChunk) * (kHeadDim / kChunk) + c / kChunk; }

// Codes of 32 consecutive channels of one token (x: 32 fp16 values, 16-byte aligned),
// packed into BITS words of the token's bitstream.  grp(i) is the quantizer of channel
// i of the chunk; excl has bit i set for an excluded channel (code 0).
template <int BITS, class Params>
__device__ __forceinline__ void pack_chunk(const uint16_t* x, const Params& grp, uint32_t excl, uint32_t* out,
                                           const float* thr) {
  constexpr int L = (1 << BITS) - 1;
  uint32_t w[BITS];
#pragma unroll
  for (int k = 0; k < BITS; ++k) w[k] = 0;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
#pragma unroll
  for (int q4 = 0; q4 < kChunk / 8; ++q4) {
    const uint4 v = xv[q4];
    const uint32_t pair[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = q4 * 8 + j;
      const uint16_t bits = (uint16_t)(j & 1 ? pair[j >> 1] >> 16 : pair[j >> 1] & 0xFFFFu);
      const uint32_t c = code_of(h2f(bits), grp(i), L, thr);  // then masked: no branch per code
      const uint32_t code = (excl >> i) & 1u ? 0u : c;
      const int b = i * BITS;
      w[b >> 5] |= code << (b & 31);
      if ((b & 31) + BITS > 32) w[(b >> 5) + 1] |= code >> (32 - (b & 31));
    }
  }
#pragma unroll
  for (int k = 0; k < BITS; ++k) out[k] = w[k];
}

// Threads of one page CTA: the common-shape variant runs 512 (it needs about 35 registers, and
// its fragment packing gives keys and values to separate halves), the general one 256.
template <bool STD>
__host__ __device__ constexpr int quant_threads() { return STD ? 2 * kQuantThreads : kQuantThreads; }

template <int BK, int BV, bool STD>
__global__ void __launch_bounds__(quant_threads<STD>(), STD ? 3 : 2) quantize_pages_kernel(const QuantizeParams p) {
  constexpr int NT = quant_threads<STD>();
  const int page = blockIdx.x;
  const int unit = blockIdx.y;
  // STD: the common page shape (StdPage) with compile-time sizes and offsets
  using SP = StdPage<BK, BV>;
  const int D = STD ? kHeadDim : p.D, R = STD ? 128 : p.R, G = STD ? 32 : p.G, nsp = STD ? 0 : p.nsp;
  const bool frag = STD ? true : p.lay.frag != 0;
  const int lay_bytes = STD ? SP::bytes : p.lay.bytes;
  const int off_kc = STD ? SP::kc : p.lay.off_kc, off_km = STD ? SP::km : p.lay.off_km;
  const int off_vc = STD ? SP::vc : p.lay.off_vc, off_vm = STD ? SP::vm : p.lay.off_vm;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int LK = (1 << BK) - 1, LV = (1 << BV) - 1;

  extern __shared__ __align__(128) uint8_t smem[];
  // the common shape writes its page straight to global memory (16-byte stores, coalesced per warp),
  // which leaves room for three CTAs per SM; the general kernel assembles it in shared memory
  const QuantSmem sm = quant_smem(R, D, G, STD ? 0 : lay_bytes);
  uint16_t* kt = reinterpret_cast<uint16_t*>(smem + sm.kt);  // [R][D]
  uint16_t* vt = reinterpret_cast<uint16_t*>(smem + sm.vt);  // [R][D]
  GroupQ* kq = reinterpret_cast<GroupQ*>(smem + sm.kq);      // [R/G][D]
  GroupQ* vq = reinterpret_cast<GroupQ*>(smem + sm.vq);      // [R][D/G]
  uint8_t* sidx = smem + sm.sidx;                            // [R][kMaxSparse]
  uint8_t* const dst_page =
      p.pages + (int64_t)unit * p.unit_page_stride + (p.page0 + page) * (int64_t)lay_bytes;
  uint8_t* pg = STD ? dst_page : smem + sm.pg;                // page image (or the page itself)
  __shared__ __align__(8) uint64_t bar;
  __shared__ float thr_s[2][16];  // codebook decision thresholds (keys, values)

  const int64_t tok0 = p.src_tok0 + (int64_t)page * R;
  const uint16_t* ksrc = p.k_src + (int64_t)unit * p.src_unit_stride + tok0 * D;
  const uint16_t* vsrc = p.v_src + (int64_t)unit * p.src_unit_stride + tok0 * D;
  uint8_t* dst = p.pages + (int64_t)unit * p.unit_page_stride + (p.page0 + page) * (int64_t)lay_bytes;

  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (tid < 16) {
    thr_s[0][tid] = p.k_thr[tid];
    thr_s[1][tid] = p.v_thr[tid];
  }
  __syncthreads();
  const float* kthr = p.lut ? thr_s[0] : nullptr;
  const float* vthr = p.lut ? thr_s[1] : nullptr;
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
    for (int t = warp; t < R; t += NT / 32) {
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
    for (int i = si_used + tid; i < p.lay.off_sv - p.lay.off_si; i += NT) pg[p.lay.off_si + i] = 0;
    for (int i = sv_used + tid; i < p.lay.bytes - p.lay.off_sv; i += NT) pg[p.lay.off_sv + i] = 0;
    __syncthreads();
  }
  auto excluded = [&](int t, int c) {
    if (nsp == 0) return false;
    bool ex = false;
    for (int k = 0; k < nsp; ++k) ex |= sidx[t * kMaxSparse + k] == c;
    return ex;
  };

  // ---- keys: one quantizer per (G-token group, channel)
  const int ngk = R / G;
  if (nsp == 0) {
    // two channels per thread: fp16 minimum and maximum are exact, so the scan runs on half2
    for (int idx = tid; idx < ngk * D / 2; idx += NT) {
      const int g = idx / (D / 2), c = 2 * (idx - g * (D / 2));
      const __half2* col = reinterpret_cast<const __half2*>(kt + (g * G) * D + c);
      __half2 mn = col[0], mx = mn;
#pragma unroll 8
      for (int t = 1; t < G; ++t) {
        const __half2 v = col[t * (D / 2)];
        mn = __hmin2(mn, v);
        mx = __hmax2(mx, v);
      }
      const float2 fmn = __half22float2(mn), fmx = __half22float2(mx);
      const GroupQ q0 = group_params(fmn.x, fmx.x, LK), q1 = group_params(fmn.y, fmx.y, LK);
      kq[g * D + (frag ? c : kq_slot(c))] = q0;  // fragment packing reads them channel by channel
      kq[g * D + (frag ? c + 1 : kq_slot(c + 1))] = q1;
      *reinterpret_cast<uint2*>(reinterpret_cast<uint32_t*>(pg + off_km) + g * D + c) = make_uint2(q0.bits, q1.bits);
    }
  } else {
    for (int idx = tid; idx < ngk * D; idx += NT) {
      const int g = idx / D, c = idx - g * D;
      bool any = false;
      float mn = 0.0f, mx = 0.0f;
      for (int t = g * G; t < g * G + G; ++t) {
        if (excluded(t, c)) continue;
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
      const GroupQ q = group_params(mn, mx, LK);
      kq[g * D + (frag ? c : kq_slot(c))] = q;
      reinterpret_cast<uint32_t*>(pg + off_km)[idx] = q.bits;
    }
  }

  // ---- values: one quantizer per (token, G-channel group); a warp per token,
  //      4 consecutive channels per lane, G/4 lanes per group
  {
    const int lanes_per_group = G / 4;
    const int c0 = lane * 4;
    const int ng = D / G;
    for (int t = warp; t < R; t += NT / 32) {
      float x[4];
      {
        const uint2 w = *reinterpret_cast<const uint2*>(vt + t * D + c0);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
        x[0] = a.x;
        x[1] = a.y;
        x[2] = b.x;
        x[3] = b.y;
      }
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
      if ((lane & (lanes_per_group - 1)) == 0) {
        const GroupQ q = group_params(mn, mx, LV);
        const int g = c0 / G;
        vq[t * ng + g] = q;
        reinterpret_cast<uint32_t*>(pg + off_vm)[t * ng + g] = q.bits;
      }
    }
  }
  __syncthreads();

  // ---- codes in fragment order (2- and 4-bit codes, keys without RoPE): one word per thread
  //      and step, its code pairs placed as frag_key_pair / frag_value_pair describe
  if (frag) {
    constexpr int KB = (BK == 2 || BK == 4) ? BK : 2, VB = (BV == 2 || BV == 4) ? BV : 2;
    uint32_t* kc = reinterpret_cast<uint32_t*>(pg + off_kc);
    uint32_t* vc = reinterpret_cast<uint32_t*>(pg + off_vc);
    const int ng = D / G;
    // one thread per (16-token tile, lane) owns that lane's 2B words of the tile; with 512 threads
    // the first half packs the keys and the second half the values
    const int items = (R / 16) * 32;
    const bool split = NT >= 2 * items;
    const int first = split && tid >= items ? items : 0;
    for (int id2 = tid - first; id2 < items; id2 += split ? 2 * items : NT) {
      const int idx = id2;
      const int tile = idx >> 5, ln = idx & 31, g = ln >> 2, t = ln & 3;
      if (!split || first == 0) {
        // keys: tokens 16*tile + g (+8), channels 16kk + 8h + 2t (+1); one key group per tile
        const int tk0 = 16 * tile + g;
        const GroupQ* gq = kq + (tk0 / G) * D;
        uint32_t wk[2 * KB];
#pragma unroll
        for (int i = 0; i < 2 * KB; ++i) wk[i] = 0;
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c0 = 16 * kk + 8 * h + 2 * t;
            const GroupQ q0 = gq[c0], q1 = gq[c0 + 1];
            const int j = 2 * (kk % (8 / KB)) + h;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int tok = tk0 + 8 * r;
              const uint32_t xx = *reinterpret_cast<const uint32_t*>(kt + tok * D + c0);
              uint32_t a = quant_code(h2f((uint16_t)(xx & 0xFFFFu)), q0, LK);
              uint32_t b = quant_code(h2f((uint16_t)(xx >> 16)), q1, LK);
              if (nsp > 0) {
                a = excluded(tok, c0) ? 0u : a;
                b = excluded(tok, c0 + 1) ? 0u : b;
              }
              wk[r * KB + kk / (8 / KB)] |= (a << (KB * j)) | (b << (16 + KB * j));
            }
          }
        uint4* dstk = reinterpret_cast<uint4*>(kc + (size_t)idx * 2 * KB);
#pragma unroll
        for (int i = 0; i < 2 * KB / 4; ++i) dstk[i] = make_uint4(wk[4 * i], wk[4 * i + 1], wk[4 * i + 2], wk[4 * i + 3]);
      }
      if (!split || first != 0) {
        // values: tokens s, s+1 with s = 16*tile + 8*tb + 2t; channel 16mc + g + 8rr; one
        // quantizer per (token, channel group), used for every channel of the lane in that group
        uint32_t wv[2 * VB];
#pragma unroll
        for (int i = 0; i < 2 * VB; ++i) wv[i] = 0;
#pragma unroll
        for (int tb = 0; tb < 2; ++tb) {
          const int s0 = 16 * tile + 8 * tb + 2 * t;
          for (int grp = 0; grp < ng; ++grp) {
            const GroupQ q0 = vq[s0 * ng + grp], q1 = vq[(s0 + 1) * ng + grp];
            for (int mc = grp * (G / 16); mc < (grp + 1) * (G / 16); ++mc)
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                const int ch = 16 * mc + g + 8 * rr;
                const uint32_t a = quant_code(h2f(vt[s0 * D + ch]), q0, LV);
                const uint32_t b = quant_code(h2f(vt[(s0 + 1) * D + ch]), q1, LV);
                const int r = 2 * tb + rr, j = mc % (16 / VB);
                wv[r * (VB / 2) + mc / (16 / VB)] |= (a << (VB * j)) | (b << (16 + VB * j));
              }
          }
        }
        uint4* dstv = reinterpret_cast<uint4*>(vc + (size_t)idx * 2 * VB);
#pragma unroll
        for (int i = 0; i < 2 * VB / 4; ++i) dstv[i] = make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
      }
    }
  } else {
    // ---- codes as token-major bitstreams, computed and packed a 32-channel chunk (BITS words) at a time
    constexpr int NCH = kHeadDim / kChunk;
    constexpr int WKW = kHeadDim * BK / 32, WVW = kHeadDim * BV / 32;
    uint32_t* kc = reinterpret_cast<uint32_t*>(pg + off_kc);
    uint32_t* vc = reinterpret_cast<uint32_t*>(pg + off_vc);
    for (int idx = tid; idx < R * NCH; idx += NT) {
      const int t = idx / NCH, ch = idx - t * NCH;
      uint32_t excl = 0;
      for (int k = 0; k < nsp; ++k) {
        const int c = sidx[t * kMaxSparse + k] - ch * kChunk;
        if (c >= 0 && c < kChunk) excl |= 1u << c;
      }
      const GroupQ* gq = kq + (t / G) * D + ch;
      pack_chunk<BK>(kt + t * D + ch * kChunk, [&](int i) -> const GroupQ& { return gq[i * NCH]; }, excl,
                     kc + t * WKW + ch * BK, kthr);
    }
    const int ng = D / G;
    for (int idx = tid; idx < R * NCH; idx += NT) {
      const int t = idx / NCH, ch = idx - t * NCH;
      const GroupQ& gq = vq[t * ng + (ch * kChunk) / G];
      pack_chunk<BV>(vt + t * D + ch * kChunk, [&](int) -> const GroupQ& { return gq; }, 0u, vc + t * WVW + ch * BV,
                     vthr);
    }
  }
  if constexpr (!STD) {
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_s2g(dst, pg, (uint32_t)lay_bytes);
      bulk_commit();
      bulk_wait_all();
    }
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
  using SP = StdPage<BK, BV>;
  constexpr bool can_std = (BK == 2 || BK == 4) && (BV == 2 || BV == 4);  // fragment-order pages only
  const bool std_shape = can_std && p.R == 128 && p.D == kHeadDim && p.G == 32 && p.nsp == 0 && p.lay.frag &&
                         !p.lut && p.lay.bytes == SP::bytes && p.lay.off_kc == SP::kc && p.lay.off_km == SP::km &&
                         p.lay.off_vc == SP::vc && p.lay.off_vm == SP::vm;
  auto kern = std_shape ? quantize_pages_kernel<BK, BV, can_std> : quantize_pages_kernel<BK, BV, false>;
  const size_t smem = std_shape ? quant_smem(p.R, p.D, p.G, 0).total : quantize_smem_bytes(p.R, p.D, p.G, p.lay);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)n_pages, (unsigned)p.n_units);
  kern<<<grid, std_shape ? quant_threads<can_std>() : kQuantThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t quantize_smem_bytes(int R, int D, int G, const PageLayout& lay) { return quant_smem(R, D, G, lay.bytes).total; }

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
