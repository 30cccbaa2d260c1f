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
// Two kernels.  The general one (any R, G, sparse entries, code order,
// codebooks): the two fp16 input tiles (R x D each) arrive by bulk copy into
// shared memory, each thread computes and packs whole 32-bit code words
// straight from the tile, the page is assembled in shared memory and leaves
// by one bulk copy.  The common page shape (R = 128, G = 32, 2- or 4-bit codes
// in fragment order) has a kernel of its own, quantize_std_kernel, which
// takes 2-bit codes by comparing fp16 inputs with exact per-group decision
// thresholds (kvq_quantizer.cuh) instead of dividing.
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

// The general page kernel: any R, G, sparse entries, bitstream or fragment order, codebooks.  The
// common page shape has its own kernel below (quantize_std_kernel).
template <int BK, int BV>
__global__ void __launch_bounds__(kQuantThreads, 2) quantize_pages_kernel(const QuantizeParams p) {
  constexpr int NT = kQuantThreads;
  const int page = blockIdx.x;
  const int unit = blockIdx.y;
  const int D = p.D, R = p.R, G = p.G, nsp = p.nsp;
  const bool frag = p.lay.frag != 0;
  const int lay_bytes = p.lay.bytes;
  const int off_kc = p.lay.off_kc, off_km = p.lay.off_km;
  const int off_vc = p.lay.off_vc, off_vm = p.lay.off_vm;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int LK = (1 << BK) - 1, LV = (1 << BV) - 1;

  extern __shared__ __align__(128) uint8_t smem[];
  // the page is assembled in shared memory and leaves by one bulk copy
  const QuantSmem sm = quant_smem(R, D, G, lay_bytes);
  uint16_t* kt = reinterpret_cast<uint16_t*>(smem + sm.kt);  // [R][D]
  uint16_t* vt = reinterpret_cast<uint16_t*>(smem + sm.vt);  // [R][D]
  GroupQ* kq = reinterpret_cast<GroupQ*>(smem + sm.kq);      // [R/G][D]
  GroupQ* vq = reinterpret_cast<GroupQ*>(smem + sm.vq);      // [R][D/G]
  uint8_t* sidx = smem + sm.sidx;                            // [R][kMaxSparse]
  uint8_t* pg = smem + sm.pg;                                // page image
  __shared__ __align__(8) uint64_t bar;
  __shared__ float thr_s[2][16];  // codebook decision thresholds (keys, values)

  const int64_t tok0 = p.src_tok0 + (int64_t)page * R;
  const uint16_t* ksrc = p.k_src + (int64_t)unit * p.src_unit_stride + tok0 * D;
  const uint16_t* vsrc = p.v_src + (int64_t)unit * p.src_unit_stride + tok0 * D;
  uint8_t* dst = p.pages + (int64_t)unit * p.unit_page_stride + (p.page0 + page) * (int64_t)lay_bytes;
#ifdef KVQ_DEBUG_CHECKS
  {
    const int64_t so = (int64_t)unit * p.src_unit_stride + tok0 * D;
    const int64_t po = (int64_t)unit * p.unit_page_stride + (p.page0 + page) * (int64_t)lay_bytes;
    if (so < 0 || so + (int64_t)R * D > p.src_elems || po < 0 || po + lay_bytes > p.pages_bytes) {
      if (tid == 0) report_error(p.err, kDevBounds);
      return;  // the whole CTA, before any barrier
    }
  }
#endif

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
  {
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_s2g(dst, pg, (uint32_t)lay_bytes);
      bulk_commit();
      bulk_wait_all();
    }
  }
}

// ---------------------------------------------------------------------------------------------
// The common page shape (R = 128, D = 128, G = 32, 2- or 4-bit codes in fragment order, no sparse
// entries, uniform codes): one CTA of 512 threads per page, three CTAs per SM.  Warps 0-7 take the
// keys and warps 8-15 the values, through three phases separated by two barriers:
//   fill    keys: 16-byte cp.async copies into a token-major tile; values: 16-byte loads of 8
//           tokens x 8 channels, transposed in registers into a channel-major tile of token pairs
//           (every operand register of the value products pairs two tokens of one channel);
//   ranges  keys: a thread per (32-token group, channel pair) walks its column; values: a thread
//           per (token pair, 32-channel group) walks its row; both on fp16 pairs (fp16 minimum and
//           maximum are exact), then the zero point, the step and -- for 2-bit codes -- the three
//           fp16 decision thresholds of each group (kvq::qthr), or the group quantizer (4-bit);
//   codes   a thread per (16-token tile, lane) builds that lane's fragment words: 2-bit codes by
//           comparing fp16 pairs with the thresholds (two packed compares and a select per two
//           codes: bit 1 from t1, bit 0 from t2 or t0 as bit 1 says), 4-bit
//           codes with the group quantizer; each thread stores its words with 16-byte stores.
// Both tiles are XOR-swizzled in 16-byte chunks so that no phase has shared-memory bank
// conflicts: key row t keeps chunk c at c ^ (t & 7); value row (channel) c keeps chunk q at
// q ^ ((c ^ (c >> 3)) & 7).
constexpr int kStdThreads = 512;

__device__ __forceinline__ int kswz(int cp, int tok) { return (((cp >> 2) ^ (tok & 7)) << 2) | (cp & 3); }
__device__ __forceinline__ int vswz(int tp, int ch) { return (((tp >> 2) ^ ((ch ^ (ch >> 3)) & 7)) << 2) | (tp & 3); }

// Shared memory of the common-shape kernel, in 32-bit words.
template <int BK, int BV>
struct StdSmem {
  static constexpr int ks = 0;                                            // [128 tok][64] key pairs
  static constexpr int vt = ks + 128 * 64;                                // [128 ch][64] value token pairs
  static constexpr int kt = vt + 128 * 64;                                // thresholds [4][3][64] | GroupQ [4][128]
  static constexpr int vth = kt + (BK == 2 ? 4 * 3 * 64 : 4 * 128 * 2);  // thresholds [4][3][64] | GroupQ [128][4]
  static constexpr int vms = vth + (BV == 2 ? 4 * 3 * 64 : 128 * 4 * 2);  // value zero point / step words [128][4]
  static constexpr int words = vms + 128 * 4;
  static constexpr size_t bytes = (size_t)words * 4;
};

__device__ __forceinline__ __half2 as_h2(uint32_t x) {
  __half2 h;
  memcpy(&h, &x, 4);
  return h;
}

// 4-bit codes of an fp16 pair of group values (x >= the group's minimum) with each half's quantizer,
// codes at bits 0-3 and 16-19, on packed fp32 pairs: r = (x - z) * (1/s), t = r + 1.5*2^23 holds
// rint(r) in its low mantissa bits, the clamp is one integer minimum.  Where r lies within 2^-14 of a
// half-integer (where it could round differently from the IEEE quotient) the pair's bit 0 / 1 of
// `near` is set and the caller takes that code again with code4_exact.
__device__ __forceinline__ uint32_t code4_pair_fast(uint32_t x, const GroupQ& q0, const GroupQ& q1, uint32_t& near) {
  constexpr float M = 0x1.8p23f;
  const float2 d = __fadd2_rn(__half22float2(as_h2(x)), make_float2(-q0.zf(), -q1.zf()));
  const float2 r = __fmul2_rn(d, make_float2(q0.inv, q1.inv));
  const float2 t = __fadd2_rn(r, make_float2(M, M));
  const float2 e = __ffma2_rn(__fadd2_rn(t, make_float2(-M, -M)), make_float2(-1.0f, -1.0f), r);
  near = (fabsf(e.x) >= 0.5f - 0x1.0p-14f ? 1u : 0u) | (fabsf(e.y) >= 0.5f - 0x1.0p-14f ? 2u : 0u);
  return min(__float_as_uint(t.x) - __float_as_uint(M), 15u) | (min(__float_as_uint(t.y) - __float_as_uint(M), 15u) << 16);
}
__device__ __forceinline__ uint32_t code4_exact(float x, const GroupQ& g) {
  const float q = rintf(__fdiv_rn(__fsub_rn(x, g.zf()), g.sf()));  // s > 0: a zero step is never near
  return (uint32_t)fminf(fmaxf(q, 0.0f), 15.0f);
}

// 4-bit codes of an fp16 pair with each half's quantizer: codes at bits 0-3 and 16-19.
__device__ __forceinline__ uint32_t code4_pair(uint32_t x, const GroupQ& q0, const GroupQ& q1) {
  const float2 f = __half22float2(as_h2(x));
  return quant_code(f.x, q0, 15) | (quant_code(f.y, q1, 15) << 16);
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

// A barrier over one half of the 512 threads (warps 0-7 or warps 8-15).
__device__ __forceinline__ void half_barrier(bool first_half) {
  if (first_half) asm volatile("bar.sync 1, 256;" ::: "memory");
  else asm volatile("bar.sync 2, 256;" ::: "memory");
}

template <int BK, int BV>
__global__ void __launch_bounds__(kStdThreads, 3) quantize_std_kernel(const QuantizeParams p) {
  static_assert((BK == 2 || BK == 4) && (BV == 2 || BV == 4), "fragment-order pages hold 2- or 4-bit codes");
  using SP = StdPage<BK, BV>;
  using SM = StdSmem<BK, BV>;
  constexpr int D = kHeadDim;
  const int page = blockIdx.x, unit = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool keys = warp < 8;
  const int wl = warp & 7, ht = tid & 255;
  extern __shared__ __align__(128) uint32_t sw[];
  uint32_t* const ks = sw + SM::ks;
  uint32_t* const vt = sw + SM::vt;

  const int64_t tok0 = p.src_tok0 + (int64_t)page * 128;
  const uint16_t* ksrc = p.k_src + (int64_t)unit * p.src_unit_stride + tok0 * D;
  const uint16_t* vsrc = p.v_src + (int64_t)unit * p.src_unit_stride + tok0 * D;
  uint8_t* const dst = p.pages + (int64_t)unit * p.unit_page_stride + (p.page0 + page) * (int64_t)SP::bytes;
#ifdef KVQ_DEBUG_CHECKS
  {
    const int64_t so = (int64_t)unit * p.src_unit_stride + tok0 * D;
    const int64_t po = (int64_t)unit * p.unit_page_stride + (p.page0 + page) * (int64_t)SP::bytes;
    if (so < 0 || so + 128 * D > p.src_elems || po < 0 || po + SP::bytes > p.pages_bytes) {
      if (tid == 0) report_error(p.err, kDevBounds);
      return;  // the whole CTA, before any barrier
    }
  }
#endif

  // ---- fill
  if (keys) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = ht + 256 * i, row = q >> 4, c16 = q & 15;
      cp_async16(ks + row * 64 + ((c16 ^ (row & 7)) << 2), ksrc + row * D + c16 * 8);
    }
    cp_async_commit();
    cp_async_wait_all();
  } else {
    const int o = ht >> 4, c8 = ht & 15;  // token octet, channel octet
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      // the upper channel octets take the two token quads in the other order: the 16 lanes of a
      // half-warp then store to 16 different 8-byte slots
      const int half = hh ^ (c8 >> 3);
      uint4 r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        r[i] = __ldcs(reinterpret_cast<const uint4*>(vsrc + (8 * o + 4 * half + i) * D + 8 * c8));
      const int tp = 4 * o + 2 * half;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t a0 = comp(r[0], w), a1 = comp(r[1], w), a2 = comp(r[2], w), a3 = comp(r[3], w);
        const int ch0 = 8 * c8 + 2 * w, ch1 = ch0 + 1;
        *reinterpret_cast<uint2*>(vt + ch0 * 64 + vswz(tp, ch0)) =
            make_uint2(__byte_perm(a0, a1, 0x5410), __byte_perm(a2, a3, 0x5410));
        *reinterpret_cast<uint2*>(vt + ch1 * 64 + vswz(tp, ch1)) =
            make_uint2(__byte_perm(a0, a1, 0x7632), __byte_perm(a2, a3, 0x7632));
      }
    }
  }
  // keys (warps 0-7) and values (warps 8-15) share nothing until the end: each half waits only for
  // itself, so one half computes while the other still waits for its data (barriers 1 and 2, as
  // immediates: a barrier index in a register would reserve all sixteen and cost occupancy)
  half_barrier(keys);

  // ---- ranges, zero points and steps, thresholds
  {
    const int grp = wl >> 1, pos = 32 * (wl & 1) + lane;  // keys: (token group, channel pair); values: (channel group, token pair)
    // the swizzled word of this thread's column in row i of its group is base[(i & 7) ^ ...]: eight
    // per-thread offsets cover the 32 rows of the scan
    __half2 mn, mx;
    if (keys) {
      // key row 32*grp + t keeps chunk (pos >> 2) at (pos >> 2) ^ (t & 7)
      const uint32_t* col = ks + 32 * grp * 64;
      int off[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) off[k] = (((pos >> 2) ^ k) << 2) | (pos & 3);
      mn = mx = as_h2(col[off[0]]);
#pragma unroll
      for (int t = 1; t < 32; ++t) {
        const __half2 v = as_h2(col[t * 64 + off[t & 7]]);
        mn = __hmin2(mn, v);
        mx = __hmax2(mx, v);
      }
    } else {
      // value row (channel) 32*grp + c keeps chunk (pos >> 2) at (pos >> 2) ^ ((c & 7) ^ (c >> 3) ^ 4*(grp & 1))
      const uint32_t* col = vt + 32 * grp * 64;
      int off[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) off[k] = (((pos >> 2) ^ k ^ (4 * (grp & 1))) << 2) | (pos & 3);
      mn = mx = as_h2(col[off[0]]);
#pragma unroll
      for (int c = 1; c < 32; ++c) {
        const __half2 v = as_h2(col[c * 64 + off[(c & 7) ^ (c >> 3)]]);
        mn = __hmin2(mn, v);
        mx = __hmax2(mx, v);
      }
    }
    const float2 fmn = __half22float2(mn), fmx = __half22float2(mx);
    // the two groups of this thread: keys channels 2*pos, 2*pos + 1; values tokens 2*pos, 2*pos + 1
    const int B = keys ? BK : BV;
    uint32_t zs0, zs1;
    if (B == 2) {
      uint32_t ta[3], tb[3];
      zs0 = qthr::thresholds2(fmn.x, fmx.x, ta);
      zs1 = qthr::thresholds2(fmn.y, fmx.y, tb);
      uint32_t* th = sw + (keys ? SM::kt : SM::vth) + grp * 3 * 64 + pos;
#pragma unroll
      for (int k = 0; k < 3; ++k) th[k * 64] = ta[k] | (tb[k] << 16);
    } else {
      const GroupQ q0 = group_params(fmn.x, fmx.x, 15), q1 = group_params(fmn.y, fmx.y, 15);
      zs0 = q0.bits;
      zs1 = q1.bits;
      GroupQ* gq = reinterpret_cast<GroupQ*>(sw + (keys ? SM::kt : SM::vth));
      if (keys) {
        gq[grp * 128 + 2 * pos] = q0;
        gq[grp * 128 + 2 * pos + 1] = q1;
      } else {
        gq[(2 * pos) * 4 + grp] = q0;
        gq[(2 * pos + 1) * 4 + grp] = q1;
      }
    }
    if (keys) {
      *reinterpret_cast<uint2*>(dst + SP::km + (grp * 128 + 2 * pos) * 4) = make_uint2(zs0, zs1);
    } else {
      sw[SM::vms + (2 * pos) * 4 + grp] = zs0;
      sw[SM::vms + (2 * pos + 1) * 4 + grp] = zs1;
    }
  }
  half_barrier(keys);

  // ---- codes in fragment order: thread = (16-token tile wl, lane).  Every load address is a
  //      per-lane base plus a compile-time offset: the XOR swizzle only depends on the lane (g8)
  //      and on loop constants, so the swizzled chunk offsets are taken once per lane.
  const int g8 = lane >> 2, t4 = lane & 3;
  if (keys) {
    // key rows 16m + g8 + 8r (row & 7 = g8); the lane's channel pairs are cp = 16q + 4j + t4 (4-bit
    // words: q = word index u) or 32u + 4j + t4 (2-bit words), chunk cp >> 2, swizzled by g8
    const int m = wl, gk = m >> 1;
    const uint32_t* kr = ks + (16 * m + g8) * 64 + t4;
    int sj[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) sj[j] = (j ^ g8) << 2;
    uint32_t wd[2 * BK];
#pragma unroll
    for (int i = 0; i < 2 * BK; ++i) wd[i] = 0;
    if constexpr (BK == 2) {
      // word r*2 + u, pair j: channel pair 32u + 4j + t4 (chunk 8u + j)
      const uint32_t* th = sw + SM::kt + gk * 3 * 64 + t4;
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t t0 = th[32 * u + 4 * j], t1 = th[64 + 32 * u + 4 * j], t2 = th[128 + 32 * u + 4 * j];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const __half2 x = as_h2(kr[r * 8 * 64 + 32 * u + sj[j]]);
            // code = thresholds reached (t0 <= t1 <= t2): bit 1 = x >= t1; bit 0 = x >= t2 where
            // x >= t1, else x >= t0 -- two packed compares and a select per two codes
            const uint32_t m1 = __hge2_mask(x, as_h2(t1));
            const uint32_t m0 = __hge2_mask(x, as_h2((m1 & t2) | (~m1 & t0)));
            wd[r * 2 + u] |= (m0 & (0x00010001u << (2 * j))) | (m1 & (0x00020002u << (2 * j)));
          }
        }
    } else {
      // word r*4 + u, pair j: channel pair 16u + 4j + t4 (chunk 4u + j)
      const GroupQ* gq = reinterpret_cast<const GroupQ*>(sw + SM::kt) + gk * 128 + 2 * t4;
      uint32_t nm0 = 0, nm1 = 0;  // near-tie elements: bit 4c + 2r + e of element e of pair (chunk c, row r)
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = 4 * u + j;  // chunk
          const GroupQ q0 = gq[2 * (16 * u + 4 * j)], q1 = gq[2 * (16 * u + 4 * j) + 1];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const uint32_t x = kr[r * 8 * 64 + 4 * (c & 8) + sj[c & 7]];
            uint32_t nb;
            wd[r * 4 + u] |= code4_pair_fast(x, q0, q1, nb) << (4 * j);
            const int b = 4 * c + 2 * r;
            if (b < 32) nm0 |= nb << b;
            else nm1 |= nb << (b - 32);
          }
        }
      // the rare near-tie elements again with the IEEE quotient, behind one vote
      if (__any_sync(0xffffffffu, (nm0 | nm1) != 0)) {
        uint64_t nm = ((uint64_t)nm1 << 32) | nm0;
        while (nm) {
          const int b = __ffsll((long long)nm) - 1;
          nm &= nm - 1;
          const int e = b & 1, r = (b >> 1) & 1, c = b >> 2, u = c >> 2, j = c & 3;
          const uint32_t x = kr[r * 8 * 64 + 4 * (c & 8) + (((c & 7) ^ g8) << 2)];
          const uint32_t code = code4_exact(h2f((uint16_t)(e ? (x >> 16) : (x & 0xFFFFu))), gq[2 * (16 * u + 4 * j) + e]);
          const int sh = 4 * j + 16 * e;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i == r * 4 + u) wd[i] = (wd[i] & ~(0xFu << sh)) | (code << sh);
        }
      }
    }
    uint4* o = reinterpret_cast<uint4*>(dst + SP::kc) + (m * 32 + lane) * (2 * BK / 4);
#pragma unroll
    for (int i = 0; i < 2 * BK / 4; ++i) o[i] = make_uint4(wd[4 * i], wd[4 * i + 1], wd[4 * i + 2], wd[4 * i + 3]);
  } else {
    // value token pairs tp = 8m + 4(r >> 1) + t4 (chunk 2m ^ (r >> 1)), channels ch = 16mc + g8 + 8(r & 1)
    // (ch & 7 = g8, ch >> 3 = 2mc + (r & 1)): the swizzled chunk is (2m ^ g8) ^ K with
    // K = (r >> 1) ^ ((2mc + (r & 1)) & 7), so eight per-lane bases cover every load
    const int m = wl;
    const int A = (2 * m) ^ g8;
    const uint32_t* vb[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) vb[k] = vt + g8 * 64 + (((A ^ k) << 2) | t4);
    uint32_t wd[2 * BV];
#pragma unroll
    for (int i = 0; i < 2 * BV; ++i) wd[i] = 0;
    if constexpr (BV == 2) {
      // word r, pair j = M-tile mc; thresholds of (token pair, group mc >> 1)
      const uint32_t* th = sw + SM::vth + 8 * m + t4;
#pragma unroll
      for (int rh = 0; rh < 2; ++rh)
#pragma unroll
        for (int gv = 0; gv < 4; ++gv) {
          const uint32_t t0 = th[gv * 192 + 4 * rh], t1 = th[gv * 192 + 64 + 4 * rh], t2 = th[gv * 192 + 128 + 4 * rh];
#pragma unroll
          for (int rl = 0; rl < 2; ++rl)
#pragma unroll
            for (int jl = 0; jl < 2; ++jl) {
              const int r = 2 * rh + rl, j = 2 * gv + jl;
              const int K = rh ^ ((2 * j + rl) & 7);
              const __half2 x = as_h2(vb[K][(16 * j + 8 * rl) * 64]);
              const uint32_t m1 = __hge2_mask(x, as_h2(t1));
              const uint32_t m0 = __hge2_mask(x, as_h2((m1 & t2) | (~m1 & t0)));
              wd[r] |= (m0 & (0x00010001u << (2 * j))) | (m1 & (0x00020002u << (2 * j)));
            }
        }
    } else {
      // word r*2 + u, pair j: M-tile mc = 4u + j
      const GroupQ* gq = reinterpret_cast<const GroupQ*>(sw + SM::vth) + (2 * (8 * m + t4)) * 4;
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int mc = 4 * u + j, gv = mc >> 1;
            const int K = (r >> 1) ^ ((2 * mc + (r & 1)) & 7);
            const uint32_t x = vb[K][(16 * mc + 8 * (r & 1)) * 64];
            const int tb = 2 * 4 * (r >> 1);  // token offset 8(r >> 1), times 4 groups per token
            wd[r * 2 + u] |= code4_pair(x, gq[tb * 4 + gv], gq[(tb + 1) * 4 + gv]) << (4 * j);
          }
    }
    uint4* o = reinterpret_cast<uint4*>(dst + SP::vc) + (m * 32 + lane) * (2 * BV / 4);
#pragma unroll
    for (int i = 0; i < 2 * BV / 4; ++i) o[i] = make_uint4(wd[4 * i], wd[4 * i + 1], wd[4 * i + 2], wd[4 * i + 3]);
    // the value zero points and steps (2 KB) leave in 16-byte stores
    if (ht < 128) reinterpret_cast<uint4*>(dst + SP::vm)[ht] = reinterpret_cast<const uint4*>(sw + SM::vms)[ht];
  }
}

// ---------------------------------------------------------------------------------------------
// Pages whose codes are token-major bitstreams (3-bit codes, or keys rotated at decode; uniform
// codes), R = 128, D = 128, G = 32 or 64, up to four sparse entries per key vector: one CTA of 512
// threads per page, two CTAs per SM (64 registers), the tiles and swizzles of quantize_std_kernel.
//   fill     as in quantize_std_kernel;
//   sparse   warps 0-7: a thread per (token, 64-channel half) finds the half's largest |x| in
//            channel order, the two lanes of a token merge their lists by a shuffle (larger |x|
//            first, ties to the lower channel); each entry is written out and replaced in the tile by a
//            NaN, which the fp16 minimum and maximum skip and which quantizes to code 0 --
//            exactly the exclusion the method asks for;
//   ranges   warps 0-7: key ranges and quantizers, a thread per (token group, channel pair);
//            warps 8-15: value ranges and quantizers, a thread per (token pair, channel group);
//   codes    warps 0-7 the key codes, warps 8-15 the value codes: two (token, 32-channel chunk)
//            per thread, each packed 32 at a time into B words.
// The key half (warps 0-7) and the value half (warps 8-15) share nothing, so each waits at barriers
// of its own and computes while the other still waits for its data.
// A code comes from the group's reciprocal; elements whose product lies within 2^-14 of a
// half-integer (where it could round differently from the IEEE quotient) are collected in a mask
// and taken again with the IEEE quotient after the loop, behind one vote per chunk.
struct __align__(8) QuantF {  // a group quantizer in the form the code loop uses
  float inv, nz;  // 1/s and -z
};
// shared memory of quantize_bits_kernel: the two tiles, the key and value quantizers (QuantF) and
// their stored (zero point, step) words
constexpr size_t kBitsSmemBytes = (size_t)(2 * 128 * 64 + 4 * 128 * 2 + 128 * 4 * 2 + 4 * 128 + 128 * 4) * 4;

// Codes of 32 channels of one token (x: fp16 values, e-th of chunk at (w4[e/2] >> 16*(e&1))) into
// BITS words; q(c) gives channel c's quantizer and bits(c) its stored (zero point, step).
// xval(c) is called with compile-time c in the main loop; xdyn(c) and qbits(c) only in the rare
// pass over near-tie elements, with a run-time c (so they read shared memory, not register arrays).
template <int BITS, class QF, class QB, class XF, class XD>
__device__ __forceinline__ void code_chunk(const XF& xval, const XD& xdyn, const QF& qf, const QB& qbits,
                                           uint32_t (&w)[BITS]) {
  constexpr int L = (1 << BITS) - 1;
  constexpr float M = 0x1.8p23f;  // r + M has rint(r) in its low mantissa bits (0 <= r < 2^22)
#pragma unroll
  for (int i = 0; i < BITS; ++i) w[i] = 0;
  uint32_t near = 0;
  // two codes at a time on packed fp32 pairs: d = max(x - z, 0) (a sparse entry, NaN, gives 0 and
  // code 0; every other x is at least the group minimum z), r = d / s as d * (1/s), t = r + M,
  // code = min(rint(r), L) from t's bits; near when |r - rint(r)| >= 1/2 - 2^-14 (exact difference)
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    const QuantF q0 = qf(c), q1 = qf(c + 1);
    float2 d = __fadd2_rn(make_float2(xval(c), xval(c + 1)), make_float2(q0.nz, q1.nz));
    d = make_float2(fmaxf(d.x, 0.0f), fmaxf(d.y, 0.0f));
    const float2 r = __fmul2_rn(d, make_float2(q0.inv, q1.inv));
    const float2 t = __fadd2_rn(r, make_float2(M, M));
    const float2 e = __ffma2_rn(__fadd2_rn(t, make_float2(-M, -M)), make_float2(-1.0f, -1.0f), r);
    near |= (fabsf(e.x) >= 0.5f - 0x1.0p-14f ? 1u << c : 0u) | (fabsf(e.y) >= 0.5f - 0x1.0p-14f ? 2u << c : 0u);
    const uint32_t code0 = min(__float_as_uint(t.x) - __float_as_uint(M), (uint32_t)L);
    const uint32_t code1 = min(__float_as_uint(t.y) - __float_as_uint(M), (uint32_t)L);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t code = k ? code1 : code0;
      const int b = BITS * (c + k);
      w[b >> 5] |= code << (b & 31);
      if ((b & 31) + BITS > 32) w[(b >> 5) + 1] |= code >> (32 - (b & 31));
    }
  }
  if (__any_sync(0xffffffffu, near != 0)) {
    while (near) {
      const int c = __ffs(near) - 1;
      near &= near - 1;
      const uint32_t zs = qbits(c);
      const float sf = h2f((uint16_t)(zs >> 16));
      const float rq = rintf(__fdiv_rn(__fsub_rn(xdyn(c), h2f((uint16_t)(zs & 0xFFFFu))), sf));  // s > 0 here
      const uint32_t code = (uint32_t)fminf(fmaxf(rq, 0.0f), (float)L);
      const int b = BITS * c;
      const uint64_t m = (uint64_t)L << (b & 31);
      const uint64_t v = (uint64_t)code << (b & 31);
#pragma unroll
      for (int i = 0; i < BITS; ++i) {  // word b >> 5 and, for a code that straddles, the next one
        if (i == (b >> 5)) w[i] = (w[i] & ~(uint32_t)m) | (uint32_t)v;
        if (i == (b >> 5) + 1) w[i] = (w[i] & ~(uint32_t)(m >> 32)) | (uint32_t)(v >> 32);
      }
    }
  }
}

template <int BK, int BV>
__global__ void __launch_bounds__(kStdThreads, 2) quantize_bits_kernel(const QuantizeParams p) {
  constexpr int D = kHeadDim, R = 128;
  constexpr int LK = (1 << BK) - 1, LV = (1 << BV) - 1;
  constexpr int WK = D * BK / 32, WV = D * BV / 32;  // words of one token's bitstream
  const int G = p.G, nsp = p.nsp;
  const int ngv = D / G, ngk = R / G;  // value groups per token, key groups per page
  const int page = blockIdx.x, unit = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ht = tid & 255;
  extern __shared__ __align__(128) uint32_t sw[];
  uint32_t* const ks = sw;                                           // [128 tok][64] key pairs
  uint32_t* const vt = sw + 128 * 64;                                // [128 ch][64] value token pairs
  QuantF* const kqf = reinterpret_cast<QuantF*>(sw + 2 * 128 * 64);  // [R/G][D]
  QuantF* const vqf = kqf + 4 * 128;                                 // [R][D/G]
  uint32_t* const kzs = reinterpret_cast<uint32_t*>(vqf + 128 * 4);  // [R/G][D] stored (zero point, step)
  uint32_t* const vzs = kzs + 4 * 128;                               // [R][D/G]
  const int64_t tok0 = p.src_tok0 + (int64_t)page * R;
  const uint16_t* ksrc = p.k_src + (int64_t)unit * p.src_unit_stride + tok0 * D;
  const uint16_t* vsrc = p.v_src + (int64_t)unit * p.src_unit_stride + tok0 * D;
  uint8_t* const dst = p.pages + (int64_t)unit * p.unit_page_stride + (p.page0 + page) * (int64_t)p.lay.bytes;
#ifdef KVQ_DEBUG_CHECKS
  {
    const int64_t so = (int64_t)unit * p.src_unit_stride + tok0 * D;
    const int64_t po = (int64_t)unit * p.unit_page_stride + (p.page0 + page) * (int64_t)p.lay.bytes;
    if (so < 0 || so + R * D > p.src_elems || po < 0 || po + p.lay.bytes > p.pages_bytes) {
      if (tid == 0) report_error(p.err, kDevBounds);
      return;  // the whole CTA, before any barrier
    }
  }
#endif

  // ---- fill (as in quantize_std_kernel)
  if (warp < 8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = ht + 256 * i, row = q >> 4, c16 = q & 15;
      cp_async16(ks + row * 64 + ((c16 ^ (row & 7)) << 2), ksrc + row * D + c16 * 8);
    }
    cp_async_commit();
    cp_async_wait_all();
  } else {
    const int o = ht >> 4, c8 = ht & 15;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int half = hh ^ (c8 >> 3);
      uint4 r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        r[i] = __ldcs(reinterpret_cast<const uint4*>(vsrc + (8 * o + 4 * half + i) * D + 8 * c8));
      const int tp = 4 * o + 2 * half;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t a0 = comp(r[0], w), a1 = comp(r[1], w), a2 = comp(r[2], w), a3 = comp(r[3], w);
        const int ch0 = 8 * c8 + 2 * w, ch1 = ch0 + 1;
        *reinterpret_cast<uint2*>(vt + ch0 * 64 + vswz(tp, ch0)) =
            make_uint2(__byte_perm(a0, a1, 0x5410), __byte_perm(a2, a3, 0x5410));
        *reinterpret_cast<uint2*>(vt + ch1 * 64 + vswz(tp, ch1)) =
            make_uint2(__byte_perm(a0, a1, 0x7632), __byte_perm(a2, a3, 0x7632));
      }
    }
  }
  half_barrier(warp < 8);

  // ---- sparse key entries (warps 0-7): thread = (token t, half qt of 64 channels); lanes 2t', 2t'+1
  //      of a warp hold one token's two halves.  |x| as fp16 bits orders like its value; entry (v, c)
  //      outranks (v', c') when v > v', or v == v' and c < c' (ties to the lower channel).
  if (nsp > 0 && warp < 8) {
    const int t = tid >> 1, qt = tid & 1;
    const uint32_t* row = ks + t * 64;
    int bc[kMaxSparse];  // the chosen channels (unused slots hold a channel past the end)
    if (nsp <= 2) {
      // two slots, branch-free: each entry as the key (|x| bits << 7) | (127 - channel), so that a
      // larger key is a larger |x|, or the same |x| at a lower channel, and no two keys are equal;
      // the two largest keys take three integer min/max per entry
      int k0 = -1, k1 = -1;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int ch = 8 * qt + i;  // 16-byte chunk: channels 8ch .. 8ch+7
        const uint4 v = *reinterpret_cast<const uint4*>(row + ((ch ^ (t & 7)) << 2));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t w = w4[e >> 1];
          const int k = (int)((e & 1) ? (((w >> 9) & (0x7FFFu << 7)) | (uint32_t)(127 - (8 * ch + e)))
                                      : (((w & 0x7FFFu) << 7) | (uint32_t)(127 - (8 * ch + e))));
          k1 = max(k1, min(k0, k));
          k0 = max(k0, k);
        }
      }
      // merge the two halves' pairs
#pragma unroll
      for (int off = 1; off < 2; off <<= 1) {
        const int o0 = __shfl_xor_sync(0xffffffffu, k0, off), o1 = __shfl_xor_sync(0xffffffffu, k1, off);
        k1 = max(min(k0, o0), max(k1, o1));
        k0 = max(k0, o0);
      }
      const int c0 = 127 - (k0 & 127), c1 = 127 - (k1 & 127);
      bc[0] = min(c0, c1);
      bc[1] = nsp == 2 ? max(c0, c1) : (1 << 20);
      bc[0] = nsp == 2 ? bc[0] : c0;
#pragma unroll
      for (int k = 2; k < kMaxSparse; ++k) bc[k] = 1 << 20;
    } else {
      int bv[kMaxSparse];
#pragma unroll
      for (int k = 0; k < kMaxSparse; ++k) {
        bv[k] = -1;
        bc[k] = 1 << 20;
      }
      auto outranks = [](int v, int c, int v2, int c2) { return v > v2 || (v == v2 && c < c2); };
      auto insert = [&](int v, int c) {
#pragma unroll
        for (int k = kMaxSparse - 1; k >= 0; --k) {
          if (k >= nsp || !outranks(v, c, bv[k], bc[k])) continue;
          if (k == 0 || !outranks(v, c, bv[k - 1], bc[k - 1])) {
            bv[k] = v;
            bc[k] = c;
          } else {
            bv[k] = bv[k - 1];
            bc[k] = bc[k - 1];
          }
        }
      };
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int ch = 8 * qt + i;
        const uint4 v = *reinterpret_cast<const uint4*>(row + ((ch ^ (t & 7)) << 2));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) insert((int)((w4[e >> 1] >> (16 * (e & 1))) & 0x7FFFu), 8 * ch + e);
      }
#pragma unroll
      for (int off = 1; off < 2; off <<= 1) {
        int ov[kMaxSparse], oc[kMaxSparse];
#pragma unroll
        for (int k = 0; k < kMaxSparse; ++k) {
          ov[k] = __shfl_xor_sync(0xffffffffu, bv[k], off);
          oc[k] = __shfl_xor_sync(0xffffffffu, bc[k], off);
        }
#pragma unroll
        for (int k = 0; k < kMaxSparse; ++k)
          if (k < nsp) insert(ov[k], oc[k]);
      }
      // ascending channel order (a sorting network; unused slots stay last)
      auto order = [&](int i, int j) {
        const int lo = min(bc[i], bc[j]), hi = max(bc[i], bc[j]);
        bc[i] = lo;
        bc[j] = hi;
      };
      order(0, 1);
      order(2, 3);
      order(0, 2);
      order(1, 3);
      order(1, 2);
    }
    // each lane writes and masks the entries of its own half
    uint16_t* rowh = reinterpret_cast<uint16_t*>(ks + t * 64);
#pragma unroll
    for (int k = 0; k < kMaxSparse; ++k) {
      const int c = bc[k];
      if (k >= nsp || (c >> 6) != qt) continue;
      const int hw = 2 * ((((c >> 3) ^ (t & 7)) << 2) | ((c >> 1) & 3)) + (c & 1);  // half index in the row
      dst[p.lay.off_si + t * nsp + k] = (uint8_t)c;
      reinterpret_cast<uint16_t*>(dst + p.lay.off_sv)[t * nsp + k] = rowh[hw];
      rowh[hw] = 0x7E00u;  // NaN
    }
    half_barrier(true);  // the key half only
  }

  // ---- ranges and quantizers: keys (warps 0-7), values (warps 8-15)
  if (warp < 8) {
    for (int it = tid; it < ngk * 64; it += 256) {
      const int gk = it >> 6, cp = it & 63;  // token group, channel pair
      const uint32_t* col = ks + G * gk * 64;
      int off[8];  // row 8*b + k keeps chunk cp >> 2 at (cp >> 2) ^ k
#pragma unroll
      for (int k = 0; k < 8; ++k) off[k] = (((cp >> 2) ^ k) << 2) | (cp & 3);
      // NaN (a sparse entry) never wins a minimum or maximum against a number: start from NaN
      __half2 mn = as_h2(0x7E007E00u), mx = mn;
      for (int tb = 0; tb < G; tb += 8) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const __half2 v = as_h2(col[(tb + k) * 64 + off[k]]);
          mn = __hmin2(mn, v);
          mx = __hmax2(mx, v);
        }
      }
      float2 fmn = __half22float2(mn), fmx = __half22float2(mx);
      if (fmn.x != fmn.x) fmn.x = fmx.x = 0.0f;  // every entry sparse: range 0
      if (fmn.y != fmn.y) fmn.y = fmx.y = 0.0f;
      const GroupQ q0 = group_params(fmn.x, fmx.x, LK), q1 = group_params(fmn.y, fmx.y, LK);
      kqf[gk * 128 + 2 * cp] = QuantF{q0.inv, -q0.zf()};
      kqf[gk * 128 + 2 * cp + 1] = QuantF{q1.inv, -q1.zf()};
      kzs[gk * 128 + 2 * cp] = q0.bits;
      kzs[gk * 128 + 2 * cp + 1] = q1.bits;
      *reinterpret_cast<uint2*>(dst + p.lay.off_km + (gk * 128 + 2 * cp) * 4) = make_uint2(q0.bits, q1.bits);
    }
  } else {
    for (int it = ht; it < 64 * ngv; it += 256) {
      const int g = it >> 6, tp = it & 63;  // channel group, tokens 2*tp, 2*tp + 1
      const int c0 = G * g;
      __half2 mn = as_h2(0x7E007E00u), mx = mn;  // values hold no NaN: the first row replaces these
      for (int cb = 0; cb < G; cb += 8) {
        // rows c0 + cb + k keep chunk tp >> 2 at (tp >> 2) ^ k ^ (((c0 + cb) >> 3) & 7)
        const int u = (tp >> 2) ^ (((c0 + cb) >> 3) & 7);
        const uint32_t* rows = vt + (c0 + cb) * 64 + (tp & 3);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const __half2 v = as_h2(rows[k * 64 + ((u ^ k) << 2)]);
          mn = __hmin2(mn, v);
          mx = __hmax2(mx, v);
        }
      }
      const float2 fmn = __half22float2(mn), fmx = __half22float2(mx);
      const GroupQ q0 = group_params(fmn.x, fmx.x, LV), q1 = group_params(fmn.y, fmx.y, LV);
      vqf[(2 * tp) * ngv + g] = QuantF{q0.inv, -q0.zf()};
      vqf[(2 * tp + 1) * ngv + g] = QuantF{q1.inv, -q1.zf()};
      vzs[(2 * tp) * ngv + g] = q0.bits;
      vzs[(2 * tp + 1) * ngv + g] = q1.bits;
      uint32_t* vm = reinterpret_cast<uint32_t*>(dst + p.lay.off_vm);
      vm[(2 * tp) * ngv + g] = q0.bits;
      vm[(2 * tp + 1) * ngv + g] = q1.bits;
    }
  }
  half_barrier(warp < 8);

  // ---- codes: the key half codes the keys and the value half the values, two 32-channel chunks a
  //      thread, so each half goes on as soon as its own ranges are done
  if (warp < 8) {
    // keys: (token t, chunk q); the quarter-warps read rows t .. t+7, whose swizzles differ
    const int t = ((warp & 3) << 5) | lane;
    const int gk = t / G;
    const uint16_t* rowh = reinterpret_cast<const uint16_t*>(ks + t * 64);
    uint32_t* kc = reinterpret_cast<uint32_t*>(dst + p.lay.off_kc);
#pragma unroll 1
    for (int qq = 0; qq < 2; ++qq) {
      const int q = (warp >> 2) + 2 * qq;
      uint32_t xw[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(ks + t * 64 + (((4 * q + i) ^ (t & 7)) << 2));
        xw[4 * i] = v.x;
        xw[4 * i + 1] = v.y;
        xw[4 * i + 2] = v.z;
        xw[4 * i + 3] = v.w;
      }
      const QuantF* qf = kqf + gk * 128 + 32 * q;
      const uint32_t* qb = kzs + gk * 128 + 32 * q;
      uint32_t w[BK];
      code_chunk<BK>([&](int c) { return h2f((uint16_t)((c & 1) ? (xw[c >> 1] >> 16) : (xw[c >> 1] & 0xFFFFu))); },
                     [&](int c) {
                       const int ch = 32 * q + c;
                       return h2f(rowh[2 * ((((ch >> 3) ^ (t & 7)) << 2) | ((ch >> 1) & 3)) + (ch & 1)]);
                     },
                     [&](int c) { return qf[c]; }, [&](int c) { return qb[c]; }, w);
#pragma unroll
      for (int i = 0; i < BK; ++i) kc[t * WK + q * BK + i] = w[i];
    }
  } else {
    // values: (token 2tp + hf, chunk q); the two lanes of a token pair read the same words
    const int hf = lane & 1, tp = ((warp & 3) << 4) | (lane >> 1);
    const int tok = 2 * tp + hf;
    uint32_t* vc = reinterpret_cast<uint32_t*>(dst + p.lay.off_vc);
#pragma unroll 1
    for (int qq = 0; qq < 2; ++qq) {
      const int q = ((warp - 8) >> 2) + 2 * qq;
      const int g = (32 * q) / G;
      const QuantF qv = vqf[tok * ngv + g];
      const uint32_t qvb = vzs[tok * ngv + g];
      const int c0 = 32 * q;
      int off[8];  // row c0 + c keeps chunk tp >> 2 at (tp >> 2) ^ ((c ^ (c >> 3)) & 7) ^ ((c0 >> 3) & 7)
#pragma unroll
      for (int k = 0; k < 8; ++k) off[k] = (((tp >> 2) ^ k ^ ((c0 >> 3) & 7)) << 2) | (tp & 3);
      const uint32_t* col = vt + c0 * 64;
      uint32_t w[BV];
      code_chunk<BV>(
          [&](int c) {
            const uint32_t x = col[c * 64 + off[(c ^ (c >> 3)) & 7]];
            return h2f((uint16_t)(hf ? (x >> 16) : (x & 0xFFFFu)));
          },
          [&](int c) {
            const uint32_t x = vt[(c0 + c) * 64 + vswz(tp, c0 + c)];
            return h2f((uint16_t)(hf ? (x >> 16) : (x & 0xFFFFu)));
          },
          [&](int) { return qv; }, [&](int) { return qvb; }, w);
#pragma unroll
      for (int i = 0; i < BV; ++i) vc[tok * WV + q * BV + i] = w[i];
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
  dim3 grid((unsigned)n_pages, (unsigned)p.n_units);
  if constexpr (can_std) {
    if (std_shape) {
      constexpr size_t smem = StdSmem<BK, BV>::bytes;
      cudaError_t e = cudaFuncSetAttribute(quantize_std_kernel<BK, BV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
      if (e != cudaSuccess) return e;
      quantize_std_kernel<BK, BV><<<grid, kStdThreads, smem, s>>>(p);
      return cudaGetLastError();
    }
  }
  if (!p.lay.frag && !p.lut && p.R == 128 && p.D == kHeadDim && (p.G == 32 || p.G == 64) && p.nsp <= kMaxSparse) {
    constexpr size_t smem = kBitsSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(quantize_bits_kernel<BK, BV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    quantize_bits_kernel<BK, BV><<<grid, kStdThreads, smem, s>>>(p);
    return cudaGetLastError();
  }
  auto kern = quantize_pages_kernel<BK, BV>;
  const size_t smem = quantize_smem_bytes(p.R, p.D, p.G, p.lay);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kQuantThreads, smem, s>>>(p);
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
