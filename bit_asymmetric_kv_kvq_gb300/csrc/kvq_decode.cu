// Split-K flash-decoding attention over the packed cache, with the merge of
// the splits fused into the same launch.
//
// Decode reads the whole cache for every generated token ("KV cache has a
// geometry problem, not a bit problem", section "Why the KV cache is a
// problem"), so the kernel is built around streaming pages: a producer warp
// issues one bulk (TMA) copy per page into a ring of shared-memory stages,
// four consumer warps dequantize in registers and never touch global memory
// for the cache, and the grid is (token splits) x (batch * kv heads).
//
// Keys are quantized per channel over G-token groups, so inside a group the
// score is linear in the codes:
//   q . k_t = sum_c q_c (z_c + s_c code_tc) = Z + sum_c q'_c code_tc,
//   Z = sum_c q_c z_c,  q'_c = q_c s_c,
// which removes the per-element dequantization multiply.  Values are
// quantized per token over G-channel groups, so
//   sum_t p_t v_tc = sum_t (p_t s_tg) code_tc + sum_t p_t z_tg.
// With pre-RoPE keys the rotation mixes channels c and c + D/2 at a
// token-dependent angle, so keys are dequantized, rotated and then dotted
// (unite.ai page, section "Rotary embeddings complicate keys").
//
// Softmax is online in base 2 with a lazy maximum: the running maximum only
// moves when a score exceeds it by more than 8 (log2 units), which keeps
// every weight below 2^8 and skips most rescales.  Each CTA writes one
// unnormalised partial (m, l, acc[D]) per query head; the last CTA of a
// (batch, kv head) to finish (an atomic ticket, no waiting) merges the splits
// with a log-sum-exp weighting and writes the fp16 output.  One split writes
// the output directly.
#include <cuda_fp16.h>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 4;
constexpr float kLazyRescale = 8.0f;

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// Exact small-integer to float: 2^23 + code has code in the low mantissa bits.
__device__ __forceinline__ float code_to_float(uint32_t code) {
  return __uint_as_float(0x4B000000u | code) - 8388608.0f;
}

template <int BK, int BV, int HG, bool ROPE>
struct Shape {
  static constexpr int D = kHeadDim;
  static constexpr int CPL = 32 / HG;    // channels per lane
  static constexpr int KAPPA = D / CPL;  // lanes sharing one token (channel chunks)
  static constexpr int TAU = 32 / KAPPA; // token slots per warp
  static constexpr int TPL = 32 / TAU;   // tokens per lane in a 32-token sub-tile
  static constexpr int HALF = CPL / 2;   // rope: channels per lane in each half of the head
};

// Extract `n` codes of `bits` bits starting at bit `bit0` of a token record
// held in shared memory, into codes[0..n).
template <int BITS, int N>
__device__ __forceinline__ void load_codes(const uint32_t* rec, int bit0, uint32_t (&codes)[N]) {
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  if constexpr (N * BITS <= 32 + 0) {
    // fits in one 64-bit window from the first word
    const int w = bit0 >> 5, off = bit0 & 31;
    uint64_t win = rec[w];
    if (off + N * BITS > 32) win |= (uint64_t)rec[w + 1] << 32;
    win >>= off;
#pragma unroll
    for (int i = 0; i < N; ++i) codes[i] = (uint32_t)(win >> (i * BITS)) & MASK;
  } else if constexpr (N * BITS <= 48) {
    const int w = bit0 >> 5, off = bit0 & 31;
    uint64_t win = (uint64_t)rec[w] | ((uint64_t)rec[w + 1] << 32);
    win >>= off;
#pragma unroll
    for (int i = 0; i < N; ++i) codes[i] = (uint32_t)(win >> (i * BITS)) & MASK;
  } else {
    // word aligned: bit0 % 32 == 0 and N*BITS % 32 == 0
    constexpr int NW = N * BITS / 32;
    uint32_t wds[NW];
    const int w = bit0 >> 5;
#pragma unroll
    for (int i = 0; i < NW; ++i) wds[i] = rec[w + i];
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int b = i * BITS;
      const int wi = b >> 5, o = b & 31;
      uint32_t v = wds[wi] >> o;
      if (o + BITS > 32) v |= wds[wi + 1] << (32 - o);
      codes[i] = v & MASK;
    }
  }
}

// cos/sin of theta_i * t, with theta_i / (2 pi) given as a 0.64 fixed-point
// fraction of a turn: the turn count t * F mod 1 is exact integer arithmetic.
__device__ __forceinline__ void rope_cs(unsigned long long F, uint32_t t, float& c, float& s) {
  const uint32_t flo = (uint32_t)F, fhi = (uint32_t)(F >> 32);
  const uint32_t top = __umulhi(t, flo) + t * fhi;  // bits 32..63 of t*F = turns * 2^32 (mod 2^32)
  const float x = (float)(top >> 8) * 0x1.0p-23f;   // angle / pi in [0, 2)
  sincospif(x, &s, &c);
}

template <int BK, int BV, int HG, bool ROPE>
__global__ void __launch_bounds__(kDecodeThreads) decode_split_kernel(const DecodeParams p) {
  using S = Shape<BK, BV, HG, ROPE>;
  constexpr int D = S::D, CPL = S::CPL, KAPPA = S::KAPPA, TAU = S::TAU, TPL = S::TPL;

  const int split = blockIdx.x;
  const int unit = blockIdx.y;  // b * Hkv + kvh
  const int b = unit / p.Hkv, kvh = unit - b * p.Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ float q_s[HG][D];
  __shared__ float qp_s[kConsumerWarps][HG][D];
  __shared__ float wacc[kConsumerWarps][HG][D];
  __shared__ float wml[kConsumerWarps][HG][2];
  __shared__ int abort_flag;
  __shared__ int last_cta;

  // page range of this split; the last split also reads the fp16 window
  const int64_t pg_begin = (int64_t)split * p.n_pages / p.splits;
  const int64_t pg_end = (int64_t)(split + 1) * p.n_pages / p.splits;
  const int n_pg = (int)(pg_end - pg_begin);
  const bool do_window = split == p.splits - 1 && p.n_r > 0;
  const int page_bytes = p.lay.bytes;
  const uint8_t* unit_pages = p.pages + (int64_t)unit * p.unit_page_stride;

  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    fence_mbar_init();
  }
  for (int i = tid; i < HG * D; i += kDecodeThreads) {
    const int h = i / D, c = i - h * D;
    q_s[h][c] = h2f(p.q[((int64_t)b * p.Hq + kvh * HG + h) * D + c]);
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------- producer: one bulk copy per page into the stage ring
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n_pg; ++i) {
        const int st = i % kStages, k = i / kStages;
        if (k > 0 && !mbar_wait(&empty_bar[st], (k - 1) & 1)) {
          report_error(p.err, kDevWaitTimeout);
          atomicExch(&abort_flag, 1);
          break;
        }
        if (*(volatile int*)&abort_flag) break;
        mbar_arrive_expect_tx(&full_bar[st], (uint32_t)page_bytes);
        bulk_g2s(stage_mem + (size_t)st * page_bytes, unit_pages + (pg_begin + i) * (int64_t)page_bytes,
                 (uint32_t)page_bytes, &full_bar[st]);
        ++issued;
      }
      // never leave with a copy in flight: wait (bounded) for the last copy of every stage
      for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
        mbar_wait(&full_bar[i % kStages], (i / kStages) & 1);
    }
    return;
  }

  // ---------------- consumers
  const int kap = lane % KAPPA;  // channel chunk
  const int tau = lane / KAPPA;  // token slot
  float m_run[HG], l_run[HG], zsum[HG], acc[HG][CPL];
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.0f;
    zsum[h] = 0.0f;
#pragma unroll
    for (int i = 0; i < CPL; ++i) acc[h][i] = 0.0f;
  }
  // key channels of this lane: a contiguous chunk, or (rope) half a chunk in each half of the head
  const int kc_lo = ROPE ? kap * S::HALF : kap * CPL;
  const int vc_lo = kap * CPL;
  const int sub_tiles = p.R / 32;
  const int ng = D / p.G;

  // Online-softmax update of one sub-tile; sc[j][h] are final scores (log2 units) of the
  // lane's tokens (-inf for masked ones).  Returns the weights in sc.
  auto softmax_update = [&](float (&sc)[TPL][HG]) {
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      float tmax = sc[0][h];
#pragma unroll
      for (int j = 1; j < TPL; ++j) tmax = fmaxf(tmax, sc[j][h]);
#pragma unroll
      for (int off = KAPPA; off < 32; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      if (tmax > m_run[h] + kLazyRescale || (m_run[h] == -INFINITY && tmax != -INFINITY)) {
        const float mnew = fmaxf(tmax, m_run[h]);
        const float f = m_run[h] == -INFINITY ? 0.0f : exp2f(m_run[h] - mnew);
        l_run[h] *= f;
        zsum[h] *= f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) acc[h][i] *= f;
        m_run[h] = mnew;
      }
      const bool live = m_run[h] != -INFINITY;
#pragma unroll
      for (int j = 0; j < TPL; ++j) sc[j][h] = live ? exp2f(sc[j][h] - m_run[h]) : 0.0f;
    }
  };

  int pg_i = 0;
  for (; pg_i < n_pg; ++pg_i) {
    const int st = pg_i % kStages;
    if (!mbar_wait(&full_bar[st], (pg_i / kStages) & 1)) {
      report_error(p.err, kDevWaitTimeout);
      atomicExch(&abort_flag, 1);
      break;
    }
    const uint8_t* pgm = stage_mem + (size_t)st * page_bytes;
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_kc);
    const uint32_t* km = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_km);
    const uint32_t* vcw = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_vc);
    const uint32_t* vm = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_vm);
    const uint8_t* si = pgm + p.lay.off_si;
    const uint16_t* sv = reinterpret_cast<const uint16_t*>(pgm + p.lay.off_sv);
    const int64_t page_tok0 = (pg_begin + pg_i) * (int64_t)p.R;

    for (int stt = warp; stt < sub_tiles; stt += kConsumerWarps) {
      const int g = (stt * 32) / p.G;  // key group of this sub-tile (G >= 32)
      float sc[TPL][HG];

      if constexpr (!ROPE) {
        // cooperative q'_c = q_c * s_c and Z = sum_c q_c z_c for the group
        __syncwarp();  // every lane has finished reading the previous sub-tile's q'
        float zp[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) zp[h] = 0.0f;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
          const int c = lane + 32 * j;
          const uint32_t mz = km[g * D + c];
          const float z = h2f((uint16_t)(mz & 0xFFFFu)), s = h2f((uint16_t)(mz >> 16));
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            qp_s[warp][h][c] = q_s[h][c] * s;
            zp[h] = fmaf(q_s[h][c], z, zp[h]);
          }
        }
#pragma unroll
        for (int h = 0; h < HG; ++h)
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) zp[h] += __shfl_xor_sync(0xffffffffu, zp[h], off);
        __syncwarp();
        float qp[HG][CPL];
#pragma unroll
        for (int h = 0; h < HG; ++h)
#pragma unroll
          for (int i = 0; i < CPL; ++i) qp[h][i] = qp_s[warp][h][kc_lo + i];

#pragma unroll
        for (int j = 0; j < TPL; ++j) {
          const int tt = stt * 32 + tau + TAU * j;  // token within the page
          uint32_t codes[CPL];
          load_codes<BK, CPL>(kc + tt * (D * BK / 32), kc_lo * BK, codes);
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) a = fmaf(qp[h][i], code_to_float(codes[i]), a);
            sc[j][h] = a;
          }
          // sparse entries: the dense code there is 0 (value z); add q_c (x_c - z_c)
          for (int k = 0; k < p.nsp; ++k) {
            const int c = si[tt * p.nsp + k];
            if (c >= kc_lo && c < kc_lo + CPL) {
              const float z = h2f((uint16_t)(km[g * D + c] & 0xFFFFu));
              const float x = h2f(sv[tt * p.nsp + k]);
#pragma unroll
              for (int h = 0; h < HG; ++h) sc[j][h] = fmaf(q_s[h][c], x - z, sc[j][h]);
            }
          }
        }
        // sum the channel chunks of each token, then add the group constant
#pragma unroll
        for (int j = 0; j < TPL; ++j)
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            float a = sc[j][h];
#pragma unroll
            for (int off = 1; off < KAPPA; off <<= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            sc[j][h] = (a + zp[h]) * p.qk_scale_log2;
          }
      } else {
        // pre-RoPE keys: dequantize, restore sparse entries, rotate, dot
        constexpr int HF = S::HALF;
        float zl[HF], sl[HF], zh[HF], sh[HF];
#pragma unroll
        for (int i = 0; i < HF; ++i) {
          const uint32_t a = km[g * D + kc_lo + i], c2 = km[g * D + kc_lo + D / 2 + i];
          zl[i] = h2f((uint16_t)(a & 0xFFFFu));
          sl[i] = h2f((uint16_t)(a >> 16));
          zh[i] = h2f((uint16_t)(c2 & 0xFFFFu));
          sh[i] = h2f((uint16_t)(c2 >> 16));
        }
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
          const int tt = stt * 32 + tau + TAU * j;
          const uint32_t* rec = kc + tt * (D * BK / 32);
          uint32_t cl[HF], ch[HF];
          load_codes<BK, HF>(rec, kc_lo * BK, cl);
          load_codes<BK, HF>(rec, (kc_lo + D / 2) * BK, ch);
          float kl[HF], kh[HF];
#pragma unroll
          for (int i = 0; i < HF; ++i) {
            kl[i] = fmaf(sl[i], code_to_float(cl[i]), zl[i]);
            kh[i] = fmaf(sh[i], code_to_float(ch[i]), zh[i]);
          }
          for (int k = 0; k < p.nsp; ++k) {
            const int c = si[tt * p.nsp + k];
            const float x = h2f(sv[tt * p.nsp + k]);
#pragma unroll
            for (int i = 0; i < HF; ++i) {
              if (c == kc_lo + i) kl[i] = x;
              if (c == kc_lo + D / 2 + i) kh[i] = x;
            }
          }
          const uint32_t tpos = (uint32_t)(page_tok0 + tt);
          float a[HG];
#pragma unroll
          for (int h = 0; h < HG; ++h) a[h] = 0.0f;
#pragma unroll
          for (int i = 0; i < HF; ++i) {
            float cs, sn;
            rope_cs(p.rope_turns[kc_lo + i], tpos, cs, sn);
            const float rl = kl[i] * cs - kh[i] * sn;
            const float rh = kh[i] * cs + kl[i] * sn;
#pragma unroll
            for (int h = 0; h < HG; ++h) a[h] = fmaf(q_s[h][kc_lo + i], rl, fmaf(q_s[h][kc_lo + D / 2 + i], rh, a[h]));
          }
#pragma unroll
          for (int h = 0; h < HG; ++h) sc[j][h] = a[h];
        }
#pragma unroll
        for (int j = 0; j < TPL; ++j)
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            float a = sc[j][h];
#pragma unroll
            for (int off = 1; off < KAPPA; off <<= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            sc[j][h] = a * p.qk_scale_log2;
          }
      }

      softmax_update(sc);

      // P.V over the value codes of the lane's channel chunk
      const int gv = vc_lo / p.G;
#pragma unroll
      for (int j = 0; j < TPL; ++j) {
        const int tt = stt * 32 + tau + TAU * j;
        const uint32_t mv = vm[tt * ng + gv];
        const float z = h2f((uint16_t)(mv & 0xFFFFu)), s = h2f((uint16_t)(mv >> 16));
        uint32_t codes[CPL];
        load_codes<BV, CPL>(vcw + tt * (D * BV / 32), vc_lo * BV, codes);
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float pw = sc[j][h];
          l_run[h] += pw;
          zsum[h] = fmaf(pw, z, zsum[h]);
          const float ps = pw * s;
#pragma unroll
          for (int i = 0; i < CPL; ++i) acc[h][i] = fmaf(ps, code_to_float(codes[i]), acc[h][i]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[st]);
  }

  // fold the value zero-point sums into the accumulators (quantized tokens only)
#pragma unroll
  for (int h = 0; h < HG; ++h) {
#pragma unroll
    for (int i = 0; i < CPL; ++i) acc[h][i] += zsum[h];
  }

  // ---------------- fp16 window (last split): tokens Tq .. Tq + n_r - 1
  if (do_window && !*(volatile int*)&abort_flag) {
    const int64_t tq = p.n_pages * (int64_t)p.R;
    const uint16_t* wk = p.wk + (int64_t)unit * p.win_unit_stride;
    const uint16_t* wv = p.wv + (int64_t)unit * p.win_unit_stride;
    const int wtiles = (p.n_r + 31) / 32;
    for (int stt = warp; stt < wtiles; stt += kConsumerWarps) {
      float sc[TPL][HG];
#pragma unroll
      for (int j = 0; j < TPL; ++j) {
        const int tt = stt * 32 + tau + TAU * j;
        if (tt >= p.n_r) {
#pragma unroll
          for (int h = 0; h < HG; ++h) sc[j][h] = 0.0f;
          continue;
        }
        const uint16_t* kr = wk + (int64_t)tt * D;
        float a[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) a[h] = 0.0f;
        if constexpr (!ROPE) {
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const float x = h2f(kr[kc_lo + i]);
#pragma unroll
            for (int h = 0; h < HG; ++h) a[h] = fmaf(q_s[h][kc_lo + i], x, a[h]);
          }
        } else {
          const uint32_t tpos = (uint32_t)(tq + tt);
#pragma unroll
          for (int i = 0; i < S::HALF; ++i) {
            const float xl = h2f(kr[kc_lo + i]), xh = h2f(kr[kc_lo + D / 2 + i]);
            float cs, sn;
            rope_cs(p.rope_turns[kc_lo + i], tpos, cs, sn);
            const float rl = xl * cs - xh * sn, rh = xh * cs + xl * sn;
#pragma unroll
            for (int h = 0; h < HG; ++h) a[h] = fmaf(q_s[h][kc_lo + i], rl, fmaf(q_s[h][kc_lo + D / 2 + i], rh, a[h]));
          }
        }
#pragma unroll
        for (int h = 0; h < HG; ++h) sc[j][h] = a[h];
      }
#pragma unroll
      for (int j = 0; j < TPL; ++j) {
        const int tt = stt * 32 + tau + TAU * j;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          float a = sc[j][h];
#pragma unroll
          for (int off = 1; off < KAPPA; off <<= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
          sc[j][h] = tt < p.n_r ? a * p.qk_scale_log2 : -INFINITY;
        }
      }
      softmax_update(sc);
#pragma unroll
      for (int j = 0; j < TPL; ++j) {
        const int tt = stt * 32 + tau + TAU * j;
        if (tt >= p.n_r) continue;
        const uint16_t* vr = wv + (int64_t)tt * D;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float pw = sc[j][h];
          l_run[h] += pw;
#pragma unroll
          for (int i = 0; i < CPL; ++i) acc[h][i] = fmaf(pw, h2f(vr[vc_lo + i]), acc[h][i]);
        }
      }
    }
  }

  // ---------------- reduce the token slots of the warp, then the warps of the CTA
#pragma unroll
  for (int h = 0; h < HG; ++h) {
#pragma unroll
    for (int off = KAPPA; off < 32; off <<= 1) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], off);
#pragma unroll
      for (int i = 0; i < CPL; ++i) acc[h][i] += __shfl_xor_sync(0xffffffffu, acc[h][i], off);
    }
  }
  if (tau == 0) {
#pragma unroll
    for (int h = 0; h < HG; ++h)
#pragma unroll
      for (int i = 0; i < CPL; ++i) wacc[warp][h][vc_lo + i] = acc[h][i];
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      wml[warp][h][0] = m_run[h];
      wml[warp][h][1] = l_run[h];
    }
  }
  named_barrier_sync(1, kConsumerWarps * 32);
  // this CTA's partial for (head h, channel c) = (i / D, i % D), i = tid + 128 k
  constexpr int PER = HG * D / (kConsumerWarps * 32);
  float pa[PER], pm[PER], pl[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid + k * kConsumerWarps * 32;
    const int h = i / D, c = i - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wml[w][h][0]);
    float a = 0.0f, L = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        if (wml[w][h][0] == -INFINITY) continue;
        const float f = exp2f(wml[w][h][0] - M);
        a = fmaf(f, wacc[w][h][c], a);
        L = fmaf(f, wml[w][h][1], L);
      }
    }
    pa[k] = a;
    pm[k] = M;
    pl[k] = L;
  }
  const int64_t bh0 = (int64_t)b * p.Hq + kvh * HG;
  if (p.splits == 1) {
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = tid + k * kConsumerWarps * 32;
      p.out[bh0 * D + i] = __half_as_ushort(__float2half_rn(pa[k] / pl[k]));
    }
    return;
  }
  // publish the partial; the last CTA of the unit to finish merges all splits
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid + k * kConsumerWarps * 32;
    const int h = i / D, c = i - h * D;
    const int64_t slot = (bh0 + h) * p.splits + split;
    p.part_acc[slot * D + c] = pa[k];
    if (c == 0) {
      p.part_ml[slot * 2] = pm[k];
      p.part_ml[slot * 2 + 1] = pl[k];
    }
  }
  __threadfence();
  named_barrier_sync(1, kConsumerWarps * 32);
  if (tid == 0) last_cta = atomicAdd(&p.counters[unit], 1) == p.splits - 1;
  named_barrier_sync(1, kConsumerWarps * 32);
  if (!last_cta) return;
  __threadfence();
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid + k * kConsumerWarps * 32;
    const int h = i / D, c = i - h * D;
    const float* ml = p.part_ml + (bh0 + h) * p.splits * 2;
    const float* pacc = p.part_acc + (bh0 + h) * p.splits * D + c;
    float M = -INFINITY;
    for (int sp = 0; sp < p.splits; ++sp) M = fmaxf(M, __ldcg(ml + 2 * sp));
    float a = 0.0f, L = 0.0f;
    for (int sp = 0; sp < p.splits; ++sp) {
      const float m = __ldcg(ml + 2 * sp);
      if (m == -INFINITY) continue;
      const float f = exp2f(m - M);
      L = fmaf(f, __ldcg(ml + 2 * sp + 1), L);
      a = fmaf(f, __ldcg(pacc + (int64_t)sp * D), a);
    }
    p.out[bh0 * D + i] = __half_as_ushort(__float2half_rn(a / L));
  }
  if (tid == 0) p.counters[unit] = 0;  // ready for the next call on this stream
}

template <int BK, int BV, int HG, bool ROPE>
cudaError_t launch_decode_t(const DecodeParams& p, int n_units, cudaStream_t s) {
  const size_t smem = (size_t)kStages * p.lay.bytes;
  auto kern = decode_split_kernel<BK, BV, HG, ROPE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.splits, (unsigned)n_units);
  kern<<<grid, kDecodeThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

#define KVQ_DECODE_CASES(X)                                                                                 \
  X(2, 2, 1, false) X(2, 2, 2, false) X(2, 2, 4, false) X(4, 2, 1, false) X(4, 2, 2, false) X(4, 2, 4, false) \
  X(3, 3, 1, false) X(3, 3, 2, false) X(3, 3, 4, false) X(4, 4, 1, false) X(4, 4, 2, false) X(4, 4, 4, false) \
  X(2, 2, 1, true) X(2, 2, 4, true) X(3, 3, 1, true) X(3, 3, 4, true) X(4, 2, 1, true) X(4, 2, 4, true)       \
  X(4, 4, 1, true) X(4, 4, 4, true)

bool decode_supported(int bk, int bv, int hg, bool rope) {
#define KVQ_SUP(BKV, BVV, HGV, RP) \
  if (bk == BKV && bv == BVV && hg == HGV && rope == RP) return true;
  KVQ_DECODE_CASES(KVQ_SUP)
#undef KVQ_SUP
  return false;
}

cudaError_t launch_decode(const DecodeParams& p, int bk, int bv, int hg, bool rope, int n_units, cudaStream_t s,
                          bool* supported) {
  *supported = true;
#define KVQ_DEC(BKV, BVV, HGV, RP) \
  if (bk == BKV && bv == BVV && hg == HGV && rope == RP) return launch_decode_t<BKV, BVV, HGV, RP>(p, n_units, s);
  KVQ_DECODE_CASES(KVQ_DEC)
#undef KVQ_DEC
  *supported = false;
  return cudaErrorInvalidValue;
}

}  // namespace kvq
