// Decode attention over the packed cache: one persistent, load-balanced launch.
//
// Decode reads the whole cache for every generated token ("KV cache has a
// geometry problem, not a bit problem", section "Why the KV cache is a
// problem"), so the kernel is built around streaming pages at full bandwidth:
//
//  * Work list.  Every (batch, kv head) unit contributes n_pages page items
//    and, when the fp16 window is not empty, one window item.  The items of
//    all units are laid end to end and the grid (sized to the resident CTA
//    count) takes equal contiguous slices of that list, so every SM streams
//    the same number of pages whatever the batch/head/length mix, and a CTA
//    crosses from one unit into the next without a new launch.
//  * Streaming.  A producer warp issues one bulk (TMA) copy per page into a
//    ring of shared-memory stages guarded by mbarriers; four consumer warps
//    take one 32-token sub-tile of each page and dequantize in registers.
//  * Merge.  Each CTA writes one unnormalised partial (m, l, acc[D]) per
//    query head for every unit it touched; the CTA that completes a unit's
//    item count (an atomic ticket, no waiting) merges the unit's partials
//    with log-sum-exp weights and writes the fp16 output.  A unit covered by
//    one CTA is written directly.
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
// every weight below 2^8 and skips most rescales.
#include <cuda_fp16.h>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kDecodeThreads = kConsumerThreads;  // every warp computes; copies are issued by whichever warp frees a stage
constexpr int kStages = 4;
constexpr float kLazyRescale = 8.0f;

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// Exact small-integer to float: 2^23 + code has code in the low mantissa bits.
__device__ __forceinline__ float code_to_float(uint32_t code) {
  return __uint_as_float(0x4B000000u | code) - 8388608.0f;
}

// Power of two that the fast paths keep their products scaled by (see MaskCodes).
constexpr int kCodeExp = 64;

// Codes of one 32-bit word of a B-bit bitstream as fp32 subnormals, one logic
// op per code: masking the code at position p in place gives the float
// code * 2^(B*p) * 2^-149 exactly for the first NDIRECT positions (they fit in
// the 23 mantissa bits); the rest are read the same way from the word shifted
// right by NDIRECT*B.  The factor each code multiplies carries
// scale_in(p) = 2^(149 - kCodeExp - B*p), so every product is
// code * factor * 2^-kCodeExp, a normal number, with no offset to remove;
// scale_out(p) = 2^(kCodeExp - B*p) undoes the position scale of an
// accumulator that summed subnormal codes against unscaled factors.
template <int BITS>
struct MaskCodes {
  static constexpr int PER_WORD = 32 / BITS;
  static constexpr int NDIRECT = BITS == 2 ? 11 : 5;  // (2^B - 1) * 2^(B*(n-1)) < 2^23
  static constexpr uint32_t MASK = (1u << BITS) - 1u;
  __device__ static constexpr int pos(int i) { return i < NDIRECT ? i : i - NDIRECT; }
  __device__ static float scale_in(int i) {
    return __uint_as_float((uint32_t)(127 + 149 - kCodeExp - BITS * pos(i)) << 23);
  }
  __device__ static float scale_out(int i) { return __uint_as_float((uint32_t)(127 + kCodeExp - BITS * pos(i)) << 23); }
  __device__ __forceinline__ static void to_float(uint32_t w, float (&f)[PER_WORD]) {
    const uint32_t ws = w >> (NDIRECT * BITS);
#pragma unroll
    for (int i = 0; i < PER_WORD; ++i) {
      const uint32_t src = i < NDIRECT ? w : ws;
      f[i] = __uint_as_float(src & (MASK << (BITS * pos(i))));
    }
  }
};

template <int BK, int BV, int HG, bool ROPE>
struct Shape {
  static constexpr int D = kHeadDim;
  static constexpr int CPL = 32 / HG;    // channels per lane
  static constexpr int KAPPA = D / CPL;  // lanes sharing one token (channel chunks)
  static constexpr int TAU = 32 / KAPPA; // token slots per warp
  static constexpr int TPL = 32 / TAU;   // tokens per lane in a 32-token sub-tile
  static constexpr int HALF = CPL / 2;   // rope: channels per lane in each half of the head
  // one query head per kv head with 2- or 4-bit codes: mask extraction and packed fp32x2 math
  static constexpr bool FAST_K = HG == 1 && !ROPE && (BK == 2 || BK == 4);
  static constexpr bool FAST_V = HG == 1 && (BV == 2 || BV == 4);
  static constexpr int KBITS_FAST = (BK == 2 || BK == 4) ? BK : 2;
  // resident CTAs per SM the register budget is sized for (128 threads each)
  static constexpr int MIN_BLOCKS = ROPE ? (HG == 1 ? 3 : 2) : (HG == 4 ? 2 : 4);
};

// Extract N codes of BITS bits starting at bit `bit0` of a token record held
// in shared memory, into codes[0..N).
template <int BITS, int N>
__device__ __forceinline__ void load_codes(const uint32_t* rec, int bit0, uint32_t (&codes)[N]) {
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  if constexpr (N * BITS <= 32) {
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

// N consecutive fp16 values (N a multiple of 4, src aligned to 2N bytes up to 16) as floats,
// in 8- or 16-byte loads.
template <int N>
__device__ __forceinline__ void load_halves(const uint16_t* src, float (&dst)[N]) {
  static_assert(N % 4 == 0, "rows are read in groups of four");
  if constexpr (N % 8 == 0) {
#pragma unroll
    for (int v = 0; v < N / 8; ++v) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + v);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ws[i]));
        dst[8 * v + 2 * i] = f.x;
        dst[8 * v + 2 * i + 1] = f.y;
      }
    }
  } else {
#pragma unroll
    for (int v = 0; v < N / 4; ++v) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(src) + v);
      const uint32_t ws[2] = {w.x, w.y};
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ws[i]));
        dst[4 * v + 2 * i] = f.x;
        dst[4 * v + 2 * i + 1] = f.y;
      }
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

// The CTA whose slice of the work list holds item x (slices [k*total/grid, (k+1)*total/grid)).
__device__ __forceinline__ int cta_of(int64_t x, int64_t total, int grid) {
  return (int)(((x + 1) * (int64_t)grid - 1) / total);
}

// Running softmax state of one lane for the current unit.
template <int HG, int CPL>
struct LaneState {
  float m[HG], l[HG], zsum[HG], acc[HG][CPL];
  bool folded;
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.0f;
      zsum[h] = 0.0f;
#pragma unroll
      for (int i = 0; i < CPL; ++i) acc[h][i] = 0.0f;
    }
    folded = false;
  }
};

template <int BK, int BV, int HG, bool ROPE>
__global__ void __launch_bounds__(kDecodeThreads, (Shape<BK, BV, HG, ROPE>::MIN_BLOCKS))
    decode_kernel(const DecodeParams p) {
  using S = Shape<BK, BV, HG, ROPE>;
  constexpr int D = S::D, CPL = S::CPL, KAPPA = S::KAPPA, TAU = S::TAU, TPL = S::TPL;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x, grid = gridDim.x;
  const int64_t wpu = p.work_per_unit;
  const int64_t total = p.n_units * wpu;
  const int64_t w_begin = (int64_t)cta * total / grid;
  const int64_t w_end = (int64_t)(cta + 1) * total / grid;
  const int page_bytes = p.lay.bytes;

  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ int stage_cnt[kStages];  // warps that finished each stage (mod kConsumerWarps: the last one refills)
  __shared__ __align__(16) uint16_t q_stage[2][HG * D];  // fp16 query rows of the next units
  __shared__ __align__(8) uint64_t q_full[2];
  __shared__ float q_s[HG][D];
  __shared__ __align__(16) float qp_s[kConsumerWarps][HG][D];
  __shared__ float wacc[kConsumerWarps][HG][D];
  __shared__ float wml[kConsumerWarps][HG][2];
  __shared__ int abort_flag;
  __shared__ int last_cta;
  __shared__ int stage_issued[kStages];  // copies issued into each stage / query buffer so far
  __shared__ int qbuf_issued[2];

  // Page items of this slice, numbered k = 0, 1, ... in list order.  Before item x the list
  // holds unit(x) * n_pages + min(loc(x), n_pages) page items, so page k of the slice is global
  // page P_begin + k: unit (P_begin + k) / n_pages, page (P_begin + k) % n_pages of that unit.
  auto pages_before = [&](int64_t x) -> int64_t {
    const int64_t u = x / wpu, l = x - u * wpu;
    return u * p.n_pages + (l < p.n_pages ? l : p.n_pages);
  };
  const int64_t P_begin = pages_before(w_begin);
  const int n_pg = (int)(pages_before(w_end) - P_begin);
  const int64_t unit_first = w_begin / wpu;
  const int n_cta_units = w_end > w_begin ? (int)((w_end - 1) / wpu - unit_first + 1) : 0;
  const uint32_t q_bytes = (uint32_t)(HG * D * 2);

  // page k of the slice into stage k % kStages (one thread)
  auto issue_page = [&](int k) {
    // 32-bit division: a cache never holds 2^32 pages
    const uint32_t P = (uint32_t)(P_begin + k), np = (uint32_t)p.n_pages;
    const uint32_t u = P / np, loc = P - u * np;
    const int st = k % kStages;
    mbar_arrive_expect_tx(&full_bar[st], (uint32_t)page_bytes);
    bulk_g2s(stage_mem + (size_t)st * page_bytes, p.pages + (int64_t)u * p.unit_page_stride + (int64_t)loc * page_bytes,
             (uint32_t)page_bytes, &full_bar[st]);
    stage_issued[st] = k / kStages + 1;
  };
  // query rows q[b][kvh*HG .. kvh*HG+HG-1][:] (contiguous) of the slice's j-th unit into buffer j % 2 (one thread)
  auto issue_q = [&](int j) {
    const int64_t u = unit_first + j;
    const int64_t b = u / p.Hkv, kvh = u - b * p.Hkv;
    mbar_arrive_expect_tx(&q_full[j & 1], q_bytes);
    bulk_g2s(q_stage[j & 1], p.q + (b * p.Hq + kvh * HG) * D, q_bytes, &q_full[j & 1]);
    qbuf_issued[j & 1] = (j >> 1) + 1;
  };

  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
      stage_cnt[i] = 0;
      stage_issued[i] = 0;
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      qbuf_issued[i] = 0;
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int k = 0; k < n_pg && k < kStages; ++k) issue_page(k);
    for (int j = 0; j < n_cta_units && j < 2; ++j) issue_q(j);
  }

  // ---------------- consumers
  const int kap = lane % KAPPA;  // channel chunk
  const int tau = lane / KAPPA;  // token slot
  // key channels of this lane: a contiguous chunk, or (rope) half a chunk in each half of the head
  const int kc_lo = ROPE ? kap * S::HALF : kap * CPL;
  const int vc_lo = kap * CPL;
  const int sub_tiles = p.R / 32;
  const int ng = D >> p.log2G;
  const int gv = vc_lo >> p.log2G;
  // fast key path: 2^(-B*p) of the channels this lane prepares for the group products
  float k_unscale[D / 32];
#pragma unroll
  for (int j = 0; j < D / 32; ++j)
    k_unscale[j] = S::FAST_K ? MaskCodes<S::KBITS_FAST>::scale_in((lane + 32 * j) % MaskCodes<S::KBITS_FAST>::PER_WORD)
                             : 1.0f;

  LaneState<HG, CPL> st;
  st.reset();

  // Online-softmax update of one sub-tile: sc[j][h] are final scores (log2 units) of the
  // lane's tokens (-inf for masked ones); returns the weights in sc.
  auto softmax_update = [&](float (&sc)[TPL][HG]) {
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      float tmax = sc[0][h];
#pragma unroll
      for (int j = 1; j < TPL; ++j) tmax = fmaxf(tmax, sc[j][h]);
      // the running maximum only moves when a score passes it by the lazy threshold: a vote
      // settles the common case without a reduction
      const bool over = tmax > st.m[h] + kLazyRescale || (st.m[h] == -INFINITY && tmax != -INFINITY);
      if (__any_sync(0xffffffffu, over)) {
#pragma unroll
        for (int off = KAPPA; off < 32; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
        const float mnew = fmaxf(tmax, st.m[h]);
        const float f = st.m[h] == -INFINITY ? 0.0f : exp2f(st.m[h] - mnew);
        st.l[h] *= f;
        st.zsum[h] *= f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) st.acc[h][i] *= f;
        st.m[h] = mnew;
      }
      const bool live = st.m[h] != -INFINITY;
#pragma unroll
      for (int j = 0; j < TPL; ++j) sc[j][h] = live ? exp2f(sc[j][h] - st.m[h]) : 0.0f;
    }
  };

  // undo the per-position code scale of the fast value path and add the value
  // zero-point sums (quantized tokens only); done once per unit, before any fp16 token
  auto fold = [&]() {
    if (st.folded) return;
#pragma unroll
    for (int h = 0; h < HG; ++h)
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        if constexpr (S::FAST_V) st.acc[h][i] *= MaskCodes<S::FAST_V ? BV : 2>::scale_out(i % MaskCodes<S::FAST_V ? BV : 2>::PER_WORD);
        st.acc[h][i] += st.zsum[h];
      }
    st.folded = true;
  };

  int q_seq = 0;
  auto load_q = [&]() {
    const int qs = q_seq & 1;
    if (!mbar_wait(&q_full[qs], (q_seq >> 1) & 1)) {
      report_error(p.err, kDevWaitTimeout);
      atomicExch(&abort_flag, 1);
    }
    for (int i = tid; i < HG * D; i += kConsumerThreads) {
      const int h = i / D, c = i - h * D;
      q_s[h][c] = h2f(q_stage[qs][i]);
    }
    named_barrier_sync(1, kConsumerThreads);
    // buffer qs is free again: fetch the unit after next into it
    if (tid == 0 && q_seq + 2 < n_cta_units && !*(volatile int*)&abort_flag) issue_q(q_seq + 2);
    ++q_seq;
  };

  // Partial of this CTA for `unit` (covering `done` of its items); merges when it completes the unit.
  auto epilogue = [&](int64_t unit, int done) {
    fold();
#pragma unroll
    for (int h = 0; h < HG; ++h) {
#pragma unroll
      for (int off = KAPPA; off < 32; off <<= 1) {
        st.l[h] += __shfl_xor_sync(0xffffffffu, st.l[h], off);
#pragma unroll
        for (int i = 0; i < CPL; ++i) st.acc[h][i] += __shfl_xor_sync(0xffffffffu, st.acc[h][i], off);
      }
    }
    if (tau == 0) {
#pragma unroll
      for (int h = 0; h < HG; ++h)
#pragma unroll
        for (int i = 0; i < CPL; ++i) wacc[warp][h][vc_lo + i] = st.acc[h][i];
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        wml[warp][h][0] = st.m[h];
        wml[warp][h][1] = st.l[h];
      }
    }
    named_barrier_sync(1, kConsumerThreads);
    constexpr int PER = HG * D / kConsumerThreads;
    float pa[PER], pm[PER], pl[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = tid + k * kConsumerThreads;
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
    const int64_t b = unit / p.Hkv, kvh = unit - b * p.Hkv;
    const int64_t bh0 = b * p.Hq + kvh * HG;
    const int k_first = cta_of(unit * wpu, total, grid);
    const int k_last = cta_of(unit * wpu + wpu - 1, total, grid);
    if (k_first == k_last) {
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int i = tid + k * kConsumerThreads;
        p.out[bh0 * D + i] = __half_as_ushort(__float2half_rn(pa[k] / pl[k]));
      }
    } else {
      const int slot = cta - k_first;
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int i = tid + k * kConsumerThreads;
        const int h = i / D, c = i - h * D;
        const int64_t so = (bh0 + h) * p.max_slots + slot;
        p.part_acc[so * D + c] = pa[k];
        if (c == 0) {
          p.part_ml[so * 2] = pm[k];
          p.part_ml[so * 2 + 1] = pl[k];
        }
      }
      __threadfence();
      named_barrier_sync(1, kConsumerThreads);
      if (tid == 0) last_cta = atomicAdd(&p.counters[unit], done) + done == wpu;
      named_barrier_sync(1, kConsumerThreads);
      if (last_cta) {
        __threadfence();
        const int nslots = k_last - k_first + 1;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
          const int i = tid + k * kConsumerThreads;
          const int h = i / D, c = i - h * D;
          const float* ml = p.part_ml + (bh0 + h) * p.max_slots * 2;
          const float* pacc = p.part_acc + (bh0 + h) * p.max_slots * D + c;
          float M = -INFINITY;
#pragma unroll 4
          for (int sp = 0; sp < nslots; ++sp) M = fmaxf(M, __ldcg(ml + 2 * sp));
          float a = 0.0f, L = 0.0f;
#pragma unroll 4
          for (int sp = 0; sp < nslots; ++sp) {
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
    }
    named_barrier_sync(1, kConsumerThreads);  // shared scratch is free again
  };

  int64_t cur = -1;
  int done = 0;
  int pg_seq = 0;
  int64_t unit = w_begin / wpu;
  int loc = (int)(w_begin - unit * wpu);
  for (int64_t x = w_begin; x < w_end; ++x, ++loc) {
    if (loc == wpu) {
      loc = 0;
      ++unit;
    }
    if (unit != cur) {
      if (cur >= 0) epilogue(cur, done);
      cur = unit;
      done = 0;
      st.reset();
      load_q();
    }
    ++done;
    if (*(volatile int*)&abort_flag) continue;

    if (loc < p.n_pages) {
      // ---------------- a page of quantized tokens
      const int stg = pg_seq % kStages;
      if (!mbar_wait(&full_bar[stg], (pg_seq / kStages) & 1)) {
        report_error(p.err, kDevWaitTimeout);
        atomicExch(&abort_flag, 1);
        continue;
      }
      const uint8_t* pgm = stage_mem + (size_t)stg * page_bytes;
      const uint32_t* kc = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_kc);
      const uint32_t* km = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_km);
      const uint32_t* vcw = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_vc);
      const uint32_t* vm = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_vm);
      const uint8_t* si = pgm + p.lay.off_si;
      const uint16_t* sv = reinterpret_cast<const uint16_t*>(pgm + p.lay.off_sv);
      const int64_t page_tok0 = loc * (int64_t)p.R;

      for (int stt = warp; stt < sub_tiles; stt += kConsumerWarps) {
        const int g = (stt * 32) >> p.log2G;  // key group of this sub-tile (G >= 32)
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
            const float z = h2f((uint16_t)(mz & 0xFFFFu));
            const float s = h2f((uint16_t)(mz >> 16)) * k_unscale[j];
#pragma unroll
            for (int h = 0; h < HG; ++h) {
              qp_s[warp][h][c] = q_s[h][c] * s;
              zp[h] = fmaf(q_s[h][c], z, zp[h]);
            }
          }
          __syncwarp();
          float qp[HG][CPL];
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            const float4* src = reinterpret_cast<const float4*>(&qp_s[warp][h][kc_lo]);
#pragma unroll
            for (int i = 0; i < CPL / 4; ++i) {
              const float4 v = src[i];
              qp[h][4 * i] = v.x;
              qp[h][4 * i + 1] = v.y;
              qp[h][4 * i + 2] = v.z;
              qp[h][4 * i + 3] = v.w;
            }
          }

#pragma unroll
          for (int j = 0; j < TPL; ++j) {
            const int tt = stt * 32 + tau + TAU * j;  // token within the page
            if constexpr (S::FAST_K) {
              using MC = MaskCodes<S::KBITS_FAST>;
              constexpr int NW = CPL * BK / 32;
              const uint32_t* rec = kc + tt * (D * BK / 32) + kap * NW;
              // four independent partial sums keep the packed FMA chains short
              float2 a2[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                              make_float2(0.0f, 0.0f)};
#pragma unroll
              for (int wi = 0; wi < NW; ++wi) {
                float f[MC::PER_WORD];
                MC::to_float(rec[wi], f);
#pragma unroll
                for (int m = 0; m < MC::PER_WORD / 2; ++m) {
                  const int i = wi * MC::PER_WORD + 2 * m;
                  a2[m & 3] = __ffma2_rn(make_float2(f[2 * m], f[2 * m + 1]), make_float2(qp[0][i], qp[0][i + 1]),
                                         a2[m & 3]);
                }
              }
              const float2 s01 = __fadd2_rn(a2[0], a2[1]), s23 = __fadd2_rn(a2[2], a2[3]);
              const float2 s03 = __fadd2_rn(s01, s23);
              sc[j][0] = (s03.x + s03.y) * __uint_as_float((uint32_t)(127 + kCodeExp) << 23);
            } else {
              uint32_t codes[CPL];
              load_codes<BK, CPL>(kc + tt * (D * BK / 32), kc_lo * BK, codes);
#pragma unroll
              for (int h = 0; h < HG; ++h) {
                float a = 0.0f;
#pragma unroll
                for (int i = 0; i < CPL; ++i) a = fmaf(qp[h][i], code_to_float(codes[i]), a);
                sc[j][h] = a;
              }
            }
          }
          if (p.nsp > 0) {
            // sparse entries: the dense code there is 0 (value z); add q_c (x_c - z_c)
#pragma unroll
            for (int j = 0; j < TPL; ++j) {
              const int tt = stt * 32 + tau + TAU * j;
              for (int k = 0; k < p.nsp; ++k) {
                const int c = si[tt * p.nsp + k];
                if (c >= kc_lo && c < kc_lo + CPL) {
                  const float z = h2f((uint16_t)(km[g * D + c] & 0xFFFFu));
                  const float xv = h2f(sv[tt * p.nsp + k]);
#pragma unroll
                  for (int h = 0; h < HG; ++h) sc[j][h] = fmaf(q_s[h][c], xv - z, sc[j][h]);
                }
              }
            }
          }
          // the group constant Z (reduced here, off the path of the code products)
#pragma unroll
          for (int h = 0; h < HG; ++h)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) zp[h] += __shfl_xor_sync(0xffffffffu, zp[h], off);
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
              const float xv = h2f(sv[tt * p.nsp + k]);
#pragma unroll
              for (int i = 0; i < HF; ++i) {
                if (c == kc_lo + i) kl[i] = xv;
                if (c == kc_lo + D / 2 + i) kh[i] = xv;
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
              for (int h = 0; h < HG; ++h)
                a[h] = fmaf(q_s[h][kc_lo + i], rl, fmaf(q_s[h][kc_lo + D / 2 + i], rh, a[h]));
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
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
          const int tt = stt * 32 + tau + TAU * j;
          const uint32_t mv = vm[tt * ng + gv];
          const float z = h2f((uint16_t)(mv & 0xFFFFu)), s = h2f((uint16_t)(mv >> 16));
          if constexpr (S::FAST_V) {
            using MC = MaskCodes<S::FAST_V ? BV : 2>;
            constexpr int NW = CPL * BV / 32;
            const uint32_t* rec = vcw + tt * (D * BV / 32) + kap * NW;
            const float pw = sc[j][0];
            st.l[0] += pw;
            st.zsum[0] = fmaf(pw, z, st.zsum[0]);
            // subnormal codes against p*s*2^(149-kCodeExp): acc[i] gathers code*p*s*2^(B*pos-kCodeExp)
            const float ps = pw * (s * __uint_as_float((uint32_t)(127 + 149 - kCodeExp) << 23));
            const float2 ps2 = make_float2(ps, ps);
#pragma unroll
            for (int wi = 0; wi < NW; ++wi) {
              float f[MC::PER_WORD];
              MC::to_float(rec[wi], f);
#pragma unroll
              for (int m = 0; m < MC::PER_WORD / 2; ++m) {
                const int i = wi * MC::PER_WORD + 2 * m;
                const float2 r = __ffma2_rn(make_float2(f[2 * m], f[2 * m + 1]), ps2,
                                            make_float2(st.acc[0][i], st.acc[0][i + 1]));
                st.acc[0][i] = r.x;
                st.acc[0][i + 1] = r.y;
              }
            }
          } else {
            uint32_t codes[CPL];
            load_codes<BV, CPL>(vcw + tt * (D * BV / 32), vc_lo * BV, codes);
#pragma unroll
            for (int h = 0; h < HG; ++h) {
              const float pw = sc[j][h];
              st.l[h] += pw;
              st.zsum[h] = fmaf(pw, z, st.zsum[h]);
              const float ps = pw * s;
#pragma unroll
              for (int i = 0; i < CPL; ++i) st.acc[h][i] = fmaf(ps, code_to_float(codes[i]), st.acc[h][i]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        // release the stage; the last warp to release it refills it with page pg_seq + kStages
        mbar_arrive(&empty_bar[stg]);
        if (atomicAdd(&stage_cnt[stg], 1) % kConsumerWarps == kConsumerWarps - 1 && pg_seq + kStages < n_pg &&
            !*(volatile int*)&abort_flag) {
          if (mbar_wait(&empty_bar[stg], (pg_seq / kStages) & 1)) {
            issue_page(pg_seq + kStages);
          } else {
            report_error(p.err, kDevWaitTimeout);
            atomicExch(&abort_flag, 1);
          }
        }
      }
      ++pg_seq;
    } else {
      // ---------------- the fp16 window: tokens Tq .. Tq + n_r - 1, read directly
      fold();
      const int64_t tq = p.n_pages * (int64_t)p.R;
      const uint16_t* wk = p.wk + unit * p.win_unit_stride;
      const uint16_t* wv = p.wv + unit * p.win_unit_stride;
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
            float xk[CPL];
            load_halves<CPL>(kr + kc_lo, xk);
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
#pragma unroll
              for (int h = 0; h < HG; ++h) a[h] = fmaf(q_s[h][kc_lo + i], xk[i], a[h]);
            }
          } else {
            const uint32_t tpos = (uint32_t)(tq + tt);
            float xlo[S::HALF], xhi[S::HALF];
            load_halves<S::HALF>(kr + kc_lo, xlo);
            load_halves<S::HALF>(kr + kc_lo + D / 2, xhi);
#pragma unroll
            for (int i = 0; i < S::HALF; ++i) {
              const float xl = xlo[i], xh = xhi[i];
              float cs, sn;
              rope_cs(p.rope_turns[kc_lo + i], tpos, cs, sn);
              const float rl = xl * cs - xh * sn, rh = xh * cs + xl * sn;
#pragma unroll
              for (int h = 0; h < HG; ++h)
                a[h] = fmaf(q_s[h][kc_lo + i], rl, fmaf(q_s[h][kc_lo + D / 2 + i], rh, a[h]));
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
          float xv[CPL];
          load_halves<CPL>(wv + (int64_t)tt * D + vc_lo, xv);
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            const float pw = sc[j][h];
            st.l[h] += pw;
#pragma unroll
            for (int i = 0; i < CPL; ++i) st.acc[h][i] = fmaf(pw, xv[i], st.acc[h][i]);
          }
        }
      }
    }
  }
  if (cur >= 0) epilogue(cur, done);
  // never leave with a copy in flight (only possible after an abort): wait, bounded, for the
  // last copy issued into every stage and query buffer
  __syncthreads();
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i)
      if (stage_issued[i] > 0) mbar_wait(&full_bar[i], (stage_issued[i] - 1) & 1);
    for (int i = 0; i < 2; ++i)
      if (qbuf_issued[i] > 0) mbar_wait(&q_full[i], (qbuf_issued[i] - 1) & 1);
  }
}

template <int BK, int BV, int HG, bool ROPE>
cudaError_t launch_decode_t(const DecodeParams& p, int grid, cudaStream_t s) {
  const size_t smem = (size_t)kStages * p.lay.bytes;
  auto kern = decode_kernel<BK, BV, HG, ROPE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kDecodeThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int BK, int BV, int HG, bool ROPE>
int resident_t(int page_bytes) {
  const size_t smem = (size_t)kStages * page_bytes;
  auto kern = decode_kernel<BK, BV, HG, ROPE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDecodeThreads, smem) != cudaSuccess) return 0;
  return n;
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

int decode_resident_ctas_per_sm(int bk, int bv, int hg, bool rope, int page_bytes) {
#define KVQ_RES(BKV, BVV, HGV, RP) \
  if (bk == BKV && bv == BVV && hg == HGV && rope == RP) return resident_t<BKV, BVV, HGV, RP>(page_bytes);
  KVQ_DECODE_CASES(KVQ_RES)
#undef KVQ_RES
  return 0;
}

cudaError_t launch_decode(const DecodeParams& p, int bk, int bv, int hg, bool rope, int grid, cudaStream_t s,
                          bool* supported) {
  *supported = true;
#define KVQ_DEC(BKV, BVV, HGV, RP) \
  if (bk == BKV && bv == BVV && hg == HGV && rope == RP) return launch_decode_t<BKV, BVV, HGV, RP>(p, grid, s);
  KVQ_DECODE_CASES(KVQ_DEC)
#undef KVQ_DEC
  *supported = false;
  return cudaErrorInvalidValue;
}

}  // namespace kvq
