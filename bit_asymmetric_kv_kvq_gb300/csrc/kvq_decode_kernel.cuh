// The CUDA-core decode kernel template and its launch helpers, shared by kvq_decode.cu (uniform
// codes) and kvq_decode_lut.cu (codebook codes), which instantiate it in separate translation
// units so that the library builds in parallel.
//
// Decode attention over the packed cache: one persistent, load-balanced launch.
//
// Decode reads the whole cache for every generated token ("KV cache has a
// geometry problem, not a bit problem", section "Why the KV cache is a
// problem"), so the kernel is built around streaming pages at full bandwidth:
//
//  * Work list.  Every (batch, kv head) unit contributes its fp16 items (sink
//    and window rows, when there are any), then n_pages page items.  The items of
//    all units are laid end to end and the grid (sized to the resident CTA
//    count) takes equal contiguous slices of that list, so every SM streams
//    the same number of pages whatever the batch/head/length mix, and a CTA
//    crosses from one unit into the next without a new launch.
//  * Streaming.  Pages arrive by one bulk (TMA) copy each into a ring of
//    shared-memory stages guarded by mbarriers; the warps of a CTA take the
//    pages' 32-token sub-tiles from a shared counter and dequantize in
//    registers, and the last warp to finish with a stage issues the copy that
//    refills it (no warp is set aside to issue copies).
//  * Merge.  Each warp writes one unnormalised partial (m, l, acc[D]) per
//    query head for every unit it touched.  A small kernel launched right
//    after (one CTA per unit) combines a unit's partials with log-sum-exp
//    weights and writes the fp16 output; merging inside the decode launch put
//    chains of L2 round trips at the end of every CTA's slice.
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
#pragma once

#include <cuda_fp16.h>

#include "kvq_internal.h"
#include "kvq_merge.cuh"
#include "kvq_ptx.cuh"

namespace kvq {

namespace {

constexpr int kMaxStages = 16;  // shared-memory page stages per CTA (a power of two, sized per launch)
constexpr unsigned kFull = 0xffffffffu;
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
// accumulator that summed subnormal codes against unscaled factors, and
// scale_back(p) = 1 / scale_out(p) puts real-valued sums into those units.
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
  __device__ static float scale_back(int i) { return __uint_as_float((uint32_t)(127 - kCodeExp + BITS * pos(i)) << 23); }
  __device__ __forceinline__ static void to_float(uint32_t w, float (&f)[PER_WORD]) {
    const uint32_t ws = w >> (NDIRECT * BITS);
#pragma unroll
    for (int i = 0; i < PER_WORD; ++i) {
      const uint32_t src = i < NDIRECT ? w : ws;
      f[i] = __uint_as_float(src & (MASK << (BITS * pos(i))));
    }
  }
};

template <int BK, int BV, int HG, bool ROPE, bool LUT = false>
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
  // keys rotated at decode with four query heads per kv head: the page sub-tiles on packed fp32
  // pairs with masked codes (rope_subtile in decode_kernel)
  static constexpr bool FAST_ROPE = ROPE && HG == 4 && !LUT;
  // warps of the one CTA per SM: as many as the register budget of the path allows (keys
  // rotated at decode need about 255 registers: at 168, one head per kv head spilled 1.4 KB)
  // (rope_subtile keeps each lane's value accumulators in shared memory between sub-tiles, which
  // brings it to 128 registers)
  static constexpr int WARPS = FAST_ROPE ? 16 : ROPE ? 8 : (HG == 4 ? 8 : 16);
  // dynamic shared memory beside the page stages: rope_subtile's accumulators, 4 KB per warp
  static constexpr int ACC_SMEM = FAST_ROPE ? WARPS * 32 * HG * CPL * 4 : 0;
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

// Running softmax state of one lane for the current unit.
template <int HG, int CPL>
struct LaneState {
  float m[HG], l[HG], zsum[HG], acc[HG][CPL];
  float lp;  // rope_subtile: this lane's share of l for head (lane % KAPPA) % 4, merged in the epilogue
  __device__ __forceinline__ void reset() {
    lp = 0.0f;
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.0f;
      zsum[h] = 0.0f;
#pragma unroll
      for (int i = 0; i < CPL; ++i) acc[h][i] = 0.0f;
    }
  }
};

// One CTA per SM.  The CTA streams a contiguous slice of the work list through a ring of
// shared-memory page stages; its warps take the slice's 32-token sub-tiles one at a time from a
// shared counter, so a warp that the scheduler serves less often simply takes fewer of them.
// Every warp keeps its own online-softmax state per unit and, when it leaves a unit, writes one
// partial (m, l, acc) into the next free slot of that unit; merge_kernel combines them after the
// launch.  There is no CTA-wide barrier after the start.
//
// LUT: codes index caller-supplied codebooks (non-uniform levels in step units) instead of
// standing for themselves; the mask-based fast paths, which rely on linear codes, are off.
template <int BK, int BV, int HG, bool ROPE, bool LUT>
__global__ void __launch_bounds__(Shape<BK, BV, HG, ROPE, LUT>::WARPS * 32, 1) decode_kernel(const DecodeParams p) {
  using S = Shape<BK, BV, HG, ROPE, LUT>;
  constexpr int D = S::D, CPL = S::CPL, KAPPA = S::KAPPA, TAU = S::TAU, TPL = S::TPL, W = S::WARPS;
  // the mask-based fast paths need codes that stand for themselves
  constexpr bool FAST_K = S::FAST_K && !LUT, FAST_V = S::FAST_V && !LUT;
  constexpr bool FAST_ROPE = S::FAST_ROPE && !LUT;
  // rope_subtile's value units: the accumulator of channel i of a lane's chunk holds
  // value * 2^(BV*(i%4) - kCodeExp) (codes masked in place at bit BV*(i%4) of a four-code run)
  auto rope_v_scale_out = [](int i) { return __uint_as_float((uint32_t)(127 + kCodeExp - BV * (i & 3)) << 23); };
  auto rope_v_scale_back = [](int i) { return __uint_as_float((uint32_t)(127 - kCodeExp + BV * (i & 3)) << 23); };

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x, grid = gridDim.x;
  const int64_t wpu = p.work_per_unit;
  const int64_t total = p.n_units * wpu;
  const int64_t w_begin = (int64_t)cta * total / grid;
  const int64_t w_end = (int64_t)(cta + 1) * total / grid;
  const int page_bytes = p.lay.bytes;
  const int log2S = p.log2_stages, n_stages = 1 << log2S;
  const int SPP = p.R / 32;  // sub-tiles per item (1..4)
  const int n_sub = (int)(w_end - w_begin) * SPP;

  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ int stage_cnt[kMaxStages];     // sub-tiles released per stage (mod SPP: the last refills)
  __shared__ int stage_issued[kMaxStages];  // copies issued into each stage so far
  __shared__ int stage_page[kMaxStages];    // page of the slice a stage holds or is being filled with
  __shared__ __align__(16) float qw_s[W][HG][D];  // each warp's query rows (fp32) for its unit
  __shared__ __align__(16) float qp_s[ROPE ? 1 : W][HG][D];  // each warp's q' for its key group
  __shared__ int next_sub;
  __shared__ int abort_flag;
  // rope: the turn of frequency i over TAU tokens (cos, sin), the step between a lane's tokens
  __shared__ float2 rope_step[ROPE ? kHeadDim / 2 : 1];
  // codebooks: the level (in steps) of every key and value code
  __shared__ float lut_s[2][LUT ? 16 : 1];

  // A unit's items are its fp16 items (hw = ceil(n_w / R) of them: the sink rows, then the window
  // rows) followed by its pages.  Page items of this slice are numbered k = 0, 1, ... in list
  // order.  Before item x the list holds unit(x) * n_pages + max(loc(x) - hw, 0) page items, so page
  // k of the slice is global page P_begin + k: unit (P_begin + k) / n_pages, page
  // (P_begin + k) % n_pages of that unit.
  const int hw = (int)(wpu - p.n_pages);
  auto pages_before = [&](int64_t x) -> int64_t {
    const int64_t u = x / wpu, l = x - u * wpu;
    return u * p.n_pages + (l > hw ? l - hw : 0);
  };
  const int64_t P_begin = pages_before(w_begin);
  const int n_pg = (int)(pages_before(w_end) - P_begin);

  // page k of the slice into stage k % n_stages (one thread)
  const unsigned long long wlim = p.wait_ns ? p.wait_ns : kWaitLimitNs;  // page and stage waits
  auto issue_page = [&](int k) {
    if (k + 1 == p.test_withhold) return;  // test hook: this page is never copied
    // 32-bit division: a cache never holds 2^32 pages
    const uint32_t P = (uint32_t)(P_begin + k), np = (uint32_t)p.n_pages;
    const uint32_t u = P / np, loc = P - u * np;
#ifdef KVQ_DEBUG_CHECKS
    {
      const int64_t off = (int64_t)u * p.unit_page_stride + (int64_t)loc * page_bytes;
      if (off < 0 || off + page_bytes > p.pages_bytes) {
        report_error(p.err, kDevBounds);  // not copied: the waits for it run out and end the launch
        return;
      }
    }
#endif
    const int st = k & (n_stages - 1);
    mbar_arrive_expect_tx(&full_bar[st], (uint32_t)page_bytes);
    bulk_g2s(stage_mem + (size_t)st * page_bytes, p.pages + (int64_t)u * p.unit_page_stride + (int64_t)loc * page_bytes,
             (uint32_t)page_bytes, &full_bar[st]);
    stage_issued[st] = (k >> log2S) + 1;
    stage_page[st] = k;
  };
  // A warp may have taken a sub-tile of page k while a stage still serves page k - n_stages
  // (or an older one: warps run ahead of a warp that holds a page while it writes a partial), and a
  // parity wait cannot tell phases 2*n_stages pages apart.  So wait until the stage is assigned
  // page k, then for its copy.  Bounded like every wait here.
  auto wait_page = [&](int k) -> bool {
    const int st = k & (n_stages - 1);
    if (*(volatile int*)&stage_page[st] != k) {
      const unsigned long long t0 = global_ns();
      while (*(volatile int*)&stage_page[st] != k) {
        if (global_ns() - t0 > wlim) return false;
        __nanosleep(128);
      }
    }
    return mbar_wait(&full_bar[st], (k >> log2S) & 1, wlim);
  };

  if (tid == 0) {
    abort_flag = 0;
    next_sub = 0;
    for (int i = 0; i < n_stages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], SPP);
      stage_cnt[i] = 0;
      stage_issued[i] = 0;
      stage_page[i] = -1;
    }
    fence_mbar_init();
  }
  pdl_allow_next();  // the merge kernel may take SMs as this grid's CTAs leave
  pdl_wait();        // the cache, the query, the slot counts and the RoPE table come from earlier work
  if constexpr (ROPE) {
    for (int i = tid; i < D / 2; i += blockDim.x) {
      float c, s;
      rope_cs(p.rope_turns[i], (uint32_t)S::TAU, c, s);
      rope_step[i] = make_float2(c, s);
    }
  }
  if constexpr (LUT) {
    if (tid < 16) {
      lut_s[0][tid] = p.k_lev[tid];
      lut_s[1][tid] = p.v_lev[tid];
    }
  }
  __syncthreads();
  if (tid == 0)
    for (int k = 0; k < n_pg && k < n_stages; ++k) issue_page(k);
  // value of a key / value code: the code itself, or its codebook level
  auto kval = [&](uint32_t c) -> float {
    if constexpr (LUT) return lut_s[0][c];
    else return code_to_float(c);
  };
  auto vval = [&](uint32_t c) -> float {
    if constexpr (LUT) return lut_s[1][c];
    else return code_to_float(c);
  };

  // ---------------- per-warp work
  const int kap = lane % KAPPA;  // channel chunk
  const int tau = lane / KAPPA;  // token slot
  // key channels of this lane: a contiguous chunk, or (rope) half a chunk in each half of the head
  const int kc_lo = ROPE ? kap * S::HALF : kap * CPL;
  const int vc_lo = kap * CPL;
  const int ng = D >> p.log2G;
  const int gv = vc_lo >> p.log2G;
  // fast key path: 2^(149-kCodeExp-B*pos) of the channels this lane prepares for the group products
  float k_unscale[D / 32];
#pragma unroll
  for (int j = 0; j < D / 32; ++j)
    k_unscale[j] = FAST_K ? MaskCodes<S::KBITS_FAST>::scale_in((lane + 32 * j) % MaskCodes<S::KBITS_FAST>::PER_WORD)
                             : 1.0f;
  float (*qs)[D] = qw_s[warp];
  // rope_subtile lane constants: where the lane's key channels (kc_lo .. +3 and the same in the
  // second half of the head) and value channels (vc_lo .. +7) sit in a token's bitstream record,
  // and the turn of its four frequencies over TAU tokens
  const int rk_wl = (kc_lo * BK) >> 5, rk_sl = (kc_lo * BK) & 31;
  const int rk_wh = ((kc_lo + D / 2) * BK) >> 5, rk_sh = ((kc_lo + D / 2) * BK) & 31;
  const int rv_w = (vc_lo * BV) >> 5, rv_s = (vc_lo * BV) & 31;
  float2 rstep_c[2], rstep_s[2], rstep_ns[2];
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    if constexpr (FAST_ROPE) {
      const float2 a = rope_step[kc_lo + 2 * m], b = rope_step[kc_lo + 2 * m + 1];
      rstep_c[m] = make_float2(a.x, b.x);
      rstep_s[m] = make_float2(a.y, b.y);
      rstep_ns[m] = make_float2(-a.y, -b.y);
    } else {
      rstep_c[m] = rstep_s[m] = rstep_ns[m] = make_float2(0.0f, 0.0f);
    }
  }

  LaneState<HG, CPL> st;
  // rope_subtile: st.acc lives in this warp's shared-memory slot between sub-tiles (float4 i of
  // lane l at [i][l]: conflict-free), and in registers only where values are accumulated
  float4* acc_s = reinterpret_cast<float4*>(stage_mem + ((size_t)page_bytes << log2S)) + warp * (HG * CPL / 4) * 32;
  auto acc_store = [&]() {
    if constexpr (FAST_ROPE) {
#pragma unroll
      for (int i = 0; i < HG * CPL / 4; ++i)
        acc_s[i * 32 + lane] = make_float4(st.acc[i / (CPL / 4)][4 * (i % (CPL / 4))], st.acc[i / (CPL / 4)][4 * (i % (CPL / 4)) + 1],
                                           st.acc[i / (CPL / 4)][4 * (i % (CPL / 4)) + 2], st.acc[i / (CPL / 4)][4 * (i % (CPL / 4)) + 3]);
    }
  };
  auto acc_load = [&]() {
    if constexpr (FAST_ROPE) {
#pragma unroll
      for (int i = 0; i < HG * CPL / 4; ++i) {
        const float4 v = acc_s[i * 32 + lane];
        st.acc[i / (CPL / 4)][4 * (i % (CPL / 4))] = v.x;
        st.acc[i / (CPL / 4)][4 * (i % (CPL / 4)) + 1] = v.y;
        st.acc[i / (CPL / 4)][4 * (i % (CPL / 4)) + 2] = v.z;
        st.acc[i / (CPL / 4)][4 * (i % (CPL / 4)) + 3] = v.w;
      }
    }
  };
  st.reset();
  acc_store();

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
      if (__any_sync(kFull, over)) {
#pragma unroll
        for (int off = KAPPA; off < 32; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, off));
        const float mnew = fmaxf(tmax, st.m[h]);
        const float f = st.m[h] == -INFINITY ? 0.0f : exp2f(st.m[h] - mnew);
        st.l[h] *= f;
        st.zsum[h] *= f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) st.acc[h][i] *= f;
        if constexpr (FAST_ROPE) {
          if (((lane % KAPPA) & 3) == h) st.lp *= f;
        }
        st.m[h] = mnew;
      }
      const bool live = st.m[h] != -INFINITY;
#pragma unroll
      for (int j = 0; j < TPL; ++j) sc[j][h] = live ? exp2f(sc[j][h] - st.m[h]) : 0.0f;
    }
  };

  // this warp's query rows q[b][kvh*HG .. kvh*HG+HG-1][:] (contiguous fp16) as floats
  auto load_q = [&](int64_t unit) {
    constexpr int PERL = HG * D / 32;
    const int64_t b = unit / p.Hkv, kvh = unit - b * p.Hkv;
    float v[PERL];
    load_halves<PERL>(p.q + (b * p.Hq + kvh * HG) * D + lane * PERL, v);
    __syncwarp();  // every lane is done with the previous unit's rows
#pragma unroll
    for (int i = 0; i < PERL; ++i) (&qs[0][0])[lane * PERL + i] = v[i];
    __syncwarp();
  };

  // This warp leaves `unit`: one partial into the unit's next free slot (the merge kernel that
  // follows the launch combines the slots).
  auto epilogue = [&](int64_t unit) {
    constexpr int NOUT = CPL / TAU;  // channels per head a lane holds after the reduction
    static_assert(NOUT == 4, "the partial of a lane is one float4 per head");
    acc_load();
    if constexpr (FAST_ROPE) {
      // page weights: lane kap of a slot summed head kap % 4; gather them into every lane's l
      float lq = st.lp;
      lq += __shfl_xor_sync(kFull, lq, 4);
      lq += __shfl_xor_sync(kFull, lq, 8);
#pragma unroll
      for (int h = 0; h < HG; ++h) st.l[h] += __shfl_sync(kFull, lq, tau * KAPPA + h);
      st.lp = 0.0f;
    }
    // l and the value zero-point sums over the warp's token slots (lanes of one slot hold copies)
#pragma unroll
    for (int h = 0; h < HG; ++h)
#pragma unroll
      for (int off = KAPPA; off < 32; off <<= 1) {
        st.l[h] += __shfl_xor_sync(kFull, st.l[h], off);
        st.zsum[h] += __shfl_xor_sync(kFull, st.zsum[h], off);
      }
    // reduce-scatter of acc over the token slots: each step keeps the half of the chunk that the
    // lane's slot bit selects, so the lane ends with channels vc_lo + NOUT*tau .. + NOUT - 1
#pragma unroll
    for (int h = 0; h < HG; ++h) {
#pragma unroll
      for (int half = CPL / 2, bit = TAU / 2; half >= NOUT; half >>= 1, bit >>= 1) {
        const bool up = (tau & bit) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float send = up ? st.acc[h][i] : st.acc[h][i + half];
          const float keep = up ? st.acc[h][i + half] : st.acc[h][i];
          st.acc[h][i] = keep + __shfl_xor_sync(kFull, send, bit * KAPPA);
        }
      }
    }
    // undo the per-position code scale of the fast value path; add the value zero-point sums
#pragma unroll
    for (int h = 0; h < HG; ++h)
#pragma unroll
      for (int i = 0; i < NOUT; ++i) {
        float a = st.acc[h][i];
        if constexpr (FAST_V) a *= MaskCodes<FAST_V ? BV : 2>::scale_out((vc_lo + NOUT * tau + i) % (32 / BV));
        if constexpr (FAST_ROPE) a *= rope_v_scale_out(i);  // channel 4*tau + i of the chunk: position i
        st.acc[h][i] = a + st.zsum[h];
      }
    const int64_t b = unit / p.Hkv, kvh = unit - b * p.Hkv;
    const int64_t bh0 = b * p.Hq + kvh * HG;
    int slot = 0;
    if (lane == 0) slot = atomicAdd(p.nslot + unit, 1);
    slot = __shfl_sync(kFull, slot, 0);
    if (slot < p.max_slots) {
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const int64_t so = (bh0 + h) * p.max_slots + slot;
        *reinterpret_cast<float4*>(p.part_acc + so * D + vc_lo + NOUT * tau) =
            make_float4(st.acc[h][0], st.acc[h][1], st.acc[h][2], st.acc[h][3]);
        if (lane == 0) *reinterpret_cast<float2*>(p.part_ml + so * 2) = make_float2(st.m[h], st.l[h]);
      }
    } else if (lane == 0) {
      report_error(p.err, kDevBadArgument);  // slots are sized for the grid: not reached
    }
  };

  // ---------------- keys stored before RoPE, four query heads per kv head: one 32-token page
  // sub-tile on packed fp32 pairs.  Lane (tau, kap) covers tokens tau + TAU*j (j < 16) on key
  // channels kc_lo + i and kc_lo + D/2 + i (i < 4: four frequencies) and value channels vc_lo + i
  // (i < 8).
  //  * Keys: the lane's two 4-code runs of a token are funnel-shifted out of the record; code i,
  //    masked in place, is the fp32 subnormal code * 2^(BK*i) * 2^-149, so one FMA against
  //    s * 2^(85 - BK*i) and z * 2^-64 gives the dequantized key times 2^-64, exactly as rounded as
  //    z + s*code.  The pairs (c, c + D/2) are rotated by the token's angle, turned on from the
  //    lane's first token by angle addition, and dotted with the four heads' query rows.
  //  * Sparse entries: the dense code there is 0 (value z), so each adds (x - z) times the rotated
  //    query at its channel, computed once per entry by the lane of its token.
  //  * Scores of four tokens x four heads are reduce-scattered over the slot's 16 lanes (15
  //    exchanges instead of 64 butterflies), so lane kap ends with token 4b + kap/4, head kap%4 of
  //    block b and the softmax runs once per score, not once per lane.
  //  * Values: the lane's eight codes are two masked 4-code runs against p*s*2^(149 - kCodeExp)
  //    (accumulator units as rope_v_scale_out undoes), four heads per code in packed FMAs.
  auto rope_subtile = [&](const uint8_t* pgm, int stt, int64_t page_tok0) {
    if constexpr (FAST_ROPE) {
      static_assert(HG == 4 && S::HALF == 4 && CPL == 8 && KAPPA == 16 && TAU == 2 && TPL == 16, "one layout");
      const uint32_t* kc = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_kc);
      const uint32_t* km = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_km);
      const uint32_t* vcw = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_vc);
      const uint32_t* vm = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_vm);
      constexpr uint32_t KMASK = (1u << BK) - 1u, VMASK = (1u << BV) - 1u;
      constexpr int KW = D * BK / 32, VW = D * BV / 32;  // words of a token's key / value record
      const int g = (stt * 32) >> p.log2G;                 // key group (G >= 32)
      const int hl = kap & 3;                              // head of this lane's scores
      // query rows of the lane's key channels, as pairs of neighbouring channels
      float2 ql[HG][2], qh[HG][2];
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float4 a = *reinterpret_cast<const float4*>(&qs[h][kc_lo]);
        const float4 b = *reinterpret_cast<const float4*>(&qs[h][kc_lo + D / 2]);
        ql[h][0] = make_float2(a.x, a.y);
        ql[h][1] = make_float2(a.z, a.w);
        qh[h][0] = make_float2(b.x, b.y);
        qh[h][1] = make_float2(b.z, b.w);
      }
      // the group's zero points and steps in the masked codes' units (see above)
      float2 zl2[2], sl2[2], zh2[2], sh2[2];
      {
        const uint4 a = *reinterpret_cast<const uint4*>(km + g * D + kc_lo);
        const uint4 b = *reinterpret_cast<const uint4*>(km + g * D + kc_lo + D / 2);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
        float zl[4], sl[4], zh[4], sh[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float pos = __uint_as_float((uint32_t)(127 + 85 - BK * i) << 23);
          const float2 za = __half22float2(*reinterpret_cast<const __half2*>(&aw[i]));
          const float2 zb = __half22float2(*reinterpret_cast<const __half2*>(&bw[i]));
          zl[i] = za.x * 0x1.0p-64f;
          sl[i] = za.y * pos;
          zh[i] = zb.x * 0x1.0p-64f;
          sh[i] = zb.y * pos;
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          zl2[m] = make_float2(zl[2 * m], zl[2 * m + 1]);
          sl2[m] = make_float2(sl[2 * m], sl[2 * m + 1]);
          zh2[m] = make_float2(zh[2 * m], zh[2 * m + 1]);
          sh2[m] = make_float2(sh[2 * m], sh[2 * m + 1]);
        }
      }
      // cos/sin of the lane's four frequencies at its first token (exact from the turn count)
      float2 rc[2], rs[2];
      {
        float c[4], sn[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) rope_cs(p.rope_turns[kc_lo + i], (uint32_t)(page_tok0 + stt * 32 + tau), c[i], sn[i]);
        rc[0] = make_float2(c[0], c[1]);
        rc[1] = make_float2(c[2], c[3]);
        rs[0] = make_float2(sn[0], sn[1]);
        rs[1] = make_float2(sn[2], sn[3]);
      }
      // sparse entries of token `lane` of the sub-tile: their score corrections per head
      float dlt[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) dlt[h] = 0.0f;
      const int nsp = p.nsp;
      if (nsp > 0) {
        const int tt = stt * 32 + lane;
        const uint8_t* si = pgm + p.lay.off_si;
        const uint16_t* sv = reinterpret_cast<const uint16_t*>(pgm + p.lay.off_sv);
        for (int k = 0; k < nsp; ++k) {
          const int c = si[tt * nsp + k];
          const float dx = h2f(sv[tt * nsp + k]) - h2f((uint16_t)(km[g * D + c] & 0xFFFFu));
          float cs, sn;
          rope_cs(p.rope_turns[c & (D / 2 - 1)], (uint32_t)(page_tok0 + tt), cs, sn);
          const float sg = c < D / 2 ? sn : -sn;  // the rotated query at c: q_c cos +- q_(c^D/2) sin
#pragma unroll
          for (int h = 0; h < HG; ++h) dlt[h] = fmaf(dx, fmaf(qs[h][c], cs, qs[h][c ^ (D / 2)] * sg), dlt[h]);
        }
      }
      // ---- scores, four tokens at a time (one block in registers at a time)
      float r0 = 0.0f, r1 = 0.0f, r2 = 0.0f, r3 = 0.0f;
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        float v[16];  // entry 4*jj + h: token 4b + jj, head h (this lane's channels only)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * b + jj;
          const uint32_t* rec = kc + (stt * 32 + tau + TAU * j) * KW;
          const uint32_t xl = __funnelshift_r(rec[rk_wl], rec[rk_wl + 1], rk_sl);
          const uint32_t xh = __funnelshift_r(rec[rk_wh], rec[rk_wh + 1], rk_sh);
          float2 acc[HG];
#pragma unroll
          for (int h = 0; h < HG; ++h) acc[h] = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const float2 fl = make_float2(__uint_as_float(xl & (KMASK << (BK * 2 * m))),
                                          __uint_as_float(xl & (KMASK << (BK * (2 * m + 1)))));
            const float2 fh = make_float2(__uint_as_float(xh & (KMASK << (BK * 2 * m))),
                                          __uint_as_float(xh & (KMASK << (BK * (2 * m + 1)))));
            const float2 kl = __ffma2_rn(fl, sl2[m], zl2[m]);
            const float2 kh = __ffma2_rn(fh, sh2[m], zh2[m]);
            const float2 nsn = make_float2(-rs[m].x, -rs[m].y);
            const float2 rl = __ffma2_rn(kh, nsn, __fmul2_rn(kl, rc[m]));   // kl cos - kh sin
            const float2 rh = __ffma2_rn(kl, rs[m], __fmul2_rn(kh, rc[m]));  // kh cos + kl sin
#pragma unroll
            for (int h = 0; h < HG; ++h) acc[h] = __ffma2_rn(qh[h][m], rh, __ffma2_rn(ql[h][m], rl, acc[h]));
          }
#pragma unroll
          for (int h = 0; h < HG; ++h) v[4 * jj + h] = acc[h].x + acc[h].y;
          {  // (the turn past the last token is not used)
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const float2 c = rc[m], sn = rs[m];
              rc[m] = __ffma2_rn(c, rstep_c[m], __fmul2_rn(sn, rstep_ns[m]));  // cos(a + d)
              rs[m] = __ffma2_rn(sn, rstep_c[m], __fmul2_rn(c, rstep_s[m]));   // sin(a + d)
            }
          }
        }
        // reduce-scatter over the slot's lanes (kap bits 3..0): lane kap keeps entry kap
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) {
          const bool up = (kap & off) != 0;
#pragma unroll
          for (int i = 0; i < off; ++i) {
            const float send = up ? v[i] : v[i + off];
            const float keep = up ? v[i + off] : v[i];
            v[i] = keep + __shfl_xor_sync(kFull, send, off);
          }
        }
        r0 = b == 0 ? v[0] : r0;
        r1 = b == 1 ? v[0] : r1;
        r2 = b == 2 ? v[0] : r2;
        r3 = b == 3 ? v[0] : r3;
      }
      const float r[4] = {r0, r1, r2, r3};
      // final scores (log2 units) of token 4b + kap/4 of the slot, head hl
      const float sgl = 0x1.0p64f * p.qk_scale_log2;
      float sb[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float d = 0.0f;
        if (nsp > 0) {
          const int src = tau + TAU * (4 * b + (kap >> 2));  // the lane that holds that token's corrections
          const float d0 = __shfl_sync(kFull, dlt[0], src), d1 = __shfl_sync(kFull, dlt[1], src);
          const float d2 = __shfl_sync(kFull, dlt[2], src), d3 = __shfl_sync(kFull, dlt[3], src);
          d = hl == 0 ? d0 : hl == 1 ? d1 : hl == 2 ? d2 : d3;
        }
        sb[b] = fmaf(r[b], sgl, d * p.qk_scale_log2);
      }
      // ---- online softmax: the lane's four scores all belong to head hl
      auto mof = [&](int h) { return h == 0 ? st.m[0] : h == 1 ? st.m[1] : h == 2 ? st.m[2] : st.m[3]; };
      float ml = mof(hl);
      const float tmax = fmaxf(fmaxf(sb[0], sb[1]), fmaxf(sb[2], sb[3]));
      const bool over = tmax > ml + kLazyRescale || (ml == -INFINITY && tmax != -INFINITY);
      float fac[HG];  // rescale of the accumulators (applied when they are loaded for the values)
#pragma unroll
      for (int h = 0; h < HG; ++h) fac[h] = 1.0f;
      if (__any_sync(kFull, over)) {
        float mx = tmax;  // the largest of head hl over the sub-tile: lanes kap % 4 == hl of both slots
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float mnew = fmaxf(__shfl_sync(kFull, mx, h), st.m[h]);  // lane h holds head h
          const float f = st.m[h] == -INFINITY ? 0.0f : exp2f(st.m[h] - mnew);
          st.l[h] *= f;
          st.zsum[h] *= f;
          fac[h] = f;
          if (hl == h) st.lp *= f;
          st.m[h] = mnew;
        }
        ml = mof(hl);
      }
      float pb[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        pb[b] = exp2f(sb[b] - ml);
        st.lp += pb[b];
      }
      // ---- values
      acc_load();
#pragma unroll
      for (int h = 0; h < HG; ++h)
#pragma unroll
        for (int i = 0; i < CPL; ++i) st.acc[h][i] *= fac[h];
      // while the accumulators are in registers their shared-memory slot holds the sub-tile's
      // weights, [slot tau][token j][head h]: one 16-byte load gives a token's four heads
      __syncwarp();
      float* const p_s = reinterpret_cast<float*>(acc_s);
#pragma unroll
      for (int b = 0; b < 4; ++b) p_s[tau * 64 + 16 * b + kap] = pb[b];  // token 4b + kap/4, head kap%4
      __syncwarp();
      float2 z01 = make_float2(st.zsum[0], st.zsum[1]), z23 = make_float2(st.zsum[2], st.zsum[3]);
      const float kScIn = __uint_as_float((uint32_t)(127 + 149 - kCodeExp) << 23);
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = 4 * b + jj;
        const int tt = stt * 32 + tau + TAU * j;
        const float4 pq = *reinterpret_cast<const float4*>(p_s + (tau * 16 + j) * 4);
        const float2 p01 = make_float2(pq.x, pq.y), p23 = make_float2(pq.z, pq.w);
        const float2 zs = __half22float2(*reinterpret_cast<const __half2*>(vm + tt * ng + gv));
        const float sv = zs.y * kScIn;
        const uint32_t* rec = vcw + tt * VW;
        const uint32_t x = __funnelshift_r(rec[rv_w], rec[rv_w + 1], rv_s);
        const uint32_t x2 = x >> (4 * BV);
        float2 f2[4];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          f2[m] = make_float2(__uint_as_float(x & (VMASK << (BV * 2 * m))), __uint_as_float(x & (VMASK << (BV * (2 * m + 1)))));
          f2[2 + m] = make_float2(__uint_as_float(x2 & (VMASK << (BV * 2 * m))),
                                  __uint_as_float(x2 & (VMASK << (BV * (2 * m + 1)))));
        }
        const float2 ps01 = __fmul2_rn(p01, make_float2(sv, sv)), ps23 = __fmul2_rn(p23, make_float2(sv, sv));
        const float psh[HG] = {ps01.x, ps01.y, ps23.x, ps23.y};
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float2 ps2 = make_float2(psh[h], psh[h]);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float2 a = __ffma2_rn(f2[m], ps2, make_float2(st.acc[h][2 * m], st.acc[h][2 * m + 1]));
            st.acc[h][2 * m] = a.x;
            st.acc[h][2 * m + 1] = a.y;
          }
        }
        z01 = __ffma2_rn(p01, make_float2(zs.x, zs.x), z01);
        z23 = __ffma2_rn(p23, make_float2(zs.x, zs.x), z23);
      }
      }
      st.zsum[0] = z01.x;
      st.zsum[1] = z01.y;
      st.zsum[2] = z23.x;
      st.zsum[3] = z23.y;
      __syncwarp();  // every lane is done with the weights before the accumulators go back
      acc_store();
    }
  };

  int64_t cur = -1, ustart = 0;
  while (true) {
    int s = 0;
    if (lane == 0) s = atomicAdd(&next_sub, 1);
    s = __shfl_sync(kFull, s, 0);
    if (s >= n_sub || *(volatile int*)&abort_flag) break;
    const int sx = SPP == 4 ? s >> 2 : SPP == 2 ? s >> 1 : SPP == 1 ? s : s / 3;
    const int stt = s - sx * SPP;  // sub-tile: tokens 32*stt .. 32*stt+31 of the item
    const int64_t x = w_begin + sx;
    if (cur < 0 || x >= ustart + wpu) {
      if (cur >= 0) epilogue(cur);
      cur = x / wpu;
      ustart = cur * wpu;
      st.reset();
      acc_store();
      load_q(cur);
    }
    const int loc = (int)(x - ustart);

    if (loc >= hw) {
      // ---------------- a sub-tile of a page of quantized tokens
      const int kpg = (int)(cur * p.n_pages + (loc - hw) - P_begin);
      const int stg = kpg & (n_stages - 1);
      if (!wait_page(kpg)) {
        report_error(p.err, kDevWaitTimeout);
        atomicExch(&abort_flag, 1);
        break;
      }
      const uint8_t* pgm = stage_mem + (size_t)stg * page_bytes;
      const uint32_t* kc = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_kc);
      const uint32_t* km = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_km);
      const uint32_t* vcw = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_vc);
      const uint32_t* vm = reinterpret_cast<const uint32_t*>(pgm + p.lay.off_vm);
      const uint8_t* si = pgm + p.lay.off_si;
      const uint16_t* sv = reinterpret_cast<const uint16_t*>(pgm + p.lay.off_sv);
      const int64_t page_tok0 = p.n_s + (loc - hw) * (int64_t)p.R;

      if constexpr (FAST_ROPE) {
        rope_subtile(pgm, stt, page_tok0);
      } else {
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
            qp_s[warp][h][c] = qs[h][c] * s;
            zp[h] = fmaf(qs[h][c], z, zp[h]);
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
          if constexpr (FAST_K) {
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
              for (int i = 0; i < CPL; ++i) a = fmaf(qp[h][i], kval(codes[i]), a);
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
                for (int h = 0; h < HG; ++h) sc[j][h] = fmaf(qs[h][c], xv - z, sc[j][h]);
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
        // cos/sin of the lane's first token, exact from the turn count, then turned by TAU
        // tokens per step (angle addition; a few fp32 roundings per step)
        float rc[HF], rs[HF];
#pragma unroll
        for (int i = 0; i < HF; ++i)
          rope_cs(p.rope_turns[kc_lo + i], (uint32_t)(page_tok0 + stt * 32 + tau), rc[i], rs[i]);
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
            kl[i] = fmaf(sl[i], kval(cl[i]), zl[i]);
            kh[i] = fmaf(sh[i], kval(ch[i]), zh[i]);
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
          float a[HG];
#pragma unroll
          for (int h = 0; h < HG; ++h) a[h] = 0.0f;
#pragma unroll
          for (int i = 0; i < HF; ++i) {
            const float cs = rc[i], sn = rs[i];
            const float rl = kl[i] * cs - kh[i] * sn;
            const float rh = kh[i] * cs + kl[i] * sn;
#pragma unroll
            for (int h = 0; h < HG; ++h)
              a[h] = fmaf(qs[h][kc_lo + i], rl, fmaf(qs[h][kc_lo + D / 2 + i], rh, a[h]));
            if (j + 1 < TPL) {
              const float2 st = rope_step[kc_lo + i];
              rc[i] = cs * st.x - sn * st.y;
              rs[i] = sn * st.x + cs * st.y;
            }
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
        if constexpr (FAST_V) {
          using MC = MaskCodes<FAST_V ? BV : 2>;
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
            for (int i = 0; i < CPL; ++i) st.acc[h][i] = fmaf(ps, vval(codes[i]), st.acc[h][i]);
          }
        }
      }
      }  // !FAST_ROPE
      __syncwarp();
      if (lane == 0) {
        // release this sub-tile of the stage; the warp releasing its last sub-tile refills the
        // stage with page kpg + n_stages of the slice
        mbar_arrive(&empty_bar[stg]);
        if (atomicAdd(&stage_cnt[stg], 1) % SPP == SPP - 1 && kpg + n_stages < n_pg &&
            !*(volatile int*)&abort_flag) {
          if (mbar_wait(&empty_bar[stg], (kpg >> log2S) & 1, wlim)) {
            issue_page(kpg + n_stages);
          } else {
            report_error(p.err, kDevWaitTimeout);
            atomicExch(&abort_flag, 1);
          }
        }
      }
    } else {
      // ---------------- the fp16 rows, read directly: the n_s sink tokens (positions 0..n_s),
      // then the n_r window tokens (positions n_s + Tq ..).  They are the unit's first items, so
      // their loads overlap the prefetch of the unit's pages.
      const int64_t tq = p.n_pages * (int64_t)p.R;
      const uint16_t* wk = p.wk + cur * p.win_unit_stride;
      const uint16_t* wv = p.wv + cur * p.win_unit_stride;
      const int f = loc * SPP + stt;  // sub-tile of the unit's fp16 rows
      // the newest token comes from the caller's buffers when the step appends it; the warp
      // that covers it also stores it into its window slot
      const int newest = p.k_new ? p.n_w - 1 : -1;
      if (newest >= 32 * f && newest < 32 * f + 32) {
        const uint16_t* src = lane < 16 ? p.k_new + cur * D : p.v_new + cur * D;
        uint16_t* dst = const_cast<uint16_t*>(lane < 16 ? wk : wv) + (int64_t)newest * D;
        reinterpret_cast<uint4*>(dst)[lane & 15] = __ldg(reinterpret_cast<const uint4*>(src) + (lane & 15));
      }
      if (32 * f < p.n_w) {
        acc_load();
        float sc[TPL][HG];
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
          const int tt = f * 32 + tau + TAU * j;
          if (tt >= p.n_w) {
#pragma unroll
            for (int h = 0; h < HG; ++h) sc[j][h] = 0.0f;
            continue;
          }
          const uint16_t* kr = tt == newest ? p.k_new + cur * D : wk + (int64_t)tt * D;
          float a[HG];
#pragma unroll
          for (int h = 0; h < HG; ++h) a[h] = 0.0f;
          if constexpr (!ROPE) {
            float xk[CPL];
            load_halves<CPL>(kr + kc_lo, xk);
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
#pragma unroll
              for (int h = 0; h < HG; ++h) a[h] = fmaf(qs[h][kc_lo + i], xk[i], a[h]);
            }
          } else {
            const uint32_t tpos = (uint32_t)(tt < p.n_s ? tt : tq + tt);
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
                a[h] = fmaf(qs[h][kc_lo + i], rl, fmaf(qs[h][kc_lo + D / 2 + i], rh, a[h]));
            }
          }
#pragma unroll
          for (int h = 0; h < HG; ++h) sc[j][h] = a[h];
        }
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
          const int tt = f * 32 + tau + TAU * j;
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            float a = sc[j][h];
#pragma unroll
            for (int off = 1; off < KAPPA; off <<= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            sc[j][h] = tt < p.n_w ? a * p.qk_scale_log2 : -INFINITY;
          }
        }
        softmax_update(sc);
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
          const int tt = f * 32 + tau + TAU * j;
          if (tt >= p.n_w) continue;
          float xv[CPL];
          const uint16_t* vr = tt == newest ? p.v_new + cur * D : wv + (int64_t)tt * D;
          load_halves<CPL>(vr + vc_lo, xv);
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            const float pw = sc[j][h];
            st.l[h] += pw;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
              // in the units of the fast value path (exact powers of two), undone by the fold
              const float sb = FAST_ROPE ? rope_v_scale_back(i)
                               : FAST_V ? MaskCodes<FAST_V ? BV : 2>::scale_back((vc_lo + i) % (32 / (FAST_V ? BV : 2)))
                                        : 1.0f;
              st.acc[h][i] = fmaf(pw * sb, xv[i], st.acc[h][i]);
            }
          }
        }
        acc_store();
      }
    }
  }
  if (cur >= 0) epilogue(cur);
  // never leave with a copy in flight (only possible after an abort): wait, bounded, for the
  // last copy issued into every stage
  __syncthreads();
  if (tid == 0) {
    for (int i = 0; i < n_stages; ++i)
      if (stage_issued[i] > 0) mbar_wait(&full_bar[i], (stage_issued[i] - 1) & 1);
  }
}

// Page stages of one CTA: the largest power of two up to kMaxStages whose pages fit the opt-in
// shared memory beside the kernel's static arrays; -1 when not even one fits.
template <int BK, int BV, int HG, bool ROPE, bool LUT>
int log2_stages_t(int page_bytes) {
  auto kern = decode_kernel<BK, BV, HG, ROPE, LUT>;
  static int static_smem = -1, optin = -1;
  if (static_smem < 0) {
    cudaFuncAttributes a{};
    int dev = 0;
    if (cudaFuncGetAttributes(&a, kern) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return -1;
    static_smem = (int)a.sharedSizeBytes;
  }
  if (static_smem > 48 * 1024) return -1;  // more static shared memory than a kernel may declare
  const int avail = optin - static_smem - Shape<BK, BV, HG, ROPE, LUT>::ACC_SMEM;
  int l = 4;  // kMaxStages = 16
  while (l >= 0 && ((int64_t)page_bytes << l) > avail) --l;
  return l;
}

template <int BK, int BV, int HG, bool ROPE, bool LUT>
cudaError_t launch_decode_t(const DecodeParams& p, int grid, cudaStream_t s) {
  const int l = log2_stages_t<BK, BV, HG, ROPE, LUT>(p.lay.bytes);
  if (l < 0) return cudaErrorInvalidValue;
  DecodeParams q = p;
  q.log2_stages = l;
  const size_t smem = ((size_t)p.lay.bytes << l) + Shape<BK, BV, HG, ROPE, LUT>::ACC_SMEM;
  auto kern = decode_kernel<BK, BV, HG, ROPE, LUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, (unsigned)grid, Shape<BK, BV, HG, ROPE, LUT>::WARPS * 32, smem, s, q);
}

template <int BK, int BV, int HG, bool ROPE, bool LUT>
int resident_t(int page_bytes, int* warps) {
  *warps = Shape<BK, BV, HG, ROPE, LUT>::WARPS;
  const int l = log2_stages_t<BK, BV, HG, ROPE, LUT>(page_bytes);
  if (l < 0) return 0;
  const size_t smem = ((size_t)page_bytes << l) + Shape<BK, BV, HG, ROPE, LUT>::ACC_SMEM;
  auto kern = decode_kernel<BK, BV, HG, ROPE, LUT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Shape<BK, BV, HG, ROPE, LUT>::WARPS * 32, smem) !=
      cudaSuccess)
    return 0;
  return n;
}

}  // namespace
}  // namespace kvq
