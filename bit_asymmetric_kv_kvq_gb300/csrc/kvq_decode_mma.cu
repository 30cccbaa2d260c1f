// Decode attention on the tensor cores, for pages whose codes are stored in
// fragment order (2- or 4-bit keys and values, keys stored after RoPE).
//
// Both halves of decode attention are small matrix products per 16-token tile
// ("KV cache has a geometry problem, not a bit problem", section "Why the KV
// cache is a problem": every generated token reads the whole cache):
//
//   scores  S[token][head]   = sum_c code_k[token][c] * q'_h[c]  + Z_h,
//           q'_h[c] = q_h[c] s_c, Z_h = sum_c q_h[c] z_c   (keys per channel over G tokens)
//   values  O[c][head]      += sum_t code_v[t][c] * p_h[t] s_{t,g(c)}  (+ sum_t p_h[t] z_{t,g(c)})
//                                                          (values per token over G channels)
//
// Each is issued as mma.sync m16n8k16 (fp16 in, fp32 accumulate) with the codes
// as the A operand.  A code pair is turned into an A register with one AND:
// masked in place, the two codes are exact fp16 subnormals code * 2^(B*p) * 2^-24
// (see frag_key_pair / frag_value_pair for where each lane's codes sit).  The
// position scale 2^(B*p) is folded into the B operand for keys (the B row of
// that k-slot) and into the output scale for values (one position per M-tile).
// Key B values are split into a high and a low fp16 part (two of the eight N
// columns per head), which keeps them to about 22 significant bits: a score
// error moves a softmax weight by the same relative amount.  Value B values
// p_t * s_t are single fp16 numbers (one column per (group, head)): their
// rounding (2^-12 relative per product) moves the output far less than the
// 2e-3 the outputs are held to, and one column per head halves the value
// operands to build.
//
// Scheduling is that of the CUDA-core kernel: one CTA per SM streams a
// contiguous slice of the (window, pages) work list through a ring of page
// stages, its warps take 32-token sub-tiles from a shared counter, keep their
// own online-softmax state per unit, and leave one partial per unit they
// touched; the merge kernel launched after combines them.  A window sub-tile
// (fp16 tokens not yet quantized) is computed on the CUDA cores as a
// partial of its own.
#include <cuda_fp16.h>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

namespace {

// Warps of the one CTA per SM: 16 at up to 128 registers.  (Four query heads per kv head once held
// value operands split into high and low parts and a scale per head, spilled at 128 registers and
// ran 12 warps; with single fp16 value operands and one key scale they fit.)
template <int HG>
__host__ __device__ constexpr int mma_warps() { return 16; }
constexpr int kMmaMaxStages = 16;
constexpr unsigned kAll = 0xffffffffu;
constexpr float kLazy = 8.0f;  // the running maximum moves only when a score passes it by 8 (log2 units)
// Running maximum before the first score: finite, below every score, so the first sub-tile raises it
// by the plain lazy test and the rescale factor 2^(kNoMax - m) of the (empty) sums is 0.
constexpr float kNoMax = -1.0e30f;

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }  // |e| <= 126

// 2^x by the hardware approximation, results below 2^-126 flushed to zero: softmax weights that
// small (relative to a running maximum at most 2^8 below the largest) change no sum.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Code pairs of one fragment word (B-bit codes): pair j read in place for j < DIR, from the
// word shifted down by SHIFT bits otherwise; pos(j) is the exponent of its position scale.
template <int B>
struct Pairs {
  static constexpr int PER = 16 / B;
  static constexpr int DIR = 10 / B;
  static constexpr int SHIFT = B * DIR;
  __host__ __device__ static constexpr int pos(int j) { return B * (j < DIR ? j : j - DIR); }
  __device__ __forceinline__ static uint32_t get(uint32_t w, uint32_t ws, int j) {
    const uint32_t m = ((((1u << B) - 1u) * 0x00010001u) << pos(j));
    return (j < DIR ? w : ws) & m;
  }
};

__device__ __forceinline__ uint32_t h2bits(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }

// x = q * s for a pair of channels, split into fp16 high parts and the fp16 rounding of what they
// leave, for |x| < 2^(15 - pk).  With M = 1.5 * 2^(27 - pk), fl(x + M) lies in [2^(27-pk), 2^(28-pk))
// whose fp32 spacing is 2^(4 - pk), so fl(x + M) - M is x rounded to that grid (exact subtraction):
// a multiple of 2^(4-pk) below 2^(15-pk) in magnitude, at most 11 significant bits, exact in fp16.
// What it leaves (|r| <= 2^(3-pk), exact in fp32) is rounded to fp16 once: hi + lo = x within
// 2^-23 of the bound.  Two values per instruction, no conversion back from fp16.
__device__ __forceinline__ void split_qs(float2 q, float2 s, float2 M, uint32_t& hi, uint32_t& lo) {
  const float2 t = __ffma2_rn(q, s, M);
  const float2 h = __fadd2_rn(t, make_float2(-M.x, -M.y));
  const float2 r = __ffma2_rn(q, s, make_float2(-h.x, -h.y));
  hi = h2bits(__float22half2_rn(h));
  lo = h2bits(__float22half2_rn(r));
}

template <int BK, int BV, int HG, bool STD>
__global__ void __launch_bounds__(mma_warps<HG>() * 32, 1) decode_mma_kernel(const DecodeParams p) {
  constexpr int D = kHeadDim, W = mma_warps<HG>();
  constexpr int NCOL = HG;       // value B columns per value group: one per head
  constexpr int GPB = 8 / NCOL;  // value groups per B fragment
  constexpr int NBM = (D / 32 + GPB - 1) / GPB;  // B fragments per value tile at most (G = 32)
  // value group g sits in B fragment g % NBM, column block g / NBM: the groups a lane feeds are
  // consecutive (one 8-byte load per token when NBM = 2)
  constexpr int KCOL = 2 * HG;   // key B columns: (head, high/low)
  constexpr int KPW = 8 / BK;    // key k-chunks per fragment word
  using PK = Pairs<BK>;
  using PV = Pairs<BV>;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g8 = lane >> 2, t4 = lane & 3;  // mma fragment coordinates
  const int cta = blockIdx.x, grid = gridDim.x;
  const int64_t wpu = p.work_per_unit;
  const int64_t total = p.n_units * wpu;
  const int64_t w_begin = (int64_t)cta * total / grid;
  const int64_t w_end = (int64_t)(cta + 1) * total / grid;
  using SP = StdPage<BK, BV>;
  const int page_bytes = STD ? SP::bytes : p.lay.bytes;
  const int off_kc = STD ? SP::kc : p.lay.off_kc, off_km = STD ? SP::km : p.lay.off_km;
  const int off_vc = STD ? SP::vc : p.lay.off_vc, off_vm = STD ? SP::vm : p.lay.off_vm;
  const int log2G = STD ? 5 : p.log2G;
  const int nsp = STD ? 0 : p.nsp;
  // the page ring: page k of the slice goes to stage k mod n_stages on lap k / n_stages
  const int n_stages = p.n_stages;
  const uint32_t smagic = p.stage_magic;
  auto lap_of = [&](int k) { return (int)__umulhi((uint32_t)k, smagic); };
  const int SPP = STD ? 4 : p.R / 32;
  const int n_sub = (int)(w_end - w_begin) * SPP;
  const int ng = D >> log2G;               // value groups per token

  // dynamic shared memory: the page stages, then each warp's query rows (fp32) and key B
  // fragments (static arrays stay small: static shared memory is limited to 48 KB)
  extern __shared__ __align__(128) uint8_t stage_mem[];
  float(*qw_s)[HG][D] = reinterpret_cast<float(*)[HG][D]>(stage_mem + (size_t)page_bytes * n_stages);
  uint32_t(*bk_s)[KCOL][4][16] = reinterpret_cast<uint32_t(*)[KCOL][4][16]>(qw_s + W);
  __shared__ __align__(8) uint64_t full_bar[kMmaMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMmaMaxStages];
  __shared__ int stage_cnt[kMmaMaxStages];
  __shared__ int stage_issued[kMmaMaxStages];
  __shared__ int stage_page[kMmaMaxStages];     // page of the slice a stage holds or is being filled with
  __shared__ int next_sub;
  __shared__ int abort_flag;
  __shared__ __align__(16) uint32_t zero_frag[4][16];  // B fragments of the unused columns

  const int hw = (int)(wpu - p.n_pages);
  auto pages_before = [&](int64_t x) -> int64_t {
    const int64_t u = x / wpu, l = x - u * wpu;
    return u * p.n_pages + (l > hw ? l - hw : 0);
  };
  const int64_t P_begin = pages_before(w_begin);
  const int n_pg = (int)(pages_before(w_end) - P_begin);
  const unsigned long long wlim = p.wait_ns ? p.wait_ns : kWaitLimitNs;  // page and stage waits
  auto issue_page = [&](int k) {
    if (k + 1 == p.test_withhold) return;  // test hook: this page is never copied
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
    const int lap = lap_of(k), st = k - lap * n_stages;
    mbar_arrive_expect_tx(&full_bar[st], (uint32_t)page_bytes);
    bulk_g2s(stage_mem + (size_t)st * page_bytes, p.pages + (int64_t)u * p.unit_page_stride + (int64_t)loc * page_bytes,
             (uint32_t)page_bytes, &full_bar[st]);
    stage_issued[st] = lap + 1;
    stage_page[st] = k;
  };
  // A warp may have taken a sub-tile of page k while a stage still serves page k - n_stages
  // (or an older one: warps run ahead of a warp that holds a page while it writes a partial), and a
  // parity wait cannot tell phases 2*n_stages pages apart.  So wait until the stage is assigned
  // page k, then for its copy.  Bounded like every wait here.
  auto wait_page = [&](int k) -> bool {
    const int lap = lap_of(k), st = k - lap * n_stages;
    if (*(volatile int*)&stage_page[st] != k) {
      const unsigned long long t0 = global_ns();
      while (*(volatile int*)&stage_page[st] != k) {
        if (global_ns() - t0 > wlim) return false;
        __nanosleep(128);
      }
    }
    return mbar_wait(&full_bar[st], lap & 1, wlim);
  };

  if (tid < 64) (&zero_frag[0][0])[tid] = 0u;
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
  pdl_wait();        // the cache, the query and the slot counts come from earlier kernels
  __syncthreads();
  if (tid == 0)
    for (int k = 0; k < n_pg && k < n_stages; ++k) issue_page(k);

  float (*qs)[D] = qw_s[warp];
  const int hcol = g8 % HG;          // head of this lane's value B column g8
  const int gl = g8 / HG;            // value group of that column within a B fragment
  const int hmine = t4 % HG;         // head of this lane's scores (lanes t4 < HG) and running maximum
  // the lane's value D columns n = 2*t4 + e are (group n / HG within the fragment, head n % HG)
  const int hd0 = (2 * t4) % HG, hd1 = (2 * t4 + 1) % HG;

  // ---- per-warp state for the current unit
  float dv[8][4];            // value accumulators, one m16n8 tile per 16 channels
  float mrun;                // running maximum of head hmine (log2 units), kNoMax before the first score
  float lacc, zacc[NBM];     // sum of p (column owners) and p*z per B fragment
  int es;                    // exponent bound of the value scales seen (B values carry 2^(6-es));
                             // starts below every fp16 scale (>= 2^-24)
  auto reset = [&]() {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) dv[i][j] = 0.0f;
    mrun = kNoMax;
    lacc = 0.0f;
#pragma unroll
    for (int i = 0; i < NBM; ++i) zacc[i] = 0.0f;
    es = -30;
  };

  int eq = 0;  // exponent of the current unit's largest |q| (over its heads)
  auto load_q = [&](int64_t unit) {
    constexpr int PERL = HG * D / 32;
    const int64_t b = unit / p.Hkv, kvh = unit - b * p.Hkv;
    const uint16_t* src = p.q + (b * p.Hq + kvh * HG) * D + lane * PERL;
    float v[PERL];
#pragma unroll
    for (int i = 0; i < PERL; i += 4) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(src + i));
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
      const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
      v[i] = a.x;
      v[i + 1] = a.y;
      v[i + 2] = c.x;
      v[i + 3] = c.y;
    }
    float mq = 0.0f;
#pragma unroll
    for (int i = 0; i < PERL; ++i) mq = fmaxf(mq, fabsf(v[i]));
    // |q| >= 0 orders like its bit pattern: one integer reduction finds the unit's largest
    const uint32_t mqb = __reduce_max_sync(kAll, __float_as_uint(mq));
    eq = mqb != 0u ? (int)((mqb >> 23) & 0xFF) - 127 : 0;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < PERL; ++i) (&qs[0][0])[lane * PERL + i] = v[i];
    __syncwarp();
  };

  auto slot_of = [&](int64_t unit) {
    int slot = 0;
    if (lane == 0) slot = atomicAdd(p.nslot + unit, 1);
    return __shfl_sync(kAll, slot, 0);
  };

  // This warp leaves `unit`: its partial (m, l, acc) per head into a fresh slot (the merge
  // kernel that follows the launch combines the slots).
  auto epilogue = [&](int64_t unit) {
    const int64_t b = unit / p.Hkv, kvh = unit - b * p.Hkv;
    const int64_t bh0 = b * p.Hq + kvh * HG;
    // column owners' sums over the four lanes of a fragment row (t4)
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      lacc += __shfl_xor_sync(kAll, lacc, off);
#pragma unroll
      for (int i = 0; i < NBM; ++i) zacc[i] += __shfl_xor_sync(kAll, zacc[i], off);
    }
    const int slot = slot_of(unit);
    if (slot < p.max_slots) {
      // zero-point sums of the (group, head) of this lane's D columns n = 2*t4 + e: owned by the
      // lanes of B column n (lane 4n)
      float zs[2][NBM];
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int i = 0; i < NBM; ++i) zs[e][i] = __shfl_sync(kAll, zacc[i], 4 * (2 * t4 + e));
      const float osc = pow2f(24 - (6 - es));
#pragma unroll
      for (int mc = 0; mc < 8; ++mc) {
        const int grp = (16 * mc) >> log2G;
        const float s = osc * pow2f(-PV::pos(mc % PV::PER));
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int n = 2 * t4 + e;
          if (n / HG != grp / NBM) continue;  // this column holds another group's products
          float z = zs[e][0];
#pragma unroll
          for (int i = 1; i < NBM; ++i)
            if (grp % NBM == i) z = zs[e][i];
          float* dst = p.part_acc + ((bh0 + n % HG) * p.max_slots + slot) * D + 16 * mc + g8;
          dst[0] = fmaf(dv[mc][e], s, z);
          dst[8] = fmaf(dv[mc][2 + e], s, z);
        }
      }
      // (m, l) of head h: m from lane h, l from the owners of B column h (lane 4h)
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float mh = __shfl_sync(kAll, mrun, h);
        const float lh = __shfl_sync(kAll, lacc, 4 * h);
        if (lane == 0) *reinterpret_cast<float2*>(p.part_ml + ((bh0 + h) * p.max_slots + slot) * 2) = make_float2(mh, lh);
      }
    } else if (lane == 0) {
      report_error(p.err, kDevBadArgument);  // slots are sized for the grid: not reached
    }
  };

  // A sub-tile of the fp16 rows (the sink tokens, then the window tokens; rows 32*stt ..) as a
  // partial of its own: lane l scores row 32*stt + l, then owns channels 4l .. 4l+3 of the
  // weighted sum.
  auto window_subtile = [&](int64_t unit, int stt) {
    const int64_t b = unit / p.Hkv, kvh = unit - b * p.Hkv;
    const int64_t bh0 = b * p.Hq + kvh * HG;
    const uint16_t* wk = p.wk + unit * p.win_unit_stride;
    const uint16_t* wv = p.wv + unit * p.win_unit_stride;
    const int tok = 32 * stt + lane;
    const bool live = tok < p.n_w;
    // the newest token comes from the caller's buffers when the step appends it (stored below)
    const int newest = p.k_new ? p.n_w - 1 : -1;
    // the slot early, so the atomic's round trip overlaps the row loads
    int slot = 0;
    if (lane == 0) slot = atomicAdd(p.nslot + unit, 1);
    // the value row of this lane's token heads for L2 while the key rows are read
    if (live) {
      const uint16_t* vr = tok == newest ? p.v_new + unit * D : wv + (int64_t)tok * D;
      prefetch_l2(vr);
      prefetch_l2(vr + 64);
    }
    // rows come from DRAM: with one query head the whole 256-byte key row of a lane is in flight at
    // once (one round trip), and sixteen value rows; more heads keep half of that (registers)
    constexpr int NK = HG == 1 ? 16 : 8, NV = HG == 1 ? 16 : 8;
    float s[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) s[h] = 0.0f;
    if (live) {
      const uint4* row =
          reinterpret_cast<const uint4*>(tok == newest ? p.k_new + unit * D : wk + (int64_t)tok * D);
#pragma unroll
      for (int v0 = 0; v0 < D / 8; v0 += NK) {
        uint4 w[NK];
#pragma unroll
        for (int v = 0; v < NK; ++v) w[v] = __ldg(row + v0 + v);
#pragma unroll
        for (int v = 0; v < NK; ++v) {
          const uint32_t ws[4] = {w[v].x, w[v].y, w[v].z, w[v].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ws[i]));
            const int c = 8 * (v0 + v) + 2 * i;
#pragma unroll
            for (int h = 0; h < HG; ++h) s[h] = fmaf(qs[h][c], f.x, fmaf(qs[h][c + 1], f.y, s[h]));
          }
        }
      }
    }
    const int nt = min(32, p.n_w - 32 * stt);
    float m[HG], pw[HG], l[HG], a[HG][4];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      const float sc = live ? s[h] * p.qk_scale_log2 : -INFINITY;
      m[h] = sc;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m[h] = fmaxf(m[h], __shfl_xor_sync(kAll, m[h], off));
      pw[h] = live ? ex2_ftz(sc - m[h]) : 0.0f;
      l[h] = pw[h];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l[h] += __shfl_xor_sync(kAll, l[h], off);
#pragma unroll
      for (int i = 0; i < 4; ++i) a[h][i] = 0.0f;
    }
    // values: lane l owns channels 4l .. 4l+3 of every row; NV rows' loads in flight
    for (int j0 = 0; j0 < nt; j0 += NV) {
      uint2 w[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int r = 32 * stt + j0 + i;
        const uint16_t* vrow = r == newest ? p.v_new + unit * D : wv + (int64_t)r * D;
        w[i] = j0 + i < nt ? __ldg(reinterpret_cast<const uint2*>(vrow + 4 * lane)) : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&w[i].x));
        const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&w[i].y));
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float pj = __shfl_sync(kAll, pw[h], (j0 + i) & 31);  // 0 past nt: those lanes are not live
          a[h][0] = fmaf(pj, x01.x, a[h][0]);
          a[h][1] = fmaf(pj, x01.y, a[h][1]);
          a[h][2] = fmaf(pj, x23.x, a[h][2]);
          a[h][3] = fmaf(pj, x23.y, a[h][3]);
        }
      }
    }
    slot = __shfl_sync(kAll, slot, 0);
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      if (slot < p.max_slots) {
        const int64_t so = (bh0 + h) * p.max_slots + slot;
        *reinterpret_cast<float4*>(p.part_acc + so * D + 4 * lane) = make_float4(a[h][0], a[h][1], a[h][2], a[h][3]);
        if (lane == 0) *reinterpret_cast<float2*>(p.part_ml + so * 2) = make_float2(m[h], l[h]);
      }
    }
    if (newest >= 32 * stt && newest < 32 * stt + 32) {
      // store the appended token into its window slot: lanes 0-15 the key row, 16-31 the value row
      const uint16_t* src = lane < 16 ? p.k_new + unit * D : p.v_new + unit * D;
      uint16_t* dst = const_cast<uint16_t*>(lane < 16 ? wk : wv) + (int64_t)newest * D;
      reinterpret_cast<uint4*>(dst)[lane & 15] = __ldg(reinterpret_cast<const uint4*>(src) + (lane & 15));
    }
  };

  int64_t cur = -1;
  // for the current unit, relative to the slice's item index sx: the first item past the unit,
  // the unit's item of index 0 and the slice page of its first page (32-bit: a slice is small)
  int uend = 0, lofs = 0, kofs = 0;
  bool touched = false;  // the warp has state (page sub-tiles) for the current unit
  // sub-tiles taken at a time: two (of one page) when a page has an even number of them, which
  // halves the scheduling, page-wait and release work per sub-tile
  const int GR = (SPP & 1) ? 1 : 2;
  while (true) {
    int s = 0;
    if (lane == 0) s = atomicAdd(&next_sub, GR);
    s = __shfl_sync(kAll, s, 0);
    if (s >= n_sub || *(volatile int*)&abort_flag) break;
    const int sx = SPP == 4 ? s >> 2 : SPP == 2 ? s >> 1 : SPP == 1 ? s : s / 3;
    const int stt0 = s - sx * SPP;
    if (cur < 0 || sx >= uend) {
      if (cur >= 0 && touched) epilogue(cur);
      const int64_t x = w_begin + sx;
      cur = x / wpu;
      const int64_t ustart = cur * wpu;
      uend = (int)(ustart + wpu - w_begin);
      lofs = (int)(w_begin - ustart);
      kofs = (int)(cur * p.n_pages - hw - P_begin) + lofs;
      touched = false;
      reset();
      load_q(cur);
    }
    const int loc = sx + lofs;
    if (loc < hw) {
      for (int qq = 0; qq < GR; ++qq) {
        const int f = loc * SPP + stt0 + qq;  // sub-tile of the unit's fp16 rows
        if (32 * f < p.n_w) window_subtile(cur, f);
      }
      continue;
    }

    // ---------------- sub-tiles of a page: tokens 32*stt .. 32*stt+31 for stt = stt0 .. stt0+GR-1
    touched = true;
    const int kpg = sx + kofs;  // = cur * n_pages + (loc - hw) - P_begin
    const int kpg_lap = lap_of(kpg), stg = kpg - kpg_lap * n_stages;
    if (!wait_page(kpg)) {
      report_error(p.err, kDevWaitTimeout);
      atomicExch(&abort_flag, 1);
      break;
    }
    const uint8_t* pgm = stage_mem + (size_t)stg * page_bytes;
    const uint32_t* km = reinterpret_cast<const uint32_t*>(pgm + off_km);
    const uint32_t* vm = reinterpret_cast<const uint32_t*>(pgm + off_vm);
    for (int qq = 0; qq < GR; ++qq) {
    const int stt = stt0 + qq;
    const int gk = (32 * stt) >> log2G;  // key group

    // -- key B fragments: q'_h[c] 2^(sig - pos) split high/low, four channels per lane.  One
    //    exponent serves every head: |q_h[c] s_c| < 2^(eq+1) 2^(es+1) with eq the unit's largest |q|
    //    and es the group's largest step, so sig = 13 - eq - es keeps every |B| below 2^15.
    float zl;   // Z = sum_c q_h[c] z_c of head (lane >> 3) (HG = 4), (lane >> 4) (HG = 2) or the head
    float sgk;  // score = D * 2^(24 - sig)
    {
      const uint4 mz = *reinterpret_cast<const uint4*>(km + gk * D + 4 * lane);
      // (z, s) of channels 4*lane + i
      const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&mz.x));
      const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&mz.y));
      const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&mz.z));
      const float2 f3 = __half22float2(*reinterpret_cast<const __half2*>(&mz.w));
      // channel c = 4*lane + i = 16*kk + 8*hh + 2*tt + e
      const int kk = lane >> 2, hh = (lane >> 1) & 1;
      const int pk = PK::pos(2 * (kk % KPW) + hh);
      // steps are >= 0: the largest orders like its bit pattern
      const float smx = fmaxf(fmaxf(f0.y, f1.y), fmaxf(f2.y, f3.y));
      const uint32_t smxb = __reduce_max_sync(kAll, __float_as_uint(smx));
      const int esk = smxb != 0u ? (int)((smxb >> 23) & 0xFF) - 127 : 0;
      const int sig = 13 - eq - esk;  // fp16 exponents: within [-17, 61]
      sgk = pow2f(24 - sig);
      const float sscale = pow2f(sig - pk);
      const float2 ss01 = __fmul2_rn(make_float2(f0.y, f1.y), make_float2(sscale, sscale));
      const float2 ss23 = __fmul2_rn(make_float2(f2.y, f3.y), make_float2(sscale, sscale));
      const float2 z01 = make_float2(f0.x, f1.x), z23 = make_float2(f2.x, f3.x);
      const float mg = pow2f(27 - pk) * 1.5f;
      const float2 M = make_float2(mg, mg);
      float zp[HG];
      const int tt0 = 2 * (lane & 1);
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float4 q4 = *reinterpret_cast<const float4*>(&qs[h][4 * lane]);
        const float2 q01 = make_float2(q4.x, q4.y), q23 = make_float2(q4.z, q4.w);
        const float2 zq = __ffma2_rn(q23, z23, __fmul2_rn(q01, z01));
        zp[h] = zq.x + zq.y;
        uint32_t hi01, lo01, hi23, lo23;
        split_qs(q01, ss01, M, hi01, lo01);
        split_qs(q23, ss23, M, hi23, lo23);
        bk_s[warp][2 * h][tt0][2 * kk + hh] = hi01;
        bk_s[warp][2 * h][tt0 + 1][2 * kk + hh] = hi23;
        bk_s[warp][2 * h + 1][tt0][2 * kk + hh] = lo01;
        bk_s[warp][2 * h + 1][tt0 + 1][2 * kk + hh] = lo23;
      }
      // Z of every head summed over the lanes, transposed as it goes: each exchange hands the
      // partner the heads it keeps, so the warp ends with head (lane >> (5 - log2 HG)) on each lane
      if constexpr (HG == 4) {
        const bool b4 = lane & 16, b3 = lane & 8;
        const float k0 = (b4 ? zp[2] : zp[0]) + __shfl_xor_sync(kAll, b4 ? zp[0] : zp[2], 16);
        const float k1 = (b4 ? zp[3] : zp[1]) + __shfl_xor_sync(kAll, b4 ? zp[1] : zp[3], 16);
        zl = (b3 ? k1 : k0) + __shfl_xor_sync(kAll, b3 ? k0 : k1, 8);
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) zl += __shfl_xor_sync(kAll, zl, off);
      } else if constexpr (HG == 2) {
        const bool b4 = lane & 16;
        zl = (b4 ? zp[1] : zp[0]) + __shfl_xor_sync(kAll, b4 ? zp[0] : zp[1], 16);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) zl += __shfl_xor_sync(kAll, zl, off);
      } else {
        zl = zp[0];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) zl += __shfl_xor_sync(kAll, zl, off);
      }
    }
    __syncwarp();
    uint32_t bf[16];
    {
      // lanes of the unused B columns read a block of zeros: one path for every lane
      const uint4* src = reinterpret_cast<const uint4*>(g8 < KCOL ? &bk_s[warp][g8][t4][0] : &zero_frag[t4][0]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = src[i];
        bf[4 * i] = v.x;
        bf[4 * i + 1] = v.y;
        bf[4 * i + 2] = v.z;
        bf[4 * i + 3] = v.w;
      }
    }
    __syncwarp();  // bk_s is free for the next sub-tile

    // -- scores of the two 16-token tiles: lane (g8, t4 < HG) gets head t4 of tokens g8, g8 + 8.
    //    The two tiles' products are interleaved: two accumulator chains of eight products each
    //    (splitting each chain in two and adding the halves measured slower: the adds cost more
    //    than the latency they hide behind the other warps).
    float dsum[2][4];
    {
      uint32_t wd[2][2 * BK];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const uint4* wsrc =
            reinterpret_cast<const uint4*>(pgm + off_kc) + ((int64_t)(2 * stt + mt) * 32 + lane) * (2 * BK / 4);
#pragma unroll
        for (int i = 0; i < 2 * BK / 4; ++i) {
          const uint4 v = wsrc[i];
          wd[mt][4 * i] = v.x;
          wd[mt][4 * i + 1] = v.y;
          wd[mt][4 * i + 2] = v.z;
          wd[mt][4 * i + 3] = v.w;
        }
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dsum[mt][e] = 0.0f;
#pragma unroll
      for (int u = 0; u < BK; ++u) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const uint32_t X = wd[mt][u], Y = wd[mt][BK + u];
          const uint32_t Xs = X >> PK::SHIFT, Ys = Y >> PK::SHIFT;
#pragma unroll
          for (int jj = 0; jj < KPW; ++jj) {
            const int kk = u * KPW + jj;
            mma16816(dsum[mt], PK::get(X, Xs, 2 * jj), PK::get(Y, Ys, 2 * jj), PK::get(X, Xs, 2 * jj + 1),
                     PK::get(Y, Ys, 2 * jj + 1), bf[2 * kk], bf[2 * kk + 1]);
          }
        }
      }
    }
    float sc[2][2];
    // every lane computes (no branch); lanes past the heads take head 0 and are masked below
    const int hq = t4 < HG ? t4 : 0;
    // scores in log2 units: the softmax scale folded into the product's scale and into Z
    const float zz = (HG == 1 ? zl : __shfl_sync(kAll, zl, (32 / HG) * hq)) * p.qk_scale_log2;
    const float sgl = sgk * p.qk_scale_log2;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const float* d = dsum[mt];
      float s0 = -INFINITY, s1 = -INFINITY;
      {
        s0 = fmaf(d[0] + d[1], sgl, zz);
        s1 = fmaf(d[2] + d[3], sgl, zz);
        if (nsp > 0) {
          // sparse entries: the dense code there is 0 (value z); add q_c (x_c - z_c)
          const uint8_t* si = pgm + p.lay.off_si;
          const uint16_t* sv = reinterpret_cast<const uint16_t*>(pgm + p.lay.off_sv);
#pragma unroll
          for (int rh = 0; rh < 2; ++rh) {
            const int tok = 32 * stt + 16 * mt + g8 + 8 * rh;
            float add = 0.0f;
            for (int k = 0; k < p.nsp; ++k) {
              const int c = si[tok * p.nsp + k];
              const float xv = __half2float(__ushort_as_half(sv[tok * p.nsp + k]));
              const float z = __half2float(__ushort_as_half((uint16_t)(km[gk * D + c] & 0xFFFFu)));
              add = fmaf(qs[hq][c], xv - z, add);
            }
            if (rh == 0) s0 = fmaf(add, p.qk_scale_log2, s0);
            else s1 = fmaf(add, p.qk_scale_log2, s1);
          }
        }
        s0 = t4 < HG ? s0 : -INFINITY;
        s1 = t4 < HG ? s1 : -INFINITY;
      }
      sc[mt][0] = s0;
      sc[mt][1] = s1;
    }

    // -- online softmax (lazy maximum), per head over lanes t4 = head
    {
      const float tmax = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      const bool over = tmax > mrun + kLazy;  // masked lanes hold -inf
      if (__any_sync(kAll, over)) {
        float mx = tmax;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, off));
        mx = __shfl_sync(kAll, mx, (lane & ~3) | hmine);  // the maximum of this lane's head
        const float mnew = fmaxf(mx, mrun);
        const float f = ex2_ftz(mrun - mnew);  // 0 on the first sub-tile
        // the lane's D columns belong to heads hd0, hd1 (f of head h is on the lanes t4 = h)
        const float f0 = HG == 1 ? f : __shfl_sync(kAll, f, (lane & ~3) | hd0);
        const float f1 = HG == 1 ? f : __shfl_sync(kAll, f, (lane & ~3) | hd1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          dv[i][0] *= f0;
          dv[i][1] *= f1;
          dv[i][2] *= f0;
          dv[i][3] *= f1;
        }
        // lacc and zacc belong to head hcol
        const float fc = __shfl_sync(kAll, f, hcol);
        lacc *= fc;
#pragma unroll
        for (int i = 0; i < NBM; ++i) zacc[i] *= fc;
        mrun = mnew;
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) sc[mt][rh] = t4 < HG ? ex2_ftz(sc[mt][rh] - mrun) : 0.0f;
    }

    // -- values: scales and zero points of the lane's column groups for the 8 tokens it feeds
    //    (tokens 2t4, 2t4+1, 2t4+8, 2t4+9 of both 16-token tiles)
    float vs[2][NBM][4], vz[2][NBM][4];
    {
      float smax = 0.0f;
#pragma unroll
      for (int kc = 0; kc < 2; ++kc) {
        const int tb = 16 * (2 * stt + kc) + 2 * t4;
        if constexpr (STD && NBM == 2) {
          // groups 2*gl and 2*gl + 1 of a token: adjacent words
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tok = tb + (i & 1) + 8 * (i >> 1);
            const uint2 w = *reinterpret_cast<const uint2*>(vm + tok * 4 + 2 * gl);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
            vz[kc][0][i] = a.x;
            vs[kc][0][i] = a.y;
            vz[kc][1][i] = b.x;
            vs[kc][1][i] = b.y;
            smax = fmaxf(smax, fmaxf(a.y, b.y));
          }
        } else {
#pragma unroll
          for (int bi = 0; bi < NBM; ++bi) {
            const int grp = gl * NBM + bi;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int tok = tb + (i & 1) + 8 * (i >> 1);
              float2 zsv = make_float2(0.0f, 0.0f);
              if (grp < ng) zsv = __half22float2(*reinterpret_cast<const __half2*>(vm + tok * ng + grp));
              vz[kc][bi][i] = zsv.x;
              vs[kc][bi][i] = zsv.y;
              smax = fmaxf(smax, zsv.y);
            }
          }
        }
      }
      const uint32_t smaxb = __reduce_max_sync(kAll, __float_as_uint(smax));  // scales are >= 0
      const int enew = smaxb != 0u ? (int)((smaxb >> 23) & 0xFF) - 127 : -30;
      if (enew > es) {  // larger scales: lower the B scale, rescale what is accumulated (exact)
        const float f = pow2f(es - enew);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) dv[i][j] *= f;
        es = enew;
      }
    }
    const float bscale = pow2f(6 - es);  // p <= 2^8 and s < 2^(es+1): |B| < 2^15

    // -- values, one 16-token tile (k-chunk) at a time
#pragma unroll
    for (int kc = 0; kc < 2; ++kc) {
      const int tile = 2 * stt + kc;
      // p of head hcol for tokens 2t4, 2t4+1, 2t4+8, 2t4+9 of the tile
      const int la = 4 * (2 * t4) + hcol, lb = 4 * (2 * t4 + 1) + hcol;
      const float p0 = __shfl_sync(kAll, sc[kc][0], la), p1 = __shfl_sync(kAll, sc[kc][0], lb);
      const float p2 = __shfl_sync(kAll, sc[kc][1], la), p3 = __shfl_sync(kAll, sc[kc][1], lb);
      const float2 p01 = make_float2(p0, p1), p23 = make_float2(p2, p3);
      const float2 pb01 = __fmul2_rn(p01, make_float2(bscale, bscale)), pb23 = __fmul2_rn(p23, make_float2(bscale, bscale));
      uint32_t bv[NBM][2];
#pragma unroll
      for (int bi = 0; bi < NBM; ++bi) {
        const float2 b01 = __fmul2_rn(pb01, make_float2(vs[kc][bi][0], vs[kc][bi][1]));
        const float2 b23 = __fmul2_rn(pb23, make_float2(vs[kc][bi][2], vs[kc][bi][3]));
        bv[bi][0] = h2bits(__floats2half2_rn(b01.x, b01.y));
        bv[bi][1] = h2bits(__floats2half2_rn(b23.x, b23.y));
      }
      if constexpr (NBM == 2) {
        // both fragments' zero-point sums at once: (zacc[0], zacc[1]) += p_i (z of either group)
        float2 za = make_float2(zacc[0], zacc[1]);
        za = __ffma2_rn(make_float2(p3, p3), make_float2(vz[kc][0][3], vz[kc][1][3]), za);
        za = __ffma2_rn(make_float2(p2, p2), make_float2(vz[kc][0][2], vz[kc][1][2]), za);
        za = __ffma2_rn(make_float2(p1, p1), make_float2(vz[kc][0][1], vz[kc][1][1]), za);
        za = __ffma2_rn(make_float2(p0, p0), make_float2(vz[kc][0][0], vz[kc][1][0]), za);
        zacc[0] = za.x;
        zacc[1] = za.y;
      } else {
#pragma unroll
        for (int bi = 0; bi < NBM; ++bi)
          zacc[bi] = fmaf(p0, vz[kc][bi][0], fmaf(p1, vz[kc][bi][1], fmaf(p2, vz[kc][bi][2], fmaf(p3, vz[kc][bi][3], zacc[bi]))));
      }
      lacc += (p0 + p1) + (p2 + p3);  // read from the lanes of B column h (lane 4h)

      uint32_t wd[2 * BV];
      const uint4* wsrc = reinterpret_cast<const uint4*>(pgm + off_vc) + ((int64_t)tile * 32 + lane) * (2 * BV / 4);
#pragma unroll
      for (int i = 0; i < 2 * BV / 4; ++i) {
        const uint4 v = wsrc[i];
        wd[4 * i] = v.x;
        wd[4 * i + 1] = v.y;
        wd[4 * i + 2] = v.z;
        wd[4 * i + 3] = v.w;
      }
      uint32_t wsh[2 * BV];
#pragma unroll
      for (int i = 0; i < 2 * BV; ++i) wsh[i] = wd[i] >> PV::SHIFT;
#pragma unroll
      for (int mc = 0; mc < 8; ++mc) {
        const int u = mc / PV::PER, j = mc % PV::PER;
        constexpr int WPR = BV / 2;  // words per register slot
        uint32_t b0 = bv[0][0], b1 = bv[0][1];
        if constexpr (NBM > 1) {
          const int bi = ((16 * mc) >> log2G) % NBM;
#pragma unroll
          for (int i = 1; i < NBM; ++i)
            if (bi == i) {
              b0 = bv[i][0];
              b1 = bv[i][1];
            }
        }
        mma16816(dv[mc], PV::get(wd[0 * WPR + u], wsh[0 * WPR + u], j), PV::get(wd[1 * WPR + u], wsh[1 * WPR + u], j),
                 PV::get(wd[2 * WPR + u], wsh[2 * WPR + u], j), PV::get(wd[3 * WPR + u], wsh[3 * WPR + u], j), b0, b1);
      }
    }

    }  // sub-tiles of the grab

    // -- release the sub-tiles; the warp releasing a stage's last sub-tile refills it
    __syncwarp();
    if (lane == 0) {
      for (int qq = 0; qq < GR; ++qq) mbar_arrive(&empty_bar[stg]);
      if (atomicAdd(&stage_cnt[stg], GR) % SPP == SPP - GR && kpg + n_stages < n_pg && !*(volatile int*)&abort_flag) {
        if (mbar_wait(&empty_bar[stg], kpg_lap & 1, wlim)) {
          issue_page(kpg + n_stages);
        } else {
          report_error(p.err, kDevWaitTimeout);
          atomicExch(&abort_flag, 1);
        }
      }
    }
  }
  if (cur >= 0 && touched) epilogue(cur);
  __syncthreads();
  if (tid == 0) {
    for (int i = 0; i < n_stages; ++i)
      if (stage_issued[i] > 0) mbar_wait(&full_bar[i], (stage_issued[i] - 1) & 1);
  }
}

// Per-warp buffers in dynamic shared memory (bytes per CTA): query rows and key B fragments.
template <int HG>
constexpr size_t warp_bufs_bytes() {
  return (size_t)mma_warps<HG>() * (HG * kHeadDim * sizeof(float) + 2 * HG * 4 * 16 * sizeof(uint32_t));
}

// Page stages of one CTA: as many as fit (up to kMmaMaxStages) in the opt-in shared memory beside
// the static arrays and the per-warp buffers; -1 when fewer than two fit (or the static arrays
// exceed the 48 KB a kernel may declare).  Two at least: the ring's lap is a multiply-high by
// ceil(2^32 / n), which fits in 32 bits only for n >= 2 (pages of R <= 128 tokens leave room for
// seven or more).
template <int BK, int BV, int HG>
int stages_mma(int page_bytes) {
  auto kern = decode_mma_kernel<BK, BV, HG, false>;  // both variants declare the same static arrays
  static int static_smem = -1, optin = -1;
  if (static_smem < 0) {
    cudaFuncAttributes a{};
    int dev = 0;
    if (cudaFuncGetAttributes(&a, kern) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return -1;
    static_smem = (int)a.sharedSizeBytes;
  }
  if (static_smem > 48 * 1024) return -1;
  const int64_t avail = (int64_t)optin - static_smem - (int64_t)warp_bufs_bytes<HG>();
  const int64_t n = avail / page_bytes;
  return n < 2 ? -1 : (int)(n < kMmaMaxStages ? n : kMmaMaxStages);
}

template <int BK, int BV, int HG>
cudaError_t launch_mma_t(const DecodeParams& p, int grid, cudaStream_t s) {
  const int n = stages_mma<BK, BV, HG>(p.lay.bytes);
  if (n < 0) return cudaErrorInvalidValue;
  DecodeParams q = p;
  q.n_stages = n;
  q.stage_magic = (uint32_t)((0x100000000ull + (uint64_t)n - 1) / (uint64_t)n);  // ceil(2^32 / n)
  const size_t smem = (size_t)p.lay.bytes * n + warp_bufs_bytes<HG>();
  const bool std_shape = p.R == 128 && p.G == 32 && p.nsp == 0 && p.lay.bytes == StdPage<BK, BV>::bytes &&
                         p.lay.off_km == StdPage<BK, BV>::km && p.lay.off_vc == StdPage<BK, BV>::vc &&
                         p.lay.off_vm == StdPage<BK, BV>::vm && p.lay.off_kc == 0;
  auto kern = std_shape ? decode_mma_kernel<BK, BV, HG, true> : decode_mma_kernel<BK, BV, HG, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, (unsigned)grid, mma_warps<HG>() * 32, smem, s, q);
}

template <int BK, int BV, int HG>
int resident_mma_t(int page_bytes) {
  const int n = stages_mma<BK, BV, HG>(page_bytes);
  if (n < 0) return 0;
  const size_t smem = (size_t)page_bytes * n + warp_bufs_bytes<HG>();
  auto kern = decode_mma_kernel<BK, BV, HG, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
  if (cudaFuncSetAttribute(decode_mma_kernel<BK, BV, HG, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return 0;
  int n_ctas = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n_ctas, kern, mma_warps<HG>() * 32, smem) != cudaSuccess)
    return 0;
  return n_ctas;
}

}  // namespace

#define KVQ_MMA_CASES(X) X(2, 2, 1) X(2, 2, 2) X(2, 2, 4) X(4, 2, 1) X(4, 2, 2) X(4, 2, 4) X(4, 4, 1) X(4, 4, 2) X(4, 4, 4)

bool decode_mma_supported(int bk, int bv, int hg) {
#define KVQ_MS(BKV, BVV, HGV) \
  if (bk == BKV && bv == BVV && hg == HGV) return true;
  KVQ_MMA_CASES(KVQ_MS)
#undef KVQ_MS
  return false;
}

int decode_mma_resident(int bk, int bv, int hg, int page_bytes, int* warps) {
  *warps = hg == 4 ? mma_warps<4>() : mma_warps<1>();
#define KVQ_MR(BKV, BVV, HGV) \
  if (bk == BKV && bv == BVV && hg == HGV) return resident_mma_t<BKV, BVV, HGV>(page_bytes);
  KVQ_MMA_CASES(KVQ_MR)
#undef KVQ_MR
  return 0;
}

cudaError_t launch_decode_mma(const DecodeParams& p, int bk, int bv, int hg, int grid, cudaStream_t s) {
#define KVQ_ML(BKV, BVV, HGV) \
  if (bk == BKV && bv == BVV && hg == HGV) return launch_mma_t<BKV, BVV, HGV>(p, grid, s);
  KVQ_MMA_CASES(KVQ_ML)
#undef KVQ_ML
  return cudaErrorInvalidValue;
}

}  // namespace kvq
