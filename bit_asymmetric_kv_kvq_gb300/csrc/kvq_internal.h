// Internal declarations shared by the library's translation units.
//
// Device layout of one (batch, kv-head) unit:
//   pages  : [n_pages_cap][page_bytes]; page p holds the R quantized tokens
//            [p*R, p*R + R) as five 16-byte aligned sections
//              kc  key codes    [R][D*BK/32] u32  (token-major channel bitstream)
//              km  key meta     [R/G][D] u32      (fp16 zero point in the low half, scale in the high half)
//              vc  value codes  [R][D*BV/32] u32
//              vm  value meta   [R][D/G] u32      (zero point low, scale high)
//              si  sparse idx   [R][NSP] u8       (padded to 16 bytes)
//              sv  sparse vals  [R][NSP] fp16     (padded to 16 bytes)
//   window : K and V fp16 [R][D] each (the recent, not yet quantized tokens).
// A page is one flush unit, so a flush writes exactly one page and a decode
// split streams whole pages with one bulk copy each.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "kvq.h"

namespace kvq {

constexpr int kHeadDim = 128;

struct PageLayout {
  int32_t off_kc, off_km, off_vc, off_vm, off_si, off_sv, bytes;
  int32_t frag;  // 1: key and value codes in tensor-core fragment order (see below), 0: bitstreams
};

// Fragment order is used when both code widths are 2 or 4 bits and keys are stored after
// RoPE (no rotation at decode); otherwise codes are token-major bitstreams.
PageLayout make_layout(int R, int D, int G, int bk, int bv, int nsp, bool rope, bool codebook = false);

// Fragment order of the codes of a page (D = 128, B = 2 or 4 bits).  Both sections are cut
// into 16-token tiles; in each tile every lane l = 4g + t (g = l / 4, t = l % 4) of a warp
// owns 2B consecutive 32-bit words (word index (tile*32 + l)*2B + w).  A word holds 16/B code
// pairs; pair j keeps its first code at bits [B*j, B*j + B) and its second at bits
// [16 + B*j, 16 + B*j + B), so masking a pair in place leaves two fp16 subnormals
// code * 2^(B*j) * 2^-24 (pairs j >= 10/B are first shifted down by B*(10/B) bits).
//
// Keys, tile = tokens 16m .. 16m+15: word w = r*B + u holds token 16m + g + 8r; its pair j
// covers channels c and c + 1 with c = 16*(u*(8/B) + j/2) + 8*(j%2) + 2t.
__host__ __device__ inline void frag_key_pair(int bits, int tile, int lane, int w, int j, int* token, int* c0) {
  const int g = lane >> 2, t = lane & 3;
  const int r = w / bits, u = w % bits;
  *token = 16 * tile + g + 8 * r;
  *c0 = 16 * (u * (8 / bits) + j / 2) + 8 * (j % 2) + 2 * t;
}
// Values, tile = tokens 16k .. 16k+15: word w = r*(B/2) + u, r = 0..3; its pair j covers
// channel 16*(u*(16/B) + j) + g + 8*(r%2) of tokens s and s + 1, s = 16k + 8*(r/2) + 2t.
__host__ __device__ inline void frag_value_pair(int bits, int tile, int lane, int w, int j, int* tok0, int* ch) {
  const int g = lane >> 2, t = lane & 3;
  const int r = w / (bits / 2), u = w % (bits / 2);
  *ch = 16 * (u * (16 / bits) + j) + g + 8 * (r % 2);
  *tok0 = 16 * tile + 8 * (r / 2) + 2 * t;
}

// The common page shape -- R = 128 tokens, D = 128, G = 32, no sparse entries -- as compile-time
// offsets (the layout make_layout gives it).  The page and decode kernels have variants compiled
// for it (chosen at launch when a cache's layout matches), in which the page addressing folds.
template <int BK, int BV>
struct StdPage {
  static constexpr int kc = 0;
  static constexpr int km = 128 * 128 * BK / 8;
  static constexpr int vc = km + (128 / 32) * 128 * 4;
  static constexpr int vm = vc + 128 * 128 * BV / 8;
  static constexpr int bytes = vm + 128 * (128 / 32) * 4;
};

// Host-side validation of a configuration (the checks kvq_create applies).
kvq_status check_config(const kvq_config& cfg);

// theta_i / (2 pi) as 0.64 fixed-point turns, theta_i = base^(-2i/D), i < D/2.
void rope_table(double base, int D, unsigned long long* out);

// Device error codes written by kernels into the cache's error word.
enum DeviceError : int {
  kDevOk = 0,
  kDevWaitTimeout = 1,    // an mbarrier wait gave up
  kDevBadArgument = 2,    // a kernel saw parameters it cannot handle
  kDevBounds = 3,         // debug builds: an access fell outside its buffer (and was skipped)
};

struct QuantizeParams {
  const uint16_t* k_src;     // fp16 bits; token t of unit u at k_src + u*src_unit_stride + t*D
  const uint16_t* v_src;
  int64_t src_unit_stride;   // elements
  int64_t src_tok0;          // source token of the first page of this launch
  uint8_t* pages;            // base of all units' pages
  int64_t unit_page_stride;  // bytes between units
  int64_t page0;             // index of the first page written by this launch
  int32_t n_units, Hkv, D, G, R, nsp;
  PageLayout lay;
  int* err;
  int64_t src_elems;         // extent of k_src and v_src (elements) and of the pages (bytes):
  int64_t pages_bytes;       //   the bounds checks of debug builds
  int32_t lut;               // 1: codes are codebook indices chosen by the thresholds below
  float k_thr[16];           // decision thresholds between consecutive key / value levels
  float v_thr[16];
};

struct CopyTokensParams {
  const uint16_t* k_src;
  const uint16_t* v_src;
  int64_t src_unit_stride;  // elements
  int64_t src_tok0;
  uint16_t* k_dst;          // window base
  uint16_t* v_dst;
  int64_t dst_unit_stride;  // elements
  int64_t dst_tok0;
  int32_t n_tok, n_units, D;
};

struct DecodeParams {
  const uint16_t* q;        // [B][Hq][D] fp16 bits
  const uint8_t* pages;
  int64_t unit_page_stride;
  const uint16_t* wk;       // fp16 rows [units][S + R][D]: the sink rows, then the window rows
  const uint16_t* wv;       //   (rows 0 .. n_w are contiguous: the window fills only after the sink)
  int64_t win_unit_stride;  // elements
  const uint16_t* k_new;    // null, or [B*Hkv][D] fp16: the window's newest token (slot n_r - 1),
  const uint16_t* v_new;    //   read from here and stored into the window by the decode kernel
  int64_t n_units;          // B * Hkv
  int64_t n_pages;          // quantized pages per unit (Tq / R)
  int32_t work_per_unit;    // ceil(n_w / R) fp16 items, then the n_pages page items
  int32_t n_r;              // window tokens
  int32_t n_s;              // sink tokens; positions: sink 0..n_s, pages n_s.., window n_s + Tq..
  int32_t n_w;              // fp16 rows n_s + n_r: the sink rows, then the window rows
  int32_t max_slots;        // partial slots per query head
  int32_t log2_stages;      // page stages per CTA (set by the launcher; CUDA-core kernels)
  int32_t n_stages;         // page stages per CTA of the tensor-core kernel (any count up to 16)
  uint32_t stage_magic;     //   and ceil(2^32 / n_stages): k / n_stages = umulhi(k, stage_magic)
  int32_t Hkv, Hq, D, G, R, nsp;
  int32_t log2G;            // G = 1 << log2G
  PageLayout lay;
  float qk_scale_log2;      // softmax_scale * log2(e)
  const unsigned long long* rope_turns;  // [D/2] theta_i / (2*pi) as 0.64 fixed point (rope only)
  float* part_ml;           // [B*Hq][max_slots][2]  (running max in log2 units, sum)
  float* part_acc;          // [B*Hq][max_slots][D]
  int* nslot;               // [B*Hkv] partial slots taken per unit, zero between calls (the
                            //   merge kernel clears them)
  uint16_t* out;            // [B][Hq][D] fp16 bits
  int* err;
  int32_t lut;              // 1: codebook cache (the CUDA-core kernel with level lookups)
  float k_lev[16];          // codebook caches: the level (in steps) of each key / value code
  float v_lev[16];
  // test hooks (zero in normal use): a limit for the page and stage waits in place of the default
  // kWaitLimitNs, and k + 1 to leave page k of every CTA's slice uncopied (its waits then run out)
  unsigned long long wait_ns;
  int32_t test_withhold;
  int64_t pages_bytes;      // extent of the pages (the bounds checks of debug builds)
};

// Launchers (return cudaGetLastError() after the launch).
cudaError_t launch_quantize(const QuantizeParams& p, int bk, int bv, int n_pages, cudaStream_t s);
cudaError_t launch_copy_tokens(const CopyTokensParams& p, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, int bk, int bv, int hg, bool rope, int grid, cudaStream_t s,
                          bool* supported);
// Decode CTAs resident per SM (0: unsupported), and in *warps the warps of one CTA: the partial
// slots a unit needs are warps * (CTAs whose slices meet the unit).
int decode_resident_ctas_per_sm(int bk, int bv, int hg, bool rope, int R, int nsp, int page_bytes, int* warps,
                                bool codebook = false);
// Tensor-core decode over fragment-ordered pages (2/4-bit codes, keys without RoPE).
bool decode_mma_supported(int bk, int bv, int hg);
int decode_mma_resident(int bk, int bv, int hg, int page_bytes, int* warps);
cudaError_t launch_decode_mma(const DecodeParams& p, int bk, int bv, int hg, int grid, cudaStream_t s);
// CUDA-core decode of codebook caches (kvq_decode_lut.cu).
bool decode_lut_supported(int bk, int bv, int hg, bool rope);
int decode_lut_resident(int bk, int bv, int hg, bool rope, int page_bytes, int* warps);
cudaError_t launch_decode_lut(const DecodeParams& p, int bk, int bv, int hg, bool rope, int grid, cudaStream_t s);
bool decode_supported(int bk, int bv, int hg, bool rope, bool codebook = false);
bool quantize_supported(int bk, int bv);
size_t quantize_smem_bytes(int R, int D, int G, const PageLayout& lay);

}  // namespace kvq
