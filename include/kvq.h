/*
 * kvq.h - asymmetric low-bit KV cache with quantized decode attention, C ABI.
 *
 * The library keeps one layer's KV cache for a batch of sequences on one GPU:
 *
 *  - Keys are quantized per channel: each group of G consecutive tokens of a
 *    channel shares one fp16 zero point and one fp16 scale ("KV cache has a
 *    geometry problem, not a bit problem", section "Keys"; KIVI summary page,
 *    section "Method").
 *  - Values are quantized per token: each group of G consecutive channels of a
 *    token shares one zero point and scale (same page, section "Values").
 *  - The quantizer is uniform and asymmetric: zero point = group minimum,
 *    step = range / (2^B - 1), every element rounds to the nearest step (same
 *    page, section "Quantization error in practice").  B is 2, 3 or 4 bits and
 *    may differ between keys and values, e.g. K4V2 ("Quantize What Counts:
 *    More for Keys, Less for Values").
 *  - The most recent tokens stay in an fp16 window of R tokens; a full window
 *    is quantized as one block (unite.ai page, section "System tax"; KIVI
 *    summary page, section "Method": buffer of 128 recent tokens).
 *  - Optionally keys are kept pre-RoPE and rotated after dequantization, and
 *    the largest-magnitude entries of each key vector are kept sparse in fp16
 *    outside the group ranges (KVQuant review, "Proposed method").
 *
 * Decode attention reads the whole cache every generated token, which makes
 * it bound by memory bandwidth (unite.ai page, section "Why the KV cache is a
 * problem").  kvq_decode_attention computes softmax(q.K^T * scale).V over all
 * cached tokens for every query head, reading the packed codes directly.
 *
 * Conventions for every call:
 *  - Return value: KVQ_OK (0) or a negative kvq_status.  No exception or
 *    longjmp crosses the ABI.  Argument, state and capacity errors are found
 *    on the host before anything is launched and leave the cache unchanged.
 *  - Device pointers are plain CUDA device addresses of the cache's device;
 *    `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *    asynchronous on that stream; the caller's buffers must stay valid until
 *    the stream has passed the call.  The cache state (token counts) is
 *    tracked on the host, so no call waits for the GPU except kvq_export_unit
 *    and kvq_sync_status.
 *  - Input device buffers must be 16-byte aligned and densely packed.
 *  - The cache owns all of its device memory; it is allocated once by
 *    kvq_create and freed by kvq_destroy.  The hot calls allocate nothing.
 *  - One cache must not be used from two host threads or two streams at
 *    once.  Different caches are independent.
 *  - A CUDA error inside a call (launch failure, or a device-side wait that
 *    ran out) makes the cache return KVQ_ERR_CUDA from then on.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned buffer, bad config value */
  KVQ_ERR_UNSUPPORTED = -2, /* a valid config outside what this build implements */
  KVQ_ERR_CAPACITY = -3,    /* more tokens than cfg.max_tokens */
  KVQ_ERR_STATE = -4,       /* call not allowed in the cache's current state */
  KVQ_ERR_CUDA = -5,        /* CUDA runtime error or device-side timeout (sticky) */
  KVQ_ERR_OOM = -6          /* device allocation failed in kvq_create */
} kvq_status;

typedef struct {
  int32_t batch;         /* B >= 1 sequences */
  int32_t num_kv_heads;  /* Hkv >= 1 */
  int32_t num_q_heads;   /* Hq, a multiple of Hkv; q head h reads kv head h / (Hq/Hkv) */
  int32_t head_dim;      /* D (this build: 128) */
  int64_t max_tokens;    /* capacity: tokens per sequence after all appends */
  int32_t k_bits;        /* bits per key code: 2, 3 or 4 */
  int32_t v_bits;        /* bits per value code: 2, 3 or 4 */
  int32_t group_size;    /* G: tokens per key group and channels per value group; 32 or 64, divides D and R */
  int32_t residual;      /* R: fp16 window length; a multiple of 32 and of G, at most 128 */
  int32_t k_sparse;      /* fp16 outliers kept per key vector, 0..4 (0 = dense keys) */
  int32_t rope;          /* 0: keys arrive already rotated; 1: keys arrive pre-RoPE and are rotated
                            after dequantization (rotate-half pairs (i, i+D/2), theta_i = base^(-2i/D),
                            position = absolute token index) */
  float rope_base;       /* RoPE base, e.g. 10000 (used when rope = 1) */
  float softmax_scale;   /* scale applied to q.k, e.g. 1/sqrt(D) */
  int32_t sink_tokens;   /* S, 0..R: the first S tokens of every sequence are kept fp16 (attention sinks)
                            and never quantized; 0 = no sinks.  unite.ai page and dothoosh.com page,
                            research-direction sections (InnerQ keeps high-precision windows for the
                            recent tokens and for the attention-sink tokens). */
  int32_t codebook;      /* 0: uniform levels (code c stands for z + c*s).  1: non-uniform levels (the
                            nuqX datatype of the KVQuant review, "Proposed method", without its
                            calibration): code c stands for z + lev[c]*s with per-cache key and value
                            levels set by kvq_set_codebooks before the first prefill or append;
                            rope = 0 with (k_bits, v_bits) in {(2,2), (3,3), (4,4), (4,2)} and 1 or 4
                            query heads per kv head, or rope = 1 with 3/3 bits and 4. */
} kvq_config;

typedef struct kvq_cache kvq_cache; /* opaque */

/*
 * Create an empty cache on CUDA device `device` and allocate all its device
 * memory: the packed pages for max_tokens tokens, the fp16 window and the
 * split-attention workspace.  On success *out receives the handle.
 * Errors: KVQ_ERR_INVALID_ARG (null, out-of-range field), KVQ_ERR_UNSUPPORTED,
 * KVQ_ERR_OOM, KVQ_ERR_CUDA.  On error *out is set to NULL.
 */
kvq_status kvq_create(const kvq_config* cfg, int device, kvq_cache** out);

/*
 * Device memory of the caches created from now on (process-wide; each cache keeps the functions
 * it was created with and frees through them).  alloc(bytes, device, user) returns device memory
 * of `device` aligned to 256 bytes, or NULL when it has none; free_fn(ptr, device, user) gives it
 * back.  For callers that manage GPU memory in a pool of their own.  Both NULL: cudaMalloc and
 * cudaFree (the default).  A cache allocates only in kvq_create and kvq_set_splits; when an
 * allocation fails, kvq_create frees what it had allocated and returns KVQ_ERR_OOM (a block that
 * is not 256-byte aligned is handed back and counts as KVQ_ERR_INVALID_ARG).  Not thread-safe
 * against a concurrent kvq_create.  KVQ_ERR_INVALID_ARG if exactly one of the two is NULL.
 * (The method pages have no counterpart.)
 */
typedef void* (*kvq_alloc_fn)(size_t bytes, int device, void* user);
typedef void (*kvq_free_fn)(void* ptr, int device, void* user);
kvq_status kvq_set_device_allocator(kvq_alloc_fn alloc, kvq_free_fn free_fn, void* user);

/* Free the cache and its device memory (synchronizes the device first).
   NULL is a no-op returning KVQ_OK. */
kvq_status kvq_destroy(kvq_cache* cache);

/*
 * Prefill: cache the prompt's keys and values, k and v device fp16
 * [B][Hkv][n_tokens][D], 1 <= n_tokens <= max_tokens.  The first
 * n_s = min(n_tokens, S) tokens are copied into the fp16 sink store (S =
 * sink_tokens, usually 0); of the T' = n_tokens - n_s tokens after them the
 * first Tq = R*floor((T'-1)/R) are quantized into packed pages (keys per
 * channel over G-token groups, values per token over G-channel groups, the
 * sparse outliers first when k_sparse > 0) and the last T' - Tq (1..R, or 0
 * when T' = 0) are copied into the fp16 window.  Allowed once, on an empty cache
 * (otherwise KVQ_ERR_STATE).  KIVI summary page, section "Method"; unite.ai
 * page, sections "Keys", "Values", "System tax".
 */
kvq_status kvq_prefill_quantize(kvq_cache* cache, const void* k_f16, const void* v_f16, int64_t n_tokens,
                                void* cuda_stream);

/*
 * Append one decode token: k and v device fp16 [B][Hkv][D].  While the sink
 * store holds fewer than S tokens the token goes there.  Otherwise, if the
 * window already holds R tokens it is first quantized as one block (the
 * flush), then the new token is stored in the window.  An append on an empty cache acts as
 * a prefill of one token.  KVQ_ERR_CAPACITY when the cache already holds
 * max_tokens tokens.  unite.ai page, section "System tax".
 */
kvq_status kvq_append(kvq_cache* cache, const void* k_f16, const void* v_f16, void* cuda_stream);

/*
 * Decode attention for one query token per sequence and head: q and out
 * device fp16 [B][Hq][D].  q arrives already rotated (post-RoPE at its own
 * position).  out[b][h] = softmax(scale * q[b][h] . K^T) . V over all T
 * cached tokens of sequence b and kv head h/(Hq/Hkv), where K and V are the
 * dequantized pages (z + s*code; sparse entries restored; keys rotated when
 * rope = 1) followed by the fp16 window.  Computed as split-K flash decoding
 * in fp32 (token ranges in parallel, online softmax, log-sum-exp merge), then
 * rounded to fp16.  KVQ_ERR_STATE on an empty cache.
 *
 * Outputs are not bitwise reproducible from launch to launch: the warps of a
 * launch take token ranges as they become free, and the partials are merged
 * in the order they finish, so fp32 sums are taken in a different order each
 * time and an fp16 output may differ by an ulp between two launches over the
 * same cache (about 0.5 % of the outputs of a full-size launch do).  Every
 * launch stays within the error bound against exact attention over the
 * dequantized cache.
 */
kvq_status kvq_decode_attention(kvq_cache* cache, const void* q_f16, void* out_f16, void* cuda_stream);

/*
 * One decode step of a layer in one call: kvq_append(k, v) followed by
 * kvq_decode_attention(q, out): the same cache state bit for bit, and the
 * same attention up to the launch-to-launch rounding differences described
 * for kvq_decode_attention.  The append's flush, when the window is full,
 * is its own launch; the new token is read by the attention launch straight
 * from k and v and stored into its window slot by that launch, so a step costs
 * one launch (two on a flush) instead of two (three).  Buffers as for
 * kvq_append and kvq_decode_attention; the same errors (KVQ_ERR_CAPACITY
 * before any work when the cache is full).  unite.ai page, section "System
 * tax": each generated token appends to the window, flushes a full window as
 * one block, and reads the whole cache.
 */
kvq_status kvq_decode_step(kvq_cache* cache, const void* k_f16, const void* v_f16, const void* q_f16, void* out_f16,
                           void* cuda_stream);

/*
 * Codebooks of a cache created with codebook = 1: k_levels[0 .. 2^k_bits) and v_levels[0 .. 2^v_bits),
 * host fp32 arrays (copied), the level of each code in quantization steps, strictly increasing from
 * lev[0] = 0 to lev[L] = L (L = 2^bits - 1), so a group's minimum and maximum stay exact.  A value
 * x of a group with zero point z and step s takes the code of the nearest level to
 * y = (x - z) / s (fp32 quotient): the number of thresholds fp32((lev[j] + lev[j+1]) * 0.5),
 * j < L, that y exceeds (a value on a threshold takes the lower level).  lev[c] = c is the
 * uniform quantizer except on exact ties.  Must run before the first prefill or append
 * (KVQ_ERR_STATE otherwise; those calls return KVQ_ERR_STATE until it has run); kvq_reset keeps
 * the codebooks.  KVQ_ERR_INVALID_ARG for a uniform cache or levels that break the rules above.
 */
kvq_status kvq_set_codebooks(kvq_cache* cache, const float* k_levels, const float* v_levels);

/*
 * Forget every cached token so the cache can take a new batch of sequences
 * (the next call may be a prefill).  Host-only: no device work, no memory
 * is freed or cleared; the pages are simply overwritten by later calls.
 */
kvq_status kvq_reset(kvq_cache* cache);

/*
 * Decode attention with no device allocation, over packed buffers the caller
 * owns.  (The method pages have no counterpart for this entry point.)
 *
 * For callers that cannot allocate device memory when they run attention --
 * an engine that carves all GPU memory from its own pool and does not let
 * libraries allocate, or a latency-critical path that must not enter the
 * allocator -- and that therefore keep the cache in their own buffers instead
 * of a kvq_cache.  It computes exactly what kvq_decode_attention computes for
 * a cache holding n_tokens tokens in the layout below; the split-attention
 * partials, which kvq_decode_attention keeps in each cache's workspace, live
 * in one 8 MiB file-scope device array inside the library instead (every GPU
 * that loads the library holds it until the process exits).
 *
 *   cfg            a configuration kvq_create would accept
 *   pages          device, [B*Hkv][pages_per_unit][page_bytes]; page p of a unit
 *                  holds tokens [p*R, p*R+R) as consecutive sections, each padded
 *                  to a multiple of 16 bytes: key codes (R*D*k_bits/32 u32), key
 *                  zero point/scale [R/G][D] u32 (fp16 zero point in the low half,
 *                  scale in the high half), value codes (R*D*v_bits/32 u32), value
 *                  zero point/scale [R][D/G] u32, sparse channels [R][k_sparse] u8,
 *                  sparse values [R][k_sparse] fp16.
 *                  Codes are token-major bitstreams [R][D*bits/32] (as in
 *                  kvq_unit_view) unless both widths are 2 or 4 bits and rope = 0;
 *                  then both code sections are in tensor-core fragment order: per
 *                  16-token tile m and lane l = 4g + t (g = l/4, t = l%4), 2B
 *                  consecutive words (word index (m*32 + l)*2B + w), each holding
 *                  16/B code pairs; pair j has its first code at bits [B*j, B*j+B)
 *                  and its second at bits [16+B*j, 16+B*j+B).  Keys: word
 *                  w = r*B + u, token 16m + g + 8r, channels c and c+1 with
 *                  c = 16*(u*(8/B) + j/2) + 8*(j%2) + 2t.  Values: word
 *                  w = r*(B/2) + u (r = 0..3), channel 16*(u*(16/B) + j) + g + 8*(r%2)
 *                  of tokens s and s+1 with s = 16m + 8*(r/2) + 2t.
 *   window_k/_v    device fp16 [B*Hkv][R][D]; slots 0..n_r-1 hold the newest tokens
 *   n_tokens       cached tokens T >= 1: Tq = R*floor((T-1)/R) are in the pages,
 *                  n_r = T - Tq in the window
 *   q_f16, out_f16 device fp16 [B][Hq][D]
 *
 * Errors: KVQ_ERR_INVALID_ARG (nulls, misalignment, Tq/R > pages_per_unit),
 * KVQ_ERR_UNSUPPORTED, and KVQ_ERR_CAPACITY when even the smallest launch's
 * partials do not fit the 8 MiB array: B*Hq*(D+2)*4 bytes per partial slot,
 * 3*W slots per query head for a one-CTA launch (W = warps of one decode CTA:
 * 16 on the tensor-core kernel, 8 to 16 on the CUDA-core kernel), plus one
 * counter per unit, after a fixed
 * head of 4.3 KB.  Larger sizes run on fewer CTAs than the GPU holds, as many
 * as the array allows.  KVQ_ERR_CAPACITY also refuses a ninth distinct
 * rope_base on one device (the array keeps the turn tables of eight).
 *
 * The device is the current one.  The first call on a device looks up the
 * array's address (a runtime symbol lookup) and clears its error word, and
 * the first call with rope = 1 and a given rope_base on a device writes that
 * base's turn table into the array with a synchronous copy; make those first
 * calls before any stream capture.  Later calls issue only a memset of the
 * counters and the two kernel launches.  The address is remembered for the
 * life of the process: after cudaDeviceReset (or anything else that destroys
 * the device's primary context) the remembered address is stale, so do not
 * call this function on that device again in the same process.
 *
 * Every call shares the one array: it clears the counters it needs at the
 * start of each call, but calls whose work overlaps on the GPU (different
 * streams, or several host threads) race on it.  A device-side wait that runs
 * out (see kvq_sync_status) is recorded in the array's error word; the call
 * has then returned KVQ_OK with an unusable output, and
 * kvq_noalloc_sync_status reports it.  Nothing is allocated and no allocator
 * is called.
 */
kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, const void* pages, int64_t pages_per_unit,
                                        const void* window_k, const void* window_v, int64_t n_tokens,
                                        const void* q_f16, void* out_f16, void* cuda_stream);

/*
 * Device-side status of kvq_decode_attention_noalloc on the current device: waits for
 * cuda_stream, then reads the scratch array's error word.  KVQ_OK if no call since the last
 * check recorded an error; otherwise KVQ_ERR_CUDA, and the word is cleared.  Also KVQ_ERR_CUDA
 * when the stream reports an error.  (The method pages have no counterpart.)
 */
kvq_status kvq_noalloc_sync_status(void* cuda_stream);

/*
 * Page layout of a configuration, for callers that build or size the packed
 * pages themselves (kvq_decode_attention_noalloc takes them in this layout).
 * Host arithmetic only: no CUDA call, no device needed.  One page holds R
 * tokens of one (batch, kv head) unit; its sections are those listed for
 * kvq_decode_attention_noalloc, in that order, each padded to a multiple of
 * 16 bytes; every offset is in bytes from the start of the page.
 *   page_bytes      bytes of one page (the stride of pages within a unit)
 *   kcodes_offset   key codes, R*D*k_bits/8 bytes
 *   kmeta_offset    key zero point / scale, [R/G][D] u32
 *   vcodes_offset   value codes, R*D*v_bits/8 bytes
 *   vmeta_offset    value zero point / scale, [R][D/G] u32
 *   sp_idx_offset   sparse key channels, [R][k_sparse] u8
 *   sp_val_offset   sparse key values, [R][k_sparse] fp16
 *   tokens_per_page R
 *   fragment_order  1: both code sections in tensor-core fragment order,
 *                   0: token-major bitstreams
 * Errors: KVQ_ERR_INVALID_ARG (null pointer, or a configuration kvq_create
 * refuses as invalid), KVQ_ERR_UNSUPPORTED (a valid configuration this build
 * does not implement).  kvq_create also checks the device's limits (shared
 * memory, resident CTAs), which this call, having no device, does not.
 */
typedef struct {
  int64_t page_bytes;
  int64_t kcodes_offset, kmeta_offset, vcodes_offset, vmeta_offset, sp_idx_offset, sp_val_offset;
  int32_t tokens_per_page;
  int32_t fragment_order;
} kvq_page_info;

kvq_status kvq_page_layout(const kvq_config* cfg, kvq_page_info* info);

/* ---------------- helpers (not on the hot path) ---------------- */

/* Host-tracked state: tokens cached, tokens quantized (Tq), tokens in the window. */
kvq_status kvq_get_state(const kvq_cache* cache, int64_t* t_total, int64_t* t_quant, int32_t* n_resid);

/*
 * Host view of one (batch, kv head) unit in the canonical layout.  Every
 * pointer is caller-allocated host memory of at least the byte size that
 * kvq_unit_sizes reports for the current state; a NULL pointer skips that
 * array.  Layouts (Tq = quantized tokens, n_r = window tokens):
 *   kcodes uint32 [Tq][D*k_bits/32]  codes of one token's D channels as a
 *                                     little-endian bitstream: code of channel
 *                                     c at bits [c*k_bits, c*k_bits + k_bits)
 *   kz, ks uint16 [Tq/G][D]          key zero point / scale (fp16 bits)
 *   vcodes uint32 [Tq][D*v_bits/32]  same bitstream layout for values
 *   vz, vs uint16 [Tq][D/G]          value zero point / scale
 *   sp_idx uint8  [Tq][k_sparse]     sparse key channels, ascending
 *   sp_val uint16 [Tq][k_sparse]     sparse key values (exact fp16)
 *   wk, wv uint16 [n_r][D]           fp16 window (tokens n_s+Tq .. n_s+Tq+n_r-1)
 */
typedef struct {
  void* kcodes; void* kz; void* ks;
  void* vcodes; void* vz; void* vs;
  void* sp_idx; void* sp_val;
  void* wk; void* wv;
  int64_t kcodes_bytes, kmeta_bytes, vcodes_bytes, vmeta_bytes, sp_idx_bytes, sp_val_bytes, window_bytes;
  void* sk; void* sv;    /* sink tokens uint16 [n_s][D] (fp16 bits), n_s = T - Tq - n_r */
  int64_t sink_bytes;
} kvq_unit_view;

/* Fill the *_bytes fields of `sizes` for the current state (pointers untouched). */
kvq_status kvq_unit_sizes(const kvq_cache* cache, kvq_unit_view* sizes);

/*
 * Copy unit (b, kvh) to the host in the canonical layout; waits for `stream` (synchronous).  This
 * is the cache export in per-unit form: a caller exports the whole cache by calling it for every
 * (b, kvh), with host buffers sized by kvq_unit_sizes.  Pages stored in fragment order are converted
 * back to the canonical bitstreams above, so the export is the same for every page layout.
 */
kvq_status kvq_export_unit(kvq_cache* cache, int32_t b, int32_t kvh, kvq_unit_view* dst, void* cuda_stream);

/*
 * Decode work partition.  Decode attention runs as one persistent launch whose
 * CTAs take equal contiguous slices of the list of all units' pages (plus one
 * window item per unit); by default the grid is the number of CTAs the GPU
 * keeps resident.  kvq_set_splits(n) with n > 0 forces a grid of n CTAs per
 * (batch, kv head) unit instead (clamped to 16; 0 restores the default) -- a
 * test and tuning aid that changes where units are cut, not the result
 * beyond rounding.  kvq_get_splits reports the CTAs per unit (rounded up) of
 * the next decode.
 */
kvq_status kvq_set_splits(kvq_cache* cache, int32_t splits);
kvq_status kvq_get_splits(const kvq_cache* cache, int32_t* splits);

/*
 * Wait for `stream`, then report the cache's device-side status: KVQ_OK, or
 * KVQ_ERR_CUDA if a kernel recorded a failed bounded wait or CUDA reports an
 * error.  Every device-side wait in the kernels gives up after a time limit
 * and records an error code instead of hanging.
 */
kvq_status kvq_sync_status(kvq_cache* cache, void* cuda_stream);

/*
 * Test hook for the device-side time limits (not for production use).  Every wait of the decode
 * kernels -- for a page copy to land, for a stage to be released -- gives up after a time limit
 * (2 s by default), records an error in the cache's error word and lets the kernel finish without
 * leaving copies in flight; kvq_sync_status then reports KVQ_ERR_CUDA.  This hook makes that path
 * testable without a fault: for the decode launches that follow, wait_limit_ns > 0 replaces the
 * default limit, and withhold_page = k >= 0 leaves page k of every CTA's slice of the work list
 * uncopied, so the warps that reach it wait until the limit runs out.  (-1, 0) restores normal
 * operation.  Outputs of affected launches are not meaningful.  KVQ_ERR_INVALID_ARG for
 * withhold_page < -1 or wait_limit_ns < 0.  (The method pages have no counterpart.)
 */
kvq_status kvq_test_inject(kvq_cache* cache, int32_t withhold_page, int64_t wait_limit_ns);

/*
 * Debug builds only (the library compiled with KVQ_DEBUG_CHECKS, e.g. bit_asymmetric_kv_kvq_gb300/_build.py
 * --debug): waits for the device, then checks the cache's error word -- where the kernels' bounds
 * checks of debug builds and the time limits of every build record -- and the canary bytes that
 * follow each of the cache's device buffers in debug builds.  KVQ_OK when all are intact,
 * KVQ_ERR_CUDA otherwise; KVQ_ERR_UNSUPPORTED in a normal build.  A stand-in for a device memory
 * checker.  (The method pages have no counterpart.)
 */
kvq_status kvq_debug_check(kvq_cache* cache);

/* Kernel launches issued by this cache since creation (decode, append, flush...). */
int64_t kvq_launch_count(const kvq_cache* cache);

/* Static text for a status code. */
const char* kvq_status_string(kvq_status status);

/* Library version, (major << 16) | minor. */
int32_t kvq_version(void);

/* ---------------- axis ablation (analysis beside the cache, not the cache) ----------------
 *
 * The comparison at the centre of "KV cache has a geometry problem, not a bit problem"
 * (sections "Keys" and "Values"; restated on the dothoosh.com page): quantize keys or values
 * with groups along either axis and measure what that does to attention scores and outputs.
 * These calls run on device buffers the caller owns; nothing is allocated.  Errors are detected
 * on the host before any launch (KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED); KVQ_ERR_CUDA if the
 * launch fails.  All are asynchronous on cuda_stream.
 */
#define KVQ_AXIS_TOKENS 0   /* groups of G tokens of one channel ("per-channel"; the cache's keys) */
#define KVQ_AXIS_CHANNELS 1 /* groups of G channels of one token ("per-token"; the cache's values) */

/*
 * Quantize x, device fp16 [n_units][n_tokens][head_dim] (8-byte aligned), with the cache's group
 * quantizer (zero point = group minimum, step = range / (2^bits - 1), round to nearest; unite.ai
 * page, section "Quantization error in practice") along `axis`.  Outputs, device:
 * codes_u8 uint8 [n_units][n_tokens][head_dim] (4-byte aligned), one code per byte;
 * zero_f16 and scale_f16 fp16 bits, [n_units][n_tokens/G][head_dim] for KVQ_AXIS_TOKENS
 * (n_tokens a multiple of G, n_units <= 65535) or [n_units][n_tokens][head_dim/G] for
 * KVQ_AXIS_CHANNELS.  bits 2..4; group_size 32 or 64; head_dim 128.
 */
kvq_status kvq_axis_quantize(const void* x_f16, int64_t n_units, int64_t n_tokens, int32_t head_dim, int32_t bits,
                             int32_t group_size, int32_t axis, void* codes_u8, void* zero_f16, void* scale_f16,
                             void* cuda_stream);

/* z + s*code (one rounding) for the output of kvq_axis_quantize: out_f32 device fp32
   [n_units][n_tokens][head_dim], 16-byte aligned. */
kvq_status kvq_axis_dequantize(const void* codes_u8, const void* zero_f16, const void* scale_f16, int64_t n_units,
                               int64_t n_tokens, int32_t head_dim, int32_t group_size, int32_t axis, void* out_f32,
                               void* cuda_stream);

/*
 * Exact decode attention (fp32 arithmetic) of heads_per_unit (1, 2 or 4) query heads per unit:
 * q_f16 device fp16 [n_units][heads_per_unit][head_dim]; k and v device [n_units][n_tokens][head_dim],
 * fp32 when kv_f32 = 1 (16-byte aligned), fp16 when kv_f32 = 0 (8-byte aligned).  out_f32 device
 * fp32 [n_units][heads_per_unit][head_dim] = softmax(softmax_scale * q.K^T) V; scores_f32, if not
 * NULL, receives softmax_scale * q.k per [n_units][heads_per_unit][n_tokens].
 */
kvq_status kvq_axis_attention(const void* k, const void* v, int32_t kv_f32, const void* q_f16, int64_t n_units,
                              int32_t heads_per_unit, int64_t n_tokens, int32_t head_dim, float softmax_scale,
                              void* scores_f32, void* out_f32, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
