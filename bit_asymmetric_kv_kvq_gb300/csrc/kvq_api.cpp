// Host side of the C ABI declared in include/kvq.h: the cache handle, the
// cache state machine, argument checks and kernel launches.
//
// State machine (unite.ai page, section "System tax"; KIVI summary page,
// section "Method"): the most recent tokens stay in an fp16 window of R
// tokens; an append that finds the window full first quantizes those R tokens
// as one page (the flush) and then stores the new token.  So for T >= 1
// cached tokens the window holds n_r in [1, R] tokens and Tq = R*floor((T-1)/R)
// tokens are quantized.  All counts live on the host: no call reads the GPU.
//
// Attention sinks (unite.ai page and dothoosh.com page, research-direction sections: InnerQ keeps
// the attention-sink tokens in high precision as well as the recent ones): with sink_tokens = S
// the first n_s = min(T, S) tokens are stored fp16 and never quantized; the window/flush machine
// above runs on the tokens after them, so Tq = R*floor((T-n_s-1)/R).  Each unit keeps its fp16
// rows in one buffer of S + R rows: the sink rows 0 .. n_s, then the window rows S .. S + n_r.  The
// window fills only once the sink is full, so the rows in use are always 0 .. n_s + n_r.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

// Device memory of a cache: the caller's allocator (kvq_set_device_allocator) or cudaMalloc.
struct DeviceAllocator {
  kvq_alloc_fn alloc = nullptr;
  kvq_free_fn free = nullptr;
  void* user = nullptr;
};
std::mutex g_alloc_mutex;
DeviceAllocator g_alloc;

#ifdef KVQ_DEBUG_CHECKS
// Debug builds put a canary of this many bytes after every device buffer of a cache and check it
// in kvq_debug_check (a stand-in for a memory checker).
constexpr size_t kCanaryBytes = 256;
constexpr unsigned char kCanaryByte = 0xA5;
#endif

}  // namespace

struct kvq_cache {
  kvq_config cfg;
  DeviceAllocator alloc;
#ifdef KVQ_DEBUG_CHECKS
  std::vector<std::pair<unsigned char*, size_t>> canaries;  // (buffer, bytes in use): a canary follows each
#endif
  int device = 0;
  int sm_count = 0;
  kvq::PageLayout lay{};
  int64_t n_units = 0;        // B * Hkv
  int64_t n_pages_cap = 0;    // pages per unit
  int64_t unit_page_stride = 0;
  uint8_t* pages = nullptr;
  uint16_t* wk = nullptr;     // fp16 rows [units][S + R][D]: sink rows, then window rows
  uint16_t* wv = nullptr;
  float* part_ml = nullptr;
  float* part_acc = nullptr;
  int* counters = nullptr;
  int* err = nullptr;
  unsigned long long* rope_turns = nullptr;
  int32_t max_slots = 1;      // partial slots per query head
  int32_t forced_splits = 0;  // 0: grid = resident CTAs; n: grid = n CTAs per unit
  int64_t resident = 1;       // decode CTAs resident on the whole GPU
  int32_t decode_warps = 1;   // warps of one decode CTA
  int64_t T = 0, Tq = 0;
  int32_t n_r = 0;
  int32_t n_s = 0;            // sink tokens held (<= S)
  bool lut_set = false;       // codebook caches: kvq_set_codebooks has run
  float k_lev[16] = {}, v_lev[16] = {};  // codebook levels (in steps) and the decision thresholds
  float k_thr[16] = {}, v_thr[16] = {};  //   between consecutive levels
  bool prefilled = false;
  bool broken = false;
  int64_t launches = 0;
  unsigned long long test_wait_ns = 0;  // test hooks (kvq_test_inject)
  int32_t test_withhold = 0;
};

namespace {

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvq_status fail_cuda(kvq_cache* c) {
  c->broken = true;
  return KVQ_ERR_CUDA;
}

int64_t quantized_tokens(int64_t T, int R) { return T <= 0 ? 0 : (int64_t)R * ((T - 1) / R); }

// One device buffer of the cache, through its allocator (debug builds add a canary after it).
cudaError_t dev_alloc(kvq_cache* c, void** p, size_t bytes) {
  *p = nullptr;
  if (bytes < 16) bytes = 16;
#ifdef KVQ_DEBUG_CHECKS
  const size_t total = bytes + kCanaryBytes;
#else
  const size_t total = bytes;
#endif
  if (c->alloc.alloc) {
    void* q = c->alloc.alloc(total, c->device, c->alloc.user);
    if (!q) return cudaErrorMemoryAllocation;
    if (reinterpret_cast<uintptr_t>(q) & 255u) {
      c->alloc.free(q, c->device, c->alloc.user);
      return cudaErrorInvalidValue;
    }
    *p = q;
  } else {
    const cudaError_t e = cudaMalloc(p, total);
    if (e != cudaSuccess) {
      *p = nullptr;
      return e;
    }
  }
#ifdef KVQ_DEBUG_CHECKS
  const cudaError_t e = cudaMemset(static_cast<unsigned char*>(*p) + bytes, kCanaryByte, kCanaryBytes);
  if (e != cudaSuccess) return e;
  c->canaries.push_back({static_cast<unsigned char*>(*p), bytes});
#endif
  return cudaSuccess;
}

void dev_free(kvq_cache* c, void* p) {
  if (!p) return;
#ifdef KVQ_DEBUG_CHECKS
  for (size_t i = 0; i < c->canaries.size(); ++i)
    if (c->canaries[i].first == p) {
      c->canaries.erase(c->canaries.begin() + (long)i);
      break;
    }
#endif
  if (c->alloc.free) c->alloc.free(p, c->device, c->alloc.user);
  else cudaFree(p);
}

void free_all(kvq_cache* c) {
  dev_free(c, c->pages);
  dev_free(c, c->wk);
  dev_free(c, c->wv);
  dev_free(c, c->part_ml);
  dev_free(c, c->part_acc);
  dev_free(c, c->counters);
  dev_free(c, c->err);
  dev_free(c, c->rope_turns);
  c->pages = nullptr;
  c->wk = c->wv = nullptr;
  c->part_ml = c->part_acc = nullptr;
  c->err = nullptr;
  c->counters = nullptr;
  c->rope_turns = nullptr;
}

kvq_status validate(const kvq_config& k) {
  if (k.batch < 1 || k.num_kv_heads < 1 || k.num_q_heads < 1 || k.head_dim < 1 || k.max_tokens < 1)
    return KVQ_ERR_INVALID_ARG;
  if (k.num_q_heads % k.num_kv_heads) return KVQ_ERR_INVALID_ARG;
  if (k.k_bits < 2 || k.k_bits > 4 || k.v_bits < 2 || k.v_bits > 4) return KVQ_ERR_INVALID_ARG;
  if (k.group_size < 1 || k.residual < 1 || k.k_sparse < 0 || (k.rope != 0 && k.rope != 1))
    return KVQ_ERR_INVALID_ARG;
  if (k.head_dim % k.group_size || k.residual % k.group_size) return KVQ_ERR_INVALID_ARG;
  if (!(k.softmax_scale > 0.0f) || !std::isfinite(k.softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if (k.rope && (!(k.rope_base > 1.0f) || !std::isfinite(k.rope_base))) return KVQ_ERR_INVALID_ARG;
  if (k.k_sparse > k.head_dim || k.sink_tokens < 0) return KVQ_ERR_INVALID_ARG;
  if (k.codebook != 0 && k.codebook != 1) return KVQ_ERR_INVALID_ARG;
  // what this build implements
  if (k.head_dim != kvq::kHeadDim) return KVQ_ERR_UNSUPPORTED;
  if (k.group_size != 32 && k.group_size != 64) return KVQ_ERR_UNSUPPORTED;
  if (k.residual % 32 || k.residual > 128) return KVQ_ERR_UNSUPPORTED;
  if (k.k_sparse > 4) return KVQ_ERR_UNSUPPORTED;
  if (k.sink_tokens > k.residual) return KVQ_ERR_UNSUPPORTED;
  if ((int64_t)k.batch * k.num_q_heads > (int64_t)1 << 30) return KVQ_ERR_UNSUPPORTED;
  if (k.max_tokens >= ((int64_t)1 << 31)) return KVQ_ERR_UNSUPPORTED;
  const int hg = k.num_q_heads / k.num_kv_heads;
  if (!kvq::decode_supported(k.k_bits, k.v_bits, hg, k.rope != 0, k.codebook != 0)) return KVQ_ERR_UNSUPPORTED;
  if (!kvq::quantize_supported(k.k_bits, k.v_bits)) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

constexpr int32_t kMaxForcedSplits = 16;

// Grid of the decode launch: the resident CTAs (one per SM), or n per unit when forced; never
// more CTAs than work items.
int64_t rows_per_unit(const kvq_cache* c) { return (int64_t)c->cfg.sink_tokens + c->cfg.residual; }

int64_t fp16_items(const kvq_cache* c) { return (c->n_s + c->n_r + c->cfg.residual - 1) / c->cfg.residual; }

int64_t decode_grid(const kvq_cache* c) {
  const int64_t wpu = c->Tq / c->cfg.residual + fp16_items(c);
  const int64_t total = c->n_units * wpu;
  int64_t g = c->forced_splits > 0 ? c->n_units * c->forced_splits : c->resident;
  if (g > total) g = total;
  return g < 1 ? 1 : g;
}

// Partial slots one query head needs for a grid of `grid` CTAs: every warp of every CTA whose
// slice meets the unit may leave one, and fewer than ceil(grid / units) + 2 slices meet a unit.
int64_t slots_for_grid(const kvq_cache* c, int64_t grid) {
  return (int64_t)c->decode_warps * ((grid + c->n_units - 1) / c->n_units + 2);
}

// Grow the partial buffers to `slots` per query head (never shrinks).
cudaError_t ensure_slots(kvq_cache* c, int64_t slots) {
  if (slots <= c->max_slots) return cudaSuccess;
  const int64_t heads = (int64_t)c->cfg.batch * c->cfg.num_q_heads;
  float *ml = nullptr, *acc = nullptr;
  cudaError_t e = dev_alloc(c, (void**)&ml, (size_t)(heads * slots * 2 * sizeof(float)));
  if (e == cudaSuccess) e = dev_alloc(c, (void**)&acc, (size_t)(heads * slots * c->cfg.head_dim * sizeof(float)));
  if (e != cudaSuccess) {
    dev_free(c, ml);
    dev_free(c, acc);
    return e;
  }
  // the buffers may still be read by work in flight on any stream
  cudaDeviceSynchronize();
  dev_free(c, c->part_ml);
  dev_free(c, c->part_acc);
  c->part_ml = ml;
  c->part_acc = acc;
  c->max_slots = (int32_t)slots;
  return cudaSuccess;
}

// 0.64 fixed-point turns per token of frequency i: theta_i / (2 pi), theta_i = base^(-2i/D).
unsigned long long rope_turn_fraction(double base, int i, int D) {
  const double theta = std::pow(base, -2.0 * (double)i / (double)D);
  long double x = (long double)theta / (2.0L * 3.14159265358979323846264338327950288L);
  x -= std::floor((double)x);
  const long double hi = std::floor(x * 4294967296.0L);
  const long double lo = std::floor((x * 4294967296.0L - hi) * 4294967296.0L);
  return ((unsigned long long)hi << 32) | (unsigned long long)lo;
}

}  // namespace

namespace kvq {

kvq_status check_config(const kvq_config& cfg) { return validate(cfg); }

void rope_table(double base, int D, unsigned long long* out) {
  for (int i = 0; i < D / 2; ++i) out[i] = rope_turn_fraction(base, i, D);
}

PageLayout make_layout(int R, int D, int G, int bk, int bv, int nsp, bool rope, bool codebook) {
  auto r16 = [](int64_t x) { return (int32_t)((x + 15) / 16 * 16); };
  PageLayout l{};
  l.frag = (bk == 2 || bk == 4) && (bv == 2 || bv == 4) && !rope && !codebook ? 1 : 0;
  l.off_kc = 0;
  l.off_km = l.off_kc + r16((int64_t)R * D * bk / 8);
  l.off_vc = l.off_km + r16((int64_t)(R / G) * D * 4);
  l.off_vm = l.off_vc + r16((int64_t)R * D * bv / 8);
  l.off_si = l.off_vm + r16((int64_t)R * (D / G) * 4);
  l.off_sv = l.off_si + r16((int64_t)R * nsp);
  l.bytes = l.off_sv + r16((int64_t)R * nsp * 2);
  return l;
}

}  // namespace kvq

// Codebook caches quantize with the decision thresholds between their levels.
void set_codebook(const kvq_cache* c, kvq::QuantizeParams* qp) {
  if (!c->cfg.codebook) return;
  qp->lut = 1;
  std::memcpy(qp->k_thr, c->k_thr, sizeof(qp->k_thr));
  std::memcpy(qp->v_thr, c->v_thr, sizeof(qp->v_thr));
}

// The full window of every unit becomes page Tq/R (the flush of an append that finds n_r = R).
cudaError_t flush_window(kvq_cache* c, cudaStream_t s) {
  const int R = c->cfg.residual, D = c->cfg.head_dim;
  kvq::QuantizeParams qp{};
  qp.k_src = c->wk;  // the window rows follow the sink rows
  qp.v_src = c->wv;
  qp.src_unit_stride = rows_per_unit(c) * D;
  qp.src_tok0 = c->cfg.sink_tokens;
  qp.pages = c->pages;
  qp.unit_page_stride = c->unit_page_stride;
  qp.page0 = c->Tq / R;
  qp.n_units = (int32_t)c->n_units;
  qp.Hkv = c->cfg.num_kv_heads;
  qp.D = D;
  qp.G = c->cfg.group_size;
  qp.R = R;
  qp.nsp = c->cfg.k_sparse;
  qp.lay = c->lay;
  qp.err = c->err;
  qp.src_elems = c->n_units * rows_per_unit(c) * D;
  qp.pages_bytes = c->n_units * c->unit_page_stride;
  set_codebook(c, &qp);
  const cudaError_t e = kvq::launch_quantize(qp, c->cfg.k_bits, c->cfg.v_bits, 1, s);
  if (e == cudaSuccess) {
    c->launches++;
    c->Tq += R;
    c->n_r = 0;
  }
  return e;
}

// Copy n_tok tokens (from token src_tok0 of a [units][src_tokens][D] pair of buffers) into the sink
// rows from row n_s.
cudaError_t copy_to_sink(kvq_cache* c, const void* k, const void* v, int64_t src_tokens, int64_t src_tok0,
                         int32_t n_tok, cudaStream_t s) {
  const int D = c->cfg.head_dim;
  kvq::CopyTokensParams cp{};
  cp.k_src = static_cast<const uint16_t*>(k);
  cp.v_src = static_cast<const uint16_t*>(v);
  cp.src_unit_stride = src_tokens * D;
  cp.src_tok0 = src_tok0;
  cp.k_dst = c->wk;
  cp.v_dst = c->wv;
  cp.dst_unit_stride = rows_per_unit(c) * D;
  cp.dst_tok0 = c->n_s;
  cp.n_tok = n_tok;
  cp.n_units = (int32_t)c->n_units;
  cp.D = D;
  const cudaError_t e = kvq::launch_copy_tokens(cp, s);
  if (e == cudaSuccess) {
    c->launches++;
    c->n_s += n_tok;
  }
  return e;
}

// Decode attention over the cache's current state.  k_new/v_new are null, or hold the window's
// newest token (slot n_r - 1), which the kernel then reads from there and stores into the window.
kvq_status launch_decode_for(kvq_cache* c, const void* q, void* out, const void* k_new, const void* v_new,
                             cudaStream_t s) {
  const int R = c->cfg.residual;
  const int64_t grid = decode_grid(c);
  const int hg = c->cfg.num_q_heads / c->cfg.num_kv_heads;
  kvq::DecodeParams dp{};
  dp.q = static_cast<const uint16_t*>(q);
  dp.pages = c->pages;
  dp.unit_page_stride = c->unit_page_stride;
  dp.wk = c->wk;
  dp.wv = c->wv;
  dp.win_unit_stride = rows_per_unit(c) * c->cfg.head_dim;
  dp.k_new = static_cast<const uint16_t*>(k_new);
  dp.v_new = static_cast<const uint16_t*>(v_new);
  dp.n_units = c->n_units;
  dp.n_pages = c->Tq / R;
  dp.work_per_unit = (int32_t)(dp.n_pages + fp16_items(c));
  dp.n_r = c->n_r;
  dp.n_s = c->n_s;
  dp.n_w = c->n_s + c->n_r;
  dp.max_slots = c->max_slots;
  dp.Hkv = c->cfg.num_kv_heads;
  dp.Hq = c->cfg.num_q_heads;
  dp.D = c->cfg.head_dim;
  dp.G = c->cfg.group_size;
  dp.log2G = c->cfg.group_size == 64 ? 6 : 5;
  dp.R = R;
  dp.nsp = c->cfg.k_sparse;
  dp.lay = c->lay;
  dp.qk_scale_log2 = c->cfg.softmax_scale * 1.4426950408889634f;
  dp.rope_turns = c->rope_turns;
  dp.part_ml = c->part_ml;
  dp.part_acc = c->part_acc;
  dp.nslot = c->counters;
  dp.out = static_cast<uint16_t*>(out);
  dp.err = c->err;
  dp.wait_ns = c->test_wait_ns;
  dp.test_withhold = c->test_withhold;
  dp.pages_bytes = c->n_units * c->unit_page_stride;
  if (c->cfg.codebook) {
    dp.lut = 1;
    std::memcpy(dp.k_lev, c->k_lev, sizeof(dp.k_lev));
    std::memcpy(dp.v_lev, c->v_lev, sizeof(dp.v_lev));
  }
  bool supported = false;
  if (kvq::launch_decode(dp, c->cfg.k_bits, c->cfg.v_bits, hg, c->cfg.rope != 0, (int)grid, s, &supported) !=
      cudaSuccess)
    return supported ? fail_cuda(c) : KVQ_ERR_UNSUPPORTED;
  c->launches += 2;  // the decode kernel and the merge of its partials
  return KVQ_OK;
}

extern "C" {

int32_t kvq_version(void) { return (1 << 16) | 0; }

kvq_status kvq_page_layout(const kvq_config* cfg, kvq_page_info* info) {
  if (!cfg || !info) return KVQ_ERR_INVALID_ARG;
  const kvq_status st = validate(*cfg);
  if (st != KVQ_OK) return st;
  // the layout kvq_create gives the cache's pages
  const kvq::PageLayout l = kvq::make_layout(cfg->residual, cfg->head_dim, cfg->group_size, cfg->k_bits, cfg->v_bits,
                                             cfg->k_sparse, cfg->rope != 0, cfg->codebook != 0);
  info->page_bytes = l.bytes;
  info->kcodes_offset = l.off_kc;
  info->kmeta_offset = l.off_km;
  info->vcodes_offset = l.off_vc;
  info->vmeta_offset = l.off_vm;
  info->sp_idx_offset = l.off_si;
  info->sp_val_offset = l.off_sv;
  info->tokens_per_page = cfg->residual;
  info->fragment_order = l.frag;
  return KVQ_OK;
}

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "configuration not supported by this build";
    case KVQ_ERR_CAPACITY: return "cache capacity exceeded";
    case KVQ_ERR_STATE: return "call not allowed in the current cache state";
    case KVQ_ERR_CUDA: return "CUDA error or device-side timeout";
    case KVQ_ERR_OOM: return "device allocation failed";
  }
  return "unknown status";
}

kvq_status kvq_create(const kvq_config* cfg, int device, kvq_cache** out) {
  if (!out) return KVQ_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg) return KVQ_ERR_INVALID_ARG;
  kvq_status st = validate(*cfg);
  if (st != KVQ_OK) return st;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return device < 0 ? KVQ_ERR_INVALID_ARG : KVQ_ERR_CUDA;
  }
  DeviceGuard g(device);
  if (!g.ok) return KVQ_ERR_CUDA;

  kvq_cache* c = new kvq_cache();
  c->cfg = *cfg;
  c->device = device;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
    delete c;
    return KVQ_ERR_CUDA;
  }
  c->sm_count = prop.multiProcessorCount;
  const int D = cfg->head_dim, R = cfg->residual, G = cfg->group_size;
  c->lay = kvq::make_layout(R, D, G, cfg->k_bits, cfg->v_bits, cfg->k_sparse, cfg->rope != 0, cfg->codebook != 0);
  if (kvq::quantize_smem_bytes(R, D, G, c->lay) > (size_t)prop.sharedMemPerBlockOptin) {
    delete c;
    return KVQ_ERR_UNSUPPORTED;
  }
  c->n_units = (int64_t)cfg->batch * cfg->num_kv_heads;
  c->n_pages_cap = quantized_tokens(cfg->max_tokens, R) / R;
  c->unit_page_stride = c->n_pages_cap * (int64_t)c->lay.bytes;
  const int hg = cfg->num_q_heads / cfg->num_kv_heads;
  int warps = 0;
  const int per_sm = kvq::decode_resident_ctas_per_sm(cfg->k_bits, cfg->v_bits, hg, cfg->rope != 0, cfg->residual,
                                                     cfg->k_sparse, c->lay.bytes, &warps, cfg->codebook != 0);
  if (per_sm < 1) {
    cudaGetLastError();
    delete c;
    return KVQ_ERR_UNSUPPORTED;
  }
  c->resident = (int64_t)per_sm * c->sm_count;
  c->decode_warps = warps;
  c->max_slots = (int32_t)slots_for_grid(c, c->resident);

  const int64_t heads = (int64_t)cfg->batch * cfg->num_q_heads;
  {
    std::lock_guard<std::mutex> lock(g_alloc_mutex);
    c->alloc = g_alloc;
  }
  cudaError_t e = cudaSuccess;
  auto alloc = [&](void** p, size_t bytes) {
    if (e == cudaSuccess) e = dev_alloc(c, p, bytes);
  };
  alloc((void**)&c->pages, (size_t)(c->n_units * c->unit_page_stride));
  alloc((void**)&c->wk, (size_t)(c->n_units * rows_per_unit(c) * D * 2));
  alloc((void**)&c->wv, (size_t)(c->n_units * rows_per_unit(c) * D * 2));
  alloc((void**)&c->part_ml, (size_t)(heads * c->max_slots * 2 * sizeof(float)));
  alloc((void**)&c->part_acc, (size_t)(heads * c->max_slots * D * sizeof(float)));
  alloc((void**)&c->counters, (size_t)c->n_units * sizeof(int));  // partial slots taken per unit
  alloc((void**)&c->err, sizeof(int));
  alloc((void**)&c->rope_turns, (size_t)(D / 2) * sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(c->err, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(c->counters, 0, (size_t)c->n_units * sizeof(int));
  if (e == cudaSuccess) {
    std::vector<unsigned long long> turns(D / 2);
    for (int i = 0; i < D / 2; ++i) turns[i] = rope_turn_fraction(cfg->rope ? cfg->rope_base : 10000.0, i, D);
    e = cudaMemcpy(c->rope_turns, turns.data(), turns.size() * sizeof(unsigned long long), cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) {
    const kvq_status st = e == cudaErrorMemoryAllocation ? KVQ_ERR_OOM
                          : e == cudaErrorInvalidValue  ? KVQ_ERR_INVALID_ARG
                                                        : KVQ_ERR_CUDA;
    cudaGetLastError();
    free_all(c);
    delete c;
    return st;
  }
  *out = c;
  return KVQ_OK;
}

kvq_status kvq_set_device_allocator(kvq_alloc_fn alloc, kvq_free_fn free_fn, void* user) {
  if ((alloc == nullptr) != (free_fn == nullptr)) return KVQ_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_alloc_mutex);
  g_alloc.alloc = alloc;
  g_alloc.free = free_fn;
  g_alloc.user = alloc ? user : nullptr;
  return KVQ_OK;
}

kvq_status kvq_debug_check(kvq_cache* c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
#ifdef KVQ_DEBUG_CHECKS
  DeviceGuard g(c->device);
  if (!g.ok || cudaDeviceSynchronize() != cudaSuccess) return fail_cuda(c);
  int err = 0;
  if (cudaMemcpy(&err, c->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return fail_cuda(c);
  if (err != 0) return fail_cuda(c);
  std::vector<unsigned char> buf(kCanaryBytes);
  for (const auto& cn : c->canaries) {
    if (cudaMemcpy(buf.data(), cn.first + cn.second, kCanaryBytes, cudaMemcpyDeviceToHost) != cudaSuccess)
      return fail_cuda(c);
    for (unsigned char b : buf)
      if (b != kCanaryByte) return fail_cuda(c);
  }
  return KVQ_OK;
#else
  return KVQ_ERR_UNSUPPORTED;
#endif
}

kvq_status kvq_destroy(kvq_cache* c) {
  if (!c) return KVQ_OK;
  {
    DeviceGuard g(c->device);
    cudaDeviceSynchronize();
    free_all(c);
  }
  delete c;
  return KVQ_OK;
}

kvq_status kvq_get_state(const kvq_cache* c, int64_t* t_total, int64_t* t_quant, int32_t* n_resid) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (t_total) *t_total = c->T;
  if (t_quant) *t_quant = c->Tq;
  if (n_resid) *n_resid = c->n_r;
  return KVQ_OK;
}

int64_t kvq_launch_count(const kvq_cache* c) { return c ? c->launches : -1; }

kvq_status kvq_reset(kvq_cache* c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->broken) return KVQ_ERR_CUDA;
  c->T = 0;
  c->Tq = 0;
  c->n_r = 0;
  c->n_s = 0;
  c->prefilled = false;
  return KVQ_OK;
}

kvq_status kvq_set_codebooks(kvq_cache* c, const float* k_levels, const float* v_levels) {
  if (!c || !k_levels || !v_levels) return KVQ_ERR_INVALID_ARG;
  if (!c->cfg.codebook) return KVQ_ERR_INVALID_ARG;
  if (c->prefilled || c->T != 0) return KVQ_ERR_STATE;
  auto check = [](const float* lev, int bits) {
    const int L = (1 << bits) - 1;
    if (lev[0] != 0.0f || lev[L] != (float)L) return false;
    for (int j = 0; j < L; ++j)
      if (!(lev[j + 1] > lev[j]) || !std::isfinite(lev[j + 1])) return false;
    return true;
  };
  if (!check(k_levels, c->cfg.k_bits) || !check(v_levels, c->cfg.v_bits)) return KVQ_ERR_INVALID_ARG;
  auto store = [](const float* lev, int bits, float* dst_lev, float* dst_thr) {
    const int L = (1 << bits) - 1;
    for (int j = 0; j < 16; ++j) dst_lev[j] = j <= L ? lev[j] : 0.0f;
    for (int j = 0; j < 16; ++j) {
      if (j < L) {
        volatile float sum = lev[j] + lev[j + 1];  // one rounding, then an exact halving
        dst_thr[j] = sum * 0.5f;
      } else {
        dst_thr[j] = 0.0f;
      }
    }
  };
  store(k_levels, c->cfg.k_bits, c->k_lev, c->k_thr);
  store(v_levels, c->cfg.v_bits, c->v_lev, c->v_thr);
  c->lut_set = true;
  return KVQ_OK;
}

kvq_status kvq_set_splits(kvq_cache* c, int32_t splits) {
  if (!c || splits < 0) return KVQ_ERR_INVALID_ARG;
  const int32_t n = splits > kMaxForcedSplits ? kMaxForcedSplits : splits;
  if (n > 0) {
    DeviceGuard g(c->device);
    if (!g.ok) return fail_cuda(c);
    const cudaError_t e = ensure_slots(c, slots_for_grid(c, c->n_units * n));
    if (e != cudaSuccess) {
      cudaGetLastError();
      return e == cudaErrorMemoryAllocation ? KVQ_ERR_OOM : fail_cuda(c);
    }
  }
  c->forced_splits = n;
  return KVQ_OK;
}

kvq_status kvq_get_splits(const kvq_cache* c, int32_t* splits) {
  if (!c || !splits) return KVQ_ERR_INVALID_ARG;
  *splits = (int32_t)((decode_grid(c) + c->n_units - 1) / c->n_units);
  return KVQ_OK;
}

kvq_status kvq_prefill_quantize(kvq_cache* c, const void* k, const void* v, int64_t n_tokens, void* stream) {
  if (!c || !k || !v) return KVQ_ERR_INVALID_ARG;
  if (c->broken) return KVQ_ERR_CUDA;
  if (!aligned16(k) || !aligned16(v)) return KVQ_ERR_INVALID_ARG;
  if (n_tokens < 1) return KVQ_ERR_INVALID_ARG;
  if (c->prefilled || c->T != 0 || (c->cfg.codebook && !c->lut_set)) return KVQ_ERR_STATE;
  if (n_tokens > c->cfg.max_tokens) return KVQ_ERR_CAPACITY;
  DeviceGuard g(c->device);
  if (!g.ok) return fail_cuda(c);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int R = c->cfg.residual, D = c->cfg.head_dim;
  // the first min(n_tokens, S) tokens go to the sink; the window machine takes the rest
  const int64_t ns = n_tokens < c->cfg.sink_tokens ? n_tokens : c->cfg.sink_tokens;
  if (ns > 0 && copy_to_sink(c, k, v, n_tokens, 0, (int32_t)ns, s) != cudaSuccess) return fail_cuda(c);
  const int64_t Tq = quantized_tokens(n_tokens - ns, R);
  const int64_t n_pages = Tq / R;
  // one launch per at most 65535 pages in grid.x
  for (int64_t p0 = 0; p0 < n_pages; p0 += 65535) {
    const int64_t np = n_pages - p0 < 65535 ? n_pages - p0 : 65535;
    kvq::QuantizeParams qp{};
    qp.k_src = static_cast<const uint16_t*>(k);
    qp.v_src = static_cast<const uint16_t*>(v);
    qp.src_unit_stride = n_tokens * D;
    qp.src_tok0 = ns + p0 * R;
    qp.pages = c->pages;
    qp.unit_page_stride = c->unit_page_stride;
    qp.page0 = p0;
    qp.n_units = (int32_t)c->n_units;
    qp.Hkv = c->cfg.num_kv_heads;
    qp.D = D;
    qp.G = c->cfg.group_size;
    qp.R = R;
    qp.nsp = c->cfg.k_sparse;
    qp.lay = c->lay;
    qp.err = c->err;
    qp.src_elems = c->n_units * n_tokens * D;
    qp.pages_bytes = c->n_units * c->unit_page_stride;
    set_codebook(c, &qp);
    if (kvq::launch_quantize(qp, c->cfg.k_bits, c->cfg.v_bits, (int)np, s) != cudaSuccess) return fail_cuda(c);
    c->launches++;
  }
  kvq::CopyTokensParams cp{};
  cp.k_src = static_cast<const uint16_t*>(k);
  cp.v_src = static_cast<const uint16_t*>(v);
  cp.src_unit_stride = n_tokens * D;
  cp.src_tok0 = ns + Tq;
  cp.k_dst = c->wk;
  cp.v_dst = c->wv;
  cp.dst_unit_stride = rows_per_unit(c) * D;
  cp.dst_tok0 = ns;  // = S whenever window tokens remain
  cp.n_tok = (int32_t)(n_tokens - ns - Tq);
  cp.n_units = (int32_t)c->n_units;
  cp.D = D;
  if (cp.n_tok > 0) {
    if (kvq::launch_copy_tokens(cp, s) != cudaSuccess) return fail_cuda(c);
    c->launches++;
  }
  c->T = n_tokens;
  c->Tq = Tq;
  c->n_r = (int32_t)(n_tokens - ns - Tq);
  c->prefilled = true;
  return KVQ_OK;
}

kvq_status kvq_append(kvq_cache* c, const void* k, const void* v, void* stream) {
  if (!c || !k || !v) return KVQ_ERR_INVALID_ARG;
  if (c->broken) return KVQ_ERR_CUDA;
  if (!aligned16(k) || !aligned16(v)) return KVQ_ERR_INVALID_ARG;
  if (c->cfg.codebook && !c->lut_set) return KVQ_ERR_STATE;
  if (c->T + 1 > c->cfg.max_tokens) return KVQ_ERR_CAPACITY;
  DeviceGuard g(c->device);
  if (!g.ok) return fail_cuda(c);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int R = c->cfg.residual, D = c->cfg.head_dim;
  if (c->n_s < c->cfg.sink_tokens) {  // the sink still has room
    if (copy_to_sink(c, k, v, 1, 0, 1, s) != cudaSuccess) return fail_cuda(c);
    c->T += 1;
    c->prefilled = true;
    return KVQ_OK;
  }
  if (c->n_r == R && flush_window(c, s) != cudaSuccess) return fail_cuda(c);
  kvq::CopyTokensParams cp{};
  cp.k_src = static_cast<const uint16_t*>(k);
  cp.v_src = static_cast<const uint16_t*>(v);
  cp.src_unit_stride = D;
  cp.src_tok0 = 0;
  cp.k_dst = c->wk;
  cp.v_dst = c->wv;
  cp.dst_unit_stride = rows_per_unit(c) * D;
  cp.dst_tok0 = c->n_s + c->n_r;  // the sink is full here: n_s = S
  cp.n_tok = 1;
  cp.n_units = (int32_t)c->n_units;
  cp.D = D;
  if (kvq::launch_copy_tokens(cp, s) != cudaSuccess) return fail_cuda(c);
  c->launches++;
  c->n_r += 1;
  c->T += 1;
  c->prefilled = true;
  return KVQ_OK;
}

kvq_status kvq_decode_attention(kvq_cache* c, const void* q, void* out, void* stream) {
  if (!c || !q || !out) return KVQ_ERR_INVALID_ARG;
  if (c->broken) return KVQ_ERR_CUDA;
  if (!aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
  if (c->T < 1) return KVQ_ERR_STATE;
  DeviceGuard g(c->device);
  if (!g.ok) return fail_cuda(c);
  return launch_decode_for(c, q, out, nullptr, nullptr, static_cast<cudaStream_t>(stream));
}

kvq_status kvq_decode_step(kvq_cache* c, const void* k, const void* v, const void* q, void* out, void* stream) {
  if (!c || !k || !v || !q || !out) return KVQ_ERR_INVALID_ARG;
  if (c->broken) return KVQ_ERR_CUDA;
  if (!aligned16(k) || !aligned16(v) || !aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
  if (c->cfg.codebook && !c->lut_set) return KVQ_ERR_STATE;
  if (c->T + 1 > c->cfg.max_tokens) return KVQ_ERR_CAPACITY;
  DeviceGuard g(c->device);
  if (!g.ok) return fail_cuda(c);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c->n_s < c->cfg.sink_tokens) {  // the token goes to the sink: a copy, then plain decode
    if (copy_to_sink(c, k, v, 1, 0, 1, s) != cudaSuccess) return fail_cuda(c);
    c->T += 1;
    c->prefilled = true;
    return launch_decode_for(c, q, out, nullptr, nullptr, s);
  }
  if (c->n_r == c->cfg.residual && flush_window(c, s) != cudaSuccess) return fail_cuda(c);
  // the new token is window slot n_r; the decode launch stores it there as it reads it
  c->n_r += 1;
  c->T += 1;
  c->prefilled = true;
  return launch_decode_for(c, q, out, k, v, s);
}

kvq_status kvq_test_inject(kvq_cache* c, int32_t withhold_page, int64_t wait_limit_ns) {
  if (!c || withhold_page < -1 || wait_limit_ns < 0) return KVQ_ERR_INVALID_ARG;
  c->test_withhold = withhold_page + 1;
  c->test_wait_ns = (unsigned long long)wait_limit_ns;
  return KVQ_OK;
}

kvq_status kvq_sync_status(kvq_cache* c, void* stream) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return fail_cuda(c);
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return fail_cuda(c);
  int err = 0;
  if (cudaMemcpy(&err, c->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return fail_cuda(c);
  if (err != 0) return fail_cuda(c);
  return c->broken ? KVQ_ERR_CUDA : KVQ_OK;
}

kvq_status kvq_unit_sizes(const kvq_cache* c, kvq_unit_view* v) {
  if (!c || !v) return KVQ_ERR_INVALID_ARG;
  const int D = c->cfg.head_dim, G = c->cfg.group_size, nsp = c->cfg.k_sparse;
  const int64_t Tq = c->Tq;
  v->kcodes_bytes = Tq * D * c->cfg.k_bits / 8;
  v->kmeta_bytes = (Tq / G) * D * 2;
  v->vcodes_bytes = Tq * D * c->cfg.v_bits / 8;
  v->vmeta_bytes = Tq * (D / G) * 2;
  v->sp_idx_bytes = Tq * nsp;
  v->sp_val_bytes = Tq * nsp * 2;
  v->window_bytes = (int64_t)c->n_r * D * 2;
  v->sink_bytes = (int64_t)c->n_s * D * 2;
  return KVQ_OK;
}

kvq_status kvq_export_unit(kvq_cache* c, int32_t b, int32_t kvh, kvq_unit_view* dst, void* stream) {
  if (!c || !dst) return KVQ_ERR_INVALID_ARG;
  if (b < 0 || b >= c->cfg.batch || kvh < 0 || kvh >= c->cfg.num_kv_heads) return KVQ_ERR_INVALID_ARG;
  if (c->broken) return KVQ_ERR_CUDA;
  DeviceGuard g(c->device);
  if (!g.ok) return fail_cuda(c);
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return fail_cuda(c);
  const int D = c->cfg.head_dim, G = c->cfg.group_size, R = c->cfg.residual, nsp = c->cfg.k_sparse;
  const int bk = c->cfg.k_bits, bv = c->cfg.v_bits;
  const int64_t unit = (int64_t)b * c->cfg.num_kv_heads + kvh;
  const int64_t n_pages = c->Tq / R;
  const kvq::PageLayout& L = c->lay;
  std::vector<uint8_t> pg((size_t)(n_pages * L.bytes));
  if (n_pages > 0 && cudaMemcpy(pg.data(), c->pages + unit * c->unit_page_stride, pg.size(), cudaMemcpyDeviceToHost) !=
                         cudaSuccess)
    return fail_cuda(c);
  const int64_t kc_row = (int64_t)D * bk / 8, vc_row = (int64_t)D * bv / 8;
  // code of (token, channel) into a token-major bitstream of `bits`-bit codes
  auto put = [](uint8_t* rows, int64_t row_bytes, int bits, int token, int ch, uint32_t code) {
    uint32_t* w = reinterpret_cast<uint32_t*>(rows + token * row_bytes);
    const int b = ch * bits;
    w[b >> 5] |= code << (b & 31);
    if ((b & 31) + bits > 32) w[(b >> 5) + 1] |= code >> (32 - (b & 31));
  };
  for (int64_t p = 0; p < n_pages; ++p) {
    const uint8_t* src = pg.data() + p * L.bytes;
    if (!L.frag) {
      if (dst->kcodes) std::memcpy((uint8_t*)dst->kcodes + p * R * kc_row, src + L.off_kc, (size_t)(R * kc_row));
      if (dst->vcodes) std::memcpy((uint8_t*)dst->vcodes + p * R * vc_row, src + L.off_vc, (size_t)(R * vc_row));
    } else {
      // fragment order (see frag_key_pair / frag_value_pair) back to token-major bitstreams
      const uint32_t* kw = reinterpret_cast<const uint32_t*>(src + L.off_kc);
      const uint32_t* vw = reinterpret_cast<const uint32_t*>(src + L.off_vc);
      uint8_t* kout = dst->kcodes ? (uint8_t*)dst->kcodes + p * R * kc_row : nullptr;
      uint8_t* vout = dst->vcodes ? (uint8_t*)dst->vcodes + p * R * vc_row : nullptr;
      if (kout) std::memset(kout, 0, (size_t)(R * kc_row));
      if (vout) std::memset(vout, 0, (size_t)(R * vc_row));
      for (int tile = 0; tile < R / 16; ++tile)
        for (int lane = 0; lane < 32; ++lane) {
          for (int w = 0; w < 2 * bk && kout; ++w) {
            const uint32_t word = kw[((int64_t)tile * 32 + lane) * 2 * bk + w];
            for (int j = 0; j < 16 / bk; ++j) {
              int tok, c0;
              kvq::frag_key_pair(bk, tile, lane, w, j, &tok, &c0);
              const uint32_t m = (1u << bk) - 1u;
              put(kout, kc_row, bk, tok, c0, (word >> (bk * j)) & m);
              put(kout, kc_row, bk, tok, c0 + 1, (word >> (16 + bk * j)) & m);
            }
          }
          for (int w = 0; w < 2 * bv && vout; ++w) {
            const uint32_t word = vw[((int64_t)tile * 32 + lane) * 2 * bv + w];
            for (int j = 0; j < 16 / bv; ++j) {
              int tok, ch;
              kvq::frag_value_pair(bv, tile, lane, w, j, &tok, &ch);
              const uint32_t m = (1u << bv) - 1u;
              put(vout, vc_row, bv, tok, ch, (word >> (bv * j)) & m);
              put(vout, vc_row, bv, tok + 1, ch, (word >> (16 + bv * j)) & m);
            }
          }
        }
    }
    const uint32_t* km = reinterpret_cast<const uint32_t*>(src + L.off_km);
    for (int64_t i = 0; i < (int64_t)(R / G) * D; ++i) {
      const int64_t o = p * (R / G) * D + i;
      if (dst->kz) ((uint16_t*)dst->kz)[o] = (uint16_t)(km[i] & 0xFFFFu);
      if (dst->ks) ((uint16_t*)dst->ks)[o] = (uint16_t)(km[i] >> 16);
    }
    const uint32_t* vm = reinterpret_cast<const uint32_t*>(src + L.off_vm);
    for (int64_t i = 0; i < (int64_t)R * (D / G); ++i) {
      const int64_t o = p * R * (D / G) + i;
      if (dst->vz) ((uint16_t*)dst->vz)[o] = (uint16_t)(vm[i] & 0xFFFFu);
      if (dst->vs) ((uint16_t*)dst->vs)[o] = (uint16_t)(vm[i] >> 16);
    }
    if (nsp > 0) {
      if (dst->sp_idx) std::memcpy((uint8_t*)dst->sp_idx + p * R * nsp, src + L.off_si, (size_t)(R * nsp));
      if (dst->sp_val) std::memcpy((uint8_t*)dst->sp_val + p * R * nsp * 2, src + L.off_sv, (size_t)(R * nsp * 2));
    }
  }
  const int64_t S = c->cfg.sink_tokens;
  const size_t wbytes = (size_t)c->n_r * D * 2;
  if (wbytes) {
    if (dst->wk && cudaMemcpy(dst->wk, c->wk + (unit * rows_per_unit(c) + S) * D, wbytes, cudaMemcpyDeviceToHost) !=
                       cudaSuccess)
      return fail_cuda(c);
    if (dst->wv && cudaMemcpy(dst->wv, c->wv + (unit * rows_per_unit(c) + S) * D, wbytes, cudaMemcpyDeviceToHost) !=
                       cudaSuccess)
      return fail_cuda(c);
  }
  const size_t sbytes = (size_t)c->n_s * D * 2;
  if (sbytes) {
    if (dst->sk && cudaMemcpy(dst->sk, c->wk + unit * rows_per_unit(c) * D, sbytes, cudaMemcpyDeviceToHost) !=
                       cudaSuccess)
      return fail_cuda(c);
    if (dst->sv && cudaMemcpy(dst->sv, c->wv + unit * rows_per_unit(c) * D, sbytes, cudaMemcpyDeviceToHost) !=
                       cudaSuccess)
      return fail_cuda(c);
  }
  return KVQ_OK;
}

}  // extern "C"
