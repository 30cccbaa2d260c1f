// Decode attention over caller-owned packed buffers with no device allocation.
//
// Some callers cannot call cudaMalloc when they need attention: an engine
// that carves all device memory out of its own pool up front and forbids
// libraries from allocating behind its back, or code that must not take the
// allocator's locks or synchronisation on a latency-critical path.  They
// keep the packed pages and the fp16 window in memory they own and call
// kvq_decode_attention_noalloc.  The split-attention partials that
// kvq_decode_attention keeps in each cache's workspace live here instead in
// one file-scope device array, sized once for the whole process.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

// Scratch for split partials and per-unit counters, shared by every call in
// the process.  Every GPU that loads the library holds it until exit.
constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on `device` (which must be current).
// The first call on a device looks the symbol up once and remembers it.
cudaError_t scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[device]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[device] = ptr;
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, const void* pages, int64_t pages_per_unit,
                                                   const void* window_k, const void* window_v, int64_t n_tokens,
                                                   const void* q_f16, void* out_f16, void* cuda_stream) {
  if (!cfg || !pages || !window_k || !window_v || !q_f16 || !out_f16) return KVQ_ERR_INVALID_ARG;
  const kvq_status st = kvq::check_config(*cfg);
  if (st != KVQ_OK) return st;
  if (n_tokens < 1 || n_tokens > cfg->max_tokens || pages_per_unit < 0) return KVQ_ERR_INVALID_ARG;
  if (cfg->sink_tokens != 0 || cfg->codebook != 0) return KVQ_ERR_UNSUPPORTED;  // the buffers hold neither
  if (!aligned16(pages) || !aligned16(window_k) || !aligned16(window_v) || !aligned16(q_f16) || !aligned16(out_f16))
    return KVQ_ERR_INVALID_ARG;
  const int D = cfg->head_dim, R = cfg->residual, G = cfg->group_size;
  const int64_t tq = (int64_t)R * ((n_tokens - 1) / R);
  const int64_t n_pages = tq / R;
  if (n_pages > pages_per_unit) return KVQ_ERR_INVALID_ARG;
  const int hg = cfg->num_q_heads / cfg->num_kv_heads;
  const int64_t n_units = (int64_t)cfg->batch * cfg->num_kv_heads;
  const int64_t heads = (int64_t)cfg->batch * cfg->num_q_heads;
  const kvq::PageLayout lay = kvq::make_layout(R, D, G, cfg->k_bits, cfg->v_bits, cfg->k_sparse, cfg->rope != 0);

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return KVQ_ERR_CUDA;
  void* scratch = nullptr;
  if (scratch_address(device, &scratch) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ERR_CUDA;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return KVQ_ERR_CUDA;
  int warps = 0;
  const int per_sm = kvq::decode_resident_ctas_per_sm(cfg->k_bits, cfg->v_bits, hg, cfg->rope != 0, cfg->residual,
                                                     cfg->k_sparse, lay.bytes, &warps);
  if (per_sm < 1) {
    cudaGetLastError();
    return KVQ_ERR_UNSUPPORTED;
  }

  // Scratch layout: the RoPE turn table, per-unit tickets and slot counts, then (m, l) and acc[D]
  // per query head and partial slot.  The grid is the resident CTA count, lowered until the
  // slots it needs (warps * (ceil(grid / units) + 2) per query head) fit; a size that does not
  // fit even one CTA is refused.
  const int64_t wpu = n_pages + (n_tokens - tq > 0 ? 1 : 0);
  const size_t rope_bytes = 256 * 8;  // room for the RoPE turn table (D/2 entries)
  const size_t counter_bytes = rope_bytes + ((size_t)n_units * 2 * sizeof(int) + 255) / 256 * 256;
  auto slots_for = [&](int64_t g) { return (int64_t)warps * ((g + n_units - 1) / n_units + 2); };
  auto ml_bytes_for = [&](int64_t sl) { return ((size_t)heads * sl * 2 * sizeof(float) + 255) / 256 * 256; };
  auto bytes_for = [&](int64_t g) {
    const int64_t sl = slots_for(g);
    return counter_bytes + ml_bytes_for(sl) + (size_t)heads * sl * D * sizeof(float);
  };
  int64_t grid = (int64_t)per_sm * sms;
  if (grid > n_units * wpu) grid = n_units * wpu;
  while (grid > 1 && bytes_for(grid) > kScratchBytes) grid = grid * 3 / 4;
  if (bytes_for(grid) > kScratchBytes) return KVQ_ERR_CAPACITY;
  const int64_t slots = slots_for(grid);

  unsigned char* base = static_cast<unsigned char*>(scratch);
  unsigned long long* rope_turns = reinterpret_cast<unsigned long long*>(base);
  int* counters = reinterpret_cast<int*>(base + rope_bytes);
  float* part_ml = reinterpret_cast<float*>(base + counter_bytes);
  float* part_acc = reinterpret_cast<float*>(base + counter_bytes + ml_bytes_for(slots));
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  // the counters must start at zero; a call that stopped early may have left them set
  if (cudaMemsetAsync(counters, 0, (size_t)n_units * 2 * sizeof(int), s) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cfg->rope) {
    // pageable source: the copy has taken the table by the time the call returns
    unsigned long long table[kvq::kHeadDim / 2];
    kvq::rope_table(cfg->rope_base, D, table);
    if (cudaMemcpyAsync(rope_turns, table, sizeof(table), cudaMemcpyHostToDevice, s) != cudaSuccess)
      return KVQ_ERR_CUDA;
  }

  kvq::DecodeParams dp{};
  dp.q = static_cast<const uint16_t*>(q_f16);
  dp.pages = static_cast<const uint8_t*>(pages);
  dp.unit_page_stride = pages_per_unit * (int64_t)lay.bytes;
  dp.wk = static_cast<const uint16_t*>(window_k);
  dp.wv = static_cast<const uint16_t*>(window_v);
  dp.win_unit_stride = (int64_t)R * D;
  dp.n_units = n_units;
  dp.n_pages = n_pages;
  dp.work_per_unit = (int32_t)wpu;
  dp.n_r = (int32_t)(n_tokens - tq);
  dp.n_w = dp.n_r;  // no sink tokens here
  dp.max_slots = (int32_t)slots;
  dp.Hkv = cfg->num_kv_heads;
  dp.Hq = cfg->num_q_heads;
  dp.D = D;
  dp.G = G;
  dp.log2G = G == 64 ? 6 : 5;
  dp.R = R;
  dp.nsp = cfg->k_sparse;
  dp.lay = lay;
  dp.qk_scale_log2 = cfg->softmax_scale * 1.4426950408889634f;
  dp.rope_turns = rope_turns;
  dp.part_ml = part_ml;
  dp.part_acc = part_acc;
  dp.nslot = counters;
  dp.out = static_cast<uint16_t*>(out_f16);
  dp.err = nullptr;
  bool supported = false;
  if (kvq::launch_decode(dp, cfg->k_bits, cfg->v_bits, hg, cfg->rope != 0, (int)grid, s, &supported) != cudaSuccess)
    return supported ? KVQ_ERR_CUDA : KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}
