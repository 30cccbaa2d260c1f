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

// Fixed head of the array: the error word (256-byte block), then up to kRopeTables RoPE turn tables
// (D/2 = 64 entries each), written once per device and rope base; the counters and partials follow.
constexpr size_t kErrBytes = 256;
constexpr int kRopeTables = 8;
constexpr size_t kRopeTableBytes = (kvq::kHeadDim / 2) * sizeof(unsigned long long);
constexpr size_t kHeadBytes = kErrBytes + kRopeTables * kRopeTableBytes;

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};
float g_rope_base[kMaxDevices][kRopeTables];  // bases whose tables are in place
int g_rope_used[kMaxDevices] = {};

// Device address of the scratch array on `device` (which must be current).
// The first call on a device looks the symbol up once and remembers it.
cudaError_t scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[device]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess) return e;
    // a fresh array holds zeros; clear the error word anyway (synchronous, once per device)
    const cudaError_t z = cudaMemset(ptr, 0, kErrBytes);
    if (z != cudaSuccess) return z;
    g_scratch_addr[device] = ptr;
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

// The RoPE turn table of `base` inside the scratch array of `device`: written by a synchronous copy
// the first time a base is used on the device, found again by later calls (which then copy nothing).
// More than kRopeTables distinct bases on one device are refused: *full is set and nothing is copied.
cudaError_t rope_table_address(int device, unsigned char* base_addr, float rope_base, unsigned long long** out,
                               bool* full) {
  *full = false;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  for (int i = 0; i < g_rope_used[device]; ++i)
    if (g_rope_base[device][i] == rope_base) {
      *out = reinterpret_cast<unsigned long long*>(base_addr + kErrBytes + i * kRopeTableBytes);
      return cudaSuccess;
    }
  if (g_rope_used[device] >= kRopeTables) {
    *full = true;
    return cudaSuccess;
  }
  const int i = g_rope_used[device];
  unsigned long long table[kvq::kHeadDim / 2];
  kvq::rope_table(rope_base, kvq::kHeadDim, table);
  unsigned long long* dst = reinterpret_cast<unsigned long long*>(base_addr + kErrBytes + i * kRopeTableBytes);
  const cudaError_t e = cudaMemcpy(dst, table, sizeof(table), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return e;
  g_rope_base[device][i] = rope_base;
  g_rope_used[device] = i + 1;
  *out = dst;
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

  // Scratch layout after the fixed head (error word, RoPE tables): the per-unit slot counters, then
  // (m, l) and acc[D] per query head and partial slot.  The grid is the resident CTA count, lowered
  // until the slots it needs (warps * (ceil(grid / units) + 2) per query head) fit; a size that does
  // not fit even one CTA is refused.
  const int64_t wpu = n_pages + (n_tokens - tq > 0 ? 1 : 0);
  const size_t counter_bytes = kHeadBytes + ((size_t)n_units * sizeof(int) + 255) / 256 * 256;
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
  int* err_word = reinterpret_cast<int*>(base);
  unsigned long long* rope_turns = nullptr;
  if (cfg->rope) {
    bool full = false;
    const cudaError_t e = rope_table_address(device, base, cfg->rope_base, &rope_turns, &full);
    if (full) return KVQ_ERR_CAPACITY;  // a ninth distinct rope base on this device
    if (e != cudaSuccess) {
      cudaGetLastError();
      return KVQ_ERR_CUDA;
    }
  }
  int* counters = reinterpret_cast<int*>(base + kHeadBytes);
  float* part_ml = reinterpret_cast<float*>(base + counter_bytes);
  float* part_acc = reinterpret_cast<float*>(base + counter_bytes + ml_bytes_for(slots));
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  // the slot counters must start at zero; a call that stopped early may have left them set
  if (cudaMemsetAsync(counters, 0, (size_t)n_units * sizeof(int), s) != cudaSuccess) return KVQ_ERR_CUDA;

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
  dp.pages_bytes = n_units * dp.unit_page_stride;
  dp.err = err_word;  // a device-side wait that runs out is recorded here (kvq_noalloc_sync_status)
  bool supported = false;
  if (kvq::launch_decode(dp, cfg->k_bits, cfg->v_bits, hg, cfg->rope != 0, (int)grid, s, &supported) != cudaSuccess)
    return supported ? KVQ_ERR_CUDA : KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

extern "C" kvq_status kvq_noalloc_sync_status(void* cuda_stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return KVQ_ERR_CUDA;
  void* scratch = nullptr;
  if (scratch_address(device, &scratch) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ERR_CUDA;
  }
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  int err = 0;
  if (cudaMemcpy(&err, scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KVQ_ERR_CUDA;
  if (err == 0) return KVQ_OK;
  if (cudaMemset(scratch, 0, sizeof(int)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_ERR_CUDA;
}
