// Decode attention on the CUDA cores (3-bit codes, keys rotated at decode): the instantiations
// and the dispatch over every configuration, including the hand-off to the tensor-core kernel
// (kvq_decode_mma.cu), the codebook kernels (kvq_decode_lut.cu) and the merge of the partials.
// The kernel itself is in kvq_decode_kernel.cuh.
#include "kvq_decode_kernel.cuh"

namespace kvq {

// configurations the CUDA-core kernel serves: codes of 3 bits, or keys rotated at decode
#define KVQ_DECODE_CASES(X)                                                                                      \
  X(3, 3, 1, false) X(3, 3, 2, false) X(3, 3, 4, false) X(2, 2, 1, true) X(2, 2, 4, true) X(3, 3, 1, true)       \
  X(3, 3, 4, true) X(4, 2, 1, true) X(4, 2, 4, true) X(4, 4, 1, true) X(4, 4, 4, true)

namespace {
bool frag_codes(int bk, int bv, bool rope) { return (bk == 2 || bk == 4) && (bv == 2 || bv == 4) && !rope; }
}  // namespace

bool decode_supported(int bk, int bv, int hg, bool rope, bool codebook) {
  if (codebook) return decode_lut_supported(bk, bv, hg, rope);
  if (frag_codes(bk, bv, rope)) return decode_mma_supported(bk, bv, hg);
#define KVQ_SUP(BKV, BVV, HGV, RP) \
  if (bk == BKV && bv == BVV && hg == HGV && rope == RP) return true;
  KVQ_DECODE_CASES(KVQ_SUP)
#undef KVQ_SUP
  return false;
}

int decode_resident_ctas_per_sm(int bk, int bv, int hg, bool rope, int R, int nsp, int page_bytes, int* warps,
                                bool codebook) {
  (void)R;
  (void)nsp;
  *warps = 0;
  if (codebook) return decode_lut_resident(bk, bv, hg, rope, page_bytes, warps);
  if (frag_codes(bk, bv, rope)) return decode_mma_resident(bk, bv, hg, page_bytes, warps);
#define KVQ_RES(BKV, BVV, HGV, RP) \
  if (bk == BKV && bv == BVV && hg == HGV && rope == RP) return resident_t<BKV, BVV, HGV, RP, false>(page_bytes, warps);
  KVQ_DECODE_CASES(KVQ_RES)
#undef KVQ_RES
  return 0;
}

namespace {

cudaError_t launch_merge(const DecodeParams& p, int hg, cudaStream_t s) {
  const unsigned grid = (unsigned)p.n_units;
  auto run = [&](auto kern, int threads) -> cudaError_t { return launch_pdl(kern, grid, (unsigned)threads, 0, s, p); };
  switch (hg) {
    case 1: return run(merge_kernel<1>, 1 * kMergeWarpsPerHead * 32);
    case 2: return run(merge_kernel<2>, 2 * kMergeWarpsPerHead * 32);
    case 4: return run(merge_kernel<4>, 4 * kMergeWarpsPerHead * 32);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_only(const DecodeParams& p, int bk, int bv, int hg, bool rope, int grid, cudaStream_t s,
                               bool* supported) {
  if (p.lut) return launch_decode_lut(p, bk, bv, hg, rope, grid, s);
  if (p.lay.frag) return launch_decode_mma(p, bk, bv, hg, grid, s);
#define KVQ_DEC(BKV, BVV, HGV, RP) \
  if (bk == BKV && bv == BVV && hg == HGV && rope == RP) return launch_decode_t<BKV, BVV, HGV, RP, false>(p, grid, s);
  KVQ_DECODE_CASES(KVQ_DEC)
#undef KVQ_DEC
  *supported = false;
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int bk, int bv, int hg, bool rope, int grid, cudaStream_t s,
                          bool* supported) {
  *supported = decode_supported(bk, bv, hg, rope, p.lut != 0);
  if (!*supported) return cudaErrorInvalidValue;
  const cudaError_t e = launch_decode_only(p, bk, bv, hg, rope, grid, s, supported);
  if (e != cudaSuccess) return e;
  return launch_merge(p, hg, s);
}

}  // namespace kvq
