// Decode attention for codebook caches (non-uniform levels: the nuqX datatype of the KVQuant
// review, "Proposed method", with levels the caller supplies instead of a calibrated set): the
// CUDA-core kernel with every code looked up in a 16-entry shared-memory table of levels.  Kept in
// its own translation unit so that the library's sources compile in parallel.
#include "kvq_decode_kernel.cuh"

namespace kvq {

#define KVQ_LUT_CASES(X)                                                                                    \
  X(2, 2, 1, false) X(2, 2, 4, false) X(3, 3, 1, false) X(3, 3, 4, false) X(4, 4, 1, false) X(4, 4, 4, false) \
  X(4, 2, 1, false) X(4, 2, 4, false) X(3, 3, 4, true)

bool decode_lut_supported(int bk, int bv, int hg, bool rope) {
#define KVQ_SUP(BKV, BVV, HGV, RP) \
  if (bk == BKV && bv == BVV && hg == HGV && rope == RP) return true;
  KVQ_LUT_CASES(KVQ_SUP)
#undef KVQ_SUP
  return false;
}

int decode_lut_resident(int bk, int bv, int hg, bool rope, int page_bytes, int* warps) {
  *warps = 0;
#define KVQ_RES(BKV, BVV, HGV, RP) \
  if (bk == BKV && bv == BVV && hg == HGV && rope == RP) return resident_t<BKV, BVV, HGV, RP, true>(page_bytes, warps);
  KVQ_LUT_CASES(KVQ_RES)
#undef KVQ_RES
  return 0;
}

cudaError_t launch_decode_lut(const DecodeParams& p, int bk, int bv, int hg, bool rope, int grid, cudaStream_t s) {
#define KVQ_DEC(BKV, BVV, HGV, RP) \
  if (bk == BKV && bv == BVV && hg == HGV && rope == RP) return launch_decode_t<BKV, BVV, HGV, RP, true>(p, grid, s);
  KVQ_LUT_CASES(KVQ_DEC)
#undef KVQ_DEC
  return cudaErrorInvalidValue;
}

}  // namespace kvq
