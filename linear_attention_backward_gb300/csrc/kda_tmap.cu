// kda_tmap.cu -- host-side encoding of the TMA tensor maps of the token-major
// inputs.  The driver's encoder is looked up through the runtime once per
// process, so the library needs no link against the driver library.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kda_params.h"

namespace kda {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// [ntok, H, 128] bf16, box = 64 tokens x 1 head x `width` channels; width
// 128 without swizzling (row-major rows of 256 bytes), or 64 with 128-byte
// swizzling (rows of 128 bytes, 16-byte chunks permuted by row % 8)
bool encode(CUtensorMap *m, const void *base, int64_t ntok, int H, int width = 128,
            bool swizzle = false) {
  auto fn = encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)ntok};
  const cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};  // bytes, dims 1 and 2
  const cuuint32_t box[3] = {(cuuint32_t)width, 1, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_token_maps(const KdaParams &p, TokenMaps &m) {
  const int64_t ntok = (int64_t)p.B * p.T;
  if (ntok <= 0) return true;  // nothing is launched
  // a tensor the call does not have (dO in the forward) keeps an empty map
  auto enc = [&](CUtensorMap *mp, const void *base) {
    return base == nullptr || encode(mp, base, ntok, p.H);
  };
  return enc(&m.q, p.q) && enc(&m.k, p.k) && enc(&m.g, p.g) && enc(&m.v, p.v) &&
         enc(&m.dO, p.dO) && enc(&m.dq, p.dq) && enc(&m.dk, p.dk) && enc(&m.dv, p.dv) &&
         enc(&m.dg, p.dg) &&
         (p.dO == nullptr || encode(&m.dO_sw, p.dO, ntok, p.H, 64, true)) &&
         (p.v == nullptr || encode(&m.v_sw, p.v, ntok, p.H, 64, true));
}

}  // namespace kda
