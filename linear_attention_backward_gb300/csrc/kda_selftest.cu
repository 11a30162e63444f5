// kda_selftest.cu -- device self-test of the tcgen05 building blocks: one
// M = 128 tile D = A B^T (K up to 128) through shared-memory descriptors,
// Tensor Memory and tcgen05.ld, with A and B in K-major or MN-major
// core-matrix layout (packed or padded) or in the 128-byte swizzled layout.
// Used by the test-suite to pin the descriptor encodings on the device
// before the kernels rely on them.
#include <cuda_runtime.h>

#include "kda.h"
#include "kda_umma.cuh"

namespace kda {

// A: [M = 128][K] bf16 row-major, B: [N][K] bf16 row-major, D: [128][N] fp32.
__global__ void __launch_bounds__(128) kda_selftest_umma_kernel(const bf16 *A, const bf16 *B,
                                                                 float *D, int N, int K,
                                                                 int a_mn, int b_mn,
                                                                 int layout) {
  extern __shared__ __align__(1024) char smem[];
  constexpr int M = 128;
  bf16 *As = reinterpret_cast<bf16 *>(smem);
  // a padded 128 x 128 tile takes 36 KB
  bf16 *Bs = reinterpret_cast<bf16 *>(smem + 40960);
  uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + 81920);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + 81920 + 64);
  const int tid = threadIdx.x, warp = tid >> 5;
  // the swizzled layout's atoms need 1024-byte aligned tiles
  const bool aligned = (smem_u32(smem) & 1023u) == 0u;
  // slab strides of the swizzled layout: K-major tiles stack their 64-column
  // K slabs (rows x 128 bytes each), MN-major ones their 64-wide M / N slabs
  // (K x 128 bytes each)
  const uint32_t a_slab = a_mn ? (uint32_t)K * 128u : (uint32_t)M * 128u;
  const uint32_t b_slab = b_mn ? (uint32_t)K * 128u : (uint32_t)N * 128u;
  // A element (m, k): K-major -> core_off(m, k, K); MN-major -> core_off(k, m, M)
  for (int e = tid; e < M * K; e += 128) {
    const int m = e / K, k = e % K;
    const uint32_t off =
        layout == 2 ? (a_mn ? umma::sw128_off(k, m, a_slab) : umma::sw128_off(m, k, a_slab))
        : layout == 1 ? (a_mn ? umma::pcore_off(k, m, M) : umma::pcore_off(m, k, K))
                      : (a_mn ? umma::core_off(k, m, M) : umma::core_off(m, k, K));
    *reinterpret_cast<bf16 *>(reinterpret_cast<char *>(As) + off) = A[e];
  }
  for (int e = tid; e < N * K; e += 128) {
    const int n = e / K, k = e % K;
    const uint32_t off =
        layout == 2 ? (b_mn ? umma::sw128_off(k, n, b_slab) : umma::sw128_off(n, k, b_slab))
        : layout == 1 ? (b_mn ? umma::pcore_off(k, n, N) : umma::pcore_off(n, k, K))
                      : (b_mn ? umma::core_off(k, n, N) : umma::core_off(n, k, K));
    *reinterpret_cast<bf16 *>(reinterpret_cast<char *>(Bs) + off) = B[e];
  }
  if (tid == 0) umma::mbar_init(mbar, 1);
  umma::fence_async_smem();
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  __syncthreads();
  if (warp == 0) umma::tmem_alloc(tslot, N < 32 ? 32 : N);
  umma::tc_fence_before();
  __syncthreads();
  umma::tc_fence_after();
  const uint32_t tbase = *tslot;
  if (tid == 0 && aligned && layout == 2) {
    const uint32_t idesc = umma::idesc_bf16(M, N, a_mn != 0, b_mn != 0);
    const uint32_t a0 = smem_u32(As), b0 = smem_u32(Bs);
    for (int s = 0; s < K / 16; ++s) {
      // K-major: 32 bytes along the 128-byte rows per step, four steps per
      // slab; MN-major: two 8-row groups (2048 bytes) per step
      const uint32_t a_at = a_mn ? a0 + 2048u * s : a0 + (s >> 2) * a_slab + 32u * (s & 3);
      const uint32_t b_at = b_mn ? b0 + 2048u * s : b0 + (s >> 2) * b_slab + 32u * (s & 3);
      const uint64_t ad = umma::smem_desc_sw128(a_at, a_mn ? a_slab : 16u, 1024u);
      const uint64_t bd = umma::smem_desc_sw128(b_at, b_mn ? b_slab : 16u, 1024u);
      umma::mma_bf16(tbase, ad, bd, idesc, s > 0);
    }
    umma::mma_commit(mbar);
  } else if (tid == 0 && layout != 2) {
    const uint32_t idesc = umma::idesc_bf16(M, N, a_mn != 0, b_mn != 0);
    const uint32_t a0 = smem_u32(As), b0 = smem_u32(Bs);
    for (int s = 0; s < K / 16; ++s) {
      // Descriptor strides: LBO = distance between core matrices along K,
      // SBO = distance between core matrices along M (or N).  Each step
      // consumes two core matrices along K.
      uint32_t a_lead, a_str, a_step, b_lead, b_str, b_step;
      if (!a_mn) { a_lead = 128; a_str = (K / 8) * 128; a_step = 256; }
      else { a_lead = (M / 8) * 128; a_str = 128; a_step = 2 * (M / 8) * 128; }
      if (!b_mn) { b_lead = 128; b_str = (K / 8) * 128; b_step = 256; }
      else { b_lead = (N / 8) * 128; b_str = 128; b_step = 2 * (N / 8) * 128; }
      if (layout == 1) {  // padded core layout
        const uint32_t cs = umma::kCoreStride;
        if (!a_mn) { a_lead = cs; a_str = (K / 8) * cs; a_step = 2 * cs; }
        else { a_lead = (M / 8) * cs; a_str = cs; a_step = 2 * (M / 8) * cs; }
        if (!b_mn) { b_lead = cs; b_str = (K / 8) * cs; b_step = 2 * cs; }
        else { b_lead = (N / 8) * cs; b_str = cs; b_step = 2 * (N / 8) * cs; }
      }
      const uint64_t ad = umma::smem_desc(a0 + s * a_step, a_lead, a_str);
      const uint64_t bd = umma::smem_desc(b0 + s * b_step, b_lead, b_str);
      umma::mma_bf16(tbase, ad, bd, idesc, s > 0);
    }
    umma::mma_commit(mbar);
  }
  const bool ok = (aligned || layout != 2) && umma::mbar_wait(mbar, 0);
  umma::tc_fence_after();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 16) {
      float v[16];
      umma::tmem_ld16(tbase + ((uint32_t)(32 * warp) << 16) + c0, v);
      umma::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) D[(32 * warp + (tid & 31)) * N + c0 + j] = v[j];
    }
  }
  umma::tc_fence_before();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tbase, N < 32 ? 32 : N);
}

}  // namespace kda

extern "C" kda_status kda_selftest_umma(const void *A, const void *B, float *D, int N, int K,
                                        int a_mn, int b_mn, int layout,
                                        kda_stream_t stream) {
  if (!A || !B || !D || (N != 32 && N != 64 && N != 128) || K < 16 || K > 128 || K % 16 ||
      (layout != 0 && layout != 1 && layout != 2))
    return KDA_ERR_INVALID_ARG;
  // the swizzled layout's MN-major slabs are 64 wide; its K-major slabs take
  // K in steps of 64
  if (layout == 2 && ((b_mn && N < 64) || K % 64 != 0)) return KDA_ERR_INVALID_ARG;
  auto k = kda::kda_selftest_umma_kernel;
  // generous allocation: the tiles use the first 80 KB only
  const int smem = 180 * 1024;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return KDA_ERR_CUDA;
  k<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const kda::bf16 *>(A), static_cast<const kda::bf16 *>(B), D, N, K, a_mn, b_mn,
      layout);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
