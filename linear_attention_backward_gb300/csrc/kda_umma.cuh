// kda_umma.cuh -- fifth-generation tensor-core (tcgen05) building blocks for
// sm_100-family GPUs, written from the PTX ISA: Tensor Memory allocation,
// shared-memory matrix descriptors, the kind::f16 instruction descriptor,
// MMA issue / commit, bounded mbarrier waits and Tensor Memory loads.
//
// Operand layout used throughout: the no-swizzle ("interleaved") canonical
// layout, built from 8 x 16-byte core matrices (8 rows x 8 bf16, 128
// contiguous bytes).  A tile is stored core-matrix by core-matrix:
//   K-major tile  [R rows][C cols], C contiguous in the logical matrix:
//     element (r, c) at ((r / 8) * (C / 8) + c / 8) * 128 + (r % 8) * 16 + (c % 8) * 2
// i.e. core matrices run along the columns first, then down the row groups.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_device.cuh"

namespace kda {
namespace umma {

// ---- byte offset of element (r, c) of an R x C bf16 tile in core-matrix order
__host__ __device__ __forceinline__ uint32_t core_off(int r, int c, int C) {
  return (uint32_t)((((r >> 3) * (C >> 3) + (c >> 3)) << 7) + ((r & 7) << 4) + ((c & 7) << 1));
}
// Padded variant: core matrices along a row of cores sit 144 bytes apart
// (128 + 16), so that the 16-byte rows of the four cores a warp's 32 columns
// touch fall on different banks.  Row groups of 8 are (C / 8) * 144 apart.
constexpr uint32_t kCoreStride = 144;
__host__ __device__ __forceinline__ uint32_t pcore_off(int r, int c, int C) {
  return (uint32_t)((r >> 3) * (C >> 3) * kCoreStride + (c >> 3) * kCoreStride + ((r & 7) << 4) +
                    ((c & 7) << 1));
}
__host__ __device__ constexpr uint32_t ptile_bytes(int R, int C) {
  return (uint32_t)((R / 8) * (C / 8) * kCoreStride);
}

// ---- shared-memory matrix descriptor (no swizzle) ----------------------------
// lbo = byte distance between core matrices adjacent along K, sbo = along M
// (or N); the same rule holds for K-major and MN-major tiles (pinned by the
// device self-test).
// bits  0-13 start address >> 4
// bits 16-29 leading-dimension byte offset >> 4
// bits 32-45 stride-dimension byte offset >> 4
// bits 46-47 descriptor version (1 on sm_100)
// bits 49-51 base offset (0), bit 52 LBO mode (0), bits 61-63 layout (0 = none)
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// ---- 128-byte swizzled layout (SWIZZLE_128B) --------------------------------
// A tile is cut into slabs of 64 contiguous-index elements (128 bytes) and
// each slab into atoms of 8 rows x 128 bytes (1024 bytes, 1024-byte aligned);
// within an atom the 16-byte chunk j of row r sits at chunk j ^ (r % 8).  This
// is the pattern a TMA copy with CU_TENSOR_MAP_SWIZZLE_128B writes (box rows
// of 128 bytes, destination 1024-byte aligned) and the tensor core reads with
// layout type 2.  Element (row, col) -- col the contiguous index -- of a tile
// whose 64-column slabs lie slab_bytes apart sits at sw128_off(row, col,
// slab_bytes).  Read K-major (col = K): each MMA's K = 16 step moves the
// descriptor start 32 bytes along the row (four steps per slab, then the
// next slab); SBO = 1024 (8-row groups), LBO unused.  Read MN-major
// (col = M or N, row = K): each K = 16 step moves the start 2048 bytes (two
// 8-row groups); SBO = 1024, LBO = slab_bytes (the next 64 M / N).
__host__ __device__ __forceinline__ uint32_t sw128_off(int row, int col, uint32_t slab_bytes) {
  return (uint32_t)(col >> 6) * slab_bytes + (uint32_t)((row >> 3) << 10) +
         (uint32_t)((row & 7) << 7) + (uint32_t)((((col & 63) >> 3) ^ (row & 7)) << 4) +
         (uint32_t)((col & 7) << 1);
}
// descriptor of a 128-byte swizzled operand (layout type 2 in bits 61-63)
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return smem_desc(saddr, lbo, sbo) | ((uint64_t)2 << 61);
}

// ---- instruction descriptor, kind::f16 with bf16 inputs and fp32 accumulate
// bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format
// (1 = bf16), 15 A major (0 = K, 1 = MN), 16 B major, 17-22 N >> 3,
// 24-28 M >> 4
__host__ __device__ __forceinline__ uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  uint32_t d = 0;
  d |= 1u << 4;
  d |= 1u << 7;
  d |= 1u << 10;
  d |= (a_mn ? 1u : 0u) << 15;
  d |= (b_mn ? 1u : 0u) << 16;
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}

// ---- Tensor Memory allocation (one warp) ----------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(smem_dst)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols));
}

// ---- MMA: D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread ---------------
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0));
}
// arrive on an mbarrier once every MMA issued so far by this thread is done
__device__ __forceinline__ void mma_commit(uint64_t *mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(mbar)));
}

// ---- mbarrier ----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(mbar)), "r"(count));
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *mbar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(mbar)), "r"(parity));
  return ok != 0;
}
// Poll limits of the bounded waits: copies from HBM, MMA completion, and the
// last wait for work still in flight after a wait has given up (the drain).
constexpr uint32_t kPollLoads = 1u << 24;
constexpr uint32_t kPollMma = 1u << 20;
constexpr uint32_t kPollDrain = 1u << 16;
// Bounded wait: gives up after `limit` polls, flags the device status word
// (timeout) and returns false; the caller must then skip the dependent work,
// drain what is in flight (another bounded wait) and release its resources.
__device__ __forceinline__ bool mbar_wait(uint64_t *mbar, uint32_t parity,
                                          uint32_t limit = kPollLoads) {
  for (uint32_t n = 0; n < limit; ++n)
    if (mbar_try_wait(mbar, parity)) return true;
  set_status(5);
  return false;
}

// ---- bulk copies (the non-tensor TMA path) ------------------------------------
// One thread arms the barrier with the byte count of the copies that complete it.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(mbar)),
               "r"(bytes)
               : "memory");
}
// global -> shared, `bytes` a multiple of 16, both addresses 16-byte aligned
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(mbar))
      : "memory");
}
// One box of a 3-D tensor map (tiled, no swizzle) -> shared memory at dst
// (128-byte aligned), completing `mbar` with the box's bytes.  `map` is the
// address of a __grid_constant__ kernel parameter.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *map, int x, int y, int z,
                                            uint64_t *mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(mbar))
      : "memory");
}

// one box of a 3-D tensor map, shared -> global, tracked by the issuing
// thread's bulk-group counter (the source rows are the box, row-major)
__device__ __forceinline__ void tma_store_3d(const void *map, int x, int y, int z,
                                             const void *src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];\n" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
      : "memory");
}
// shared -> global, tracked by the issuing thread's bulk-group counter
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// all committed bulk stores of this thread have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
// all but the most recent committed group have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_but1() {
  asm volatile("cp.async.bulk.wait_group.read 1;\n" ::: "memory");
}
// ... and are complete
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}

// ---- fences ------------------------------------------------------------------
// generic-proxy smem writes -> visible to the tensor core (async proxy)
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}

// ---- Tensor Memory -> registers: 32 lanes x 16 columns (one warp; lane t of
// the warp reads TMEM lane base + t, columns col .. col + 15) ---------------------
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

}  // namespace umma
}  // namespace kda
