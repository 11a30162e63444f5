// kda_device.cuh -- device-side building blocks shared by the KDA kernels:
// bf16 packing, ldmatrix / mma.sync wrappers, a warp-level 16-row GEMM on
// shared-memory tiles (bf16 tensor-core version and an fp32 SIMT version with
// the same accumulator layout), and the device status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

using bf16 = __nv_bfloat16;

constexpr int CHUNK = 64;        // tokens per chunk
constexpr int NTHREADS = 256;    // 8 warps per CTA in every kernel
constexpr int NWARPS = NTHREADS / 32;

// Device status word of this translation unit (one per device and per
// kernel file; read and cleared through the host API).
static __device__ int g_status = 0;

__device__ __forceinline__ void set_status(int code) { atomicCAS(&g_status, 0, code); }

// Programmatic dependent launch: a kernel launched by pdl_launch (kda_params.h)
// may start while the kernel before it on the stream finishes its last CTAs;
// it waits here, before it touches anything that kernel writes (a no-op for a
// kernel launched the ordinary way).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// The intra-chunk products carry the gate through 16-row block factors
// e^(gc_i - m_I) and e^(m_I - gc_j) around each block's reference row (up to
// 7 and 8 tokens of log-decay).  Past 88 nats such a factor is infinite in
// fp32 and the gradients cannot be finite: the tcgen05 prep flags the chunk
// for the exact kernels (kda_range.cu), the other prep kernels raise this
// status code (KDA_ERR_GATE_RANGE) instead of returning them silently.
// (Below it the factors are finite; sums of them stay finite for ordinary
// operands: a parity test reaches 85.6 nats.)
constexpr float kMaxBlockLogDecay = 88.f;
// The tcgen05 path also flags a chunk in which every channel decays by more
// than this many nats per token on average over the chunk's rows.  There the
// true dg is of order e^(-gk) while the block-factored products leave an
// absolute error of about 1e-5 of the terms that cancel in it (measured on a
// GB300 with uniform gates: dg's relative error 3.5e-3 at 6 nats per token,
// 3.1e-2 at 8, 0.16 at 10); with one weaker channel the tensor's dg is
// carried by that channel and stays accurate.
constexpr float kStrongTokenDecay = 6.f;
constexpr int kStatusGateRange = 8;
__device__ __forceinline__ void check_block_log_decay(float span) {
  if (span > kMaxBlockLogDecay) set_status(kStatusGateRange);
}

// Row stride (elements) of a shared tile with `cols` columns: 16 bytes of
// padding per row for bf16 keeps ldmatrix row addresses on distinct 16-byte
// bank groups (stride = 16 mod 128 bytes).  fp32 tiles feed the SIMT path
// only and stay unpadded (rows remain 16-byte aligned).
template <typename E> __host__ __device__ constexpr int tile_ld(int cols) {
  return cols + (sizeof(E) == 2 ? 8 : 0);
}

template <typename E> __device__ __forceinline__ float to_f(E x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 x) { return __bfloat162float(x); }

template <typename E> __device__ __forceinline__ E from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// store two consecutive elements
__device__ __forceinline__ void store2(float *p, float a, float b) {
  *reinterpret_cast<float2 *>(p) = make_float2(a, b);
}
__device__ __forceinline__ void store2(bf16 *p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
}
__device__ __forceinline__ float2 load2(const float *p) {
  return *reinterpret_cast<const float2 *>(p);
}
__device__ __forceinline__ float2 load2(const bf16 *p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const bf16 *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const bf16 *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// D(16x8) += A(16x16) * B(16x8), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t scale_pair(uint32_t v, float s0, float s1) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&v);
  float2 f = __bfloat1622float2(h);
  __nv_bfloat162 o = __floats2bfloat162_rn(f.x * s0, f.y * s1);
  return *reinterpret_cast<uint32_t *>(&o);
}

// Accumulator layout (both versions): for a 16 x (8*NF) output, lane l holds
//   acc[f][0] -> (row l/4,     col 8f + 2(l%4))     acc[f][1] -> col + 1
//   acc[f][2] -> (row l/4 + 8, col 8f + 2(l%4))     acc[f][3] -> col + 1
// Operand addressing:
//   AK = true : A(m, k) = a[m * lda + k]      AK = false: A(m, k) = a[k * lda + m]
//   BK = true : B(k, n) = b[n * ldb + k]      BK = false: B(k, n) = b[k * ldb + n]
// kscale (nullable): per-k factor applied to A, i.e. A(m, k) * kscale[k].
template <int NF, bool AK, bool BK>
__device__ __forceinline__ void warp_gemm(float (&acc)[NF][4], const bf16 *a, int lda,
                                          const bf16 *b, int ldb, int kdim,
                                          const float *kscale = nullptr) {
  static_assert(NF % 2 == 0, "NF must be even");
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k0 = 0; k0 < kdim; k0 += 16) {
    uint32_t af[4];
    if (AK)
      ldsm_x4(af, a + (lane & 15) * lda + k0 + (lane >> 4) * 8);
    else
      ldsm_x4_t(af, a + (k0 + (lane & 7) + (lane >> 4) * 8) * lda + ((lane >> 3) & 1) * 8);
    if (kscale != nullptr) {
      const int c = k0 + 2 * (lane & 3);
      const float s0 = kscale[c], s1 = kscale[c + 1], s8 = kscale[c + 8], s9 = kscale[c + 9];
      af[0] = scale_pair(af[0], s0, s1);
      af[1] = scale_pair(af[1], s0, s1);
      af[2] = scale_pair(af[2], s8, s9);
      af[3] = scale_pair(af[3], s8, s9);
    }
#pragma unroll
    for (int f = 0; f < NF; f += 2) {
      uint32_t bfr[4];
      if (BK)
        ldsm_x4(bfr, b + (f * 8 + (lane & 7) + (lane >> 4) * 8) * ldb + k0 + ((lane >> 3) & 1) * 8);
      else
        ldsm_x4_t(bfr, b + (k0 + (lane & 7) + ((lane >> 3) & 1) * 8) * ldb + f * 8 + (lane >> 4) * 8);
      mma_16816(acc[f], af, bfr[0], bfr[1]);
      mma_16816(acc[f + 1], af, bfr[2], bfr[3]);
    }
  }
}

// fp32 SIMT version: same operands, same accumulator layout.
template <int NF, bool AK, bool BK>
__device__ __forceinline__ void warp_gemm(float (&acc)[NF][4], const float *a, int lda,
                                          const float *b, int ldb, int kdim,
                                          const float *kscale = nullptr) {
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2, c = 2 * (lane & 3);
  for (int k = 0; k < kdim; ++k) {
    float a0 = AK ? a[r * lda + k] : a[k * lda + r];
    float a1 = AK ? a[(r + 8) * lda + k] : a[k * lda + r + 8];
    if (kscale != nullptr) {
      a0 *= kscale[k];
      a1 *= kscale[k];
    }
#pragma unroll
    for (int f = 0; f < NF; ++f) {
      const int n = 8 * f + c;
      const float b0 = BK ? b[n * ldb + k] : b[k * ldb + n];
      const float b1 = BK ? b[(n + 1) * ldb + k] : b[k * ldb + n + 1];
      acc[f][0] = fmaf(a0, b0, acc[f][0]);
      acc[f][1] = fmaf(a0, b1, acc[f][1]);
      acc[f][2] = fmaf(a1, b0, acc[f][2]);
      acc[f][3] = fmaf(a1, b1, acc[f][3]);
    }
  }
}

template <int NF> __device__ __forceinline__ void zero_acc(float (&acc)[NF][4]) {
#pragma unroll
  for (int f = 0; f < NF; ++f) acc[f][0] = acc[f][1] = acc[f][2] = acc[f][3] = 0.f;
}

// Visit every accumulator element: fn(row, col, value&) with row/col local to
// the 16 x (8*NF) warp tile.
template <int NF, typename Fn>
__device__ __forceinline__ void for_acc(float (&acc)[NF][4], Fn fn) {
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2, c = 2 * (lane & 3);
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    fn(r, 8 * f + c, acc[f][0]);
    fn(r, 8 * f + c + 1, acc[f][1]);
    fn(r + 8, 8 * f + c, acc[f][2]);
    fn(r + 8, 8 * f + c + 1, acc[f][3]);
  }
}

// Store a warp accumulator tile to a shared/global tile (row stride ld).
template <int NF, typename E>
__device__ __forceinline__ void store_acc(E *dst, int ld, float (&acc)[NF][4], float mul = 1.f) {
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2, c = 2 * (lane & 3);
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    store2(dst + r * ld + 8 * f + c, acc[f][0] * mul, acc[f][1] * mul);
    store2(dst + (r + 8) * ld + 8 * f + c, acc[f][2] * mul, acc[f][3] * mul);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// sum over the 4 lanes that share accumulator rows (lane % 4)
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

// log(1 + t) for t in [0, 1].  The fast log of the rounded sum 1 + t keeps
// an absolute error of ~1e-7 but loses the relative precision of small t
// (1 + t rounds to 1 below 2^-24), so arguments below 2^-5 take the Taylor
// series t - t^2/2 + t^3/3 - t^4/4 + t^5/5 instead (relative truncation
// error below t^5 / 6 < 1e-8 there).
__device__ __forceinline__ float log1p_series(float t) {
  return t * fmaf(-t, fmaf(-t, fmaf(-t, fmaf(-t, 0.2f, 0.25f), 0.33333334f), 0.5f), 1.f);
}
__device__ __forceinline__ float log1p_unit(float t) {
  return t < 0.03125f ? log1p_series(t) : __logf(1.f + t);
}
// The same for a warp whose 32 arguments are mostly not small: the fast log,
// replaced by the series only where t < 2^-14 (where the fast log's error of
// ~6e-8 reaches 1e-3 of the value), behind a warp vote so that the common
// case pays one vote.  All 32 lanes must call it together.
__device__ __forceinline__ float log1p_unit_warp(float t) {
  float l = __logf(1.f + t);
  const bool tiny = t < 6.103515625e-05f;
  if (__any_sync(0xffffffffu, tiny) && tiny) l = log1p_series(t);
  return l;
}
// softplus for the dA_log terms dgk * gk, whose sum needs gk's relative
// precision: log(1 + e^x) = max(x, 0) + log(1 + e^-|x|) with the accurate
// log1p above (softplus(-30) ~ 1e-13 is not rounded to zero)
__device__ __forceinline__ float softplus_f(float x) {
  return fmaxf(x, 0.f) + log1p_unit(__expf(-fabsf(x)));
}
// softplus for the gate's running sums, which feed the decays e^gc: there an
// absolute error of ~1e-7 per token is far below the bf16 operands' own, so
// the plain fast log of 1 + e^-|x| serves (it rounds values below ~1e-7 to 0)
__device__ __forceinline__ float softplus_gate(float x) {
  return fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x)));
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + __expf(-x)); }

}  // namespace kda
