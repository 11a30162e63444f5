// kda_tc_tiles.cuh -- shared-memory tile helpers for the tcgen05 kernels:
// element access in the padded core-matrix layout, tcgen05 operand
// descriptors for tiles read K-major or MN-major, and mma.sync products on
// the same padded tiles (used for the small 16-row pair blocks).
#pragma once

#include "kda_umma.cuh"

namespace kda {
namespace tct {

using umma::pcore_off;
constexpr uint32_t CS = umma::kCoreStride;  // padded core stride (144 bytes)
constexpr uint32_t CP = 128;                // packed core stride


__device__ __forceinline__ bf16 *pel(void *t, int r, int c, int C) {
  return reinterpret_cast<bf16 *>(reinterpret_cast<char *>(t) + pcore_off(r, c, C));
}
__device__ __forceinline__ float pget(const void *t, int r, int c, int C) {
  return __bfloat162float(
      *reinterpret_cast<const bf16 *>(reinterpret_cast<const char *>(t) + pcore_off(r, c, C)));
}
// 8 consecutive columns c0 .. c0 + 7 (c0 % 8 == 0) of row r, one 16-byte store
__device__ __forceinline__ void pstore8(void *t, int r, int c0, int C, const float *v) {
  __nv_bfloat162 h[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) h[q] = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
  *reinterpret_cast<uint4 *>(reinterpret_cast<char *>(t) + pcore_off(r, c0, C)) =
      *reinterpret_cast<uint4 *>(h);
}
__device__ __forceinline__ void pload8(const void *t, int r, int c0, int C, float *v) {
  const uint4 u =
      *reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(t) + pcore_off(r, c0, C));
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __bfloat1622float2(h[q]);
    v[2 * q] = f.x;
    v[2 * q + 1] = f.y;
  }
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}
__device__ __forceinline__ uint32_t f2_to_bf2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}
// Four consecutive fp32 values from shared memory, one 16-byte load (p must be
// 16-byte aligned); used for per-row vectors such as the row norms and beta,
// which every lane of a warp reads at the same address
__device__ __forceinline__ void lds4(const float *p, float *v) {
  const float4 t = *reinterpret_cast<const float4 *>(p);
  v[0] = t.x;
  v[1] = t.y;
  v[2] = t.z;
  v[3] = t.w;
}

// Sums over the warp's 32 lanes of each of 16 per-lane values (a row each):
// lanes 2 r and 2 r + 1 return the sum of row r.  Four halving steps exchange
// 8, 4, 2 and 1 values (a lane keeps the half of the rows that its bit 4, 3,
// 2, 1 selects and sends the other), then lanes 2 r, 2 r + 1 add their two
// partial sums: 16 shuffles in all.  v is consumed.
__device__ __forceinline__ float rows16_sum(float (&v)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const int n = 8 >> st, s = 16 >> st;
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int k = 0; k < n; ++k) {
      const float send = up ? v[k] : v[k + n];
      const float keep = up ? v[k + n] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// 8 fp32 -> one 16-byte row of a packed core tile (global or shared)
__device__ __forceinline__ void st16_bf(void *dst, const float *v) {
  uint4 u;
  u.x = f2_to_bf2(v[0], v[1]);
  u.y = f2_to_bf2(v[2], v[3]);
  u.z = f2_to_bf2(v[4], v[5]);
  u.w = f2_to_bf2(v[6], v[7]);
  *reinterpret_cast<uint4 *>(dst) = u;
}
// one 16-byte row of 8 bf16 -> 8 fp32
__device__ __forceinline__ void ld16_bf(const void *src, float *v) {
  const uint4 u = *reinterpret_cast<const uint4 *>(src);
  const float2 a = bf2_to_f2(u.x), b = bf2_to_f2(u.y), c = bf2_to_f2(u.z), d = bf2_to_f2(u.w);
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  v[4] = c.x; v[5] = c.y; v[6] = d.x; v[7] = d.y;
}

// ---- tcgen05 operands -------------------------------------------------------
struct Op {
  uint32_t addr, lbo, sbo, step;
  uint32_t swz = 0;   // descriptor layout type (0: none, 2: 128-byte swizzle)
  uint32_t slab = 0;  // per > 0: K = 16 steps advance by `step` within a slab,
  uint32_t per = 0;   // `per` steps per slab, slabs `slab` bytes apart
};
// stored tile [R][C] read with K along its columns, from column k0
__device__ __forceinline__ Op opk(const void *t, int C, int k0 = 0, uint32_t cs = CS) {
  return Op{smem_u32(t) + (uint32_t)(k0 / 8) * cs, cs, (uint32_t)(C / 8) * cs, 2 * cs};
}
// stored tile [R][C] read with K along its rows, from row r0
__device__ __forceinline__ Op opmn(const void *t, int C, int r0 = 0, uint32_t cs = CS) {
  return Op{smem_u32(t) + (uint32_t)(r0 / 8) * (C / 8) * cs, (uint32_t)(C / 8) * cs, cs,
            2 * (uint32_t)(C / 8) * cs};
}
// a tile in the 128-byte swizzled layout (umma::sw128_off, 1024-byte
// aligned), read MN-major: slabs of 64 M / N columns slab_bytes apart, K
// down its rows (two 8-row atoms per K = 16 step)
__device__ __forceinline__ Op opsw_mn(const void *t, uint32_t slab_bytes) {
  return Op{smem_u32(t), slab_bytes, 1024u, 2048u, 2u};
}
// the same layout read K-major: K along the 128-byte rows (32 bytes per
// K = 16 step, four steps per slab), slabs of 64 K columns slab_bytes apart,
// M / N down the rows
__device__ __forceinline__ Op opsw_k(const void *t, uint32_t slab_bytes) {
  return Op{smem_u32(t), 16u, 1024u, 32u, 2u, slab_bytes, 4u};
}
// D (+)= A B^T over `ksteps` K = 16 steps, issued by one thread; a step
// advances the descriptors' start-address field by step >> 4.
__device__ __forceinline__ void gemm(uint32_t d, Op a, bool amn, Op b, bool bmn, int N, int ksteps,
                                     bool accumulate) {
  const uint32_t id = umma::idesc_bf16(128, N, amn, bmn);
  const uint64_t da = umma::smem_desc(a.addr, a.lbo, a.sbo) | ((uint64_t)a.swz << 61);
  const uint64_t db = umma::smem_desc(b.addr, b.lbo, b.sbo) | ((uint64_t)b.swz << 61);
  auto at = [](const Op &o, int s) {  // byte offset of K step s
    return o.per ? (uint32_t)(s / (int)o.per) * o.slab + (uint32_t)(s % (int)o.per) * o.step
                 : (uint32_t)s * o.step;
  };
  for (int s = 0; s < ksteps; ++s)
    umma::mma_bf16(d, da + (at(a, s) >> 4), db + (at(b, s) >> 4), id, accumulate || s > 0);
}

// Precomputed form of an operand: its descriptor, and the descriptor step
// (start address >> 4) per K = 16 step.
struct Desc {
  uint64_t d;
  uint32_t step;
};
__device__ __forceinline__ Desc mkdesc(Op o) {
  return Desc{umma::smem_desc(o.addr, o.lbo, o.sbo), o.step >> 4};
}
// the descriptor of the same operand shifted by `bytes` (a multiple of 16)
__device__ __forceinline__ uint64_t dshift(const Desc &o, uint32_t bytes) {
  return o.d + (bytes >> 4);
}
// one K = 16 MMA from precomputed descriptors
__device__ __forceinline__ void mma1(uint32_t d, uint64_t da, uint64_t db, uint32_t idesc,
                                     bool accumulate) {
  umma::mma_bf16(d, da, db, idesc, accumulate);
}

// ---- mma.sync on padded core tiles (pair matrices) ---------------------------
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
// acc (16 x 8 NF) += A (16 x kdim) B (kdim x 8 NF); A(m, k) = tile A[ar0 + m][ac0 + k],
// B(k, n) = tile B[br0 + n][bc0 + k]; both K-contiguous tiles; kscale per k.
// The fragments of step k + 16 are loaded before the MMAs of step k are
// issued (the loads and MMAs are ordered asm statements), so that no MMA waits
// on the shared-memory latency of its own operands.
template <int NF>
__device__ __forceinline__ void wg_core(float (&acc)[NF][4], const void *A, int AC, int ar0,
                                        int ac0, const void *B, int BC, int br0, int bc0,
                                        int kdim, const float *kscale) {
  const int lane = threadIdx.x & 31;
  const uint32_t a0 = smem_u32(A), b0 = smem_u32(B);
  uint32_t af[2][4], bfr[2][NF / 2][4];
  auto load = [&](int k0, int buf) {
    ldsm4(af[buf], a0 + pcore_off(ar0 + (lane & 15), ac0 + k0 + (lane >> 4) * 8, AC));
#pragma unroll
    for (int f = 0; f < NF; f += 2)
      ldsm4(bfr[buf][f / 2], b0 + pcore_off(br0 + f * 8 + (lane & 7) + (lane >> 4) * 8,
                                            bc0 + k0 + ((lane >> 3) & 1) * 8, BC));
  };
  load(0, 0);
#pragma unroll
  for (int k0 = 0; k0 < kdim; k0 += 16) {
    const int cur = (k0 >> 4) & 1;
    if (k0 + 16 < kdim) load(k0 + 16, cur ^ 1);
    uint32_t a[4] = {af[cur][0], af[cur][1], af[cur][2], af[cur][3]};
    if (kscale != nullptr) {
      const int c = k0 + 2 * (lane & 3);  // even: 8-byte pairs (kscale is 8-byte aligned)
      const float2 s01 = *reinterpret_cast<const float2 *>(kscale + c);
      const float2 s89 = *reinterpret_cast<const float2 *>(kscale + c + 8);
      a[0] = scale_pair(a[0], s01.x, s01.y);
      a[1] = scale_pair(a[1], s01.x, s01.y);
      a[2] = scale_pair(a[2], s89.x, s89.y);
      a[3] = scale_pair(a[3], s89.x, s89.y);
    }
#pragma unroll
    for (int f = 0; f < NF; f += 2) {
      mma_16816(acc[f], a, bfr[cur][f / 2][0], bfr[cur][f / 2][1]);
      mma_16816(acc[f + 1], a, bfr[cur][f / 2][2], bfr[cur][f / 2][3]);
    }
  }
}

// fp32 -> tf32 (round to nearest, ties away) and one mma.m16n8k8 tf32 step:
// acc (16 x 8, fp32) += A (16 x 8) B (8 x 8), register fragments of the PTX
// ISA's m16n8k8 layouts (g = lane / 4, t = lane % 4): a = A[g][t], A[g+8][t],
// A[g][t+4], A[g+8][t+4]; b = B[t][g], B[t+4][g]; acc = C[g][2t], C[g][2t+1],
// C[g+8][2t], C[g+8][2t+1].
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float (&acc)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Row stride (floats) of the fp32 G / INV tile: 68, so that the 8 rows a
// warp reads at once in the block levels fall on different banks.
constexpr int kGfStride = 68;
// Gf [64][kGfStride] fp32 holds G (strictly lower) on entry and
// (I + diag(beta) G)^-1 on exit (block forward substitution in place, as
// wy_inverse in kda_chunk.cuh).  While warps 0-3 invert the diagonal blocks,
// warps 4 and up run side(warp - 4) (independent work of the caller's that
// touches neither Gf nor tbuf).
template <typename Side>
__device__ inline void inverse_inplace(float *Gf, const float *beta, float *tbuf, Side side) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int LG = kGfStride;
  if (warp >= 4) side(warp - 4);
  if (warp < 4) {
    const int o = 16 * warp, col = lane & 15;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      // x_r = e_r - beta_r sum_{j < r} G_rj x_j, the row's G entries by
      // 16-byte loads (rows are 16-byte aligned: kGfStride = 68)
      const float br = beta[o + r];
      const float *grow = Gf + (o + r) * LG + o;
      float g16[16];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (4 * q < r) lds4(grow + 4 * q, g16 + 4 * q);
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int j = 0; j < r; ++j) {
        if (j & 1)
          s1 = fmaf(g16[j], x[j], s1);
        else
          s0 = fmaf(g16[j], x[j], s0);
      }
      x[r] = fmaf(-br, s0 + s1, (r == col) ? 1.f : 0.f);
    }
    __syncwarp();
    if (lane < 16) {
#pragma unroll
      for (int r = 0; r < 16; ++r) Gf[(o + r) * LG + o + col] = x[r];
    }
  }
  __syncthreads();
  // Block levels, X_IJ = -X_II diag(beta_I) sum_{L=J}^{I-1} G_IL X_LJ, on the
  // tensor cores: warp J < I takes block (I, J) with mma.m16n8k8 tf32 (fp32
  // accumulation).  tf32 operands round to 2^-11, finer than the bf16 in
  // which the inverse is used.
  // The sum runs over L = 0 .. I - 1 for every J: the blocks X_LJ above the
  // diagonal (L < J) hold zeros, so the extra terms vanish and each level's
  // terms are a fixed, fully unrolled set whose loads overlap.
  const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int I = 1; I < 4; ++I) {
    float *tw = tbuf + warp * 256;  // this warp's 16 x 16 scratch
    if (warp < I) {
      const int J = warp;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int L = 0; L < I; ++L) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const float *ga = Gf + (16 * I + gid) * LG + 16 * L + 8 * kk + tig;
          const uint32_t af[4] = {to_tf32(ga[0]), to_tf32(ga[8 * LG]), to_tf32(ga[4]),
                                  to_tf32(ga[8 * LG + 4])};
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const float *xb = Gf + (16 * L + 8 * kk + tig) * LG + 16 * J + 8 * nt + gid;
            const uint32_t bf[2] = {to_tf32(xb[0]), to_tf32(xb[4 * LG])};
            mma_tf32(acc[nt], af, bf);
          }
        }
      }
      // T' = diag(beta_I) T into the scratch (row-major 16 x 16)
      const float b0 = beta[16 * I + gid], b8 = beta[16 * I + gid + 8];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        tw[gid * 16 + 8 * nt + 2 * tig] = b0 * acc[nt][0];
        tw[gid * 16 + 8 * nt + 2 * tig + 1] = b0 * acc[nt][1];
        tw[(gid + 8) * 16 + 8 * nt + 2 * tig] = b8 * acc[nt][2];
        tw[(gid + 8) * 16 + 8 * nt + 2 * tig + 1] = b8 * acc[nt][3];
      }
    }
    __syncthreads();  // every warp has read the G blocks of row I before any is overwritten
    if (warp < I) {
      const int J = warp;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const float *xa = Gf + (16 * I + gid) * LG + 16 * I + 8 * kk + tig;  // X_II
        const uint32_t af[4] = {to_tf32(xa[0]), to_tf32(xa[8 * LG]), to_tf32(xa[4]),
                                to_tf32(xa[8 * LG + 4])};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float *tb = tw + (8 * kk + tig) * 16 + 8 * nt + gid;
          const uint32_t bf[2] = {to_tf32(tb[0]), to_tf32(tb[4 * 16])};
          mma_tf32(acc[nt], af, bf);
        }
      }
      float *xo = Gf + (16 * I + gid) * LG + 16 * J;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        xo[8 * nt + 2 * tig] = -acc[nt][0];
        xo[8 * nt + 2 * tig + 1] = -acc[nt][1];
        xo[8 * LG + 8 * nt + 2 * tig] = -acc[nt][2];
        xo[8 * LG + 8 * nt + 2 * tig + 1] = -acc[nt][3];
      }
    }
    __syncthreads();
  }
}

// Row sums over the warp's 32 lanes for 32 rows at once: lane l returns
// sum over lanes of v[l] (31 shuffles instead of 32 x 5); v is consumed.
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int k = 0; k < s; ++k) {
      const float send = up ? v[k] : v[k + s];
      const float keep = up ? v[k + s] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return v[0];
}

// TMEM address of this thread's lane (warp quarter) at column col
__device__ __forceinline__ uint32_t tm(uint32_t tbase, int col) {
  return tbase + ((uint32_t)(32 * ((threadIdx.x >> 5) & 3)) << 16) + (uint32_t)col;
}
// this thread's 32 columns [col0 + 32 g, +32) of its lane
__device__ __forceinline__ void tld32(uint32_t tbase, int col0, float (&v)[32]) {
  const int g = threadIdx.x >> 7;
  float a[16], b[16];
  umma::tmem_ld16(tm(tbase, col0 + 32 * g), a);
  umma::tmem_ld16(tm(tbase, col0 + 32 * g + 16), b);
  umma::tmem_ld_wait();
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    v[q] = a[q];
    v[16 + q] = b[q];
  }
}

}  // namespace tct
}  // namespace kda
