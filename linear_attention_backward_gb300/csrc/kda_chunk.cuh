// kda_chunk.cuh -- per-chunk preparation shared by the scan and gradient
// kernels: L2 norms, the gate log-decay and its within-chunk running sum, the
// decay-scaled operand tiles, the intra-chunk pair matrices (Akk, Mqk) and the
// WY / UT inverse (I + Akk)^-1.
//
// Names follow the kernel-B guide ("bwd-kernelB-beginner-guide-full", Part 2):
//   qd = q^ e^gc, kd = k^ e^gc, kr = k^ e^(gT - gc)   (R1 reconstruction in B1)
// and the intra-chunk products q^_i . k^_j e^(gc_i - gc_j) (j <= i).
//
// Range safety.  gc reaches -200 and below within a chunk, so e^-gc is not
// representable in fp32 and a plain q e^gc . (k e^-gc) product overflows.
// The chunk is cut into four 16-row blocks; block I has the reference gate
// m_I = gc[16 I + 7] (per channel), and every intra-chunk product between
// rows i in block I and j in block J <= I is formed as
//   (x_i e^(gc_i - m_I)) * F_IJ * (z_j e^(m_J - gc_j)),   F_IJ = e^(m_I - m_J) <= 1
// so that no factor exceeds e^(decay over 8 tokens).  (The pages work at the
// same 16-row granularity: guide Part 2, B3 optimisation 7, the K = 16
// contraction and the 16-row reverse cumsum.)
#pragma once

#include <type_traits>

#include "kda_device.cuh"
#include "kda_params.h"

namespace kda {

// Gate arithmetic by input type.  fp32 inputs are held to 1e-4 relative
// error, so their gate path takes the accurate softplus and exponential (the
// fast exponential's error bound grows with |x|, and gate exponents reach
// tens of nats); bf16 operands are rounded to 2^-9, far above either fast
// form's error, and keep the fast ones.
template <typename E> __device__ __forceinline__ float gate_exp(float x) {
  if constexpr (std::is_same<E, float>::value) return expf(x);
  else return __expf(x);
}
template <typename E> __device__ __forceinline__ float gate_softplus(float x) {
  if constexpr (std::is_same<E, float>::value) return softplus_f(x);
  else return softplus_gate(x);
}


// Mean log-decay per token, on every channel of a chunk, past which the
// block-factored dg leaves the input type's tolerance (kda_device.cuh): fp32
// inputs are held to 1e-4 (dg's error measured 1.2e-5 at 4 nats per token,
// 1.1e-4 at 6), bf16 to 2e-2 (3.5e-3 at 6, 3.1e-2 at 8 on the tcgen05 kernels).
template <typename E> __host__ __device__ constexpr float sustained_decay_limit() {
  return std::is_same<E, float>::value ? 5.f : kStrongTokenDecay;
}

// Bounds of sequence s.  Returns false (and flags the device status) on a
// malformed cu_seqlens entry.
__device__ __forceinline__ bool seq_bounds(const KdaParams &p, int s, int64_t &tok0, int &L,
                                           int64_t &slot0) {
  if (p.cu == nullptr) {
    tok0 = (int64_t)s * p.T;
    L = p.T;
    slot0 = (int64_t)s * p.nps;
    return true;
  }
  const int a = p.cu[s], b = p.cu[s + 1];
  if (a < 0 || b < a || b > p.T || (s == 0 && a != 0) || (s == p.num_seqs - 1 && b != p.T)) {
    set_status(6);
    return false;
  }
  tok0 = a;
  L = b - a;
  slot0 = (int64_t)(a / CHUNK) + s;
  return true;
}

// Inverse of the slot map: the sequence and chunk index that own `slot`.
// The gate's bias for head h, channel c (zero without one): the gate is
// gk = -exp(A_log[h]) * softplus(g + dt_bias[h][c]).
__device__ __forceinline__ float gate_bias(const KdaParams &p, int h, int c, int K) {
  return p.dt_bias != nullptr ? p.dt_bias[h * K + c] : 0.f;
}

__device__ __forceinline__ bool slot_owner(const KdaParams &p, int64_t slot, int &s, int &j,
                                           int64_t &tok0, int &len) {
  int64_t t0;
  int L;
  int64_t s0;
  if (p.cu == nullptr) {
    // slots number fewer than 2^31 (B * T <= 2^31 tokens): 32-bit division
    // (the 64-bit one is a subroutine call)
    const uint32_t sl = (uint32_t)slot, nps = (uint32_t)p.nps;
    s = (int)(sl / nps);
    j = (int)(sl - (uint32_t)s * nps);
    if (s >= p.B) return false;
  } else {
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {  // largest s with floor(cu[s]/64) + s <= slot
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)(p.cu[mid] / CHUNK) + mid <= slot) lo = mid; else hi = mid - 1;
    }
    s = lo;
  }
  if (!seq_bounds(p, s, t0, L, s0)) return false;
  j = (int)(slot - s0);
  if (j < 0 || (int64_t)j * CHUNK >= L) return false;
  tok0 = t0 + (int64_t)j * CHUNK;
  len = min(CHUNK, L - j * CHUNK);
  return true;
}

// ---------------------------------------------------------------------------
// Asynchronous staging of the chunk's raw rows into shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
  // src-size 0 fills the 16 bytes with zeros (phantom rows)
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
               "l"(gmem), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }

// Rows [0, 64) of the head-h slice of a token-major [*, H, D] tensor starting
// at token tok0, columns [col0, col0 + ncols), into dst (row stride ld
// elements).  Rows >= len are zero-filled; their source is never read.
template <typename E>
__device__ __forceinline__ void stage_rows(E *dst, int ld, const void *src, int64_t tok0, int len,
                                           int H, int h, int D, int col0, int ncols) {
  constexpr int EPC = 16 / sizeof(E);  // elements per 16-byte chunk
  const int cpr = ncols / EPC;          // chunks per row
  const E *base = reinterpret_cast<const E *>(src);
  for (int e = threadIdx.x; e < CHUNK * cpr; e += NTHREADS) {
    const int i = e / cpr, c = (e % cpr) * EPC;
    const bool valid = i < len;
    const E *g = base + ((tok0 + (valid ? i : 0)) * H + h) * (int64_t)D + col0 + c;
    cp_async16(dst + i * ld + c, g, valid);
  }
}

// A dense row-major [rows][cols] matrix (row stride cols) into dst (row
// stride ld elements).
template <typename E>
__device__ __forceinline__ void stage_dense(E *dst, int ld, const E *src, int rows, int cols) {
  constexpr int EPC = 16 / sizeof(E);
  const int cpr = cols / EPC;
  for (int e = threadIdx.x; e < rows * cpr; e += NTHREADS) {
    const int r = e / cpr, c = (e % cpr) * EPC;
    cp_async16(dst + r * ld + c, src + (int64_t)r * cols + c, true);
  }
}

// L2 prefetch of the same rows (used for the next chunk of a serial scan).
__device__ __forceinline__ void prefetch_rows_l2(const void *src, int64_t tok0, int len, int H,
                                                 int h, int rowbytes, int elem, int D,
                                                 int col0) {
  const char *base = reinterpret_cast<const char *>(src);
  const int lines = (rowbytes + 127) / 128;
  for (int e = threadIdx.x; e < len * lines; e += NTHREADS) {
    const int i = e / lines, l = e % lines;
    const char *ptr = base + (((tok0 + i) * H + h) * (int64_t)D + col0) * elem + 128 * l;
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(ptr));
  }
}

// ---------------------------------------------------------------------------
// Shared-memory views used by the prep.
// ---------------------------------------------------------------------------
template <typename E, int K> struct PrepView {
  float *m;       // [4][K]   scratch (block partial sums of the gate)
  float *em;      // [4][K]   e^(m_I)
  float *egm;     // [4][K]   e^(gT - m_I)
  float *F;       // [6][K]   e^(m_I - m_J), J < I, pair index I(I-1)/2 + J
  float *gT;      // [K]
  float *rq, *rk; // [64] 1 / sqrt(|x|^2 + eps)
  float *beta;    // [64]
  float *part;    // [2 NTHREADS / K][K] column partial sums (scratch)
  static constexpr int LDF = K + 4;
  static constexpr int LD = tile_ld<E>(K);
  static constexpr size_t floats = 19 * K + 3 * 64 + 2 * NTHREADS;
};

template <typename E, int K>
__device__ __forceinline__ PrepView<E, K> make_view(float *s) {
  PrepView<E, K> v;
  v.m = s;
  v.em = s + 4 * K;
  v.egm = s + 8 * K;
  v.F = s + 12 * K;
  v.gT = s + 18 * K;
  v.rq = s + 19 * K;
  v.rk = v.rq + 64;
  v.beta = v.rk + 64;
  v.part = v.beta + 64;
  return v;
}

__device__ __forceinline__ int pair_index(int I, int J) { return I * (I - 1) / 2 + J; }

template <typename E> __device__ __forceinline__ const E *elem_ptr(const void *base, int64_t off) {
  return reinterpret_cast<const E *>(base) + off;
}

// Operand tiles the prep can build (nullptr = skip).  All [64][LD] of E.
template <typename E> struct PrepTiles {
  E *QM = nullptr;   // q^ e^(gc - m)
  E *KM = nullptr;   // k^ e^(gc - m)
  E *KP = nullptr;   // k^ e^(m - gc)
  E *KD = nullptr;   // k^ e^gc
  E *KR = nullptr;   // k^ e^(gT - gc)
  E *QD = nullptr;   // scale * q^ e^gc
  float *Et = nullptr;  // optional fp32 [64][LDF]: E = e^(gc - m)
};

// Stage the chunk's raw q (optional), k, g rows (cp.async, zero-filled past
// len) and beta; the caller waits (cp_async_wait_all + __syncthreads) before
// chunk_prep.
template <typename E, int K>
__device__ __forceinline__ void stage_chunk(const KdaParams &p, int h, int64_t tok0, int len,
                                            bool need_q, E *Qr, E *Kr, E *Gr, float *beta) {
  if (need_q) stage_rows<E>(Qr, K, p.q, tok0, len, p.H, h, K, 0, K);
  stage_rows<E>(Kr, K, p.k, tok0, len, p.H, h, K, 0, K);
  stage_rows<E>(Gr, K, p.g, tok0, len, p.H, h, K, 0, K);
  if (threadIdx.x < CHUNK)
    beta[threadIdx.x] =
        threadIdx.x < len ? to_f(elem_ptr<E>(p.beta, (tok0 + threadIdx.x) * p.H + h)[0]) : 0.f;
}

// Per-chunk prep from the staged raw rows.  Rows >= len are phantom rows:
// q = k = 0, beta = 0 and a zero log-decay, so they change nothing and the
// last real row's gc is gT.
template <typename E, int K>
__device__ void chunk_prep(const KdaParams &p, int h, int len, bool need_q, const E *Qr,
                           const E *Kr, const E *Gr, const PrepView<E, K> &sv,
                           const PrepTiles<E> &tiles, bool grads = false) {
  constexpr int LD = PrepView<E, K>::LD;
  constexpr int LDF = PrepView<E, K>::LDF;
  constexpr int PAIRS = K / 2;               // column pairs
  constexpr int PARTS = NTHREADS / PAIRS;    // row segments
  constexpr int ROWS = CHUNK / PARTS;        // rows per segment (16 or 8)
  static_assert(ROWS == 16 || ROWS == 8, "segment must tile the 16-row blocks");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float A = gate_exp<E>(p.A_log[h]);
  // 1. L2 norms: one warp per row, 4 (K = 128) or 2 (K = 64) channels per lane
  for (int i = warp; i < CHUNK; i += NWARPS) {
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int c = 2 * lane; c < K; c += 64) {
      const float2 kv = load2(Kr + i * K + c);
      sk = fmaf(kv.x, kv.x, fmaf(kv.y, kv.y, sk));
      if (need_q) {
        const float2 qv = load2(Qr + i * K + c);
        sq = fmaf(qv.x, qv.x, fmaf(qv.y, qv.y, sq));
      }
    }
    sk = warp_sum(sk);
    sq = warp_sum(sq);
    if (lane == 0) {
      sv.rk[i] = rsqrtf(sk + p.eps);
      sv.rq[i] = rsqrtf(sq + p.eps);
    }
  }
  // 2. gate log-decay and its running sum, two channels per thread, one
  //    ROWS-row segment per thread, held in registers as sums local to the
  //    segment.  Every exponent used below is formed from such local sums
  //    (gc - m_I within a block, and block partials for m_I - m_J and
  //    gT - m_I), never as a difference of two chunk-long sums, which would
  //    cost ~|gc| * 2^-24 of absolute accuracy.
  const int cp = tid % PAIRS, seg = tid / PAIRS;
  const int c = 2 * cp, r0 = seg * ROWS;
  const int I = r0 >> 4;  // 16-row block of this segment
  float g0[ROWS], g1[ROWS];
  float run0 = 0.f, run1 = 0.f;
  const float bias0 = gate_bias(p, h, c, K), bias1 = gate_bias(p, h, c + 1, K);
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    const int i = r0 + r;
    const float2 gv = load2(Gr + i * K + c);
    const bool ok = i < len;
    run0 += ok ? -A * gate_softplus<E>(gv.x + bias0) : 0.f;
    run1 += ok ? -A * gate_softplus<E>(gv.y + bias1) : 0.f;
    g0[r] = run0;
    g1[r] = run1;
  }
  // log-decay around the block's reference row 16 I + 7 that the block
  // factors carry: a whole block (rows 0..7 before it, 8..15 after it), or a
  // half block ending at it (rows 0..7) or starting after it (rows 8..15)
  if constexpr (ROWS == 16) {
    check_block_log_decay(fmaxf(fmaxf(g0[0] - g0[7], g0[7] - g0[ROWS - 1]),
                                fmaxf(g1[0] - g1[7], g1[7] - g1[ROWS - 1])));
  } else if ((r0 & 15) == 0) {
    check_block_log_decay(fmaxf(g0[0] - g0[ROWS - 1], g1[0] - g1[ROWS - 1]));
  } else {
    check_block_log_decay(fmaxf(-g0[ROWS - 1], -g1[ROWS - 1]));
  }
  // a channel that decays by at most the sustained-decay limit over the chunk
  // (below): set by step 3, read after its barrier
  __shared__ int weak_any;
  if (tid == 0) weak_any = 0;
  // block partials: Ablk = sum of rows 16I .. 16I+7 (through the reference
  // row), Bblk = rows 16I+8 .. 16I+15
  float *Ablk = sv.part, *Bblk = sv.m;  // [4][K] each (sv.m reused as scratch)
  if (ROWS == 16) {
    Ablk[I * K + c] = g0[7];
    Ablk[I * K + c + 1] = g1[7];
    Bblk[I * K + c] = g0[ROWS - 1] - g0[7];
    Bblk[I * K + c + 1] = g1[ROWS - 1] - g1[7];
  } else {
    float *dst = (r0 & 15) ? Bblk : Ablk;
    dst[I * K + c] = run0;
    dst[I * K + c + 1] = run1;
  }
  __syncthreads();
  // 3. per-(block, channel) factors from the block partials
  for (int e = tid; e < K; e += NTHREADS) {
    float a[4], bb[4];
#pragma unroll
    for (int L = 0; L < 4; ++L) {
      a[L] = Ablk[L * K + e];
      bb[L] = Bblk[L * K + e];
    }
    float before = 0.f, tot = 0.f;
#pragma unroll
    for (int L = 0; L < 4; ++L) tot += a[L] + bb[L];
#pragma unroll
    for (int L = 0; L < 4; ++L) {
      float after = bb[L];
#pragma unroll
      for (int L2 = L + 1; L2 < 4; ++L2) after += a[L2] + bb[L2];
      sv.em[L * K + e] = gate_exp<E>(before + a[L]);   // e^(m_L)
      sv.egm[L * K + e] = gate_exp<E>(after);       // e^(gT - m_L)
      before += a[L] + bb[L];
    }
#pragma unroll
    for (int I2 = 1; I2 < 4; ++I2)
#pragma unroll
      for (int J = 0; J < I2; ++J) {
        float d = bb[J] + a[I2];
#pragma unroll
        for (int L = J + 1; L < I2; ++L) d += a[L] + bb[L];
        sv.F[pair_index(I2, J) * K + e] = gate_exp<E>(d);  // e^(m_I - m_J)
      }
    sv.gT[e] = tot;
    if (-tot <= sustained_decay_limit<E>() * (float)len) weak_any = 1;
  }
  __syncthreads();
  // When every channel decays by more than the limit per token, the
  // block-factored products leave dg (then tiny) outside the tolerance of the
  // input type (measured on a GB300: fp32 dg error 1.1e-4 at 6 nats per token
  // on every channel, 6e-2 at 8); the gradient kernel (grads) reports it as a
  // range error.  The states the scans compute stay accurate.
  if (grads && tid == 0 && weak_any == 0 && len > 0) set_status(kStatusGateRange);
  // 4. operand tiles.  gc_i - m_I from the segment's local sums: the
  //    reference row 16I+7 lies in this segment (local index 7) unless the
  //    segment is the second half of its block, where it is the row just
  //    before the segment.
  const bool ref_here = (r0 & 15) == 0;
  const float ref0 = ref_here ? g0[7] : 0.f, ref1 = ref_here ? g1[7] : 0.f;
  const float em0 = sv.em[I * K + c], em1 = sv.em[I * K + c + 1];
  const float eg0 = sv.egm[I * K + c], eg1 = sv.egm[I * K + c + 1];
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    const int i = r0 + r;
    const float2 kv = load2(Kr + i * K + c);
    const float rk = sv.rk[i];
    const float kh0 = kv.x * rk, kh1 = kv.y * rk;
    const float d0 = g0[r] - ref0, d1 = g1[r] - ref1;
    const float e0 = gate_exp<E>(d0), e1 = gate_exp<E>(d1);
    const float ei0 = gate_exp<E>(-d0), ei1 = gate_exp<E>(-d1);
    if (tiles.KM) store2(tiles.KM + i * LD + c, kh0 * e0, kh1 * e1);
    if (tiles.KP) store2(tiles.KP + i * LD + c, kh0 * ei0, kh1 * ei1);
    if (tiles.KD) store2(tiles.KD + i * LD + c, (kh0 * e0) * em0, (kh1 * e1) * em1);
    if (tiles.KR) store2(tiles.KR + i * LD + c, (kh0 * ei0) * eg0, (kh1 * ei1) * eg1);
    if (need_q) {
      const float2 qv = load2(Qr + i * K + c);
      const float rq = sv.rq[i];
      const float qh0 = qv.x * rq, qh1 = qv.y * rq;
      if (tiles.QM) store2(tiles.QM + i * LD + c, qh0 * e0, qh1 * e1);
      if (tiles.QD)
        store2(tiles.QD + i * LD + c, p.scale * (qh0 * e0) * em0, p.scale * (qh1 * e1) * em1);
    }
    if (tiles.Et) {
      tiles.Et[i * LDF + c] = e0;
      tiles.Et[i * LDF + c + 1] = e1;
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Intra-chunk pair matrices.  Warps 0..3 form G (k-k, strictly lower, fp32)
// for row block I = warp; warps 4..7 (when Mqk != nullptr) form
// scale * Mqk (q-k, lower including the diagonal) for row block I = warp - 4.
// ---------------------------------------------------------------------------
template <typename E, int K>
__device__ void intra_pairs(const E *QM, const E *KM, const E *KP, const float *F, float *G,
                            int ldg, E *Mqk, int ldm, float scale) {
  constexpr int LD = tile_ld<E>(K);
  const int warp = threadIdx.x >> 5;
  const int I = warp & 3;
  const bool is_q = warp >= 4;
  if (is_q && Mqk == nullptr) return;
  const E *X = is_q ? QM : KM;
  for (int J = 0; J < 4; ++J) {
    float acc[2][4];
    zero_acc(acc);
    if (J <= I)
      warp_gemm<2, true, true>(acc, X + 16 * I * LD, LD, KP + 16 * J * LD, LD, K,
                               J < I ? F + pair_index(I, J) * K : nullptr);
    for_acc(acc, [&](int r, int c, float &v) {
      const int i = 16 * I + r, j = 16 * J + c;
      if (is_q)
        Mqk[i * ldm + j] = from_f<E>(j <= i ? scale * v : 0.f);
      else
        G[i * ldg + j] = j < i ? v : 0.f;
    });
  }
}

// ---------------------------------------------------------------------------
// WY / UT inverse: INV = (I + A)^-1 with A_ij = beta_i G_ij (j < i), all fp32.
// The four 16x16 diagonal blocks are inverted by forward substitution, one
// warp per block with one column per lane held in registers; the off-diagonal
// blocks follow by block forward substitution,
//   X_IJ = -X_II sum_{J <= L < I} A_IL X_LJ,
// one level (block row) at a time over all threads.  inv32 is [64][68] fp32
// scratch, tbuf holds 3 * 256 floats.  Output INV in E, [64][ldi].
// ---------------------------------------------------------------------------
// One level of the block forward substitution: block row I, all J < I.
// Thread t owns row r = t / 4 % 16 and columns 4 (t % 4) .. + 4 of one J
// block; X rows are read as float4, G rows once per thread.
template <int I>
__device__ __forceinline__ void inv_level(const float *G, int ldg, const float *beta,
                                          float *inv32, float *tbuf) {
  constexpr int L32 = 68;
  const int tid = threadIdx.x;
  const int J = tid >> 6, r = (tid >> 2) & 15, c4 = 4 * (tid & 3);
  const int row = 16 * I + r;
  if (J < I) {
    const float *grow = G + row * ldg;
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int Lb = 0; Lb < I; ++Lb) {
      if (Lb < J) continue;
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const float gv = grow[16 * Lb + x];
        const float4 xv = *reinterpret_cast<const float4 *>(inv32 + (16 * Lb + x) * L32 + 16 * J + c4);
        t.x = fmaf(gv, xv.x, t.x);
        t.y = fmaf(gv, xv.y, t.y);
        t.z = fmaf(gv, xv.z, t.z);
        t.w = fmaf(gv, xv.w, t.w);
      }
    }
    const float br = beta[row];
    *reinterpret_cast<float4 *>(tbuf + (J << 8) + (r << 4) + c4) =
        make_float4(br * t.x, br * t.y, br * t.z, br * t.w);
  }
  __syncthreads();
  if (J < I) {
    const float *xr = inv32 + row * L32 + 16 * I;
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int x = 0; x < 16; ++x) {
      const float xv = xr[x];
      const float4 tv = *reinterpret_cast<const float4 *>(tbuf + (J << 8) + (x << 4) + c4);
      t.x = fmaf(xv, tv.x, t.x);
      t.y = fmaf(xv, tv.y, t.y);
      t.z = fmaf(xv, tv.z, t.z);
      t.w = fmaf(xv, tv.w, t.w);
    }
    *reinterpret_cast<float4 *>(inv32 + row * L32 + 16 * J + c4) =
        make_float4(-t.x, -t.y, -t.z, -t.w);
  }
  __syncthreads();
}

template <typename E>
__device__ void wy_inverse(const float *G, int ldg, const float *beta, float *inv32, float *tbuf,
                           E *inv, int ldi) {
  constexpr int L32 = 68;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // zero everything above the diagonal blocks
  for (int e = tid; e < 64 * 64; e += NTHREADS) {
    const int r = e >> 6, c = e & 63;
    if ((c >> 4) > (r >> 4)) inv32[r * L32 + c] = 0.f;
  }
  if (warp < 4) {
    const int o = 16 * warp, col = lane & 15;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float br = beta[o + r];
      const float *grow = G + (o + r) * ldg + o;
      float s0 = (r == col) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
      for (int j = 0; j < r; ++j) {
        if (j & 1)
          s1 = fmaf(-br * grow[j], x[j], s1);
        else
          s0 = fmaf(-br * grow[j], x[j], s0);
      }
      x[r] = s0 + s1;
    }
    if (lane < 16) {
#pragma unroll
      for (int r = 0; r < 16; ++r) inv32[(o + r) * L32 + o + col] = x[r];
    }
  }
  __syncthreads();
  inv_level<1>(G, ldg, beta, inv32, tbuf);
  inv_level<2>(G, ldg, beta, inv32, tbuf);
  inv_level<3>(G, ldg, beta, inv32, tbuf);
  for (int e = tid; e < 64 * 32; e += NTHREADS) {
    const int r = e >> 5, cc = 2 * (e & 31);
    store2(inv + r * ldi + cc, inv32[r * L32 + cc], inv32[r * L32 + cc + 1]);
  }
  __syncthreads();
}

}  // namespace kda
