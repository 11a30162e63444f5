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

#include "kda_device.cuh"
#include "kda_params.h"

namespace kda {



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
__device__ __forceinline__ bool slot_owner(const KdaParams &p, int64_t slot, int &s, int &j,
                                           int64_t &tok0, int &len) {
  int64_t t0;
  int L;
  int64_t s0;
  if (p.cu == nullptr) {
    s = (int)(slot / p.nps);
    j = (int)(slot % p.nps);
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
// Shared-memory views used by the prep.
// ---------------------------------------------------------------------------
template <typename E, int K> struct PrepView {
  float *gc;      // [64][LDF] fp32: gk, then gc, then (optionally) E = e^(gc - m)
  float *m;       // [4][K]   block reference gates
  float *em;      // [4][K]   e^(m_I)
  float *egm;     // [4][K]   e^(gT - m_I)
  float *F;       // [6][K]   e^(m_I - m_J), J < I, pair index I(I-1)/2 + J
  float *gT;      // [K]
  float *rq, *rk; // [64] 1 / sqrt(|x|^2 + eps)
  float *beta;    // [64]
  static constexpr int LDF = K + 4;
  static constexpr int LD = tile_ld<E>(K);
};

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
  bool keep_E = false;  // leave E = e^(gc - m) in view.gc
};

// Per-chunk prep.  Rows >= len are phantom rows: q = k = 0, beta = 0 and a
// zero log-decay, so they change nothing and the last real row's gc is gT.
template <typename E, int K>
__device__ void chunk_prep(const KdaParams &p, int h, int64_t tok0, int len, bool need_q,
                           const PrepView<E, K> &sv, const PrepTiles<E> &tiles) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.H;
  const float A = __expf(p.A_log[h]);
  constexpr int LDF = PrepView<E, K>::LDF;
  constexpr int LD = PrepView<E, K>::LD;
  // 1. log-decay gk (fp32) and beta
  for (int e = tid; e < CHUNK * K; e += NTHREADS) {
    const int i = e / K, c = e % K;
    float gk = 0.f;
    if (i < len) {
      const float gv = to_f(elem_ptr<E>(p.g, ((tok0 + i) * H + h) * K)[c]);
      gk = -A * softplus_f(gv);
    }
    sv.gc[i * LDF + c] = gk;
  }
  if (tid < CHUNK)
    sv.beta[tid] = tid < len ? to_f(elem_ptr<E>(p.beta, (tok0 + tid) * H + h)[0]) : 0.f;
  // 2. L2 norms (one warp per row)
  for (int i = warp; i < CHUNK; i += NWARPS) {
    float sk = 0.f, sq = 0.f;
    if (i < len) {
      const E *kr = elem_ptr<E>(p.k, ((tok0 + i) * H + h) * K);
      const E *qr = elem_ptr<E>(p.q, ((tok0 + i) * H + h) * K);
      for (int c = lane; c < K; c += 32) {
        const float kv = to_f(kr[c]);
        sk = fmaf(kv, kv, sk);
        if (need_q) {
          const float qv = to_f(qr[c]);
          sq = fmaf(qv, qv, sq);
        }
      }
    }
    sk = warp_sum(sk);
    sq = warp_sum(sq);
    if (lane == 0) {
      sv.rk[i] = rsqrtf(sk + p.eps);
      sv.rq[i] = rsqrtf(sq + p.eps);
    }
  }
  __syncthreads();
  // 3. running sum over the chunk rows (one thread per channel)
  if (tid < K) {
    float run = 0.f;
    for (int i = 0; i < CHUNK; ++i) {
      run += sv.gc[i * LDF + tid];
      sv.gc[i * LDF + tid] = run;
      if ((i & 15) == 7) sv.m[(i >> 4) * K + tid] = run;
    }
    sv.gT[tid] = run;
  }
  __syncthreads();
  for (int e = tid; e < 4 * K; e += NTHREADS) {
    const int I = e / K, c = e % K;
    const float mI = sv.m[I * K + c];
    sv.em[e] = __expf(mI);
    sv.egm[e] = __expf(sv.gT[c] - mI);
  }
  for (int e = tid; e < 6 * K; e += NTHREADS) {
    const int pi = e / K, c = e % K;
    const int I = pi < 1 ? 1 : (pi < 3 ? 2 : 3);
    const int J = pi - pair_index(I, 0);
    sv.F[e] = __expf(sv.m[I * K + c] - sv.m[J * K + c]);
  }
  __syncthreads();
  // 4. operand tiles (two consecutive channels per thread)
  for (int e = tid; e < CHUNK * K / 2; e += NTHREADS) {
    const int i = e / (K / 2), c = 2 * (e % (K / 2));
    const int I = i >> 4;
    float kh0 = 0.f, kh1 = 0.f, qh0 = 0.f, qh1 = 0.f;
    if (i < len) {
      const float2 kv = load2(elem_ptr<E>(p.k, ((tok0 + i) * H + h) * K + c));
      kh0 = kv.x * sv.rk[i];
      kh1 = kv.y * sv.rk[i];
      if (need_q) {
        const float2 qv = load2(elem_ptr<E>(p.q, ((tok0 + i) * H + h) * K + c));
        qh0 = qv.x * sv.rq[i];
        qh1 = qv.y * sv.rq[i];
      }
    }
    const float gc0 = sv.gc[i * LDF + c], gc1 = sv.gc[i * LDF + c + 1];
    const float m0 = sv.m[I * K + c], m1 = sv.m[I * K + c + 1];
    const float e0 = __expf(gc0 - m0), e1 = __expf(gc1 - m1);
    const float ei0 = __expf(m0 - gc0), ei1 = __expf(m1 - gc1);
    const float em0 = sv.em[I * K + c], em1 = sv.em[I * K + c + 1];
    const float eg0 = sv.egm[I * K + c], eg1 = sv.egm[I * K + c + 1];
    if (tiles.QM) store2(tiles.QM + i * LD + c, qh0 * e0, qh1 * e1);
    if (tiles.KM) store2(tiles.KM + i * LD + c, kh0 * e0, kh1 * e1);
    if (tiles.KP) store2(tiles.KP + i * LD + c, kh0 * ei0, kh1 * ei1);
    if (tiles.KD) store2(tiles.KD + i * LD + c, (kh0 * e0) * em0, (kh1 * e1) * em1);
    if (tiles.KR) store2(tiles.KR + i * LD + c, (kh0 * ei0) * eg0, (kh1 * ei1) * eg1);
    if (tiles.QD)
      store2(tiles.QD + i * LD + c, p.scale * (qh0 * e0) * em0, p.scale * (qh1 * e1) * em1);
    if (tiles.keep_E) {
      sv.gc[i * LDF + c] = e0;
      sv.gc[i * LDF + c + 1] = e1;
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
// WY / UT inverse: INV = (I + A)^-1 with A_ij = beta_i G_ij (j < i), by 16x16
// diagonal-block forward substitution followed by block forward substitution
// for the off-diagonal blocks, all in fp32.  inv32 is [64][68] fp32 scratch,
// tbuf holds 3 * 256 floats.  Output INV in E, [64][tile_ld(64)].
// ---------------------------------------------------------------------------
template <typename E>
__device__ void wy_inverse(const float *G, int ldg, const float *beta, float *inv32, float *tbuf,
                           E *inv, int ldi) {
  constexpr int L32 = 68;
  const int tid = threadIdx.x;
  // zero everything above the diagonal blocks
  for (int e = tid; e < 64 * 64; e += NTHREADS) {
    const int r = e >> 6, c = e & 63;
    if ((c >> 4) > (r >> 4)) inv32[r * L32 + c] = 0.f;
  }
  if (tid < 64) {
    const int b = tid >> 4, c = tid & 15;
    const int o = 16 * b;
    for (int r = 0; r < 16; ++r) {
      float x = (r == c) ? 1.f : 0.f;
      const float br = beta[o + r];
      for (int j = c; j < r; ++j) x -= br * G[(o + r) * ldg + o + j] * inv32[(o + j) * L32 + o + c];
      inv32[(o + r) * L32 + o + c] = (r >= c) ? x : 0.f;
    }
  }
  __syncthreads();
  for (int I = 1; I < 4; ++I) {
    for (int e = tid; e < I * 256; e += NTHREADS) {
      const int J = e >> 8, r = (e >> 4) & 15, c = e & 15;
      const int row = 16 * I + r;
      const float br = beta[row];
      float t = 0.f;
      for (int Lb = J; Lb < I; ++Lb)
        for (int x = 0; x < 16; ++x)
          t = fmaf(br * G[row * ldg + 16 * Lb + x], inv32[(16 * Lb + x) * L32 + 16 * J + c], t);
      tbuf[e] = t;
    }
    __syncthreads();
    for (int e = tid; e < I * 256; e += NTHREADS) {
      const int J = e >> 8, r = (e >> 4) & 15, c = e & 15;
      float t = 0.f;
      for (int x = 0; x < 16; ++x)
        t = fmaf(inv32[(16 * I + r) * L32 + 16 * I + x], tbuf[(J << 8) + (x << 4) + c], t);
      inv32[(16 * I + r) * L32 + 16 * J + c] = -t;
    }
    __syncthreads();
  }
  for (int e = tid; e < 64 * 32; e += NTHREADS) {
    const int r = e >> 5, c = 2 * (e & 31);
    store2(inv + r * ldi + c, inv32[r * L32 + c], inv32[r * L32 + c + 1]);
  }
  __syncthreads();
}

}  // namespace kda
