// kda_scan.cu -- the two serial chunk scans of the KDA backward, one CTA per
// (sequence, head, V band):
//
//  * forward role: the chunk-state recompute ("all_states", read by kernel
//    B2 in "bwd-kernelB-beginner-guide-full", Part 2, B2 optimisation 4)
//      U       = (I + Akk)^-1 diag(beta) (v - kd S_n)            (v_new)
//      S_{n+1} = diag(e^gT) S_n + kr^T U
//  * backward role: Kernel A, the reverse scan of the per-chunk state
//    gradient ("bwd-ncu-and-optimization-playbook", A/B table; guide Part 2,
//    B1 for dU and dvcorr)
//      dU      = scale Mqk^T dO + kr dS_{n+1}
//      dvcorr  = (I + Akk)^-T dU
//      dS_n    = diag(e^gT) dS_{n+1} + scale qd^T dO - kd^T diag(beta) dvcorr
//
// Both recurrences are column-separable in V, so the V axis is split into
// bands (the split-V grid (N, H, VSplit) of the playbook, section 3.5); every
// band recomputes the chunk prep.  The two roles do not depend on each other
// and run side by side in one launch (blockIdx.y = role).  The running state
// stays in registers (mma accumulators) across chunks: warp w owns state rows
// [16 (w % (K/16)), +16).
#include "kda_chunk.cuh"

namespace kda {

template <typename E, int K, int BV> struct ScanSmem {
  static constexpr int LD = tile_ld<E>(K);
  static constexpr int LDB = tile_ld<E>(BV);
  static constexpr size_t cmax(size_t a, size_t b) { return a > b ? a : b; }
  static constexpr size_t sz_small = ((PrepView<E, K>::floats * 4 + 127) / 128) * 128;
  static constexpr size_t sz_raw = 3 * 64 * K * sizeof(E);
  static constexpr size_t sz_tile = 64 * LD * sizeof(E);
  static constexpr size_t sz_band = 64 * LDB * sizeof(E);
  static constexpr size_t sz_G = 64 * 68 * 4;
  static constexpr size_t sz_sq = 64 * tile_ld<E>(64) * sizeof(E);
  static constexpr size_t sz_state = K * LDB * sizeof(E);
  // offsets
  static constexpr size_t o_small = 0;
  static constexpr size_t o_raw = o_small + sz_small;     // raw q, k, g (next chunk's
                                                          // land here during the chain)
  static constexpr size_t o_G = o_raw + sz_raw;           // G, later W
  static constexpr size_t o_QM = o_G + cmax(sz_G, sz_band);
  static constexpr size_t o_KM = o_QM + sz_tile;          // QM, KM, KP; later inverse
  static constexpr size_t o_KP = o_KM + sz_tile;          // scratch, then state + U
  static constexpr size_t o_KD = o_KP + sz_tile;
  static constexpr size_t o_KR = o_KD + sz_tile;
  static constexpr size_t o_QD = o_KR + sz_tile;
  static constexpr size_t o_INV = o_QD + sz_tile;
  static constexpr size_t o_MQK = o_INV + sz_sq;
  static constexpr size_t o_BAND = o_MQK + sz_sq;         // v band (fwd) / dO band (bwd)
  static constexpr size_t total = o_BAND + sz_band;
  static constexpr size_t o_W = o_G;
  static constexpr size_t o_STATE = o_QM;
  static constexpr size_t o_U = o_QM + sz_state;
  static_assert(sz_state + sz_band <= 3 * sz_tile, "state + U must fit in QM/KM/KP");
  static_assert(64 * 68 * 4 + 768 * 4 <= 3 * sz_tile, "inverse scratch must fit in QM/KM/KP");
};

template <typename E, int K, int BV>
__global__ void __launch_bounds__(NTHREADS, 1) kda_scan_kernel(KdaParams p) {
  using SM = ScanSmem<E, K, BV>;
  extern __shared__ __align__(128) char smem[];
  constexpr int LD = SM::LD, LDB = SM::LDB;
  constexpr int WM = K / 16;          // warps along state rows
  constexpr int WN = NWARPS / WM;     // warps along the band columns
  constexpr int SCOLS = BV / WN;      // state columns per warp
  constexpr int NFS = SCOLS / 8;
  constexpr int NFC = BV / 16;        // chunk-row GEMMs: 4 row blocks x 2 column halves

  const int role = p.role_base + blockIdx.y;  // 0: forward states, 1: reverse dS scan
  const int unit = blockIdx.x;
  const int band = unit % p.nb;
  const int sh = unit / p.nb;
  const int h = sh % p.H, s = sh / p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H;
  int64_t tok_seq, slot0;
  int L;
  if (!seq_bounds(p, s, tok_seq, L, slot0)) return;
  const int nck = (L + CHUNK - 1) / CHUNK;
  const int v0 = band * BV;

  PrepView<E, K> sv = make_view<E, K>(reinterpret_cast<float *>(smem + SM::o_small));
  E *Qr = reinterpret_cast<E *>(smem + SM::o_raw);
  E *Kr = Qr + 64 * K;
  E *Gr = Kr + 64 * K;
  E *QM = reinterpret_cast<E *>(smem + SM::o_QM);
  E *KM = reinterpret_cast<E *>(smem + SM::o_KM);
  E *KP = reinterpret_cast<E *>(smem + SM::o_KP);
  E *KD = reinterpret_cast<E *>(smem + SM::o_KD);
  E *KR = reinterpret_cast<E *>(smem + SM::o_KR);
  E *QD = reinterpret_cast<E *>(smem + SM::o_QD);
  float *G = reinterpret_cast<float *>(smem + SM::o_G);
  E *W = reinterpret_cast<E *>(smem + SM::o_W);
  E *INV = reinterpret_cast<E *>(smem + SM::o_INV);
  E *MQK = reinterpret_cast<E *>(smem + SM::o_MQK);
  E *BAND = reinterpret_cast<E *>(smem + SM::o_BAND);
  E *ST = reinterpret_cast<E *>(smem + SM::o_STATE);
  E *UB = reinterpret_cast<E *>(smem + SM::o_U);
  float *inv32 = reinterpret_cast<float *>(smem + SM::o_QM);
  float *tbuf = inv32 + 64 * 68;

  // state rows owned by this warp
  const int srow0 = 16 * (warp % WM);
  const int scol0 = SCOLS * (warp / WM);
  float S[NFS][4];
  const size_t KV = (size_t)K * (size_t)(BV * p.nb);
  const int Vtot = BV * p.nb;
  {
    const float *init = role == 0 ? p.h0 : p.dhT;
    for_acc(S, [&](int r, int c, float &x) {
      x = init ? init[((size_t)s * H + h) * KV + (size_t)(srow0 + r) * Vtot + v0 + scol0 + c] : 0.f;
    });
  }
  const int rb = warp & 3;            // chunk-row block of this warp
  const int ch = (warp >> 2) * (BV / 2);  // column half of the band

  const void *bsrc = role == 0 ? p.v : p.dO;
  const int es = sizeof(E);
  auto chunk_rows = [&](int jj, int64_t &t0, int &ln) {
    t0 = tok_seq + (int64_t)jj * CHUNK;
    ln = min(CHUNK, L - jj * CHUNK);
  };
  // Pipeline: the raw q / k / g rows of chunk j+1 are copied (cp.async)
  // while chunk j's intra products, inverse and chain run; the v / dO band
  // of chunk j+1 while... after chunk j's chain.  Commit groups alternate
  // raw(j), band(j), raw(j+1), band(j+1), ...
  if (nck > 0) {
    int64_t t0;
    int ln;
    chunk_rows(role == 0 ? 0 : nck - 1, t0, ln);
    stage_chunk<E, K>(p, h, t0, ln, role == 1, Qr, Kr, Gr, sv.beta);
    cp_async_commit();
    stage_rows<E>(BAND, LDB, bsrc, t0, ln, H, h, Vtot, v0, BV);
    cp_async_commit();
  }
  float beta_next = 0.f;
  for (int it = 0; it < nck; ++it) {
    const int j = role == 0 ? it : nck - 1 - it;
    const int jn = role == 0 ? j + 1 : j - 1;
    int64_t tok0;
    int len;
    chunk_rows(j, tok0, len);
    const int64_t slot = slot0 + j;
    if (it + 2 < nck) {  // warm L2 for the chunk after next
      int64_t t2;
      int l2;
      chunk_rows(role == 0 ? j + 2 : j - 2, t2, l2);
      prefetch_rows_l2(p.k, t2, l2, H, h, K * es, es, K, 0);
      prefetch_rows_l2(p.g, t2, l2, H, h, K * es, es, K, 0);
      prefetch_rows_l2(bsrc, t2, l2, H, h, BV * es, es, Vtot, v0);
      if (role == 1) prefetch_rows_l2(p.q, t2, l2, H, h, K * es, es, K, 0);
    }
    if (it > 0 && tid < CHUNK) sv.beta[tid] = beta_next;  // chunk j's beta
    asm volatile("cp.async.wait_group 1;\n" ::);  // raw(j) has landed
    __syncthreads();
    PrepTiles<E> tl;
    tl.KM = KM;
    tl.KP = KP;
    tl.KD = KD;
    tl.KR = KR;
    if (role == 1) {
      tl.QM = QM;
      tl.QD = QD;
    }
    chunk_prep<E, K>(p, h, len, role == 1, Qr, Kr, Gr, sv, tl);
    if (it + 1 < nck) {
      int64_t tn;
      int ln;
      chunk_rows(jn, tn, ln);
      if (role == 1) stage_rows<E>(Qr, K, p.q, tn, ln, H, h, K, 0, K);
      stage_rows<E>(Kr, K, p.k, tn, ln, H, h, K, 0, K);
      stage_rows<E>(Gr, K, p.g, tn, ln, H, h, K, 0, K);
      if (tid < CHUNK)  // beta(j+1) waits in a register until chunk j is done
        beta_next = tid < ln ? to_f(elem_ptr<E>(p.beta, (tn + tid) * H + h)[0]) : 0.f;
    }
    cp_async_commit();
    intra_pairs<E, K>(QM, KM, KP, sv.F, G, 68, role == 1 ? MQK : nullptr, tile_ld<E>(64), p.scale);
    __syncthreads();
    wy_inverse<E>(G, 68, sv.beta, inv32, tbuf, INV, tile_ld<E>(64));
    // publish the current state: to HBM (states / dstates) and to smem as an operand
    {
      E *dst = reinterpret_cast<E *>(role == 0 ? p.states : p.dstates) +
               ((size_t)slot * H + h) * (size_t)K * Vtot + v0;
      for_acc(S, [&](int r, int c, float &x) {
        ST[(srow0 + r) * LDB + scol0 + c] = from_f<E>(x);
      });
      asm volatile("cp.async.wait_group 1;\n" ::);  // band(j) has landed
      __syncthreads();
      for (int e = tid; e < K * BV / 2; e += NTHREADS) {
        const int r = e / (BV / 2), c = 2 * (e % (BV / 2));
        const float2 x = load2(ST + r * LDB + c);
        store2(dst + (size_t)r * Vtot + c, x.x, x.y);
      }
    }
    if (role == 0) {
      // kdS = kd S_n ; Xr = v - kdS  (in place in BAND)
      float acc[NFC][4];
      zero_acc(acc);
      warp_gemm<NFC, true, false>(acc, KD + 16 * rb * LD, LD, ST + ch, LDB, K);
      for_acc(acc, [&](int r, int c, float &x) {
        E *pv = BAND + (16 * rb + r) * LDB + ch + c;
        *pv = from_f<E>(to_f(*pv) - x);
      });
      __syncthreads();
      // U = INV diag(beta) Xr
      zero_acc(acc);
      warp_gemm<NFC, true, false>(acc, INV + 16 * rb * tile_ld<E>(64), tile_ld<E>(64), BAND + ch, LDB, 64,
                                  sv.beta);
      store_acc(UB + 16 * rb * LDB + ch, LDB, acc);
      __syncthreads();
      // S <- diag(e^gT) S + kr^T U
      for_acc(S, [&](int r, int c, float &x) { x *= gate_exp<E>(sv.gT[srow0 + r]); });
      warp_gemm<NFS, false, false>(S, KR + srow0, LD, UB + scol0, LDB, 64);
    } else {
      // dU = scale Mqk^T dO + kr dS
      float acc[NFC][4];
      zero_acc(acc);
      warp_gemm<NFC, false, false>(acc, MQK + 16 * rb, tile_ld<E>(64), BAND + ch, LDB, 64);
      warp_gemm<NFC, true, false>(acc, KR + 16 * rb * LD, LD, ST + ch, LDB, K);
      store_acc(UB + 16 * rb * LDB + ch, LDB, acc);
      __syncthreads();
      // dvcorr = INV^T dU ; W = -beta dvcorr
      zero_acc(acc);
      warp_gemm<NFC, false, false>(acc, INV + 16 * rb, tile_ld<E>(64), UB + ch, LDB, 64);
      for_acc(acc, [&](int r, int c, float &x) {
        W[(16 * rb + r) * LDB + ch + c] = from_f<E>(-sv.beta[16 * rb + r] * x);
      });
      __syncthreads();
      // dS <- diag(e^gT) dS + scale qd^T dO - kd^T diag(beta) dvcorr
      for_acc(S, [&](int r, int c, float &x) { x *= gate_exp<E>(sv.gT[srow0 + r]); });
      warp_gemm<NFS, false, false>(S, QD + srow0, LD, BAND + scol0, LDB, 64);
      warp_gemm<NFS, false, false>(S, KD + srow0, LD, W + scol0, LDB, 64);
    }
    __syncthreads();  // the band, beta and the chain's tiles are free again
    if (it + 1 < nck) {
      int64_t tn;
      int ln;
      chunk_rows(jn, tn, ln);
      stage_rows<E>(BAND, LDB, bsrc, tn, ln, H, h, Vtot, v0, BV);
    }
    cp_async_commit();
  }
  cp_async_wait_all();
  float *fin = role == 0 ? p.hT : p.dh0;
  if (fin != nullptr) {
    for_acc(S, [&](int r, int c, float &x) {
      fin[((size_t)s * H + h) * KV + (size_t)(srow0 + r) * Vtot + v0 + scol0 + c] = x;
    });
  }
  (void)lane;
}

template <typename E, int K, int BV>
static cudaError_t launch_scan(const KdaParams &p, int nroles, cudaStream_t st) {
  using SM = ScanSmem<E, K, BV>;
  auto kfn = kda_scan_kernel<E, K, BV>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SM::total);
  if (e != cudaSuccess) return e;
  const int nunits = (p.cu ? p.num_seqs : p.B) * p.H * p.nb;
  if (nunits == 0 || nroles == 0) return cudaSuccess;
  kfn<<<dim3(nunits, nroles), NTHREADS, SM::total, st>>>(p);
  return cudaGetLastError();
}

#define KDA_SCAN_CASES(X)            \
  X(bf16, 128, 128) X(bf16, 128, 64) \
  X(bf16, 128, 32) X(bf16, 64, 64)   \
  X(bf16, 64, 32) X(float, 64, 64)   \
  X(float, 64, 32)

cudaError_t scan_dispatch(const KdaParams &p, int K, bool is_bf16, int bv, int nroles,
                          cudaStream_t st) {
#define X(E, KK, BB)                                                          \
  if (is_bf16 == (sizeof(E) == 2) && K == KK && bv == BB)                     \
    return launch_scan<E, KK, BB>(p, nroles, st);
  KDA_SCAN_CASES(X)
#undef X
  return cudaErrorInvalidValue;
}

size_t scan_smem_bytes(int K, bool is_bf16, int bv) {
#define X(E, KK, BB)                                                          \
  if (is_bf16 == (sizeof(E) == 2) && K == KK && bv == BB) return ScanSmem<E, KK, BB>::total;
  KDA_SCAN_CASES(X)
#undef X
  return 0;
}

int scan_status_take() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_status, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

}  // namespace kda
