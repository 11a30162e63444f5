// kda_grads_tc.cu -- per-chunk gradients of the KDA backward on the
// fifth-generation tensor cores (tcgen05, Tensor Memory), bf16, K = V = 128.
//
// The work per (chunk, head) is the same as kda_grads.cu (the B1 / B2 / B0 /
// B3 / K1 split of "bwd-kernelB-beginner-guide-full", Part 1, in one CTA), laid
// out for tcgen05: every large contraction is taken TRANSPOSED, with the
// channel (K or V = 128) dimension as the MMA's M, so that M = 128 and the
// result lands in Tensor Memory with lane = channel.  The CTA has 512
// threads (16 warps); thread t owns channel c = t % 128 and the 16-row block
// I = t / 128 of the chunk (rows 16 I .. 16 I + 15), reads exactly its lane
// and its 16 columns of every accumulator, keeps E = e^(gc - m_I) for its
// (i, c) in registers for the whole kernel, and runs the gate epilogue (the
// reverse cumulative sum over the chunk) over its block with the carry of
// the later blocks.
//
// Products (D = A B^T, A: 128 x K, B: N x K; tiles in the padded or packed
// core-matrix layout, "K" / "MN" = how the stored tile is read):
//   P1  kdS^T[d][i]   = S[c][d] (MN)            x kd[i][c] (K)          N = 64
//   P2  U^T[d][i]     = Xr^T[d][j] (K)          x INVb[i][j] (K)        N = 64
//   P3  dU^T[d][i]    = dO[i'][d] (MN) x Mqk[i'][i] (MN)
//                     + dS[c][d] (MN)  x kr[i][c] (K)                   N = 64
//       dkr^T[c][i]   = dS[c][d] (K)            x U[i][d] (K)           N = 64
//   P5  dvcorr^T[d][i]= dU^T[d][i'] (K)         x INV[i'][i] (MN)       N = 64
//   P6  [dO; dvcorr] U^T = [dMqk / s | -dAkk] (rows: dO, then dvcorr)   N = 64
//   P8  S [dO; dvcorr]^T = [dO S^T | dvcorr S^T]^T                     N = 128
// dO arrives by TMA as two 64-channel boxes in the 128-byte swizzled layout
// and is read as it lands: MN-major by P3a, and K-major, stacked over the
// dvcorr rows the R3 epilogue writes in the same layout, by P6 and P8.
//   P9  intra-chunk terms with hi + lo operands: per key block J the dMqk and
//       dA sides in one product (N = 128 - 32 J), per query block X the
//       P9c sums (N = 16 (X + 1))
// The pair matrices G = strict_lower(kd ki^T), scale Mqk, the WY inverse
// INV = (I + Akk)^-1 and INV diag(beta), kr^T and the 16-row block factors
// and row norms come from the prep kernel's per-chunk block (kda_prep_tc.cu).
#include "kda_chunk.cuh"
#include "kda_tc_tiles.cuh"

namespace kda {
namespace gtc {

using namespace tct;
constexpr int D = 128;
constexpr uint32_t T64x128 = umma::ptile_bytes(64, 128);    // 18432
constexpr uint32_t T128x128 = umma::ptile_bytes(128, 128);  // 36864
constexpr uint32_t T64x64 = umma::ptile_bytes(64, 64);      // 9216
constexpr uint32_t T128x64 = umma::ptile_bytes(128, 64);    // 18432

constexpr int NT = 512;            // threads per CTA
constexpr int NW = NT / 32;        // warps
// the thread that issues the TMA stores of the gradient rows (and waits on
// them): not thread 0, which issues the MMAs that follow some of them
constexpr int kStoreT = 32;

// ---- shared memory plan (bytes) ----------------------------------------------
struct Smem {
  static constexpr size_t n_view = PrepView<bf16, D>::floats;
  // extra floats: tbuf 768 (ddt_bias partials, gate scalars), dgT 4 x 128, red 16 x 64,
  // red2 4 x 64, dbeta 64, dA 16
  static constexpr size_t n_extra = 768 + 512 + 1024 + 256 + 64 + 16;
  static constexpr size_t sz_small = (((n_view + n_extra) * 4 + 64 + 1023) / 1024) * 1024;
  static constexpr size_t o_small = 0;
  // R_A: raw q, k, g rows (prep phase)  ->  [0, 16K): dv rows, then g rows (K1);
  // [16K, 48K): Mqk, INV, INVb, G (packed 64 x 64, the prep block's order, one
  // bulk copy), then dq / dg rows and dk rows
  static constexpr size_t o_A = o_small + sz_small;
  static constexpr size_t o_Mqk = o_A + 16384;
  static constexpr size_t o_INV = o_Mqk + 8192;
  static constexpr size_t o_INVb = o_INV + 8192;
  static constexpr size_t o_Gbf = o_INVb + 8192;
  static constexpr size_t sz_A = 64 * 64 * 4 + 4 * T64x64;  // >= 3 raw tiles
  // R_B: S | v rows  ->  S | U^T  ->  hi tiles QMh, KMh, KPh (intra)
  static constexpr size_t o_B = o_A + sz_A;
  static constexpr size_t o_S = o_B;
  static constexpr size_t o_U = o_B + T128x128;
  static constexpr size_t sz_B = 3 * T64x128;
  // R_C: kd^T, kr^T  ->  Xr^T, dU^T  ->  lo tiles QMl, KMl (intra)
  static constexpr size_t o_C = o_B + sz_B;
  static constexpr size_t sz_C = 2 * T64x128;
  // R_D: the stacked 128-row operand [dO; dvcorr] of P3a / P6 / P8 in the
  // 128-byte swizzled layout, two 64-column slabs kStk apart (slab 0: dO
  // [0, 8K), dvcorr [8K, 16K); slab 1: dO [40K, 48K), dvcorr [48K, 56K)),
  // and dS (packed 128 x 128) in [8K, 40K) until R3 has consumed it (the
  // dvcorr rows of slab 0 are written over it after) -> dMqk | dA (interleaved
  // by 16-row blocks, 128 x 64) in [0, 18K) and KPl (intra) after it
  static constexpr size_t o_D = o_C + sz_C;
  static constexpr uint32_t kStk = 40960;
  static constexpr size_t o_stk = o_D;
  static constexpr size_t o_dS = o_D + 8192;
  static constexpr size_t o_dMqk = o_D;
  static constexpr size_t o_KPl = o_D + T128x64;
  static constexpr size_t sz_D = kStk + 16384;
  static constexpr size_t total = o_D + sz_D;
  static_assert(sz_A >= 3 * 64 * D * 2, "raw tiles must fit R_A");
  static_assert(o_Gbf + 8192 <= o_A + sz_A, "prep tiles must fit R_A");
  static_assert(kPrepINV == kPrepMqk + 8192 && kPrepINVb == kPrepINV + 8192 &&
                    kPrepG == kPrepINVb + 8192,
                "prep tiles are copied as one block");
  static_assert(T128x128 + T128x64 <= sz_B, "S + U must fit R_B");
  static_assert(o_D % 1024 == 0 && kStk % 1024 == 0, "swizzled atoms are 1024-byte aligned");
  static_assert(o_dS + 32768 <= o_stk + kStk, "dS ends where slab 1 begins");
  static_assert(o_KPl + T64x128 <= o_stk + kStk, "KPl stays clear of slab 1");
  static_assert(total <= 232448, "shared memory budget");
  static_assert(o_small % 16 == 0 && (19 * D * 4) % 16 == 0,
                "the view's rq, rk and beta rows start on 16-byte boundaries (lds4)");
};

// TMEM address of this thread's lane (warp quarter) at column col
__device__ __forceinline__ uint32_t tlane(uint32_t tbase, int col) {
  return tbase + ((uint32_t)(32 * ((threadIdx.x >> 5) & 3)) << 16) + (uint32_t)col;
}
// this thread's 16 columns [col0 + 16 I, +16) of its lane, I = tid / 128
__device__ __forceinline__ void tld16(uint32_t tbase, int col0, float (&v)[16]) {
  umma::tmem_ld16(tlane(tbase, col0 + 16 * (int)(threadIdx.x >> 7)), v);
  umma::tmem_ld_wait();
}
// the same load without the wait (batch several, then umma::tmem_ld_wait)
__device__ __forceinline__ void tld16_nw(uint32_t tbase, int col0, float (&v)[16]) {
  umma::tmem_ld16(tlane(tbase, col0 + 16 * (int)(threadIdx.x >> 7)), v);
}

// Two bf16 values (raw bits) in one register, and back to fp32 (exact).
__device__ __forceinline__ uint32_t pack_bf(bf16 a, bf16 b) {
  return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
// element r of 16 values packed two per register
#define BF16_AT(arr, r) (((r) & 1) ? bf_hi((arr)[(r) >> 1]) : bf_lo((arr)[(r) >> 1]))

// Triangle-sized accumulators of the intra-chunk products.  dMqk and dA share
// one 128 x 64 tile, interleaved by 16-row blocks (rows 32 b .. 32 b + 15 =
// dMqk block b, the next 16 = dA block b), so that P9a and P9b of key block J
// are ONE product over the tile's rows 32 J .. 127 (N = 128 - 32 J): its
// columns 32 (I - J) .. + 15 hold the dMqk side of query block I, the next 16
// the dA side.  Query-block X of P9c holds output columns j < 16 (X + 1) only
// (N = 16 (X + 1)).  TMEM column bases: P9ab in [0, 256) and [384, 448) (P8's
// results sit in [256, 384) and dkr in [448, 512)), P9c in [0, 160).
__device__ __forceinline__ int col_p9ab(int J) { return J == 0 ? 0 : (J == 1 ? 128 : (J == 2 ? 384 : 224)); }
__device__ __forceinline__ int col_p9c(int X) { return X == 0 ? 0 : (X == 1 ? 16 : (X == 2 ? 48 : 96)); }
// row of the interleaved dMqk | dA tile holding row i of dMqk (side 0) or dA (side 1)
__device__ __forceinline__ int dma_row(int i, int side) { return 32 * (i >> 4) + 16 * side + (i & 15); }

// prep in the (channel, 16-row block) mapping; E kept in registers.  The row
// norms and the block factors (em, egm, F, gT) come with the prep kernel's
// operand block; here only the thread's own gate running sum (for E) and the
// kd^T tile are formed.
// Once every thread holds its raw rows, thread 0 issues the copy of the
// prep block's 64 x 64 tiles (Mqk, INV, INVb, G: 32 KB) over them (tiles, on
// barrier pbar), so that it lands while the gate and kd^T are formed.
__device__ void prep_tc(const KdaParams &p, int h, int len, const bf16 *Qr, const bf16 *Kr,
                        const bf16 *Gr, const PrepView<bf16, D> &sv, float (&E)[16], void *KDt,
                        uint32_t (&q2)[8], uint32_t (&k2)[8], uint32_t (&g2)[8],
                        const char *tiles_src, void *tiles, uint64_t *pbar, const float *gsc) {
  const int tid = threadIdx.x;
  const int c = tid & 127, I = tid >> 7;
  const float A = gsc[0], bias = gsc[D + c];  // e^A_log[h], dt_bias[h][c]
  // gate: running sum over the block, local to the block (see kda_chunk.cuh)
  float d[16];
  {
    float run = 0.f;
#pragma unroll
    for (int r = 0; r < 16; r += 2) {
      const int i = 16 * I + r;
      g2[r >> 1] = pack_bf(Gr[i * D + c], Gr[(i + 1) * D + c]);
      q2[r >> 1] = pack_bf(Qr[i * D + c], Qr[(i + 1) * D + c]);
      k2[r >> 1] = pack_bf(Kr[i * D + c], Kr[(i + 1) * D + c]);
    }
    __syncthreads();  // the raw rows are dead
    if (tid == 0) {
      umma::mbar_expect_tx(pbar, 32768u);
      umma::bulk_g2s(tiles, tiles_src, 32768u, pbar);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int i = 16 * I + r;
      const float gv = BF16_AT(g2, r) + bias;
      run += i < len ? -A * softplus_gate(gv) : 0.f;
      d[r] = run;
    }
    const float ref = d[7];
#pragma unroll
    for (int r = 0; r < 16; ++r) d[r] -= ref;  // gc - m_I
  }
  // kd^T [c][i] (128 x 64, read MN-major as MMA operand B with K = c), one
  // 16-byte store per 8 rows
  const float em = sv.em[I * D + c];
#pragma unroll
  for (int q8 = 0; q8 < 2; ++q8) {
    float vkd[8];
#pragma unroll
    for (int t4 = 0; t4 < 8; t4 += 4) {
      float rk4[4];
      lds4(sv.rk + 16 * I + 8 * q8 + t4, rk4);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = t4 + u, r = 8 * q8 + t;
        const float e = __expf(d[r]);
        E[r] = e;
        const float kh = BF16_AT(k2, r) * rk4[u];
        vkd[t] = (kh * e) * em;
      }
    }
    pstore8(KDt, c, 16 * I + 8 * q8, 64, vkd);
  }
  __syncthreads();
}

}  // namespace gtc

__global__ void __launch_bounds__(gtc::NT, 1)
    kda_grads_tc_kernel(KdaParams p, const __grid_constant__ TokenMaps tm, const void *states) {
  using namespace gtc;
  using SM = Smem;
  extern __shared__ __align__(1024) char smem[];
  pdl_wait();  // the scans' states and state gradients
  const int64_t slot = blockIdx.x;
  const int h = blockIdx.y;
  const int H = p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = tid & 127, I = tid >> 7;  // channel (TMEM lane) and 16-row block
  int s_, j_, len;
  int64_t tok0;
  if (!slot_owner(p, slot, s_, j_, tok0, len)) {
    if (tid == 0) p.dA_part[slot * H + h] = 0.f;
    if (p.ddt_part != nullptr && tid < D) p.ddt_part[(slot * H + h) * D + tid] = 0.f;
    return;
  }
  // ---- views ----
  float *smf = reinterpret_cast<float *>(smem + SM::o_small);
  PrepView<bf16, D> sv = make_view<bf16, D>(smf);
  float *tbuf = smf + SM::n_view;  // [0, 512): ddt_bias partials (K1)
  float *gsc = tbuf + 512;         // [0]: e^A_log[h]; [128, 256): dt_bias[h][c]
  float *dgT = tbuf + 768;         // [4][128] per-block partials of the gT gradient
  float *red = dgT + 512;          // [16 warps][64]
  float *red2 = red + 1024;        // [4][64]
  float *dbs = red2 + 256;         // [64]
  float *dAred = dbs + 64;         // [16]
  uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + SM::o_small + (SM::n_view + SM::n_extra) * 4);
  uint64_t *lbar = mbar + 1;   // bulk copies of S, dS, kr^T
  uint64_t *pbar = mbar + 2;   // bulk copy of the prep tiles (its own barrier: it is armed
                               // while the first group may still be in flight)
  uint64_t *rbar = mbar + 3;   // TMA boxes of the raw q, k, g, v rows
  uint32_t *tslot = reinterpret_cast<uint32_t *>(mbar + 4);
  bf16 *Qr = reinterpret_cast<bf16 *>(smem + SM::o_A);
  bf16 *Kr = Qr + 64 * D;
  bf16 *Gr = Kr + 64 * D;
  char *Gbf = smem + SM::o_Gbf, *Mqk = smem + SM::o_Mqk, *INV = smem + SM::o_INV,
       *INVb = smem + SM::o_INVb;
  char *QMh = smem + SM::o_B, *KMh = QMh + T64x128, *KPh = KMh + T64x128;
  char *St = smem + SM::o_S, *Ut = smem + SM::o_U;
  char *KDt = smem + SM::o_C, *KRt = KDt + T64x128;
  char *XrT = KDt, *dUT = KRt, *QMl = KDt, *KMl = KRt;
  char *dSt = smem + SM::o_dS, *dMA = smem + SM::o_dMqk, *stk = smem + SM::o_stk,
       *KPl = smem + SM::o_KPl;
  const float scale = p.scale;
  const size_t DD = (size_t)D * D;
  const bf16 *Sg = reinterpret_cast<const bf16 *>(states) + ((size_t)slot * H + h) * DD;
  const bf16 *dSg = reinterpret_cast<const bf16 *>(p.dstates) + ((size_t)slot * H + h) * DD;
  const char *unit = p.prep + ((size_t)slot * H + h) * kPrepUnitBytes;

  // beta, loaded by the last two warps and stored after the CTA barrier
  // below: the raw bits stay in a register until then, so no warp waits for
  // the load before the barrier
  constexpr int kBetaT0 = NT - CHUNK;
  uint32_t beta_bits = 0u;
  if (tid >= kBetaT0 && tid - kBetaT0 < len)
    beta_bits = reinterpret_cast<const unsigned short *>(p.beta)[(tok0 + (tid - kBetaT0)) * H + h];
  // the gate's scalars likewise, by the four warps before them: A_log[h] (its
  // exponential is taken after the barrier) and the per-channel bias, kept in
  // shared memory (gsc) for the prep and K1 phases
  constexpr int kGateT0 = kBetaT0 - D;
  float gate_s = 0.f;
  if (tid >= kGateT0 && tid < kBetaT0) gate_s = gate_bias(p, h, tid - kGateT0, D);
  const float a_log = tid == kGateT0 ? p.A_log[h] : 0.f;
  // ---- barriers, the first copies, then Tensor Memory (all 512 columns) ----
  // Thread 0 initialises the barriers and at once issues the copies: the raw
  // q, k, g rows (row-major, R_A) and the block factors first, the prep phase
  // waits on them; then v rows (U's slot, free until P2), S (packed in the
  // workspace), dS and kr^T, which stream in during the prep phase.  Warp 0
  // allocates Tensor Memory meanwhile.
  // (a timeout test starves both barriers: they are armed, no copy is issued)
  const bool starve = (p.starve & kStarveGrads) != 0u;
  if (tid == 0) {
    umma::mbar_init(mbar, 1);
    umma::mbar_init(lbar, 1);
    umma::mbar_init(pbar, 1);
    umma::mbar_init(rbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    umma::mbar_expect_tx(rbar, 3 * 16384u + (uint32_t)kPrepSVBytes);
    if (!starve) {
      umma::tma_load_3d(Qr, &tm.q, 0, h, (int)tok0, rbar);
      umma::tma_load_3d(Kr, &tm.k, 0, h, (int)tok0, rbar);
      umma::tma_load_3d(Gr, &tm.g, 0, h, (int)tok0, rbar);
      umma::bulk_g2s(sv.em, unit + kPrepSV, (uint32_t)kPrepSVBytes, rbar);  // factors, norms
    }
    const uint32_t bytes = 16384u + (p.states_packed ? 32768u : 0u) +
                           (p.dstates_packed ? 32768u : 0u) + 16384u + 16384u;
    umma::mbar_expect_tx(lbar, bytes);
    if (!starve) {
      umma::tma_load_3d(Ut, &tm.v, 0, h, (int)tok0, lbar);
      // dO: two swizzled 64-channel boxes, the rows of the stacked operand
      umma::tma_load_3d(stk, &tm.dO_sw, 0, h, (int)tok0, lbar);
      umma::tma_load_3d(stk + SM::kStk, &tm.dO_sw, 64, h, (int)tok0, lbar);
      if (p.states_packed) umma::bulk_g2s(St, Sg, 32768u, lbar);
      if (p.dstates_packed) umma::bulk_g2s(dSt, dSg, 32768u, lbar);
      umma::bulk_g2s(KRt, unit + kPrepKR, 16384u, lbar);
    }
  }
  if (warp == 0) umma::tmem_alloc(tslot, 512);
  __syncthreads();
  // ---- row-major states (the per-band scans' or a caller's) by cp.async ----
  if (!p.states_packed) {  // row-major states (caller-provided) -> packed tile
    for (int e = tid; e < D * (D / 8); e += NT) {
      const int r = e >> 4, c8 = (e & 15) * 8;
      cp_async16(St + umma::core_off(r, c8, D), Sg + (size_t)r * D + c8, true);
    }
  }
  if (!p.dstates_packed) {  // row-major state gradients (the per-band scans)
    for (int e = tid; e < D * (D / 8); e += NT) {
      const int r = e >> 4, c8 = (e & 15) * 8;
      cp_async16(dSt + umma::core_off(r, c8, D), dSg + (size_t)r * D + c8, true);
    }
  }
  cp_async_commit();
  umma::tc_fence_before();
  if (tid >= kBetaT0) sv.beta[tid - kBetaT0] = __uint_as_float(beta_bits << 16);  // bf16 -> fp32
  if (tid >= kGateT0 && tid < kBetaT0) gsc[D + tid - kGateT0] = gate_s;
  if (tid == kGateT0) gsc[0] = __expf(a_log);
  // Every bounded wait below folds its result into `ok`.  The CTA decides at
  // its barriers (__syncthreads_or): once any thread's wait has given up, no
  // further MMA is issued and no result leaves the CTA (what a timed-out
  // product may have left in Tensor Memory reaches shared memory only); the
  // CTA drains what is in flight and releases Tensor Memory (`drain` below).
  const uint32_t lim_ld = poll_cap(p, umma::kPollLoads), lim_mma = poll_cap(p, umma::kPollMma);
  bool ok = umma::mbar_wait(rbar, 0, lim_ld);
  uint32_t phase = 0;         // completions of the MMA barrier waited for
  bool past_first = false;    // the prep-tile copy (pbar) has been issued
  if (len < CHUNK) {  // the boxes' rows past the chunk belong to the next sequence: zero them
    for (int e = tid; e < 3 * 64 * 16; e += NT) {
      const int t = e >> 10, i = (e >> 4) & 63, c8 = (e & 15) * 8;
      if (i >= len) {
        bf16 *base = t == 0 ? Qr : (t == 1 ? Kr : Gr);
        *reinterpret_cast<uint4 *>(base + i * D + c8) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  if (__syncthreads_or(!ok)) { ok = false; goto drain; }
  {
  past_first = true;
  umma::tc_fence_after();
  const uint32_t tbase = *tslot;
  auto mma_wait = [&]() {
    ok = umma::mbar_wait(mbar, phase & 1, lim_mma) && ok;
    phase++;
    umma::tc_fence_after();
  };

  // ---- prep ----
  float E[16];
  uint32_t q2[8], k2[8], g2[8];  // the thread's raw q, k, g rows, two per register
  // (the pair matrices and inverses formed by the prep kernel -- Mqk, INV,
  // INVb, G, packed 64 x 64 -- come into R_A over the raw rows from inside)
  prep_tc(p, h, len, Qr, Kr, Gr, sv, E, KDt, q2, k2, g2, unit + kPrepMqk, Mqk, pbar, gsc);
  cp_async_wait_all();                 // row-major S / dS, if any
  ok = umma::mbar_wait(lbar, 0, lim_ld) && ok;  // v, dO, S, dS, kr^T
  if (len < CHUNK) {
    // a sequence's partial last chunk: the dO and v boxes' rows past it hold
    // the next sequence's rows; zero them (a dO row's 128 bytes stay within
    // the row; v rows are row-major, 256 bytes)
    for (int e = tid; e < 2 * 64 * 8; e += NT) {
      const int row = (e >> 3) & 63;
      if (row >= len)
        *reinterpret_cast<uint4 *>(stk + (e >> 9) * SM::kStk + row * 128 + (e & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
    }
    for (int e = tid; e < 64 * 16; e += NT) {
      const int row = e >> 4;
      if (row >= len)
        *reinterpret_cast<uint4 *>(Ut + row * 256 + (e & 15) * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  umma::fence_async_smem();
  if (__syncthreads_or(!ok)) { ok = false; goto drain; }

  // ---- R1 = P1: kdS^T = S^T kd^T ; the epilogue forms Xr^T = v^T - kdS^T ----
  if (tid == 0) {
    umma::tc_fence_after();
    gemm(tbase + 0, opmn(St, D, 0, CP), true, opmn(KDt, 64), true, 64, D / 16, false);
    umma::mma_commit(mbar);
  }
  mma_wait();
  float acc[16];
  tld16(tbase, 0, acc);
#pragma unroll
  for (int r = 0; r < 16; ++r)  // v rows, row-major in U's slot (rows past the chunk: zeroed)
    acc[r] = __bfloat162float(reinterpret_cast<const bf16 *>(Ut)[(16 * I + r) * D + c]) - acc[r];
#pragma unroll
  for (int q = 0; q < 2; ++q) pstore8(XrT, c, 16 * I + 8 * q, 64, acc + 8 * q);  // Xr^T[d][i]
  ok = umma::mbar_wait(pbar, 0, lim_ld) && ok;  // Mqk, INV, INVb, G
  umma::fence_async_smem();
  umma::tc_fence_before();
  if (__syncthreads_or(!ok)) { ok = false; goto drain; }

  // ---- R2 = P2 + P3a: U^T = Xr^T INVb^T ; dU^T = dO^T Mqk + dS^T kr^T (dU needs no U) ----
  if (tid == 0) {
    umma::tc_fence_after();
    gemm(tbase + 64, opk(XrT, 64), false, opk(INVb, 64, 0, CP), false, 64, 4, false);
    gemm(tbase + 128, opsw_mn(stk, SM::kStk), true, opmn(Mqk, 64, 0, CP), true, 64, 4, false);
    gemm(tbase + 128, opmn(dSt, D, 0, CP), true, opmn(KRt, 64, 0, CP), true, 64, D / 16, true);
    umma::mma_commit(mbar);
  }
  {
    // B0: p_c = e^gT_c sum_d dS[c][d] S[c][d]; thread (c, I) takes d in [32 I, 32 I + 32)
    float pp = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float a8[8], b8[8];
      ld16_bf(dSt + umma::core_off(c, 32 * I + 8 * q, D), a8);
      ld16_bf(St + umma::core_off(c, 32 * I + 8 * q, D), b8);
#pragma unroll
      for (int t = 0; t < 8; ++t) pp = fmaf(a8[t], b8[t], pp);
    }
    dgT[I * D + c] = __expf(sv.gT[c]) * pp;
  }
  mma_wait();
  {
    float acc2[16];  // both loads in flight before one wait
    tld16_nw(tbase, 64, acc);
    tld16_nw(tbase, 128, acc2);
    umma::tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 2; ++q) pstore8(Ut, c, 16 * I + 8 * q, 64, acc + 8 * q);  // U^T[d][i]
#pragma unroll
    for (int q = 0; q < 2; ++q) pstore8(dUT, c, 16 * I + 8 * q, 64, acc2 + 8 * q);  // dU^T[d][i]
  }
  umma::fence_async_smem();
  umma::tc_fence_before();
  if (__syncthreads_or(!ok)) { ok = false; goto drain; }

  // ---- R3 = P5 + P3b: dvcorr^T = dU^T INV ; dkr^T = dS U^T ; dv, dbeta1, dvcorr[i][d] ----
  if (tid == 0) {
    umma::tc_fence_after();
    gemm(tbase + 0, opk(dUT, 64), false, opmn(INV, 64, 0, CP), true, 64, 4, false);
    gemm(tbase + 448, opk(dSt, D, 0, CP), false, opmn(Ut, 64), true, 64, D / 16, false);
    umma::mma_commit(mbar);
  }
  mma_wait();
  tld16(tbase, 0, acc);
  {
    bf16 *dvs = reinterpret_cast<bf16 *>(smem + SM::o_A);  // dv rows [64][128]
    float xr[16];
#pragma unroll
    for (int q = 0; q < 2; ++q) pload8(XrT, c, 16 * I + 8 * q, 64, xr + 8 * q);
    float pr[16];
#pragma unroll
    for (int r4 = 0; r4 < 16; r4 += 4) {
      float b4[4];
      lds4(sv.beta + 16 * I + r4, b4);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = r4 + u, i = 16 * I + r;
        // dvcorr row i = row 64 + i of the stacked swizzled operand
        *reinterpret_cast<bf16 *>(stk + umma::sw128_off(64 + i, c, SM::kStk)) =
            __float2bfloat16_rn(acc[r]);
        dvs[i * D + c] = __float2bfloat16_rn(b4[u] * acc[r]);
        pr[r] = acc[r] * xr[r];
      }
    }
    // sums over this warp's 32 channels; lanes 2 l, 2 l + 1 hold row 16 I + l
    const float t = rows16_sum(pr);
    if ((lane & 1) == 0) red[warp * 16 + (lane >> 1)] = t;
  }
  umma::fence_async_smem();
  umma::tc_fence_before();
  if (__syncthreads_or(!ok)) { ok = false; goto drain; }
  if (tid < 64) {  // dbeta1_i: block i / 16 lives in warps 4 (i / 16) .. + 3
    const int i = tid, w0 = (i >> 4) * 4, r = i & 15;
    dbs[i] = red[(w0 + 0) * 16 + r] + red[(w0 + 1) * 16 + r] + red[(w0 + 2) * 16 + r] +
             red[(w0 + 3) * 16 + r];
  }
  {  // dv rows: one TMA box for a whole chunk, else 16-byte row pieces (alongside P6 / P8)
    const bf16 *dvs = reinterpret_cast<const bf16 *>(smem + SM::o_A);
    if (len == CHUNK) {
      if (tid == kStoreT) {
        umma::tma_store_3d(&tm.dv, 0, h, (int)tok0, dvs);
        umma::bulk_commit();
      }
    } else {
      bf16 *dvg = reinterpret_cast<bf16 *>(p.dv);
#pragma unroll 1
      for (int e = tid; e < 64 * (D / 8); e += NT) {
        const int i = e >> 4, c8 = (e & 15) * 8;
        if (i < len)
          *reinterpret_cast<uint4 *>(dvg + ((tok0 + i) * H + h) * D + c8) =
              *reinterpret_cast<const uint4 *>(dvs + i * D + c8);
      }
    }
  }

  // ---- P6: [dO; dvcorr] U^T  and  P8: S [dO; dvcorr]^T ----
  if (tid == 0) {
    umma::tc_fence_after();
    gemm(tbase + 64, opsw_k(stk, SM::kStk), false, opmn(Ut, 64), true, 64, D / 16, false);
    gemm(tbase + 256, opk(St, D, 0, CP), false, opsw_k(stk, SM::kStk), false, 128, D / 16,
         false);
    umma::mma_commit(mbar);
  }
  mma_wait();
  {
    // lanes 0..63: dMqk / scale rows (dO U^T), lanes 64..127: -dAkk rows
    float v16[16];
    tld16(tbase, 64, v16);  // columns j in [16 I, 16 I + 16)
    if (c >= 64) {
      const int i = c - 64;
      const float bi = sv.beta[i];
      float db2 = 0.f;
      float o8[8];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float g8[8];  // G[i][16 I + 8 q .. + 7], one 16-byte row of a core matrix
        ld16_bf(Gbf + umma::core_off(i, 16 * I + 8 * q, 64), g8);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int jj = 16 * I + 8 * q + t;
          const float dak = jj < i ? -v16[8 * q + t] : 0.f;
          db2 = fmaf(dak, g8[t], db2);
          o8[t] = bi * dak;
        }
        pstore8(dMA, dma_row(i, 1), 16 * I + 8 * q, 64, o8);
      }
      red2[I * 64 + i] = db2;
    } else {
      const int i = c;
      float o8[8];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int jj = 16 * I + 8 * q + t;
          o8[t] = jj <= i ? scale * v16[8 * q + t] : 0.f;
        }
        pstore8(dMA, dma_row(i, 0), 16 * I + 8 * q, 64, o8);
      }
    }
  }
  umma::fence_async_smem();
  umma::tc_fence_before();
  if (tid == kStoreT) umma::bulk_wait_read();  // the dv box has left R_A [0, 16K) (the g rows go there)
  if (__syncthreads_or(!ok)) { ok = false; goto drain; }
  if (tid < 64 && tid < len) {
    const float db = dbs[tid] + red2[tid] + red2[64 + tid] + red2[128 + tid] + red2[192 + tid];
    reinterpret_cast<bf16 *>(p.dbeta)[(tok0 + tid) * H + h] = __float2bfloat16_rn(db);
  }
  // ---- intra-chunk operands, hi + lo (see kda_grads.cu) ----
  // (R_A [0, 16K), the old raw q rows, keeps the g rows for the gate epilogue)
  bf16 *gs = reinterpret_cast<bf16 *>(smem + SM::o_A);
#pragma unroll
  for (int r = 0; r < 16; r += 2) {
    *reinterpret_cast<uint32_t *>(gs + (r >> 1) * 2 * NT + 2 * tid) = g2[r >> 1];
  }
  float qh[16], kh[16];
#pragma unroll
  for (int q8 = 0; q8 < 2; ++q8) {
    // two rows at a time: hi = bf16 pair (one conversion), lo = the pair of
    // remainders x - hi (exact in fp32), rounded as a pair
    uint32_t hp[3][4], lp[3][4];
    float rq8[8], rk8[8];
    lds4(sv.rq + 16 * I + 8 * q8, rq8);
    lds4(sv.rq + 16 * I + 8 * q8 + 4, rq8 + 4);
    lds4(sv.rk + 16 * I + 8 * q8, rk8);
    lds4(sv.rk + 16 * I + 8 * q8 + 4, rk8 + 4);
#pragma unroll
    for (int t2 = 0; t2 < 4; ++t2) {
      float x[3][2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = 8 * q8 + 2 * t2 + e;
        qh[r] = BF16_AT(q2, r) * rq8[2 * t2 + e];
        kh[r] = BF16_AT(k2, r) * rk8[2 * t2 + e];
        x[0][e] = qh[r] * E[r];
        x[1][e] = kh[r] * E[r];
        x[2][e] = __fdividef(kh[r], E[r]);
      }
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        const uint32_t h2 = f2_to_bf2(x[u][0], x[u][1]);
        hp[u][t2] = h2;
        lp[u][t2] = f2_to_bf2(x[u][0] - bf_lo(h2), x[u][1] - bf_hi(h2));
      }
    }
    const uint32_t off = pcore_off(c, 16 * I + 8 * q8, 64);  // rows i0 .. i0 + 7 of channel c
    char *hi[3] = {QMh, KMh, KPh};
    char *lo[3] = {QMl, KMl, KPl};
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      *reinterpret_cast<uint4 *>(hi[u] + off) = make_uint4(hp[u][0], hp[u][1], hp[u][2], hp[u][3]);
      *reinterpret_cast<uint4 *>(lo[u] + off) = make_uint4(lp[u][0], lp[u][1], lp[u][2], lp[u][3]);
    }
  }
  umma::fence_async_smem();
  umma::tc_fence_before();
  __syncthreads();

  // per-thread block factors: Fq[J] = F_{I,J} (J <= I) for the query-side
  // sums, Fk[X] = F_{X,I} (X >= I) for the key side
  float Fq[4], Fk[4];
#pragma unroll
  for (int X = 0; X < 4; ++X) {
    Fq[X] = X < I ? sv.F[pair_index(I, X) * D + c] : (X == I ? 1.f : 0.f);
    Fk[X] = X > I ? sv.F[pair_index(X, I) * D + c] : (X == I ? 1.f : 0.f);
  }
  const float emI = sv.em[I * D + c];
  // ---- R5 = P9a + P9b: dq^ intra (dMqk with kp) and dkd' intra (dA with kp), per key block J,
  // both sides in one product over the interleaved tile (8 MMAs, hi + lo) ----
  if (tid == 0) {
    umma::tc_fence_after();
    const Desc aH = mkdesc(opk(KPh, 64)), aL = mkdesc(opk(KPl, 64));
    const Desc bMA = mkdesc(opk(dMA, 64));
#pragma unroll
    for (int J = 0; J < 4; ++J) {
      const uint32_t id = umma::idesc_bf16(128, 128 - 32 * J, false, false);
      const uint32_t ka = (uint32_t)(2 * J) * CS;                      // K offset (columns 16 J)
      const uint32_t kb = ka + (uint32_t)(4 * J) * (64 / 8) * CS;      // and rows 32 J of B
      mma1(tbase + col_p9ab(J), dshift(aH, ka), dshift(bMA, kb), id, false);
      mma1(tbase + col_p9ab(J), dshift(aL, ka), dshift(bMA, kb), id, true);
    }
    umma::mma_commit(mbar);
  }
  mma_wait();
  // dq / dk rows are finished in shared memory (R_A [16K, 48K): the prep tiles
  // are dead after P6) and written to HBM as 16-byte row pieces
  bf16 *dqs = reinterpret_cast<bf16 *>(smem + SM::o_A + 16384);
  bf16 *dks = dqs + 64 * D;
  float dgc[16];
  {
    // dO S^T (rows 0..63 of the stacked operand) and key blocks J <= I
    // (F_{I,J} = 0 above the diagonal blocks; rows 16 I .. of block J's
    // accumulator), TMEM loads in two batches
    float bq[16], in[16];
    {
      float a0[16], a1[16];
      tld16_nw(tbase, 256, bq);
      // (tld16 adds 16 I: key block J's dMqk side of block I is at col_p9ab(J) + 32 (I - J))
      tld16_nw(tbase, col_p9ab(0) + 16 * I, a0);
      if (I >= 1) tld16_nw(tbase, col_p9ab(1) - 32 + 16 * I, a1);
      umma::tmem_ld_wait();
#pragma unroll
      for (int r = 0; r < 16; ++r) in[r] = Fq[0] * a0[r] + (I >= 1 ? Fq[1] * a1[r] : 0.f);
      if (I >= 2) {
        tld16_nw(tbase, col_p9ab(2) - 64 + 16 * I, a0);
        if (I >= 3) tld16_nw(tbase, col_p9ab(3) - 96 + 16 * I, a1);
        umma::tmem_ld_wait();
#pragma unroll
        for (int r = 0; r < 16; ++r)
          in[r] = fmaf(Fq[2], a0[r], in[r]) + (I >= 3 ? Fq[3] * a1[r] : 0.f);
      }
    }
    float dq[16], pr[16];
    const float sem = scale * emI;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      dq[r] = E[r] * fmaf(sem, bq[r], in[r]);
      dgc[r] = dq[r] * qh[r];
      pr[r] = dgc[r];
    }
    const float t = rows16_sum(pr);
    if ((lane & 1) == 0) red[warp * 16 + (lane >> 1)] = t;
    umma::tc_fence_before();
    if (__syncthreads_or(!ok)) { ok = false; goto drain; }
    // lane l < 16: row 16 I + l summed over the block's 4 warps; broadcast below
    const float tot = red[(4 * I) * 16 + (lane & 15)] + red[(4 * I + 1) * 16 + (lane & 15)] +
                      red[(4 * I + 2) * 16 + (lane & 15)] + red[(4 * I + 3) * 16 + (lane & 15)];
#pragma unroll
    for (int r4 = 0; r4 < 16; r4 += 4) {
      float rq4[4];
      lds4(sv.rq + 16 * I + r4, rq4);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = r4 + u;
        const float rd = __shfl_sync(0xffffffffu, tot, r);
        dqs[(16 * I + r) * D + c] = __float2bfloat16_rn((dq[r] - qh[r] * rd) * rq4[u]);
      }
    }
  }

  float dkt[16];
  {
    float bk[16];  // dvcorr S^T, and the key blocks as for dq
    {
      float a0[16], a1[16];
      tld16_nw(tbase, 320, bk);
      tld16_nw(tbase, col_p9ab(0) + 16 + 16 * I, a0);  // the dA side: 16 further
      if (I >= 1) tld16_nw(tbase, col_p9ab(1) - 16 + 16 * I, a1);
      umma::tmem_ld_wait();
#pragma unroll
      for (int r = 0; r < 16; ++r) dkt[r] = Fq[0] * a0[r] + (I >= 1 ? Fq[1] * a1[r] : 0.f);
      if (I >= 2) {
        tld16_nw(tbase, col_p9ab(2) - 48 + 16 * I, a0);
        if (I >= 3) tld16_nw(tbase, col_p9ab(3) - 80 + 16 * I, a1);
        umma::tmem_ld_wait();
#pragma unroll
        for (int r = 0; r < 16; ++r)
          dkt[r] = fmaf(Fq[2], a0[r], dkt[r]) + (I >= 3 ? Fq[3] * a1[r] : 0.f);
      }
    }
#pragma unroll
    for (int r4 = 0; r4 < 16; r4 += 4) {
      float b4[4];
      lds4(sv.beta + 16 * I + r4, b4);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = r4 + u;
        dkt[r] = E[r] * fmaf(-b4[u] * emI, bk[r], dkt[r]);
      }
    }
  }
  umma::fence_async_smem();  // the dq rows, for the TMA store
  umma::tc_fence_before();
  __syncthreads();
  if (len == CHUNK) {
    if (tid == kStoreT) {
      umma::tma_store_3d(&tm.dq, 0, h, (int)tok0, dqs);
      umma::bulk_commit();
    }
  } else {
    bf16 *dqg = reinterpret_cast<bf16 *>(p.dq);
#pragma unroll 1
    for (int e = tid; e < 64 * (D / 8); e += NT) {
      const int i = e >> 4, c8 = (e & 15) * 8;
      if (i < len)
        *reinterpret_cast<uint4 *>(dqg + ((tok0 + i) * H + h) * D + c8) =
            *reinterpret_cast<const uint4 *>(dqs + i * D + c8);
    }
  }

  // ---- R6 = P9c: dki' = E^-1 sum_{X >= J} (Mqk-side + A-side) with qm / km, per query block X ----
  if (tid == 0) {
    umma::tc_fence_after();
    const Desc aQH = mkdesc(opk(QMh, 64)), aQL = mkdesc(opk(QMl, 64));
    const Desc aKH = mkdesc(opk(KMh, 64)), aKL = mkdesc(opk(KMl, 64));
    const Desc bMA = mkdesc(opmn(dMA, 64));
#pragma unroll
    for (int X = 0; X < 4; ++X) {
      const uint32_t d = tbase + col_p9c(X);
      const uint32_t id = umma::idesc_bf16(128, 16 * (X + 1), false, true);
      const uint32_t ka = (uint32_t)(2 * X) * CS;                      // K offset (columns 16 X)
      const uint32_t kbm = (uint32_t)(4 * X) * (64 / 8) * CS;          // dMqk block X: rows 32 X
      const uint32_t kba = kbm + (uint32_t)2 * (64 / 8) * CS;          // dA block X: 16 rows on
      mma1(d, dshift(aQH, ka), dshift(bMA, kbm), id, false);
      mma1(d, dshift(aQL, ka), dshift(bMA, kbm), id, true);
      mma1(d, dshift(aKH, ka), dshift(bMA, kba), id, true);
      mma1(d, dshift(aKL, ka), dshift(bMA, kba), id, true);
    }
    umma::mma_commit(mbar);
  }
  mma_wait();
  {
    // query blocks X >= I (F_{X,I} = 0 for X < I) and dkr, in two batches
    float dki[16], dkr[16];
    {
      float a0[16], a1[16];
      tld16_nw(tbase, 448, dkr);
      tld16_nw(tbase, col_p9c(3), a0);
      if (I <= 2) tld16_nw(tbase, col_p9c(2), a1);
      umma::tmem_ld_wait();
#pragma unroll
      for (int r = 0; r < 16; ++r) dki[r] = Fk[3] * a0[r] + (I <= 2 ? Fk[2] * a1[r] : 0.f);
      if (I <= 1) {
        tld16_nw(tbase, col_p9c(1), a0);
        if (I == 0) tld16_nw(tbase, col_p9c(0), a1);
        umma::tmem_ld_wait();
#pragma unroll
        for (int r = 0; r < 16; ++r)
          dki[r] = fmaf(Fk[1], a0[r], dki[r]) + (I == 0 ? Fk[0] * a1[r] : 0.f);
      }
    }
    float dk[16], pr[16], colp = 0.f;
    const float egI = sv.egm[I * D + c];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      // dki' + dkr' = E^-1 (dki + e^(gT - m_I) dkr); dkr' alone enters dgT
      const float rE = __fdividef(1.f, E[r]);
      const float w = dkr[r] * egI;
      const float sk = (dki[r] + w) * rE;
      dk[r] = dkt[r] + sk;
      dgc[r] = fmaf(dkt[r] - sk, kh[r], dgc[r]);
      colp = fmaf(w * rE, kh[r], colp);
      pr[r] = dk[r] * kh[r];
    }
    const float t = rows16_sum(pr);
    if ((lane & 1) == 0) red[warp * 16 + (lane >> 1)] = t;
    dgT[I * D + c] += colp;
    if (__syncthreads_or(!ok)) { ok = false; goto drain; }
    const float tot = red[(4 * I) * 16 + (lane & 15)] + red[(4 * I + 1) * 16 + (lane & 15)] +
                      red[(4 * I + 2) * 16 + (lane & 15)] + red[(4 * I + 3) * 16 + (lane & 15)];
#pragma unroll
    for (int r4 = 0; r4 < 16; r4 += 4) {
      float rk4[4];
      lds4(sv.rk + 16 * I + r4, rk4);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = r4 + u;
        const float rd = __shfl_sync(0xffffffffu, tot, r);
        dks[(16 * I + r) * D + c] = __float2bfloat16_rn((dk[r] - kh[r] * rd) * rk4[u]);
      }
    }
  }

  // ---- K1: reverse cumsum over the chunk rows, dg, dA_log ----
  {
    float tot = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) tot += dgc[r];
    umma::fence_async_smem();  // the dk rows, for the TMA store
    __syncthreads();           // red is free again; the dk rows are complete
    red[I * 128 + c] = tot;  // block totals per channel
    if (len == CHUNK) {
      if (tid == kStoreT) {
        umma::tma_store_3d(&tm.dk, 0, h, (int)tok0, dks);
        umma::bulk_commit();
      }
    } else {
      bf16 *dkg = reinterpret_cast<bf16 *>(p.dk);
#pragma unroll 1
      for (int e = tid; e < 64 * (D / 8); e += NT) {
        const int i = e >> 4, c8 = (e & 15) * 8;
        if (i < len)
          *reinterpret_cast<uint4 *>(dkg + ((tok0 + i) * H + h) * D + c8) =
              *reinterpret_cast<const uint4 *>(dks + i * D + c8);
      }
    }
    if (tid == kStoreT) umma::bulk_wait_read_but1();  // the dq box has left (dg rows go there)
    __syncthreads();
    float run = dgT[c] + dgT[D + c] + dgT[2 * D + c] + dgT[3 * D + c];
#pragma unroll
    for (int X = 1; X < 4; ++X)
      if (X > I) run += red[X * 128 + c];
    const float nA = -gsc[0], bias = gsc[D + c];  // -e^A_log[h], dt_bias[h][c]
    float dA = 0.f, ddt = 0.f;  // dA: sum of dgk softplus (times -e^A_log below)
    bf16 *dgsm = dqs;  // dg rows, [64][128]
#pragma unroll
    for (int r2 = 7; r2 >= 0; --r2) {
      // the g rows 2 r2 (low half) and 2 r2 + 1 (high half), one load
      const uint32_t gp = *reinterpret_cast<const uint32_t *>(gs + r2 * 2 * NT + 2 * tid);
#pragma unroll
      for (int e = 1; e >= 0; --e) {
        const int r = 2 * r2 + e, i = 16 * I + r;
        run += dgc[r];
        const float gv = (e ? bf_hi(gp) : bf_lo(gp)) + bias;
        // sigmoid and softplus from one exponential, t = e^-|g|
        const float t = __expf(-fabsf(gv));
        const float inv = __fdividef(1.f, 1.f + t);
        const float sg = gv >= 0.f ? inv : t * inv;
        const float sp = fmaxf(gv, 0.f) + log1p_unit_warp(t);
        const float dgv = run * nA * sg;
        dgsm[i * D + c] = __float2bfloat16_rn(dgv);
        if (i < len) {
          dA = fmaf(run, sp, dA);
          ddt += dgv;
        }
      }
    }
    dA = warp_sum(dA * nA);
    if (lane == 0) dAred[warp] = dA;
    tbuf[I * D + c] = ddt;  // ddt_bias partial: this block's dg column sum
    umma::fence_async_smem();  // the dg rows, for the TMA store
    umma::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < NW; ++w) t += dAred[w];
      p.dA_part[slot * H + h] = t;
    }
    if (p.ddt_part != nullptr && tid < D)
      p.ddt_part[(slot * H + h) * D + tid] =
          (tbuf[tid] + tbuf[D + tid]) + (tbuf[2 * D + tid] + tbuf[3 * D + tid]);
    if (len == CHUNK) {
      if (tid == kStoreT) {
        umma::tma_store_3d(&tm.dg, 0, h, (int)tok0, dgsm);
        umma::bulk_commit();
      }
    } else {
      bf16 *dgg = reinterpret_cast<bf16 *>(p.dg);
#pragma unroll 1
      for (int e = tid; e < 64 * (D / 8); e += NT) {
        const int i = e >> 4, c8 = (e & 15) * 8;
        if (i < len)
          *reinterpret_cast<uint4 *>(dgg + ((tok0 + i) * H + h) * D + c8) =
              *reinterpret_cast<const uint4 *>(dgsm + i * D + c8);
      }
    }
  }
  }
drain:
  // `ok` is uniform here: every decision above sets it for the whole CTA
  // before jumping, and no wait follows the last one
  if (!ok) {
    // a bounded wait gave up (the status word says so): let the copies and the
    // MMA batch that may still be in flight land before the CTA releases its
    // shared memory and Tensor Memory
    if (tid == 0) {
      const uint32_t lim = poll_cap(p, umma::kPollDrain);
      umma::mbar_wait(rbar, 0, lim);
      umma::mbar_wait(lbar, 0, lim);
      if (past_first) umma::mbar_wait(pbar, 0, lim);
      if (phase > 0) umma::mbar_wait(mbar, (phase - 1) & 1, lim);
    }
    cp_async_wait_all();
    umma::tc_fence_before();
    __syncthreads();
  }
  // the stored boxes have read shared memory before the CTA ends (their
  // global writes complete before the grid does); on the normal path every
  // Tensor Memory load completed before the gate epilogue's barriers
  if (tid == kStoreT) umma::bulk_wait_read();
  if (warp == 0) {
    __syncwarp();  // thread 0 may have drained alone: the release is warp-collective
    umma::tc_fence_after();
    umma::tmem_dealloc(*tslot, 512);
  }
}

cudaError_t grads_tc_launch(const KdaParams &p, const TokenMaps &tm, const void *states,
                            cudaStream_t st) {
  auto kfn = kda_grads_tc_kernel;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)gtc::Smem::total);
  if (e != cudaSuccess) return e;
  if (p.nslots > 0) {
    e = pdl_launch(kfn, dim3((unsigned)p.nslots, p.H), dim3(gtc::NT), gtc::Smem::total, st, p, tm,
                   states);
  }
  return e;
}

size_t grads_tc_smem_bytes() { return gtc::Smem::total; }

int grads_tc_status_take() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_status, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

}  // namespace kda
