// kda_grads.cu -- per-chunk gradients of the KDA backward, one CTA per
// (chunk slot, head).  It is the work the kernel-B guide
// ("bwd-kernelB-beginner-guide-full") splits into B1 / B2 / B0 / B3 (Part 1
// table), done in one CTA from the chunk inputs, the chunk-start state S_n
// and the chunk-end state gradient dS_{n+1}:
//
//   B1  U = INV diag(beta) (v - kd S_n)        dU = scale Mqk^T dO + kr dS_{n+1}
//       dvcorr = INV^T dU      dv = beta dvcorr      dkr = U dS_{n+1}^T
//   B2  dqd = scale dO S_n^T + dMqk ki        dkd = -diag(beta) dvcorr S_n^T + dA ki
//       dbeta = rowsum(dvcorr (v - kd S_n)) + rowsum(dAkk * G)
//   B0  p = e^gT rowdot(dS_{n+1}, S_n)        (gradient of the chunk-end decay)
//   B3  dMqk = lower(scale dO U^T)   dAkk = -strict_lower(dvcorr U^T)   dA = diag(beta) dAkk
//       dki = dMqk^T qd + dA^T kd
//   K1  dgc = dq^ q^ + (dkd' - dki' - dkr') k^          (fp32 only, guide Part 2, B3)
//       dgk = reverse_cumsum(dgc) + dgT,  dg = dgk (-e^A_log) sigmoid(g),
//       dA_log = sum dgk gk,  dq = (dq^ - q^ (q^ . dq^)) / |q|  (and dk)
//
// with ki = k^ e^-gc formed only inside 16-row blocks relative to a block
// reference gate (see kda_chunk.cuh).  Primed gradients are taken in the
// normalised-key frame: dq^ = dqd e^gc, dkd' = dkd e^gc, dki' = dki e^-gc,
// dkr' = dkr e^(gT - gc); dk^ = dkd' + dki' + dkr'.  Everything after the
// bf16 tensor-core products is fp32 (the guide's fp32-only gate epilogue).
#include <stdlib.h>

#include "kda_chunk.cuh"

namespace kda {

// Accumulator of the gate gradient's carries.  The chunk-end term dgT (the
// row dot e^gT dS_{n+1} . S_n plus the kr column sums) is large next to dgk
// and cancels against the reverse cumulative sum of dgc, and dA_log = sum
// dgk gk cancels once more over the rows; one fp32 rounding of dgT alone
// moves dA_log by ~5e-5 relative on ordinary inputs.  fp32 inputs are held
// to 1e-4, so their dgT, the cumulative sum and the dA_log partial are
// accumulated in fp64 (exact products of the fp32 factors); bf16 inputs keep
// fp32, far below their own 2e-2 bound.
template <typename E>
using GAcc = typename std::conditional<std::is_same<E, float>::value, double, float>::type;

template <typename E, int D> struct GradSmem {
  static constexpr int LD = tile_ld<E>(D);
  static constexpr int LDS = tile_ld<E>(64);
  static constexpr int LDF = D + 4;
  static constexpr size_t sz_E = 64 * LDF * 4;
  // the prep view, then dgT (D) and dA (8) as GAcc; the dbeta parts and
  // row dots reuse the view's column-partial scratch between the prep and the
  // cumsum, and so do the cumsum's segment totals (GAcc)
  static constexpr size_t n_small = PrepView<E, D>::floats + (D + 8) * (sizeof(GAcc<E>) / 4);
  static_assert(PrepView<E, D>::floats % 2 == 0, "dgT must be 8-byte aligned");
  static_assert((NTHREADS / D) * D * sizeof(GAcc<E>) <= 2 * NTHREADS * 4,
                "segment totals must fit the column-partial scratch");
  static constexpr size_t sz_small = ((n_small * 4 + 127) / 128) * 128;
  static constexpr size_t sz_G = 64 * 68 * 4;
  static constexpr size_t sz_sq = 64 * LDS * sizeof(E);
  static constexpr size_t sz_tile = 64 * LD * sizeof(E);
  static constexpr size_t o_E = 0;
  static constexpr size_t o_small = o_E + sz_E;
  static constexpr size_t o_INV = o_small + sz_small;
  static constexpr size_t o_MQK = o_INV + sz_sq;
  static constexpr size_t o_DA = o_MQK + sz_sq;
  static constexpr size_t o_BIG1 = o_DA + sz_sq;          // QM, KM -> S_n [D][LD]
  static constexpr size_t o_BIG2 = o_BIG1 + 2 * sz_tile;  // KP, KD -> dS_{n+1} -> QM, KM
  static constexpr size_t o_KR = o_BIG2 + 2 * sz_tile;    // KR -> dU -> dvcorr
  static constexpr size_t o_U = o_KR + sz_tile;           // inverse scratch -> U -> KP
  static constexpr size_t o_DO = o_U + sz_tile;           // inverse scratch -> dO
  static constexpr size_t o_V = o_DO + sz_tile;           // inverse scratch -> v -> Xr -> dgc
  static constexpr size_t o_G = o_V + sz_tile;
  static constexpr size_t total = o_G + (sz_G > sz_tile ? sz_G : sz_tile);
  static_assert(D * LD * sizeof(E) <= 2 * sz_tile, "state tile must fit two chunk tiles");
  static_assert(64 * 68 * 4 + 768 * 4 <= 3 * sz_tile, "inverse scratch must fit in U, dO, V");
  static_assert(3 * 64 * D * sizeof(E) <= 3 * sz_tile, "raw q, k, g must fit in U, dO, V");
  static_assert(64 * LDF * 4 <= sz_tile + (sz_G > sz_tile ? sz_G : sz_tile), "dgc must fit");
};

template <typename E, int D>
__global__ void __launch_bounds__(NTHREADS, 1) kda_grads_kernel(KdaParams p, const void *states) {
  using SM = GradSmem<E, D>;
  extern __shared__ __align__(128) char smem[];
  constexpr int LD = SM::LD, LDS = SM::LDS, LDF = SM::LDF;
  constexpr int NF = D / 16;  // 16 x (D/2) warp tiles
  const int64_t slot = blockIdx.x;
  const int h = blockIdx.y;
  const int H = p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int s, j, len;
  int64_t tok0;
  if (!slot_owner(p, slot, s, j, tok0, len)) {
    if (tid == 0) p.dA_part[slot * H + h] = 0.f;
    if (p.ddt_part != nullptr && tid < D) p.ddt_part[(slot * H + h) * D + tid] = 0.f;
    return;
  }
  (void)s;
  (void)j;

  // ---- shared memory views ----
  float *Eg = reinterpret_cast<float *>(smem + SM::o_E);
  float *sm = reinterpret_cast<float *>(smem + SM::o_small);
  PrepView<E, D> sv = make_view<E, D>(sm);
  using Acc = GAcc<E>;
  Acc *dgT = reinterpret_cast<Acc *>(sm + PrepView<E, D>::floats);  // [D]
  Acc *dAred = dgT + D;             // [8]
  float *dbp = sv.part;             // [4][64]: dbeta1 halves, dbeta2 halves
  float *rowdot = sv.part + 256;    // [2][64]
  Acc *partsum = reinterpret_cast<Acc *>(sv.part);  // [NTHREADS / D][D], the gate cumsum
  E *INV = reinterpret_cast<E *>(smem + SM::o_INV);
  E *MQK = reinterpret_cast<E *>(smem + SM::o_MQK);
  E *DA = reinterpret_cast<E *>(smem + SM::o_DA);
  E *BIG1 = reinterpret_cast<E *>(smem + SM::o_BIG1);
  E *BIG2 = reinterpret_cast<E *>(smem + SM::o_BIG2);
  E *KRt = reinterpret_cast<E *>(smem + SM::o_KR);
  E *Ut = reinterpret_cast<E *>(smem + SM::o_U);
  E *DOt = reinterpret_cast<E *>(smem + SM::o_DO);
  E *Vt = reinterpret_cast<E *>(smem + SM::o_V);
  float *G = reinterpret_cast<float *>(smem + SM::o_G);
  float *inv32 = reinterpret_cast<float *>(smem + SM::o_U);
  float *tbuf = inv32 + 64 * 68;
  float *dgc = reinterpret_cast<float *>(smem + SM::o_V);  // [64][LDF] over V and G

  const int rb = warp & 3;                 // row block of this warp
  const int ch = (warp >> 2) * (D / 2);    // column half
  const float scale = p.scale;
  const size_t DD = (size_t)D * D;
  const E *Sg = reinterpret_cast<const E *>(states) + ((size_t)slot * H + h) * DD;
  const E *dSg = reinterpret_cast<const E *>(p.dstates) + ((size_t)slot * H + h) * DD;

  if (tid < D) dgT[tid] = Acc(0);

  // ---- prep: norms, gates, operand tiles, pair matrices, inverse ----
  {
    // raw q, k, g rows staged into the (still unused) U / dO / v tiles
    E *Qr = reinterpret_cast<E *>(smem + SM::o_U);
    E *Kr = Qr + 64 * D;
    E *Gr = Kr + 64 * D;
    stage_chunk<E, D>(p, h, tok0, len, true, Qr, Kr, Gr, sv.beta);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    PrepTiles<E> tl;
    tl.QM = BIG1;
    tl.KM = BIG1 + 64 * LD;
    tl.KP = BIG2;
    tl.KD = BIG2 + 64 * LD;
    tl.KR = KRt;
    tl.Et = Eg;
    chunk_prep<E, D>(p, h, len, true, Qr, Kr, Gr, sv, tl, true);
  }
  intra_pairs<E, D>(BIG1, BIG1 + 64 * LD, BIG2, sv.F, G, 68, MQK, LDS, scale);
  __syncthreads();
  wy_inverse<E>(G, 68, sv.beta, inv32, tbuf, INV, LDS);
  // S_n -> BIG1, v -> Vt, asynchronously
  stage_dense<E>(BIG1, LD, Sg, D, D);
  stage_rows<E>(Vt, LD, p.v, tok0, len, H, h, D, 0, D);
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();

  float acc[NF][4], tmp[NF][4], dkr[NF][4];
  // ---- B2 (kdS) : Xr = v - kd S_n, in place ----
  zero_acc(acc);
  warp_gemm<NF, true, false>(acc, BIG2 + 64 * LD + 16 * rb * LD, LD, BIG1 + ch, LD, D);
  for_acc(acc, [&](int r, int c, float &x) {
    E *pv = Vt + (16 * rb + r) * LD + ch + c;
    *pv = from_f<E>(to_f(*pv) - x);
  });
  __syncthreads();
  // ---- U = INV diag(beta) Xr ; load dS_{n+1} -> BIG2, dO -> DOt ----
  zero_acc(acc);
  warp_gemm<NF, true, false>(acc, INV + 16 * rb * LDS, LDS, Vt + ch, LD, 64, sv.beta);
  // dS_{n+1} -> BIG2 (kd is dead), dO -> DOt (inverse scratch is dead)
  stage_dense<E>(BIG2, LD, dSg, D, D);
  stage_rows<E>(DOt, LD, p.dO, tok0, len, H, h, D, 0, D);
  cp_async_commit();
  store_acc(Ut + 16 * rb * LD + ch, LD, acc);
  cp_async_wait_all();
  __syncthreads();

  // ---- B1: dU = scale Mqk^T dO + kr dS ; dkr = U dS^T ; B0: p ----
  zero_acc(acc);
  warp_gemm<NF, false, false>(acc, MQK + 16 * rb, LDS, DOt + ch, LD, 64);
  warp_gemm<NF, true, false>(acc, KRt + 16 * rb * LD, LD, BIG2 + ch, LD, D);
  zero_acc(dkr);
  warp_gemm<NF, true, true>(dkr, Ut + 16 * rb * LD, LD, BIG2 + ch * LD, LD, D);
  // dkr' = dkr e^(gT - gc) (its column sums enter dgT in pass 2)
  for_acc(dkr, [&](int r, int c, float &x) {
    const int i = 16 * rb + r, cc = ch + c;
    x *= sv.egm[rb * D + cc] / Eg[i * LDF + cc];
  });
  // p_c = e^gT_c sum_d dS_cd S_cd  (D rows, 256 / D threads per row)
  {
    constexpr int TPR = NTHREADS / D;
    const int r = tid / TPR, part = tid % TPR;
    Acc acc_p = Acc(0);
    for (int d = part * (D / TPR); d < (part + 1) * (D / TPR); d += 2) {
      const float2 a = load2(BIG2 + r * LD + d);
      const float2 b = load2(BIG1 + r * LD + d);
      acc_p = fma(Acc(a.x), Acc(b.x), fma(Acc(a.y), Acc(b.y), acc_p));
    }
#pragma unroll
    for (int o = 1; o < TPR; o <<= 1) acc_p += __shfl_xor_sync(0xffffffffu, acc_p, o);
    if (part == 0) atomicAdd(&dgT[r], Acc(gate_exp<E>(sv.gT[r])) * acc_p);
  }
  __syncthreads();  // all reads of KRt, MQK, BIG2 (dS) done
  store_acc(KRt + 16 * rb * LD + ch, LD, acc);  // dU
  __syncthreads();

  // ---- dvcorr = INV^T dU ; dv ; dbeta1 ----
  zero_acc(acc);
  warp_gemm<NF, false, false>(acc, INV + 16 * rb, LDS, KRt + ch, LD, 64);
  {
    float rp[2] = {0.f, 0.f};
    for_acc(acc, [&](int r, int c, float &x) {
      const float xr = to_f(Vt[(16 * rb + r) * LD + ch + c]);
      rp[r >= 8] = fmaf(x, xr, rp[r >= 8]);
    });
    const int r0 = lane >> 2;
    rp[0] = quad_sum(rp[0]);
    rp[1] = quad_sum(rp[1]);
    if ((lane & 3) == 0) {
      dbp[(warp >> 2) * 64 + 16 * rb + r0] = rp[0];
      dbp[(warp >> 2) * 64 + 16 * rb + r0 + 8] = rp[1];
    }
    // dv = beta dvcorr
    E *dvg = reinterpret_cast<E *>(p.dv);
    const int c0 = 2 * (lane & 3);
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = 16 * rb + r0 + 8 * hh;
        if (i < len) {
          const float b = sv.beta[i];
          store2(dvg + ((tok0 + i) * H + h) * D + ch + 8 * f + c0, b * acc[f][2 * hh],
                 b * acc[f][2 * hh + 1]);
        }
      }
  }
  __syncthreads();  // all reads of dU done
  store_acc(KRt + 16 * rb * LD + ch, LD, acc);  // dvcorr
  __syncthreads();

  // ---- B3: dMqk = lower(scale dO U^T), dAkk = -strict_lower(dvcorr U^T) ----
  {
    const int jh = (warp >> 2) * 32;  // 32 columns (chunk rows j) per warp
    float am[4][4], aa[4][4];
    zero_acc(am);
    zero_acc(aa);
    warp_gemm<4, true, true>(am, DOt + 16 * rb * LD, LD, Ut + jh * LD, LD, D);
    warp_gemm<4, true, true>(aa, KRt + 16 * rb * LD, LD, Ut + jh * LD, LD, D);
    float rp[2] = {0.f, 0.f};
    const int lr = lane >> 2, lc = 2 * (lane & 3);
#pragma unroll
    for (int f = 0; f < 4; ++f)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 16 * rb + lr + ((e >> 1) << 3);
        const int jj = jh + 8 * f + lc + (e & 1);
        const float vm = jj <= i ? scale * am[f][e] : 0.f;
        const float va = jj < i ? -aa[f][e] : 0.f;
        MQK[i * LDS + jj] = from_f<E>(vm);
        DA[i * LDS + jj] = from_f<E>(sv.beta[i] * va);
        rp[e >> 1] = fmaf(va, G[i * 68 + jj], rp[e >> 1]);
      }
    rp[0] = quad_sum(rp[0]);
    rp[1] = quad_sum(rp[1]);
    if ((lane & 3) == 0) {
      dbp[128 + (warp >> 2) * 64 + 16 * rb + lr] = rp[0];
      dbp[128 + (warp >> 2) * 64 + 16 * rb + lr + 8] = rp[1];
    }
  }
  __syncthreads();
  // dbeta
  if (tid < len) {
    const float db = dbp[tid] + dbp[64 + tid] + dbp[128 + tid] + dbp[192 + tid];
    reinterpret_cast<E *>(p.dbeta)[(tok0 + tid) * H + h] = from_f<E>(db);
  }
  // raw q, k rows -> the v / G tiles (both dead after B3), in flight while
  // the inter-chunk products run
  E *Qraw = Vt, *Kraw = Vt + 64 * D;
  stage_rows<E>(Qraw, D, p.q, tok0, len, H, h, D, 0, D);
  stage_rows<E>(Kraw, D, p.k, tok0, len, H, h, D, 0, D);
  cp_async_commit();
  // ---- B2 inter-chunk products while S_n and dO are resident ----
  float bq[NF][4], bk[NF][4];
  zero_acc(bq);
  zero_acc(bk);
  warp_gemm<NF, true, true>(bq, DOt + 16 * rb * LD, LD, BIG1 + ch * LD, LD, D);  // dO S^T
  warp_gemm<NF, true, true>(bk, KRt + 16 * rb * LD, LD, BIG1 + ch * LD, LD, D);  // dvcorr S^T
  __syncthreads();  // S_n (BIG1), dO (DOt) and dvcorr (KRt) are dead from here on
  // raw g rows -> KRt, for the gate epilogue
  E *Graw = KRt;
  stage_rows<E>(Graw, D, p.g, tok0, len, H, h, D, 0, D);
  cp_async_commit();
  asm volatile("cp.async.wait_group 1;\n" ::);  // q, k have landed
  __syncthreads();
  // Operands of the intra-chunk gradient products, rebuilt in fp32 from q, k
  // and E.  These products feed the gate gradient, whose reverse cumulative
  // sum cancels them pairwise; bf16 rounding of the keys / queries alone
  // would leave a residue of a few 1e-2 in dg.  They are therefore carried
  // as two bf16 terms, hi = bf16(x) and lo = bf16(x - hi) (about 16 mantissa
  // bits), and every product is taken twice on the tensor cores.
  E *QMt = BIG2, *KMt = BIG2 + 64 * LD, *KPt = Ut;
  E *QMl = BIG1, *KMl = BIG1 + 64 * LD, *KPl = DOt;
  constexpr bool kSplit = sizeof(E) == 2;
  for (int e = tid; e < 64 * D / 2; e += NTHREADS) {
    const int i = e / (D / 2), c = 2 * (e % (D / 2));
    const float2 qv = load2(Qraw + i * D + c);
    const float2 kv = load2(Kraw + i * D + c);
    const float q0 = qv.x * sv.rq[i], q1 = qv.y * sv.rq[i];
    const float k0 = kv.x * sv.rk[i], k1 = kv.y * sv.rk[i];
    const float e0 = Eg[i * LDF + c], e1 = Eg[i * LDF + c + 1];
    const float x[6] = {q0 * e0, q1 * e1, k0 * e0, k1 * e1, k0 / e0, k1 / e1};
    E *hi[3] = {QMt, KMt, KPt};
    E *lo[3] = {QMl, KMl, KPl};
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      store2(hi[t] + i * LD + c, x[2 * t], x[2 * t + 1]);
      if (kSplit) {
        const float2 hv = load2(hi[t] + i * LD + c);
        store2(lo[t] + i * LD + c, x[2 * t] - hv.x, x[2 * t + 1] - hv.y);
      }
    }
  }
  __syncthreads();
  // normalised q / k of an element from the resident operand tiles
  auto qhat = [&](int i, int c) {
    float x = to_f(QMt[i * LD + c]);
    if (kSplit) x += to_f(QMl[i * LD + c]);
    return x / Eg[i * LDF + c];
  };
  auto khat = [&](int i, int c) {
    float x = to_f(KMt[i * LD + c]);
    if (kSplit) x += to_f(KMl[i * LD + c]);
    return x / Eg[i * LDF + c];
  };

  const int r0 = lane >> 2, c0 = 2 * (lane & 3);
  // W_I,J (16 x 16 block of W) times the hi + lo operand rows of block J
  auto intra_b = [&](float (&out)[NF][4], const E *Wt, const E *Zh, const E *Zl) {
    zero_acc(out);
    for (int J = 0; J <= rb; ++J) {
      zero_acc(tmp);
      warp_gemm<NF, true, false>(tmp, Wt + 16 * rb * LDS + 16 * J, LDS, Zh + 16 * J * LD + ch,
                                 LD, 16);
      if (kSplit)
        warp_gemm<NF, true, false>(tmp, Wt + 16 * rb * LDS + 16 * J, LDS,
                                   Zl + 16 * J * LD + ch, LD, 16);
      const float *Fp = J < rb ? sv.F + pair_index(rb, J) * D + ch : nullptr;
#pragma unroll
      for (int f = 0; f < NF; ++f)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float fct = Fp ? Fp[8 * f + c0 + (e & 1)] : 1.f;
          out[f][e] = fmaf(tmp[f][e], fct, out[f][e]);
        }
    }
  };

  // ---- pass 1: dq^ = gamma (scale dO S^T) + E sum_J (dMqk_IJ KP_J) F_IJ ----
  {
    float intra[NF][4];
    intra_b(intra, MQK, KPt, KPl);
    float rp[2] = {0.f, 0.f};
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 16 * rb + r0 + ((e >> 1) << 3);
        const int c = ch + 8 * f + c0 + (e & 1);
        const float Ev = Eg[i * LDF + c];
        const float gam = Ev * sv.em[rb * D + c];
        const float dqh = scale * gam * bq[f][e] + Ev * intra[f][e];
        bq[f][e] = dqh;
        const float qh = qhat(i, c);
        tmp[f][e] = qh;
        dgc[i * LDF + c] = dqh * qh;
        rp[e >> 1] = fmaf(dqh, qh, rp[e >> 1]);
      }
    rp[0] = quad_sum(rp[0]);
    rp[1] = quad_sum(rp[1]);
    if ((lane & 3) == 0) {
      rowdot[(warp >> 2) * 64 + 16 * rb + r0] = rp[0];
      rowdot[(warp >> 2) * 64 + 16 * rb + r0 + 8] = rp[1];
    }
    __syncthreads();
    E *dqg = reinterpret_cast<E *>(p.dq);
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = 16 * rb + r0 + 8 * hh;
        if (i < len) {
          const float rd = rowdot[i] + rowdot[64 + i];
          const int c = ch + 8 * f + c0;
          const float a0 = (bq[f][2 * hh] - tmp[f][2 * hh] * rd) * sv.rq[i];
          const float a1 = (bq[f][2 * hh + 1] - tmp[f][2 * hh + 1] * rd) * sv.rq[i];
          store2(dqg + ((tok0 + i) * H + h) * D + c, a0, a1);
        }
      }
    __syncthreads();  // rowdot reused below
  }

  // ---- pass 2: dk ----
  {
    // dkd' = -beta gamma (dvcorr S^T) + E sum_J (dA_IJ KP_J) F_IJ
    float intra[NF][4];
    intra_b(intra, DA, KPt, KPl);
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 16 * rb + r0 + ((e >> 1) << 3);
        const int c = ch + 8 * f + c0 + (e & 1);
        const float Ev = Eg[i * LDF + c];
        const float gam = Ev * sv.em[rb * D + c];
        bk[f][e] = -sv.beta[i] * gam * bk[f][e] + Ev * intra[f][e];
      }
    // dki' = E^-1 sum_{I >= rb} (dMqk_I,rb^T QM_I + dA_I,rb^T KM_I) F_I,rb
    zero_acc(intra);
    for (int I = rb; I < 4; ++I) {
      zero_acc(tmp);
      const E *Wq = MQK + 16 * I * LDS + 16 * rb, *Wk = DA + 16 * I * LDS + 16 * rb;
      warp_gemm<NF, false, false>(tmp, Wq, LDS, QMt + 16 * I * LD + ch, LD, 16);
      warp_gemm<NF, false, false>(tmp, Wk, LDS, KMt + 16 * I * LD + ch, LD, 16);
      if (kSplit) {
        warp_gemm<NF, false, false>(tmp, Wq, LDS, QMl + 16 * I * LD + ch, LD, 16);
        warp_gemm<NF, false, false>(tmp, Wk, LDS, KMl + 16 * I * LD + ch, LD, 16);
      }
      const float *Fp = I > rb ? sv.F + pair_index(I, rb) * D + ch : nullptr;
#pragma unroll
      for (int f = 0; f < NF; ++f)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float fct = Fp ? Fp[8 * f + c0 + (e & 1)] : 1.f;
          intra[f][e] = fmaf(tmp[f][e], fct, intra[f][e]);
        }
    }
    float rp[2] = {0.f, 0.f};
    Acc colp[NF][2];
#pragma unroll
    for (int f = 0; f < NF; ++f) colp[f][0] = colp[f][1] = Acc(0);
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 16 * rb + r0 + ((e >> 1) << 3);
        const int c = ch + 8 * f + c0 + (e & 1);
        const float dki = intra[f][e] / Eg[i * LDF + c];
        const float dkd = bk[f][e];
        const float dkh = dkd + dki + dkr[f][e];
        const float dks = dkd - dki - dkr[f][e];
        const float kh = khat(i, c);
        bk[f][e] = dkh;
        tmp[f][e] = kh;
        dgc[i * LDF + c] += dks * kh;
        rp[e >> 1] = fmaf(dkh, kh, rp[e >> 1]);
        colp[f][e & 1] = fma(Acc(dkr[f][e]), Acc(kh), colp[f][e & 1]);
      }
    // dgT += sum over the chunk rows of dkr' k^ (same k^ as the cancelling term)
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        Acc v = colp[f][x];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        if ((lane >> 2) == 0) atomicAdd(&dgT[ch + 8 * f + c0 + x], v);
      }
    rp[0] = quad_sum(rp[0]);
    rp[1] = quad_sum(rp[1]);
    if ((lane & 3) == 0) {
      rowdot[(warp >> 2) * 64 + 16 * rb + r0] = rp[0];
      rowdot[(warp >> 2) * 64 + 16 * rb + r0 + 8] = rp[1];
    }
    __syncthreads();
    E *dkg = reinterpret_cast<E *>(p.dk);
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = 16 * rb + r0 + 8 * hh;
        if (i < len) {
          const float rd = rowdot[i] + rowdot[64 + i];
          const int c = ch + 8 * f + c0;
          const float a0 = (bk[f][2 * hh] - tmp[f][2 * hh] * rd) * sv.rk[i];
          const float a1 = (bk[f][2 * hh + 1] - tmp[f][2 * hh + 1] * rd) * sv.rk[i];
          store2(dkg + ((tok0 + i) * H + h) * D + c, a0, a1);
        }
      }
  }
  cp_async_wait_all();  // raw g
  __syncthreads();

  // ---- K1: reverse cumsum of dgc over the chunk rows, dg, dA_log ----
  {
    constexpr int PARTS = NTHREADS / D;     // row segments per column
    constexpr int SEG = 64 / PARTS;
    const int c = tid % D, part = tid / D;
    const int ra = part * SEG;
    Acc tot = Acc(0);
    for (int i = ra; i < ra + SEG; ++i) tot += dgc[i * LDF + c];
    partsum[part * D + c] = tot;
    __syncthreads();
    Acc run = dgT[c];
    for (int q2 = part + 1; q2 < PARTS; ++q2) run += partsum[q2 * D + c];
    const float A = gate_exp<E>(p.A_log[h]);
    const float bias = gate_bias(p, h, c, D);
    Acc dA = Acc(0);
    float ddt = 0.f;
    E *dgg = reinterpret_cast<E *>(p.dg);
    for (int i = ra + SEG - 1; i >= ra; --i) {
      run += dgc[i * LDF + c];
      if (i < len) {
        const float gv = to_f(Graw[i * D + c]) + bias;
        const float gk = -A * softplus_f(gv);
        const float dgv = (float)run * (-A) / (1.f + gate_exp<E>(-gv));
        dgg[((tok0 + i) * H + h) * D + c] = from_f<E>(dgv);
        dA = fma(run, Acc(gk), dA);
        ddt += dgv;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dA += __shfl_xor_sync(0xffffffffu, dA, o);
    if (lane == 0) dAred[warp] = dA;
    __syncthreads();
    if (tid == 0) {
      Acc t = Acc(0);
      for (int w = 0; w < NWARPS; ++w) t += dAred[w];
      p.dA_part[slot * H + h] = (float)t;
    }
    if (p.ddt_part != nullptr) {  // ddt_bias partial of the chunk: the dg column sums
      partsum[part * D + c] = ddt;  // (every thread has read partsum above)
      __syncthreads();
      if (part == 0) {
        Acc t = Acc(0);
        for (int q2 = 0; q2 < PARTS; ++q2) t += partsum[q2 * D + c];
        p.ddt_part[(slot * H + h) * D + c] = (float)t;
      }
    }
  }
}

// Deterministic dA_log: one CTA per head sums the per-chunk partials in a
// fixed order.
__global__ void kda_dalog_reduce_kernel(const float *part, int64_t nslots, int H, float *dA) {
  __shared__ float red[NWARPS];
  pdl_wait();  // the gradient kernels' partials
  const int h = blockIdx.x;
  float t = 0.f;
  for (int64_t s = threadIdx.x; s < nslots; s += NTHREADS) t += part[s * H + h];
  t = warp_sum(t);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    float x = 0.f;
    for (int w = 0; w < NWARPS; ++w) x += red[w];
    dA[h] = x;
  }
}

// Deterministic ddt_bias: one CTA per head, thread (c, r) sums the partials of
// channel c over the slots s = r, r + R, ... (coalesced over c), then the R
// sums of each channel in a fixed order.
__global__ void __launch_bounds__(1024) kda_ddt_reduce_kernel(const float *part, int64_t nslots,
                                                              int H, int K, float *ddt) {
  __shared__ float red[1024];
  const int h = blockIdx.x, c = threadIdx.x, r = threadIdx.y, R = blockDim.y;
  float t = 0.f;
  for (int64_t s = r; s < nslots; s += R) t += part[(s * H + h) * K + c];
  red[r * K + c] = t;
  __syncthreads();
  if (r == 0) {
    float x = 0.f;
    for (int q = 0; q < R; ++q) x += red[q * K + c];
    ddt[h * K + c] = x;
  }
}

// bf16 K = V = 128 runs on the tcgen05 kernel (kda_grads_tc.cu) unless the
// environment variable KDA_GRADS_MMA_SYNC is set (A/B comparisons).
static bool use_tc_kernel() {
  static const bool tc = getenv("KDA_GRADS_MMA_SYNC") == nullptr;
  return tc;
}

template <typename E, int D>
static cudaError_t launch_grads(const KdaParams &p, const void *states, cudaStream_t st,
                                void *after, const TokenMaps *tm) {
  using SM = GradSmem<E, D>;
  cudaError_t e;
  // packed state tiles (tcgen05 scans) are read by the tcgen05 kernel only
  if ((p.states_packed || p.dstates_packed) && tm == nullptr) return cudaErrorInvalidValue;
  if (sizeof(E) == 2 && D == 128 && tm != nullptr &&
      (use_tc_kernel() || p.states_packed || p.dstates_packed)) {
    e = grads_tc_launch(p, *tm, states, st);
    if (e == cudaSuccess) e = range_grads_launch(p, states, st);  // flagged chunks, exactly
    if (e != cudaSuccess) return e;
  } else {
    auto kfn = kda_grads_kernel<E, D>;
    e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM::total);
    if (e != cudaSuccess) return e;
    if (p.nslots > 0) {
      kfn<<<dim3((unsigned)p.nslots, p.H), NTHREADS, SM::total, st>>>(p, states);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  if (after != nullptr) cudaEventRecord(reinterpret_cast<cudaEvent_t>(after), st);
  cudaError_t er = pdl_launch(kda_dalog_reduce_kernel, dim3(p.H), dim3(NTHREADS), 0, st, p.dA_part,
                              p.nslots, p.H, p.dA_log);
  if (er == cudaSuccess && p.ddt_bias != nullptr && p.H > 0)
    kda_ddt_reduce_kernel<<<p.H, dim3(D, 1024 / D), 0, st>>>(p.ddt_part, p.nslots, p.H, D,
                                                             p.ddt_bias);
  return er != cudaSuccess ? er : cudaGetLastError();
}

cudaError_t grads_dispatch(const KdaParams &p, int K, bool is_bf16, const void *states,
                           cudaStream_t st, void *after, const TokenMaps *tm) {
  if (is_bf16) {
    if (K == 128) return launch_grads<bf16, 128>(p, states, st, after, tm);
    if (K == 64) return launch_grads<bf16, 64>(p, states, st, after, tm);
  } else {
    if (K == 64) return launch_grads<float, 64>(p, states, st, after, tm);
  }
  return cudaErrorInvalidValue;
}

size_t grads_smem_bytes(int K, bool is_bf16) {
  if (is_bf16) return K == 128 ? GradSmem<bf16, 128>::total : GradSmem<bf16, 64>::total;
  return GradSmem<float, 64>::total;
}

int grads_status_take() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_status, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

}  // namespace kda
