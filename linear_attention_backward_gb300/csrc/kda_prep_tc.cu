// kda_prep_tc.cu -- chunk-parallel prep of the state-scan operands (bf16,
// K = V = 128): one CTA per (chunk slot, head), two CTAs per SM.
//
// Per chunk it forms, from q, k, v, g and beta (gate and range-safety
// conventions as in kda_chunk.cuh):
//   W  = (I + Akk)^-1 diag(beta) kd       U0 = (I + Akk)^-1 diag(beta) v
//   QE = scale (qd - Mqk W)               kr = k^ e^(gT - gc),  gT
// (all four 64 x 128 tiles stored transposed, channel-major, see kda_params.h)
// and keeps the pair matrices G, scale Mqk and the inverses INV, INV diag(beta)
// for the gradient kernel, which then does not form them again.
// With these the two serial recurrences of the backward ("all_states" of
// kernel B2 and Kernel A, "bwd-kernelB-beginner-guide-full", Part 2, and the
// A/B table of "bwd-ncu-and-optimization-playbook") need nothing else per
// chunk than products with the running state:
//   U     = U0 - W S_n,                  S_{n+1} = e^gT S_n + kr^T U
//   dS_n  = e^gT dS_{n+1} - W^T (kr dS_{n+1}) + QE^T dO
// The second line is Kernel A's update with dU and dvcorr substituted:
// kd^T diag(beta) (I + Akk)^-T = W^T, so
//   scale qd^T dO - kd^T diag(beta) dvcorr
//     = scale qd^T dO - W^T (scale Mqk^T dO + kr dS_{n+1}).
//
// Layout of the work: thread (channel pair, 16-row block) for the gate, the
// norms and the decay-scaled tiles (loaded straight from HBM into
// registers); mma.sync for the 16-row pair blocks of Akk and Mqk (they carry
// a per-channel factor on the contraction index, see kda_chunk.cuh); the
// WY inverse in fp32; tcgen05 for the three 64 x 64 x 128 products, whose
// results land transposed (channel = TMEM lane) and are written to HBM as
// 16-byte rows of packed core matrices, the byte order the scans copy into
// shared memory as one bulk copy.
#include "kda_chunk.cuh"
#include "kda_tc_tiles.cuh"

namespace kda {
namespace ptc {

using namespace tct;
constexpr int D = 128;
constexpr uint32_t T64x128 = umma::ptile_bytes(64, 128);  // 18432 (padded)
constexpr uint32_t T64x64 = umma::ptile_bytes(64, 64);    // 9216 (padded)

struct Smem {
  static constexpr size_t n_view = PrepView<bf16, D>::floats;
  // extra floats: tbuf 768 (inverse), red 2 x 8 x 16 (row norms)
  static constexpr size_t n_extra = 768 + 256;
  static constexpr size_t sz_small = (((n_view + n_extra) * 4 + 64 + 1023) / 1024) * 1024;
  static constexpr size_t o_QM = sz_small;          // q^ e^(gc - m)  [i][c] padded
  static constexpr size_t o_KM = o_QM + T64x128;    // k^ e^(gc - m)  [i][c] padded
  static constexpr size_t o_KP = o_KM + T64x128;    // k^ e^(m - gc)  -> later Mqk [i][j]
  static constexpr size_t o_V = o_KP + T64x128;     // v: two 64-channel swizzled boxes [j][v]
  static constexpr size_t o_G = o_V + 16384;        // G / INV fp32 [64][68] -> later W^T
  static constexpr size_t o_INVb = o_G + 64 * kGfStride * 4;  // INV diag(beta) [i][j] padded
  static constexpr size_t total = o_INVb + T64x64;
  static_assert(total + 1024 <= 233472 / 2, "two CTAs per SM");
  static_assert(o_V % 1024 == 0, "swizzled boxes start on 1024-byte atoms");
  static_assert(o_G % 16 == 0 && (kGfStride * 4) % 16 == 0 && (19 * D * 4) % 16 == 0,
                "16-byte loads (lds4) of the inverse's rows and the view's rq, rk, beta");
};

}  // namespace ptc

// kMode: what the kernel writes beyond the scans' operands (kPrepAll,
// kPrepReadout, kPrepStates; kda_params.h), one instance each
template <uint32_t kMode>
__global__ void __launch_bounds__(NTHREADS, 2)
    kda_prep_tc_kernel(KdaParams p, const __grid_constant__ TokenMaps tm, char *prep) {
  using namespace ptc;
  using SM = ptc::Smem;
  extern __shared__ __align__(1024) char smem[];
  const int64_t slot = blockIdx.x;
  const int h = blockIdx.y;
  const int H = p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int s_, j_, len;
  int64_t tok0;
  if (!slot_owner(p, slot, s_, j_, tok0, len)) {  // padding slot: never read
    if (tid == 0 && p.range_flags != nullptr) p.range_flags[slot * H + h] = 0;
    return;
  }
  char *unit = prep + ((size_t)slot * H + h) * kPrepUnitBytes;
  // the gate's per-head scale and per-channel bias, loaded now (first used
  // after the raw rows have landed, so their latency hides behind that wait)
  const int c_g = 2 * (tid & 63);
  const float a_log = p.A_log[h];
  const float bias0 = gate_bias(p, h, c_g, D), bias1 = gate_bias(p, h, c_g + 1, D);

  float *smf = reinterpret_cast<float *>(smem);
  PrepView<bf16, D> sv = make_view<bf16, D>(smf);
  float *tbuf = smf + SM::n_view;
  float *red = tbuf + 768;  // [2 (k, q)][8 warps][16 rows]
  uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + (SM::n_view + SM::n_extra) * 4);
  uint64_t *rbar = mbar + 1;  // TMA boxes of the raw q, k, g rows
  uint64_t *vbar = mbar + 2;  // TMA boxes of the v rows
  uint32_t *tslot = reinterpret_cast<uint32_t *>(mbar + 3);
  int *far_s = reinterpret_cast<int *>(tslot + 1);  // a channel passes the block range
  int *weak_s = far_s + 1;  // a live channel decays by at most kStrongTokenDecay per token
  // live channels (a nonzero key row in the chunk; a zero-padded channel is not):
  // word 2 q + o, bit l = channel 64 q + 2 l + o
  uint32_t *live_s = reinterpret_cast<uint32_t *>(weak_s + 1);
  char *QM = smem + SM::o_QM, *KM = smem + SM::o_KM, *KP = smem + SM::o_KP;
  char *Mqk = KP;
  char *Vt = smem + SM::o_V;
  float *Gf = reinterpret_cast<float *>(smem + SM::o_G);
  char *Wt = smem + SM::o_G;
  char *INVb = smem + SM::o_INVb;
  const float scale = p.scale;

  // raw q, k, g rows (row-major [64][128]) into the tile region, which the
  // tiles overwrite only after every thread has taken its rows; thread 0 issues
  // them as soon as the barriers exist, and the v rows as two 64-channel boxes
  // in the 128-byte swizzled layout, which the U0^T product reads MN-major as
  // they land; warp 0 then allocates Tensor Memory
  const bf16 *Qraw = reinterpret_cast<const bf16 *>(QM);
  const bf16 *Kraw = Qraw + 64 * D, *Graw = Kraw + 64 * D;
  if (tid == 0) {
    umma::mbar_init(mbar, 1);
    umma::mbar_init(rbar, 1);
    umma::mbar_init(vbar, 1);
    *far_s = 0;
    *weak_s = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) live_s[w] = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    umma::mbar_expect_tx(rbar, 3 * 16384u);
    umma::mbar_expect_tx(vbar, 16384u);
    if ((p.starve & kStarvePrep) == 0u) {  // (a timeout test arms the barriers only)
      umma::tma_load_3d(QM, &tm.q, 0, h, (int)tok0, rbar);
      umma::tma_load_3d(QM + 16384, &tm.k, 0, h, (int)tok0, rbar);
      umma::tma_load_3d(QM + 32768, &tm.g, 0, h, (int)tok0, rbar);
      umma::tma_load_3d(Vt, &tm.v_sw, 0, h, (int)tok0, vbar);
      umma::tma_load_3d(Vt + 8192, &tm.v_sw, 64, h, (int)tok0, vbar);
    }
  }
  if (warp == 0) umma::tmem_alloc(tslot, 256);
  __syncthreads();
  if (tid < CHUNK)
    sv.beta[tid] = tid < len ? __bfloat162float(reinterpret_cast<const bf16 *>(p.beta)[(tok0 + tid) * H + h])
                             : 0.f;

  // ---- raw rows straight into registers: thread (channel pair cp, block I) ----
  const int cp = tid & 63, I = tid >> 6, c = 2 * cp;
  uint32_t kraw[16], qraw[16];
  float g0[16], g1[16];
  // Every bounded wait folds its result into `ok`; the CTA decides at its
  // barriers (__syncthreads_or).  Once a wait has given up no further MMA is
  // issued, the CTA drains what is in flight and releases Tensor Memory
  // (`drain` below).  What a timed-out product left in Tensor Memory may
  // reach this call's operand blocks, whose status word then reports the
  // timeout.
  bool ok;
  uint32_t phase = 0;  // completions of the MMA barrier waited for
  {
    uint32_t graw[16];
    ok = umma::mbar_wait(rbar, 0, poll_cap(p, umma::kPollLoads));
#pragma unroll
    for (int r = 0; r < 16; ++r) {  // rows past the chunk (the next sequence's) read as zero
      const int i = 16 * I + r;
      const bool ok = i < len;
      kraw[r] = ok ? *reinterpret_cast<const uint32_t *>(Kraw + i * D + c) : 0u;
      qraw[r] = ok ? *reinterpret_cast<const uint32_t *>(Qraw + i * D + c) : 0u;
      graw[r] = ok ? *reinterpret_cast<const uint32_t *>(Graw + i * D + c) : 0u;
    }
    // norms: per-row partial sums over this thread's two channels
    float sk[16], sq[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float2 kv = bf2_to_f2(kraw[r]), qv = bf2_to_f2(qraw[r]);
      sk[r] = fmaf(kv.x, kv.x, kv.y * kv.y);
      sq[r] = fmaf(qv.x, qv.x, qv.y * qv.y);
    }
    const float tk = rows16_sum(sk);
    const float tq = rows16_sum(sq);
    if ((lane & 1) == 0) {  // lanes 2 r, 2 r + 1 hold row 16 I + r
      red[warp * 16 + (lane >> 1)] = tk;
      red[128 + warp * 16 + (lane >> 1)] = tq;
    }
    // gate: running sum over the block (sums local to the block)
    const float A = __expf(a_log);
    float run0 = 0.f, run1 = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const bool ok = 16 * I + r < len;
      const float2 gv = bf2_to_f2(graw[r]);
      run0 += ok ? -A * softplus_gate(gv.x + bias0) : 0.f;
      run1 += ok ? -A * softplus_gate(gv.y + bias1) : 0.f;
      g0[r] = run0;
      g1[r] = run1;
    }
    // log-decay around the block's reference row (row 7): rows 0..7 and 8..15.
    // Past the range the chunk is flagged for the exact kernels of
    // kda_range.cu (or, without a flag array, reported)
    const float span = fmaxf(fmaxf(g0[0] - g0[7], g0[7] - g0[15]),
                             fmaxf(g1[0] - g1[7], g1[7] - g1[15]));
    if (p.range_flags == nullptr) check_block_log_decay(span);
    else if (span > kMaxBlockLogDecay) *far_s = 1;
    {
      uint32_t any = 0u;
#pragma unroll
      for (int r = 0; r < 16; ++r) any |= kraw[r];
      // this warp's lanes hold channels 64 (warp & 1) + 2 lane (+ 1)
      const uint32_t m0 = __ballot_sync(0xffffffffu, (any & 0xffffu) != 0u);
      const uint32_t m1 = __ballot_sync(0xffffffffu, (any >> 16) != 0u);
      if (lane == 0) {
        atomicOr(live_s + 2 * (warp & 1), m0);
        atomicOr(live_s + 2 * (warp & 1) + 1, m1);
      }
    }
    float *Ablk = sv.part, *Bblk = sv.m;
    Ablk[I * D + c] = g0[7];
    Ablk[I * D + c + 1] = g1[7];
    Bblk[I * D + c] = g0[15] - g0[7];
    Bblk[I * D + c + 1] = g1[15] - g1[7];
  }
  if (__syncthreads_or(!ok)) {
    if (tid == 0 && p.range_flags != nullptr) p.range_flags[slot * H + h] = *far_s;
    ok = false;
    goto drain;
  }
  {
  if (tid < CHUNK) {  // row norms: block I's rows live in warps 2I, 2I + 1
    const int ib = tid >> 4, r = tid & 15;
    sv.rk[tid] = rsqrtf(red[(2 * ib) * 16 + r] + red[(2 * ib + 1) * 16 + r] + p.eps);
    sv.rq[tid] = rsqrtf(red[128 + (2 * ib) * 16 + r] + red[128 + (2 * ib + 1) * 16 + r] + p.eps);
  } else if (tid >= 128) {  // per-(block, channel) factors from the block partials
    const int e = tid - 128;
    float a[4], bb[4];
#pragma unroll
    for (int L = 0; L < 4; ++L) {
      a[L] = sv.part[L * D + e];
      bb[L] = sv.m[L * D + e];
    }
    float before = 0.f, tot = 0.f;
#pragma unroll
    for (int L = 0; L < 4; ++L) tot += a[L] + bb[L];
#pragma unroll
    for (int L = 0; L < 4; ++L) {
      float after = bb[L];
#pragma unroll
      for (int L2 = L + 1; L2 < 4; ++L2) after += a[L2] + bb[L2];
      sv.em[L * D + e] = __expf(before + a[L]);  // e^(m_L)
      sv.egm[L * D + e] = __expf(after);         // e^(gT - m_L)
      before += a[L] + bb[L];
    }
#pragma unroll
    for (int I2 = 1; I2 < 4; ++I2)
#pragma unroll
      for (int J = 0; J < I2; ++J) {
        float d = bb[J] + a[I2];
#pragma unroll
        for (int L = J + 1; L < I2; ++L) d += a[L] + bb[L];
        sv.F[pair_index(I2, J) * D + e] = __expf(d);  // e^(m_I - m_J)
      }
    reinterpret_cast<float *>(unit + kPrepGT)[e] = tot;
    sv.gT[e] = tot;
    const bool live = (live_s[2 * (e >> 6) + (e & 1)] >> ((e & 63) >> 1)) & 1u;
    if (live && -tot <= kStrongTokenDecay * (float)len) *weak_s = 1;  // (same value from all)
  }
  __syncthreads();
  // the chunk goes to the exact kernels if a channel passes the block range,
  // or if every live channel decays strongly (kda_device.cuh)
  if (tid == 0) {
    if (p.range_flags != nullptr)
      p.range_flags[slot * H + h] = (*far_s != 0 || *weak_s == 0) ? 1 : 0;
    else if (*weak_s == 0)  // (only the backward runs without flags)
      set_status(kStatusGateRange);
  }
  // the block factors and the row norms for the gradient kernel (one 8 KB span
  // of the view: e^(m_I), e^(gT - m_I), e^(m_I - m_J), gT, 1/|q|, 1/|k|)
  static_assert(19 * D + 128 - 4 * D == kPrepSVBytes / 4, "factor span");
  constexpr bool grad_tiles = kMode == kPrepAll, readout = kMode != kPrepStates;
  if constexpr (grad_tiles)
    for (int e = tid; e < (int)(kPrepSVBytes / 16); e += NTHREADS)
      reinterpret_cast<uint4 *>(unit + kPrepSV)[e] = reinterpret_cast<const uint4 *>(sv.em)[e];
  // ---- decay-scaled tiles; kr^T goes straight to HBM ----
  {
    const float eg0 = sv.egm[I * D + c], eg1 = sv.egm[I * D + c + 1];
    char *kr_out = unit + kPrepKR;
#pragma unroll
    for (int h8 = 0; h8 < 2; ++h8) {
      float kr0[8], kr1[8];
      float rk8[8], rq8[8];  // the rows' norms, 16-byte loads
      lds4(sv.rk + 16 * I + 8 * h8, rk8);
      lds4(sv.rk + 16 * I + 8 * h8 + 4, rk8 + 4);
      lds4(sv.rq + 16 * I + 8 * h8, rq8);
      lds4(sv.rq + 16 * I + 8 * h8 + 4, rq8 + 4);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int r = 8 * h8 + t, i = 16 * I + r;
        const float rk = rk8[t], rq = rq8[t];
        const float2 kv = bf2_to_f2(kraw[r]), qv = bf2_to_f2(qraw[r]);
        const float kh0 = kv.x * rk, kh1 = kv.y * rk, qh0 = qv.x * rq, qh1 = qv.y * rq;
        const float d0 = g0[r] - g0[7], d1 = g1[r] - g1[7];
        const float e0 = __expf(d0), e1 = __expf(d1);
        const float ei0 = __expf(-d0), ei1 = __expf(-d1);
        const uint32_t off = pcore_off(i, c, D);
        *reinterpret_cast<uint32_t *>(QM + off) = f2_to_bf2(qh0 * e0, qh1 * e1);
        *reinterpret_cast<uint32_t *>(KM + off) = f2_to_bf2(kh0 * e0, kh1 * e1);
        *reinterpret_cast<uint32_t *>(KP + off) = f2_to_bf2(kh0 * ei0, kh1 * ei1);
        kr0[t] = (kh0 * ei0) * eg0;
        kr1[t] = (kh1 * ei1) * eg1;
      }
      // kr^T [c][i]: rows 16 I + 8 h8 .. + 7 of channels c and c + 1, 16-byte rows
      st16_bf(kr_out + umma::core_off(c, 16 * I + 8 * h8, 64), kr0);
      st16_bf(kr_out + umma::core_off(c + 1, 16 * I + 8 * h8, 64), kr1);
    }
  }
  __syncthreads();
  // ---- pair blocks: G = kd ki^T (strictly lower, fp32), scale * Mqk (lower) ----
  // 20 nonzero 16 x 16 blocks (I >= J, two sides); the 12 off-diagonal ones
  // carry the per-channel factor F_IJ.  Warp w takes one diagonal block
  // (side w / 4, I = w % 4) and off-diagonal blocks w and w + 8 of the list
  // below, so no warp does more than one diagonal and two scaled blocks.
  {
    const int Ib0 = warp & 3;
    const bool q0 = warp >= 4;
    float acc[3][2][4];
    int tI[3], tJ[3];
    bool tq[3], tv[3];
    tI[0] = Ib0; tJ[0] = Ib0; tq[0] = q0; tv[0] = true;
#pragma unroll
    for (int t = 1; t < 3; ++t) {
      const int o = warp + 8 * (t - 1);  // off-diagonal task index, 0..11
      tv[t] = o < 12;
      const int oi = o % 6;               // (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
      tI[t] = oi == 0 ? 1 : (oi < 3 ? 2 : 3);
      tJ[t] = oi == 0 ? 0 : (oi == 1 ? 0 : (oi == 2 ? 1 : oi - 3));
      tq[t] = o >= 6;
    }
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      zero_acc(acc[t]);
      if (tv[t])
        wg_core<2>(acc[t], tq[t] ? QM : KM, D, 16 * tI[t], 0, KP, D, 16 * tJ[t], 0, D,
                   t > 0 ? sv.F + pair_index(tI[t], tJ[t]) * D : nullptr);
    }
    // G (fp32, strictly lower) and the zero blocks above the diagonal
#pragma unroll
    for (int t = 0; t < 3; ++t)
      if (tv[t] && !tq[t])
        for_acc(acc[t], [&](int r, int cc, float &v) {
          const int i = 16 * tI[t] + r, jj = 16 * tJ[t] + cc;
          Gf[i * kGfStride + jj] = jj < i ? v : 0.f;
        });
    // blocks above the diagonal, u -> (I, J): (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
    for (int e = tid; e < 6 * 256; e += NTHREADS) {
      const int u = e >> 8, r = (e >> 4) & 15, cc = e & 15;
      const int Iu = u < 3 ? 0 : (u < 5 ? 1 : 2), Ju = u < 3 ? u + 1 : (u < 5 ? u - 1 : 3);
      Gf[(16 * Iu + r) * kGfStride + 16 * Ju + cc] = 0.f;
    }
    __syncthreads();  // KP is read by every warp above; Mqk overwrites it
#pragma unroll
    for (int t = 0; t < 3; ++t)
      if (tv[t] && tq[t])
        for_acc(acc[t], [&](int r, int cc, float &v) {
          const int i = 16 * tI[t] + r, jj = 16 * tJ[t] + cc;
          *pel(Mqk, i, jj, 64) = __float2bfloat16_rn(jj <= i ? scale * v : 0.f);
        });
    for (int e = tid; e < 6 * 256; e += NTHREADS) {  // the same blocks of Mqk
      const int u = e >> 8, r = (e >> 4) & 15, cc = e & 15;
      const int Iu = u < 3 ? 0 : (u < 5 ? 1 : 2), Ju = u < 3 ? u + 1 : (u < 5 ? u - 1 : 3);
      *pel(Mqk, 16 * Iu + r, 16 * Ju + cc, 64) = __float2bfloat16_rn(0.f);
    }
  }
  __syncthreads();
  // G for the gradient kernel (packed 64 x 64 tile; the inverse overwrites Gf)
  if constexpr (grad_tiles) {
    for (int e8 = tid; e8 < 64 * 8; e8 += NTHREADS) {
      const int i = e8 >> 3, j0 = (e8 & 7) * 8;
      st16_bf(unit + kPrepG + umma::core_off(i, j0, 64), Gf + i * kGfStride + j0);
    }
    __syncthreads();
  }
  // scale * Mqk for the gradient kernel, stored by the warps the inverse's
  // diagonal phase leaves idle
  inverse_inplace(Gf, sv.beta, tbuf, [&](int w4) {
    if constexpr (readout) {
      for (int e8 = 32 * w4 + lane; e8 < 64 * 8; e8 += 32 * (NWARPS - 4)) {
        const int i = e8 >> 3, j0 = (e8 & 7) * 8;
        *reinterpret_cast<uint4 *>(unit + kPrepMqk + umma::core_off(i, j0, 64)) =
            *reinterpret_cast<const uint4 *>(Mqk + pcore_off(i, j0, 64));
      }
    }
  });
  // INV diag(beta) as the W^T product's operand first; INV and INV diag(beta)
  // go to HBM while that product runs (it reads only the shared tile)
  for (int e8 = tid; e8 < 64 * 8; e8 += NTHREADS) {
    const int i = e8 >> 3, j0 = (e8 & 7) * 8;
    float x[8], b8[8];
    lds4(Gf + i * kGfStride + j0, x);
    lds4(Gf + i * kGfStride + j0 + 4, x + 4);
    lds4(sv.beta + j0, b8);
    lds4(sv.beta + j0 + 4, b8 + 4);
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] *= b8[u];
    pstore8(INVb, i, j0, 64, x);
  }
  umma::fence_async_smem();
  umma::tc_fence_before();
  __syncthreads();
  umma::tc_fence_after();
  const uint32_t tbase = *tslot;
  auto mma_wait = [&]() {
    ok = umma::mbar_wait(mbar, phase & 1, poll_cap(p, umma::kPollMma)) && ok;
    phase++;
    umma::tc_fence_after();
  };
  // ---- W^T per key block J (the block factor e^(m_J) is applied per lane below) ----
  if (tid == 0) {
    for (int J = 0; J < 4; ++J)
      gemm(tbase + 64 * J, opmn(KM, D, 16 * J), true, opk(INVb, 64, 16 * J), false, 64, 1, false);
    umma::mma_commit(mbar);
  }
  for (int e8 = tid; e8 < 64 * 8; e8 += NTHREADS) {
    const int i = e8 >> 3, j0 = (e8 & 7) * 8;
    float g8[8], x[8], b8[8];
    lds4(Gf + i * kGfStride + j0, g8);
    lds4(Gf + i * kGfStride + j0 + 4, g8 + 4);
    lds4(sv.beta + j0, b8);
    lds4(sv.beta + j0 + 4, b8 + 4);
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] = g8[u] * b8[u];
    if constexpr (grad_tiles) {
      const uint32_t off = umma::core_off(i, j0, 64);
      st16_bf(unit + kPrepINV + off, g8);
      st16_bf(unit + kPrepINVb + off, x);
    }
  }
  mma_wait();
  const int ch = tid & 127, gq = tid >> 7;  // TMEM lane (channel) and 32-column group
  {
    float w[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) w[r] = 0.f;
#pragma unroll
    for (int J = 0; J < 4; ++J) {
      float a[32];
      tld32(tbase, 64 * J, a);
      const float em = sv.em[J * D + ch];
#pragma unroll
      for (int r = 0; r < 32; ++r) w[r] = fmaf(em, a[r], w[r]);
    }
    // W^T's tile lies over INV's fp32 rows, which the stores above read; and
    // nothing leaves a CTA whose product wait gave up
    if (__syncthreads_or(!ok)) { ok = false; goto drain; }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t off = umma::core_off(ch, 32 * gq + 8 * q, 64);
      st16_bf(Wt + off, w + 8 * q);
      st16_bf(unit + kPrepW + off, w + 8 * q);
    }
  }
  ok = umma::mbar_wait(vbar, 0, poll_cap(p, umma::kPollLoads)) && ok;  // v has landed
  if (len < CHUNK) {
    // a sequence's partial last chunk: the v boxes' rows past it hold the next
    // sequence's rows; zero them (a row's 128 bytes stay within the row)
    for (int e = tid; e < 2 * 64 * 8; e += NTHREADS) {
      const int row = (e >> 3) & 63;
      if (row >= len)
        *reinterpret_cast<uint4 *>(Vt + (e >> 9) * 8192 + row * 128 + (e & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
    }
  }
  umma::fence_async_smem();
  umma::tc_fence_before();
  if (__syncthreads_or(!ok)) { ok = false; goto drain; }
  // ---- U0^T = v^T (INV diag(beta))^T ;  (Mqk W)^T = W^T Mqk^T ----
  if (tid == 0) {
    umma::tc_fence_after();
    gemm(tbase + 0, opsw_mn(Vt, 8192u), true, opk(INVb, 64), false, 64, 4, false);
    if constexpr (readout)
      gemm(tbase + 64, opk(Wt, 64, 0, CP), false, opk(Mqk, 64), false, 64, 4, false);
    umma::mma_commit(mbar);
  }
  mma_wait();
  if (__syncthreads_or(!ok)) { ok = false; goto drain; }  // nothing leaves after a timeout
  {
    float a[32];
    tld32(tbase, 0, a);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st16_bf(unit + kPrepU0 + umma::core_off(ch, 32 * gq + 8 * q, 64), a + 8 * q);
    if constexpr (!readout) goto drain;
    tld32(tbase, 64, a);
    const float em0 = sv.em[(2 * gq) * D + ch], em1 = sv.em[(2 * gq + 1) * D + ch];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const int i = 32 * gq + r;
      const float qd = pget(QM, i, ch, D) * (r < 16 ? em0 : em1);
      a[r] = fmaf(scale, qd, -a[r]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st16_bf(unit + kPrepQE + umma::core_off(ch, 32 * gq + 8 * q, 64), a + 8 * q);
  }
  }
drain:
  // every thread gets here (through a decision above, which set `ok` for the
  // whole CTA, or at the end of the work, after the last products' wait);
  // the barrier both ends every thread's Tensor Memory loads before the
  // release and lets the CTA agree on whether any wait gave up
  umma::tc_fence_before();
  if (__syncthreads_or(!ok)) {
    // a bounded wait gave up (the status word says so): let the copies and the
    // MMA batch that may still be in flight land before the CTA releases its
    // shared memory and Tensor Memory (thread 0, in warp 0, waits before the
    // release below)
    if (tid == 0) {
      const uint32_t lim = poll_cap(p, umma::kPollDrain);
      umma::mbar_wait(rbar, 0, lim);
      umma::mbar_wait(vbar, 0, lim);
      if (phase > 0) umma::mbar_wait(mbar, (phase - 1) & 1, lim);
    }
  }
  if (warp == 0) {
    __syncwarp();  // thread 0 may have drained alone: the release is warp-collective
    umma::tc_fence_after();
    umma::tmem_dealloc(*tslot, 256);
  }
}

cudaError_t prep_tc_launch(const KdaParams &p, const TokenMaps &tm, void *prep, cudaStream_t st) {
  auto kfn = p.prep_mode == kPrepStates    ? kda_prep_tc_kernel<kPrepStates>
             : p.prep_mode == kPrepReadout ? kda_prep_tc_kernel<kPrepReadout>
                                           : kda_prep_tc_kernel<kPrepAll>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)ptc::Smem::total);
  if (e != cudaSuccess) return e;
  if (p.nslots > 0) {
    kfn<<<dim3((unsigned)p.nslots, p.H), NTHREADS, ptc::Smem::total, st>>>(
        p, tm, static_cast<char *>(prep));
    e = cudaGetLastError();
  }
  return e;
}

int prep_tc_status_take() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_status, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

}  // namespace kda
