// kda_scan_tc.cu -- the two serial chunk scans of the KDA backward on the
// fifth-generation tensor cores (bf16, K = V = 128), streaming the per-chunk
// operands written by the prep kernel (kda_prep_tc.cu):
//
//  * forward role: the chunk-state recompute ("all_states", read by kernel
//    B2 of "bwd-kernelB-beginner-guide-full", Part 2, B2 optimisation 4)
//      U = U0 - W S_n,          S_{n+1} = e^gT S_n + kr^T U
//  * reverse role: Kernel A, the reverse scan of the per-chunk state
//    gradient ("bwd-ncu-and-optimization-playbook", A/B table)
//      dS_n = e^gT dS_{n+1} - W^T (kr dS_{n+1}) + QE^T dO
//
// One CTA per (sequence, head, role), two CTAs per SM, all 256 threads on
// the epilogues.  Per chunk two tcgen05 products, both with the channel
// dimension (128) as M:
//   MMA1  T1[v][i] = sum_c X[c][v] B1[i][c]       N = 64,  K = 128
//         (B1 = W forward, kr reverse; T1^T = W S_n or kr dS_{n+1})
//   MMA2  T2[c][v] = sum_i A2[i][c] U[i][v] (+ sum_i QE[i][c] dO[i][v])
//         (A2 = kr forward, W reverse)             N = 128, K = 64
// The fp32 running state X stays in registers (thread = TMEM lane c and one
// half of the V columns); its bf16 copy in shared memory is MMA1's operand
// and is what goes to HBM as the chunk's state (the grads kernel reads the
// same rounding the scan used), stored from the tile with one bulk copy per
// chunk: states and dstates written here are in packed core-matrix order.  The chunk's
// operands (gT, W^T, kr^T, U0^T or QE^T; 48.5 KB) arrive by bulk TMA copies
// into three regions with one mbarrier each; a region is refilled with the
// next chunk's data as soon as its consumer (MMA1, the U epilogue or MMA2)
// is done, behind an L2 prefetch two chunks ahead.  The reverse role's dO
// rows come with MMA2's region as two TMA boxes (64 tokens x 64 channels)
// in the 128-byte swizzled layout, which MMA2 reads as they land.
//
// With few (sequence, head) chains the same kernel runs context-parallel
// (see scan_tc_cp_launch below): chains over segments of a sequence, a third
// role that forms a segment's transfer product from the identity, and a
// combine kernel that chains the segment boundaries between the two passes.
#include "kda_chunk.cuh"
#include "kda_tc_tiles.cuh"

namespace kda {
namespace stc {

using namespace tct;
constexpr int D = 128;
constexpr uint32_t kInFwd = (uint32_t)kPrepQE;                 // gT, W^T, kr, U0^T
constexpr uint32_t kInRevA = (uint32_t)kPrepU0;                // gT, W^T, kr
constexpr uint32_t kQEHere = (uint32_t)kPrepU0;                // QE^T lands where U0^T would
struct Smem {
  static constexpr size_t o_X = 0;                 // state [c][v] packed, 32 KB
  static constexpr size_t o_dO = o_X + 32768;      // dO [i][v], two 128-byte swizzled boxes
  static constexpr size_t o_U = o_dO + 16384;      // U^T [v][i] packed
  static constexpr size_t o_IN = o_U + 16384;      // operand block, 48.5 KB
  static constexpr size_t o_bar = o_IN + kInFwd;
  static constexpr size_t total = o_bar + 64;
  static_assert(total + 1024 <= 233472 / 2, "two CTAs per SM");
  static_assert(o_IN % 16 == 0, "bulk copy alignment");
  static_assert(o_dO % 1024 == 0, "the swizzled boxes' atoms are 1024-byte aligned");
};
constexpr uint32_t kDOBox = 8192;  // one 64 x 64 swizzled dO box

}  // namespace stc

__global__ void __launch_bounds__(NTHREADS, 2)
    kda_scan_tc_kernel(KdaParams p, const __grid_constant__ TokenMaps tm, const char *prep) {
  using namespace stc;
  using SM = stc::Smem;
  extern __shared__ __align__(1024) char smem[];
  pdl_wait();  // the prep kernels' operand blocks
  // the swizzled dO boxes need 1024-byte aligned atoms; the dynamic window of
  // a kernel without static shared memory is, and a launch where it were not
  // records KDA_ERR_CUDA and does nothing rather than issue a misaligned copy
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) set_status(4);
    return;
  }
  const int H = p.H;
  const int nseq = p.cu ? p.num_seqs : p.B;
  const int tid = threadIdx.x, warp = tid >> 5;
  const size_t DD = (size_t)D * D;
  int r, h, role;
  int g = -1;  // context-parallel segment (-1: the whole sequence)
  if (p.cp_segs >= 3) {
    // context-parallel chain kinds, kind-major then (sequence, head):
    //  phase 1: reverse-local g = 1..P-1, forward-local g = 0..P-2 (zero
    //           start, or dh_T / h0 for the outermost), transfers g = 1..P-2;
    //  phase 3: reverse g = 0..P-2, forward g = 1..P-1 from the combined
    //           boundaries.
    const int P = p.cp_segs;
    const bool has_rev = p.role_base + p.cp_nroles > 1, has_fwd = p.role_base == 0;
    int kind = (int)(blockIdx.x / (unsigned)(nseq * H));
    const int rem = (int)(blockIdx.x % (unsigned)(nseq * H));
    r = rem / H;
    h = rem % H;
    role = -1;
    if (has_rev) {
      if (kind < P - 1) {
        role = 1;
        g = p.cp_phase == 1 ? kind + 1 : kind;
      }
      kind -= P - 1;
    }
    if (role < 0 && has_fwd) {
      if (kind >= 0 && kind < P - 1) {
        role = 0;
        g = p.cp_phase == 1 ? kind : kind + 1;
      }
      kind -= P - 1;
    }
    if (role < 0 && p.cp_phase == 1 && kind >= 0 && kind < P - 2) {
      role = 2;
      g = kind + 1;
    }
    if (role < 0) return;
  } else {
    // block b -> (sequence rank r, role, head) for varlen: the chains of the
    // longest sequences are dispatched first, so that short chains fill in
    // behind them instead of a long one starting last; fixed length (all
    // chains equally long): (role, sequence, head).  The reverse role (the
    // longer chain of work per chunk) goes first in both.
    const int nroles = (int)(gridDim.x / (unsigned)(nseq * H));
    int rl;
    if (p.seq_order != nullptr) {
      r = (int)(blockIdx.x / (unsigned)(nroles * H));
      const int rem = (int)(blockIdx.x % (unsigned)(nroles * H));
      rl = nroles - 1 - rem / H;
      h = rem % H;
    } else {
      rl = nroles - 1 - (int)(blockIdx.x / (unsigned)(nseq * H));
      const int rem = (int)(blockIdx.x % (unsigned)(nseq * H));
      r = rem / H;
      h = rem % H;
    }
    role = p.role_base + rl;
  }
  // role 0: forward states, 1: reverse dS scan, 2: forward transfer matrix
  // (the forward update with U0 = 0 from the identity: the product of the
  // segment's chunk transitions S -> e^gT S - kr^T W S)
  const bool fwd = role != 1;
  const int s = p.seq_order ? p.seq_order[r] : r;
  int64_t tok_seq, slot0;
  int L;
  if (!seq_bounds(p, s, tok_seq, L, slot0)) return;
  const int nck_seq = (L + CHUNK - 1) / CHUNK;
  // this chain's chunks [c0, c0 + nck), its start and end tiles (row-major
  // fp32 K x V, nullable) and whether it stores the chunk states
  int c0 = 0, nck = nck_seq;
  const float *init;
  float *fin;
  bool pub = true;
  {
    const size_t sh = ((size_t)s * H + h) * DD;
    const float *outer_in = role == 1 ? p.dhT : p.h0;
    float *outer_out = role == 1 ? p.dh0 : p.hT;
    init = outer_in ? outer_in + sh : nullptr;
    fin = outer_out ? outer_out + sh : nullptr;
    if (g >= 0) {
      const int P = p.cp_segs;
      c0 = (int)((int64_t)g * nck_seq / P);
      nck = (int)((int64_t)(g + 1) * nck_seq / P) - c0;
      float *tiles = p.cp_buf + ((size_t)s * H + h) * (size_t)kda_cp_tiles(P) * DD;
      if (p.cp_phase == 1) {
        if (role == 0) {  // local from h0 (g = 0, the true states) or zero
          if (g > 0) init = nullptr;
          pub = g == 0;
          fin = tiles + (size_t)g * DD;
        } else if (role == 1) {  // local from dh_T (g = P - 1) or zero
          if (g < P - 1) init = nullptr;
          pub = g == P - 1;
          fin = tiles + (size_t)(P - 1 + g - 1) * DD;
        } else {
          init = nullptr;
          pub = false;
          fin = tiles + (size_t)(2 * (P - 1) + g - 1) * DD;
        }
      } else {
        if (role == 0) {
          init = tiles + (size_t)(g - 1) * DD;
          if (g < P - 1) fin = nullptr;
        } else {
          init = tiles + (size_t)(P - 1 + g) * DD;
          if (g > 0) fin = nullptr;
        }
      }
    }
  }
  char *Xs = smem + SM::o_X, *IN = smem + SM::o_IN, *dOs = smem + SM::o_dO, *Us = smem + SM::o_U;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::o_bar);  // 3 operand slots + MMA
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 4);

  const int ch = tid & 127, hf = tid >> 7;  // TMEM lane; half of the columns
  // running state: row ch, columns [64 hf, 64 hf + 64)
  float X[64];
  {
    const float *src = init ? init + (size_t)ch * D + 64 * hf : nullptr;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float4 v = src ? *reinterpret_cast<const float4 *>(src + 4 * q)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      X[4 * q] = v.x;
      X[4 * q + 1] = v.y;
      X[4 * q + 2] = v.z;
      X[4 * q + 3] = v.w;
    }
    if (role == 2) {  // the identity
#pragma unroll
      for (int q = 0; q < 64; ++q) X[q] = 64 * hf + q == ch ? 1.f : 0.f;
    }
  }
  if (warp == 0) umma::tmem_alloc(tslot, 256);
  if (tid == 0) {
    for (int k = 0; k < 4; ++k) umma::mbar_init(bars + k, 1);
  }
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  __syncthreads();

  auto chunk_of = [&](int it) { return fwd ? c0 + it : c0 + nck - 1 - it; };
  auto unit_of = [&](int j) {
    return prep + ((size_t)(slot0 + j) * H + h) * kPrepUnitBytes;
  };
  const bf16 *dOg = reinterpret_cast<const bf16 *>(p.dO);
  // Operand regions of IN and the barrier each one completes on:
  //   forward: slot 0 = gT | W^T (MMA1), slot 1 = U0^T (epilogue 1), slot 2 = kr^T (MMA2)
  //   reverse: slot 0 = kr^T (MMA1), slot 1 = gT | W^T, QE^T (+ dO rows) (MMA2)
  // A slot is refilled with the next chunk's data as soon as its consumer is done.
  // Slot sl's copies are issued by thread 32 (sl + 1) (warps 1-3), publishing
  // and prefetching by threads 160 and 192: thread 0 only issues the MMAs.
  // (a timeout test arms the first chunk's barriers but issues no copies)
  const bool starve = (p.starve & kStarveScan) != 0u;
  auto load_slot = [&](int sl, int it) {
    const char *u = unit_of(chunk_of(it));
    if (starve && it == 0) {
      if (tid == 32 * (sl + 1)) umma::mbar_expect_tx(bars + sl, 16u);
      return;
    }
    if (tid == 32 * (sl + 1)) {
      if (fwd) {
        if (sl == 0) {
          umma::mbar_expect_tx(bars + 0, kPrepKR);
          umma::bulk_g2s(IN, u, kPrepKR, bars + 0);
        } else if (sl == 1) {
          umma::mbar_expect_tx(bars + 1, 16384u);
          umma::bulk_g2s(IN + kPrepU0, u + kPrepU0, 16384u, bars + 1);
        } else {
          umma::mbar_expect_tx(bars + 2, 16384u);
          umma::bulk_g2s(IN + kPrepKR, u + kPrepKR, 16384u, bars + 2);
        }
      } else {
        if (sl == 0) {
          umma::mbar_expect_tx(bars + 0, 16384u);
          umma::bulk_g2s(IN + kPrepKR, u + kPrepKR, 16384u, bars + 0);
        } else {
          // gT | W^T, QE^T, and the chunk's dO rows as two swizzled boxes
          // (channels 0-63, 64-127); rows past the tensor's end read as zero
          const int t0 = (int)(tok_seq + (int64_t)chunk_of(it) * CHUNK);
          umma::mbar_expect_tx(bars + 1, kPrepKR + 16384u + 2 * kDOBox);
          umma::bulk_g2s(IN, u, kPrepKR, bars + 1);
          umma::bulk_g2s(IN + kQEHere, u + kPrepQE, 16384u, bars + 1);
          umma::tma_load_3d(dOs, &tm.dO_sw, 0, h, t0, bars + 1);
          umma::tma_load_3d(dOs + kDOBox, &tm.dO_sw, 64, h, t0, bars + 1);
        }
      }
    }
  };
  auto prefetch = [&](int it) {
    const int j = chunk_of(it);
    const char *u = unit_of(j);
    if (tid == 192) {
      if (fwd) {
        umma::bulk_prefetch_l2(u, kInFwd);
      } else {
        umma::bulk_prefetch_l2(u, kInRevA);
        umma::bulk_prefetch_l2(u + kPrepQE, 16384u);
      }
    }
    if (!fwd && tid >= 128) {  // dO rows: two 128-byte lines each, plain L2 prefetches
      const int i = (tid - 128) >> 1;
      const int64_t t0 = tok_seq + (int64_t)j * CHUNK;
      if (i < L - j * CHUNK) {
        const bf16 *row = dOg + ((t0 + i) * H + h) * D + 64 * (tid & 1);
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(row));
      }
    }
  };
  bf16 *states_out = reinterpret_cast<bf16 *>(fwd ? p.states : p.dstates);
  // bf16 running state -> MMA1's operand tile
  auto to_tile = [&]() {
#pragma unroll
    for (int q = 0; q < 8; ++q) st16_bf(Xs + umma::core_off(ch, 64 * hf + 8 * q, D), X + 8 * q);
  };
  // the bf16 tile (the state chunk j starts from) -> the chunk's slot in HBM,
  // one bulk copy by thread 160 once the tile is complete and fenced
  auto publish = [&](int j) {
    if (pub && tid == 160) {
      umma::bulk_s2g(states_out + ((size_t)(slot0 + j) * H + h) * DD, Xs, (uint32_t)(DD * 2));
      umma::bulk_commit();
    }
  };
  const int nslots_in = fwd ? 3 : 2;
  if (nck > 0) {
    for (int sl = 0; sl < nslots_in; ++sl) load_slot(sl, 0);
    if (nck > 1) prefetch(1);
    to_tile();
  }
  umma::fence_async_smem();
  umma::tc_fence_before();
  __syncthreads();
  umma::tc_fence_after();
  if (nck > 0) publish(chunk_of(0));
  const uint32_t tbase = *tslot;
  uint32_t ph[4] = {0u, 0u, 0u, 0u};  // phase of each barrier (bars[3] = MMA completion)
  auto wait_bar = [&](int k) {
    const bool ok = umma::mbar_wait(bars + k, ph[k] & 1,
                                    poll_cap(p, k == 3 ? umma::kPollMma : umma::kPollLoads));
    ph[k]++;
    return ok;
  };
  bool bad = false;
  const uint32_t tl = tbase + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's TMEM lanes
  float eg = 1.f;

  for (int it = 0; it < nck; ++it) {
    const bool more = it + 1 < nck;
    if (it + 2 < nck) prefetch(it + 2);
    bool ok = true;
    // ---- MMA1: T1 = (B1 X)^T into columns [0, 64) ----
    if (fwd) {
      ok = wait_bar(0);  // gT | W^T (every thread reads gT)
      eg = __expf(reinterpret_cast<const float *>(IN + kPrepGT)[ch]);
    } else if (tid == 0) {
      ok = wait_bar(0);  // kr^T
    }
    if (__syncthreads_or(!ok)) {
      bad = true;
      break;
    }
    if (tid == 0) {
      umma::tc_fence_after();
      const Op a = opmn(Xs, D, 0, CP);
      const Op b1 = opmn(IN + (fwd ? kPrepW : kPrepKR), 64, 0, CP);  // W^T / kr^T, [c][i]
      gemm(tbase, a, true, b1, true, 64, D / 16, false);
      umma::mma_commit(bars + 3);
    }
    ok = wait_bar(3);
    umma::tc_fence_after();
    if (more) load_slot(0, it + 1);  // MMA1's operand is consumed
    // ---- U^T[v][i] for lane v = ch, i in [32 hf, 32 hf + 32) ----
    {
      float t[32];
      tld32(tbase, 0, t);
      if (fwd) {
        ok = wait_bar(1) && ok;  // U0^T
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float u0[8];
          ld16_bf(IN + kPrepU0 + umma::core_off(ch, 32 * hf + 8 * q, 64), u0);
          const float keep = role == 0 ? 1.f : 0.f;  // the transfer drops U0
#pragma unroll
          for (int n = 0; n < 8; ++n) t[8 * q + n] = fmaf(keep, u0[n], -t[8 * q + n]);
        }
      } else {
#pragma unroll
        for (int n = 0; n < 32; ++n) t[n] = -t[n];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) st16_bf(Us + umma::core_off(ch, 32 * hf + 8 * q, 64), t + 8 * q);
    }
    if (!fwd) {
      ok = wait_bar(1) && ok;  // gT | W^T, QE^T, dO
      eg = __expf(reinterpret_cast<const float *>(IN + kPrepGT)[ch]);
      // a sequence's partial last chunk: the boxes' rows past it hold the next
      // sequence's dO; zero them (a row's 128 bytes stay within the row)
      const int ln = L - chunk_of(it) * CHUNK;
      if (ln < CHUNK) {
        for (int e = tid; e < 2 * 64 * 8; e += NTHREADS) {
          const int row = (e >> 3) & 63;
          if (row >= ln)
            *reinterpret_cast<uint4 *>(dOs + (e >> 9) * kDOBox + row * 128 + (e & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    umma::fence_async_smem();
    umma::tc_fence_before();
    if (__syncthreads_or(!ok)) {
      bad = true;
      break;
    }
    if (fwd && more) load_slot(1, it + 1);  // U0^T is consumed
    // ---- MMA2: T2 into columns [64, 192) ----
    if (tid == 0) {
      bool ok2 = true;
      if (fwd) ok2 = wait_bar(2);  // kr^T
      umma::tc_fence_after();
      const Op b = opk(Us, 64, 0, CP);
      if (ok2) {
        if (fwd) {
          gemm(tbase + 64, opk(IN + kPrepKR, 64, 0, CP), false, b, false, 128, 4, false);
        } else {
          gemm(tbase + 64, opk(IN + kPrepW, 64, 0, CP), false, b, false, 128, 4, false);
          // + QE^T dO: dO read MN-major from the swizzled boxes (N = 128 as
          // two 64-wide slabs kDOBox apart, K = 16 tokens = two 8-row atoms)
          gemm(tbase + 64, opk(IN + kQEHere, 64, 0, CP), false, opsw_mn(dOs, kDOBox), true, 128,
               4, true);
        }
      }
      umma::mma_commit(bars + 3);
      ok = ok2;
    }
    ok = wait_bar(3) && ok;
    umma::tc_fence_after();
    if (tid == 160) umma::bulk_wait_read();  // the tile's previous store has read it
    if (__syncthreads_or(!ok)) {
      bad = true;
      break;
    }
    // MMA2's operands are consumed: refill for the next chunk
    if (more) load_slot(fwd ? 2 : 1, it + 1);
    // ---- state update: X = e^gT X + T2 ----
#pragma unroll
    for (int q = 0; q < 4; q += 2) {
      float t0[16], t1[16];
      umma::tmem_ld16(tl + 64 + 64 * hf + 16 * q, t0);
      umma::tmem_ld16(tl + 64 + 64 * hf + 16 * (q + 1), t1);
      umma::tmem_ld_wait();
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        X[16 * q + n] = fmaf(eg, X[16 * q + n], t0[n]);
        X[16 * (q + 1) + n] = fmaf(eg, X[16 * (q + 1) + n], t1[n]);
      }
    }
    if (more) to_tile();
    umma::fence_async_smem();
    umma::tc_fence_before();
    __syncthreads();
    if (more) publish(chunk_of(it + 1));
  }
  if (bad) {
    // a bounded wait gave up (status already flagged): let copies and MMAs in
    // flight land before the buffers and Tensor Memory are released
    if (tid == 0) {
      for (int k = 0; k < 4; ++k) umma::mbar_wait(bars + k, ph[k] & 1, poll_cap(p, umma::kPollDrain));
    }
    cp_async_wait_all();
    __syncthreads();
  } else {
    if (fin != nullptr) {
      float *dst = fin + (size_t)ch * D + 64 * hf;
#pragma unroll
      for (int q = 0; q < 16; ++q)
        *reinterpret_cast<float4 *>(dst + 4 * q) =
            make_float4(X[4 * q], X[4 * q + 1], X[4 * q + 2], X[4 * q + 3]);
    }
  }
  if (tid == 160) umma::bulk_wait_read();  // (the global writes complete before the grid does)
  umma::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    umma::tc_fence_after();
    umma::tmem_dealloc(tbase, 256);
  }
}

cudaError_t scan_tc_launch(const KdaParams &p, const TokenMaps &tm, const void *prep, int nroles,
                           cudaStream_t st) {
  auto kfn = kda_scan_tc_kernel;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)stc::Smem::total);
  if (e != cudaSuccess) return e;
  const int64_t nunits = (int64_t)(p.cu ? p.num_seqs : p.B) * p.H;
  if (nunits == 0 || nroles == 0) return cudaSuccess;
  if (nroles < 1 || p.role_base + nroles > 2) return cudaErrorInvalidValue;
  return pdl_launch(kfn, dim3((unsigned)(nunits * nroles)), dim3(NTHREADS), stc::Smem::total, st,
                    p, tm, static_cast<const char *>(prep));
}

// ---------------------------------------------------------------------------
// Context-parallel scans.  With A_n = e^gT - kr^T W the forward update is
// S_{n+1} = A_n S_n + kr^T U0 and the reverse one dS_n = A_n^T dS_{n+1} +
// QE^T dO, so over a segment of chunks [a, b), with P_g = A_{b-1} ... A_a,
//   S_b  = P_g S_a + E_g       (E_g: the segment's forward scan from zero)
//   dS_a = P_g^T dS_b + F_g    (F_g: its reverse scan from zero)
// Phase 1 scans every segment from zero (the first forward and the last
// reverse segment from h0 / dh_T, which makes their states final) and the
// inner segments' P_g from the identity; the combine kernel below chains the
// boundaries; phase 3 rescans the remaining segments from them.  Tiles per
// (sequence, head), fp32 row-major K x V:
//   [0, P-1)        forward start of segment g + 1 (E_g, combined in place)
//   [P-1, 2P-2)     reverse end of segment g (F_{g+1}, combined in place)
//   [2P-2, 3P-4)    P_g of the inner segments g = 1 .. P-2
// ---------------------------------------------------------------------------
namespace stc {
constexpr int kCombCols = 32;  // V columns per combine CTA
constexpr int kSinLd = 40;     // row stride (floats) of the staged columns: B fragments conflict-free
}  // namespace stc

// One CTA per (sequence, head) x 32-column block of V x direction (0 forward,
// 1 reverse); the columns of a state evolve independently.  P - 2 dependent
// steps, each a 128 x 128 by 128 x 32 product on the tensor cores (mma.sync
// m16n8k8 tf32, fp32 accumulation; tf32 rounds to 2^-11, finer than the
// bf16 of the published states) plus the local tile:
//   forward  start(g) = P_{g-1} start(g-1) + E_{g-1},        g = 2 .. P-1
//   reverse  end(g)   = P_{g+1}^T end(g+1) + F_{g+1},        g = P-3 .. 0
// Warp w owns rows [16 w, 16 w + 16) and all 32 columns (four n-tiles).  The
// transfer products do not depend on the chain: each thread's A fragments of
// the next step (64 floats, read straight from L2) are loaded while the
// current step multiplies.
__global__ void __launch_bounds__(NTHREADS) kda_cp_combine_kernel(KdaParams p) {
  using namespace stc;
  __shared__ __align__(16) float Sin[D * kSinLd];
  pdl_wait();  // the first pass's segment boundaries and transfer matrices
  const int P = p.cp_segs;
  const int dir = p.role_base + (int)blockIdx.z;
  const int j0 = (int)blockIdx.y * kCombCols;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3, r0 = 16 * w + gq;
  const size_t DD = (size_t)D * D;
  float *tiles = p.cp_buf + (size_t)blockIdx.x * (size_t)kda_cp_tiles(P) * DD;
  // tile indices of step st: input boundary, output boundary, transfer
  auto t_in = [&](int st) { return dir == 0 ? st : 2 * P - 3 - st; };
  auto t_out = [&](int st) { return dir == 0 ? st + 1 : 2 * P - 4 - st; };
  auto t_p = [&](int st) { return dir == 0 ? 2 * P - 2 + st : 3 * P - 5 - st; };
  // A = P_g (forward) or P_g^T (reverse); fragment q of k-step ks holds
  // A[r0 + 8 (q & 1)][8 ks + tq + 4 (q >> 1)]
  float pa[D / 8][4];
  auto load_a = [&](int st) {
    const float *Pg = tiles + (size_t)t_p(st) * DD;
#pragma unroll
    for (int ks = 0; ks < D / 8; ++ks) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = r0 + 8 * (q & 1), k = 8 * ks + tq + 4 * (q >> 1);
        pa[ks][q] = dir == 0 ? Pg[r * D + k] : Pg[k * D + r];
      }
    }
  };
  if (P >= 3) load_a(0);
  {  // the first input: the outermost boundary tile's columns [j0, j0 + 32)
    const float *src = tiles + (size_t)t_in(0) * DD;
    float4 v[D * kCombCols / 4 / NTHREADS];
#pragma unroll
    for (int i = 0; i < D * kCombCols / 4 / NTHREADS; ++i) {
      const int e = tid + i * NTHREADS;
      v[i] = *reinterpret_cast<const float4 *>(src + (size_t)(e >> 3) * D + j0 + 4 * (e & 7));
    }
#pragma unroll
    for (int i = 0; i < D * kCombCols / 4 / NTHREADS; ++i) {
      const int e = tid + i * NTHREADS;
      *reinterpret_cast<float4 *>(Sin + (e >> 3) * kSinLd + 4 * (e & 7)) = v[i];
    }
  }
  __syncthreads();
  for (int st = 0; st < P - 2; ++st) {
    uint32_t af[D / 8][4];
#pragma unroll
    for (int ks = 0; ks < D / 8; ++ks)
#pragma unroll
      for (int q = 0; q < 4; ++q) af[ks][q] = to_tf32(pa[ks][q]);
    if (st + 1 < P - 2) load_a(st + 1);
    float *out = tiles + (size_t)t_out(st) * DD;
    float acc[4][4];  // [n-tile][fragment]: the local tile plus the product
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float2 lo = *reinterpret_cast<const float2 *>(out + (size_t)r0 * D + j0 + 8 * nt + 2 * tq);
      const float2 hi =
          *reinterpret_cast<const float2 *>(out + (size_t)(r0 + 8) * D + j0 + 8 * nt + 2 * tq);
      acc[nt][0] = lo.x;
      acc[nt][1] = lo.y;
      acc[nt][2] = hi.x;
      acc[nt][3] = hi.y;
    }
#pragma unroll
    for (int ks = 0; ks < D / 8; ++ks) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float *b = Sin + (8 * ks + tq) * kSinLd + 8 * nt + gq;
        const uint32_t bf[2] = {to_tf32(b[0]), to_tf32(b[4 * kSinLd])};
        mma_tf32(acc[nt], af[ks], bf);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      *reinterpret_cast<float2 *>(out + (size_t)r0 * D + j0 + 8 * nt + 2 * tq) =
          make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2 *>(out + (size_t)(r0 + 8) * D + j0 + 8 * nt + 2 * tq) =
          make_float2(acc[nt][2], acc[nt][3]);
    }
    __syncthreads();  // every warp is done reading Sin
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      *reinterpret_cast<float2 *>(Sin + r0 * kSinLd + 8 * nt + 2 * tq) =
          make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2 *>(Sin + (r0 + 8) * kSinLd + 8 * nt + 2 * tq) =
          make_float2(acc[nt][2], acc[nt][3]);
    }
    __syncthreads();
  }
}

cudaError_t scan_tc_cp_launch(KdaParams p, const TokenMaps &tm, const void *prep, int nroles,
                              cudaStream_t st) {
  const int P = p.cp_segs;
  if (P < 3 || p.cp_buf == nullptr) return cudaErrorInvalidValue;
  if (nroles < 1 || p.role_base < 0 || p.role_base + nroles > 2) return cudaErrorInvalidValue;
  auto kfn = kda_scan_tc_kernel;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)stc::Smem::total);
  if (e != cudaSuccess) return e;
  const int64_t nunits = (int64_t)(p.cu ? p.num_seqs : p.B) * p.H;
  if (nunits == 0) return cudaSuccess;
  const bool has_fwd = p.role_base == 0, has_rev = p.role_base + nroles > 1;
  const int roles = (has_fwd ? 1 : 0) + (has_rev ? 1 : 0);
  p.cp_nroles = nroles;
  p.seq_order = nullptr;
  // 1. local segment scans and the inner transfer matrices
  p.cp_phase = 1;
  e = pdl_launch(kfn, dim3((unsigned)(nunits * (roles * (P - 1) + (P - 2)))), dim3(NTHREADS),
                 stc::Smem::total, st, p, tm, static_cast<const char *>(prep));
  if (e != cudaSuccess) return e;
  // 2. the segment boundaries
  p.cp_phase = 2;
  e = pdl_launch(kda_cp_combine_kernel, dim3((unsigned)nunits, stc::D / stc::kCombCols, (unsigned)roles),
                 dim3(NTHREADS), 0, st, p);
  if (e != cudaSuccess) return e;
  // 3. the remaining segments from their true boundaries
  p.cp_phase = 3;
  return pdl_launch(kfn, dim3((unsigned)(nunits * roles * (P - 1))), dim3(NTHREADS),
                    stc::Smem::total, st, p, tm, static_cast<const char *>(prep));
}

// rank of sequence s = the number of sequences longer than s, or as long and
// before it; every thread ranks one sequence against all (num_seqs reads)
__global__ void kda_seq_order_kernel(const int32_t *cu, int n, int32_t *order) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= n) return;
  const int Ls = cu[s + 1] - cu[s];
  int r = 0;
  for (int t = 0; t < n; ++t) {
    const int Lt = cu[t + 1] - cu[t];
    r += (Lt > Ls || (Lt == Ls && t < s)) ? 1 : 0;
  }
  order[r] = s;
}

cudaError_t seq_order_launch(const int32_t *cu, int num_seqs, int32_t *order, cudaStream_t st) {
  if (num_seqs <= 0) return cudaSuccess;
  kda_seq_order_kernel<<<(num_seqs + 255) / 256, 256, 0, st>>>(cu, num_seqs, order);
  return cudaGetLastError();
}

int scan_tc_status_take() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_status, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

}  // namespace kda
