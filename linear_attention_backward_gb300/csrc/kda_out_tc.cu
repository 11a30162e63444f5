// kda_out_tc.cu -- chunk outputs of the KDA forward on the fifth-generation
// tensor cores (bf16, K = V = 128), from the prep kernel's per-chunk operands
// and the forward scan's chunk states.
//
// With the WY form of the chunk (the same algebra as the scans: U = U0 - W S_n
// the corrected values, Mqk = scale * lower(qd ki^T) with the diagonal), the
// read-out o_i = scale * S_i^T q^_i of every row of chunk n is
//   o = scale * qd S_n + Mqk U = (scale * qd - Mqk W) S_n + Mqk U0
//     = QE S_n + Mqk U0,
// two products per chunk whose operands the prep block already holds (QE^T,
// U0^T, Mqk) next to the state S_n the scan stored.  Taken transposed, with
// the V channel as the MMA's M:
//   o^T[v][i] = sum_c S_n[c][v] QE[i][c]  +  sum_j U0^T[v][j] Mqk[i][j]
//               (N = 64, K = 128)            (N = 64, K = 64)
// One CTA of 128 threads per (chunk slot, head), three per SM; thread v reads
// TMEM lane v and writes column v of the chunk's rows, which leave as 16-byte
// row pieces.
#include "kda_chunk.cuh"
#include "kda_tc_tiles.cuh"

namespace kda {
namespace otc {

using namespace tct;
constexpr int D = 128;
constexpr int NT = 128;
struct Smem {
  static constexpr size_t o_S = 0;                 // S_n [c][v] packed, 32 KB
  static constexpr size_t o_B = o_S + 32768;       // U0^T | QE^T | Mqk, as in the prep block
  static constexpr size_t nB = kPrepINV - kPrepU0;  // 40 KB
  static constexpr size_t o_U0 = o_B;
  static constexpr size_t o_QE = o_B + (kPrepQE - kPrepU0);
  static constexpr size_t o_Mqk = o_B + (kPrepMqk - kPrepU0);
  static constexpr size_t o_O = o_S;               // the chunk's o rows [i][v], after the MMAs
  static constexpr size_t o_bar = o_B + nB;
  static constexpr size_t total = o_bar + 64;
  static_assert(kPrepQE == kPrepU0 + 16384 && kPrepMqk == kPrepQE + 16384 &&
                    kPrepINV == kPrepMqk + 8192,
                "U0^T, QE^T and Mqk are copied as one block");
  static_assert(3 * (total + 1024) <= 233472, "three CTAs per SM");
};

}  // namespace otc

__global__ void __launch_bounds__(otc::NT) kda_out_tc_kernel(KdaParams p, const void *states,
                                                            void *out) {
  using namespace otc;
  using SM = otc::Smem;
  extern __shared__ __align__(1024) char smem[];
  pdl_wait();  // the scan's chunk states
  const int64_t slot = blockIdx.x;
  const int h = blockIdx.y;
  const int H = p.H;
  const int tid = threadIdx.x, warp = tid >> 5;
  int s_, j_, len;
  int64_t tok0;
  if (!slot_owner(p, slot, s_, j_, tok0, len)) return;  // padding slot
  char *St = smem + SM::o_S;
  char *U0t = smem + SM::o_U0, *QEt = smem + SM::o_QE, *Mqk = smem + SM::o_Mqk;
  bf16 *Os = reinterpret_cast<bf16 *>(smem + SM::o_O);
  uint64_t *lbar = reinterpret_cast<uint64_t *>(smem + SM::o_bar);
  uint64_t *mbar = lbar + 1;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(lbar + 2);
  const size_t unit = (size_t)slot * H + h;

  if (warp == 0) umma::tmem_alloc(tslot, 64);
  if (tid == 0) {
    umma::mbar_init(lbar, 1);
    umma::mbar_init(mbar, 1);
  }
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  __syncthreads();
  umma::tc_fence_after();
  const uint32_t tbase = *tslot;
  // Bounded waits: thread 0 waits for the copies and issues the products only
  // if they landed; the CTA learns the outcome at a barrier, and after a wait
  // that gave up it writes nothing, drains what is in flight and releases
  // Tensor Memory.
  bool ok = true;
  if (tid == 0) {
    umma::mbar_expect_tx(lbar, 32768u + (uint32_t)SM::nB);
    if ((p.starve & kStarveOut) == 0u) {  // (a timeout test arms the barrier only)
      umma::bulk_g2s(St, static_cast<const char *>(states) + unit * 32768, 32768u, lbar);
      umma::bulk_g2s(U0t, p.prep + unit * kPrepUnitBytes + kPrepU0, (uint32_t)SM::nB, lbar);
    }
    ok = umma::mbar_wait(lbar, 0, poll_cap(p, umma::kPollLoads));
    umma::tc_fence_after();
    if (ok) {
      // o^T = S_n^T QE^T  (A = S read MN-major, B = QE^T [c][i] read MN-major)
      gemm(tbase, opmn(St, D, 0, CP), true, opmn(QEt, 64, 0, CP), true, 64, D / 16, false);
      //     + U0^T Mqk^T  (A = U0^T [v][j], B = Mqk [i][j], both read with K = j)
      gemm(tbase, opk(U0t, 64, 0, CP), false, opk(Mqk, 64, 0, CP), false, 64, 4, true);
      umma::mma_commit(mbar);
    }
  }
  const bool loaded = !__syncthreads_or(!ok);
  if (loaded) ok = umma::mbar_wait(mbar, 0, poll_cap(p, umma::kPollMma));
  umma::tc_fence_after();
  // thread v = tid: TMEM lane v holds o^T[v][0..63]; rows land in Os [i][v]
  // (S's region: the products are complete)
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float a[16];
    umma::tmem_ld16(tbase + ((uint32_t)(32 * warp) << 16) + (uint32_t)(16 * q), a);
    umma::tmem_ld_wait();
#pragma unroll
    for (int r = 0; r < 16; ++r) Os[(16 * q + r) * D + tid] = __float2bfloat16_rn(a[r]);
  }
  umma::tc_fence_before();
  if (__syncthreads_or(!ok)) {
    // a bounded wait gave up (the status word says so): the copies or the
    // products may still be in flight; give them a last bounded wait
    if (tid == 0) {
      const uint32_t lim = poll_cap(p, umma::kPollDrain);
      if (!loaded) umma::mbar_wait(lbar, 0, lim);
      else umma::mbar_wait(mbar, 0, lim);
    }
    __syncthreads();
  } else {
    bf16 *og = static_cast<bf16 *>(out);
#pragma unroll 1
    for (int e = tid; e < 64 * (D / 8); e += NT) {
      const int i = e >> 4, c8 = (e & 15) * 8;
      if (i < len)
        *reinterpret_cast<uint4 *>(og + ((tok0 + i) * H + h) * D + c8) =
            *reinterpret_cast<const uint4 *>(Os + i * D + c8);
    }
  }
  if (warp == 0) {
    umma::tc_fence_after();
    umma::tmem_dealloc(tbase, 64);
  }
}

cudaError_t out_tc_launch(const KdaParams &p, const void *states, void *o, cudaStream_t st) {
  auto kfn = kda_out_tc_kernel;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)otc::Smem::total);
  if (e != cudaSuccess) return e;
  if (p.nslots > 0 && p.H > 0) {
    e = pdl_launch(kfn, dim3((unsigned)p.nslots, p.H), dim3(otc::NT), otc::Smem::total, st, p,
                   states, o);
  }
  return e;
}

int out_tc_status_take() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_status, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

}  // namespace kda
