// kda_range.cu -- exact chunk arithmetic for gates beyond the range of the
// 16-row block factors (bf16, K = V = 128, the tcgen05 path).
//
// The tensor-core kernels form every intra-chunk product between rows i and
// j <= i through factors referenced to a row of each 16-row block
// (kda_chunk.cuh).  Those factors are finite in fp32 only while a channel's
// gate log-decay between a row and its block's reference row stays below 88
// nats.  Past that (more than 11 nats per token, sustained over half a block,
// e.g. e^A_log = 8 with softplus(g + dt_bias) above 1.4) they overflow,
// although every product they stand for is at most 1 in magnitude.  The prep
// kernel marks such a (chunk, head) in a flag array, and also a chunk in
// which every channel decays by more than 6 nats per token (kda_device.cuh:
// there the block-factored products leave dg, which is then tiny, less
// accurate than bf16 allows).  The two kernels here redo a marked chunk's
// arithmetic in plain fp32 with one exponential per (row pair, channel),
// e_ij = e^(gc_i - gc_j) <= 1 for j <= i, which cannot overflow:
//
//   kda_range_prep_kernel   after the prep kernel, before the scans: the
//       scans' operands gT, W^T, kr^T, U0^T and, for the read-out, QE^T and
//       scale * Mqk, over the prep kernel's (non-finite) ones;
//   kda_range_grads_kernel  after the gradient kernel: the chunk's dq, dk, dv,
//       dg and dbeta rows and its dA_log / ddt_bias partials, from the chunk
//       states S_n and dS_{n+1} that the scans stored (then exact too).
//
// Per chunk (rows i, j < 64; rows past a sequence's end have q = k = 0,
// beta = 0 and no decay; s the read-out scale), the chunked form of the
// recurrence ("bwd-kernelB-beginner-guide-full", Part 1, the B1 / B2 / B0 / B3
// terms) written without block factors:
//   G_ij  = sum_c k^_i k^_j e_ij  (j < i),    Mq_ij = sum_c q^_i k^_j e_ij  (j <= i)
//   T     = (I + diag(beta) G)^-1
//   X     = v - kd S_n,   U = T diag(beta) X          (kd = k^ e^gc, qd = q^ e^gc)
//   o     = s (qd S_n + Mq U),    S_{n+1} = e^gT S_n + kr^T U    (kr = k^ e^(gT - gc))
// and its reverse mode:
//   dU    = s Mq^T dO + kr dS_{n+1},   dY = T^T dU,   dv = diag(beta) dY
//   dA    = -strict_lower(dY U^T),     dG = diag(beta) dA,   dMq = s lower(dO U^T)
//   dbeta = rowsum(dY o X) + rowsum(dA o G)
//   dqd   = s dO S_n^T,   dkd = -diag(beta) dY S_n^T,   dkr = U dS_{n+1}^T
// then per (i, c) the pair matrices' terms (sums over j with e_ij), the L2-norm
// backward, and the gate epilogue: the reverse cumulative sum of the
// log-decay gradient over the chunk plus dgT, dg, and the dA_log and ddt_bias
// partials, with the gradient kernel's conventions.
//
// Each kernel launches one CTA per SM, which walks its contiguous share of
// the flag array: a chunk that is not flagged costs one flag read.
#include "kda_chunk.cuh"
#include "kda_tc_tiles.cuh"

namespace kda {
namespace rng {

using namespace tct;

constexpr int D = 128;
constexpr int NT = 512;
constexpr int RS = D + 1;          // row stride of the [64][128] fp32 tiles
constexpr int PS = CHUNK + 1;      // row stride of the [64][64] fp32 tiles
constexpr int kRow = CHUNK * RS;   // floats of a [64][128] tile
constexpr int kPair = CHUNK * PS;  // floats of a [64][64] tile
constexpr int RB = CHUNK * D / NT;      // rows per thread, (channel, row block) mappings
constexpr int CG = CHUNK * D / NT;      // columns per thread, (row, column group) mappings
constexpr int PB = CHUNK * CHUNK / NT;  // rows per thread, (pair column, row block) mapping
static_assert(NT == 8 * CHUNK && RB % 8 == 0 && CG % 8 == 0, "the mappings below");

// Shared-memory views common to both kernels.
struct Basics {
  float *qh, *kh, *gc;         // [64][RS]: q^, k^ and the running log-decay gc
  float *G, *Mq, *T;           // [64][PS]
  float *beta, *rq, *rk, *gT;  // [64], [64], [64], [128]
};
constexpr int kBasicFloats = 3 * kRow + 3 * kPair + 3 * CHUNK + D;

__device__ __forceinline__ Basics basics_view(float *s) {
  Basics b;
  b.qh = s;
  b.kh = s + kRow;
  b.gc = s + 2 * kRow;
  b.G = s + 3 * kRow;
  b.Mq = b.G + kPair;
  b.T = b.Mq + kPair;
  b.beta = b.T + kPair;
  b.rq = b.beta + CHUNK;
  b.rk = b.rq + CHUNK;
  b.gT = b.rk + CHUNK;
  return b;
}

// Calls f(u) for every flagged unit u = slot * H + h of this CTA's contiguous
// share of the flag array, taken NT flags at a time.  Every thread calls f
// the same number of times.  The order within a piece follows the shared
// atomic and may vary; each unit's results depend on that unit alone.
template <typename F>
__device__ __forceinline__ void for_each_flagged(const int32_t *flags, int64_t nunits, int *list,
                                                 int *count, F &&f) {
  const int64_t per = (nunits + gridDim.x - 1) / gridDim.x;
  const int64_t u0 = (int64_t)blockIdx.x * per;
  const int64_t u1 = u0 + per < nunits ? u0 + per : nunits;
  for (int64_t base = u0; base < u1; base += NT) {
    if (threadIdx.x == 0) *count = 0;
    __syncthreads();
    const int64_t u = base + threadIdx.x;
    if (u < u1 && flags[u] != 0) list[atomicAdd(count, 1)] = (int)threadIdx.x;
    __syncthreads();
    const int n = *count;
    for (int k = 0; k < n; ++k) f(base + list[k]);
    __syncthreads();  // list and count are read by every thread above
  }
}

// The chunk's k, g (and with kQ q) rows into the fp32 tiles, zero past len;
// beta; the row norms (rows scaled in place); the gate's running sum over the
// chunk, gc and gT, with the prep kernel's gate arithmetic.  Ends with a
// barrier.
template <bool kQ>
__device__ void chunk_basics(const KdaParams &p, int h, int64_t tok0, int len, const Basics &b) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H;
  const bf16 *qg = static_cast<const bf16 *>(p.q), *kg = static_cast<const bf16 *>(p.k);
  const bf16 *gg = static_cast<const bf16 *>(p.g);
  for (int e = tid; e < CHUNK * (D / 8); e += NT) {
    const int i = e >> 4, c8 = (e & 15) * 8;
    float kv[8], gv[8], qv[8];
    if (i < len) {
      const int64_t off = ((tok0 + i) * H + h) * D + c8;
      ld16_bf(kg + off, kv);
      ld16_bf(gg + off, gv);
      if (kQ) ld16_bf(qg + off, qv);
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) kv[u] = gv[u] = qv[u] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      b.kh[i * RS + c8 + u] = kv[u];
      b.gc[i * RS + c8 + u] = gv[u];
      if (kQ) b.qh[i * RS + c8 + u] = qv[u];
    }
  }
  if (tid < CHUNK)
    b.beta[tid] = tid < len
                      ? __bfloat162float(static_cast<const bf16 *>(p.beta)[(tok0 + tid) * H + h])
                      : 0.f;
  __syncthreads();
  for (int i = warp; i < CHUNK; i += NT / 32) {  // row norms: a warp per row
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float x = b.kh[i * RS + lane + 32 * m];
      sk = fmaf(x, x, sk);
      if (kQ) {
        const float y = b.qh[i * RS + lane + 32 * m];
        sq = fmaf(y, y, sq);
      }
    }
    const float rk = rsqrtf(warp_sum(sk) + p.eps);
    const float rq = kQ ? rsqrtf(warp_sum(sq) + p.eps) : 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      b.kh[i * RS + lane + 32 * m] *= rk;
      if (kQ) b.qh[i * RS + lane + 32 * m] *= rq;
    }
    if (lane == 0) {
      b.rk[i] = rk;
      b.rq[i] = rq;
    }
  }
  if (tid < D) {  // channel tid: gk = -e^A_log softplus(g + dt_bias), summed down the chunk
    const float A = __expf(p.A_log[h]), bias = gate_bias(p, h, tid, D);
    float run = 0.f;
    for (int i = 0; i < CHUNK; ++i) {
      if (i < len) run += -A * softplus_gate(b.gc[i * RS + tid] + bias);
      b.gc[i * RS + tid] = run;
    }
    b.gT[tid] = run;
  }
  __syncthreads();
}

// G (strictly lower) and, with kQ, Mq (lower, diagonal included): one thread
// per pair (i, j <= i) of the 2080, the exponential shared by both; zero
// above the diagonal.  Ends with a barrier.
template <bool kQ>
__device__ void pair_matrices(const Basics &b) {
  for (int e = threadIdx.x; e < CHUNK * (CHUNK + 1) / 2; e += NT) {
    int i = (int)((sqrtf(8.f * (float)e + 1.f) - 1.f) * 0.5f);
    while ((i + 1) * (i + 2) / 2 <= e) ++i;
    while (i * (i + 1) / 2 > e) --i;
    const int j = e - i * (i + 1) / 2;
    const float *ki = b.kh + i * RS, *kj = b.kh + j * RS, *qi = b.qh + i * RS;
    const float *gi = b.gc + i * RS, *gj = b.gc + j * RS;
    float sg = 0.f, sm = 0.f;
#pragma unroll 4
    for (int c = 0; c < D; ++c) {
      const float t = kj[c] * __expf(gi[c] - gj[c]);  // gc_i <= gc_j: at most k^_j
      sg = fmaf(ki[c], t, sg);
      if (kQ) sm = fmaf(qi[c], t, sm);
    }
    b.G[i * PS + j] = j < i ? sg : 0.f;
    if (kQ) b.Mq[i * PS + j] = sm;
  }
  for (int e = threadIdx.x; e < CHUNK * CHUNK; e += NT) {
    const int i = e >> 6, j = e & 63;
    if (j > i) {
      b.G[i * PS + j] = 0.f;
      if (kQ) b.Mq[i * PS + j] = 0.f;
    }
  }
  __syncthreads();
}

// T = (I + diag(beta) G)^-1 (unit lower triangular) by forward substitution:
// column j by lanes 8 (j % 4) .. + 7 of warp j / 4, each dot product split
// over the eight lanes.  Ends with a barrier.
__device__ void wy_inverse_exact(const Basics &b) {
  const int j = threadIdx.x >> 3, part = threadIdx.x & 7;
  for (int i = 0; i < CHUNK; ++i) {
    float t = 0.f;
    if (i > j)
      for (int l = j + part; l < i; l += 8) t = fmaf(b.G[i * PS + l], b.T[l * PS + j], t);
    t += __shfl_xor_sync(0xffffffffu, t, 1);
    t += __shfl_xor_sync(0xffffffffu, t, 2);
    t += __shfl_xor_sync(0xffffffffu, t, 4);
    if (part == 0) b.T[i * PS + j] = i < j ? 0.f : (i == j ? 1.f : -b.beta[i] * t);
    __syncwarp();
  }
  __syncthreads();
}

// n16 16-byte pieces from global to shared memory
__device__ __forceinline__ void copy16(void *dst, const void *src, int n16) {
  for (int e = threadIdx.x; e < n16; e += NT)
    reinterpret_cast<uint4 *>(dst)[e] = reinterpret_cast<const uint4 *>(src)[e];
}

// 8 values of row c of a packed 128 x 128 bf16 state tile, columns v8 .. + 7
__device__ __forceinline__ void state_row8(const bf16 *S, int c, int v8, float *x) {
  ld16_bf(reinterpret_cast<const char *>(S) + umma::core_off(c, v8, D), x);
}

constexpr size_t kListBytes = (NT + 1) * 4;
constexpr size_t kPrepBytes = (size_t)(kBasicFloats + kRow) * 4 + kListBytes;
constexpr size_t kGradBytes = (size_t)(kBasicFloats + D + 8) * 4 + 32768 + 16384 + kListBytes;
static_assert(kPrepBytes <= 232448 && kGradBytes <= 232448, "shared memory budget");
static_assert((size_t)(kBasicFloats + D + 8) * 4 % 16 == 0, "16-byte aligned state tile");

}  // namespace rng

// The scans' operands (and the read-out's, by kMode) of every flagged chunk.
template <uint32_t kMode>
__global__ void __launch_bounds__(rng::NT, 1) kda_range_prep_kernel(KdaParams p, char *prep) {
  using namespace rng;
  pdl_wait();  // the prep kernel's flags and operand blocks
  constexpr bool readout = kMode != kPrepStates;
  extern __shared__ __align__(16) float rsm[];
  const Basics b = basics_view(rsm);
  float *Wf = rsm + kBasicFloats;  // [64][RS] W, fp32 (read-out)
  int *list = reinterpret_cast<int *>(Wf + kRow), *count = list + NT;
  const int H = p.H;
  for_each_flagged(p.range_flags, p.nslots * H, list, count, [&](int64_t u) {
    const int64_t slot = u / H;
    const int h = (int)(u - slot * H);
    int s_, j_, len;
    int64_t tok0;
    if (!slot_owner(p, slot, s_, j_, tok0, len)) return;  // (the prep kernel writes 0 there)
    char *unit = prep + (size_t)u * kPrepUnitBytes;
    const int tid = threadIdx.x, c = tid & 127, i0 = RB * (tid >> 7);
    chunk_basics<readout>(p, h, tok0, len, b);
    pair_matrices<readout>(b);
    wy_inverse_exact(b);
    // kr^T [c][i] and gT
#pragma unroll
    for (int q = 0; q < RB / 8; ++q) {
      float v[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int i = i0 + 8 * q + t;
        v[t] = b.kh[i * RS + c] * __expf(b.gT[c] - b.gc[i * RS + c]);
      }
      st16_bf(unit + kPrepKR + umma::core_off(c, i0 + 8 * q, 64), v);
    }
    if (tid < D) reinterpret_cast<float *>(unit + kPrepGT)[tid] = b.gT[tid];
    __syncthreads();
    // in place: kh <- diag(beta) kd, qh <- scale qd; then gc <- diag(beta) v
    for (int e = tid; e < CHUNK * D; e += NT) {
      const int i = e >> 7, cc = e & 127;
      const float eg = __expf(b.gc[i * RS + cc]);
      b.kh[i * RS + cc] *= b.beta[i] * eg;
      if (readout) b.qh[i * RS + cc] *= p.scale * eg;
    }
    __syncthreads();
    const bf16 *vg = static_cast<const bf16 *>(p.v);
    for (int e = tid; e < CHUNK * (D / 8); e += NT) {
      const int i = e >> 4, c8 = (e & 15) * 8;
      float x[8];
      if (i < len) ld16_bf(vg + ((tok0 + i) * H + h) * D + c8, x);
#pragma unroll
      for (int t = 0; t < 8; ++t) b.gc[i * RS + c8 + t] = i < len ? b.beta[i] * x[t] : 0.f;
    }
    __syncthreads();
    // W = T diag(beta) kd, U0 = T diag(beta) v: thread (channel c, rows i0 .. + 15)
    {
      float w[RB], u0[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) w[r] = u0[r] = 0.f;
      for (int j = 0; j < i0 + RB; ++j) {
        const float kj = b.kh[j * RS + c], vj = b.gc[j * RS + c];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const float t = b.T[(i0 + r) * PS + j];  // zero for j > i0 + r
          w[r] = fmaf(t, kj, w[r]);
          u0[r] = fmaf(t, vj, u0[r]);
        }
      }
#pragma unroll
      for (int q = 0; q < RB / 8; ++q) {
        const uint32_t off = umma::core_off(c, i0 + 8 * q, 64);
        st16_bf(unit + kPrepW + off, w + 8 * q);
        st16_bf(unit + kPrepU0 + off, u0 + 8 * q);
      }
      if (readout)
#pragma unroll
        for (int r = 0; r < RB; ++r) Wf[(i0 + r) * RS + c] = w[r];
    }
    if (readout) {
      __syncthreads();
      // QE = scale (qd - Mq W), and scale * Mq as the packed 64 x 64 tile
      float qe[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) qe[r] = b.qh[(i0 + r) * RS + c];
      for (int j = 0; j < i0 + RB; ++j) {
        const float wj = -p.scale * Wf[j * RS + c];
#pragma unroll
        for (int r = 0; r < RB; ++r) qe[r] = fmaf(b.Mq[(i0 + r) * PS + j], wj, qe[r]);
      }
#pragma unroll
      for (int q = 0; q < RB / 8; ++q)
        st16_bf(unit + kPrepQE + umma::core_off(c, i0 + 8 * q, 64), qe + 8 * q);
      for (int e8 = tid; e8 < CHUNK * 8; e8 += NT) {
        const int i = e8 >> 3, j0 = (e8 & 7) * 8;
        float m[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) m[t] = p.scale * b.Mq[i * PS + j0 + t];
        st16_bf(unit + kPrepMqk + umma::core_off(i, j0, 64), m);
      }
    }
    __syncthreads();  // the tiles are free for the next unit
  });
}

// The gradient rows and partials of every flagged chunk.  The chunk's prep
// block, which nothing reads after the gradient kernel, holds three fp32
// [64][128] row-major tiles: X, U, dY, later dkr / z, dqd / dgc and dkd.
__global__ void __launch_bounds__(rng::NT, 1)
    kda_range_grads_kernel(KdaParams p, const void *states) {
  using namespace rng;
  pdl_wait();  // the gradient kernel's rows and partials
  extern __shared__ __align__(16) float rsm[];
  const Basics b = basics_view(rsm);
  float *dgTs = rsm + kBasicFloats;  // [128] e^gT sum_v S dS
  float *red = dgTs + D;             // [8]
  bf16 *Sb = reinterpret_cast<bf16 *>(red + 8);   // packed 128 x 128: S_n, or dS_{n+1}
  bf16 *dOs = Sb + D * D;                         // [64][128] row-major
  int *list = reinterpret_cast<int *>(dOs + CHUNK * D), *count = list + NT;
  const int H = p.H;
  for_each_flagged(p.range_flags, p.nslots * H, list, count, [&](int64_t u) {
    const int64_t slot = u / H;
    const int h = (int)(u - slot * H);
    int s_, j_, len;
    int64_t tok0;
    if (!slot_owner(p, slot, s_, j_, tok0, len)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bf16 *Sg = static_cast<const bf16 *>(states) + (size_t)u * D * D;
    const bf16 *dSg = static_cast<const bf16 *>(p.dstates) + (size_t)u * D * D;
    float *X = reinterpret_cast<float *>(const_cast<char *>(p.prep) + (size_t)u * kPrepUnitBytes);
    float *U = X + CHUNK * D, *dY = U + CHUNK * D;
    const int64_t rowH = (int64_t)H * D;  // elements per token of a [*, H, 128] tensor
    copy16(Sb, Sg, D * D / 8);
    for (int e = tid; e < CHUNK * (D / 8); e += NT) {
      const int i = e >> 4, c8 = (e & 15) * 8;
      reinterpret_cast<uint4 *>(dOs + i * D + c8)[0] =
          i < len ? *reinterpret_cast<const uint4 *>(static_cast<const bf16 *>(p.dO) +
                                                     (tok0 + i) * rowH + h * D + c8)
                  : make_uint4(0u, 0u, 0u, 0u);
    }
    if (tid < D) {  // dgT's state term, e^gT[c] sum_v S[c][v] dS[c][v], from HBM
      float t = 0.f;
      for (int v8 = 0; v8 < D; v8 += 8) {
        float s8[8], d8[8];
        state_row8(Sg, tid, v8, s8);
        state_row8(dSg, tid, v8, d8);
#pragma unroll
        for (int x = 0; x < 8; ++x) t = fmaf(s8[x], d8[x], t);
      }
      dgTs[tid] = t;  // times e^gT below, once gT is known
    }
    chunk_basics<true>(p, h, tok0, len, b);
    pair_matrices<true>(b);
    wy_inverse_exact(b);
    // ---- X = v - kd S_n: thread (row i, columns v0 .. + 15) ----
    {
      const int i = tid >> 3, v0 = CG * (tid & 7);
      float x[CG];
      if (i < len) {
#pragma unroll
        for (int q = 0; q < CG / 8; ++q)
          ld16_bf(static_cast<const bf16 *>(p.v) + (tok0 + i) * rowH + h * D + v0 + 8 * q, x + 8 * q);
      } else {
#pragma unroll
        for (int r = 0; r < CG; ++r) x[r] = 0.f;
      }
      for (int c = 0; c < D; ++c) {
        const float kd = b.kh[i * RS + c] * __expf(b.gc[i * RS + c]);
#pragma unroll
        for (int q = 0; q < CG / 8; ++q) {
          float s8[8];
          state_row8(Sb, c, v0 + 8 * q, s8);
#pragma unroll
          for (int t = 0; t < 8; ++t) x[8 * q + t] = fmaf(-kd, s8[t], x[8 * q + t]);
        }
      }
#pragma unroll
      for (int q = 0; q < CG / 4; ++q)
        reinterpret_cast<float4 *>(X + i * D + v0)[q] =
            make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    }
    if (tid < D) dgTs[tid] *= __expf(b.gT[tid]);
    __syncthreads();
    // ---- U = T diag(beta) X: thread (column v, rows i0 .. + 15) ----
    {
      const int v = tid & 127, i0 = RB * (tid >> 7);
      float uu[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) uu[r] = 0.f;
      for (int j = 0; j < i0 + RB; ++j) {
        const float xj = b.beta[j] * X[j * D + v];
#pragma unroll
        for (int r = 0; r < RB; ++r) uu[r] = fmaf(b.T[(i0 + r) * PS + j], xj, uu[r]);
      }
#pragma unroll
      for (int r = 0; r < RB; ++r) U[(i0 + r) * D + v] = uu[r];
    }
    __syncthreads();
    copy16(Sb, dSg, D * D / 8);  // S_n is no longer read until it is copied back
    __syncthreads();
    // ---- dU = s Mq^T dO + kr dS_{n+1} (into dY's tile): thread (row i, columns v0 ..) ----
    {
      const int i = tid >> 3, v0 = CG * (tid & 7);
      float d[CG];
#pragma unroll
      for (int r = 0; r < CG; ++r) d[r] = 0.f;
      for (int l = i; l < CHUNK; ++l) {
        const float m = p.scale * b.Mq[l * PS + i];
#pragma unroll
        for (int q = 0; q < CG / 8; ++q) {
          float o8[8];
          ld16_bf(dOs + l * D + v0 + 8 * q, o8);
#pragma unroll
          for (int t = 0; t < 8; ++t) d[8 * q + t] = fmaf(m, o8[t], d[8 * q + t]);
        }
      }
      for (int c = 0; c < D; ++c) {
        const float kr = b.kh[i * RS + c] * __expf(b.gT[c] - b.gc[i * RS + c]);
#pragma unroll
        for (int q = 0; q < CG / 8; ++q) {
          float s8[8];
          state_row8(Sb, c, v0 + 8 * q, s8);
#pragma unroll
          for (int t = 0; t < 8; ++t) d[8 * q + t] = fmaf(kr, s8[t], d[8 * q + t]);
        }
      }
#pragma unroll
      for (int q = 0; q < CG / 4; ++q)
        reinterpret_cast<float4 *>(dY + i * D + v0)[q] =
            make_float4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]);
    }
    __syncthreads();
    // ---- dY = T^T dU in place: thread (column v, rows i0 .. + 15) ----
    {
      const int v = tid & 127, i0 = RB * (tid >> 7);
      float y[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) y[r] = 0.f;
      for (int i = i0; i < CHUNK; ++i) {
        const float du = dY[i * D + v];
#pragma unroll
        for (int r = 0; r < RB; ++r) y[r] = fmaf(b.T[i * PS + i0 + r], du, y[r]);  // T_ij = 0, j > i
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < RB; ++r) dY[(i0 + r) * D + v] = y[r];
    }
    __syncthreads();
    // ---- dv; U^T into shared memory (over dS_{n+1}, copied back below) ----
    {
      bf16 *dvg = static_cast<bf16 *>(p.dv);
      for (int e = tid; e < CHUNK * (D / 8); e += NT) {
        const int i = e >> 4, c8 = (e & 15) * 8;
        if (i < len) {
          float y[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) y[t] = b.beta[i] * dY[i * D + c8 + t];
          st16_bf(dvg + (tok0 + i) * rowH + h * D + c8, y);
        }
      }
      float *UT = reinterpret_cast<float *>(Sb);  // [128][64]
      for (int e = tid; e < CHUNK * D; e += NT) {
        const int j = e & 63, v = e >> 6;
        UT[v * CHUNK + j] = U[j * D + v];
      }
    }
    __syncthreads();
    // ---- the pair gradients: dG over G, dMq over Mq, dA o G over T.  Thread
    //      (column j, rows 8 iq .. + 7): dA_ij = -dY_i . U_j, dMq_ij = s dO_i . U_j ----
    {
      const float *UT = reinterpret_cast<const float *>(Sb);
      const int j = tid & 63, ib = PB * (tid >> 6);
      float a[PB], m[PB];
#pragma unroll
      for (int r = 0; r < PB; ++r) a[r] = m[r] = 0.f;
      for (int v8 = 0; v8 < D; v8 += 8) {
        float u8[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) u8[t] = UT[(v8 + t) * CHUNK + j];
#pragma unroll
        for (int r = 0; r < PB; ++r) {
          float o8[8];
          ld16_bf(dOs + (ib + r) * D + v8, o8);
          const float4 ya = reinterpret_cast<const float4 *>(dY + (ib + r) * D + v8)[0];
          const float4 yb = reinterpret_cast<const float4 *>(dY + (ib + r) * D + v8)[1];
          const float y8[8] = {ya.x, ya.y, ya.z, ya.w, yb.x, yb.y, yb.z, yb.w};
          float ta = a[r], tm = m[r];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            ta = fmaf(y8[t], u8[t], ta);
            tm = fmaf(o8[t], u8[t], tm);
          }
          a[r] = ta;
          m[r] = tm;
        }
      }
#pragma unroll
      for (int r = 0; r < PB; ++r) {
        const int i = ib + r;
        if (j <= i) {
          const float dA = j < i ? -a[r] : 0.f;
          b.T[i * PS + j] = dA * b.G[i * PS + j];
          b.G[i * PS + j] = b.beta[i] * dA;
          b.Mq[i * PS + j] = p.scale * m[r];
        }
      }
    }
    __syncthreads();
    copy16(Sb, dSg, D * D / 8);  // dS_{n+1} again, for dkr (made visible by the barrier below)
    // ---- dbeta, a warp per row ----
    for (int i = warp; i < CHUNK; i += NT / 32) {
      float t = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) t = fmaf(dY[i * D + lane + 32 * m], X[i * D + lane + 32 * m], t);
      t += b.T[i * PS + lane] + b.T[i * PS + lane + 32];
      t = warp_sum(t);
      if (lane == 0 && i < len)
        static_cast<bf16 *>(p.dbeta)[(tok0 + i) * H + h] = __float2bfloat16_rn(t);
    }
    __syncthreads();  // dS_{n+1} has landed
    // ---- dkr = U dS_{n+1}^T (over X), then dqd = s dO S_n^T (over U) and
    //      dkd = -diag(beta) dY S_n^T (over dY): thread (channel c, rows i0 .. + 15) ----
    const int c = tid & 127, i0 = RB * (tid >> 7);
    {
      float dkr[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) dkr[r] = 0.f;
      for (int v8 = 0; v8 < D; v8 += 8) {
        float s8[8];
        state_row8(Sb, c, v8, s8);
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const float4 ua = reinterpret_cast<const float4 *>(U + (i0 + r) * D + v8)[0];
          const float4 ub = reinterpret_cast<const float4 *>(U + (i0 + r) * D + v8)[1];
          float t = dkr[r];
          t = fmaf(ua.x, s8[0], t);
          t = fmaf(ua.y, s8[1], t);
          t = fmaf(ua.z, s8[2], t);
          t = fmaf(ua.w, s8[3], t);
          t = fmaf(ub.x, s8[4], t);
          t = fmaf(ub.y, s8[5], t);
          t = fmaf(ub.z, s8[6], t);
          t = fmaf(ub.w, s8[7], t);
          dkr[r] = t;
        }
      }
      __syncthreads();  // X (read by dbeta) and S's place in shared memory are free
#pragma unroll
      for (int r = 0; r < RB; ++r) X[(i0 + r) * D + c] = dkr[r];
    }
    copy16(Sb, Sg, D * D / 8);
    __syncthreads();
    // dqd, then dkd (one 32-row accumulator set at a time)
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      float acc[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) acc[r] = 0.f;
      for (int v8 = 0; v8 < D; v8 += 8) {
        float s8[8];
        state_row8(Sb, c, v8, s8);
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          float x8[8];
          if (pass == 0) {
            ld16_bf(dOs + (i0 + r) * D + v8, x8);
          } else {
            const float4 ya = reinterpret_cast<const float4 *>(dY + (i0 + r) * D + v8)[0];
            const float4 yb = reinterpret_cast<const float4 *>(dY + (i0 + r) * D + v8)[1];
            x8[0] = ya.x; x8[1] = ya.y; x8[2] = ya.z; x8[3] = ya.w;
            x8[4] = yb.x; x8[5] = yb.y; x8[6] = yb.z; x8[7] = yb.w;
          }
          float t = acc[r];
#pragma unroll
          for (int q = 0; q < 8; ++q) t = fmaf(x8[q], s8[q], t);
          acc[r] = t;
        }
      }
      __syncthreads();  // pass 0: U is read no more; pass 1: dY is read no more
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        if (pass == 0) U[(i0 + r) * D + c] = p.scale * acc[r];
        else dY[(i0 + r) * D + c] = -b.beta[i0 + r] * acc[r];
      }
    }
    __syncthreads();
    // ---- per (i, c): the pair matrices' terms, dq, dk, dgc (over dqd), z (over dkr) ----
    {
      bf16 *dqg = static_cast<bf16 *>(p.dq), *dkg = static_cast<bf16 *>(p.dk);
      for (int i = warp; i < CHUNK; i += NT / 32) {
        float dqh[4], dkh[4];
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int cc = lane + 32 * m;
          const float gci = b.gc[i * RS + cc], qi = b.qh[i * RS + cc], ki = b.kh[i * RS + cc];
          // a1 = sum_{j<i} dMq_ij k^_j e_ij,  a2 = sum_{j<i} dG_ij k^_j e_ij,
          // a3 = sum_{l>i} dG_li k^_l e_li,  a4 = sum_{l>i} dMq_li q^_l e_li
          float a1 = 0.f, a2 = 0.f, a3 = 0.f, a4 = 0.f;
          for (int j = 0; j < CHUNK; ++j) {
            const float d = gci - b.gc[j * RS + cc];
            const float kj = b.kh[j * RS + cc];
            if (j < i) {
              const float t = kj * __expf(d);
              a1 = fmaf(b.Mq[i * PS + j], t, a1);
              a2 = fmaf(b.G[i * PS + j], t, a2);
            } else if (j > i) {
              const float e = __expf(-d);
              a3 = fmaf(b.G[j * PS + i], kj * e, a3);
              a4 = fmaf(b.Mq[j * PS + i], b.qh[j * RS + cc] * e, a4);
            }
          }
          const float mii = b.Mq[i * PS + i];  // the diagonal pair, e_ii = 1
          const float eci = __expf(gci), krf = __expf(b.gT[cc] - gci);
          const float xq = U[i * D + cc] * eci;    // dqd e^gc
          const float xk = dY[i * D + cc] * eci;   // dkd e^gc
          const float xr = X[i * D + cc] * krf;    // dkr e^(gT - gc)
          dqh[m] = xq + a1 + mii * ki;
          dkh[m] = xk + xr + a2 + a3 + a4 + mii * qi;
          // the log-decay gradient.  Two pairs of its terms cancel exactly and
          // are left out rather than summed: the diagonal pair's (its factor
          // e_ii = 1 has no gate dependence), and kr's, -z_i here against +z_i
          // in dgT (gT - gc_i), which reach row t's dgk as the sum of z over
          // the rows before t (the gate epilogue).  With strong decay the
          // true dgk is many orders below those terms.
          U[i * D + cc] = qi * (xq + a1) + ki * (xk + a2 - a3 - a4);  // dgc
          X[i * D + cc] = ki * xr;                                    // z = kr dkr
          sq = fmaf(qi, dqh[m], sq);
          sk = fmaf(ki, dkh[m], sk);
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        if (i < len) {
          const float rq = b.rq[i], rk = b.rk[i];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int cc = lane + 32 * m;
            const int64_t o = (tok0 + i) * rowH + h * D + cc;
            dqg[o] = __float2bfloat16_rn(rq * (dqh[m] - b.qh[i * RS + cc] * sq));
            dkg[o] = __float2bfloat16_rn(rk * (dkh[m] - b.kh[i * RS + cc] * sk));
          }
        }
      }
    }
    __syncthreads();
    // ---- gate epilogue: channel c, reverse cumulative sum from the last row ----
    if (tid < D) {
      // dgk_t = sum_{i>=t} dgc_i + sum_{i<t} z_i + e^gT sum_v S dS: the
      // prefix sums of z first (over z)
      float pz = 0.f;
      for (int i = 0; i < CHUNK; ++i) {
        const float z = X[i * D + tid];
        X[i * D + tid] = pz;
        pz += z;
      }
      const float nA = -__expf(p.A_log[h]), bias = gate_bias(p, h, tid, D);
      const bf16 *gg = static_cast<const bf16 *>(p.g);
      bf16 *dgg = static_cast<bf16 *>(p.dg);
      float suf = dgTs[tid], dA = 0.f, ddt = 0.f;
      for (int i = CHUNK - 1; i >= 0; --i) {
        suf += U[i * D + tid];
        const float run = suf + X[i * D + tid];  // dgk of row i
        if (i < len) {
          const int64_t o = (tok0 + i) * rowH + h * D + tid;
          const float gv = __bfloat162float(gg[o]) + bias;
          const float t = __expf(-fabsf(gv));
          const float inv = 1.f / (1.f + t);
          const float sg = gv >= 0.f ? inv : t * inv;
          const float dgv = run * nA * sg;
          dgg[o] = __float2bfloat16_rn(dgv);
          dA = fmaf(run, fmaxf(gv, 0.f) + log1p_unit(t), dA);
          ddt += dgv;
        }
      }
      dA = warp_sum(dA * nA);
      if (lane == 0) red[warp] = dA;
      if (p.ddt_part != nullptr) p.ddt_part[u * D + tid] = ddt;
    }
    __syncthreads();
    if (tid == 0) p.dA_part[u] = (red[0] + red[1]) + (red[2] + red[3]);
    __syncthreads();  // shared memory is free for the next unit
  });
}

namespace {

unsigned range_grid(const KdaParams &p) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t units = p.nslots * p.H;
  return (unsigned)(units < sms ? units : sms);
}

}  // namespace

cudaError_t range_prep_launch(const KdaParams &p, void *prep, cudaStream_t st) {
  if (p.range_flags == nullptr || p.nslots * p.H == 0) return cudaSuccess;
  auto kfn = p.prep_mode == kPrepStates    ? kda_range_prep_kernel<kPrepStates>
             : p.prep_mode == kPrepReadout ? kda_range_prep_kernel<kPrepReadout>
                                           : kda_range_prep_kernel<kPrepAll>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)rng::kPrepBytes);
  if (e != cudaSuccess) return e;
  return pdl_launch(kfn, dim3(range_grid(p)), dim3(rng::NT), rng::kPrepBytes, st, p,
                    static_cast<char *>(prep));
}

cudaError_t range_grads_launch(const KdaParams &p, const void *states, cudaStream_t st) {
  if (p.range_flags == nullptr || p.nslots * p.H == 0) return cudaSuccess;
  if (!p.states_packed || !p.dstates_packed || p.prep == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kda_range_grads_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)rng::kGradBytes);
  if (e != cudaSuccess) return e;
  return pdl_launch(kda_range_grads_kernel, dim3(range_grid(p)), dim3(rng::NT), rng::kGradBytes,
                    st, p, states);
}

int range_status_take() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_status, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

}  // namespace kda
