// kda_params.h -- launch parameters shared by the host API and the kernels,
// and the host-side entry points of the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

// Launches kernel(args...) allowed to start while the previous kernel on the
// stream finishes (programmatic dependent launch); the kernel calls pdl_wait()
// (kda_device.cuh) before reading anything the previous kernels wrote.  It
// hides the gap between two dependent launches.
template <typename... K, typename... A>
inline cudaError_t pdl_launch(void (*kernel)(K...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct KdaParams {
  int B, T, H, num_seqs;
  const int32_t *cu;          // device, nullable
  int nps;                    // slots per sequence (fixed length): ceil(T / 64)
  int64_t nslots;
  float scale, eps;
  const void *q, *k, *v, *g, *beta, *dO;
  const float *A_log, *h0, *dhT;
  const float *dt_bias;       // nullable [H, K]: the gate's per-channel bias
  void *states;               // [slots, H, K, V] (written by the forward scan)
  float *hT;                  // nullable
  void *dstates;              // [slots, H, K, V]
  float *dh0;                 // nullable
  void *dq, *dk, *dv, *dg, *dbeta;
  float *dA_part;             // [slots, H]
  float *dA_log;              // [H]
  float *ddt_part;            // [slots, H, K] per-chunk partials of ddt_bias
  float *ddt_bias;            // nullable [H, K], overwritten
  int nb;                     // V bands of the scan kernels
  int role_base;              // first scan role of a launch (0 forward, 1 reverse)
  // Layout of each K x V tile of states / dstates: 0 = row-major, 1 = packed
  // core-matrix order (8 x 8 bf16 cores of 128 bytes, cores along V first),
  // the shared-memory operand layout the tcgen05 scans store with one bulk copy.
  int states_packed, dstates_packed;
  const char *prep;           // per-chunk operand blocks (bf16, K = V = 128), see below
  const int32_t *seq_order;   // tcgen05 scans: sequences longest first (varlen), or null
  // Context-parallel tcgen05 scans: each sequence's chunks (nck of them) are
  // split into cp_segs >= 3 segments, segment g holding
  // chunks [g nck / cp_segs, (g + 1) nck / cp_segs).  cp_phase 1 runs every
  // segment's local scan and the transfer matrices, 2 (the combine kernel)
  // chains them into the true segment boundaries, 3 reruns the segments
  // from those boundaries; cp_nroles roles from role_base take part.
  // cp_buf holds kda_cp_tiles(cp_segs) fp32 K x V row-major tiles per
  // (sequence, head); see kda_scan_tc.cu.  cp_segs = 0: whole-sequence chains.
  int cp_segs, cp_phase, cp_nroles;
  float *cp_buf;
  // Timeout tests: kernels named in `starve` (kStarve* bits) arm their first
  // load barrier but issue none of its copies, so that its bounded wait runs
  // out; `poll_limit` (0 = the kernels' defaults) caps every bounded wait.
  uint32_t starve, poll_limit;
  // What the prep kernel writes beyond the scans' operands (W^T, kr^T, U0^T,
  // gT): kPrepAll (0) everything, the gradient kernel's tiles and factors
  // included; kPrepReadout (1) also QE^T and scale * Mqk, which the forward
  // read-out needs; kPrepStates (2) nothing more (the chunk states alone).
  uint32_t prep_mode;
  // [slots, H] flags of the chunks whose gate passes the 16-row block
  // factors' range (kda_range.cu), written by the tcgen05 prep kernel for
  // every (chunk slot, head); null: such chunks raise KDA_ERR_GATE_RANGE.
  int32_t *range_flags;
};

constexpr uint32_t kPrepAll = 0, kPrepReadout = 1, kPrepStates = 2;

constexpr uint32_t kStarvePrep = 1, kStarveScan = 2, kStarveGrads = 4, kStarveOut = 8;

// poll limit of a bounded wait: the launch's cap, else the kernel's default
__host__ __device__ constexpr uint32_t poll_cap(const KdaParams &p, uint32_t dflt) {
  return p.poll_limit != 0u && p.poll_limit < dflt ? p.poll_limit : dflt;
}

// fp32 K x V tiles per (sequence, head) of the context-parallel scans:
// forward segment starts (P - 1), reverse segment ends (P - 1) and the
// transfer matrices of the inner segments (P - 2).
__host__ __device__ constexpr int kda_cp_tiles(int P) { return P >= 3 ? 3 * P - 4 : 0; }

// Per-chunk operands of the state scans (bf16, K = V = 128), one block of
// kPrepUnitBytes per (chunk slot, head), written by the chunk-parallel prep
// kernel and streamed by the tcgen05 scans.  Every tile is a 128 x 64 or
// 64 x 128 bf16 matrix in packed core-matrix order (8 x 8 cores of 128
// bytes, cores along the columns first):
//   gT   fp32 [128]          total log-decay of the chunk per channel
//   Wt   [c][i]  W^T,  W  = (I + Akk)^-1 diag(beta) kd
//   KRt  [c][i]  kr^T, kr = k^ e^(gT - gc)
//   U0t  [v][i]  U0^T, U0 = (I + Akk)^-1 diag(beta) v
//   QEt  [c][i]  QE^T, QE = scale (qd - Mqk W)
// and, for the gradient kernel, 64 x 64 bf16 tiles in the same order:
//   Mqk  [i][j]  scale * lower(qd ki^T) (diagonal included)
//   INV  [i][j]  (I + Akk)^-1,  INVb = INV diag(beta)
//   G    [i][j]  strict_lower(kd ki^T)  (Akk = diag(beta) G)
// and the per-chunk factors of the 16-row blocks, fp32, 8 KB:
//   SV   e^(m_I) [4][128] | e^(gT - m_I) [4][128] | e^(m_I - m_J) [6][128] |
//        gT [128] | 1/|q_i| [64] | 1/|k_i| [64]
//   (m_I = gc at row 16 I + 7; the layout of the kernels' shared-memory view
//   from its e^(m_I) array on)
constexpr size_t kPrepGT = 0;
constexpr size_t kPrepW = 512;
constexpr size_t kPrepKR = kPrepW + 16384;
constexpr size_t kPrepU0 = kPrepKR + 16384;
constexpr size_t kPrepQE = kPrepU0 + 16384;
constexpr size_t kPrepMqk = kPrepQE + 16384;
constexpr size_t kPrepINV = kPrepMqk + 8192;
constexpr size_t kPrepINVb = kPrepINV + 8192;
constexpr size_t kPrepG = kPrepINVb + 8192;
constexpr size_t kPrepSV = kPrepG + 8192;
constexpr size_t kPrepSVBytes = 8192;
constexpr size_t kPrepUnitBytes = kPrepSV + kPrepSVBytes;

// TMA tensor maps of the token-major bf16 tensors [B * T, H, 128]: one box is
// the 64 rows x 128 channels of one chunk and head, row-major (256-byte rows)
// in shared memory; rows past the tensor's end read as zero (and are not
// written by a store).  Inputs q, k, g, v, dO; gradients dq, dk, dv, dg
// (stored from shared memory for whole chunks).  dO_sw and v_sw map dO and v
// with boxes of 64 rows x 64 channels in the 128-byte swizzled layout
// (umma::sw128_off), which the tensor cores read as it lands.  A null tensor
// keeps an empty map.
struct TokenMaps {
  CUtensorMap q, k, g, v, dO;
  CUtensorMap dq, dk, dv, dg;
  CUtensorMap dO_sw, v_sw;
};
// kda_tmap.cu: encodes the five maps; false if the driver refuses one.
bool encode_token_maps(const KdaParams &p, TokenMaps &m);

// kda_prep_tc.cu: the per-chunk scan operands above (bf16, K = V = 128).
cudaError_t prep_tc_launch(const KdaParams &p, const TokenMaps &tm, void *prep, cudaStream_t st);
int prep_tc_status_take();

// kda_scan_tc.cu: both state scans on tcgen05 from the prep buffer; roles
// as in scan_dispatch.
// (the reverse role takes each chunk's dO through tm.dO_sw)
cudaError_t scan_tc_launch(const KdaParams &p, const TokenMaps &tm, const void *prep, int nroles,
                           cudaStream_t st);
// the three phases of the context-parallel scans (p.cp_segs >= 3); p.role_base
// and nroles as for scan_tc_launch
cudaError_t scan_tc_cp_launch(KdaParams p, const TokenMaps &tm, const void *prep, int nroles,
                              cudaStream_t st);
// order[r] = the sequence of rank r by length (longest first, ties by index)
cudaError_t seq_order_launch(const int32_t *cu, int num_seqs, int32_t *order, cudaStream_t st);
int scan_tc_status_take();

// kda_range.cu: exact fp32 arithmetic for the chunks p.range_flags marks
// (no-ops without flags).  range_prep_launch after prep_tc_launch (the scans'
// operands, and the read-out's by p.prep_mode), range_grads_launch after
// grads_tc_launch (the chunk's gradient rows and partials; the prep block
// serves as its scratch).
cudaError_t range_prep_launch(const KdaParams &p, void *prep, cudaStream_t st);
cudaError_t range_grads_launch(const KdaParams &p, const void *states, cudaStream_t st);
int range_status_take();

// kda_out_tc.cu: forward outputs o = QE S_n + Mqk U0 per chunk (bf16, K = V =
// 128) from the prep blocks and the packed chunk states.
cudaError_t out_tc_launch(const KdaParams &p, const void *states, void *o, cudaStream_t st);
int out_tc_status_take();

// kda_scan.cu: forward-state scan (role 0) and reverse dS scan (role 1).
cudaError_t scan_dispatch(const KdaParams &p, int K, bool bf16, int bv, int nroles,
                          cudaStream_t st);
size_t scan_smem_bytes(int K, bool bf16, int bv);
int scan_status_take();

// kda_grads.cu: per-chunk gradients and the dA_log reduction.
// `after_grads` (nullable cudaEvent_t) is recorded between the gradient
// kernel and the dA_log reduction.
cudaError_t grads_dispatch(const KdaParams &p, int K, bool bf16, const void *states,
                           cudaStream_t st, void *after_grads = nullptr,
                           const TokenMaps *tm = nullptr);
size_t grads_smem_bytes(int K, bool bf16);
int grads_status_take();

// kda_pad.cu: bf16 K = V = 64 on the 128-channel path.  rows x 64 bf16 <->
// rows x 128 bf16 (padded channels = fill), n fp32 tiles a x b <-> A x B
// (zero outside), and n row-major 64 x 64 bf16 states <-> packed 128 x 128.
cudaError_t pad_rows_launch(const void *src, void *dst, int64_t rows, float fill,
                            cudaStream_t st);
cudaError_t unpad_rows_launch(const void *src, void *dst, int64_t rows, cudaStream_t st);
cudaError_t pad_tiles_f32_launch(const float *src, float *dst, int64_t n, int a, int b, int A,
                                 int B, bool unpad, cudaStream_t st);
cudaError_t pack_states64_launch(const void *src, void *dst, int64_t n, cudaStream_t st);
cudaError_t unpack_states64_launch(const void *src, void *dst, int64_t n, cudaStream_t st);

// kda_grads_tc.cu: the same per-chunk gradients on tcgen05 (bf16, K = V = 128).
cudaError_t grads_tc_launch(const KdaParams &p, const TokenMaps &tm, const void *states,
                            cudaStream_t st);
size_t grads_tc_smem_bytes();
int grads_tc_status_take();

}  // namespace kda
