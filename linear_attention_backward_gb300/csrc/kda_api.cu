// kda_api.cu -- host side of the C ABI declared in include/kda.h: argument
// validation, workspace layout, launch sequencing and the device status word.
#include <cuda_runtime.h>

#include <stdint.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "kda.h"
#include "kda_params.h"

namespace {

constexpr int kChunk = 64;
constexpr size_t kAlign = 256;
constexpr int kTargetCtas = 152;  // one wave of the scan kernels fills the SMs

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int num_seqs_of(const kda_shape *s) { return s->cu_seqlens ? s->num_seqs : s->B; }

// Structural validation of a shape (no pointers other than cu_seqlens' presence).
kda_status check_shape(const kda_shape *s) {
  if (s == nullptr) return KDA_ERR_INVALID_ARG;
  if (s->B < 1 || s->T < 0 || s->H < 1 || s->K < 1 || s->V < 1) return KDA_ERR_INVALID_ARG;
  if (s->dtype != KDA_FP32 && s->dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (s->chunk != kChunk) return KDA_ERR_UNSUPPORTED;
  if (s->cu_seqlens != nullptr) {
    if (s->B != 1 || s->num_seqs < 1) return KDA_ERR_INVALID_ARG;
  } else if (s->num_seqs != 0) {
    return KDA_ERR_INVALID_ARG;
  }
  if (s->K != s->V) return KDA_ERR_UNSUPPORTED;
  if (s->K != 64 && s->K != 128) return KDA_ERR_UNSUPPORTED;
  if (s->dtype == KDA_FP32 && s->K != 64) return KDA_ERR_UNSUPPORTED;
  // sizes must stay inside 32-bit element offsets per row and 64-bit overall
  if ((int64_t)s->B * s->T > (int64_t)1 << 31) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

int64_t slots_of(const kda_shape *s) {
  if (s->cu_seqlens) return (int64_t)(s->T / kChunk) + s->num_seqs;
  return (int64_t)s->B * ((s->T + kChunk - 1) / kChunk);
}

size_t elem_size(const kda_shape *s) { return s->dtype == KDA_BF16 ? 2 : 4; }

size_t states_bytes(const kda_shape *s) {
  return round_up((size_t)slots_of(s) * s->H * (size_t)s->K * s->V * elem_size(s));
}

// Test hook of the timeout tests: KDA_TEST_STARVE_WAITS names kernels
// (any of prep, scan, grads, out) that arm their first load barrier without
// issuing its copies, so that their bounded waits run out; every bounded
// wait of such a call then polls at most 4096 times.
void test_hooks(kda::KdaParams &p) {
  const char *e = getenv("KDA_TEST_STARVE_WAITS");
  if (e == nullptr || e[0] == '\0') return;
  if (strstr(e, "prep")) p.starve |= kda::kStarvePrep;
  if (strstr(e, "scan")) p.starve |= kda::kStarveScan;
  if (strstr(e, "grads")) p.starve |= kda::kStarveGrads;
  if (strstr(e, "out")) p.starve |= kda::kStarveOut;
  if (p.starve != 0u) p.poll_limit = 4096u;
}

void fill_params(const kda_shape *s, kda::KdaParams &p) {
  memset(&p, 0, sizeof(p));
  p.B = s->B;
  p.T = s->T;
  p.H = s->H;
  p.num_seqs = num_seqs_of(s);
  p.cu = s->cu_seqlens;
  p.nps = (s->T + kChunk - 1) / kChunk;
  p.nslots = slots_of(s);
  p.scale = s->scale > 0.f ? s->scale : 1.0f / sqrtf((float)s->K);
  p.eps = s->l2_eps >= 0.f ? s->l2_eps : 1e-6f;
  p.nb = 1;
  test_hooks(p);
}

// V band width of the scan kernels: wide bands unless the (sequence, head,
// role) units alone leave most SMs idle.
int pick_band(const kda_shape *s, int nroles) {
  const int units = num_seqs_of(s) * s->H * nroles;
  int bv = s->V;
  while (bv > 32 && units * (s->V / bv) * 2 <= kTargetCtas) bv /= 2;
  return bv;
}

// The tcgen05 state path (chunk-parallel prep + streaming scans) serves bf16
// with K = V = 128; its per-chunk operand blocks live in the workspace.
bool tc_state_path(const kda_shape *s) { return s->dtype == KDA_BF16 && s->K == 128; }

size_t prep_bytes(const kda_shape *s) {
  if (!tc_state_path(s)) return 0;
  return round_up((size_t)slots_of(s) * s->H * kda::kPrepUnitBytes);
}

// KDA_SCAN_LEGACY=1 selects the per-band scans (which redo the chunk prep
// in every band) instead of prep + tcgen05 scans, for comparisons.
bool legacy_scan() {
  const char *e = getenv("KDA_SCAN_LEGACY");
  return e != nullptr && e[0] == '1';
}

kda_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

// Segments of the context-parallel tcgen05 scans (0: whole-sequence chains).
// Used when the whole-sequence chains (two per sequence and head) leave most
// SMs idle: the most segments (3..8, at least four chunks each) whose phase-1
// chains, kda_cp_tiles(P) per sequence and head, still fit one per SM.  When
// even three segments do not fit so but the whole-sequence chains fill at
// most half the SMs (up to 38 sequence-heads), the most whose chains fit two
// per SM, the scan kernel's residency: at B = 1, T = 8192, H = 32 four
// segments take the scans from 0.282 to 0.222 ms, where at H = 16 more than
// the one-per-SM count (four) gained nothing.  A function of the shape, so
// that the workspace size is too: for varlen the host does not read
// cu_seqlens, and the chunks per sequence are taken as the average
// T / 64 / num_seqs (shorter sequences get shorter, possibly empty, segments).
int cp_segments(const kda_shape *s) {
  if (!tc_state_path(s)) return 0;
  const int64_t units = (int64_t)num_seqs_of(s) * s->H;
  const int nck = s->cu_seqlens ? (int)((s->T / kChunk) / s->num_seqs)
                                : (s->T + kChunk - 1) / kChunk;
  if (2 * units >= kTargetCtas) return 0;
  int best = 0;
  for (int P = 3; P <= 8; ++P)
    if (kda::kda_cp_tiles(P) * units <= kTargetCtas && nck >= 4 * P) best = P;
  if (best == 0 && 4 * units <= kTargetCtas)
    for (int P = 3; P <= 8; ++P)
      if (kda::kda_cp_tiles(P) * units <= 2 * kTargetCtas && nck >= 4 * P) best = P;
  return best;
}

// Segments a call uses: KDA_SCAN_CP=0 turns the context-parallel scans off,
// KDA_SCAN_CP=n (3 <= n <= cp_segments) takes n segments, for comparisons.
int cp_segments_used(const kda_shape *s) {
  const int P = cp_segments(s);
  const char *e = getenv("KDA_SCAN_CP");
  if (e == nullptr || P == 0) return P;
  const int n = atoi(e);
  if (n == 0) return 0;
  return n >= 3 && n <= P ? n : P;
}

size_t cp_bytes(const kda_shape *s) {
  return round_up((size_t)num_seqs_of(s) * s->H * (size_t)kda::kda_cp_tiles(cp_segments(s)) *
                  s->K * s->V * sizeof(float));
}

// Workspace layout: states | dS | dA_log partials [slots, H] | ddt_bias
// partials [slots, H, K] | per-chunk operand blocks (tcgen05 path) |
// boundary tiles of the context-parallel scans | range flags [slots, H]
// (tcgen05 path: the chunks whose gate the exact kernels of kda_range.cu take).
size_t dA_part_offset(const kda_shape *s) { return 2 * states_bytes(s); }
size_t ddt_part_offset(const kda_shape *s) {
  return dA_part_offset(s) + round_up((size_t)slots_of(s) * s->H * sizeof(float));
}
size_t prep_offset(const kda_shape *s) {
  return ddt_part_offset(s) + round_up((size_t)slots_of(s) * s->H * s->K * sizeof(float));
}
size_t cp_offset(const kda_shape *s) { return prep_offset(s) + prep_bytes(s); }
size_t flags_offset(const kda_shape *s) { return cp_offset(s) + cp_bytes(s); }
size_t flags_bytes(const kda_shape *s) {
  return tc_state_path(s) ? round_up((size_t)slots_of(s) * s->H * sizeof(int32_t)) : 0;
}

// The forward half shared by kda_fwd and kda_fwd_states on the tcgen05 path:
// per-chunk operands into the workspace, then the forward state scan (whole
// sequences, or context-parallel segments when the chains alone leave most
// SMs idle), which stores every chunk-start state in packed core-matrix
// order to p.states and the final states to p.hT.  p holds the inputs, the
// outputs and p.dA_part (the sequence order of varlen scans lives there).
cudaError_t forward_states_tc(kda::KdaParams &p, const kda_shape *shape, char *w,
                              const kda::TokenMaps &tm, cudaStream_t cs) {
  void *prep = w + prep_offset(shape);
  p.prep = static_cast<const char *>(prep);
  p.range_flags = reinterpret_cast<int32_t *>(w + flags_offset(shape));
  cudaError_t e = kda::prep_tc_launch(p, tm, prep, cs);
  if (e == cudaSuccess) e = kda::range_prep_launch(p, prep, cs);
  p.role_base = 0;
  p.states_packed = 1;
  const int cp = cp_segments_used(shape);
  if (e == cudaSuccess && p.cu != nullptr && cp < 3) {
    p.seq_order = reinterpret_cast<const int32_t *>(p.dA_part);
    e = kda::seq_order_launch(p.cu, p.num_seqs, reinterpret_cast<int32_t *>(p.dA_part), cs);
  }
  if (e == cudaSuccess && cp >= 3) {
    p.cp_segs = cp;
    p.cp_buf = reinterpret_cast<float *>(w + cp_offset(shape));
    e = kda::scan_tc_cp_launch(p, tm, p.prep, 1, cs);
    p.cp_segs = 0;
  } else if (e == cudaSuccess) {
    e = kda::scan_tc_launch(p, tm, p.prep, 1, cs);
  }
  return e;
}

// ---- bf16 K = V = 64 on the 128-channel tensor-core path -------------------
// The shape's channels are zero-padded to 128 (kda_pad.cu explains why the
// result is exact); the padded copies live behind the padded shape's own
// workspace.  KDA_PAD64=0 runs such shapes on the mma.sync kernels instead,
// for comparisons.
bool pad64_shape(const kda_shape *s) {
  return s->dtype == KDA_BF16 && s->K == 64 && s->V == 64;
}
bool pad64_path(const kda_shape *s) {
  if (!pad64_shape(s)) return false;
  const char *e = getenv("KDA_PAD64");
  return e == nullptr || e[0] != '0';
}
kda_shape padded_shape(const kda_shape *s) {
  kda_shape p = *s;
  p.K = p.V = 128;
  p.scale = s->scale > 0.f ? s->scale : 0.125f;  // the 64-channel problem's 64^-1/2
  return p;
}
// byte offsets of the padded copies: the padded shape's workspace [0, inner),
// then q, k, v, g, dO and dq, dk, dv, dg ([B, T, H, 128] bf16), h0, dh_T,
// dh0 ([N, H, 128, 128] fp32), dt_bias, ddt_bias ([H, 128] fp32) and given
// states ([slots, H, 128, 128] bf16, packed)
struct Pad64 {
  size_t inner, q, k, v, g, dO, dq, dk, dv, dg, h0, dhT, dh0, dt, ddt, states, total;
};
Pad64 pad64_layout(const kda_shape *s) {
  const kda_shape ps = padded_shape(s);
  Pad64 L;
  size_t o = round_up(flags_offset(&ps) + flags_bytes(&ps));
  L.inner = o;
  const size_t tok = round_up((size_t)s->B * s->T * s->H * 128 * 2);
  size_t *toks[] = {&L.q, &L.k, &L.v, &L.g, &L.dO, &L.dq, &L.dk, &L.dv, &L.dg};
  for (size_t *t : toks) {
    *t = o;
    o += tok;
  }
  const size_t st = round_up((size_t)num_seqs_of(s) * s->H * 128 * 128 * 4);
  L.h0 = o;
  o += st;
  L.dhT = o;
  o += st;
  L.dh0 = o;
  o += st;
  const size_t bias = round_up((size_t)s->H * 128 * 4);
  L.dt = o;
  o += bias;
  L.ddt = o;
  o += bias;
  L.states = o;
  o += round_up((size_t)slots_of(s) * s->H * 128 * 128 * 2);
  L.total = o;
  return L;
}

kda_status check_ws(const kda_shape *shape, const void *ws, size_t ws_bytes) {
  const size_t need = kda_workspace_bytes(shape);
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return KDA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return KDA_ERR_WORKSPACE;
  return KDA_OK;
}

}  // namespace

extern "C" {

int kda_abi_version(void) { return 7; }

const char *kda_status_str(kda_status st) {
  switch (st) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_TIMEOUT: return "device-side wait timed out";
    case KDA_ERR_DEVICE_ARG: return "device found a malformed cu_seqlens table";
    case KDA_ERR_TOO_LARGE: return "problem exceeds the fixed no-allocation scratch";
    case KDA_ERR_GATE_RANGE: return "gate log-decay around a 16-row block exceeds 88 nats";
  }
  return "unknown status";
}

int64_t kda_num_chunk_slots(const kda_shape *shape) {
  if (check_shape(shape) != KDA_OK) return 0;
  return slots_of(shape);
}

size_t kda_workspace_dstates_offset(const kda_shape *shape) {
  if (check_shape(shape) != KDA_OK) return 0;
  if (pad64_path(shape)) {
    const kda_shape ps = padded_shape(shape);
    return states_bytes(&ps);
  }
  return states_bytes(shape);
}

int kda_scan_segments(const kda_shape *shape) {
  if (check_shape(shape) != KDA_OK) return 0;
  if (pad64_path(shape)) {
    const kda_shape ps = padded_shape(shape);
    return cp_segments_used(&ps);
  }
  return cp_segments_used(shape);
}

size_t kda_workspace_bytes(const kda_shape *shape) {
  if (check_shape(shape) != KDA_OK) return 0;
  if (pad64_shape(shape)) return pad64_layout(shape).total;  // also covers the mma.sync path
  return flags_offset(shape) + flags_bytes(shape);
}

kda_status kda_check_cu_seqlens_host(const int32_t *cu, int num_seqs, int total_T) {
  if (cu == nullptr || num_seqs < 1 || total_T < 0) return KDA_ERR_INVALID_ARG;
  if (cu[0] != 0 || cu[num_seqs] != total_T) return KDA_ERR_INVALID_ARG;
  for (int i = 0; i < num_seqs; ++i)
    if (cu[i + 1] < cu[i]) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

kda_status kda_fwd_states(const kda_shape *shape, const void *q, const void *k, const void *v,
                          const void *g, const void *beta, const float *A_log,
                          const float *dt_bias, const float *h0, void *states, float *hT,
                          void *ws, size_t ws_bytes, kda_stream_t stream) {
  kda_status st = check_shape(shape);
  if (st != KDA_OK) return st;
  const bool tokens = (int64_t)shape->B * shape->T > 0;
  const bool tc = tc_state_path(shape);
  if (!A_log) return KDA_ERR_INVALID_ARG;
  if (tokens && (!k || !v || !g || !beta || !states || (tc && !q))) return KDA_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, A_log, dt_bias, h0, states, hT};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  kda::KdaParams p;
  fill_params(shape, p);
  p.q = q;
  p.k = k;
  p.v = v;
  p.g = g;
  p.beta = beta;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.h0 = h0;
  p.states = states;
  p.hT = hT;
  if (pad64_path(shape) && ws != nullptr && (q != nullptr || !tokens)) {
    // bf16 K = V = 64 with a workspace: the 128-channel prep and forward scan
    // on padded copies, then the states' 64 x 64 corners (row-major) and hT
    // cut back out
    st = check_ws(shape, ws, ws_bytes);
    if (st != KDA_OK) return st;
    const kda_shape ps = padded_shape(shape);
    const Pad64 L = pad64_layout(shape);
    char *w = static_cast<char *>(ws);
    const int64_t rows = (int64_t)shape->B * shape->T * shape->H;
    const int64_t nst = (int64_t)num_seqs_of(shape) * shape->H;
    cudaError_t e = cudaSuccess;
    const void *src[] = {q, k, v, g};
    const size_t dst[] = {L.q, L.k, L.v, L.g};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      if (src[i]) e = kda::pad_rows_launch(src[i], w + dst[i], rows, i == 3 ? -30.f : 0.f, cs);
    float *h0p = h0 ? reinterpret_cast<float *>(w + L.h0) : nullptr;
    float *dtp = dt_bias ? reinterpret_cast<float *>(w + L.dt) : nullptr;
    float *hTp = hT ? reinterpret_cast<float *>(w + L.dh0) : nullptr;
    if (e == cudaSuccess && h0) e = kda::pad_tiles_f32_launch(h0, h0p, nst, 64, 64, 128, 128, false, cs);
    if (e == cudaSuccess && dt_bias)
      e = kda::pad_tiles_f32_launch(dt_bias, dtp, shape->H, 1, 64, 1, 128, false, cs);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    st = kda_fwd_states(&ps, w + L.q, w + L.k, w + L.v, w + L.g, beta, A_log, dtp, h0p,
                        w + L.states, hTp, w, L.inner, stream);
    if (st != KDA_OK) return st;
    if (tokens) e = kda::unpack_states64_launch(w + L.states, states, slots_of(shape) * shape->H, cs);
    if (e == cudaSuccess && hT) e = kda::pad_tiles_f32_launch(hTp, hT, nst, 64, 64, 128, 128, true, cs);
    return from_cuda(e);
  }
  if (tc) {
    // the tcgen05 path: the chunk-parallel prep and the forward scan, with
    // the operand blocks in the caller's workspace
    st = check_ws(shape, ws, ws_bytes);
    if (st != KDA_OK) return st;
    char *w = static_cast<char *>(ws);
    p.dA_part = reinterpret_cast<float *>(w + dA_part_offset(shape));
    kda::TokenMaps tm{};  // left zero when there are no tokens (no kernel then reads it)
    if (!kda::encode_token_maps(p, tm)) return KDA_ERR_CUDA;
    p.prep_mode = kda::kPrepStates;  // the scans' operands only
    return from_cuda(forward_states_tc(p, shape, w, tm, cs));
  }
  // other dtypes and head sizes (and bf16 K = V = 64 without a workspace):
  // the per-band scan (row-major states; no workspace)
  p.role_base = 0;
  const int bv = pick_band(shape, 1);
  p.nb = shape->V / bv;
  return from_cuda(kda::scan_dispatch(p, shape->K, shape->dtype == KDA_BF16, bv, 1, cs));
}

kda_status kda_fwd(const kda_shape *shape, const void *q, const void *k, const void *v,
                   const void *g, const void *beta, const float *A_log, const float *dt_bias,
                   const float *h0, void *o, float *hT, void *ws, size_t ws_bytes,
                   kda_stream_t stream) {
  kda_status st = check_shape(shape);
  if (st != KDA_OK) return st;
  if (!tc_state_path(shape) && !pad64_path(shape)) return KDA_ERR_UNSUPPORTED;
  const bool tokens = (int64_t)shape->B * shape->T > 0;
  if (!A_log) return KDA_ERR_INVALID_ARG;
  if (tokens && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, A_log, dt_bias, h0, o, hT};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return KDA_ERR_INVALID_ARG;
  st = check_ws(shape, ws, ws_bytes);
  if (st != KDA_OK) return st;
  if (pad64_path(shape)) {
    // the 128-channel forward on padded copies, then o and hT cut back
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const kda_shape ps = padded_shape(shape);
    const Pad64 L = pad64_layout(shape);
    char *w = static_cast<char *>(ws);
    const int64_t rows = (int64_t)shape->B * shape->T * shape->H;
    const int64_t nst = (int64_t)num_seqs_of(shape) * shape->H;
    cudaError_t e = cudaSuccess;
    const void *src[] = {q, k, v, g};
    const size_t dst[] = {L.q, L.k, L.v, L.g};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      if (src[i]) e = kda::pad_rows_launch(src[i], w + dst[i], rows, i == 3 ? -30.f : 0.f, cs);
    float *h0p = h0 ? reinterpret_cast<float *>(w + L.h0) : nullptr;
    float *dtp = dt_bias ? reinterpret_cast<float *>(w + L.dt) : nullptr;
    float *hTp = hT ? reinterpret_cast<float *>(w + L.dh0) : nullptr;
    if (e == cudaSuccess && h0) e = kda::pad_tiles_f32_launch(h0, h0p, nst, 64, 64, 128, 128, false, cs);
    if (e == cudaSuccess && dt_bias)
      e = kda::pad_tiles_f32_launch(dt_bias, dtp, shape->H, 1, 64, 1, 128, false, cs);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    st = kda_fwd(&ps, w + L.q, w + L.k, w + L.v, w + L.g, beta, A_log, dtp, h0p, w + L.dq, hTp,
                 w, L.inner, stream);
    if (st != KDA_OK) return st;
    e = kda::unpad_rows_launch(w + L.dq, o, rows, cs);
    if (e == cudaSuccess && hT) e = kda::pad_tiles_f32_launch(hTp, hT, nst, 64, 64, 128, 128, true, cs);
    return from_cuda(e);
  }

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  char *w = static_cast<char *>(ws);
  kda::KdaParams p;
  fill_params(shape, p);
  p.q = q;
  p.k = k;
  p.v = v;
  p.g = g;
  p.beta = beta;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.h0 = h0;
  p.hT = hT;
  p.states = w;  // packed chunk states, as kda_bwd keeps them
  p.dA_part = reinterpret_cast<float *>(w + dA_part_offset(shape));
  p.prep_mode = kda::kPrepReadout;  // the scans' operands and QE^T, scale * Mqk
  kda::TokenMaps tm{};  // left zero when there are no tokens (no kernel then reads it)
  if (!kda::encode_token_maps(p, tm)) return KDA_ERR_CUDA;
  // 1. per-chunk operands, 2. forward state scan (S_n of every chunk, hT),
  // 3. the chunk outputs
  cudaError_t e = forward_states_tc(p, shape, w, tm, cs);
  if (e == cudaSuccess) e = kda::out_tc_launch(p, p.states, o, cs);
  return from_cuda(e);
}

kda_status kda_bwd(const kda_shape *shape, const void *q, const void *k, const void *v,
                   const void *g, const void *beta, const float *A_log, const float *dt_bias,
                   const float *h0, const void *dO, const float *dh_T, void *dq, void *dk,
                   void *dv, void *dg, void *dbeta, float *dA_log, float *ddt_bias, float *dh0,
                   const void *states, void *ws, size_t ws_bytes, kda_stream_t stream) {
  return kda_bwd_timed(shape, q, k, v, g, beta, A_log, dt_bias, h0, dO, dh_T, dq, dk, dv, dg,
                       dbeta, dA_log, ddt_bias, dh0, states, ws, ws_bytes, stream, nullptr);
}

kda_status kda_bwd_timed(const kda_shape *shape, const void *q, const void *k, const void *v,
                         const void *g, const void *beta, const float *A_log,
                         const float *dt_bias, const float *h0, const void *dO,
                         const float *dh_T, void *dq, void *dk, void *dv, void *dg, void *dbeta,
                         float *dA_log, float *ddt_bias, float *dh0, const void *states,
                         void *ws, size_t ws_bytes, kda_stream_t stream, void *const *events) {
  kda_status st = check_shape(shape);
  if (st != KDA_OK) return st;
  // per-token tensors may be NULL only when there are no tokens
  const bool tokens = (int64_t)shape->B * shape->T > 0;
  if (!A_log || !dA_log) return KDA_ERR_INVALID_ARG;
  if (tokens && (!q || !k || !v || !g || !beta || !dO || !dq || !dk || !dv || !dg || !dbeta))
    return KDA_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, A_log, dt_bias, h0, dO, dh_T, dq, dk, dv, dg, dbeta,
                        dA_log, ddt_bias, dh0, states};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
  st = check_ws(shape, ws, ws_bytes);
  if (st != KDA_OK) return st;
  if (pad64_path(shape)) {
    // the 128-channel backward on padded copies, then the gradients cut back
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const kda_shape ps = padded_shape(shape);
    const Pad64 L = pad64_layout(shape);
    char *w = static_cast<char *>(ws);
    const int64_t rows = (int64_t)shape->B * shape->T * shape->H;
    const int64_t nst = (int64_t)num_seqs_of(shape) * shape->H;
    cudaError_t e = cudaSuccess;
    const void *src[] = {q, k, v, g, dO};
    const size_t dst[] = {L.q, L.k, L.v, L.g, L.dO};
    for (int i = 0; i < 5 && e == cudaSuccess; ++i)
      if (src[i]) e = kda::pad_rows_launch(src[i], w + dst[i], rows, i == 3 ? -30.f : 0.f, cs);
    float *h0p = h0 ? reinterpret_cast<float *>(w + L.h0) : nullptr;
    float *dhTp = dh_T ? reinterpret_cast<float *>(w + L.dhT) : nullptr;
    float *dh0p = dh0 ? reinterpret_cast<float *>(w + L.dh0) : nullptr;
    float *dtp = dt_bias ? reinterpret_cast<float *>(w + L.dt) : nullptr;
    float *ddtp = ddt_bias ? reinterpret_cast<float *>(w + L.ddt) : nullptr;
    void *stp = states ? w + L.states : nullptr;
    if (e == cudaSuccess && h0) e = kda::pad_tiles_f32_launch(h0, h0p, nst, 64, 64, 128, 128, false, cs);
    if (e == cudaSuccess && dh_T)
      e = kda::pad_tiles_f32_launch(dh_T, dhTp, nst, 64, 64, 128, 128, false, cs);
    if (e == cudaSuccess && dt_bias)
      e = kda::pad_tiles_f32_launch(dt_bias, dtp, shape->H, 1, 64, 1, 128, false, cs);
    if (e == cudaSuccess && states)
      e = kda::pack_states64_launch(states, stp, slots_of(shape) * shape->H, cs);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    st = kda_bwd_timed(&ps, w + L.q, w + L.k, w + L.v, w + L.g, beta, A_log, dtp, h0p, w + L.dO,
                       dhTp, w + L.dq, w + L.dk, w + L.dv, w + L.dg, dbeta, dA_log, ddtp, dh0p, stp,
                       w, L.inner, stream, events);
    if (st != KDA_OK) return st;
    void *outs[] = {dq, dk, dv, dg};
    const size_t from[] = {L.dq, L.dk, L.dv, L.dg};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      if (outs[i]) e = kda::unpad_rows_launch(w + from[i], outs[i], rows, cs);
    if (e == cudaSuccess && dh0) e = kda::pad_tiles_f32_launch(dh0p, dh0, nst, 64, 64, 128, 128, true, cs);
    if (e == cudaSuccess && ddt_bias)
      e = kda::pad_tiles_f32_launch(ddtp, ddt_bias, shape->H, 1, 64, 1, 128, true, cs);
    return from_cuda(e);
  }

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  char *w = static_cast<char *>(ws);
  const size_t sb = states_bytes(shape);
  kda::KdaParams p;
  fill_params(shape, p);
  p.q = q;
  p.k = k;
  p.v = v;
  p.g = g;
  p.beta = beta;
  p.dO = dO;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.h0 = h0;
  p.dhT = dh_T;
  p.states = states ? const_cast<void *>(states) : w;
  p.hT = nullptr;
  p.dstates = w + sb;
  p.dh0 = dh0;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dg = dg;
  p.dbeta = dbeta;
  p.dA_part = reinterpret_cast<float *>(w + dA_part_offset(shape));
  p.dA_log = dA_log;
  p.ddt_part = reinterpret_cast<float *>(w + ddt_part_offset(shape));
  p.ddt_bias = ddt_bias;
  const bool bf = shape->dtype == KDA_BF16;
  auto mark = [&](int i) {
    if (events != nullptr && events[i] != nullptr)
      cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), cs);
  };
  mark(0);
  // 1. scans: forward states (unless given) and the reverse dS scan, one launch
  const int nroles = states ? 1 : 2;
  p.role_base = states ? 1 : 0;
  cudaError_t e = cudaSuccess;
  kda::TokenMaps tm{};  // left zero when there are no tokens (no kernel then reads it)
  if (tc_state_path(shape)) {
    // TMA maps of the token-major inputs, and the per-chunk operands for the
    // tcgen05 scans and the gradient kernel
    if (!kda::encode_token_maps(p, tm)) return KDA_ERR_CUDA;
    void *prep = w + prep_offset(shape);
    p.prep = static_cast<const char *>(prep);
    // chunks whose gate passes the block factors' range are redone exactly
    // (kda_range.cu) on the tcgen05 scans' path; the per-band scans report them
    if (!legacy_scan()) p.range_flags = reinterpret_cast<int32_t *>(w + flags_offset(shape));
    e = kda::prep_tc_launch(p, tm, prep, cs);
    if (e == cudaSuccess) e = kda::range_prep_launch(p, prep, cs);
  }
  mark(1);
  if (e == cudaSuccess && tc_state_path(shape) && !legacy_scan()) {
    // the tcgen05 scans store their tiles in packed core-matrix order, the
    // layout kda_fwd_states gives the caller on this path too
    p.states_packed = 1;
    p.dstates_packed = 1;
    const int cp = cp_segments_used(shape);
    if (p.cu != nullptr && cp < 3) {
      // varlen: the scans take the sequences longest first; the order lives in
      // the dA_log partials (slots x H >= num_seqs floats), which the gradient
      // kernel overwrites only after the scans
      p.seq_order = reinterpret_cast<const int32_t *>(p.dA_part);
      e = kda::seq_order_launch(p.cu, p.num_seqs, reinterpret_cast<int32_t *>(p.dA_part), cs);
    }
    if (e == cudaSuccess && cp >= 3) {
      // few (sequence, head) chains: context-parallel scans over segments
      p.cp_segs = cp;
      p.cp_buf = reinterpret_cast<float *>(w + cp_offset(shape));
      e = kda::scan_tc_cp_launch(p, tm, p.prep, nroles, cs);
      p.cp_segs = 0;
    } else if (e == cudaSuccess) {
      e = kda::scan_tc_launch(p, tm, p.prep, nroles, cs);
    }
  } else if (e == cudaSuccess) {
    // the per-band scans write row-major tiles; caller states on the tcgen05
    // path are packed (kda_fwd_states' layout there)
    p.states_packed = states != nullptr && tc_state_path(shape) ? 1 : 0;
    const int bv = pick_band(shape, nroles);
    p.nb = shape->V / bv;
    e = kda::scan_dispatch(p, shape->K, bf, bv, nroles, cs);
  }
  if (e != cudaSuccess) return KDA_ERR_CUDA;
  mark(2);
  // 2. per-chunk gradients and the dA_log reduction
  e = kda::grads_dispatch(p, shape->K, bf, p.states, cs, events ? events[3] : nullptr,
                          tc_state_path(shape) ? &tm : nullptr);
  mark(4);
  return from_cuda(e);
}

kda_status kda_get_device_status(kda_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KDA_ERR_CUDA;
  const int words[] = {kda::scan_status_take(),     kda::prep_tc_status_take(),
                       kda::scan_tc_status_take(),  kda::grads_status_take(),
                       kda::grads_tc_status_take(), kda::out_tc_status_take(),
                       kda::range_status_take()};
  for (int v : words)
    if (v < 0) return KDA_ERR_CUDA;
  for (int v : words)
    if (v != 0) return (kda_status)v;
  return KDA_OK;
}

}  // extern "C"
