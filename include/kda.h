/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi-Delta-Attention backward library.
 *
 * The operation.  Per sequence and head, with t the token index,
 *   q^_t = q_t / sqrt(|q_t|^2 + l2_eps), k^_t likewise      (in-library L2 norm)
 *   gk_t = -exp(A_log[h]) * softplus(g_t + dt_bias[h])        (per-channel log-decay)
 *   S_t  = (I - beta_t k^_t k^_t^T) Diag(exp(gk_t)) S_{t-1} + beta_t k^_t v_t^T
 *   o_t  = scale * S_t^T q^_t,     S_0 = h0
 * and kda_bwd returns the gradients of  sum_t <dO_t, o_t> + <dh_T, S_T>  with
 * respect to q, k, v, g, beta, A_log, dt_bias and h0.  dt_bias, the gate's
 * per-channel bias (the kernel-B guide, Part 2, B3 optimisation 7: the
 * reverse cumulative sum accumulates dA_log and ddt_bias), is optional: a
 * NULL dt_bias is a zero bias, and a NULL ddt_bias skips that gradient.
 * The work is the chunked backward described on the pages
 * "bwd-kernelB-beginner-guide-full" (Part 1: the per-chunk gradient kernel
 * B1/B2/B0/B3 and its outputs dq, dk, dv, dbeta, dg, dA_log; Part 2, B3:
 * the L2-norm backward and the reverse cumulative sum of the gate gradient)
 * and "bwd-ncu-and-optimization-playbook" (A/B table: Kernel A, the serial
 * reverse scan of the per-chunk state gradient dS, grid (N, H, VSplit)).
 * Chunk size is 64 tokens.
 *
 * Head sizes.  bf16 with K = V = 128 runs the fifth-generation tensor-core
 * kernels.  bf16 with K = V = 64 runs the same kernels on copies of the
 * inputs zero-padded to 128 channels (exact: a padded channel has q^ = k^ = 0
 * and zero value columns, so its state rows and columns stay zero and every
 * gradient term touching it vanishes; the read-out scale stays 64^-1/2); the
 * padded copies live in the workspace, and the environment variable
 * KDA_PAD64=0 selects the mma.sync kernels for such shapes instead.  fp32
 * (K = V = 64) runs mma.sync / fp32 SIMT kernels, whose products keep fp32
 * precision (the fp32 tolerance of 1e-4 rules out tf32 operands).
 *
 * Conventions for every entry point.
 *  - Tensors are DEVICE pointers, contiguous, token-major ("native [T,H,D]"
 *    layout of the kernel-B guide, Part 2, B3 optimisation 8):
 *      q, k, g, dq, dk, dg : [B, T, H, K]
 *      v, dO, dv           : [B, T, H, V]
 *      beta, dbeta         : [B, T, H]
 *      A_log, dA_log       : [H] fp32
 *      dt_bias, ddt_bias   : [H, K] fp32
 *      h0, hT, dh_T, dh0   : [N, H, K, V] fp32, N = B (fixed length) or
 *                            num_seqs (varlen)
 *    q, k, v, g, beta, dO and the gradients dq, dk, dv, dg, dbeta all have the
 *    dtype given in kda_shape (fp32 or bf16).
 *  - Varlen: cu_seqlens (DEVICE int32 [num_seqs + 1], cu_seqlens[0] == 0,
 *    non-decreasing, cu_seqlens[num_seqs] == T) packs num_seqs sequences
 *    back to back in one batch row (B must be 1).  cu_seqlens == NULL means
 *    B fixed-length sequences of length T.  The library never reads
 *    cu_seqlens on the host; kernels check it and report a bad table through
 *    the device status word (kda_get_device_status).
 *  - Chunk slots.  Per-chunk buffers (the states and the workspace) are
 *    indexed by a chunk slot, not a dense chunk count, so that no host-side
 *    scan of cu_seqlens is needed:
 *      fixed length: slot(b, j) = b * ceil(T / 64) + j
 *      varlen:       slot(s, j) = floor(cu_seqlens[s] / 64) + s + j
 *    for chunk j of sequence b / s.  kda_num_chunk_slots() gives the number
 *    of slots (varlen: floor(T / 64) + num_seqs; a few slots stay unused).
 *  - Ownership: the caller owns every buffer, including the workspace.  The
 *    library never allocates or frees memory and never synchronises the
 *    stream, except kda_get_device_status which synchronises its stream.
 *  - Errors: argument errors are returned before anything is launched.  A
 *    failed launch returns KDA_ERR_CUDA.  Errors found on the device (a bad
 *    cu_seqlens table, a gate beyond the block range on the fp32 kernels, a
 *    bounded wait that gave up) are recorded in a device status word read
 *    by kda_get_device_status; the outputs of that call are then not valid.
 *  - Bounded waits.  Every wait of a kernel on a copy or a tensor-core
 *    product polls a bounded number of times (2^24 polls for copies, 2^20
 *    for products).  A CTA whose wait gives up records KDA_ERR_TIMEOUT,
 *    issues no further product and writes no further result, waits once
 *    more (2^16 polls) for what it still has in flight, releases its Tensor
 *    Memory and exits; the context stays usable.  Test hook: the environment
 *    variable KDA_TEST_STARVE_WAITS, a list of kernel names (prep, scan,
 *    grads, out), makes those kernels arm their first load barrier without
 *    issuing its copies and caps every wait of the call at 4096 polls, so
 *    that the timeout path can be exercised without a fault.
 *  - Streams: all work of one call is queued on `stream` in order.  Calls
 *    on different streams that share output or workspace buffers race.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kda_stream_t; /* == cudaStream_t; NULL = default stream */

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* null pointer, bad shape, misaligned pointer */
  KDA_ERR_UNSUPPORTED = 2, /* valid but not built: K, V not in {64, 128}, K != V */
  KDA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than kda_workspace_bytes */
  KDA_ERR_CUDA = 4,        /* a CUDA launch or runtime call failed */
  KDA_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up */
  KDA_ERR_DEVICE_ARG = 6,  /* the device found a bad cu_seqlens table */
  KDA_ERR_TOO_LARGE = 7,   /* kda_bwd_noalloc: problem needs more than its fixed scratch */
  KDA_ERR_GATE_RANGE = 8   /* fp32 inputs and the comparison switches (KDA_SCAN_LEGACY,
                              KDA_GRADS_MMA_SYNC, KDA_PAD64=0) only: the device found a
                              channel whose gate log-decay over the 7 or 8 tokens on either
                              side of a 16-row block's reference row exceeds 88 nats, where
                              the block factors e^x leave the fp32 range, or (kda_bwd) a
                              chunk in which every channel decays by more than 5 nats per
                              token (6 for bf16), where the block-factored dg misses the
                              tolerance; the outputs of that call are not valid.  bf16
                              inputs take such chunks through exact kernels (one
                              exponential per row pair) instead */
} kda_status;

typedef enum { KDA_FP32 = 0, KDA_BF16 = 1 } kda_dtype;

typedef struct {
  int B, T, H, K, V;          /* K == V, both 64 or 128 */
  int chunk;                  /* must be 64 */
  int num_seqs;               /* varlen: number of packed sequences; else 0 */
  const int32_t *cu_seqlens;  /* varlen: DEVICE pointer [num_seqs + 1]; else NULL */
  float scale;                /* read-out scale; <= 0 selects K^-1/2 */
  float l2_eps;               /* added to |x|^2 in the L2 norm; < 0 selects 1e-6 */
  kda_dtype dtype;            /* dtype of q, k, v, g, beta, dO and gradients */
} kda_shape;

/* Number of chunk slots (see "Chunk slots" above); 0 on a bad shape. */
int64_t kda_num_chunk_slots(const kda_shape *shape);

/* Bytes of workspace kda_bwd needs: the per-chunk states (dtype of the
 * shape, [slots, H, K, V]) unless the caller passes them, the per-chunk
 * state gradients dS (same size), per-chunk dA_log and ddt_bias partials
 * ([slots, H] and [slots, H, K] fp32) and, for bf16
 * with K = V = 128, the per-chunk operand blocks of the tensor-core scans
 * (107008 bytes per slot and head), where kda_scan_segments() > 0 the
 * segment boundary tiles of the context-parallel scans, and a 4-byte flag
 * per slot and head (the chunks whose gate passes the block factors' range,
 * which exact kernels then redo).  For bf16 with
 * K = V = 64 it is the workspace of the 128-channel shape plus the padded
 * copies of the inputs, gradients, h0 / dh_T / dh0, the gate bias and given
 * states.  Returns 0 on a bad shape. */
size_t kda_workspace_bytes(const kda_shape *shape);
/* Byte offset inside the workspace of the per-chunk state gradients
 * dS_{n+1} (the adjoint of the state at the END of chunk n), [slots, H]
 * tiles of K x V in the shape's dtype.  For bf16 with K = V = 128 each tile
 * is in packed core-matrix order -- element (k, v) at element offset
 * ((k / 8) * (V / 8) + v / 8) * 64 + (k % 8) * 8 + v % 8 -- and so are the
 * states kda_bwd recomputes at the start of the workspace; otherwise tiles
 * are row-major.  For bf16 with K = V = 64 (padded path) the tiles are the
 * padded 128 x 128 ones, in packed order, with the values in the 64 x 64
 * corner.  Exposed so that tests can check the scans on their own. */
size_t kda_workspace_dstates_offset(const kda_shape *shape);
/* Segments per sequence of the context-parallel state scans that kda_bwd and
 * kda_fwd run for this shape; 0 means one scan chain per (sequence, head,
 * role).  The serial chunk scans are the part of the backward that does not
 * fill the GPU when B * H is small (with a single sequence the reverse scan,
 * Kernel A of "bwd-ncu-and-optimization-playbook", A/B table, takes about
 * half of the backward there; its split-V remedy, ibid. §3.5, adds CTAs but
 * shortens no chain).  With A_n = diag(e^gT) - kr^T W the chunk
 * updates are affine (S_{n+1} = A_n S_n + kr^T U0, dS_n = A_n^T dS_{n+1} +
 * QE^T dO), so each sequence's chunks split into P segments: every segment is
 * scanned from zero, the inner segments' transfer products A_{b-1}..A_a are
 * formed, a combine kernel chains the segment boundaries, and the segments
 * are scanned again from the true boundaries (two more launches than the
 * whole-sequence scans).  Used for bf16 K = V = 128 shapes with 2 N H < 152
 * (N sequences; 152 is the SM count) and at least 4 P chunks per sequence
 * (for varlen, on average: T / 64 / N, since the host never reads
 * cu_seqlens; shorter sequences get shorter or empty segments): the most
 * segments, 3 to 8, whose first-pass chains ((3 P - 4) N H) fit one per SM;
 * if not even 3 do and 4 N H <= 152, the most whose chains fit two per SM
 * (the scan kernel's residency).  The workspace then ends with (3 P - 4)
 * fp32 K x V tiles per (sequence, head).
 * The environment variable KDA_SCAN_CP=0 turns this off per call, and
 * KDA_SCAN_CP=n (3 <= n <= the value without it) takes n segments.
 * Returns 0 on a bad shape. */
int kda_scan_segments(const kda_shape *shape);
/* Forward chunk-state recompute (the "all_states" operand of kernel B2 in
 * "bwd-kernelB-beginner-guide-full", Part 2, B2 optimisation 4).
 *   states : OUT [slots, H, K, V], dtype of the shape: S at the start of
 *            every chunk (S_0 = h0), bf16 rounded to nearest even.  For bf16
 *            with K = V = 128 each K x V tile is in packed core-matrix order
 *            (element (k, v) at element offset ((k / 8) * (V / 8) + v / 8) *
 *            64 + (k % 8) * 8 + v % 8: 8 x 8 blocks of 128 bytes, blocks along
 *            V first), the order in which the scans store them and the
 *            gradient kernel reads them; otherwise row-major.  kda_bwd takes
 *            them in the same layout.
 *   h0     : nullable (zero initial state), fp32 [N, H, K, V].
 *   hT     : nullable OUT fp32 [N, H, K, V]: the final state of each sequence.
 *   ws     : bf16: DEVICE workspace of at least kda_workspace_bytes(shape)
 *            bytes, 256-byte aligned (the layout kda_bwd uses; the per-chunk
 *            operand blocks of the chunk-parallel prep live there).
 *            Required for K = V = 128; for K = V = 64 it selects the
 *            tensor-core path below.  fp32 needs none (ws may be NULL).
 * bf16 with K = V = 128 runs the chunk-parallel prep (its pair blocks read
 * q; it writes only the scans' operands, not the read-out's or the gradient
 * kernel's) and the forward tcgen05 state scan, context-parallel where
 * kda_scan_segments() > 0; q is then required.  bf16 K = V = 64 with a
 * workspace and q runs the same kernels on zero-padded 128-channel copies and
 * returns the states' 64 x 64 corners row-major (kda_bwd packs them back into
 * the padded layout).  fp32, and bf16 K = V = 64 without a workspace, run the
 * per-band scan and ignore q. */
kda_status kda_fwd_states(const kda_shape *shape, const void *q, const void *k,
                          const void *v, const void *g, const void *beta,
                          const float *A_log, const float *dt_bias, const float *h0,
                          void *states, float *hT, void *ws, size_t ws_bytes,
                          kda_stream_t stream);

/* Forward pass: the read-out o_t = scale * S_t^T q^_t of every token and the
 * final states ("bwd-kernelB-beginner-guide-full", Part 1: the chunked KDA
 * recurrence whose backward kda_bwd computes), on the same per-chunk operands
 * as kda_bwd: with U = U0 - W S_n the corrected values of chunk n and
 * QE = scale (qd - Mqk W),  o = QE S_n + (scale Mqk) U0  row by row.
 * bf16 only (K = V = 64 on zero-padded copies); KDA_ERR_UNSUPPORTED for fp32.
 *   o      : OUT [B, T, H, V] bf16, overwritten (rows of every sequence).
 *   h0     : nullable (zero initial state), fp32 [N, H, K, V].
 *   hT     : nullable OUT fp32 [N, H, K, V]: the final state of each sequence.
 *   ws     : DEVICE workspace of at least kda_workspace_bytes(shape) bytes,
 *            256-byte aligned (the layout kda_bwd uses; its dS part is unused).
 * q, k, v, g, beta and A_log are required. */
kda_status kda_fwd(const kda_shape *shape, const void *q, const void *k, const void *v,
                   const void *g, const void *beta, const float *A_log,
                   const float *dt_bias, const float *h0, void *o, float *hT, void *ws,
                   size_t ws_bytes, kda_stream_t stream);

/* Backward pass.
 *   dh_T   : nullable (zero), fp32 [N, H, K, V].
 *   dq, dk, dv, dg, dbeta : OUT, overwritten, dtype of the shape.
 *   dA_log : OUT fp32 [H], overwritten (summed over sequences and tokens).
 *   ddt_bias : nullable OUT fp32 [H, K], overwritten (summed likewise).
 *   dh0    : nullable OUT fp32 [N, H, K, V].
 *   states : nullable; the output of kda_fwd_states for the same inputs, in
 *            its layout (packed core-matrix tiles for bf16, K = V = 128).
 *            NULL recomputes them inside the workspace.
 *   ws     : DEVICE workspace of at least kda_workspace_bytes(shape) bytes,
 *            256-byte aligned.  Its content on entry is ignored.
 * q, k, v, g, beta, A_log and dO are required. */
kda_status kda_bwd(const kda_shape *shape, const void *q, const void *k,
                   const void *v, const void *g, const void *beta,
                   const float *A_log, const float *dt_bias, const float *h0,
                   const void *dO, const float *dh_T, void *dq, void *dk, void *dv,
                   void *dg, void *dbeta, float *dA_log, float *ddt_bias, float *dh0,
                   const void *states, void *ws, size_t ws_bytes, kda_stream_t stream);

/* kda_bwd with phase timing: `events` (nullable) points at 5 cudaEvent_t
 * created by the caller (timing enabled).  They are recorded on `stream`
 * at the start of the call, after the per-chunk prep (bf16, K = V = 128;
 * otherwise right after the first), after the chunk scans (forward-state
 * recompute and reverse dS scan), after the per-chunk gradient kernel and
 * at the end (after the dA_log and ddt_bias reductions).  Otherwise identical
 * to kda_bwd. */
kda_status kda_bwd_timed(const kda_shape *shape, const void *q, const void *k,
                         const void *v, const void *g, const void *beta,
                         const float *A_log, const float *dt_bias, const float *h0,
                         const void *dO, const float *dh_T, void *dq, void *dk, void *dv,
                         void *dg, void *dbeta, float *dA_log, float *ddt_bias, float *dh0,
                         const void *states, void *ws, size_t ws_bytes, kda_stream_t stream,
                         void *const *events);

/* Backward pass for callers that cannot allocate device memory (no
 * counterpart on the pages; a service of this library).  Some callers have
 * no way to hand kda_bwd a workspace: code running inside a device-memory
 * allocator or pool that owns every device allocation, processes that may
 * only use memory reserved up front, or plugin hosts that expose no
 * allocation API.  This entry point takes the same inputs and outputs as
 * kda_bwd (states always recomputed) but keeps its scratch -- the per-chunk
 * states, state gradients and dA_log / ddt_bias partials -- in a fixed array of
 * kda_noalloc_scratch_bytes() bytes (64 MiB) compiled into the library.
 * That array exists once per GPU that loads the library and stays allocated
 * until the process exits.
 *  - Size limit: problems whose kda_workspace_bytes() exceeds the array are
 *    rejected with KDA_ERR_TOO_LARGE before anything is launched (64 MiB
 *    holds about 400 chunk-heads of 64 tokens at K = V = 128, bf16).
 *  - When the array is reserved: it belongs to the library's device image
 *    and is reserved when the CUDA runtime loads the module holding it --
 *    under lazy module loading (the default since CUDA 12.2) during the
 *    first kda_bwd_noalloc call on each device, under eager loading
 *    (CUDA_MODULE_LOADING=EAGER) when the context is created, for every
 *    process that loads the library.  Make one warm-up call per device
 *    outside any allocator callback or restricted region, and before
 *    capturing any stream; later calls reserve nothing.
 *  - Each call looks the array's device address up (cudaGetSymbolAddress,
 *    on the calling thread's current device); nothing is cached across
 *    calls, so a context that was torn down and re-created is handled.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Every call on a device shares the same array: calls whose work
 *    overlaps on the GPU (different streams, or different host threads)
 *    race on it and must be serialised by the caller.  The array needs no
 *    initial content; each call writes every part it reads. */
kda_status kda_bwd_noalloc(const kda_shape *shape, const void *q, const void *k,
                           const void *v, const void *g, const void *beta,
                           const float *A_log, const float *dt_bias, const float *h0,
                           const void *dO, const float *dh_T, void *dq, void *dk, void *dv,
                           void *dg, void *dbeta, float *dA_log, float *ddt_bias,
                           float *dh0, kda_stream_t stream);

/* Capacity in bytes of kda_bwd_noalloc's fixed scratch array. */
size_t kda_noalloc_scratch_bytes(void);

/* Device self-test of the fifth-generation tensor-core path (no counterpart
 * on the pages): computes D = A B^T for one M = 128 tile through shared-memory
 * descriptors, Tensor Memory and tcgen05 loads, with A ([128][K] bf16,
 * row-major, device) and B ([N][K] bf16, row-major, device) staged in K-major
 * (0) or MN-major (1) core-matrix layout; D is [128][N] fp32 (device).
 * N in {32, 64, 128}, K a multiple of 16 up to 128.  layout: 0 = core
 * matrices packed (128-byte stride), 1 = padded core layout (144-byte stride,
 * the one the kernels use for tiles their threads write), 2 = 128-byte
 * swizzled layout (8-row x 128-byte atoms, 16-byte chunk j of row r at
 * j ^ (r % 8): what a TMA copy with 128-byte swizzling writes; K a multiple
 * of 64, and N >= 64 when B is MN-major).  Other values are rejected
 * (KDA_ERR_INVALID_ARG). */
kda_status kda_selftest_umma(const void *A, const void *B, float *D, int N, int K, int a_mn,
                             int b_mn, int layout, kda_stream_t stream);

/* Synchronises `stream`, then returns and clears the device status word of
 * the current device (KDA_OK, KDA_ERR_DEVICE_ARG, KDA_ERR_TIMEOUT or
 * KDA_ERR_GATE_RANGE: the first error any kernel raised since the last read), or
 * KDA_ERR_CUDA if the synchronisation itself reported an error. */
kda_status kda_get_device_status(kda_stream_t stream);

/* Host-side check of a cu_seqlens table the caller holds on the host:
 * KDA_OK or KDA_ERR_INVALID_ARG. */
kda_status kda_check_cu_seqlens_host(const int32_t *cu_seqlens, int num_seqs,
                                     int total_T);

/* Static description of a status code. */
const char *kda_status_str(kda_status status);

/* Version of this ABI (increments on any signature or workspace-layout change). */
int kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
