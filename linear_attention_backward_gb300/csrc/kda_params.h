// kda_params.h -- launch parameters shared by the host API and the kernels,
// and the host-side entry points of the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

struct KdaParams {
  int B, T, H, num_seqs;
  const int32_t *cu;          // device, nullable
  int nps;                    // slots per sequence (fixed length): ceil(T / 64)
  int64_t nslots;
  float scale, eps;
  const void *q, *k, *v, *g, *beta, *dO;
  const float *A_log, *h0, *dhT;
  void *states;               // [slots, H, K, V] (written by the forward scan)
  float *hT;                  // nullable
  void *dstates;              // [slots, H, K, V]
  float *dh0;                 // nullable
  void *dq, *dk, *dv, *dg, *dbeta;
  float *dA_part;             // [slots, H]
  float *dA_log;              // [H]
  int nb;                     // V bands of the scan kernels
  int role_base;              // first scan role of a launch (0 forward, 1 reverse)
};

// kda_scan.cu: forward-state scan (role 0) and reverse dS scan (role 1).
cudaError_t scan_dispatch(const KdaParams &p, int K, bool bf16, int bv, int nroles,
                          cudaStream_t st);
size_t scan_smem_bytes(int K, bool bf16, int bv);
int scan_status_take();

// kda_grads.cu: per-chunk gradients and the dA_log reduction.
// `after_grads` (nullable cudaEvent_t) is recorded between the gradient
// kernel and the dA_log reduction.
cudaError_t grads_dispatch(const KdaParams &p, int K, bool bf16, const void *states,
                           cudaStream_t st, void *after_grads = nullptr);
size_t grads_smem_bytes(int K, bool bf16);
int grads_status_take();

// kda_grads_tc.cu: the same per-chunk gradients on tcgen05 (bf16, K = V = 128).
cudaError_t grads_tc_launch(const KdaParams &p, const void *states, cudaStream_t st);
size_t grads_tc_smem_bytes();
int grads_tc_status_take();

}  // namespace kda
