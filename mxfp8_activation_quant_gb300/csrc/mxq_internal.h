// Internal launcher interface of libmxq (host side). Arguments are validated by the C ABI
// layer (api.cu) before any of these is called.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "mxq.h"

namespace mxq {

// CUDA error -> MXQ_OK / MXQ_ERR_CUDA; records the error name for mxq_last_error_string.
mxq_status from_cuda(cudaError_t e);

struct QuantizeLaunch {
  const void* x;
  int64_t M, K, ldx;
  void* q;
  int64_t ldq;
  void* sf_rowmajor;
  void* sf_packed;
  void* sf_tiled;
};
cudaError_t launch_quantize(const QuantizeLaunch& a, cudaStream_t stream);

struct RmsnormLaunch {
  const void* x;
  const void* gamma;
  float eps;
  int64_t T, H, ldx;
  void* y;
  void* yq;
  void* sf_packed;
  void* sf_rowmajor;
  void* sf_tiled;
};
cudaError_t launch_rmsnorm(const RmsnormLaunch& a, cudaStream_t stream);

// One MXFP8 GEMM of the chain, grouped over G: for group g,
//   C_g[t, f] = sum_k deq(act)[t, g*act_k_per_group + k] * deq(wt)[g*n_feat + f, k]
// over k < k_len; outputs at column g*n_feat + f of the bf16 and/or MXFP8 outputs.
struct GemmLaunch {
  const void* act;          // E4M3 [T, act_cols], row stride act_ld bytes
  const void* act_sf;       // F8_128x4 scales of act
  int64_t act_cols, act_ld;
  int64_t act_k_per_group;  // column offset between groups in act (Ka for wo_a, 0 for wo_b)
  const void* wt;           // E4M3 [G*n_feat, k_len], row stride wt_ld bytes
  const void* wt_sf;        // F8_128x4 scales of wt
  int64_t wt_ld;
  int64_t T;
  int32_t G, n_feat, k_len;
  // outputs (any of them may be null, at least one of out_bf16 / z_q)
  void* out_bf16;           // bf16 [T, G*n_feat] (row stride ldo elements)
  int64_t ldo;
  void* z_q;                // E4M3 [T, G*n_feat] (row stride G*n_feat bytes)
  void* z_sf_tiled;         // F8_128x4 scales of z (needs z_q)
  void* z_sf_packed;        // int32-packed MN-major scales of z (needs z_q)
  int32_t* status;          // optional device status word
  // Launch as a programmatic dependent of the previous kernel on the stream: the weight
  // operand (never written by that kernel) is prefetched before waiting for it to finish.
  bool pdl;
  // A programmatic dependent grid follows this one (wo_a inside o_proj_mxfp8): prefer a
  // lighter per-CTA footprint so that the dependent's CTAs can be resident alongside.
  bool has_dependent;
  // act is bf16 [T, act_cols] (row stride act_ld elements), quantized to MXFP8 inside the
  // kernel with mxfp8_quantize's rule; act_sf is unused. T <= 16 only.
  bool act_is_bf16;
  // act_sf is MXQ_SF_PACKED_I32_MN (packed[w * Mp + m], Mp = ceil(T / 4) * 4), any T.
  bool act_sf_packed;
  // Optional device workspace of at least split_workspace_bytes(), zero-filled before its first
  // use; every launch that completes leaves its flags zero. With it, the CTA-pair kernel may cut
  // the k-block iterations of its last wave and remainder into equal ranges over all pairs
  // (stream-K tail) when its cost model says that pays; without it, pairs take whole tiles.
  void* workspace;
  int64_t workspace_bytes;
};
cudaError_t launch_gemm(const GemmLaunch& a, cudaStream_t stream);
// Workspace bytes the stream-K tail needs on the current device.
int64_t split_workspace_bytes();

}  // namespace mxq
