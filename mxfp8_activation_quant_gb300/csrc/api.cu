// C ABI of libmxq: argument checks on the host, then the kernel launches of mxq_internal.h.
// The operations and their sources are documented in include/mxq.h.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "mxq.h"
#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace {
thread_local char g_last_error[128] = "no error";

// An mbarrier that nothing will ever arrive on, waited on with the pipelines' own bounded wait
// (a shorter limit): the wait runs out and the timeout is reported the way every kernel reports
// it. Nothing faults and nothing hangs.
__global__ void selftest_wait_kernel(uint64_t limit_ns, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = mxq::smem_u32(&bar);
  if (threadIdx.x == 0) {
    mxq::mbar_init(b, 1);
    mxq::fence_mbar_init();
    if (!mxq::mbar_wait_limit(b, 0, limit_ns) && status != nullptr) atomicCAS(status, 0, MXQ_ERR_TIMEOUT);
  }
}

// Holds an SM for hold_ns: a CTA whose shared memory leaves no room for a GEMM CTA of this
// library beside it, one thread watching the clock (the wait always ends).
constexpr int kHoldSmemBytes = 160 * 1024;
__global__ void selftest_hold_kernel(uint64_t hold_ns) {
  extern __shared__ uint8_t hold_smem[];
  if (threadIdx.x == 0) {
    const uint64_t t0 = mxq::globaltimer_ns();
    while (mxq::globaltimer_ns() - t0 < hold_ns) __nanosleep(2000);
    hold_smem[0] = 0;
  }
}
}  // namespace

mxq_status mxq::from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MXQ_OK;
  std::strncpy(g_last_error, cudaGetErrorName(e), sizeof(g_last_error) - 1);
  g_last_error[sizeof(g_last_error) - 1] = '\0';
  return MXQ_ERR_CUDA;
}

namespace {

using mxq::from_cuda;

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// An MXFP8 GEMM operand: [rows, cols] E4M3 with F8_128x4 scales.
mxq_status check_operand(const mxq_mx_tensor* t, int64_t rows, int64_t cols) {
  if (t == nullptr || t->data == nullptr || t->sf == nullptr) return MXQ_ERR_INVALID_ARG;
  if (t->sf_layout != MXQ_SF_TILED_128X4) return MXQ_ERR_LAYOUT;
  if (t->rows != rows || t->cols != cols || t->ld < cols) return MXQ_ERR_UNSUPPORTED_SHAPE;
  if (!al16(t->data) || !al16(t->sf) || (t->ld % 16) != 0) return MXQ_ERR_MISALIGNED;
  if (t->ld >= (int64_t(1) << 40) || rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31))
    return MXQ_ERR_UNSUPPORTED_SHAPE;
  return MXQ_OK;
}

}  // namespace

extern "C" {

int mxq_abi_version(void) { return MXQ_ABI_VERSION; }

const char* mxq_status_string(mxq_status s) {
  switch (s) {
    case MXQ_OK: return "MXQ_OK";
    case MXQ_ERR_INVALID_ARG: return "MXQ_ERR_INVALID_ARG";
    case MXQ_ERR_UNSUPPORTED_SHAPE: return "MXQ_ERR_UNSUPPORTED_SHAPE";
    case MXQ_ERR_MISALIGNED: return "MXQ_ERR_MISALIGNED";
    case MXQ_ERR_LAYOUT: return "MXQ_ERR_LAYOUT";
    case MXQ_ERR_CUDA: return "MXQ_ERR_CUDA";
    case MXQ_ERR_TIMEOUT: return "MXQ_ERR_TIMEOUT";
  }
  return "MXQ_UNKNOWN_STATUS";
}

const char* mxq_last_error_string(void) { return g_last_error; }

size_t mxq_sf_bytes(int32_t layout, int64_t M, int64_t K) {
  if (M <= 0 || K <= 0 || K % 32 != 0) return 0;
  const int64_t Kg = K / 32;
  switch (layout) {
    case MXQ_SF_ROWMAJOR_U8: return static_cast<size_t>(M * Kg);
    case MXQ_SF_PACKED_I32_MN:
      if (K % 128 != 0) return 0;
      return static_cast<size_t>((Kg / 4) * cdiv(M, 4) * 4 * 4);
    case MXQ_SF_TILED_128X4: return static_cast<size_t>(cdiv(M, 128) * 128 * cdiv(Kg, 4) * 4);
    default: return 0;
  }
}

size_t mxq_status_bytes(void) { return 16; }

mxq_status mxq_check_status(const void* status, void* stream) {
  mxq_status st = from_cuda(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  if (st != MXQ_OK || status == nullptr) return st;
  int32_t code = 0;
  st = from_cuda(cudaMemcpy(&code, status, sizeof(code), cudaMemcpyDeviceToHost));
  if (st != MXQ_OK) return st;
  return code == 0 ? MXQ_OK : MXQ_ERR_TIMEOUT;
}

mxq_status mxfp8_quantize(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, void* q_e4m3, int64_t ldq,
                          void* sf_rowmajor, void* sf_packed_i32, void* sf_128x4, void* stream) {
  if (x_bf16 == nullptr || q_e4m3 == nullptr) return MXQ_ERR_INVALID_ARG;
  if (sf_rowmajor == nullptr && sf_packed_i32 == nullptr && sf_128x4 == nullptr) return MXQ_ERR_INVALID_ARG;
  if (M <= 0 || K <= 0) return MXQ_ERR_INVALID_ARG;
  if (K % 32 != 0 || ldx < K || ldq < K) return MXQ_ERR_UNSUPPORTED_SHAPE;
  if (sf_packed_i32 != nullptr && K % 128 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
  if (M >= (int64_t(1) << 31) || M * K >= (int64_t(1) << 40)) return MXQ_ERR_UNSUPPORTED_SHAPE;
  if (!al16(x_bf16) || !al16(q_e4m3) || !al16(sf_rowmajor) || !al16(sf_packed_i32) || !al16(sf_128x4))
    return MXQ_ERR_MISALIGNED;
  if ((ldx * 2) % 16 != 0 || ldq % 16 != 0) return MXQ_ERR_MISALIGNED;
  mxq::QuantizeLaunch l{x_bf16, M, K, ldx, q_e4m3, ldq, sf_rowmajor, sf_packed_i32, sf_128x4};
  return from_cuda(mxq::launch_quantize(l, static_cast<cudaStream_t>(stream)));
}

mxq_status rmsnorm_dual_out(const void* x_bf16, const void* gamma_bf16, float eps, int64_t T, int64_t H, int64_t ldx,
                            void* y_bf16, void* y_q, void* y_sf_packed_i32, void* y_sf_rowmajor, void* y_sf_128x4,
                            void* stream) {
  if (x_bf16 == nullptr || gamma_bf16 == nullptr || y_bf16 == nullptr || y_q == nullptr) return MXQ_ERR_INVALID_ARG;
  if (y_sf_packed_i32 == nullptr && y_sf_rowmajor == nullptr && y_sf_128x4 == nullptr) return MXQ_ERR_INVALID_ARG;
  if (T <= 0 || H <= 0 || !(eps >= 0.0f)) return MXQ_ERR_INVALID_ARG;
  if (H % 32 != 0 || H > 16384 || ldx < H) return MXQ_ERR_UNSUPPORTED_SHAPE;
  if (y_sf_packed_i32 != nullptr && H % 128 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
  if (T >= (int64_t(1) << 31)) return MXQ_ERR_UNSUPPORTED_SHAPE;
  if (!al16(x_bf16) || !al16(gamma_bf16) || !al16(y_bf16) || !al16(y_q) || !al16(y_sf_packed_i32) ||
      !al16(y_sf_rowmajor) || !al16(y_sf_128x4))
    return MXQ_ERR_MISALIGNED;
  if ((ldx * 2) % 16 != 0) return MXQ_ERR_MISALIGNED;
  mxq::RmsnormLaunch l{x_bf16, gamma_bf16, eps, T, H, ldx, y_bf16, y_q, y_sf_packed_i32, y_sf_rowmajor, y_sf_128x4};
  return from_cuda(mxq::launch_rmsnorm(l, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// optional split workspace: NULL, or 16-byte aligned and at least mxq_workspace_bytes()
mxq_status check_workspace(const void* ws, int64_t bytes) {
  if (ws == nullptr) return MXQ_OK;
  if (!al16(ws)) return MXQ_ERR_MISALIGNED;
  return bytes >= mxq::split_workspace_bytes() ? MXQ_OK : MXQ_ERR_INVALID_ARG;
}

mxq_status wo_a_impl(const mxq_mx_tensor* o, const mxq_mx_tensor* wa, int64_t T, int32_t G, int32_t Na, int32_t Ka,
                     void* z_q, void* z_sf_128x4, void* z_sf_packed_i32, void* z_bf16, void* ws, int64_t ws_bytes,
                     void* status, void* stream, bool has_dependent) {
  if (T <= 0 || G <= 0 || Na <= 0 || Ka <= 0) return MXQ_ERR_INVALID_ARG;
  if ((z_q == nullptr) != (z_sf_128x4 == nullptr)) return MXQ_ERR_INVALID_ARG;
  if (z_q == nullptr && z_bf16 == nullptr) return MXQ_ERR_INVALID_ARG;
  if (z_sf_packed_i32 != nullptr && z_q == nullptr) return MXQ_ERR_INVALID_ARG;
  if (Na % 128 != 0 || Ka % 128 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
  if (T >= (int64_t(1) << 31) || static_cast<int64_t>(G) * Ka >= (int64_t(1) << 31) ||
      static_cast<int64_t>(G) * Na >= (int64_t(1) << 31))
    return MXQ_ERR_UNSUPPORTED_SHAPE;
  mxq_status st = check_operand(o, T, static_cast<int64_t>(G) * Ka);
  if (st != MXQ_OK) return st;
  if ((st = check_operand(wa, static_cast<int64_t>(G) * Na, Ka)) != MXQ_OK) return st;
  if (!al16(z_q) || !al16(z_sf_128x4) || !al16(z_sf_packed_i32) || !al16(z_bf16) || !al16(status))
    return MXQ_ERR_MISALIGNED;
  if ((st = check_workspace(ws, ws_bytes)) != MXQ_OK) return st;
  mxq::GemmLaunch l = {};
  l.workspace = ws;
  l.workspace_bytes = ws_bytes;
  l.act = o->data;
  l.act_sf = o->sf;
  l.act_cols = o->cols;
  l.act_ld = o->ld;
  l.act_k_per_group = Ka;
  l.wt = wa->data;
  l.wt_sf = wa->sf;
  l.wt_ld = wa->ld;
  l.T = T;
  l.G = G;
  l.n_feat = Na;
  l.k_len = Ka;
  l.out_bf16 = z_bf16;
  l.ldo = static_cast<int64_t>(G) * Na;
  l.z_q = z_q;
  l.z_sf_tiled = z_sf_128x4;
  l.z_sf_packed = z_sf_packed_i32;
  l.status = static_cast<int32_t*>(status);
  l.has_dependent = has_dependent;
  return from_cuda(mxq::launch_gemm(l, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int64_t mxq_workspace_bytes(void) { return mxq::split_workspace_bytes(); }

mxq_status wo_a_einsum_mxfp8(const mxq_mx_tensor* o, const mxq_mx_tensor* wa, int64_t T, int32_t G, int32_t Na,
                             int32_t Ka, void* z_q, void* z_sf_128x4, void* z_sf_packed_i32, void* z_bf16,
                             void* workspace, int64_t workspace_bytes, void* status, void* stream) {
  return wo_a_impl(o, wa, T, G, Na, Ka, z_q, z_sf_128x4, z_sf_packed_i32, z_bf16, workspace, workspace_bytes, status,
                   stream, false);
}

}  // extern "C"

namespace {

// wo_b launch shared by gemm_mxfp8_bf16 and o_proj_mxfp8. `pdl` makes it a programmatic
// dependent of the previous kernel on the stream; only o_proj_mxfp8 sets it, because only
// there is that kernel known (its own wo_a, which never writes the weights wo_b prefetches).
mxq_status gemm_impl(const mxq_mx_tensor* a, const mxq_mx_tensor* b, int64_t M, int64_t N, int64_t K, void* out_bf16,
                     int64_t ldo, void* ws, int64_t ws_bytes, void* status, void* stream, bool pdl) {
  if (M <= 0 || N <= 0 || K <= 0 || out_bf16 == nullptr) return MXQ_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0 || ldo < N) return MXQ_ERR_UNSUPPORTED_SHAPE;
  if (N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return MXQ_ERR_UNSUPPORTED_SHAPE;
  // the activation may carry int32-packed MN-major scales
  const bool a_packed = a != nullptr && a->sf_layout == MXQ_SF_PACKED_I32_MN;
  mxq_status st = MXQ_OK;
  if (a_packed) {
    if (a->data == nullptr || a->sf == nullptr) return MXQ_ERR_INVALID_ARG;
    if (K % 128 != 0 || a->rows != M || a->cols != K || a->ld < K || M >= (int64_t(1) << 31))
      return MXQ_ERR_UNSUPPORTED_SHAPE;
    if (!al16(a->data) || !al16(a->sf) || (a->ld % 16) != 0) return MXQ_ERR_MISALIGNED;
  } else if ((st = check_operand(a, M, K)) != MXQ_OK) {
    return st;
  }
  if ((st = check_operand(b, N, K)) != MXQ_OK) return st;
  if (!al16(out_bf16) || !al16(status) || (ldo * 2) % 16 != 0) return MXQ_ERR_MISALIGNED;
  if ((st = check_workspace(ws, ws_bytes)) != MXQ_OK) return st;
  mxq::GemmLaunch l = {};
  l.workspace = ws;
  l.workspace_bytes = ws_bytes;
  l.act = a->data;
  l.act_sf = a->sf;
  l.act_cols = a->cols;
  l.act_ld = a->ld;
  l.act_k_per_group = 0;
  l.wt = b->data;
  l.wt_sf = b->sf;
  l.wt_ld = b->ld;
  l.T = M;
  l.G = 1;
  l.n_feat = static_cast<int32_t>(N);
  l.k_len = static_cast<int32_t>(K);
  l.out_bf16 = out_bf16;
  l.ldo = ldo;
  l.status = static_cast<int32_t*>(status);
  l.pdl = pdl;
  l.act_sf_packed = a_packed;
  return from_cuda(mxq::launch_gemm(l, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

mxq_status gemm_mxfp8_bf16(const mxq_mx_tensor* a, const mxq_mx_tensor* b, int64_t M, int64_t N, int64_t K,
                           void* out_bf16, int64_t ldo, void* workspace, int64_t workspace_bytes, void* status,
                           void* stream) {
  return gemm_impl(a, b, M, N, K, out_bf16, ldo, workspace, workspace_bytes, status, stream, false);
}

mxq_status o_proj_mxfp8(const mxq_mx_tensor* o, const mxq_mx_tensor* wa, const mxq_mx_tensor* wb, int64_t T,
                        int32_t G, int32_t Na, int32_t Ka, int32_t Nb, void* z_q, void* z_sf_128x4,
                        void* z_sf_packed_i32, void* z_bf16, void* out_bf16, void* workspace, int64_t workspace_bytes,
                        void* status, void* stream) {
  if (z_q == nullptr || z_sf_128x4 == nullptr || out_bf16 == nullptr) return MXQ_ERR_INVALID_ARG;
  if (Nb <= 0 || G <= 0 || Na <= 0) return MXQ_ERR_INVALID_ARG;
  if (Nb % 128 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
  const int64_t Kb = static_cast<int64_t>(G) * Na;
  mxq_status st = check_operand(wb, Nb, Kb);
  if (st != MXQ_OK) return st;
  if (!al16(out_bf16)) return MXQ_ERR_MISALIGNED;
  if ((st = check_workspace(workspace, workspace_bytes)) != MXQ_OK) return st;
  // The workspace serves wo_b only. wo_b is a programmatic dependent of wo_a and its epilogue
  // warps take split-tail tickets before wo_a has finished, so the two must not share the flags
  // and tickets; wo_a gains nothing from the split anyway (a tile of 32 k-blocks never pays for
  // it, and with more k-blocks measured slower).
  st = wo_a_impl(o, wa, T, G, Na, Ka, z_q, z_sf_128x4, z_sf_packed_i32, z_bf16, nullptr, 0, status, stream, true);
  if (st != MXQ_OK) return st;
  const mxq_mx_tensor z = {z_q, z_sf_128x4, MXQ_SF_TILED_128X4, T, Kb, Kb};
  return gemm_impl(&z, wb, T, Nb, Kb, out_bf16, Nb, workspace, workspace_bytes, status, stream, true);
}

mxq_status o_proj_mxfp8_from_bf16(const void* o_bf16, int64_t ld_o, const mxq_mx_tensor* wa, const mxq_mx_tensor* wb,
                                  int64_t T, int32_t G, int32_t Na, int32_t Ka, int32_t Nb, void* z_q,
                                  void* z_sf_128x4, void* z_sf_packed_i32, void* z_bf16, void* out_bf16,
                                  void* workspace, int64_t workspace_bytes, void* status, void* stream) {
  if (o_bf16 == nullptr || z_q == nullptr || z_sf_128x4 == nullptr || out_bf16 == nullptr) return MXQ_ERR_INVALID_ARG;
  if (T <= 0 || G <= 0 || Na <= 0 || Ka <= 0 || Nb <= 0) return MXQ_ERR_INVALID_ARG;
  if (Na % 128 != 0 || Ka % 128 != 0 || Nb % 128 != 0 || T >= (int64_t(1) << 31)) return MXQ_ERR_UNSUPPORTED_SHAPE;
  const int64_t Ko = static_cast<int64_t>(G) * Ka, Kb = static_cast<int64_t>(G) * Na;
  if (ld_o < Ko || Ko >= (int64_t(1) << 31) || Kb >= (int64_t(1) << 31)) return MXQ_ERR_UNSUPPORTED_SHAPE;
  mxq_status st = check_operand(wa, Kb, Ka);
  if (st != MXQ_OK) return st;
  if ((st = check_operand(wb, Nb, Kb)) != MXQ_OK) return st;
  if (!al16(o_bf16) || (ld_o * 2) % 16 != 0 || !al16(z_q) || !al16(z_sf_128x4) || !al16(z_sf_packed_i32) ||
      !al16(z_bf16) || !al16(out_bf16) || !al16(status))
    return MXQ_ERR_MISALIGNED;
  if ((st = check_workspace(workspace, workspace_bytes)) != MXQ_OK) return st;
  mxq::GemmLaunch l = {};
  l.act = o_bf16;
  l.act_cols = Ko;
  l.act_ld = ld_o;
  l.act_k_per_group = Ka;
  l.act_is_bf16 = true;
  l.wt = wa->data;
  l.wt_sf = wa->sf;
  l.wt_ld = wa->ld;
  l.T = T;
  l.G = G;
  l.n_feat = Na;
  l.k_len = Ka;
  l.out_bf16 = z_bf16;
  l.ldo = Kb;
  l.z_q = z_q;
  l.z_sf_tiled = z_sf_128x4;
  l.z_sf_packed = z_sf_packed_i32;
  l.status = static_cast<int32_t*>(status);
  l.has_dependent = true;
  st = from_cuda(mxq::launch_gemm(l, static_cast<cudaStream_t>(stream)));
  if (st != MXQ_OK) return st;
  const mxq_mx_tensor z = {z_q, z_sf_128x4, MXQ_SF_TILED_128X4, T, Kb, Kb};
  return gemm_impl(&z, wb, T, Nb, Kb, out_bf16, Nb, workspace, workspace_bytes, status, stream, true);
}

mxq_status mxq_selftest_wait_timeout(int64_t limit_us, void* status, void* stream) {
  if (status == nullptr || limit_us < 1 || limit_us > 1000000) return MXQ_ERR_INVALID_ARG;
  if (!al16(status)) return MXQ_ERR_MISALIGNED;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(limit_us) * 1000u,
                                                                      static_cast<int32_t*>(status));
  return from_cuda(cudaGetLastError());
}

mxq_status mxq_selftest_hold_sms(int64_t sm_pairs, int64_t hold_us, void* stream) {
  int dev = 0, sms = 0;
  mxq_status st = from_cuda(cudaGetDevice(&dev));
  if (st == MXQ_OK) st = from_cuda(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  if (st != MXQ_OK) return st;
  if (sm_pairs < 1 || sm_pairs > sms / 2 || hold_us < 1 || hold_us > 2000000) return MXQ_ERR_INVALID_ARG;
  static const cudaError_t attr =
      cudaFuncSetAttribute(selftest_hold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kHoldSmemBytes);
  if (attr != cudaSuccess) return from_cuda(attr);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * sm_pairs), 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.dynamicSmemBytes = kHoldSmemBytes;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;  // whole SM pairs, as the CTA-pair GEMM uses them
  a[0].val.clusterDim.x = 2;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  return from_cuda(cudaLaunchKernelEx(&cfg, selftest_hold_kernel, static_cast<uint64_t>(hold_us) * 1000u));
}

}  // extern "C"
