// o_proj_mxfp8_noalloc: the fused _o_proj pair with its z hand-off in a fixed buffer of this
// library instead of caller-owned tensors. No page describes such a variant; the pair itself
// follows "[Perf][DSv4.1] MegaAttn: wo_a writes wo_b's MXFP8 input" (Overview).
#include <cuda_runtime.h>

#include <mutex>

#include "mxq.h"
#include "mxq_internal.h"

namespace {

// z (E4M3) at offset 0, its F8_128x4 scales after it; both 256-byte aligned
static __device__ __align__(256) unsigned char g_z_scratch[MXQ_NOALLOC_Z_BYTES + MXQ_NOALLOC_SF_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_scratch[kMaxDevices] = {};

// Address of the buffer on the current device, looked up once per device.
cudaError_t scratch_for_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_scratch[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_z_scratch);
    if (e != cudaSuccess) return e;
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

mxq_status o_proj_mxfp8_noalloc(const mxq_mx_tensor* o, const mxq_mx_tensor* wa, const mxq_mx_tensor* wb, int64_t T,
                                int32_t G, int32_t Na, int32_t Ka, int32_t Nb, void* out_bf16, void* status,
                                void* stream) {
  if (T <= 0 || G <= 0 || Na <= 0) return MXQ_ERR_INVALID_ARG;
  const int64_t kz = static_cast<int64_t>(G) * Na;
  if (kz % 128 != 0) return MXQ_ERR_UNSUPPORTED_SHAPE;
  if (T > static_cast<int64_t>(MXQ_NOALLOC_Z_BYTES) / kz) return MXQ_ERR_UNSUPPORTED_SHAPE;
  const size_t sf = mxq_sf_bytes(MXQ_SF_TILED_128X4, T, kz);
  if (sf == 0 || sf > MXQ_NOALLOC_SF_BYTES) return MXQ_ERR_UNSUPPORTED_SHAPE;
  void* base = nullptr;
  const mxq_status st = mxq::from_cuda(scratch_for_current_device(&base));
  if (st != MXQ_OK) return st;
  unsigned char* z_q = static_cast<unsigned char*>(base);
  // No split workspace: at any T the buffer admits (T <= 256 at G * Na = 8192, up to 2048 with
  // G * Na = 1024) the large-T CTA-pair kernel then runs whole tiles, which needs none.
  return o_proj_mxfp8(o, wa, wb, T, G, Na, Ka, Nb, z_q, z_q + MXQ_NOALLOC_Z_BYTES, nullptr, nullptr, out_bf16, nullptr, 0,
                      status, stream);
}

}  // extern "C"
