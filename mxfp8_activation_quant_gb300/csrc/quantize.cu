// Standalone MXFP8 quantizer and the RMSNorm dual-output producer (HBM-streaming kernels).
//
// Quantizer: page "[Perf][DSv4.1] MegaAttn: wo_a writes wo_b's MXFP8 input" (Claims: the
// standalone mxfp8_quantize launch) and "[Perf][DSv4.1] Keep activations MXFP8 between
// DeepGEMM kernels" (Purpose: the "[q]" launch; one scale for each 32 elements along K).
// RMSNorm: the latter page's "mega_mhc (post+pre+RMSNorm)" producer emitting bf16 and
// "(y_fp8, y_gemm_sf)" in one kernel (RMSNorm part only).
//
// Mapping: 8 bf16 per lane in one 16-byte load, 4 lanes per 32-element group (amax with two
// xor-shuffles), 16 lanes per 128-element scale word. A warp owns one row segment of
// 4 x 256 columns, so every load instruction covers 512 contiguous bytes.
#include <cuda_runtime.h>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kWarpsPerBlock = 4;  // 128-thread blocks: about 1 % faster than 256 at every measured size
// 256-column units per warp: 4 (16 KB of loads in flight per block) from 8 M elements up, 2 below
// (more, smaller blocks: [256, 8192] 4.18 -> 3.72 us, [1024, 8192] 7.50 -> 7.19 us; at
// [32768, 8192] 2 units lose 10 %)
constexpr int64_t kSmallQuantElems = int64_t(8) << 20;
constexpr int64_t kEarlyGammaRows = 256;  // RMSNorm row counts that load gamma early (measured)

struct QuantArgs {
  const uint16_t* x;
  int64_t M, K, ldx;
  uint8_t* q;
  int64_t ldq;
  uint8_t* sf_rm;   // [M, Kg]
  uint32_t* sf_pk;  // [Kw, Mp4]
  uint8_t* sf_tl;   // F8_128x4
  int64_t Kg, Kw, Mp4, Mp128;
  int64_t rows_total;  // rows covered (padding rows write zero scale words only)
  int32_t chunks;      // warp segments per row
};

// Scales of one 256-column unit: row-major bytes, packed word, tiled word.
__device__ __forceinline__ void store_unit_scales(const QuantArgs& a, int64_t row, int64_t c, uint32_t code,
                                                  int lane) {
  if (a.sf_rm != nullptr && row < a.M && (lane & 3) == 0 && c < a.K) a.sf_rm[row * a.Kg + (c >> 5)] = code;
  uint32_t w = code;
  w |= __shfl_down_sync(0xffffffffu, code, 4) << 8;
  w |= __shfl_down_sync(0xffffffffu, code, 8) << 16;
  w |= __shfl_down_sync(0xffffffffu, code, 12) << 24;
  if ((lane & 15) == 0 && c < a.K) {
    const int64_t wi = c >> 7;
    if (a.sf_pk != nullptr && row < a.Mp4) a.sf_pk[wi * a.Mp4 + row] = w;
    if (a.sf_tl != nullptr && row < a.Mp128)
      *reinterpret_cast<uint32_t*>(a.sf_tl + tiled128x4_word_offset(row, wi, a.Kw)) = w;
  }
}

// at least 12 blocks per SM (40 registers): 75 % occupancy instead of 62.5 %, 1-2 % faster at
// large sizes (16 blocks forces spills and is slower)
template <int kUnits>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, 12) quantize_kernel(const QuantArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t row = wid / a.chunks;
  if (row >= a.rows_total) return;
  const int64_t col0 = (wid - row * a.chunks) * (256 * kUnits);
  const bool vrow = row < a.M;

  uint4 v[kUnits];
#pragma unroll
  for (int u = 0; u < kUnits; ++u) {
    const int64_t c = col0 + 256 * u + 8 * lane;
    v[u] = (vrow && c < a.K) ? ld_stream_u4(a.x + row * a.ldx + c) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int u = 0; u < kUnits; ++u) {
    const int64_t c = col0 + 256 * u + 8 * lane;
    if (col0 + 256 * u >= a.K) break;  // warp-uniform
    uint32_t amax = absmax8(v[u]);
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const uint32_t code = ue8m0_from_bf16_amax(amax);
    if (vrow && c < a.K) *reinterpret_cast<uint2*>(a.q + row * a.ldq + c) = quant8(v[u], ue8m0_inverse(code));
    store_unit_scales(a, row, c, code, lane);
  }
}

// ------------------------------------------------------------------------------------------
// RMSNorm with bf16 + MXFP8 outputs. One block of NT threads per row; thread t owns the
// 8-element chunks t, t + NT, ... of the row (CPT of them), held in registers between the two
// phases. NT is a multiple of 16, so a scale word's 16 chunks stay in 16 lanes of one warp.
// Measured at H = 5120 (cold-L2 graph timing): 256 threads are fastest up to 512 rows (T = 512:
// 6.35 -> 5.57 us), 160 (one group per thread) up to 2048 (T = 1024: 7.91 -> 7.49 us), 128 beyond.
// ------------------------------------------------------------------------------------------
struct RmsArgs {
  const uint16_t* x;
  const uint16_t* gamma;
  float eps, h;
  int64_t T, H, ldx;
  uint16_t* y;
  uint8_t* yq;
  uint8_t* sf_rm;
  uint32_t* sf_pk;
  uint8_t* sf_tl;
  int64_t Kg, Kw, Mp4, Mp128, rows_total;
};

// EARLY_G: load gamma with x instead of after the reduction. It removes one memory round trip
// from a block's critical path, which is the whole kernel when there are few rows; with many
// rows its extra registers cost more residency than it saves.
template <int CPT, bool EARLY_G, int NT>
__global__ void __launch_bounds__(NT) rmsnorm_dual_kernel(const RmsArgs a) {
  const int64_t row = blockIdx.x;
  if (row >= a.rows_total) return;  // block-uniform
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool vrow = row < a.T;
  __shared__ float red[NT / 32];

  uint4 v[CPT], gv[CPT];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int64_t c = 8 * (tid + NT * j);
    v[j] = (vrow && c < a.H) ? ld_stream_u4(a.x + row * a.ldx + c) : make_uint4(0, 0, 0, 0);
    if (EARLY_G) gv[j] = (vrow && c < a.H) ? *reinterpret_cast<const uint4*>(a.gamma + c) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = bf16_lo(w[i]), hi = bf16_hi(w[i]);
      ss = fmaf(lo, lo, ss);
      ss = fmaf(hi, hi, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float total = 0.f;
#pragma unroll
  for (int k = 0; k < NT / 32; ++k) total += red[k];
  const float r = rsqrtf(total / a.h + a.eps);

  QuantArgs qa;
  qa.M = a.T;
  qa.K = a.H;
  qa.sf_rm = a.sf_rm;
  qa.sf_pk = a.sf_pk;
  qa.sf_tl = a.sf_tl;
  qa.Kg = a.Kg;
  qa.Kw = a.Kw;
  qa.Mp4 = a.Mp4;
  qa.Mp128 = a.Mp128;

#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int64_t cbase = static_cast<int64_t>(8) * NT * j;
    if (cbase >= a.H) break;  // block-uniform
    const int64_t c = 8 * (tid + NT * j);
    uint4 y = make_uint4(0, 0, 0, 0);
    if (vrow && c < a.H) {
      const uint4 g = EARLY_G ? gv[j] : *reinterpret_cast<const uint4*>(a.gamma + c);
      y.x = bf16x2_rn((bf16_lo(v[j].x) * r) * bf16_lo(g.x), (bf16_hi(v[j].x) * r) * bf16_hi(g.x));
      y.y = bf16x2_rn((bf16_lo(v[j].y) * r) * bf16_lo(g.y), (bf16_hi(v[j].y) * r) * bf16_hi(g.y));
      y.z = bf16x2_rn((bf16_lo(v[j].z) * r) * bf16_lo(g.z), (bf16_hi(v[j].z) * r) * bf16_hi(g.z));
      y.w = bf16x2_rn((bf16_lo(v[j].w) * r) * bf16_lo(g.w), (bf16_hi(v[j].w) * r) * bf16_hi(g.w));
      *reinterpret_cast<uint4*>(a.y + row * a.H + c) = y;
    }
    uint32_t amax = absmax8(y);
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const uint32_t code = ue8m0_from_bf16_amax(amax);
    if (vrow && c < a.H) *reinterpret_cast<uint2*>(a.yq + row * a.H + c) = quant8(y, ue8m0_inverse(code));
    store_unit_scales(qa, row, c, code, lane);
  }
}

template <int CPT, int NT>
cudaError_t launch_rms_cpt(const RmsArgs& ra, cudaStream_t stream) {
  if (ra.rows_total <= kEarlyGammaRows)
    rmsnorm_dual_kernel<CPT, true, NT><<<static_cast<unsigned>(ra.rows_total), NT, 0, stream>>>(ra);
  else
    rmsnorm_dual_kernel<CPT, false, NT><<<static_cast<unsigned>(ra.rows_total), NT, 0, stream>>>(ra);
  return cudaGetLastError();
}

template <int NT>
cudaError_t launch_rms_nt(const RmsArgs& ra, int64_t H, cudaStream_t stream) {
  switch ((H / 8 + NT - 1) / NT) {  // 8-element chunks per thread
    case 1: return launch_rms_cpt<1, NT>(ra, stream);
    case 2: return launch_rms_cpt<2, NT>(ra, stream);
    case 3: return launch_rms_cpt<3, NT>(ra, stream);
    case 4: return launch_rms_cpt<4, NT>(ra, stream);
    case 5: return launch_rms_cpt<5, NT>(ra, stream);
    case 6: return launch_rms_cpt<6, NT>(ra, stream);
    case 7: case 8: return launch_rms_cpt<8, NT>(ra, stream);
    case 9: case 10: case 11: case 12: return launch_rms_cpt<12, NT>(ra, stream);
    case 13: case 14: case 15: case 16: return launch_rms_cpt<16, NT>(ra, stream);
    default: return cudaErrorInvalidValue;
  }
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

cudaError_t launch_quantize(const QuantizeLaunch& l, cudaStream_t stream) {
  QuantArgs a;
  a.x = static_cast<const uint16_t*>(l.x);
  a.M = l.M;
  a.K = l.K;
  a.ldx = l.ldx;
  a.q = static_cast<uint8_t*>(l.q);
  a.ldq = l.ldq;
  a.sf_rm = static_cast<uint8_t*>(l.sf_rowmajor);
  a.sf_pk = static_cast<uint32_t*>(l.sf_packed);
  a.sf_tl = static_cast<uint8_t*>(l.sf_tiled);
  a.Kg = l.K / 32;
  a.Kw = ceil_div(a.Kg, 4);
  a.Mp4 = ceil_div(l.M, 4) * 4;
  a.Mp128 = ceil_div(l.M, 128) * 128;
  a.rows_total = a.sf_tl ? a.Mp128 : (a.sf_pk ? a.Mp4 : l.M);
  const bool small = l.M * l.K <= kSmallQuantElems;
  const int units = small ? 2 : 4;
  a.chunks = static_cast<int32_t>(ceil_div(l.K, 256 * units));
  const int64_t warps = a.rows_total * a.chunks;
  const int64_t blocks = ceil_div(warps, kWarpsPerBlock);
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  if (small)
    quantize_kernel<2><<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, stream>>>(a);
  else
    quantize_kernel<4><<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const RmsnormLaunch& l, cudaStream_t stream) {
  RmsArgs a;
  a.x = static_cast<const uint16_t*>(l.x);
  a.gamma = static_cast<const uint16_t*>(l.gamma);
  a.eps = l.eps;
  a.h = static_cast<float>(l.H);
  a.T = l.T;
  a.H = l.H;
  a.ldx = l.ldx;
  a.y = static_cast<uint16_t*>(l.y);
  a.yq = static_cast<uint8_t*>(l.yq);
  a.sf_rm = static_cast<uint8_t*>(l.sf_rowmajor);
  a.sf_pk = static_cast<uint32_t*>(l.sf_packed);
  a.sf_tl = static_cast<uint8_t*>(l.sf_tiled);
  a.Kg = l.H / 32;
  a.Kw = ceil_div(a.Kg, 4);
  a.Mp4 = ceil_div(l.T, 4) * 4;
  a.Mp128 = ceil_div(l.T, 128) * 128;
  a.rows_total = a.sf_tl ? a.Mp128 : (a.sf_pk ? a.Mp4 : l.T);
  if (a.rows_total > 0x7FFFFFFF) return cudaErrorInvalidValue;
  if (a.rows_total <= 512) return launch_rms_nt<256>(a, l.H, stream);
  if (a.rows_total <= 2048) return launch_rms_nt<160>(a, l.H, stream);
  return launch_rms_nt<128>(a, l.H, stream);
}

}  // namespace mxq
