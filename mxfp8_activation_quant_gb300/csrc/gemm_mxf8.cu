// Block-scaled MXFP8 GEMMs of the _o_proj chain on 5th-generation tensor cores (sm_103a).
//
// Pages: "[Perf][DSv4.1] MegaAttn: wo_a writes wo_b's MXFP8 input" (Overview, Validation,
// Details): wo_a is a grouped FP8 einsum (8 groups, 4096 in, 1024 out) whose epilogue writes z as
// MXFP8 with F8_128x4 scales; wo_b is an MXFP8 GEMM "8192 -> 5120" that takes that z directly.
//
// One kernel template serves both. Per CTA (192 threads):
//   warp 0      TMA producer: operand tiles (128-byte swizzle) + 512-byte scale atoms
//   warp 1      TMEM owner and MMA issuer: tcgen05.cp copies each stage's scale atoms into
//               TMEM, then 4 x tcgen05.mma kind::mxf8f6f4 block_scale (K = 32 each)
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator, bf16 rounding, and (for wo_a)
//               per-32 MXFP8 quantization in registers
// Two orientations:
//   normal  (large T): A = activations (128 tokens / tile), B = weights (BN features / tile).
//           TMEM lane = token row, so one thread holds a 32-column quantization group.
//   swap-AB (T <= 384): A = weights (128 features / tile), B = activations (one token tile of
//           N = 16..64, or 128-token tiles). TMEM lane = feature, so a quantization group is
//           one warp (32 lanes). The K range is split over a thread-block cluster; partial sums
//           meet in distributed shared memory and are added in fixed rank order
//           (deterministic, no atomics).
// Inside o_proj_mxfp8 the wo_b grid is a programmatic dependent of the wo_a grid: its CTAs
// start while wo_a drains, fetch their first stages of weights, and only then wait for z.
// Every mbarrier wait is bounded (about 1 s); a wait that gives up records MXQ_ERR_TIMEOUT in
// the optional status word and the CTA drains its own copies and MMAs before leaving.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kThreads = 192;
constexpr int BM = 128;            // MMA M: rows of the A operand = TMEM lanes
constexpr int BK = 128;            // K bytes per stage = one 128-byte swizzle row
constexpr int kStatusTimeout = 6;  // MXQ_ERR_TIMEOUT
constexpr int kSwapMaxTokens = 384; // above this the CTA-pair kernel is faster (measured, T = 512)
// Fixed cost of the stream-K tail (partial sums through L2, flags, the finishing pass), in
// k-blocks of tile time: the split is taken only when whole tiles would waste more than this.
constexpr int kSkCostKb = 16;

struct KArgs {
  int64_t T;
  int32_t G;
  int32_t n_feat;
  int32_t kb_per_cta;       // 128-wide k-blocks per CTA
  int32_t splits;           // swap-AB: CTAs per cluster along K
  int32_t pdl;              // launched as a programmatic dependent: prefetch weights, then wait
  int32_t early;            // issue the first stages during setup (never with pdl)
  int32_t per_rank_shift;   // log2(reduction columns owned by each cluster rank)
  int64_t act_k_per_group;  // activation column offset between groups
  const uint8_t* act_sf;
  int64_t act_gp4;  // 512-byte atoms per activation row tile
  const uint8_t* wt_sf;
  int64_t wt_gp4;
  uint16_t* out_bf16;
  int64_t ldo;
  uint8_t* z_q;
  int64_t ldz;
  uint8_t* z_sf_tl;
  int64_t z_gp4, z_mp128;
  uint8_t* z_sf_pk;  // byte view of the packed words
  int64_t z_mp4;
  int32_t* status;
  int64_t act_mp4;  // packed activation scales: rows per word column (ceil(T / 4) * 4)
  // CTA-pair kernel, split tail (the SK instantiation; null otherwise). Partial sums of the
  // sharers of a split tile that do not finish it: two 128 KB slots per CTA (a pair's first and
  // last segment), [pair][segment][rank][8 epilogue warps][32 x 16-byte column groups][32 lanes];
  // ready flags [pair][segment][rank][8 epilogue warps]; arrival tickets [tail tile][rank][8
  // epilogue warps]. Flags and tickets are zero between launches.
  float4* sk_part;
  int32_t* sk_flag;
  int32_t* sk_ticket;
};

__device__ __forceinline__ void report_timeout(int32_t* status) {
  if (status != nullptr) atomicCAS(status, 0, kStatusTimeout);
}

// How the activation operand of the swap-AB kernel arrives: MXFP8 with F8_128x4 scales (the
// default), bf16 quantized in the kernel, or MXFP8 with int32-packed MN-major scales rearranged
// into the F8_128x4 atom in the kernel. The last two are decode tiles only (BN = 16).
constexpr int kActMx = 0, kActBf16 = 1, kActPackedSf = 2;

template <int BN, int STAGES, int ACT = kActMx>
struct Cfg {
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int SFB_ATOMS = (BN + 127) / 128;
  static constexpr int SF_BYTES = 512 * (1 + SFB_ATOMS);
  static constexpr int SF_COLS = 16;  // TMEM columns per stage slot (4 for A + 4 per B atom, padded)
  // kActBf16: the activation tile arrives as bf16 (BN rows of 128 elements, 256-byte rows, no
  // swizzle) in a staging slot, and the epilogue warps quantize it into the B tile and its
  // scale atom before the MMAs of the stage. kActPackedSf: the activation tile arrives as usual
  // and the stage's packed scale words (one per token row of the tile) land in the staging slot,
  // which the epilogue warps scatter into the activation's F8_128x4 atom.
  // (in the normal orientation the activation is A, 128 rows: used with BN = 128 only)
  static constexpr int BF_BYTES = ACT == kActBf16 ? BN * 256 : ACT == kActPackedSf ? BN * 4 : 0;
  // bytes on the stage's full barrier; the staged activation part has a barrier of its own, so
  // its conversion starts as soon as it lands, under the larger weight load
  static constexpr int TX_BYTES = ACT == kActBf16 ? A_BYTES + 512 : ACT == kActPackedSf ? A_BYTES + B_BYTES + 512
                                                                                       : A_BYTES + B_BYTES + SF_BYTES;
  static constexpr int OFF_B = STAGES * A_BYTES;
  // staging slots right behind the operand tiles, so that the split-K exchange below (after the
  // mainloop) may use them too
  static constexpr int OFF_BF = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SF = OFF_BF + STAGES * BF_BYTES;
  // Split-K reduction (swap-AB). Token tiles of 16 columns (decode) push their partials
  // with per-thread st.async into a dedicated receive buffer [source rank][feature][column] as
  // soon as their own MMAs are done (PUSH). Wider tiles stage their partials in the operand
  // tiles once their MMAs have completed (BN * 512 bytes, one block per owner) and receive the
  // peers' blocks there too ((splits - 1) / splits of that), after a cluster barrier that every
  // CTA reaches after its MMAs; split_fits() bounds the split accordingly.
  static constexpr bool PUSH = BN <= 16;
  static constexpr int RECV_BYTES = PUSH ? 128 * BN * 4 : 0;
  static constexpr bool split_fits(int s) { return PUSH || BN * 512 + BN * 512 / s * (s - 1) <= OFF_SF; }
  static constexpr int OFF_RECV = OFF_SF + STAGES * SF_BYTES;
  static constexpr int OFF_BAR = OFF_RECV + RECV_BYTES;
  // full, empty, 4 more, and (ACT != kActMx) "converted" and "staged part landed" per stage
  static constexpr int OFF_MISC = OFF_BAR + ((ACT != kActMx ? 4 : 2) * STAGES + 4) * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static constexpr int TMEM_USED = BN + STAGES * SF_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                   : TMEM_USED <= 64  ? 64
                                   : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256
                                                      : 512;
  // Co-resident CTAs must never need more than the SM's 512 TMEM columns in total (a CTA
  // blocked in tcgen05.alloc while a cluster peer waits for it would never resume), so the
  // launch requests enough shared memory to keep at most 512 / TMEM_COLS CTAs per SM.
  static constexpr int SM_SMEM = 228 * 1024;
  static constexpr int MAX_CO = 512 / TMEM_COLS;
  static constexpr int SMEM_FLOOR = SM_SMEM / (MAX_CO + 1) + 1024;
  static constexpr int SMEM_LAUNCH = SMEM_BYTES > SMEM_FLOOR ? SMEM_BYTES : SMEM_FLOOR;
  // byte offset of the activation's scale atom in a stage's scale slot (the weight atom is first
  // in swap-AB, second otherwise)
  static constexpr int ACT_ATOM = 512;
  // Token (swap-AB) or feature tiles of 16..128 columns: the 128 x 256 tile of this kernel,
  // with two B scale atoms, is not used (the CTA-pair kernel covers 256-wide tiles) and its
  // scale and split-K paths are not validated.
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "MMA N");
  static_assert(TMEM_USED <= 512, "TMEM");
  // unsplit swap-AB epilogue: 128 features x (BN + 4) floats staged in the tile region
  static_assert(128 * (BN + 4) * 4 <= OFF_SF, "epilogue staging must fit in the tile region");
  static_assert(SMEM_LAUNCH <= 227 * 1024, "shared memory");
  static_assert(4 * (1 + SFB_ATOMS) <= SF_COLS, "scale slot");
};

// ---- epilogue helpers ----------------------------------------------------------------------
// Split-K staging blocks: row `row` of a block holds `cpr` 16-byte chunks; chunk c is stored at
// c ^ recv_swizzle(row, cpr), which spreads 8 consecutive rows over the 8 chunk positions of a
// 128-byte bank line (fewer when a row has fewer than 8 chunks).
__device__ __forceinline__ int recv_swizzle(int row, int cpr) {
  return cpr >= 8 ? (row & 7) : ((row * cpr) >> 3) & (cpr - 1);
}

// An uneven split of n items (k-blocks, or 4-column chunks of the token tile) over US ranks:
// rank o takes [us_lo(o), us_lo(o + 1)).
template <int US>
__host__ __device__ constexpr int us_lo(int o, int n) { return o * n / (US > 0 ? US : 1); }
// the rank that owns item x
template <int US>
__host__ __device__ constexpr int us_owner(int x, int n) { return ((x + 1) * US + n - 1) / n - 1; }

__device__ __forceinline__ uint32_t amax_bf16x2_words(const uint32_t* hb, int n) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < n; ++i) m = max(m, absmax_bf16x2(hb[i]));
  return m;
}

// normal orientation: one thread = one token row, 32 consecutive feature columns
__device__ __forceinline__ void epi_row_chunk(const KArgs& p, const uint32_t (&acc)[32], int64_t row, int64_t col,
                                              uint32_t& word, int c) {
  uint32_t hb[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) hb[i] = bf16x2_rn(__uint_as_float(acc[2 * i]), __uint_as_float(acc[2 * i + 1]));
  const bool vrow = row < p.T;
  if (p.out_bf16 != nullptr && vrow) {
    uint4* dst = reinterpret_cast<uint4*>(p.out_bf16 + row * p.ldo + col);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
  }
  if (p.z_q != nullptr) {
    const uint32_t code = ue8m0_from_bf16_amax(amax_bf16x2_words(hb, 16));
    const float s = ue8m0_inverse(code);
    uint32_t qw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      qw[i] = e4m3x2(bf16_lo(hb[2 * i]) * s, bf16_hi(hb[2 * i]) * s) |
              (e4m3x2(bf16_lo(hb[2 * i + 1]) * s, bf16_hi(hb[2 * i + 1]) * s) << 16);
    if (vrow) {
      uint4* dst = reinterpret_cast<uint4*>(p.z_q + row * p.ldz + col);
      dst[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
      dst[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    }
    word |= code << (8 * (c & 3));
    if ((c & 3) == 3) {
      const int64_t wi = (col - 96) >> 7;  // first column of this 4-group word / 128
      if (p.z_sf_tl != nullptr)
        *reinterpret_cast<uint32_t*>(p.z_sf_tl + tiled128x4_word_offset(row, wi, p.z_gp4)) = word;
      if (p.z_sf_pk != nullptr && row < p.z_mp4)
        *reinterpret_cast<uint32_t*>(p.z_sf_pk + (wi * p.z_mp4 + row) * 4) = word;
      word = 0;
    }
  }
}

// normal orientation through a warp's 2 KB staging block (CTA-pair kernel): lane l holds token
// row row0 + l and 32 consecutive feature columns. The warp writes the chunk back row by row, so
// that one store instruction covers 8 rows x 64 bytes (bf16) or 16 rows x 32 bytes (E4M3): whole
// 32-byte sectors, a quarter of the requests of a 16-byte piece in each of 32 rows. Measured in
// cold-L2 graph replay: the _o_proj pair at 512 tokens 52.0 -> 49.3 us, at 2048 122.2 -> 117.9 us,
// at 4096 208.4 -> 203.3 us (with the stores removed altogether wo_b at 4096 tokens would take
// 107.6 instead of 114.5 us: the scattered pieces drained slowly in the exposed last tile). Staging
// a warp's whole 32 x 128 share of the last tile in the idle operand stages, for 128- and 256-byte
// rows, was no faster. The 16-byte pieces of a staged row are XOR-swizzled by the row, so that
// neither the staging stores nor the loads conflict on banks. Every lane of the warp calls it.
// (hb: the chunk already rounded to bf16, two columns per word)
__device__ __forceinline__ void epi_hb_chunk_staged(const KArgs& p, const uint32_t (&hb)[16], int64_t row0, int lane,
                                                    int64_t col, uint32_t& word, int c, uint32_t stage) {
  if (p.out_bf16 != nullptr) {
    // row r's 64 bytes: piece j at r * 64 + 16 * (j ^ ((r >> 1) & 3))
#pragma unroll
    for (int j = 0; j < 4; ++j)
      st_smem_v4(stage + lane * 64 + 16 * (j ^ ((lane >> 1) & 3)), hb[4 * j], hb[4 * j + 1], hb[4 * j + 2], hb[4 * j + 3]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 8 * i + (lane >> 2), j = lane & 3;
      const uint4 v = ld_smem_v4(stage + r * 64 + 16 * (j ^ ((r >> 1) & 3)));
      if (row0 + r < p.T) *reinterpret_cast<uint4*>(p.out_bf16 + (row0 + r) * p.ldo + col + 8 * j) = v;
    }
    __syncwarp();
  }
  if (p.z_q != nullptr) {
    const uint32_t code = ue8m0_from_bf16_amax(amax_bf16x2_words(hb, 16));
    const float s = ue8m0_inverse(code);
    uint32_t qw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      qw[i] = e4m3x2(bf16_lo(hb[2 * i]) * s, bf16_hi(hb[2 * i]) * s) |
              (e4m3x2(bf16_lo(hb[2 * i + 1]) * s, bf16_hi(hb[2 * i + 1]) * s) << 16);
    // row r's 32 bytes: piece j at r * 32 + 16 * (j ^ ((r >> 2) & 1))
    const int sw = (lane >> 2) & 1;
    st_smem_v4(stage + lane * 32 + 16 * sw, qw[0], qw[1], qw[2], qw[3]);
    st_smem_v4(stage + lane * 32 + 16 * (sw ^ 1), qw[4], qw[5], qw[6], qw[7]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = 16 * i + (lane >> 1), j = lane & 1;
      const uint4 v = ld_smem_v4(stage + r * 32 + 16 * (j ^ ((r >> 2) & 1)));
      if (row0 + r < p.T) *reinterpret_cast<uint4*>(p.z_q + (row0 + r) * p.ldz + col + 16 * j) = v;
    }
    __syncwarp();
    word |= code << (8 * (c & 3));
    if ((c & 3) == 3) {
      const int64_t row = row0 + lane;
      const int64_t wi = (col - 96) >> 7;  // first column of this 4-group word / 128
      if (p.z_sf_tl != nullptr)
        *reinterpret_cast<uint32_t*>(p.z_sf_tl + tiled128x4_word_offset(row, wi, p.z_gp4)) = word;
      if (p.z_sf_pk != nullptr && row < p.z_mp4)
        *reinterpret_cast<uint32_t*>(p.z_sf_pk + (wi * p.z_mp4 + row) * 4) = word;
      word = 0;
    }
  }
}

__device__ __forceinline__ void epi_row_chunk_staged(const KArgs& p, const uint32_t (&acc)[32], int64_t row0, int lane,
                                                     int64_t col, uint32_t& word, int c, uint32_t stage) {
  uint32_t hb[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) hb[i] = bf16x2_rn(__uint_as_float(acc[2 * i]), __uint_as_float(acc[2 * i + 1]));
  epi_hb_chunk_staged(p, hb, row0, lane, col, word, c, stage);
}

// scale byte 0 of a padding token row (t >= T) of the tiled / packed z scales
__device__ __forceinline__ void epi_zero_scale(const KArgs& p, int64_t t, int64_t col) {
  if (p.z_q == nullptr || t >= p.z_mp128) return;
  const int64_t gi = col >> 5;
  if (p.z_sf_tl != nullptr) p.z_sf_tl[tiled128x4_word_offset(t, gi >> 2, p.z_gp4) + (gi & 3)] = 0;
  if (p.z_sf_pk != nullptr && t < p.z_mp4) p.z_sf_pk[((gi >> 2) * p.z_mp4 + t) * 4 + (gi & 3)] = 0;
}

// swap orientation, split-K decode tiles: one warp finishes one 32-feature group of four
// consecutive tokens t0..t0+3. Lane l holds the fp32 sums of feature col + l for the four
// tokens (x, y, z, w); the group amax is one warp reduction per token.
__device__ __forceinline__ void epi_group_tokens4(const KArgs& p, const float4 s, int64_t t0, int64_t col, int lane) {
  const uint32_t h01 = bf16x2_rn(s.x, s.y), h23 = bf16x2_rn(s.z, s.w);
  const uint32_t hv[4] = {h01 & 0xFFFFu, h01 >> 16, h23 & 0xFFFFu, h23 >> 16};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t t = t0 + k;  // the same in every lane
    if (t >= p.z_mp128) break;
    if (t >= p.T) {  // padding token: only its zero scale is stored
      if (lane == 0) epi_zero_scale(p, t, col);
      continue;
    }
    if (p.out_bf16 != nullptr) p.out_bf16[t * p.ldo + col + lane] = static_cast<uint16_t>(hv[k]);
    if (p.z_q != nullptr) {
      const uint32_t code = ue8m0_from_bf16_amax(__reduce_max_sync(0xffffffffu, hv[k] & 0x7FFFu));
      p.z_q[t * p.ldz + col + lane] = static_cast<uint8_t>(e4m3x2(bf16_lo(hv[k]) * ue8m0_inverse(code), 0.f));
      if (lane == 0) {
        const int64_t gi = col >> 5;
        if (p.z_sf_tl != nullptr)
          p.z_sf_tl[tiled128x4_word_offset(t, gi >> 2, p.z_gp4) + (gi & 3)] = static_cast<uint8_t>(code);
        if (p.z_sf_pk != nullptr && t < p.z_mp4)
          p.z_sf_pk[((gi >> 2) * p.z_mp4 + t) * 4 + (gi & 3)] = static_cast<uint8_t>(code);
      }
    }
  }
}

// swap orientation, after the partial sums are in shared memory: one thread = one token and
// one 32-feature quantization group. v[0..31] are the fp32 sums for features col..col+31 of
// token t (col = first output column of the group).
__device__ __forceinline__ void epi_token_group(const KArgs& p, const float (&v)[32], int64_t t, int64_t col) {
  if (t >= p.z_mp128) return;
  uint32_t hb[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) hb[i] = bf16x2_rn(v[2 * i], v[2 * i + 1]);
  const bool vt = t < p.T;
  if (p.out_bf16 != nullptr && vt) {
    uint4* dst = reinterpret_cast<uint4*>(p.out_bf16 + t * p.ldo + col);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
  }
  if (p.z_q != nullptr) {
    const uint32_t code = ue8m0_from_bf16_amax(amax_bf16x2_words(hb, 16));
    const float s = ue8m0_inverse(code);
    uint32_t qw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      qw[i] = e4m3x2(bf16_lo(hb[2 * i]) * s, bf16_hi(hb[2 * i]) * s) |
              (e4m3x2(bf16_lo(hb[2 * i + 1]) * s, bf16_hi(hb[2 * i + 1]) * s) << 16);
    if (vt) {
      uint4* dst = reinterpret_cast<uint4*>(p.z_q + t * p.ldz + col);
      dst[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
      dst[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    }
    const int64_t gi = col >> 5;
    if (p.z_sf_tl != nullptr) p.z_sf_tl[tiled128x4_word_offset(t, gi >> 2, p.z_gp4) + (gi & 3)] = static_cast<uint8_t>(code);
    if (p.z_sf_pk != nullptr && t < p.z_mp4)
      p.z_sf_pk[((gi >> 2) * p.z_mp4 + t) * 4 + (gi & 3)] = static_cast<uint8_t>(code);
  }
}

// US > 0: the swap-AB wide-tile kernel with K split over US cluster ranks, a count that need
// not divide the k-blocks or the token columns (p.kb_per_cta then holds all k-blocks of K).
template <int BN, int STAGES, bool SWAP, int ACT = kActMx, int US = 0>
__global__ void __launch_bounds__(kThreads, 3)
    gemm_mxf8_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const KArgs p) {
  static_assert(ACT != kActBf16 || (SWAP ? BN <= 128 : BN == BM), "bf16 activations: one 128-row staging slot");
  static_assert(ACT != kActPackedSf || BN <= 128, "packed activation scales: one activation atom per stage");
  static_assert(US == 0 || (SWAP && BN >= 32 && US <= BN / 4), "uneven split: wide tiles");
  constexpr bool CVT = ACT != kActMx;  // a staged activation part converted by the epilogue warps
  using C = Cfg<BN, STAGES, ACT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sraw = smem_u32(smem_raw);
  const uint32_t sbase = (sraw + 1023u) & ~1023u;  // 128-byte-swizzled tiles need 1024-byte alignment
  uint8_t* smem = smem_raw + (sbase - sraw);
  const uint32_t bar_full = sbase + C::OFF_BAR;      // STAGES x 8 B
  const uint32_t bar_empty = bar_full + STAGES * 8;  // STAGES x 8 B
  const uint32_t bar_accf = bar_empty + STAGES * 8;  // 8 B
  const uint32_t bar_recv = bar_accf + 8;            // 8 B: split-K partials received
  const uint32_t bar_conv = bar_full + (2 * STAGES + 4) * 8;  // CVT: STAGES x 8 B, stage quantized
  const uint32_t bar_act = bar_conv + STAGES * 8;             // CVT: STAGES x 8 B, bf16 tile landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int* issued_cnt = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);
  int* consumed_cnt = reinterpret_cast<int*>(smem + C::OFF_MISC + 12);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- tile coordinates ----
  int g, split;
  int64_t a_row0, b_row0, a_xoff, b_xoff, a_rt, b_rt0, a_kc0, b_kc0;
  const uint8_t *a_sf, *b_sf;
  int64_t a_gp4, b_gp4;
  int64_t m0;  // first A row of this tile inside its group (features in swap, tokens otherwise)
  if (SWAP) {
    g = blockIdx.z / p.splits;
    split = blockIdx.z % p.splits;
    m0 = static_cast<int64_t>(blockIdx.x) * BM;
    a_row0 = static_cast<int64_t>(g) * p.n_feat + m0;  // weights
    b_row0 = static_cast<int64_t>(blockIdx.y) * BN;    // activations (token tile)
    a_xoff = 0;
    b_xoff = static_cast<int64_t>(g) * p.act_k_per_group;
    a_sf = p.wt_sf;
    a_gp4 = p.wt_gp4;
    a_rt = a_row0 >> 7;
    a_kc0 = 0;
    b_sf = p.act_sf;
    b_gp4 = p.act_gp4;
    b_rt0 = b_row0 >> 7;  // BN == 128 whenever there is more than one token tile
    b_kc0 = b_xoff >> 7;
  } else {
    g = blockIdx.z;
    split = 0;
    m0 = static_cast<int64_t>(blockIdx.y) * BM;
    a_row0 = m0;                                                                          // activations
    b_row0 = static_cast<int64_t>(g) * p.n_feat + static_cast<int64_t>(blockIdx.x) * BN;  // weights
    a_xoff = static_cast<int64_t>(g) * p.act_k_per_group;
    b_xoff = 0;
    a_sf = p.act_sf;
    a_gp4 = p.act_gp4;
    a_rt = a_row0 >> 7;
    a_kc0 = a_xoff >> 7;
    b_sf = p.wt_sf;
    b_gp4 = p.wt_gp4;
    b_rt0 = b_row0 >> 7;
    b_kc0 = 0;
  }
  const int kb_begin = US > 0 ? us_lo<US>(split, p.kb_per_cta) : split * p.kb_per_cta;
  const int nk = US > 0 ? us_lo<US>(split + 1, p.kb_per_cta) - kb_begin : p.kb_per_cta;
  const int pre = nk < STAGES ? nk : STAGES;  // stages that need no free-slot wait

  const uint32_t a_dst0 = sbase, b_dst0 = sbase + C::OFF_B, sf_dst0 = sbase + C::OFF_SF;
  // operand loads of k-block i into stage s; the weight operand is A in swap-AB, B otherwise
  auto load_act = [&](int s, int kb, uint32_t fb) {
    if (SWAP && ACT == kActPackedSf) {
      // E4M3 tile as usual; the stage's packed scale words (one per token, rows b_row0..) into
      // the staging slot. Only rows < Mp exist in each word column of the packed array.
      tma_load_2d(b_dst0 + s * C::B_BYTES, &tm_b, fb, static_cast<int32_t>(b_xoff + kb * BK), static_cast<int32_t>(b_row0));
      const uint32_t ab = bar_act + (fb - bar_full);
      const int64_t rows = p.act_mp4 - b_row0 < BN ? p.act_mp4 - b_row0 : BN;
      mbar_arrive_expect_tx(ab, static_cast<uint32_t>(rows * 4));
      bulk_load(sbase + C::OFF_BF + s * C::BF_BYTES, b_sf + ((b_kc0 + kb) * p.act_mp4 + b_row0) * 4,
                static_cast<uint32_t>(rows * 4), ab);
    } else if (SWAP && CVT) {  // bf16 activations (element coordinates) into the staging slot
      const uint32_t ab = bar_act + (fb - bar_full);
      mbar_arrive_expect_tx(ab, C::BF_BYTES);
      tma_load_2d(sbase + C::OFF_BF + s * C::BF_BYTES, &tm_b, ab, static_cast<int32_t>(b_xoff + kb * BK),
                  static_cast<int32_t>(b_row0));
    } else if (SWAP) {
      tma_load_2d(b_dst0 + s * C::B_BYTES, &tm_b, fb, static_cast<int32_t>(b_xoff + kb * BK), static_cast<int32_t>(b_row0));
#pragma unroll
      for (int j = 0; j < C::SFB_ATOMS; ++j)
        bulk_load(sf_dst0 + s * C::SF_BYTES + 512 * (1 + j), b_sf + ((b_rt0 + j) * b_gp4 + b_kc0 + kb) * 512, 512, fb);
    } else if (ACT == kActBf16) {  // normal orientation, bf16 activations (128 token rows)
      const uint32_t ab = bar_act + (fb - bar_full);
      mbar_arrive_expect_tx(ab, C::BF_BYTES);
      tma_load_2d(sbase + C::OFF_BF + s * C::BF_BYTES, &tm_a, ab, static_cast<int32_t>(a_xoff + kb * BK),
                  static_cast<int32_t>(a_row0));
    } else if (ACT == kActPackedSf) {  // normal orientation: the activation is A (128 token rows)
      tma_load_2d(a_dst0 + s * C::A_BYTES, &tm_a, fb, static_cast<int32_t>(a_xoff + kb * BK), static_cast<int32_t>(a_row0));
      const uint32_t ab = bar_act + (fb - bar_full);
      const int64_t rows = p.act_mp4 - a_row0 < BM ? p.act_mp4 - a_row0 : BM;
      mbar_arrive_expect_tx(ab, static_cast<uint32_t>(rows * 4));
      bulk_load(sbase + C::OFF_BF + s * C::BF_BYTES, a_sf + ((a_kc0 + kb) * p.act_mp4 + a_row0) * 4,
                static_cast<uint32_t>(rows * 4), ab);
    } else {
      tma_load_2d(a_dst0 + s * C::A_BYTES, &tm_a, fb, static_cast<int32_t>(a_xoff + kb * BK), static_cast<int32_t>(a_row0));
      bulk_load(sf_dst0 + s * C::SF_BYTES, a_sf + (a_rt * a_gp4 + a_kc0 + kb) * 512, 512, fb);
    }
  };
  auto load_wt = [&](int s, int kb, uint32_t fb) {
    if (SWAP) {
      tma_load_2d(a_dst0 + s * C::A_BYTES, &tm_a, fb, static_cast<int32_t>(a_xoff + kb * BK), static_cast<int32_t>(a_row0));
      bulk_load(sf_dst0 + s * C::SF_BYTES, a_sf + (a_rt * a_gp4 + a_kc0 + kb) * 512, 512, fb);
    } else {
      tma_load_2d(b_dst0 + s * C::B_BYTES, &tm_b, fb, static_cast<int32_t>(b_xoff + kb * BK), static_cast<int32_t>(b_row0));
#pragma unroll
      for (int j = 0; j < C::SFB_ATOMS; ++j)
        bulk_load(sf_dst0 + s * C::SF_BYTES + 512 * (1 + j), b_sf + ((b_rt0 + j) * b_gp4 + b_kc0 + kb) * 512, 512, fb);
    }
  };
  // ---- setup ----
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_accf, 1);
    if (CVT)
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(bar_conv + 8 * s, 4);  // one arrival per epilogue warp
        mbar_init(bar_act + 8 * s, 1);
      }
    if (SWAP && p.splits > 1) {
      mbar_init(bar_recv, 1);
      // PUSH: every rank, this one included, sends 128 features x (BN / splits) columns of fp32;
      // otherwise each other rank sends one block of that size
      mbar_arrive_expect_tx(bar_recv, static_cast<uint32_t>(C::PUSH ? 128 * BN * 4
                                                            : US > 0 ? 2048 * (us_lo<US>(split + 1, BN / 4) - us_lo<US>(split, BN / 4)) * (US - 1)
                                                                     : 128 * BN * 4 / p.splits * (p.splits - 1)));
    }
    *abort_flag = 0;
    *issued_cnt = 0;
    *consumed_cnt = 0;
    fence_mbar_init();
    // p.early: the first stages need no free slot, so they are issued here, before the TMEM
    // allocation and the block barrier (launch_gemm decides when)
    if (p.early)
      for (int j = 0; j < pre; ++j) {
        mbar_arrive_expect_tx(bar_full + 8 * j, C::TX_BYTES);
        load_wt(j, kb_begin + j, bar_full + 8 * j);
        load_act(j, kb_begin + j, bar_full + 8 * j);
      }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool recv_path = SWAP && p.splits > 1;
  // PUSH: peers may write this CTA's receive buffer once its barrier is initialized; arrive now,
  // wait just before the first push (by then every peer has long arrived)
  if (C::PUSH && recv_path) cluster_arrive();
  // A dependent grid (wo_b after wo_a) may start its prologue once every CTA of this grid has
  // passed this point: at once for the single-wave swap-AB grids, at the epilogue otherwise.
  if (SWAP && threadIdx.x == 0) pdl_launch_dependents();

  // ---- roles ----
  if (warp == 0 && lane == 0) {
    int i = p.early ? pre : 0;
    if (p.pdl) {
      // the first stages are free: fetch their weights while the producer of the activations
      // may still be running (it never writes them), then wait for it and fetch the activations
      for (int j = 0; j < pre; ++j) {
        mbar_arrive_expect_tx(bar_full + 8 * j, C::TX_BYTES);
        load_wt(j, kb_begin + j, bar_full + 8 * j);
      }
      pdl_wait_primary();
      for (int j = 0; j < pre; ++j) load_act(j, kb_begin + j, bar_full + 8 * j);
      i = pre;
    }
    for (; i < nk; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (i / STAGES) & 1;
      if (*abort_flag) break;
      if (!mbar_wait_bounded(bar_empty + 8 * s, ph ^ 1)) {
        *abort_flag = 1;
        report_timeout(p.status);
        break;
      }
      const int kb = kb_begin + i;
      const uint32_t fb = bar_full + 8 * s;
      mbar_arrive_expect_tx(fb, C::TX_BYTES);
      load_wt(s, kb, fb);
      load_act(s, kb, fb);
    }
    *issued_cnt = i;
  } else if (warp == 1 && lane == 0) {
    int i = 0;
    for (; i < nk; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (i / STAGES) & 1;
      if (*abort_flag) break;
      if (!mbar_wait_bounded(bar_full + 8 * s, ph) || (CVT && !mbar_wait_bounded(bar_conv + 8 * s, ph))) {
        *abort_flag = 1;
        report_timeout(p.status);
        break;
      }
      tc_fence_after();
      const uint32_t sf_src = sbase + C::OFF_SF + s * C::SF_BYTES;
      const uint32_t sfa_t = tmem + BN + s * C::SF_COLS;
      const uint32_t sfb_t = sfa_t + 4;
      tc_cp_sf_atom(sfa_t, sdesc_sf_atom(sf_src));
#pragma unroll
      for (int j = 0; j < C::SFB_ATOMS; ++j) tc_cp_sf_atom(sfb_t + 4 * j, sdesc_sf_atom(sf_src + 512 * (1 + j)));
      const uint64_t ad = sdesc_kmajor_sw128(sbase + s * C::A_BYTES);
      const uint64_t bd = sdesc_kmajor_sw128(sbase + C::OFF_B + s * C::B_BYTES);
#pragma unroll
      for (int k = 0; k < BK / 32; ++k)
        tc_mma_mxf8(tmem, ad + 2 * k, bd + 2 * k, idesc_mxf8(BM, BN, k, k), sfa_t, sfb_t, (i | k) != 0 ? 1u : 0u);
      tc_commit(bar_empty + 8 * s);
    }
    *consumed_cnt = i;
    tc_commit(bar_accf);  // arrives once every MMA above has completed
  }
  __syncwarp();

  // ---- epilogue ----
  const bool epi = warp >= 2;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * q) << 16);
  if (ACT == kActPackedSf && epi) {
    // During the mainloop the epilogue warps move each stage's packed scale words into the
    // activation's F8_128x4 atom: token row r's word (its 4 group bytes) goes to the atom's word
    // (r % 32) * 4 + r / 32 (bytes (r % 32) * 16 + (r / 32) * 4 ..).
    const int t = static_cast<int>(threadIdx.x) - 64;
    const int64_t row0 = SWAP ? b_row0 : a_row0;
    const int tile_rows = SWAP ? BN : BM;
    const int rows = static_cast<int>(p.act_mp4 - row0 < tile_rows ? p.act_mp4 - row0 : tile_rows);
    const int atom = SWAP ? C::ACT_ATOM : 0;
    for (int i = t; i < STAGES * 128; i += 128)  // rows past the packed array's stay zero
      reinterpret_cast<uint32_t*>(smem + C::OFF_SF + (i >> 7) * C::SF_BYTES + atom)[i & 127] = 0u;
    named_barrier(3, 128);
    for (int i = 0; i < nk; ++i) {
      const int s = i % STAGES;
      if (!mbar_wait_bounded(bar_act + 8 * s, (i / STAGES) & 1)) {
        *abort_flag = 1;
        report_timeout(p.status);
        break;
      }
      if (t < rows) {
        const uint32_t w = reinterpret_cast<const uint32_t*>(smem + C::OFF_BF + s * C::BF_BYTES)[t];
        reinterpret_cast<uint32_t*>(smem + C::OFF_SF + s * C::SF_BYTES + atom)[(t & 31) * 4 + (t >> 5)] = w;
      }
      fence_proxy_async_smem();  // the scale copy reads the atom through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_conv + 8 * s);
    }
  }
  if (ACT == kActBf16 && epi) {
    // During the mainloop the epilogue warps quantize each stage's bf16 activations exactly as
    // mxfp8_quantize does, into the activation tile (128-byte swizzle) and its F8_128x4 atom: a
    // unit is 16 elements (half a group) of one token row, thread t takes row t / 8 + 16 i and
    // half h = t % 2 of group (t / 2) % 4; the two halves of a group meet by one shuffle for the
    // amax. Rows past the last token arrive as zeros (the copy's fill) and get scale 0.
    constexpr int ROWS = SWAP ? BN : BM;
    const int t = static_cast<int>(threadIdx.x) - 64;
    const int c = (t >> 1) & 3, h = t & 1;
    const uint32_t tile0 = SWAP ? sbase + C::OFF_B : sbase;
    const int tile_bytes = SWAP ? C::B_BYTES : C::A_BYTES;
    const int atom = SWAP ? C::ACT_ATOM : 0;
    if (ROWS < 128) {  // atom rows past the tile's stay zero
      for (int i = t; i < STAGES * 128; i += 128)
        reinterpret_cast<uint32_t*>(smem + C::OFF_SF + (i >> 7) * C::SF_BYTES + atom)[i & 127] = 0u;
      named_barrier(3, 128);
    }
    for (int i = 0; i < nk; ++i) {
      const int s = i % STAGES;
      if (!mbar_wait_bounded(bar_act + 8 * s, (i / STAGES) & 1)) {
        *abort_flag = 1;
        report_timeout(p.status);
        break;
      }
#pragma unroll
      for (int u = 0; u < ROWS / 16; ++u) {
        const int r = (t >> 3) + 16 * u;
        const uint4* src = reinterpret_cast<const uint4*>(smem + C::OFF_BF + s * C::BF_BYTES + r * 256 + (32 * c + 16 * h) * 2);
        const uint4 v0 = src[0], v1 = src[1];
        uint32_t am = max(absmax8(v0), absmax8(v1));
        am = max(am, __shfl_xor_sync(0xffffffffu, am, 1));
        const uint32_t code = ue8m0_from_bf16_amax(am);
        const float sc = ue8m0_inverse(code);
        const uint2 q0 = quant8(v0, sc), q1 = quant8(v1, sc);
        const int j = 2 * c + h;  // 16-byte chunk of the 128-byte row, 128-byte swizzle
        st_smem_v4(tile0 + s * tile_bytes + r * 128 + ((j ^ (r & 7)) << 4), q0.x, q0.y, q1.x, q1.y);
        if (h == 0) smem[C::OFF_SF + s * C::SF_BYTES + atom + (r & 31) * 16 + (r >> 5) * 4 + c] = static_cast<uint8_t>(code);
      }
      fence_proxy_async_smem();  // the MMA and the scale copy read these through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_conv + 8 * s);
    }
  }
  if (epi) {
    if (!mbar_wait_bounded(bar_accf, 0)) {
      *abort_flag = 1;
      report_timeout(p.status);
    }
    tc_fence_after();
  }

  if (!SWAP) {
    if (threadIdx.x == 64) pdl_launch_dependents();
    if (epi && !__any_sync(0xffffffffu, *abort_flag)) {
      const int64_t row = m0 + 32 * q + lane;
      const int64_t col0 = static_cast<int64_t>(g) * p.n_feat + static_cast<int64_t>(blockIdx.x) * BN;
      uint32_t word = 0;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t acc[32];
        tmem_ld_x32(t_lane + 32 * c, acc);
        tmem_ld_wait();
        epi_row_chunk(p, acc, row, col0 + 32 * c, word, c);
      }
    }
  } else if (C::PUSH && recv_path) {
    // K split over the cluster, token tile of 16 columns. Each rank st.async's its fp32
    // partial of the columns owned by rank o (columns [o*per_rank, (o+1)*per_rank)) into rank
    // o's receive buffer, slot [source rank][feature][column]; the bytes complete on rank o's
    // mbarrier. Each owner adds its slots in rank order 0..splits-1 (deterministic) and
    // finishes whole (token, 32-feature group) items.
    const uint32_t rank = cluster_ctarank();
    const int per_rank = BN / p.splits;
    const int f = 32 * q + lane;
    const uint32_t recv = sbase + C::OFF_RECV;
    cluster_wait();
    if (epi && !__any_sync(0xffffffffu, *abort_flag)) {
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        uint32_t acc[16];
        tmem_ld_x16(t_lane + 16 * c, acc);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int cc = 16 * c + 4 * k;  // first of 4 columns, all owned by one rank
          const uint32_t owner = static_cast<uint32_t>(cc >> p.per_rank_shift);
          const int li = cc & (per_rank - 1);
          const uint32_t off = recv + static_cast<uint32_t>(((static_cast<int>(rank) * 128 + f) * per_rank + li) * 4);
          st_async_v4(mapa_shared(off, owner), acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3],
                      mapa_shared(bar_recv, owner));
        }
      }
    }
    if (epi) {
      if (!mbar_wait_bounded(bar_recv, 0)) {
        *abort_flag = 1;
        report_timeout(p.status);
      }
      if (!__any_sync(0xffffffffu, *abort_flag)) {
        // warp q finishes feature group q of this rank's columns, four tokens per pass; lane l
        // reads feature 32q + l of every slot as 16-byte rows (conflict-free)
        const float* red = reinterpret_cast<const float*>(smem + C::OFF_RECV);
        const int64_t col = static_cast<int64_t>(g) * p.n_feat + m0 + 32 * q;
#pragma unroll 1
        for (int j = 0; j < per_rank; j += 4) {
          float4 v = *reinterpret_cast<const float4*>(red + f * per_rank + j);
          for (int r = 1; r < p.splits; ++r) {
            const float4 u = *reinterpret_cast<const float4*>(red + (r * 128 + f) * per_rank + j);
            v.x += u.x;
            v.y += u.y;
            v.z += u.z;
            v.w += u.w;
          }
          epi_group_tokens4(p, v, b_row0 + static_cast<int>(rank) * per_rank + j, col, lane);
        }
      }
    }
  } else if (US > 0 && recv_path) {
    if constexpr (US > 0) {
    // The same exchange for an uneven split (US ranks): rank o owns the 4-column chunks
    // [us_lo(o), us_lo(o + 1)) of the token tile; the staged blocks lie in chunk order, owner o's
    // at 2 KB x us_lo(o). Chunk ownership is resolved at compile time in the fully unrolled
    // staging loop; odd chunk counts per row need no swizzle (8 consecutive rows already fall on
    // 8 different 16-byte bank positions).
    constexpr int NCH = BN / 4;
    const uint32_t rank = cluster_ctarank();
    const int own_lo = us_lo<US>(static_cast<int>(rank), NCH);
    const int own_cpr = us_lo<US>(static_cast<int>(rank) + 1, NCH) - own_lo;
    const int own_cols = 4 * own_cpr;
    const uint32_t own_blk = static_cast<uint32_t>(2048 * own_cpr);
    const uint32_t stage0 = sbase;            // this rank's partial: every owner's block
    const uint32_t recv0 = sbase + BN * 512;  // US - 1 blocks of this rank's columns
    const int f = 32 * q + lane;
    if (epi && !__any_sync(0xffffffffu, *abort_flag)) {
#pragma unroll
      for (int c = 0; c < BN / 16; ++c) {
        uint32_t acc[16];
        tmem_ld_x16(t_lane + 16 * c, acc);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int x = 4 * c + k;
          const int lo = us_lo<US>(us_owner<US>(x, NCH), NCH);
          const int cpr = us_lo<US>(us_owner<US>(x, NCH) + 1, NCH) - lo;
          const int chunk = (cpr & (cpr - 1)) == 0 ? (x - lo) ^ recv_swizzle(f, cpr) : x - lo;
          st_smem_v4(stage0 + static_cast<uint32_t>(2048 * lo + (f * cpr + chunk) * 16), acc[4 * k], acc[4 * k + 1],
                     acc[4 * k + 2], acc[4 * k + 3]);
        }
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    cluster_arrive();
    cluster_wait();
    if (threadIdx.x == 64 && !*abort_flag) {
      for (int d = 1; d < US; ++d) {
        const int o = (static_cast<int>(rank) + d) % US;
        const int slot = (static_cast<int>(rank) + US - o - 1) % US;  // this rank among o's sources
        const int lo = us_lo<US>(o, NCH);
        const uint32_t blk = static_cast<uint32_t>(2048 * (us_lo<US>(o + 1, NCH) - lo));
        bulk_s2s(mapa_shared(recv0 + slot * blk, static_cast<uint32_t>(o)), stage0 + static_cast<uint32_t>(2048 * lo), blk,
                 mapa_shared(bar_recv, static_cast<uint32_t>(o)));
      }
    }
    if (epi) {
      if (!mbar_wait_bounded(bar_recv, 0)) {
        *abort_flag = 1;
        report_timeout(p.status);
      }
    }
    __syncwarp();
    cluster_arrive();
    if (epi && !__any_sync(0xffffffffu, *abort_flag)) {
      const float* sm = reinterpret_cast<const float*>(smem);
      const bool pow2 = (own_cpr & (own_cpr - 1)) == 0;
      // own_cols takes one of two values, so the division by it is one by a constant
      constexpr int kColsLo = 4 * (NCH / US), kColsHi = 4 * ((NCH + US - 1) / US);
      for (int w = static_cast<int>(threadIdx.x) - 64; w < 4 * own_cols; w += 128) {
        const int gq = own_cols == kColsLo ? w / kColsLo : w / kColsHi;
        const int j = w - gq * own_cols;
        const int64_t t = b_row0 + 4 * own_lo + j;
        const int64_t col = static_cast<int64_t>(g) * p.n_feat + m0 + 32 * gq;
        if (t >= p.T) {  // padding token: only its zero scale is stored
          epi_zero_scale(p, t, col);
          continue;
        }
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
        for (int r = 0; r < US; ++r) {
          const uint32_t base = r == static_cast<int>(rank)
                                    ? stage0 + static_cast<uint32_t>(2048 * own_lo)
                                    : recv0 + static_cast<uint32_t>((r + US - static_cast<int>(rank) - 1) % US) * own_blk;
          const float* blkp = sm + (base - sbase) / 4;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int row = 32 * gq + i;
            const int ch = pow2 ? (j >> 2) ^ recv_swizzle(row, own_cpr) : j >> 2;
            const float x = blkp[row * own_cols + 4 * ch + (j & 3)];
            v[i] = r == 0 ? x : v[i] + x;
          }
        }
        epi_token_group(p, v, t, col);
      }
    }
    }  // if constexpr (US > 0)
  } else if (recv_path) {
    // K split over the cluster; rank o owns the token columns [o*per_rank, (o+1)*per_rank).
    // Every rank stages its fp32 partial in its own shared memory, one block per owner laid out
    // [feature][column] with the 16-byte chunks of each feature row XOR-swizzled (conflict-free
    // 16-byte writes by 8 lanes, conflict-free column reads by a warp). It then sends each other
    // owner its block with one bulk shared-to-shared copy, counted on the owner's mbarrier: a
    // handful of large transfers, where per-thread remote stores would each update that
    // mbarrier. Each owner adds the blocks of ranks 0..splits-1 in rank order (deterministic)
    // and finishes whole (token, 32-feature group) items.
    const uint32_t rank = cluster_ctarank();
    const int per_rank = BN / p.splits;
    const uint32_t blk = static_cast<uint32_t>(128 * per_rank * 4);
    const uint32_t stage0 = sbase;              // p.splits blocks: this rank's partial
    const uint32_t recv0 = sbase + BN * 512;    // p.splits - 1 blocks: the peers' partials
    const int cpr = per_rank >> 2;              // 16-byte chunks per feature row
    const int f = 32 * q + lane;
    if (epi && !__any_sync(0xffffffffu, *abort_flag)) {
      const int sw = recv_swizzle(f, cpr);
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        uint32_t acc[16];
        tmem_ld_x16(t_lane + 16 * c, acc);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int cc = 16 * c + 4 * k;  // first of 4 columns, all owned by one rank
          const uint32_t owner = static_cast<uint32_t>(cc >> p.per_rank_shift);
          const int chunk = ((cc & (per_rank - 1)) >> 2) ^ sw;
          st_smem_v4(stage0 + owner * blk + static_cast<uint32_t>((f * per_rank + 4 * chunk) * 4), acc[4 * k],
                     acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
        }
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    // every CTA of the cluster has finished its MMAs (epilogue warps arrive after bar_accf) and
    // staged its blocks: the operand regions that hold the receive blocks are idle
    cluster_arrive();
    cluster_wait();
    if (threadIdx.x == 64 && !*abort_flag) {
      for (int d = 1; d < p.splits; ++d) {
        const uint32_t o = (rank + d) % p.splits;
        const uint32_t slot = (rank + p.splits - o - 1) % p.splits;  // this rank among o's sources
        bulk_s2s(mapa_shared(recv0 + slot * blk, o), stage0 + o * blk, blk, mapa_shared(bar_recv, o));
      }
    }
    if (epi) {
      if (!mbar_wait_bounded(bar_recv, 0)) {
        *abort_flag = 1;
        report_timeout(p.status);
      }
    }
    // arrives once every copy into this CTA has landed (its senders may leave after the matching
    // wait in the teardown)
    __syncwarp();
    cluster_arrive();
    if (epi && !__any_sync(0xffffffffu, *abort_flag)) {
      const float* sm = reinterpret_cast<const float*>(smem);
      const int items = per_rank * 4;
      for (int w = static_cast<int>(threadIdx.x) - 64; w < items; w += 128) {
        const int j = w & (per_rank - 1);
        const int gq = w >> p.per_rank_shift;
        const int64_t t = b_row0 + static_cast<int>(rank) * per_rank + j;
        const int64_t col = static_cast<int64_t>(g) * p.n_feat + m0 + 32 * gq;
        if (t >= p.T) {  // padding token: only its zero scale is stored
          epi_zero_scale(p, t, col);
          continue;
        }
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
        for (int r = 0; r < p.splits; ++r) {
          const uint32_t rr = static_cast<uint32_t>(r);
          const uint32_t base = rr == rank ? stage0 + rank * blk : recv0 + ((rr + p.splits - rank - 1) % p.splits) * blk;
          const float* blkp = sm + (base - sbase) / 4;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int row = 32 * gq + i;
            const float x = blkp[row * per_rank + 4 * ((j >> 2) ^ recv_swizzle(row, cpr)) + (j & 3)];
            v[i] = r == 0 ? x : v[i] + x;
          }
        }
        epi_token_group(p, v, t, col);
      }
    }
  } else {
    // Unsplit K: the accumulator goes to shared memory as [feature][token] (rows padded by 4
    // floats: conflict-free 16-byte writes and 4-byte reads); then every thread finishes whole
    // (token, 32-feature group) items: no shuffles, 16-byte stores.
    constexpr int ps = BN + 4;
    const int f = 32 * q + lane;
    const float* red = reinterpret_cast<const float*>(smem);  // reuses the tile region
    if (epi && !__any_sync(0xffffffffu, *abort_flag)) {
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        uint32_t acc[16];
        tmem_ld_x16(t_lane + 16 * c, acc);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          st_smem_v4(sbase + static_cast<uint32_t>((f * ps + 16 * c + 4 * k) * 4), acc[4 * k], acc[4 * k + 1],
                     acc[4 * k + 2], acc[4 * k + 3]);
      }
    }
    if (epi) named_barrier(1, 128);
    if (epi && !__any_sync(0xffffffffu, *abort_flag)) {
      for (int w = static_cast<int>(threadIdx.x) - 64; w < BN * 4; w += 128) {
        const int j = w & (BN - 1);
        const int gq = w / BN;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = red[(32 * gq + i) * ps + j];
        epi_token_group(p, v, b_row0 + j, static_cast<int64_t>(g) * p.n_feat + m0 + 32 * gq);
      }
    }
  }

  // swap orientation: tiled z scales of padding token rows [BN, ceil(T/128)*128) are zero
  if (SWAP && epi && p.z_sf_tl != nullptr && split == 0 && blockIdx.y == gridDim.y - 1) {
    const int64_t wi = (static_cast<int64_t>(g) * p.n_feat + m0) >> 7;
    for (int64_t t = b_row0 + BN + (static_cast<int>(threadIdx.x) - 64); t < p.z_mp128; t += 128)
      *reinterpret_cast<uint32_t*>(p.z_sf_tl + tiled128x4_word_offset(t, wi, p.z_gp4)) = 0u;
  }

  // ---- teardown: drain own copies / MMAs if a wait gave up, then free TMEM ----
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      for (int i = *consumed_cnt; i < *issued_cnt; ++i) {
        (void)mbar_wait_bounded(bar_full + 8 * (i % STAGES), (i / STAGES) & 1);
        if (CVT) (void)mbar_wait_bounded(bar_act + 8 * (i % STAGES), (i / STAGES) & 1);
      }
    }
    if (warp == 1 && lane == 0) (void)mbar_wait_bounded(bar_accf, 0);
    __syncthreads();
  }
  // bulk path: every copy in the cluster has landed, so no peer still reads this CTA's blocks
  if (recv_path && !C::PUSH) cluster_wait();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------------
// CTA-pair persistent kernel (large T). One tcgen05 MMA of M = 256 tokens x N = 256 features
// spans the two CTAs of a cluster (cta_group::2). Each CTA streams its own 128 token rows and
// 128 of the 256 weight rows: 32 KB of operands per 128-deep k-block and CTA, against 48 KB for
// a 128 x 256 tile on one SM, for the same tensor work per SM. Both CTAs' loads complete on the
// even CTA's stage barriers; the even CTA's MMA warp issues the MMAs, and their commits arrive
// on both CTAs' barriers. Each CTA drains its half of the accumulator (its 128 token rows x 256
// columns, in its own TMEM) with four tcgen05.ld and releases it at once.
// ------------------------------------------------------------------------------------------
// PK: the activation (A) scales arrive int32-packed MN-major: each stage's 128 words of this
// CTA's token rows land in a staging slot on a barrier of the CTA's own, and warp 10 of each CTA
// scatters them into the A atom before the even CTA copies the atoms into TMEM.
template <int STAGES, bool PK = false, bool CV = false>
struct PairCfg {
  static constexpr int A_BYTES = BM * BK;   // this CTA's 128 token rows (E4M3)
  // CV: the A slot receives the 128 x 128 bf16 tile (256-byte rows, no swizzle) and its first
  // 16 KB are overwritten with the E4M3 tile the MMAs read
  static constexpr int A_SLOT = CV ? 2 * A_BYTES : A_BYTES;
  static constexpr int B_BYTES = 128 * BK;  // this CTA's 128 of the 256 weight rows
  static constexpr int SF_BYTES = 512 * 3;  // scale atoms: A (own rows), B (both 128-row atoms)
  // bytes of one stage of both CTAs (counted on the even CTA's barrier) for a tile of n features
  // (with PK the A atoms are not among them: the packed words complete on each CTA's own barrier;
  // with CV neither the A tile nor its atom: the bf16 tile completes on each CTA's own barrier)
  __host__ __device__ static constexpr uint32_t tx_bytes(int n) {
    return CV ? 2u * ((n / 2) * BK + (n / 128) * 512) : 2u * (A_BYTES + (n / 2) * BK + (PK ? 0 : 512) + (n / 128) * 512);
  }
  static constexpr int OFF_B = STAGES * A_SLOT;
  static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_PK = OFF_SF + STAGES * SF_BYTES;  // PK: STAGES x 512 B of packed words
  static constexpr int OFF_EPI = OFF_PK + (PK ? STAGES * 512 : 0);  // 2 KB staging per epilogue warp
  static constexpr int OFF_BAR = OFF_EPI + 8 * 2048;
  // full, empty, scale atoms in TMEM (STAGES each), accf, acce, drain; PK: packed words landed
  // (this CTA) and both CTAs' atoms scattered (even CTA), STAGES each; CV: bf16 tile landed (this
  // CTA), read by the 8 converting warps (this CTA), quantized by both CTAs (even CTA)
  static constexpr int OFF_MISC = OFF_BAR + ((PK ? 5 : CV ? 6 : 3) * STAGES + 4) * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int SF_COLS = 16;
  static constexpr int TMEM_COLS = 512;  // 256 accumulator columns + STAGES x 16 scale columns
  static_assert(256 + STAGES * SF_COLS <= TMEM_COLS, "TMEM");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(!(PK && CV), "one activation form");
};

constexpr int kThreadsPair = 352;  // warp 0 TMA, 1 MMA, 2..9 epilogue, 10 scale copies

// SK: the stream-K tail (p.sk_part / p.sk_flag / p.sk_ticket set); a separate instantiation keeps the
// whole-tile kernel's code exactly as without it. PK: int32-packed activation scales (PairCfg).
// CV: bf16 activations, quantized in the kernel (whole tiles only; see the converting epilogue).
template <int STAGES, bool SK, bool PK = false, bool CV = false>
__global__ void __launch_bounds__(kThreadsPair, 1)
    gemm_mxf8_pair(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_b64, const __grid_constant__ CUtensorMap tm_sfa,
                   const __grid_constant__ CUtensorMap tm_sfb, const KArgs p) {
  static_assert(!(CV && SK), "the converting kernel runs whole tiles");
  using C = PairCfg<STAGES, PK, CV>;
  constexpr int BN = 256;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sraw = smem_u32(smem_raw);
  const uint32_t sbase = (sraw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - sraw);
  const uint32_t bar_full = sbase + C::OFF_BAR;      // stage full (both CTAs' bytes), even CTA only
  const uint32_t bar_empty = bar_full + STAGES * 8;  // stage empty, arrived by the MMA commits
  const uint32_t bar_accf = bar_empty + STAGES * 8;  // accumulator full (MMA -> both epilogues)
  const uint32_t bar_acce = bar_accf + 8;            // accumulator empty (16 epilogue warps), even CTA
  const uint32_t bar_drain = bar_accf + 16;          // abort path: all tcgen05 ops completed
  const uint32_t bar_sf = bar_accf + 24;             // STAGES x 8 B: scale atoms of a stage in TMEM
  const uint32_t bar_pk = bar_sf + STAGES * 8;       // PK: STAGES x 8 B, packed words landed (own)
  const uint32_t bar_scat = bar_pk + STAGES * 8;     // PK: STAGES x 8 B, both atoms scattered (even CTA)
  const uint32_t bar_abf = bar_sf + STAGES * 8;      // CV: STAGES x 8 B, bf16 tile landed (own)
  const uint32_t bar_rd = bar_abf + STAGES * 8;      // CV: STAGES x 8 B, the 8 converting warps have read it
  const uint32_t bar_cvt = bar_rd + STAGES * 8;      // CV: STAGES x 8 B, both CTAs quantized (even CTA)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int* issued_cnt = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);
  int* consumed_cnt = reinterpret_cast<int*>(smem + C::OFF_MISC + 12);
  int* scattered_cnt = reinterpret_cast<int*>(smem + C::OFF_MISC + 16);  // PK; CV: bf16 tiles quantized
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 issues the MMAs
  const bool leader = rank == 0;

  const int n_tiles = p.n_feat / BN;
  const int m_pairs = static_cast<int>((p.T + 2 * BM - 1) / (2 * BM));
  const int per_group = m_pairs * n_tiles;
  const int total = per_group * p.G;
  const int nk = p.kb_per_cta;
  const int first_tile = static_cast<int>(blockIdx.x >> 1), tile_step = static_cast<int>(gridDim.x >> 1);
  // Work items, taken round robin by the pairs: the 256 x 256 tiles of the full waves, then, when
  // the last wave would leave more than half the pairs idle, its tiles as two 256 x 128 halves
  // each, which that wave spreads over twice as many pairs.
  constexpr bool sk = SK;
  const int tail = total % tile_step;
  const bool split_tail = !sk && tail > 0 && 2 * tail <= tile_step;
  const int n_items = split_tail ? total + tail : total;
  // item -> (group, first token of the 256-token pair tile, first feature, features)
  auto item = [&](int i, int& g, int64_t& m0, int64_t& n0, int& nf) {
    int t = i, hf = 0;
    nf = BN;
    if (split_tail && i >= total - tail) {
      const int j = i - (total - tail);
      t = total - tail + (j >> 1);
      hf = j & 1;
      nf = BN / 2;
    }
    g = t / per_group;
    const int r = t - g * per_group;
    m0 = static_cast<int64_t>(r / n_tiles) * (2 * BM);
    n0 = static_cast<int64_t>(r % n_tiles) * BN + hf * (BN / 2);
  };
  // Stream-K mode: all but the last full wave of whole tiles are taken round robin as above (pairs
  // that run at the same time work on neighbouring tiles, which share operands in L2); the
  // k-block iterations of the remaining tiles are cut into one contiguous range per pair,
  // [I * pair / P, I * (pair + 1) / P). Such a range starts inside a tile and may end inside one:
  // its segments are (tile, k-blocks [kb_lo, kb_hi)). Of the pairs that share a tile, the last to
  // finish its MMAs adds the others' partial sums (from the workspace) to its own, in k order
  // (deterministic), and writes the outputs.
  const int pair = static_cast<int>(blockIdx.x >> 1), n_pairs = tile_step;
  // the split tail is the last wave of whole tiles plus the remainder, so that every pair's range
  // covers at least one tile's worth of k-blocks and at most two pairs share a tile
  const int full_waves = sk && total / n_pairs > 0 ? total / n_pairs - 1 : 0;
  const int tail0 = full_waves * n_pairs;  // first tile of the split tail
  const int64_t iters = static_cast<int64_t>(total - tail0) * nk;
  auto range_lo = [&](int q_) { return iters * q_ / n_pairs; };
  const int64_t sk_lo = range_lo(pair), sk_hi = range_lo(pair + 1);
  // segment w of this pair (work item w in round-robin mode); false past the last one
  auto seg = [&](int w, int& t, int& g, int64_t& m0, int64_t& n0, int& nf, int& kb_lo, int& kb_hi) -> bool {
    if (!sk) {
      t = first_tile + w * tile_step;
      if (t >= n_items) return false;
      item(t, g, m0, n0, nf);
      kb_lo = 0;
      kb_hi = nk;
      return true;
    }
    if (w < full_waves) {
      t = pair + w * n_pairs;
      kb_lo = 0;
      kb_hi = nk;
    } else {
      const int64_t tt = sk_lo / nk + (w - full_waves);  // tail tile, counted from tail0
      const int64_t start = w == full_waves ? sk_lo : tt * nk;
      if (start >= sk_hi) return false;
      kb_lo = static_cast<int>(start - tt * nk);
      kb_hi = static_cast<int>(sk_hi - tt * nk < nk ? sk_hi - tt * nk : nk);
      t = tail0 + static_cast<int>(tt);
    }
    g = t / per_group;
    const int r = t - g * per_group;
    m0 = static_cast<int64_t>(r / n_tiles) * (2 * BM);
    n0 = static_cast<int64_t>(r % n_tiles) * BN;
    nf = BN;
    return true;
  };

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_b64);
    tma_prefetch_desc(&tm_sfa);
    tma_prefetch_desc(&tm_sfb);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_accf, 1);
    mbar_init(bar_acce, 16);  // one arrival per epilogue warp of both CTAs
    mbar_init(bar_drain, 2);  // the MMA thread and the scale-copy thread
    for (int s = 0; s < STAGES; ++s) mbar_init(bar_sf + 8 * s, 1);
    if (PK)
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(bar_pk + 8 * s, 1);
        mbar_init(bar_scat + 8 * s, 2);  // warp 10 of each CTA
      }
    if (CV)
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(bar_abf + 8 * s, 1);
        mbar_init(bar_rd + 8 * s, 8);    // the epilogue warps of this CTA
        mbar_init(bar_cvt + 8 * s, 16);  // the epilogue warps of both CTAs
      }
    *abort_flag = 0;
    *issued_cnt = 0;
    *consumed_cnt = 0;
    *scattered_cnt = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any load or commit can reach them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- producer (both CTAs) ----------------
    const uint32_t full0 = mapa_shared(bar_full, 0);  // the even CTA's stage barriers
    int it = 0;
    bool first = true;
    for (int w = 0; !*abort_flag; ++w) {
      int t, g, nf, kb_lo, kb_hi;
      int64_t m0, n0;
      if (!seg(w, t, g, m0, n0, nf, kb_lo, kb_hi)) break;
      const uint32_t tx = C::tx_bytes(nf);
      const int64_t a_row = m0 + BM * rank;  // this CTA's token rows
      const int64_t a_x = static_cast<int64_t>(g) * p.act_k_per_group;
      const int64_t a_atom = (a_row >> 7) * p.act_gp4 + (a_x >> 7);  // scale atom of k-block 0
      const int64_t b_first = static_cast<int64_t>(g) * p.n_feat + n0;
      const int64_t b_row = b_first + (nf / 2) * rank;  // this CTA's nf / 2 weight rows
      const int64_t b_atom = (b_first >> 7) * p.wt_gp4;
      // PK: this CTA's token rows that exist in the packed array (rows >= Mp have no word)
      const int64_t pk_rows = PK ? (p.act_mp4 - a_row < 0 ? 0 : (p.act_mp4 - a_row < BM ? p.act_mp4 - a_row : BM)) : 0;
      auto load_act = [&](int s, int kb, uint32_t fb) {
        if (CV) {  // the bf16 tile, on this CTA's own barrier: this CTA's epilogue warps quantize it
          mbar_arrive_expect_tx(bar_abf + 8 * s, 2u * C::A_BYTES);
          tma_load_2d(sbase + s * C::A_SLOT, &tm_a, bar_abf + 8 * s, static_cast<int32_t>(a_x + kb * BK),
                      static_cast<int32_t>(a_row));
          return;
        }
        tma_load_2d_pair(sbase + s * C::A_SLOT, &tm_a, fb, static_cast<int32_t>(a_x + kb * BK), static_cast<int32_t>(a_row));
        if (!PK) {
          tma_load_2d_pair(sbase + C::OFF_SF + s * C::SF_BYTES, &tm_sfa, fb, 0, static_cast<int32_t>(a_atom + kb));
        } else if (pk_rows > 0) {
          const uint32_t pb = bar_pk + 8 * s;
          mbar_arrive_expect_tx(pb, static_cast<uint32_t>(pk_rows * 4));
          bulk_load(sbase + C::OFF_PK + s * 512, p.act_sf + (((a_x >> 7) + kb) * p.act_mp4 + a_row) * 4,
                    static_cast<uint32_t>(pk_rows * 4), pb);
        } else {
          mbar_arrive(bar_pk + 8 * s);  // no token row of this CTA has scales: an all-zero atom
        }
      };
      auto load_wt = [&](int s, int kb, uint32_t fb) {
        const uint32_t sf = sbase + C::OFF_SF + s * C::SF_BYTES;
        tma_load_2d_pair(sbase + C::OFF_B + s * C::B_BYTES, nf == BN ? &tm_b : &tm_b64, fb,
                         static_cast<int32_t>(kb * BK), static_cast<int32_t>(b_row));
        tma_load_2d_pair(sf + 512, &tm_sfb, fb, 0, static_cast<int32_t>(b_atom + kb));
        if (nf == BN) tma_load_2d_pair(sf + 1024, &tm_sfb, fb, 0, static_cast<int32_t>(b_atom + p.wt_gp4 + kb));
      };
      int kb = kb_lo;
      if (first && p.pdl) {
        const int pre = kb_hi - kb_lo < STAGES ? kb_hi - kb_lo : STAGES;
        for (int j = 0; j < pre; ++j) {
          if (leader) mbar_arrive_expect_tx(bar_full + 8 * j, tx);
          load_wt(j, kb_lo + j, full0 + 8 * j);
        }
        pdl_wait_primary();
        for (int j = 0; j < pre; ++j) load_act(j, kb_lo + j, full0 + 8 * j);
        kb = kb_lo + pre;
        it = pre;
      }
      first = false;
      for (; kb < kb_hi; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!mbar_wait_bounded(bar_empty + 8 * s, ph ^ 1)) {
          *abort_flag = 1;
          report_timeout(p.status);
          break;
        }
        if (leader) mbar_arrive_expect_tx(bar_full + 8 * s, tx);
        load_wt(s, kb, full0 + 8 * s);
        load_act(s, kb, full0 + 8 * s);
      }
    }
    *issued_cnt = it;
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer (even CTA) ----------------
    if (leader) {
      // The MMAs of a stage wait for its scale atoms in TMEM (bar_sf), which warp 10 copies as
      // soon as the stage's operands have landed: the copies are issued by another thread, so
      // this thread's MMA stream never waits behind a copy of its own.
      int it = 0, ti = 0;
      for (int w = 0; !*abort_flag; ++w, ++ti) {
        int t, g, nf, kb_lo, kb_hi;
        int64_t m0, n0;
        if (!seg(w, t, g, m0, n0, nf, kb_lo, kb_hi)) break;
        if (!mbar_wait_bounded(bar_acce, (ti & 1) ^ 1)) {  // both halves drained by the epilogues
          *abort_flag = 1;
          report_timeout(p.status);
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait_bounded(bar_sf + 8 * s, (it / STAGES) & 1)) {
            *abort_flag = 1;
            report_timeout(p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem + BN + s * C::SF_COLS;
          const uint32_t sfb_t = sfa_t + 4;
          const uint64_t ad = sdesc_kmajor_sw128(sbase + s * C::A_SLOT);
          const uint64_t bd = sdesc_kmajor_sw128(sbase + C::OFF_B + s * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            tc_mma_mxf8_pair(tmem, ad + 2 * k, bd + 2 * k, idesc_mxf8(2 * BM, static_cast<uint32_t>(nf), k, k), sfa_t,
                             sfb_t, (kb != kb_lo || k != 0) ? 1u : 0u);
          tc_commit_pair(bar_empty + 8 * s, 0x3);
        }
        tc_commit_pair(bar_accf, 0x3);
        if (!ok) break;
      }
      *consumed_cnt = it;
    }
    pdl_launch_dependents();  // every tile of this pair has been issued
  } else if (warp == 10 && PK) {
    // ---------------- packed scale words -> A atom (both CTAs), then scale copies (even CTA) ----
    // Token row r's word goes to the atom's word (r % 32) * 4 + r / 32: lane l writes the four
    // words of rows l, l + 32, l + 64, l + 96 as one 16-byte store.
    const uint32_t scat0 = mapa_shared(bar_scat, 0);
    int it = 0;
    bool ok = true;
    for (int w = 0; ok; ++w) {
      int t, g, nf, kb_lo, kb_hi;
      int64_t m0, n0;
      if (!seg(w, t, g, m0, n0, nf, kb_lo, kb_hi)) break;
      const int64_t a_row = m0 + BM * rank;
      const int rows = static_cast<int>(p.act_mp4 - a_row < 0 ? 0 : (p.act_mp4 - a_row < BM ? p.act_mp4 - a_row : BM));
      const bool full_tile = nf == BN;
      for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (__any_sync(0xffffffffu, *abort_flag != 0)) {
          ok = false;
          break;
        }
        if (!mbar_wait_bounded(bar_pk + 8 * s, ph)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_timeout(p.status);
          }
          ok = false;
          break;
        }
        const uint32_t* src = reinterpret_cast<const uint32_t*>(smem + C::OFF_PK + s * 512);
        uint32_t wv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) wv[j] = lane + 32 * j < rows ? src[lane + 32 * j] : 0u;
        st_smem_v4(sbase + C::OFF_SF + s * C::SF_BYTES + lane * 16, wv[0], wv[1], wv[2], wv[3]);
        fence_proxy_async_smem();  // the scale copy reads the atom through the async proxy
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(bar_scat + 8 * s);
          else
            mbar_arrive_remote(scat0 + 8 * s);
        }
        if (leader && lane == 0) {
          if (!mbar_wait_bounded(bar_full + 8 * s, ph) || !mbar_wait_bounded(bar_scat + 8 * s, ph)) {
            *abort_flag = 1;
            report_timeout(p.status);
            ok = false;
          } else {
            tc_fence_after();
            const uint32_t sf_src = sbase + C::OFF_SF + s * C::SF_BYTES;
            const uint32_t sfa_t = tmem + BN + s * C::SF_COLS;
            tc_cp_sf_atom_pair(sfa_t, sdesc_sf_atom(sf_src));
            tc_cp_sf_atom_pair(sfa_t + 4, sdesc_sf_atom(sf_src + 512));
            if (full_tile) tc_cp_sf_atom_pair(sfa_t + 8, sdesc_sf_atom(sf_src + 1024));
            tc_commit_pair(bar_sf + 8 * s, 0x1);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
    }
    if (lane == 0) *scattered_cnt = it;
  } else if (warp == 10 && CV) {
    // ---------------- scale copies once both CTAs have quantized the stage (even CTA) --------
    if (leader && lane == 0) {
      int it = 0;
      for (int w = 0; !*abort_flag; ++w) {
        int t, g, nf, kb_lo, kb_hi;
        int64_t m0, n0;
        if (!seg(w, t, g, m0, n0, nf, kb_lo, kb_hi)) break;
        const bool full_tile = nf == BN;
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait_bounded(bar_full + 8 * s, ph) || !mbar_wait_bounded(bar_cvt + 8 * s, ph)) {
            *abort_flag = 1;
            report_timeout(p.status);
            break;
          }
          tc_fence_after();
          const uint32_t sf_src = sbase + C::OFF_SF + s * C::SF_BYTES;
          const uint32_t sfa_t = tmem + BN + s * C::SF_COLS;
          tc_cp_sf_atom_pair(sfa_t, sdesc_sf_atom(sf_src));
          tc_cp_sf_atom_pair(sfa_t + 4, sdesc_sf_atom(sf_src + 512));
          if (full_tile) tc_cp_sf_atom_pair(sfa_t + 8, sdesc_sf_atom(sf_src + 1024));
          tc_commit_pair(bar_sf + 8 * s, 0x1);
        }
      }
    }
  } else if (warp == 10) {
    // ---------------- scale copies (even CTA) ----------------
    if (leader && lane == 0) {
      int it = 0;
      for (int w = 0; !*abort_flag; ++w) {
        int t, g, nf, kb_lo, kb_hi;
        int64_t m0, n0;
        if (!seg(w, t, g, m0, n0, nf, kb_lo, kb_hi)) break;
        const bool full_tile = nf == BN;
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait_bounded(bar_full + 8 * s, (it / STAGES) & 1)) {
            *abort_flag = 1;
            report_timeout(p.status);
            break;
          }
          tc_fence_after();
          const uint32_t sf_src = sbase + C::OFF_SF + s * C::SF_BYTES;
          const uint32_t sfa_t = tmem + BN + s * C::SF_COLS;
          tc_cp_sf_atom_pair(sfa_t, sdesc_sf_atom(sf_src));
          tc_cp_sf_atom_pair(sfa_t + 4, sdesc_sf_atom(sf_src + 512));
          if (full_tile) tc_cp_sf_atom_pair(sfa_t + 8, sdesc_sf_atom(sf_src + 1024));
          tc_commit_pair(bar_sf + 8 * s, 0x1);
        }
      }
    }
  } else if (warp >= 2 && CV) {
    // ---------------- quantize the bf16 A tiles in place, and the epilogue (both CTAs) ---------
    // The 8 epilogue warps quantize every stage of bf16 activations as mxfp8_quantize does: warp
    // ew takes token rows [16 ew, 16 ew + 16) of the CTA's 128, lane l the 16-byte piece l % 16
    // (8 elements) of row 2 j + l / 16 in step j, so that a load instruction covers two whole
    // 256-byte rows; a 32-element group is 4 consecutive lanes (two xor-shuffles for its amax),
    // a scale word 16 lanes. The E4M3 row r (128 bytes, 128-byte swizzle) overwrites bytes of
    // bf16 row r / 2, so every warp reads all its rows first and waits until the other 7 have
    // read theirs. The stages of a tile are quantized before its accumulator is waited for; the
    // first stages of the next tile between the chunks of this tile's epilogue, so that the
    // MMAs of the next tile (which may start once the accumulator has been read) find them.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int ew = warp - 2;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * q) << 16) + 128 * half;
    const uint32_t acce0 = mapa_shared(bar_acce, 0);
    const uint32_t cvt0 = mapa_shared(bar_cvt, 0);
    const uint32_t stage = sbase + C::OFF_EPI + ew * 2048;
    const int pc = lane & 15;
    auto convert = [&](int i) -> bool {
      const int s = i % STAGES;
      const uint32_t ph = (i / STAGES) & 1;
      if (!mbar_wait_bounded(bar_abf + 8 * s, ph)) return false;
      const uint32_t slot = sbase + s * C::A_SLOT;
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = ld_smem_v4(slot + (16 * ew + 2 * j + (lane >> 4)) * 256 + pc * 16);
      uint2 qv[8];
      uint32_t wd[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t amax = absmax8(v[j]);
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const uint32_t code = ue8m0_from_bf16_amax(amax);
        qv[j] = quant8(v[j], ue8m0_inverse(code));
        wd[j] = code | (__shfl_down_sync(0xffffffffu, code, 4) << 8) | (__shfl_down_sync(0xffffffffu, code, 8) << 16) |
                (__shfl_down_sync(0xffffffffu, code, 12) << 24);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_rd + 8 * s);
      if (!mbar_wait_bounded(bar_rd + 8 * s, ph)) return false;
      const uint32_t atom = sbase + C::OFF_SF + s * C::SF_BYTES;  // A atom: first in the slot
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = 16 * ew + 2 * j + (lane >> 4);
        st_smem_v2(slot + r * 128 + (((pc >> 1) ^ (r & 7)) << 4) + 8 * (pc & 1), qv[j].x, qv[j].y);
        if (pc == 0) st_smem_u32(atom + (r & 31) * 16 + (r >> 5) * 4, wd[j]);
      }
      fence_proxy_async_smem();  // the MMAs and the scale copy read these through the async proxy
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(bar_cvt + 8 * s);
        else
          mbar_arrive_remote(cvt0 + 8 * s);
      }
      return true;
    };
    int ti = 0, cit = 0, it_end = 0;
    bool ok = true;
    for (int w = 0; ok; ++w, ++ti) {
      int t, g, nf, kb_lo, kb_hi;
      int64_t m0, n0;
      if (!seg(w, t, g, m0, n0, nf, kb_lo, kb_hi)) break;
      it_end += kb_hi - kb_lo;
      while (ok && cit < it_end)
        if ((ok = convert(cit))) ++cit;
      if (ok && !mbar_wait_bounded(bar_accf, ti & 1)) ok = false;
      if (!ok) {
        *abort_flag = 1;
        report_timeout(p.status);
        break;
      }
      if (__any_sync(0xffffffffu, *abort_flag)) break;
      tc_fence_after();
      const bool cols = 128 * half < nf;  // a 128-feature item has no columns for half 1
      uint32_t hb[4][16];
      if (cols) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t a[32];
          tmem_ld_x32(t_lane + 32 * c, a);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) hb[c][i] = bf16x2_rn(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // the MMA warp may overwrite this half of the accumulator now
        if (leader)
          mbar_arrive(bar_acce);
        else
          mbar_arrive_remote(acce0);
      }
      int nxt = 0;  // stages of the next tile quantized between this epilogue's chunks
      {
        int t1, g1, nf1, kl1, kh1;
        int64_t m1, n1;
        if (seg(w + 1, t1, g1, m1, n1, nf1, kl1, kh1)) nxt = kh1 - kl1 < 4 ? kh1 - kl1 : 4;
      }
      const int64_t row0 = m0 + BM * rank;
      const bool live = cols && row0 < p.z_mp128;  // (this half of a ragged last pair tile holds no token)
      const int64_t col0 = static_cast<int64_t>(g) * p.n_feat + n0 + 128 * half;
      uint32_t word = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (live) epi_hb_chunk_staged(p, hb[c], row0 + 32 * q, lane, col0 + 32 * c, word, c, stage);
        if (c < nxt && ok && (ok = convert(cit))) ++cit;
      }
      if (!ok) {
        *abort_flag = 1;
        report_timeout(p.status);
      }
    }
    if (ew == 0 && lane == 0) *scattered_cnt = cit;
  } else if (warp >= 2) {
    // ---------------- epilogue (both CTAs) ----------------
    const int q = warp & 3;            // TMEM lane quarter
    const int half = (warp - 2) >> 2;  // accumulator columns [128*half, 128*half + 128)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * q) << 16) + 128 * half;
    const uint32_t acce0 = mapa_shared(bar_acce, 0);
    const int ew = warp - 2;  // this warp's share of a partial slot and its ready flag
    const uint32_t stage = sbase + C::OFF_EPI + ew * 2048;
    int ti = 0;
    for (int w = 0;; ++w, ++ti) {
      int t, g, nf, kb_lo, kb_hi;
      int64_t m0, n0;
      if (!seg(w, t, g, m0, n0, nf, kb_lo, kb_hi)) break;
      // A tile of the split tail shared with another pair: take the tile's arrival ticket now,
      // while this segment's MMAs run, so that its latency stays off the epilogue's path (holding
      // a ticket means running, which is all the last holder relies on; see below).
      const bool split_seg = sk && (kb_lo > 0 || kb_hi < nk) && m0 + BM * rank < p.z_mp128 && 128 * half < nf;
      int arrived = 0;
      if (split_seg && lane == 0) arrived = atomicAdd(p.sk_ticket + ((t - tail0) * 2 + static_cast<int>(rank)) * 8 + ew, 1);
      if (!mbar_wait_bounded(bar_accf, ti & 1)) {
        *abort_flag = 1;
        report_timeout(p.status);
      }
      if (__any_sync(0xffffffffu, *abort_flag)) break;
      if (128 * half >= nf) {  // a 128-feature item has no columns for half 1
        if (lane == 0) {
          if (leader)
            mbar_arrive(bar_acce);
          else
            mbar_arrive_remote(acce0);
        }
        continue;
      }
      tc_fence_after();
      const int64_t row0 = m0 + BM * rank;
      const int64_t row = row0 + 32 * q + lane;
      const int64_t col0 = static_cast<int64_t>(g) * p.n_feat + n0 + 128 * half;
      // A warp's share of a split tile is 32 rows x 128 columns. Partial slots are [pair][split
      // segment 0/1][rank][8 warps][32 x 16-byte column groups][32 lanes]: a warp's 16 KB are
      // contiguous and each of its 16-byte stores or loads covers 512 contiguous bytes. Rows past
      // the last token hold zeros on every side and are neither stored nor loaded.
      const bool live = row < p.T;
      if (split_seg) {
        // A tile of the split tail shared with other pairs: its k-blocks lie in the consecutive
        // ranges of pairs [q_lo, q_hi). Every sharer takes a ticket when its segment starts; the
        // last to do so finishes the tile, the others store their partial sums and raise their
        // flag. So nobody waits for a pair that has not started: the finisher waits only for
        // sharers that already hold a ticket, whose MMAs need nothing from anyone.
        const int tt = t - tail0;
        const int64_t k_lo = static_cast<int64_t>(tt) * nk, k_hi = k_lo + nk;
        int q_lo = pair, q_hi = pair + 1;
        while (q_lo > 0 && range_lo(q_lo) > k_lo) --q_lo;
        while (q_hi < n_pairs && range_lo(q_hi) < k_hi) ++q_hi;
        // a pair's split segments: 0 = the first of its range, 1 = the last
        auto unit = [&](int qq) {
          const int j = range_lo(qq) / nk == tt ? 0 : 1;
          return ((qq * 2 + j) * 2 + static_cast<int>(rank)) * 8 + ew;
        };
        auto slot = [&](int qq) { return p.sk_part + static_cast<int64_t>(unit(qq)) * (32 * 32) + lane; };
        int sharers = 0;
        for (int qq = q_lo; qq < q_hi; ++qq) sharers += range_lo(qq + 1) > range_lo(qq) ? 1 : 0;
        int32_t* ticket = p.sk_ticket + (tt * 2 + static_cast<int>(rank)) * 8 + ew;
        arrived = __shfl_sync(0xffffffffu, arrived, 0);
        if (arrived == sharers - 1) {
          bool ok = true;
          for (int qq = q_lo; qq < q_hi && ok; ++qq) {
            if (qq == pair || range_lo(qq + 1) == range_lo(qq)) continue;
            if (lane == 0) ok = wait_flag_gpu(p.sk_flag + unit(qq));
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          }
          if (!ok) {
            if (lane == 0) {
              *abort_flag = 1;
              report_timeout(p.status);
            }
            break;
          }
          // per 32-column chunk: this pair's own sums stay in TMEM until read here; the other
          // sharer's come from its slot, 8 loads in flight. At most two pairs share a tile (every
          // range spans at least one tile's k-blocks), and the sum of two fp32 terms does not
          // depend on their order, so the bytes are the same whichever of the two finishes.
          uint32_t word = 0;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t a[32];
            tmem_ld_x32(t_lane + 32 * c, a);
            tmem_ld_wait();
            for (int qq = q_lo; qq < q_hi && live; ++qq) {
              if (qq == pair || range_lo(qq + 1) == range_lo(qq)) continue;
              const float4* src = slot(qq) + c * 8 * 32;
              float4 u[8];
#pragma unroll
              for (int x = 0; x < 8; ++x) u[x] = __ldcg(src + x * 32);
#pragma unroll
              for (int x = 0; x < 8; ++x) {
                a[4 * x] = __float_as_uint(__uint_as_float(a[4 * x]) + u[x].x);
                a[4 * x + 1] = __float_as_uint(__uint_as_float(a[4 * x + 1]) + u[x].y);
                a[4 * x + 2] = __float_as_uint(__uint_as_float(a[4 * x + 2]) + u[x].z);
                a[4 * x + 3] = __float_as_uint(__uint_as_float(a[4 * x + 3]) + u[x].w);
              }
            }
            epi_row_chunk_staged(p, a, row0 + 32 * q, lane, col0 + 32 * c, word, c, stage);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            for (int qq = q_lo; qq < q_hi; ++qq)
              if (qq != pair && range_lo(qq + 1) > range_lo(qq)) p.sk_flag[unit(qq)] = 0;
            *ticket = 0;  // every sharer has taken its ticket: ready for the next launch
            if (leader)
              mbar_arrive(bar_acce);
            else
              mbar_arrive_remote(acce0);
          }
          continue;
        }
        uint32_t acc[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_x32(t_lane + 32 * c, acc[c]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(bar_acce);
          else
            mbar_arrive_remote(acce0);
        }
        if (live) {
          float4* dst = slot(pair);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int x = 0; x < 8; ++x)
              __stcg(dst + (c * 8 + x) * 32,
                     make_float4(__uint_as_float(acc[c][4 * x]), __uint_as_float(acc[c][4 * x + 1]),
                                 __uint_as_float(acc[c][4 * x + 2]), __uint_as_float(acc[c][4 * x + 3])));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(p.sk_flag + unit(pair), 1);
        continue;
      }
      uint32_t acc[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_x32(t_lane + 32 * c, acc[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // the MMA warp may overwrite this half of the accumulator now
        if (leader)
          mbar_arrive(bar_acce);
        else
          mbar_arrive_remote(acce0);
      }
      if (row0 >= p.z_mp128) continue;  // this half of a ragged last pair tile holds no token
      uint32_t word = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) epi_row_chunk_staged(p, acc[c], row0 + 32 * q, lane, col0 + 32 * c, word, c, stage);
    }
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs have left their loops: issue counts and abort flags are final
  if (PK && warp == 0 && lane == 0) {
    // packed words this CTA loaded but warp 10 did not take: let them land before leaving
    const int peer_abort = ld_dsmem_s32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u));
    if (*abort_flag || peer_abort)
      for (int i = *scattered_cnt; i < *issued_cnt; ++i)
        (void)mbar_wait_bounded(bar_pk + 8 * (i % STAGES), (i / STAGES) & 1);
  }
  if (CV && warp == 0 && lane == 0) {
    // bf16 tiles this CTA loaded but its epilogue warps did not quantize: let them land first
    const int peer_abort = ld_dsmem_s32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u));
    if (*abort_flag || peer_abort)
      for (int i = *scattered_cnt; i < *issued_cnt; ++i)
        (void)mbar_wait_bounded(bar_abf + 8 * (i % STAGES), (i / STAGES) & 1);
  }
  if (leader && warp == 0 && lane == 0) {
    const int peer_abort = ld_dsmem_s32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), 1));
    if (*abort_flag || peer_abort) {
      // wait (bounded) for every stage either CTA issued and the MMA warp did not consume
      const int peer_issued = ld_dsmem_s32(mapa_shared(smem_u32(issued_cnt), 1));
      const int hi = *issued_cnt > peer_issued ? *issued_cnt : peer_issued;
      for (int i = *consumed_cnt; i < hi; ++i)
        (void)mbar_wait_bounded(bar_full + 8 * (i % STAGES), (i / STAGES) & 1);
      *abort_flag = 1;
    }
  }
  __syncthreads();
  if (leader && (warp == 1 || warp == 10) && lane == 0 && *abort_flag) {
    tc_commit_pair(bar_drain, 0x1);  // arrives once every MMA / copy this thread issued has completed
    if (warp == 1) (void)mbar_wait_bounded(bar_drain, 0);
  }
  __syncthreads();
  cluster_sync_all();  // the pair's MMAs and copies are over before either CTA frees TMEM or leaves
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D E4M3 tensor [rows, cols], row stride ld bytes; box = 128 bytes x box_rows, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Dynamic shared memory limit. The L1/shared split stays the driver's choice: forcing the
// largest carveout lets a programmatic dependent's CTAs (wo_b) sit beside wo_a's, where their
// early weight loads slow wo_a more than they save (measured on the T <= 16 pair).
template <typename K>
cudaError_t set_smem_attrs(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Scale atoms of an F8_128x4 array as a 2-D tensor [atoms, 128 x u32]: one 512-byte atom per box.
bool make_sf_map(CUtensorMap* m, const void* base, int64_t atoms) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {128u, static_cast<cuuint64_t>(atoms)};
  cuuint64_t strides[1] = {512u};
  cuuint32_t box[2] = {128u, 1u};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 activations [rows, cols] (row stride ld elements) in boxes of 128 elements x box_rows,
// unswizzled: 256-byte rows in shared memory.
bool make_bf16_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <int BN, int STAGES, int ACT = kActMx>
int ctas_per_sm() {
  using C = Cfg<BN, STAGES, ACT>;
  const int by_smem = C::SM_SMEM / (C::SMEM_LAUNCH + 1024);
  const int by_tmem = 512 / C::TMEM_COLS;
  return by_smem < by_tmem ? by_smem : by_tmem;
}

template <int BN, int STAGES, bool SWAP, int ACT = kActMx, int US = 0>
cudaError_t launch_cfg(const GemmLaunch& l, const KArgs& ka, dim3 grid, int cluster_z, cudaStream_t stream) {
  using C = Cfg<BN, STAGES, ACT>;
  auto kern = gemm_mxf8_kernel<BN, STAGES, SWAP, ACT, US>;
  static const cudaError_t attr_err = set_smem_attrs(kern, C::SMEM_LAUNCH);
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap tma_act, tma_wt;
  if (ACT == kActBf16) {
    if (!make_bf16_map(&tma_act, l.act, l.T, l.act_cols, l.act_ld, SWAP ? BN : BM)) return cudaErrorInvalidValue;
  } else if (!make_map(&tma_act, l.act, l.T, l.act_cols, l.act_ld, SWAP ? BN : BM)) {
    return cudaErrorInvalidValue;
  }
  if (!make_map(&tma_wt, l.wt, static_cast<int64_t>(l.G) * l.n_feat, l.k_len, l.wt_ld, SWAP ? BM : BN))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_LAUNCH;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  cfg.numAttrs = 0;
  if (cluster_z > 1) {
    attrs[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attrs[cfg.numAttrs].val.clusterDim.x = 1;
    attrs[cfg.numAttrs].val.clusterDim.y = 1;
    attrs[cfg.numAttrs].val.clusterDim.z = static_cast<unsigned>(cluster_z);
    ++cfg.numAttrs;
  }
  if (ka.pdl) {
    attrs[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  }
  cfg.attrs = attrs;
  if (SWAP) return cudaLaunchKernelEx(&cfg, kern, tma_wt, tma_act, ka);
  return cudaLaunchKernelEx(&cfg, kern, tma_act, tma_wt, ka);
}

// Largest split of the K range (cluster size) that divides the k-blocks, leaves every rank at
// least 4 token columns, fits its staging in shared memory and keeps every CTA resident in one
// wave.
template <int BN, int STAGES, int ACT = kActMx>
int pick_splits(int tiles, int kb_total, int slots) {
  for (int s = 8; s > 1; s >>= 1)
    if (kb_total % s == 0 && BN / s >= 4 && Cfg<BN, STAGES, ACT>::split_fits(s) && tiles * s <= slots) return s;
  return 1;
}

// Clusters of US CTAs of the uneven-split swap-AB kernel that fit on the device at once.
template <int BN, int STAGES, int US, int ACT>
int uneven_clusters_resident() {
  static const int n = [] {
    using C = Cfg<BN, STAGES, ACT>;
    auto kern = gemm_mxf8_kernel<BN, STAGES, true, ACT, US>;
    if (set_smem_attrs(kern, C::SMEM_LAUNCH) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, static_cast<unsigned>(8 * US));
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_LAUNCH;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = static_cast<unsigned>(US);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      return 0;
    }
    return clusters;
  }();
  return n;
}

// The split of K (cluster size) that the MXFP8-input configuration <BN, PLAN> chooses; the
// packed-scale and bf16-input variants take the same one, so that every output sums the same
// partial products in the same order as with MXFP8 input.
template <int BN, int PLAN>
int plan_splits(int tiles, int kb_total) {
  const int slots = num_sms() * ctas_per_sm<BN, PLAN>();
  const int s = pick_splits<BN, PLAN>(tiles, kb_total, slots);
  // The one-CTA-per-SM band (128-token tiles, 6 stages): when the power-of-two split leaves SMs
  // idle and 3 ranks of every tile still fit in one wave, K is cut over 3 ranks. The gate is on
  // the tile and SM counts, not on the operand: at the DeepSeek-V4.1 shapes wo_b (40 tiles: 80
  // CTAs -> 120) takes it, while wo_a (64 tiles: 3 ranks would need 192 CTAs) stays on two.
  if constexpr (BN == 128 && PLAN == 6) {
    constexpr int US = 3;
    constexpr bool fits = BN * 512 + 2048 * ((BN / 4 + US - 1) / US) * (US - 1) <= Cfg<BN, PLAN>::OFF_SF;
    if (fits && s < US && tiles * s < num_sms() && tiles * US <= slots && kb_total >= 2 * US &&
        tiles <= uneven_clusters_resident<BN, PLAN, US, kActMx>())
      return US;
  }
  return s;
}

template <int BN, int STAGES, int ACT = kActMx, int PLAN = STAGES>
cudaError_t launch_swap(const GemmLaunch& l, KArgs ka, cudaStream_t stream) {
  const int tok_tiles = static_cast<int>(ceil_div(l.T, BN));
  const int tiles = l.G * (l.n_feat / BM) * tok_tiles;
  const int kb_total = l.k_len / BK;
  int s = plan_splits<BN, PLAN>(tiles, kb_total);
  if constexpr (BN == 128) {
    constexpr int US = 3;
    constexpr bool fits = BN * 512 + 2048 * ((BN / 4 + US - 1) / US) * (US - 1) <= Cfg<BN, STAGES, ACT>::OFF_SF;
    if (s == US && !fits) s = 2;  // (a configuration with less staging room: the nearest split that fits)
    if (s == US) {
      ka.splits = US;
      ka.kb_per_cta = kb_total;  // all k-blocks: the kernel cuts the uneven ranges
      ka.per_rank_shift = 0;
      dim3 grid(static_cast<unsigned>(l.n_feat / BM), static_cast<unsigned>(tok_tiles), static_cast<unsigned>(l.G * US));
      return launch_cfg<BN, STAGES, true, ACT, US>(l, ka, grid, US, stream);
    }
  }
  while (s > 1 && (!Cfg<BN, STAGES, ACT>::split_fits(s) || kb_total % s != 0 || BN / s < 4)) s >>= 1;
  ka.splits = s;
  ka.kb_per_cta = kb_total / s;
  ka.per_rank_shift = 0;
  while ((1 << ka.per_rank_shift) < BN / s) ++ka.per_rank_shift;
  dim3 grid(static_cast<unsigned>(l.n_feat / BM), static_cast<unsigned>(tok_tiles), static_cast<unsigned>(l.G * s));
  return launch_cfg<BN, STAGES, true, ACT>(l, ka, grid, s, stream);
}

template <int BN, int STAGES, int ACT = kActMx>
cudaError_t launch_normal(const GemmLaunch& l, KArgs ka, cudaStream_t stream) {
  ka.splits = 1;
  ka.kb_per_cta = l.k_len / BK;
  dim3 grid(static_cast<unsigned>(l.n_feat / BN), static_cast<unsigned>(ceil_div(l.T, BM)),
            static_cast<unsigned>(l.G));
  return launch_cfg<BN, STAGES, false, ACT>(l, ka, grid, 1, stream);
}

}  // namespace

// Split workspace per SM pair: partial sums of two segments (the first and last of a pair's
// range) for both CTAs, 128 x 256 fp32 each; their ready flags (2 segments x 2 CTAs x 8 epilogue
// warps); and the arrival tickets of two tail tiles (the tail holds fewer than 2 tiles per pair).
constexpr int64_t kSkSlotBytes = 2 * 2 * 128 * 256 * 4;
constexpr int64_t kSkFlagBytes = 2 * 2 * 8 * 4;
constexpr int64_t kSkTicketBytes = 2 * 2 * 8 * 4;

// Clusters of the pair kernel that fit on the device at once (1 CTA per SM by its shared memory).
template <int STAGES, bool PK>
int pair_clusters_resident() {
  static const int n = [] {
    using C = PairCfg<STAGES, PK>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms()), 1, 1);
    cfg.blockDim = dim3(kThreadsPair, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_mxf8_pair<STAGES, true, PK>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      return 0;
    }
    return clusters;
  }();
  return n;
}

// CTA-pair persistent launch: clusters of two, one CTA per SM, pair tiles of 256 x 256
// CV: bf16 activations quantized in the kernel; whole tiles, the same tiles and order as the
// MXFP8-input launch of the shape (which takes the split tail only for more than 32 k-blocks per
// tile), so that the sums are those of mxfp8_quantize followed by the MXFP8-input GEMM.
template <int STAGES, bool PK = false, bool CV = false>
cudaError_t launch_pair(const GemmLaunch& l, KArgs ka, cudaStream_t stream) {
  using C = PairCfg<STAGES, PK, CV>;
  auto kern = gemm_mxf8_pair<STAGES, false, PK, CV>;
  static const cudaError_t attr_err = set_smem_attrs(kern, C::SMEM_BYTES);
  if (attr_err != cudaSuccess) return attr_err;
  ka.splits = 1;
  ka.kb_per_cta = l.k_len / BK;
  const int64_t tiles = static_cast<int64_t>(l.G) * ceil_div(l.T, 2 * BM) * (l.n_feat / 256);
  const int max_pairs = num_sms() / 2;
  // With fewer tiles than half the pairs, launch two pairs per tile: the kernel then runs every
  // tile as two 256 x 128 halves (its last-wave split), one per pair.
  const int64_t want = 2 * tiles <= max_pairs ? 2 * tiles : tiles;
  int pairs = static_cast<int>(want < max_pairs ? want : max_pairs);
  // Stream-K when a workspace is given and whole tiles would leave a ragged last wave that costs
  // more than the split's fixed cost: every pair that can be resident at once then takes an
  // equal share of the tail's k-block iterations. (Residency is a matter of speed only: a pair
  // never waits for one that has not started, so the launch completes with any number of SMs
  // available.) Whole tiles take floor(tiles / P) waves plus half a tile (the last wave split in
  // two halves) or a whole one; measured: wo_b (64 k-blocks) gains at 1024..4096 tokens, wo_a
  // (32 k-blocks) never does.
  if constexpr (!CV) {
  if (l.workspace != nullptr && tiles % max_pairs != 0) {
    auto kern_sk = gemm_mxf8_pair<STAGES, true, PK>;
    static const cudaError_t attr_err_sk = set_smem_attrs(kern_sk, C::SMEM_BYTES);
    if (attr_err_sk != cudaSuccess) return attr_err_sk;
    const int resident = pair_clusters_resident<STAGES, PK>();
    const int sk_pairs = resident < max_pairs ? resident : max_pairs;
    const int64_t rem = sk_pairs > 0 ? tiles % sk_pairs : 0;
    const double rr_tail = rem == 0 ? 0.0 : (2 * rem <= sk_pairs ? 0.5 : 1.0);
    const double waste_kb = (rr_tail - static_cast<double>(rem) / sk_pairs) * ka.kb_per_cta;
    // (with fewer tiles than pairs a pair holds less than a tile and many pairs share each one:
    // the partials cost more than the split saves, measured at T = 512)
    // Past 8 waves the tail is a small share of the launch: whole tiles then.
    if (sk_pairs >= 2 && tiles >= sk_pairs && tiles <= 8 * sk_pairs && waste_kb > kSkCostKb) {
      uint8_t* ws = static_cast<uint8_t*>(l.workspace);
      ka.sk_part = reinterpret_cast<float4*>(ws);
      ka.sk_flag = reinterpret_cast<int32_t*>(ws + static_cast<int64_t>(max_pairs) * kSkSlotBytes);
      ka.sk_ticket = reinterpret_cast<int32_t*>(ws + static_cast<int64_t>(max_pairs) * (kSkSlotBytes + kSkFlagBytes));
      pairs = sk_pairs;
      kern = kern_sk;
    }
  }
  }
  CUtensorMap tma_act, tma_wt, tma_wt64, tma_sfa, tma_sfb;
  if (CV ? !make_bf16_map(&tma_act, l.act, l.T, l.act_cols, l.act_ld, BM) : !make_map(&tma_act, l.act, l.T, l.act_cols, l.act_ld, BM))
    return cudaErrorInvalidValue;
  if (!make_map(&tma_wt, l.wt, static_cast<int64_t>(l.G) * l.n_feat, l.k_len, l.wt_ld, 128)) return cudaErrorInvalidValue;
  if (!make_map(&tma_wt64, l.wt, static_cast<int64_t>(l.G) * l.n_feat, l.k_len, l.wt_ld, 64)) return cudaErrorInvalidValue;
  // (with packed activation scales or bf16 activations the A atoms are not loaded through this map)
  if (!make_sf_map(&tma_sfa, PK || CV ? l.wt_sf : l.act_sf, PK || CV ? 1 : ceil_div(l.T, 128) * ka.act_gp4))
    return cudaErrorInvalidValue;
  if (!make_sf_map(&tma_sfb, l.wt_sf, ceil_div(static_cast<int64_t>(l.G) * l.n_feat, 128) * ka.wt_gp4))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kThreadsPair, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.numAttrs = 1;
  if (ka.pdl) {
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  cfg.attrs = attrs;
  return cudaLaunchKernelEx(&cfg, kern, tma_act, tma_wt, tma_wt64, tma_sfa, tma_sfb, ka);
}

int64_t split_workspace_bytes() {
  return static_cast<int64_t>(num_sms() / 2) * (kSkSlotBytes + kSkFlagBytes + kSkTicketBytes);
}

cudaError_t launch_gemm(const GemmLaunch& l, cudaStream_t stream) {
  KArgs ka = {};
  ka.T = l.T;
  ka.G = l.G;
  ka.n_feat = l.n_feat;
  ka.act_k_per_group = l.act_k_per_group;
  ka.act_sf = static_cast<const uint8_t*>(l.act_sf);
  ka.act_gp4 = ceil_div(l.act_cols, 128);
  ka.wt_sf = static_cast<const uint8_t*>(l.wt_sf);
  ka.wt_gp4 = ceil_div(l.k_len, 128);
  ka.out_bf16 = static_cast<uint16_t*>(l.out_bf16);
  ka.ldo = l.ldo;
  ka.z_q = static_cast<uint8_t*>(l.z_q);
  ka.ldz = static_cast<int64_t>(l.G) * l.n_feat;
  ka.z_sf_tl = static_cast<uint8_t*>(l.z_sf_tiled);
  ka.z_gp4 = ceil_div(static_cast<int64_t>(l.G) * l.n_feat, 128);
  ka.z_mp128 = ceil_div(l.T, 128) * 128;
  ka.z_sf_pk = static_cast<uint8_t*>(l.z_sf_packed);
  ka.z_mp4 = ceil_div(l.T, 4) * 4;
  ka.status = l.status;
  ka.pdl = l.pdl ? 1 : 0;
  if (l.workspace != nullptr && l.workspace_bytes < split_workspace_bytes()) return cudaErrorInvalidValue;
  // The first stages go out during setup, before the TMEM allocation and the block barrier,
  // except in the decode pair (T <= 16, wo_a followed by its dependent wo_b): standalone calls
  // and larger pairs gained (T = 1: wo_a 12.8 -> 11.9 us, wo_b 15.2 -> 14.2 us; T = 64 pair
  // 30.3 -> 30.0 us), while there the earlier wo_a loads made the pair slower (23.6 -> 24.7 us).
  // A programmatic dependent fetches only weights before its wait, in the producer role.
  ka.early = (!l.pdl && !(l.T <= 16 && l.has_dependent)) ? 1 : 0;
  ka.act_mp4 = ceil_div(l.T, 4) * 4;
  if (l.n_feat % BM != 0 || l.k_len % BK != 0) return cudaErrorInvalidValue;
  // swap-AB (weights on the MMA's M side) while the token count is small: one token tile of
  // N = 16..128, or several 128-token tiles
  // T <= 16: a grid followed by a dependent (wo_a of o_proj_mxfp8) uses 3 stages so that the
  // dependent wo_b CTAs that find room start early and fetch their first weight stages; other
  // grids keep 5 stages, about 14 MB of loads in flight
  if (l.act_is_bf16) {
    // bf16 activations, quantized in the kernel (wo_a of o_proj_mxfp8_from_bf16: a grid that a
    // dependent wo_b follows). The staging slots leave room for fewer stages; the splits are
    // those of the MXFP8-input configuration of the same band.
    constexpr int B = kActBf16;
    if (l.T <= 16) return launch_swap<16, 3, B>(l, ka, stream);
    if (l.T <= 32) return launch_swap<32, 3, B, 5>(l, ka, stream);
    if (l.T <= 64) return launch_swap<64, 2, B, 4>(l, ka, stream);
    if (l.T <= 128) return launch_swap<128, 3, B, 6>(l, ka, stream);
    if (l.T <= kSwapMaxTokens) return launch_swap<128, 3, B, 3>(l, ka, stream);
    if (l.n_feat % 256 == 0) return launch_pair<4, false, true>(l, ka, stream);
    return launch_normal<128, 3, B>(l, ka, stream);
  }
  if (l.act_sf_packed) {  // int32-packed activation scales, moved into atoms in the kernel
    // the same tiles, stages and splits as the F8_128x4 input, so the sums are the same
    constexpr int P = kActPackedSf;
    if (l.T <= 16) return l.has_dependent ? launch_swap<16, 3, P>(l, ka, stream) : launch_swap<16, 5, P>(l, ka, stream);
    if (l.T <= 32) return launch_swap<32, 5, P>(l, ka, stream);
    if (l.T <= 64) return launch_swap<64, 4, P>(l, ka, stream);
    if (l.T <= 128) return launch_swap<128, 6, P>(l, ka, stream);
    if (l.T <= kSwapMaxTokens) return launch_swap<128, 3, P>(l, ka, stream);
    if (l.n_feat % 256 == 0) return launch_pair<6, true>(l, ka, stream);
    return launch_normal<128, 6, P>(l, ka, stream);
  }
  if (l.T <= 16) return l.has_dependent ? launch_swap<16, 3>(l, ka, stream) : launch_swap<16, 5>(l, ka, stream);
  if (l.T <= 32) return launch_swap<32, 5>(l, ka, stream);
  if (l.T <= 64) return launch_swap<64, 4>(l, ka, stream);
  if (l.T <= 128) return launch_swap<128, 6>(l, ka, stream);
  if (l.T <= 256) return launch_swap<128, 3>(l, ka, stream);
  if (l.T <= kSwapMaxTokens) return launch_swap<128, 3>(l, ka, stream);
  if (l.n_feat % 256 == 0) return launch_pair<6>(l, ka, stream);
  return launch_normal<128, 6>(l, ka, stream);
}

}  // namespace mxq
