/*
 * mxq.h -- C ABI of libmxq, the GB300 (sm_103a) MXFP8 activation chain.
 *
 * The operations follow two vLLM pull-request pages:
 *   [MegaAttn]  "[Perf][DSv4.1] MegaAttn: wo_a writes wo_b's MXFP8 input" (vllm#60118)
 *   [KeepMXFP8] "[Perf][DSv4.1] Keep activations MXFP8 between DeepGEMM kernels" (vllm#57977)
 *
 * MXFP8 here means: E4M3 values (OCP FP8, "FN" variant, largest finite 448) with one UE8M0
 * scale byte b (value 2^(b-127)) per 32 consecutive elements along the contraction / row
 * dimension K (the [KeepMXFP8] review fixes one scale for each 32 elements along K). For a group with
 * largest magnitude amax the scale 2^e is the smallest power of two with amax / 2^e <= 448
 * (never below 2^-127; an all-zero group takes byte 0), and each element x is stored as the
 * E4M3 value nearest to x * 2^-e (round to nearest, ties to even, saturating at +-448; the
 * sign of a zero result follows x).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller. The library never
 *     allocates, frees or synchronizes inside a compute call; work is enqueued on `stream`
 *     (a cudaStream_t passed as void*, NULL = the legacy default stream) and returns at once.
 *   - bf16 is IEEE binary32's upper half; E4M3 and UE8M0 are bytes.
 *   - Row strides (ld*) are in ELEMENTS of the tensor's type; every pointer and every row
 *     stride in bytes must be a multiple of 16.
 *   - Argument errors are detected on the host before anything is launched and return a
 *     status other than MXQ_OK; the outputs are then untouched.
 *   - Launch failures return MXQ_ERR_CUDA (cudaGetLastError after the launch).
 *   - Device-side bounded waits that give up (a pipeline stalled for about a second) record
 *     MXQ_ERR_TIMEOUT in the optional `status` word and end the kernel cleanly; read it with
 *     mxq_check_status. Outputs of such a call are undefined.
 *   - Inputs must be finite (NaN/Inf are outside the contract).
 *
 * Scale-factor layouts (the pages name them -- "F8_128x4", "int32-packed", "MN-major" -- but do
 * not print them; these are the byte layouts this library reads and writes):
 *   MXQ_SF_ROWMAJOR_U8   : byte sf[m * Kg + g], Kg = K/32.
 *   MXQ_SF_PACKED_I32_MN : uint32 words, word w of row m holds groups 4w..4w+3 (group 4w+j in
 *                          byte j, little-endian); stored packed[w * Mp + m], Mp = ceil(M/4)*4;
 *                          requires K % 128 == 0. Padding rows hold 0.
 *   MXQ_SF_TILED_128X4   : rows padded to Mp = ceil(M/128)*128, groups to Gp = ceil(Kg/4)*4;
 *                          512-byte tiles of 128 rows x 4 groups in row-tile-major order; row r,
 *                          group c of a tile at byte (r % 32) * 16 + (r / 32) * 4 + c. This is
 *                          the block-scale layout the tensor cores read. Padding holds 0.
 * Buffer sizes: mxq_sf_bytes().
 */
#ifndef MXQ_H_
#define MXQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MXQ_ABI_VERSION 3

#if defined(__GNUC__)
#define MXQ_API __attribute__((visibility("default")))
#else
#define MXQ_API
#endif

typedef enum mxq_status {
  MXQ_OK = 0,
  MXQ_ERR_INVALID_ARG = 1,       /* required pointer NULL, size <= 0, bad layout tag value  */
  MXQ_ERR_UNSUPPORTED_SHAPE = 2, /* K % 32 != 0, packed scales with K % 128 != 0, a GEMM
                                    dimension outside the kernels' tiling (see each call)     */
  MXQ_ERR_MISALIGNED = 3,        /* a pointer or a row stride in bytes not a multiple of 16   */
  MXQ_ERR_LAYOUT = 4,            /* scale layout tag not accepted by this call               */
  MXQ_ERR_CUDA = 5,              /* CUDA error on the host side (launch, attribute, device)  */
  MXQ_ERR_TIMEOUT = 6            /* a device-side bounded wait gave up (from the status word) */
} mxq_status;

typedef enum mxq_sf_layout {
  MXQ_SF_ROWMAJOR_U8 = 0,
  MXQ_SF_PACKED_I32_MN = 1,
  MXQ_SF_TILED_128X4 = 2
} mxq_sf_layout;

/* An MXFP8 operand: E4M3 bytes [rows, cols] row-major with row stride `ld` bytes, and its
 * UE8M0 scales in `sf_layout` (the layout tag keeps producers and consumers of different
 * scale layouts from being mixed, as [KeepMXFP8] "Pieces" requires of its QuantKey). */
typedef struct mxq_mx_tensor {
  const void* data;
  const void* sf;
  int32_t sf_layout;
  int64_t rows;
  int64_t cols;
  int64_t ld;
} mxq_mx_tensor;

/* ABI version of the loaded library (MXQ_ABI_VERSION at build time). */
MXQ_API int mxq_abi_version(void);

/* Static, NUL-terminated name of a status code. */
MXQ_API const char* mxq_status_string(mxq_status s);

/* Name of the CUDA error behind the last MXQ_ERR_CUDA returned on the calling thread. */
MXQ_API const char* mxq_last_error_string(void);

/* Bytes of a scale buffer in `layout` for an [M, K] MXFP8 tensor; 0 if the shape is invalid
 * for that layout (K % 32 != 0, or packed with K % 128 != 0). */
MXQ_API size_t mxq_sf_bytes(int32_t layout, int64_t M, int64_t K);

/* Bytes of the optional device status word that the GEMM calls accept (zero it before use). */
MXQ_API size_t mxq_status_bytes(void);

/* Synchronizes `stream`, then reads the device status word written by earlier calls:
 * MXQ_OK if no bounded wait gave up, MXQ_ERR_TIMEOUT otherwise, MXQ_ERR_CUDA on a CUDA error.
 * This is the only call that synchronizes. */
MXQ_API mxq_status mxq_check_status(const void* status, void* stream);

/*
 * mxfp8_quantize -- the standalone MXFP8 quantize launch ([MegaAttn] Claims: the
 * "mxfp8_quantize kernel" that the fused path drops; [KeepMXFP8] Purpose: the "[q]" launch).
 *
 *   x_bf16       : [M, K] bf16, row stride ldx elements (ldx >= K).
 *   q_e4m3       : [M, K] E4M3 out, row stride ldq bytes (ldq >= K).
 *   sf_rowmajor  : MXQ_SF_ROWMAJOR_U8 scales out, or NULL.
 *   sf_packed_i32: MXQ_SF_PACKED_I32_MN scales out (K % 128 == 0), or NULL.
 *   sf_128x4     : MXQ_SF_TILED_128X4 scales out, or NULL.
 * Any subset of the three scale layouts is written in the same pass (at least one).
 * Requires M >= 1, K >= 32, K % 32 == 0, M * K < 2^40.
 */
MXQ_API mxq_status mxfp8_quantize(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, void* q_e4m3,
                                  int64_t ldq, void* sf_rowmajor, void* sf_packed_i32, void* sf_128x4,
                                  void* stream);

/*
 * rmsnorm_dual_out -- RMSNorm that writes bf16 and MXFP8 at once ([KeepMXFP8] Purpose:
 * "mega_mhc (post+pre+RMSNorm)" emitting bf16 plus "(y_fp8, y_gemm_sf)"; only the RMSNorm part).
 *
 *   y[t, j] = RNE_bf16( (x[t, j] * r_t) * gamma[j] ),  r_t = 1 / sqrt(mean_j x[t, j]^2 + eps)
 * computed in fp32; (y_q, scales) = mxfp8_quantize(y) applied to that bf16 y (bit-identical).
 *
 *   x_bf16 [T, H] (row stride ldx), gamma_bf16 [H], y_bf16 [T, H] out (row stride H),
 *   y_q [T, H] out (row stride H bytes), y_sf_packed_i32 / y_sf_rowmajor / y_sf_128x4: scale
 *   outputs (NULL to skip; at least one).
 * Requires T >= 1, 32 <= H <= 16384, H % 32 == 0 (H % 128 == 0 for the packed layout).
 */
MXQ_API mxq_status rmsnorm_dual_out(const void* x_bf16, const void* gamma_bf16, float eps, int64_t T,
                                    int64_t H, int64_t ldx, void* y_bf16, void* y_q,
                                    void* y_sf_packed_i32, void* y_sf_rowmajor, void* y_sf_128x4,
                                    void* stream);

/*
 * Split workspace of the large-T GEMMs (T > 384). With more than 384 tokens the GEMMs run as
 * 256 x 256 tiles on pairs of SMs; when the tile count is not a multiple of the pairs, the last
 * wave would leave pairs idle. Given a workspace, the k-block iterations of the last wave and the
 * remainder are instead divided evenly over the pairs. At most two pairs then share a tile: each
 * takes an arrival ticket when its MMAs are done, the first stores its fp32 partial sums in the
 * workspace, and the second adds them to its own and writes the outputs. The result does not
 * depend on timing or on which pair finishes, but may differ from the no-workspace result in the
 * last bit of a rounding.
 *
 * Forward progress: no pair ever waits for a pair that has not started (the finisher waits only
 * for a sharer that already holds its ticket and is storing). So a split call completes however
 * few SMs are free for it -- kernels on other streams, an MPS or green-context SM limit -- it
 * only runs slower.
 *
 * mxq_workspace_bytes() is the size for the current device: per SM pair, four 128 KB fp32
 * partial slots (a pair's first and last segment, both CTAs), then 128 bytes of ready flags and
 * 128 bytes of tickets for all pairs (flags and tickets last). The caller owns the buffer
 * (16-byte aligned). It must be zero-filled before its first use; every call that completes
 * leaves its flags and tickets zero again, so it needs no clearing between calls (after a call
 * that reported MXQ_ERR_TIMEOUT, zero it again). Calls that overlap in time (different streams)
 * need separate workspaces; calls ordered on one stream may share one. Within o_proj_mxfp8 and
 * o_proj_mxfp8_from_bf16 it serves wo_b alone (a programmatic dependent launch that overlaps
 * wo_a's end). NULL workspace: whole tiles per pair, no partials.
 */
MXQ_API int64_t mxq_workspace_bytes(void);

/*
 * wo_a_einsum_mxfp8 -- the grouped wo_a einsum of DeepSeek-V4.1's _o_proj ([MegaAttn]
 * Validation: 8 groups, 4096 in, 1024 out), read as tgk,gnk->tgn:
 *   z[t, g*Na + n] = sum_k deq(o)[t, g*Ka + k] * deq(wa)[g*Na + n, k]   (fp32 accumulation)
 * with the fused epilogue of [MegaAttn] Overview/Details: the fp32 result is rounded to bf16
 * and that bf16 z is quantized to MXFP8 in registers (scales in F8_128x4), so no standalone
 * quantize launch is needed. Bytes and scales equal mxfp8_quantize(z_bf16) of the same call.
 *
 *   o  : [T, G*Ka] MXFP8, sf_layout MXQ_SF_TILED_128X4 (scales over the [T, G*Ka] matrix).
 *   wa : [G*Na, Ka] MXFP8, sf_layout MXQ_SF_TILED_128X4.
 *   z_q, z_sf_128x4 : MXFP8 z out ([T, G*Na], row stride G*Na bytes) -- both or neither.
 *   z_sf_packed_i32 : optional second scale layout for z (MXQ_SF_PACKED_I32_MN), or NULL.
 *   z_bf16          : optional bf16 z out ([T, G*Na], row stride G*Na) -- the pre-fusion
 *                     "bf16 z" output, used for validation and the unfused arm; or NULL.
 *   workspace, workspace_bytes : optional split workspace (mxq_workspace_bytes()), or NULL, 0;
 *                     a smaller non-NULL workspace returns MXQ_ERR_INVALID_ARG.
 *   status          : optional device status word (mxq_status_bytes()), or NULL.
 * At least one of z_q / z_bf16. Requires Ka % 128 == 0, Na % 128 == 0, G >= 1, T >= 1.
 */
MXQ_API mxq_status wo_a_einsum_mxfp8(const mxq_mx_tensor* o, const mxq_mx_tensor* wa, int64_t T,
                                     int32_t G, int32_t Na, int32_t Ka, void* z_q, void* z_sf_128x4,
                                     void* z_sf_packed_i32, void* z_bf16, void* workspace,
                                     int64_t workspace_bytes, void* status, void* stream);

/*
 * gemm_mxfp8_bf16 -- the wo_b MXFP8 GEMM ([MegaAttn] Validation: "wo_b 8192 -> 5120"; it
 * consumes the quantized activation as it is):
 *   out[m, n] = RNE_bf16( sum_k deq(a)[m, k] * deq(b)[n, k] )   (fp32 accumulation)
 *   a : [M, K] MXFP8 activations, b : [N, K] MXFP8 weights, both MXQ_SF_TILED_128X4; the
 *       activation scales may also be MXQ_SF_PACKED_I32_MN ([KeepMXFP8] Pieces: the
 *       DeepGEMM-layout consumer), at any M: each stage's packed words are moved into the tensor
 *       cores' layout inside the kernel, with the same tiles and splits, so the result is
 *       bit-identical to the one from F8_128x4 scales.
 *   out_bf16 : [M, N] bf16, row stride ldo elements.
 *   workspace, workspace_bytes : optional split workspace, as in wo_a_einsum_mxfp8.
 * Requires K % 128 == 0, N % 128 == 0, M >= 1.
 */
MXQ_API mxq_status gemm_mxfp8_bf16(const mxq_mx_tensor* a, const mxq_mx_tensor* b, int64_t M, int64_t N,
                                   int64_t K, void* out_bf16, int64_t ldo, void* workspace,
                                   int64_t workspace_bytes, void* status, void* stream);

/*
 * o_proj_mxfp8 -- the fused _o_proj pair ([MegaAttn] Overview): wo_a_einsum_mxfp8 writes z as
 * MXFP8 with F8_128x4 scales, and gemm_mxfp8_bf16 consumes that z directly:
 *   out = wo_b( MXFP8( RNE_bf16( einsum(o, wa) ) ) )
 * Two kernel launches, no standalone quantize launch. Arguments as in the two calls above;
 * z_q / z_sf_128x4 are required (the hand-off buffers), z_sf_packed_i32 and z_bf16 optional.
 * out_bf16 : [T, Nb], row stride Nb. Requires Nb % 128 == 0. The workspace serves wo_b (wo_a,
 *            whose dependent wo_b may start before it ends, runs whole tiles): the call equals
 *            wo_a_einsum_mxfp8 without a workspace followed by gemm_mxfp8_bf16 with it.
 */
MXQ_API mxq_status o_proj_mxfp8(const mxq_mx_tensor* o, const mxq_mx_tensor* wa, const mxq_mx_tensor* wb,
                                int64_t T, int32_t G, int32_t Na, int32_t Ka, int32_t Nb, void* z_q,
                                void* z_sf_128x4, void* z_sf_packed_i32, void* z_bf16, void* out_bf16,
                                void* workspace, int64_t workspace_bytes, void* status, void* stream);

/*
 * mxq_selftest_wait_timeout -- exercises the failure path every kernel shares: one thread waits
 * with the pipelines' bounded mbarrier wait (here limited to limit_us microseconds, 1..10^6) on a
 * barrier nothing arrives on, gives up, and records MXQ_ERR_TIMEOUT in the status word, which
 * mxq_check_status then returns. The context stays usable. No page describes it; it is a
 * diagnostic of this library. status: a zeroed status word (required).
 */
MXQ_API mxq_status mxq_selftest_wait_timeout(int64_t limit_us, void* status, void* stream);

/*
 * mxq_selftest_hold_sms -- a diagnostic of this library (no page describes it): occupies
 * `sm_pairs` pairs of SMs (clusters of two CTAs, each with enough shared memory that no GEMM CTA
 * of this library fits beside it) for hold_us microseconds (1..2,000,000), then returns. Every
 * wait in it is on the clock, so it always ends. Used to check that calls complete while other
 * work holds SMs. Requires 1 <= sm_pairs <= the device's SMs / 2.
 */
MXQ_API mxq_status mxq_selftest_hold_sms(int64_t sm_pairs, int64_t hold_us, void* stream);

/*
 * o_proj_mxfp8_from_bf16 -- the _o_proj pair fed by bf16 o ([KeepMXFP8] Pieces: the wo_a that
 * quantizes its activation in the kernel, "pre-quantized == in-kernel"; Purpose: no quantize
 * launch between the producer of o and its consumer). wo_a loads o as bf16 and quantizes each
 * stage's tile in shared memory with exactly the rule of mxfp8_quantize (its epilogue warps do
 * it), so there is no quantize launch for o either. wo_a runs the tiles and K splits of
 * o_proj_mxfp8's wo_a (swap-AB tiles up to 384 tokens, SM pairs beyond), so z, its scales, the
 * bf16 z and out are bit-identical to mxfp8_quantize(o) followed by o_proj_mxfp8 (same
 * workspace). (Na not a multiple of 256 with T > 384: 128 x 128 tiles on single SMs, and z the
 * same up to the last bit of the bf16 rounding of some sums.) It saves time at small T only
 * (decode); from about 64 tokens on, the standalone quantizer followed by o_proj_mxfp8 is faster,
 * because every feature tile of a group quantizes the same o tile again.
 *   o_bf16 : bf16 [T, G * Ka], row stride ld_o elements (ld_o * 2 a multiple of 16 bytes).
 * Other arguments as in o_proj_mxfp8 (the workspace serves wo_b).
 */
MXQ_API mxq_status o_proj_mxfp8_from_bf16(const void* o_bf16, int64_t ld_o, const mxq_mx_tensor* wa,
                                          const mxq_mx_tensor* wb, int64_t T, int32_t G, int32_t Na, int32_t Ka,
                                          int32_t Nb, void* z_q, void* z_sf_128x4, void* z_sf_packed_i32,
                                          void* z_bf16, void* out_bf16, void* workspace, int64_t workspace_bytes,
                                          void* status, void* stream);

/*
 * o_proj_mxfp8_noalloc -- o_proj_mxfp8 with the z hand-off held in a fixed buffer inside the
 * library, so the caller passes no z buffers and nothing is allocated. The pages have no
 * counterpart: they always hand z over in a caller-owned tensor.
 *
 * For callers that cannot or will not allocate device memory per call: a plain C host with
 * no caching allocator (cudaMalloc / cudaFree synchronize the device, which would stall a
 * decode loop), or a runtime that fixes its device memory at start-up.
 *
 * Arguments as in o_proj_mxfp8 without z_q / z_sf_128x4 / z_sf_packed_i32 / z_bf16. The
 * buffer holds at most MXQ_NOALLOC_Z_BYTES of E4M3 z (T * G * Na bytes) and
 * MXQ_NOALLOC_SF_BYTES of F8_128x4 scales (mxq_sf_bytes(MXQ_SF_TILED_128X4, T, G * Na)); that is
 * T <= 256 for the DeepSeek-V4.1 shapes (G * Na = 8192). Larger shapes return
 * MXQ_ERR_UNSUPPORTED_SHAPE before anything is launched.
 *
 * Nothing in the buffer needs to start at zero: wo_a writes every z byte and scale that wo_b
 * reads in the same call. The first call on a device looks the buffer up
 * (cudaGetSymbolAddress, checked: MXQ_ERR_CUDA on failure); make that first call outside any
 * stream capture. All calls on one device share the one buffer: calls that overlap in time
 * (different streams or threads) race on it, so order them on one stream.
 */
#define MXQ_NOALLOC_Z_BYTES (2u << 20)
#define MXQ_NOALLOC_SF_BYTES (64u << 10)
MXQ_API mxq_status o_proj_mxfp8_noalloc(const mxq_mx_tensor* o, const mxq_mx_tensor* wa, const mxq_mx_tensor* wb,
                                        int64_t T, int32_t G, int32_t Na, int32_t Ka, int32_t Nb, void* out_bf16,
                                        void* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H_ */
