// MXFP8 activation-chain ORACLE — test infrastructure, not product code.
//
// A plain, slow, obviously-correct CPU statement of what the GPU library computes, used only
// by tests/, by __graft_entry__.smoke() and by bench.py's cpu_baseline / --impl reference legs.
// It shares no code, header, table or constant with the CUDA path and never calls it.
//
// Sources (vLLM pull-request pages):
//   [P3] "[Perf][DSv4.1] MegaAttn: wo_a writes wo_b's MXFP8 input" (vllm#60118),
//        sections Overview, Claims, Validation, Details.
//   [P4] "[Perf][DSv4.1] Keep activations MXFP8 between DeepGEMM kernels" (vllm#57977),
//        section Purpose (before/after diagrams, per-layer table, Pieces) and the review's
//        one scale for each 32 elements along K.
// The pages name MXFP8 (OCP FP8 E4M3 values + UE8M0 power-of-two scales per 32 elements) but
// do not define it; every reading taken where they are silent is listed at its function.
//
// Arithmetic is fp64 throughout. Every product of an E4M3 value and a power of two is exact
// in fp64, so the quantizer below is exact; the GEMMs accumulate in fp64 in plain k order.

#include <cmath>
#include <cstdint>
#include <cstring>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ----------------------------------------------------------------------------------------
// bf16: the upper 16 bits of an IEEE binary32.
// ----------------------------------------------------------------------------------------
double bf16_value(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// Round an fp64 value to the nearest bf16, ties to even (one rounding, straight from fp64).
// bf16 has 8 significant bits and binary32's exponent range: normal numbers step by
// 2^(E-7) inside the binade [2^E, 2^(E+1)), and below 2^-126 the step is 2^-133.
uint16_t bf16_round(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const bool neg = std::signbit(x);
  double a = std::fabs(x);
  double step;
  if (a >= std::ldexp(1.0, -126)) {
    int e = std::ilogb(a);
    step = std::ldexp(1.0, e - 7);
  } else {
    step = std::ldexp(1.0, -133);
  }
  double r = std::nearbyint(a / step) * step;  // a/step is exact (power-of-two divide)
  const double bf16_max = std::ldexp(255.0, 120);  // (2 - 2^-7) * 2^127
  uint16_t bits;
  if (r > bf16_max) {
    bits = 0x7F80;  // overflow to infinity under round-to-nearest
  } else {
    float f = static_cast<float>(r);  // r is exactly representable in bf16, hence binary32
    uint32_t u;
    std::memcpy(&u, &f, 4);
    bits = static_cast<uint16_t>(u >> 16);
  }
  return neg ? static_cast<uint16_t>(bits | 0x8000) : bits;
}

// ----------------------------------------------------------------------------------------
// E4M3 ("FN" variant of OCP FP8): sign, 4 exponent bits (bias 7), 3 mantissa bits.
// Exponent field 0 holds subnormals (m/8)*2^-6; field 15 with mantissa 7 is NaN; no
// infinities. Largest finite value 448 (0x7E), smallest normal 2^-6, smallest subnormal 2^-9.
// ----------------------------------------------------------------------------------------
double e4m3_value(uint8_t c) {
  const int s = c >> 7, E = (c >> 3) & 0xF, m = c & 7;
  if (E == 15 && m == 7) return std::nan("");
  double mag = (E == 0) ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, E - 7);
  return s ? -mag : mag;
}

// Encode an exact real q (held in fp64) to E4M3: round to nearest, ties to the code whose
// mantissa LSB is even, saturating to +-448. Reading (pages silent): the sign of a zero
// result follows q, as IEEE rounding does; NaN encodes as 0x7F.
uint8_t e4m3_encode(double q) {
  if (std::isnan(q)) return 0x7F;
  const uint8_t sign = std::signbit(q) ? 0x80 : 0x00;
  const double a = std::fabs(q);
  if (a >= 448.0) return sign | 0x7E;
  uint8_t mag;
  if (a < std::ldexp(1.0, -6)) {
    // subnormal binade: multiples of 2^-9; a count of 8 is the smallest normal (code 0x08)
    double n = std::nearbyint(a / std::ldexp(1.0, -9));
    mag = static_cast<uint8_t>(n);
  } else {
    int e = std::ilogb(a);                                 // a in [2^e, 2^(e+1)), e in [-6, 8]
    double n = std::nearbyint(a / std::ldexp(1.0, e - 3));  // in [8, 16]
    int ex = e, mant = static_cast<int>(n) - 8;
    if (mant == 8) { ex += 1; mant = 0; }
    int code = ((ex + 7) << 3) | mant;
    if (code > 0x7E) code = 0x7E;
    mag = static_cast<uint8_t>(code);
  }
  return sign | mag;
}

// UE8M0: an 8-bit biased exponent; byte b means 2^(b-127) (b = 255 is NaN, never produced).
// The rule of the method: the scale 2^e takes the smallest integer e with amax / 2^e <= 448
// (the largest finite E4M3 value), and no smaller than the smallest UE8M0 value 2^-127.
// An all-zero group (amax 0) satisfies every e and therefore takes byte 0.
uint8_t ue8m0_from_amax(double amax) {
  if (!(amax > 0.0)) return 0;
  int e = std::ilogb(amax) - 9;  // amax / 2^e >= 2^9 > 448: too small, walk upward
  while (amax > std::ldexp(448.0, e)) ++e;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return static_cast<uint8_t>(e + 127);
}

inline double scale_value(uint8_t b) { return std::ldexp(1.0, static_cast<int>(b) - 127); }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

int orc_abi_version(void) { return 1; }

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

// ---- element-wise formats ---------------------------------------------------------------
void orc_bf16_to_f64(const uint16_t* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_value(x[i]);
}
void orc_f64_to_bf16(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_round(x[i]);
}
void orc_e4m3_decode(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(c[i]);
}
void orc_e4m3_encode(const double* q, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(q[i]);
}
void orc_ue8m0_from_amax(const double* amax, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ue8m0_from_amax(amax[i]);
}

// ---- group quantizer ----------------------------------------------------------------------
// x: bf16 [M, K] with row stride ldx elements; K % 32 == 0. Groups are 32 consecutive
// elements along K (one scale for each 32 elements, per the review). For each group: amax = max |x_i|,
// byte b = ue8m0_from_amax(amax), e = b - 127, q_i = E4M3(x_i * 2^-e).
// Outputs q [M, K] (row stride K) and row-major scales sf [M, K/32].
void orc_quantize_bf16(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                       uint8_t* sf) {
  const int64_t Kg = K / 32;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t g = 0; g < Kg; ++g) {
      double v[32];
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) {
        v[i] = bf16_value(x[m * ldx + g * 32 + i]);
        amax = std::fmax(amax, std::fabs(v[i]));
      }
      const uint8_t b = ue8m0_from_amax(amax);
      sf[m * Kg + g] = b;
      const int e = static_cast<int>(b) - 127;
      for (int i = 0; i < 32; ++i) q[m * K + g * 32 + i] = e4m3_encode(std::ldexp(v[i], -e));
    }
  }
}

// ---- scale layouts (the pages name them; the byte layouts are this library's reading) ------
// Row-major: sf[m * Kg + g].
//
// int32-packed, MN-major: word w of row m holds the scales of groups 4w..4w+3, group 4w+j in
// byte j (little-endian significance). Words are stored column-major: packed[w * Mp + m] with
// Mp = ceil(M/4)*4 so each column of words starts on a 16-byte boundary; padding rows are 0.
// Requires Kg % 4 == 0.
void orc_sf_pack_i32(const uint8_t* sf, int64_t M, int64_t Kg, uint32_t* packed) {
  const int64_t Mp = ceil_div(M, 4) * 4, W = Kg / 4;
  for (int64_t w = 0; w < W; ++w)
    for (int64_t m = 0; m < Mp; ++m) {
      uint32_t word = 0;
      if (m < M)
        for (int j = 0; j < 4; ++j) word |= static_cast<uint32_t>(sf[m * Kg + 4 * w + j]) << (8 * j);
      packed[w * Mp + m] = word;
    }
}
void orc_sf_unpack_i32(const uint32_t* packed, int64_t M, int64_t Kg, uint8_t* sf) {
  const int64_t Mp = ceil_div(M, 4) * 4;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t g = 0; g < Kg; ++g) sf[m * Kg + g] = (packed[(g / 4) * Mp + m] >> (8 * (g % 4))) & 0xFF;
}

// F8_128x4: rows padded to Mp = ceil(M/128)*128, groups to Gp = ceil(Kg/4)*4. The scales
// form 512-byte tiles of 128 rows x 4 groups, tiles ordered row-tile major. Inside a tile,
// row r and group c sit at byte (r % 32) * 16 + (r / 32) * 4 + c. Padding is byte 0.
int64_t orc_sf_128x4_bytes(int64_t M, int64_t Kg) { return ceil_div(M, 128) * 128 * ceil_div(Kg, 4) * 4; }

void orc_sf_to_128x4(const uint8_t* sf, int64_t M, int64_t Kg, uint8_t* out) {
  const int64_t Mp = ceil_div(M, 128) * 128, Gp = ceil_div(Kg, 4) * 4;
  for (int64_t r = 0; r < Mp; ++r)
    for (int64_t g = 0; g < Gp; ++g) {
      const int64_t tile = (r / 128) * (Gp / 4) + g / 4;
      const int64_t rr = r % 128, c = g % 4;
      const int64_t off = tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + c;
      out[off] = (r < M && g < Kg) ? sf[r * Kg + g] : 0;
    }
}
void orc_sf_from_128x4(const uint8_t* in, int64_t M, int64_t Kg, uint8_t* sf) {
  const int64_t Gp = ceil_div(Kg, 4) * 4;
  for (int64_t r = 0; r < M; ++r)
    for (int64_t g = 0; g < Kg; ++g) {
      const int64_t tile = (r / 128) * (Gp / 4) + g / 4;
      const int64_t rr = r % 128, c = g % 4;
      sf[r * Kg + g] = in[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + c];
    }
}

// ---- dequantize and contract ------------------------------------------------------------
// deq[m, k] = E4M3(q[m, k]) * 2^(sf[m, k/32] - 127), exact in fp64.
void orc_dequant(const uint8_t* q, const uint8_t* sf, int64_t M, int64_t K, double* out) {
  const int64_t Kg = K / 32;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t k = 0; k < K; ++k) out[m * K + k] = e4m3_value(q[m * K + k]) * scale_value(sf[m * Kg + k / 32]);
}

// C[m, n] = sum_k A[m, k] * B[n, k]   (both operands K-contiguous, fp64, k in order)
void orc_gemm_nt(const double* A, const double* B, int64_t M, int64_t N, int64_t K, double* C) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      const double* a = A + m * K;
      const double* b = B + n * K;
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k) s += a[k] * b[k];
      C[m * N + n] = s;
    }
}

// The wo_a grouped einsum (8 groups, 4096 in, 1024 out) read as tgk,gnk->tgn:
//   z[t, g*Na + n] = sum_k o[t, g*Ka + k] * wa[g*Na + n, k]
// o: [T, G*Ka]; wa: [G*Na, Ka]; z: [T, G*Na] (g-major flattening of [T, G, Na]).
void orc_einsum_wo_a(const double* o, const double* wa, int64_t T, int64_t G, int64_t Na, int64_t Ka,
                     double* z) {
#pragma omp parallel for collapse(3) schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t g = 0; g < G; ++g)
      for (int64_t n = 0; n < Na; ++n) {
        const double* a = o + t * G * Ka + g * Ka;
        const double* b = wa + (g * Na + n) * Ka;
        double s = 0.0;
        for (int64_t k = 0; k < Ka; ++k) s += a[k] * b[k];
        z[t * G * Na + g * Na + n] = s;
      }
}

// ---- RMSNorm ------------------------------------------------------------------------------
// y[t, j] = x[t, j] * gamma[j] / sqrt(mean_j(x[t, j]^2) + eps), in fp64 (eps inside the root).
void orc_rmsnorm(const uint16_t* x, const uint16_t* gamma, double eps, int64_t T, int64_t H, int64_t ldx,
                 double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int64_t j = 0; j < H; ++j) {
      const double v = bf16_value(x[t * ldx + j]);
      ss += v * v;
    }
    const double r = 1.0 / std::sqrt(ss / static_cast<double>(H) + eps);
    for (int64_t j = 0; j < H; ++j) y[t * H + j] = bf16_value(x[t * ldx + j]) * bf16_value(gamma[j]) * r;
  }
}

}  // extern "C"
