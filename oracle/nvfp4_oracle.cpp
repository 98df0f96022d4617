// NVFP4 oracle: plain, single-threaded CPU reference of the quantizer and of
// Y = X W^T.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
// CPU baseline of the benchmark may call it; the product path never does.
// It shares no code, header, table or constant with the CUDA library.
//
// What it follows:
//  * The element types: E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa
//    bit; magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6) and E4M3 "fn" (1 sign, 4
//    exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is
//    NaN, largest finite 448), as defined by the OCP Microscaling Formats (MX)
//    v1.0 and OCP 8-bit Floating Point specifications.
//  * The NVFP4 weight format of the imp engine README ("How it works": weights
//    stored in 4 bits and multiplied without being unpacked to 16 bits) and of
//    the engineering-log entry "NVFP4 at the bit level" (four bits and two
//    scales): 16-element blocks along K, one E4M3 scale per block, one fp32
//    scale per tensor.  The scale recipe: tensor scale s = global amax /
//    (6 * 448); block scale = E4M3 round-to-nearest-even of (block amax / 6) / s.
//  * Decode is the memory-bound phase ("1. The big picture", section "Two
//    phases with very different costs"); the matmul here is its plain
//    definition, accumulated in fp64.
//
// Readings where the sources leave a step open (each is a deliberate choice):
//  * All quantizer arithmetic is IEEE fp32, correctly rounded, no contraction:
//    s = g / 2688; t = a / 6; u = t / s; d = dec(sb) * s; q = x / d.
//  * E4M3 and E2M1 rounding is to nearest, ties to the even mantissa, with
//    saturation to the largest finite value (448 and 6).
//  * The sign of an E2M1 code is copied from x (so -0.0 and tiny negatives give
//    code 0x8) except in blocks with d == 0, which are all 0x0.
//  * g == 0 gives s = 0, every block scale 0x00 and every code 0x0.
//  * Element 2i of a row is the low nibble of byte i, element 2i+1 the high one.
//
// Two more weight formats of the imp README's feature matrix (quantisation:
// "NVFP4 (native, the primary path), MXFP4, ... FP8 E4M3 weights"):
//  * MXFP4, as the OCP Microscaling Formats (MX) v1.0 define it: 32-element
//    blocks along K, one E8M0 scale per block (the byte b stands for
//    2^(b - 127); 0xFF is NaN and never produced), E2M1 elements, no tensor
//    scale.  Conversion per the MX specification: shared exponent
//    e = floor(log2(block amax)) - 2 (2 = the largest exponent of E2M1),
//    clamped to [-127, 127]; element code = E2M1(x / 2^e), round to nearest
//    even, saturating at 6.  Readings: an all-zero block takes e = -127
//    (byte 0x00); the sign of a code is copied from x; x / 2^e is one IEEE
//    fp32 division (exact but for underflow far below the E2M1 grid).
//  * FP8 E4M3 weights: one fp32 scale per tensor, s8 = global amax / 448
//    (the same recipe as the NVFP4 tensor scale, with 448 the largest E4M3
//    value), code = E4M3(x / s8), round to nearest even, saturating at 448,
//    sign copied from x; s8 == 0 gives all codes 0x00.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>

namespace {

// ---- element types, from their definitions ---------------------------------

double e2m1_value(uint8_t code) {
  int sign = (code >> 3) & 1;
  int e = (code >> 1) & 3;
  int m = code & 1;
  double mag = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -mag : mag;
}

double e4m3_value(uint8_t byte) {
  int sign = (byte >> 7) & 1;
  int e = (byte >> 3) & 15;
  int m = byte & 7;
  if (e == 15 && m == 7) return std::nan("");
  double mag = (e == 0) ? std::ldexp((double)m, -9) : std::ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -mag : mag;
}

// The non-negative finite E4M3 values, byte 0x00 .. 0x7E, in increasing order.
struct E4M3Table {
  double v[127];
  E4M3Table() { for (int b = 0; b < 127; ++b) v[b] = e4m3_value((uint8_t)b); }
};
const E4M3Table &e4m3_table() { static E4M3Table t; return t; }

// Nearest of a sorted table of non-negative values; ties go to the even index
// (the even mantissa, since index == encoding); above the top saturates.
int nearest_even(const double *v, int n, double x) {
  if (!(x > 0.0)) return 0;                 // 0 (and -0) map to index 0
  if (x >= v[n - 1]) return n - 1;          // saturate (satfinite)
  int hi = (int)(std::upper_bound(v, v + n, x) - v);  // v[hi-1] <= x < v[hi]
  int lo = hi - 1;
  double dl = x - v[lo], dh = v[hi] - x;
  if (dl < dh) return lo;
  if (dh < dl) return hi;
  return (lo % 2 == 0) ? lo : hi;
}

uint8_t e4m3_encode_nonneg(float u) {
  return (uint8_t)nearest_even(e4m3_table().v, 127, (double)u);
}

uint8_t e2m1_encode_mag(float q) {
  static const double v[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  if (std::isinf(q)) return 7;
  return (uint8_t)nearest_even(v, 8, (double)q);
}

float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// volatile stores keep each fp32 operation a separately rounded IEEE op.
float div_rn(float a, float b) { volatile float r = a / b; return r; }
float mul_rn(float a, float b) { volatile float r = a * b; return r; }

// One row of K elements with tensor scale s -> K/2 code bytes, K/16 scales.
void quantize_row(const uint16_t *x, int64_t K, float s, uint8_t *codes, uint8_t *scales) {
  for (int64_t b = 0; b < K / 16; ++b) {
    float xs[16];
    float a = 0.0f;
    for (int j = 0; j < 16; ++j) {
      xs[j] = bf16_to_f32(x[16 * b + j]);
      a = std::max(a, std::fabs(xs[j]));
    }
    float u = 0.0f;
    if (s != 0.0f) {
      float t = div_rn(a, 6.0f);
      u = div_rn(t, s);
    }
    uint8_t sb = e4m3_encode_nonneg(u);
    scales[b] = sb;
    float d = mul_rn((float)e4m3_value(sb), s);
    uint8_t c[16];
    for (int j = 0; j < 16; ++j) {
      if (d == 0.0f) { c[j] = 0; continue; }
      float q = div_rn(xs[j], d);
      uint8_t sign = std::signbit(xs[j]) ? 8 : 0;
      c[j] = (uint8_t)(sign | e2m1_encode_mag(std::fabs(q)));
    }
    for (int j = 0; j < 8; ++j) codes[8 * b + j] = (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));
  }
}

// ---- MXFP4 ------------------------------------------------------------------

double e8m0_value(uint8_t b) {
  if (b == 255) return std::nan("");
  return std::ldexp(1.0, (int)b - 127);
}

// Shared exponent of a block with largest magnitude a (finite, >= 0).
int mx_shared_exponent(float a) {
  if (a == 0.0f) return -127;
  int ex;
  std::frexp((double)a, &ex);  // a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
  int e = (ex - 1) - 2;
  return std::min(127, std::max(-127, e));
}

void mx_quantize_row(const uint16_t *x, int64_t K, uint8_t *codes, uint8_t *scales) {
  for (int64_t b = 0; b < K / 32; ++b) {
    float xs[32];
    float a = 0.0f;
    for (int j = 0; j < 32; ++j) {
      xs[j] = bf16_to_f32(x[32 * b + j]);
      a = std::max(a, std::fabs(xs[j]));
    }
    const int e = mx_shared_exponent(a);
    scales[b] = (uint8_t)(e + 127);
    const float X = std::ldexp(1.0f, e);  // 2^e, exact (2^-127 is a subnormal float)
    uint8_t c[32];
    for (int j = 0; j < 32; ++j) {
      float q = div_rn(xs[j], X);
      uint8_t sign = std::signbit(xs[j]) ? 8 : 0;
      c[j] = (uint8_t)(sign | e2m1_encode_mag(std::fabs(q)));
    }
    for (int j = 0; j < 16; ++j) codes[16 * b + j] = (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));
  }
}

// ---- FP8 E4M3 weights -------------------------------------------------------

void fp8_quantize_row(const uint16_t *x, int64_t K, float s, uint8_t *codes) {
  for (int64_t k = 0; k < K; ++k) {
    if (s == 0.0f) { codes[k] = 0; continue; }
    float v = bf16_to_f32(x[k]);
    float q = div_rn(v, s);
    uint8_t sign = std::signbit(v) ? 0x80 : 0;
    codes[k] = (uint8_t)(sign | e4m3_encode_nonneg(std::fabs(q)));
  }
}

}  // namespace

extern "C" {

double orc_e2m1_value(uint8_t code) { return e2m1_value(code); }
double orc_e4m3_value(uint8_t byte) { return e4m3_value(byte); }
uint8_t orc_e4m3_encode(float u) { return e4m3_encode_nonneg(u); }
uint8_t orc_e2m1_encode(float q) {
  uint8_t sign = std::signbit(q) ? 8 : 0;
  return (uint8_t)(sign | e2m1_encode_mag(std::fabs(q)));
}

// Global amax g = max |x| over rows x K (ld = row stride in elements) and the
// tensor scale s = g / 2688.  Returns 1 if any element is NaN or Inf, else 0.
int orc_tensor_scale(const uint16_t *x, int64_t rows, int64_t K, int64_t ld, float *amax,
                     float *tensor_scale) {
  float g = 0.0f;
  int nonfinite = 0;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < K; ++k) {
      float v = bf16_to_f32(x[r * ld + k]);
      if (!std::isfinite(v)) nonfinite = 1;
      else g = std::max(g, std::fabs(v));
    }
  *amax = g;
  *tensor_scale = div_rn(g, 2688.0f);
  return nonfinite;
}

// Quantize `rows` rows (row stride ld) with a given tensor scale s.
void orc_quantize_rows(const uint16_t *x, int64_t rows, int64_t K, int64_t ld, float s,
                       uint8_t *codes, uint8_t *scales) {
  for (int64_t r = 0; r < rows; ++r)
    quantize_row(x + r * ld, K, s, codes + r * (K / 2), scales + r * (K / 16));
}

// Whole-tensor quantizer: tensor scale, then every row.  Returns 1 on
// non-finite input (outputs then unspecified), else 0.
int orc_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ld, uint8_t *codes,
                 uint8_t *scales, float *tensor_scale) {
  float g;
  int bad = orc_tensor_scale(x, rows, K, ld, &g, tensor_scale);
  orc_quantize_rows(x, rows, K, ld, *tensor_scale, codes, scales);
  return bad;
}

// Dequantize rows: w[r][k] = e2m1(code) * e4m3(scale) * s, in fp64 (exact).
void orc_dequant(const uint8_t *codes, const uint8_t *scales, float s, int64_t rows,
                 int64_t K, double *out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = codes[r * (K / 2) + k / 2];
      uint8_t c = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
      out[r * K + k] = e2m1_value(c) * e4m3_value(scales[r * (K / 16) + k / 16]) * (double)s;
    }
}

double orc_e8m0_value(uint8_t b) { return e8m0_value(b); }

// MXFP4 quantizer: codes [rows][K/2], E8M0 scales [rows][K/32].  Returns 1
// if any element is NaN or Inf (outputs then unspecified), else 0.
int orc_mx_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ld, uint8_t *codes,
                    uint8_t *scales) {
  int bad = 0;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t k = 0; k < K; ++k)
      if (!std::isfinite(bf16_to_f32(x[r * ld + k]))) bad = 1;
    mx_quantize_row(x + r * ld, K, codes + r * (K / 2), scales + r * (K / 32));
  }
  return bad;
}

// MXFP4 dequant: w[r][k] = e2m1(code) * 2^(scale - 127), fp64 (exact).
void orc_mx_dequant(const uint8_t *codes, const uint8_t *scales, int64_t rows, int64_t K,
                    double *out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = codes[r * (K / 2) + k / 2];
      uint8_t c = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
      out[r * K + k] = e2m1_value(c) * e8m0_value(scales[r * (K / 32) + k / 32]);
    }
}

// FP8 tensor scale s8 = g / 448.  Returns 1 on NaN/Inf, else 0.
int orc_fp8_tensor_scale(const uint16_t *x, int64_t rows, int64_t K, int64_t ld, float *s8) {
  float g = 0.0f;
  int bad = 0;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < K; ++k) {
      float v = bf16_to_f32(x[r * ld + k]);
      if (!std::isfinite(v)) bad = 1;
      else g = std::max(g, std::fabs(v));
    }
  *s8 = div_rn(g, 448.0f);
  return bad;
}

// FP8 codes [rows][K] with a given tensor scale.
void orc_fp8_quantize_rows(const uint16_t *x, int64_t rows, int64_t K, int64_t ld, float s,
                           uint8_t *codes) {
  for (int64_t r = 0; r < rows; ++r) fp8_quantize_row(x + r * ld, K, s, codes + r * K);
}

// FP8 dequant: w = e4m3(code) * s, fp64 (exact).
void orc_fp8_dequant(const uint8_t *codes, float s, int64_t n, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]) * (double)s;
}

// bf16 bit patterns -> fp64.
void orc_bf16_to_f64(const uint16_t *x, int64_t n, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (double)bf16_to_f32(x[i]);
}

// y[m][n] = sum_k a[m][k] * b[n][k] and bound[m][n] = sum_k |a[m][k] * b[n][k]|,
// both accumulated in fp64 in increasing k.
void orc_matmul_abt(const double *a, int64_t M, const double *b, int64_t N, int64_t K,
                    double *y, double *bound) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = a[m * K + k] * b[n * K + k];
        acc += p;
        mag += std::fabs(p);
      }
      y[m * N + n] = acc;
      if (bound) bound[m * N + n] = mag;
    }
}

}  // extern "C"
