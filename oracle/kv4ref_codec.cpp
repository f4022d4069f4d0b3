/*
 * kv4ref_codec.cpp -- oracle codecs for the 352-byte NVFP4 KV row.
 *
 * TEST INFRASTRUCTURE ONLY (see kv4ref.h).
 *
 * Source: numinousmuses "inference-optimizations" README, section
 * "4-bit KV cache", GLM-5.3 4-bit KV bullet: a 352-byte NVFP4 row holding
 * E2M1 values with one E4M3 scale per 16 values, replacing the 576-byte FP8
 * row.  The page does not spell out the formats; the two minifloats are the
 * standard ones:
 *   E4M3 ("fn" flavour): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
 *     infinities, largest finite 448, subnormal step 2^-9.
 *   E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
 *     {0, .5, 1, 1.5, 2, 3, 4, 6}.
 * Both encoders round to nearest, ties to even mantissa, and saturate to the
 * largest finite magnitude.  Rounding is done exactly in double precision:
 * every fp32 input and every grid value is exact there, and dividing by a
 * power of two is exact.
 */
#include "kv4ref.h"

#include <cmath>
#include <cstdint>
#include <cstring>

namespace {

/* Magnitude of a minifloat code (sign stripped). */
double minifloat_value(uint32_t mag, int mbits, int bias) {
  const uint32_t e = mag >> mbits;
  const uint32_t m = mag & ((1u << mbits) - 1u);
  if (e == 0) return std::ldexp(static_cast<double>(m), 1 - bias - mbits);
  return std::ldexp(static_cast<double>((1u << mbits) + m),
                    static_cast<int>(e) - bias - mbits);
}

/* Round a >= 0 to the minifloat grid (RNE) and return the magnitude code,
 * saturating at max_mag. */
uint32_t minifloat_encode_mag(double a, int mbits, int bias, uint32_t max_mag) {
  if (a == 0.0) return 0;
  if (a >= minifloat_value(max_mag, mbits, bias)) return max_mag;
  const int emin = 1 - bias;              /* exponent of the smallest normal */
  int ex = 0;
  std::frexp(a, &ex);                     /* a = f * 2^ex, f in [0.5, 1)    */
  int e = ex - 1;                         /* floor(log2(a))                  */
  if (e < emin) e = emin;                 /* subnormals share emin's step    */
  const double step = std::ldexp(1.0, e - mbits);
  const double n = std::nearbyint(a / step);  /* exact quotient; RNE         */
  int64_t N = static_cast<int64_t>(n);
  if (N == 0) return 0;
  uint32_t ecode, mant;
  if (N >= (int64_t(1) << mbits)) {       /* normal                          */
    if (N == (int64_t(1) << (mbits + 1))) { N >>= 1; e += 1; }  /* carry     */
    ecode = static_cast<uint32_t>(e + bias);
    mant = static_cast<uint32_t>(N - (int64_t(1) << mbits));
  } else {                                /* subnormal (e == emin)           */
    ecode = 0;
    mant = static_cast<uint32_t>(N);
  }
  uint32_t code = (ecode << mbits) | mant;
  if (code > max_mag) code = max_mag;
  return code;
}

inline float bf16_to_float(uint16_t h) {
  uint32_t bits = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return f;
}

}  // namespace

extern "C" {

uint8_t kv4ref_enc_e4m3(float x) {
  const uint32_t sign = std::signbit(x) ? 0x80u : 0u;
  const uint32_t mag =
      minifloat_encode_mag(std::fabs(static_cast<double>(x)), 3, 7, 0x7Eu);
  return static_cast<uint8_t>(sign | mag);
}

float kv4ref_dec_e4m3(uint8_t c) {
  const double v = minifloat_value(c & 0x7Fu, 3, 7);
  return static_cast<float>((c & 0x80u) ? -v : v);
}

uint8_t kv4ref_enc_e2m1(float x) {
  const uint32_t sign = std::signbit(x) ? 0x8u : 0u;
  const uint32_t mag =
      minifloat_encode_mag(std::fabs(static_cast<double>(x)), 1, 1, 0x7u);
  return static_cast<uint8_t>(sign | mag);
}

float kv4ref_dec_e2m1(uint8_t c) {
  const double v = minifloat_value(c & 0x7u, 1, 1);
  return static_cast<float>((c & 0x8u) ? -v : v);
}

void kv4ref_enc_e4m3_n(const float* x, uint8_t* codes, int64_t n) {
  for (int64_t i = 0; i < n; ++i) codes[i] = kv4ref_enc_e4m3(x[i]);
}

void kv4ref_enc_e2m1_n(const float* x, uint8_t* codes, int64_t n) {
  for (int64_t i = 0; i < n; ++i) codes[i] = kv4ref_enc_e2m1(x[i]);
}

void kv4ref_quantize_row(const uint16_t* latent_bf16, const uint16_t* rope_bf16,
                         uint8_t* row) {
  uint8_t codes[512];
  for (int blk = 0; blk < 32; ++blk) {
    float x[16];
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
      x[i] = bf16_to_float(latent_bf16[blk * 16 + i]);
      const float a = std::fabs(x[i]);
      if (a > amax) amax = a;
    }
    const float s_f = amax / 6.0f;                 /* IEEE fp32 division */
    const uint8_t s8 = kv4ref_enc_e4m3(s_f);
    const float s = kv4ref_dec_e4m3(s8);
    row[256 + blk] = s8;
    for (int i = 0; i < 16; ++i) {
      if (s == 0.0f) {
        codes[blk * 16 + i] = 0;                   /* all-zero block */
      } else {
        const float r = x[i] / s;                  /* IEEE fp32 division */
        codes[blk * 16 + i] = kv4ref_enc_e2m1(r);
      }
    }
  }
  for (int j = 0; j < 256; ++j)
    row[j] = static_cast<uint8_t>(codes[2 * j] | (codes[2 * j + 1] << 4));
  for (int r = 0; r < 64; ++r)
    row[288 + r] = kv4ref_enc_e4m3(bf16_to_float(rope_bf16[r]));
}

void kv4ref_dequant_row(const uint8_t* row, float* out576) {
  for (int d = 0; d < 512; ++d) {
    const uint8_t byte = row[d / 2];
    const uint8_t code = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    const float s = kv4ref_dec_e4m3(row[256 + d / 16]);
    out576[d] = kv4ref_dec_e2m1(code) * s;          /* exact product */
  }
  for (int r = 0; r < 64; ++r) out576[512 + r] = kv4ref_dec_e4m3(row[288 + r]);
}

void kv4ref_quantize_row_mse(const uint16_t* latent_bf16, const uint16_t* rope_bf16,
                             uint8_t* row) {
  uint8_t codes[512];
  for (int blk = 0; blk < 32; ++blk) {
    float x[16];
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
      x[i] = bf16_to_float(latent_bf16[blk * 16 + i]);
      const float a = std::fabs(x[i]);
      if (a > amax) amax = a;
    }
    const int c0 = kv4ref_enc_e4m3(amax / 6.0f);     /* the amax/6 scale byte */
    const int lo = c0 - 8 < 0 ? 0 : c0 - 8;
    const int hi = c0 + 1 > 126 ? 126 : c0 + 1;
    int best_c = -1;
    float best_err = 0.0f;
    uint8_t best_codes[16] = {0};
    for (int c = lo; c <= hi; ++c) {
      const float s = kv4ref_dec_e4m3(static_cast<uint8_t>(c));
      uint8_t cand[16];
      float err = 0.0f;
      for (int i = 0; i < 16; ++i) {
        cand[i] = (s == 0.0f) ? 0 : kv4ref_enc_e2m1(x[i] / s);
        const float d = x[i] - kv4ref_dec_e2m1(cand[i]) * s;   /* product exact */
        err = err + d * d;
      }
      if (best_c < 0 || err < best_err) {
        best_c = c;
        best_err = err;
        for (int i = 0; i < 16; ++i) best_codes[i] = cand[i];
      }
    }
    row[256 + blk] = static_cast<uint8_t>(best_c);
    for (int i = 0; i < 16; ++i) codes[blk * 16 + i] = best_codes[i];
  }
  for (int j = 0; j < 256; ++j)
    row[j] = static_cast<uint8_t>(codes[2 * j] | (codes[2 * j + 1] << 4));
  for (int r = 0; r < 64; ++r)
    row[288 + r] = kv4ref_enc_e4m3(bf16_to_float(rope_bf16[r]));
}

int kv4ref_quantize_write_mse(const uint16_t* latent_bf16, int64_t latent_stride,
                              const uint16_t* rope_bf16, int64_t rope_stride,
                              const int64_t* slot_mapping, int64_t n_tokens,
                              uint8_t* pool, int64_t num_slots) {
  if (n_tokens < 0 || num_slots < 0) return KV4REF_ERR_ARG;
  if (n_tokens > 0 && (!latent_bf16 || !rope_bf16 || !slot_mapping || !pool))
    return KV4REF_ERR_ARG;
  if (latent_stride < 512 || rope_stride < 64) return KV4REF_ERR_ARG;
  int status = KV4REF_OK;
  for (int64_t t = 0; t < n_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_slots) { status = KV4REF_ERR_SLOT; continue; }
    kv4ref_quantize_row_mse(latent_bf16 + t * latent_stride,
                            rope_bf16 + t * rope_stride, pool + slot * 352);
  }
  return status;
}

int kv4ref_quantize_write_fp8(const uint16_t* latent_bf16, int64_t latent_stride,
                              const uint16_t* rope_bf16, int64_t rope_stride,
                              const int64_t* slot_mapping, int64_t n_tokens,
                              uint8_t* pool, int64_t num_slots) {
  if (n_tokens < 0 || num_slots < 0) return KV4REF_ERR_ARG;
  if (n_tokens > 0 && (!latent_bf16 || !rope_bf16 || !slot_mapping || !pool))
    return KV4REF_ERR_ARG;
  if (latent_stride < 512 || rope_stride < 64) return KV4REF_ERR_ARG;
  int status = KV4REF_OK;
  for (int64_t t = 0; t < n_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_slots) { status = KV4REF_ERR_SLOT; continue; }
    uint8_t* row = pool + slot * 576;
    for (int d = 0; d < 512; ++d)
      row[d] = kv4ref_enc_e4m3(bf16_to_float(latent_bf16[t * latent_stride + d]));
    for (int r = 0; r < 64; ++r)
      row[512 + r] = kv4ref_enc_e4m3(bf16_to_float(rope_bf16[t * rope_stride + r]));
  }
  return status;
}

void kv4ref_dequant_row_fp8(const uint8_t* row, float* out576) {
  for (int d = 0; d < 576; ++d) out576[d] = kv4ref_dec_e4m3(row[d]);
}

int kv4ref_quantize_write(const uint16_t* latent_bf16, int64_t latent_stride,
                          const uint16_t* rope_bf16, int64_t rope_stride,
                          const int64_t* slot_mapping, int64_t n_tokens,
                          uint8_t* pool, int64_t num_slots) {
  if (n_tokens < 0 || num_slots < 0) return KV4REF_ERR_ARG;
  if (n_tokens > 0 && (!latent_bf16 || !rope_bf16 || !slot_mapping || !pool))
    return KV4REF_ERR_ARG;
  if (latent_stride < 512 || rope_stride < 64) return KV4REF_ERR_ARG;
  int status = KV4REF_OK;
  for (int64_t t = 0; t < n_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_slots) { status = KV4REF_ERR_SLOT; continue; }
    kv4ref_quantize_row(latent_bf16 + t * latent_stride,
                        rope_bf16 + t * rope_stride, pool + slot * 352);
  }
  return status;
}

}  // extern "C"
