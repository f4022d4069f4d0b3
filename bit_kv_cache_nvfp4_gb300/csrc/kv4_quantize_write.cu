// kv4_quantize_write.cu -- the NVFP4 cache write (numinousmuses
// "inference-optimizations" README, "4-bit KV cache": the quantized write of
// the 352-byte row).
//
// One warp per token.  Lane i owns latent block i (elements 16i..16i+15):
// it loads 32 bytes, takes the block's amax, rounds amax/6 to an E4M3 scale
// (IEEE fp32 division, round half to even, saturating), divides each element
// by the decoded scale (IEEE fp32 division) and rounds to E2M1 (round half
// to even, saturating, sign kept).  A zero scale gives zero codes.  Lanes
// 0..7 also convert 8 rope values each to E4M3.  The row is written with
// coalesced stores: codes as 32 x 8 bytes, scales as 8 x 4 bytes, rope as
// 8 x 8 bytes.  Each warp loads its next token while it codes the current
// one.  Bytes: 1152 read, 352 written per token; at 1M tokens the IEEE
// divisions (17 per lane and token) rather than HBM bound the kernel.  Rows of 288 bytes (the latent-only layout of the same README
// section, for models whose keys carry no rope part) are the first 288
// bytes of the same row: no rope is read or written.  With a.fp8 the row is
// the 576-byte FP8 row the NVFP4 row replaces (E4M3 of every latent and rope
// value, no scale), for the comparison paths.
//
// With a.mse set, each block's scale is searched instead (README "4-bit KV
// cache", DeepSeek V4 Pro bullet: "an MSE-searched scale"; the search rule
// is this project's reading): the candidates are the E4M3 scale bytes
// c0-8 .. c0+1 around c0 = E4M3(amax/6) (clipped to 0..126); each gives codes
// E2M1(x/s) and the error sum_i (x_i - dec(code_i) s)^2 in IEEE fp32, in
// element order with every operation rounded separately; the smallest error
// wins, the lowest scale byte on ties.
#include "kv4_device.cuh"
#include "kv4_launch.h"

namespace kv4 {
namespace {

__device__ __forceinline__ float bf16_low(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_high(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// E4M3 of two floats, round half to even, saturating: hi -> high byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight floats -> four bytes of E2M1 pairs; element 2i goes to the low
// nibble of byte i.
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float (&r)[8]) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(r[0]), "f"(r[1]), "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]),
        "f"(r[7]));
  return out;
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// E2M1 magnitude of a 4-bit code's low three bits: 0, 0.5, 1, 1.5, 2, 3, 4, 6
// (two exponent bits with bias 1, one mantissa bit; exponent 0 subnormal).
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  const uint32_t e = (code >> 1) & 3u, m = code & 1u;
  const float mag = e == 0 ? 0.5f * static_cast<float>(m)
                           : __uint_as_float((126u + e) << 23) * (1.0f + 0.5f * static_cast<float>(m));
  return (code & 8u) ? -mag : mag;
}

// Squared reconstruction error of a block coded as (w0, w1) with scale s,
// summed in element order with each operation rounded to nearest.
__device__ __forceinline__ float block_error(const float (&x)[16], uint32_t w0, uint32_t w1,
                                             float s) {
  float err = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t w = i < 8 ? w0 : w1;
    const uint32_t code = (w >> (4 * (i & 7))) & 0xFu;
    const float d = __fsub_rn(x[i], __fmul_rn(e2m1_value(code), s));
    err = __fadd_rn(err, __fmul_rn(d, d));
  }
  return err;
}

__global__ void __launch_bounds__(256) quantize_write_kernel(QuantizeArgs a) {
  // the previous kernel (e.g. a decode still gathering from the pool) must
  // be complete before any row is written
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const __nv_bfloat16* latent = static_cast<const __nv_bfloat16*>(a.latent);
  const __nv_bfloat16* rope = static_cast<const __nv_bfloat16*>(a.rope);

  // The loads of a warp's next token are issued before the current token is
  // processed (slot, latent and rope of a token are independent loads), so
  // every warp keeps one token's reads in flight while it computes.
  struct TokenLoads {
    int64_t slot;
    uint4 v0, v1, rv;
  };
  auto load = [&](int64_t tt, TokenLoads& l) {
    l.slot = __ldg(a.slots + tt);
    const __nv_bfloat16* src = latent + tt * a.latent_stride + lane * 16;
    l.v0 = ld_stream(src);
    l.v1 = ld_stream(src + 8);
    l.rv = (rope != nullptr && lane < 8) ? ld_stream(rope + tt * a.rope_stride + lane * 8)
                                         : make_uint4(0, 0, 0, 0);
  };
  TokenLoads next{};
  if (warp0 < a.n_tokens) load(warp0, next);
  for (int64_t t = warp0; t < a.n_tokens; t += nwarps) {
    const TokenLoads cur = next;
    if (t + nwarps < a.n_tokens) load(t + nwarps, next);
    const int64_t slot = cur.slot;
    if (slot < 0) continue;                               // warp-uniform
    if (slot >= a.num_slots) {
      if (lane == 0) flag_error(a.dev_err, kDevBadSlot);
      continue;
    }
    const uint4 v0 = cur.v0;
    const uint4 v1 = cur.v1;
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    if (a.fp8) {
      // 576-byte FP8 row: every latent and rope value as E4M3 (no scale)
      uint8_t* row = a.pool + slot * a.row_bytes;
      uint32_t b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        b[i] = f32x2_to_e4m3x2(bf16_high(w[2 * i]), bf16_low(w[2 * i])) |
               (f32x2_to_e4m3x2(bf16_high(w[2 * i + 1]), bf16_low(w[2 * i + 1])) << 16);
      *reinterpret_cast<uint4*>(row + lane * 16) = make_uint4(b[0], b[1], b[2], b[3]);
      if (lane < 8) {
        const uint4 rv = cur.rv;
        const uint32_t lo = f32x2_to_e4m3x2(bf16_high(rv.x), bf16_low(rv.x)) |
                            (f32x2_to_e4m3x2(bf16_high(rv.y), bf16_low(rv.y)) << 16);
        const uint32_t hi = f32x2_to_e4m3x2(bf16_high(rv.z), bf16_low(rv.z)) |
                            (f32x2_to_e4m3x2(bf16_high(rv.w), bf16_low(rv.w)) << 16);
        *reinterpret_cast<uint2*>(row + 512 + lane * 8) = make_uint2(lo, hi);
      }
      continue;
    }
    float x[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = bf16_low(w[i]);
      x[2 * i + 1] = bf16_high(w[i]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    uint32_t s8 = f32x2_to_e4m3x2(0.0f, __fdiv_rn(amax, 6.0f)) & 0xFFu;
    // codes of the block for scale byte sb (all zero when it decodes to 0)
    auto encode = [&](uint32_t sb, uint32_t& w0, uint32_t& w1) {
      const float s = e4m3_to_float(sb);
      w0 = w1 = 0;
      if (s != 0.0f) {
        float r[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) r[i] = __fdiv_rn(x[i], s);
        w0 = f32x8_to_e2m1x8(r);
#pragma unroll
        for (int i = 0; i < 8; ++i) r[i] = __fdiv_rn(x[8 + i], s);
        w1 = f32x8_to_e2m1x8(r);
      }
      return s;
    };
    uint32_t c0 = 0, c1 = 0;
    if (!a.mse) {
      encode(s8, c0, c1);
    } else {
      const uint32_t lo = s8 >= 8 ? s8 - 8 : 0, hi = s8 + 1 < 126 ? s8 + 1 : 126;
      float best = 0.0f;
      uint32_t best_sb = 0xFFFFFFFFu;
      for (uint32_t sb = lo; sb <= hi; ++sb) {
        uint32_t w0, w1;
        const float s = encode(sb, w0, w1);
        const float err = block_error(x, w0, w1, s);
        if (best_sb == 0xFFFFFFFFu || err < best) {
          best = err;
          best_sb = sb;
          c0 = w0;
          c1 = w1;
        }
      }
      s8 = best_sb;
    }
    uint8_t* row = a.pool + slot * a.row_bytes;
    *reinterpret_cast<uint2*>(row + lane * 8) = make_uint2(c0, c1);

    // scale bytes: lane i holds byte i; lanes 0..7 write word k = bytes 4k..4k+3
    const uint32_t b0 = __shfl_sync(0xFFFFFFFFu, s8, (lane * 4 + 0) & 31);
    const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, s8, (lane * 4 + 1) & 31);
    const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, s8, (lane * 4 + 2) & 31);
    const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, s8, (lane * 4 + 3) & 31);
    if (lane < 8) {
      *reinterpret_cast<uint32_t*>(row + 256 + lane * 4) = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    }
    if (lane < 8 && rope != nullptr) {
      const uint4 rv = cur.rv;
      const uint32_t lo = f32x2_to_e4m3x2(bf16_high(rv.x), bf16_low(rv.x)) |
                          (f32x2_to_e4m3x2(bf16_high(rv.y), bf16_low(rv.y)) << 16);
      const uint32_t hi = f32x2_to_e4m3x2(bf16_high(rv.z), bf16_low(rv.z)) |
                          (f32x2_to_e4m3x2(bf16_high(rv.w), bf16_low(rv.w)) << 16);
      *reinterpret_cast<uint2*>(row + 288 + lane * 8) = make_uint2(lo, hi);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_write(const QuantizeArgs& a, int num_sms, cudaStream_t stream) {
  if (a.n_tokens <= 0) return cudaSuccess;
  const int64_t warps_needed = a.n_tokens;
  int64_t blocks = (warps_needed + 7) / 8;
  // at most one wave of resident blocks; each warp then walks its tokens
  static int per_sm = 0;
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_write_kernel, 256, 0) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    (void)cudaGetLastError();
  }
  const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * per_sm;
  if (blocks > cap) blocks = cap;
  // Same shared-memory carve-out as the decode kernel, which usually follows
  // in the stream: the SMs then need no reconfiguration between the two.
  static const cudaError_t carveout = cudaFuncSetAttribute(
      quantize_write_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
      cudaSharedmemCarveoutMaxShared);
  (void)carveout;
  return launch_pdl(quantize_write_kernel, static_cast<unsigned>(blocks), 256, 0, stream, 1, a);
}

}  // namespace kv4
