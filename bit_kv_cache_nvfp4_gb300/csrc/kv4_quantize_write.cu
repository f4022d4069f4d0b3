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
// 8 x 8 bytes.  The kernel is HBM-bound (1152 bytes read, 352 written per
// token).  Rows of 288 bytes (the latent-only layout of the same README
// section, for models whose keys carry no rope part) are the first 288
// bytes of the same row: no rope is read or written.
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

  for (int64_t t = warp0; t < a.n_tokens; t += nwarps) {
    const int64_t slot = __ldg(a.slots + t);
    if (slot < 0) continue;                               // warp-uniform
    if (slot >= a.num_slots) {
      if (lane == 0) flag_error(a.dev_err, kDevBadSlot);
      continue;
    }
    const __nv_bfloat16* src = latent + t * a.latent_stride + lane * 16;
    const uint4 v0 = ld_stream(src);
    const uint4 v1 = ld_stream(src + 8);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float x[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = bf16_low(w[i]);
      x[2 * i + 1] = bf16_high(w[i]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const uint32_t s8 = f32x2_to_e4m3x2(0.0f, __fdiv_rn(amax, 6.0f)) & 0xFFu;
    const float s = e4m3_to_float(s8);
    uint32_t c0 = 0, c1 = 0;
    if (s != 0.0f) {
      float r[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) r[i] = __fdiv_rn(x[i], s);
      c0 = f32x8_to_e2m1x8(r);
#pragma unroll
      for (int i = 0; i < 8; ++i) r[i] = __fdiv_rn(x[8 + i], s);
      c1 = f32x8_to_e2m1x8(r);
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
      const uint4 rv = ld_stream(rope + t * a.rope_stride + lane * 8);
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
  const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 16;
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
