// kv4_device.cuh -- device helpers shared by the kernels of libkv4mla.so:
// inline PTX for mbarriers and the 5th-generation tensor core (tcgen05 MMA,
// tensor memory), shared-memory matrix descriptors, the NVFP4 row
// dequantization and the top-k index resolution.
//
// Row format (numinousmuses "inference-optimizations" README, "4-bit KV
// cache"): 352 bytes = 256 bytes of E2M1 latent codes (byte j holds elements
// 2j in its low nibble and 2j+1 in its high nibble) + 32 E4M3 scales (one
// per 16 latent elements) + 64 E4M3 rope values.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kv4 {

constexpr int kRowBytes = 352;
constexpr int kRowBytesLatent = 288;   // latent-only row: codes + scales, no rope
constexpr int kRowBytesFp8 = 576;      // E4M3 latent + rope (the comparison row)
constexpr int kLatent = 512;
constexpr int kRope = 64;
constexpr int kQk = 576;
constexpr int kPage = 64;
constexpr int kTileKeys = 128;          // keys per MMA tile (the MMA's M)
constexpr int kChunkBytes = kTileKeys * 128;   // one 64-column slab of a tile

constexpr int kDevBadSlot = 1;
constexpr int kDevBadPage = 2;
constexpr int kDevTimeout = 4;

// ---------------------------------------------------------------------------
// small utilities
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void flag_error(int32_t* dev_err, int flag) {
  if (dev_err != nullptr) atomicOr(dev_err, flag);
}

// Byte offset inside a swizzled operand region (base 1024-byte aligned):
// the hardware XORs address bits [4, 4+B) with bits [7, 7+B), B = 3 for the
// 128-byte swizzle, 2 for 64-byte, 1 for 32-byte.
template <int B>
__device__ __forceinline__ uint32_t swizzle(uint32_t off) {
  return off ^ (((off >> 7) & ((1u << B) - 1u)) << 4);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint2 v) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that suspends the thread until the phase completes or about
// hint_ns nanoseconds have passed, instead of returning at once: waiting
// threads then take neither issue slots nor shared-memory bandwidth.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity,
                                                      uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity; gives up after timeout_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// global loads and prefetches of gathered rows
// ---------------------------------------------------------------------------
// 4- and 8-byte loads through the non-coherent path that leave no line in L1
// (every gathered row is read once).
__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_stream_u64(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}
// Ask L2 for the line that holds p; nothing comes back to the thread.
__device__ __forceinline__ void prefetch_l2_line(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---------------------------------------------------------------------------
// proxy / tensor-core fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warpgroup register reallocation: every thread of the warpgroup executes
// it.  An increase draws on the registers the block was launched with, so
// the host checks the kernel's launch register count before using a split.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------------------
// thread-block clusters: rank, cluster-wide barrier, distributed shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every block of the cluster arrives; release/acquire order
// the shared-memory writes before it with the (remote) reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of cluster_sync(), for work in between.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in block `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive (release, cluster scope) on an mbarrier of another block of the
// cluster; `bar_cluster` is its shared::cluster address (cluster_map).
__device__ __forceinline__ void mbar_remote_arrive(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// Arrive on a local mbarrier and announce `bytes` of asynchronous copies
// that will complete on it.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
      ::"r"(bar), "r"(bytes)
      : "memory");
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global memory into this block's shared memory; completes as
// transaction bytes on the block's mbarrier.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from this block's shared memory into another block's of the cluster;
// completes as transaction bytes on that block's mbarrier.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, uint32_t src,
                                                     uint32_t bytes, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst_cluster), "r"(src), "r"(bytes), "r"(bar_cluster)
      : "memory");
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: the kernels are launched so that they may
// start while the previous kernel of the stream is finishing; each waits for
// it (all of its memory operations visible) before its first global access,
// and lets the next kernel start early.  Without the launch attribute both
// are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier among `count` threads (a multiple of 32).
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also returns whether any participant passed true.
__device__ __forceinline__ bool named_sync_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------------------
// tensor memory
// ---------------------------------------------------------------------------
// Allocate ncols (power of two >= 32) TMEM columns; the base address is
// written to shared memory at dst.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp receives
// lane (quarter*32 + i); taddr carries the lane quarter in bits [16, 32).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
               "r"(r[6]), "r"(r[7])
               : "memory");
}

// Load then wait, with the destination registers tied to the wait so that
// no use of them can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld16_sync(uint32_t taddr, uint32_t (&r)[16]) {
  tmem_ld16(taddr, r);
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld8_sync(uint32_t taddr, uint32_t (&r)[8]) {
  tmem_ld8(taddr, r);
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7])
               :
               : "memory");
}

// Two 32-column loads (e.g. two partial accumulators) and one wait.
__device__ __forceinline__ void tmem_ld32x2_sync(uint32_t ta, uint32_t tb, uint32_t (&a)[32],
                                                 uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
        "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]),
        "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]),
        "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]),
        "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]),
        "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]),
        "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]),
        "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]),
        "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]),
        "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
      : "r"(ta), "r"(tb)
      : "memory");
}

// 2^x (MUFU, about 2 ulp; flushes results below 2^-126 to zero).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2(x) (MUFU, about 2 ulp for x in [1, 2]).
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 MMA (kind::f16, bf16 inputs, fp32 accumulator in TMEM)
// ---------------------------------------------------------------------------
enum : uint32_t {
  kSwizzleNone = 0,
  kSwizzle128 = 2,
  kSwizzle64 = 4,
  kSwizzle32 = 6,
};

// Shared-memory matrix descriptor: start address, leading- and stride-
// dimension byte offsets (16-byte units), descriptor version 1, swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes,
                                              uint32_t sbo_bytes, uint32_t swizzle_mode) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swizzle_mode & 7u) << 61;
  return d;
}

// Instruction descriptor for kind::f16: D fp32, A and B both f16 (format 0)
// or both bf16 (format 1), dense, no negation.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, bool a_mn_major,
                                                     bool b_mn_major, bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major,
                                                  bool b_mn_major) {
  return idesc_f16kind(M, N, a_mn_major, b_mn_major, true);
}
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major,
                                                 bool b_mn_major) {
  return idesc_f16kind(M, N, a_mn_major, b_mn_major, false);
}

__device__ __forceinline__ void mma_f16kind(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same MMA with both descriptors given as a base plus a compile-time
// offset (16-byte units), added inside the instruction sequence: the issuing
// thread then holds only the two bases in registers however many MMAs are
// unrolled.
template <uint32_t A_OFF, uint32_t B_OFF>
__device__ __forceinline__ void mma_f16kind_at(uint32_t d_tmem, uint64_t a_base, uint64_t b_base,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 ad, bd;\n\t"
      "add.s64 ad, %1, %5;\n\tadd.s64 bd, %2, %6;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_base), "l"(b_base), "r"(idesc), "r"(accumulate), "n"(A_OFF), "n"(B_OFF)
      : "memory");
}

// Arrive on an mbarrier once every MMA issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// ---------------------------------------------------------------------------
// minifloat conversions (exact)
// ---------------------------------------------------------------------------
// Four E2M1 byte pairs (8 codes) -> four f16x2 (low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) -> f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t h;
  const uint16_t v = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
  return h;
}

// One E4M3 byte -> float (exact).
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  uint32_t h = e4m3x2_to_f16x2(byte & 0xFFu);
  return __half2float(__low2half(*reinterpret_cast<const __half2*>(&h)));
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  __half2 x = *reinterpret_cast<__half2*>(&a);
  __half2 y = *reinterpret_cast<__half2*>(&b);
  __half2 z = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&z);
}

// ---------------------------------------------------------------------------
// row dequantization (to f16: every E2M1 x E4M3 product and every E4M3
// value is exact in f16 -- at most 6 significant bits, magnitudes in
// [2^-10, 2688] -- so the tensor-core operand equals the decoded value)
// ---------------------------------------------------------------------------
// A warp dequantizes one 352-byte row held as 32-bit words: lane l holds
// w_lo = word l (latent elements 8l..8l+7), w_hi = word l+32 (latent
// 256+8l..), w_ex = word l+64 for l < 24 (lanes 0..7: scale bytes 4l..4l+3,
// lanes 8..23: rope bytes 4(l-8)..4(l-8)+3).  Outputs, as f16:
//   lat_lo: latent 8l..8l+7, lat_hi: latent 256+8l..256+8l+7,
//   rope:   rope 4(l-8)..4(l-8)+3 (lanes 8..23 only).
// Every lane of the warp must call this (it shuffles).
// Two f16 values (f16x2, element 0 in the low half) -> two E4M3 bytes
// (element 0 in the low byte), round half to even, saturating at 448.  Via
// fp32, which holds every f16 value exactly.
__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h2) {
  const __half2 h = *reinterpret_cast<const __half2*>(&h2);
  const float lo = __low2float(h), hi = __high2float(h);
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

struct DequantRow {
  uint4 lat_lo, lat_hi;
  uint2 rope;
};

// Per-lane constant for dequant_row_words: the byte selector that picks this
// lane's two scale bytes out of the two shuffled scale words.
__device__ __forceinline__ uint32_t dequant_scale_selector(int lane) {
  const uint32_t b = (lane >> 1) & 3;                     // byte within each word
  return b | ((4 + b) << 4);                              // {lo word byte b, hi word byte b}
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// One latent word (8 E2M1 codes) of a row times its block's scale, as four
// f16x2; the scale word is shuffled from lane src_lane and byte_sel picks
// the block's byte in it, so every lane of the warp must call this.  The
// decode writes a row in three passes (two latent word groups, then rope).
__device__ __forceinline__ uint4 dequant_latent_part(uint32_t w, uint32_t w_ex, int src_lane,
                                                     uint32_t byte_sel) {
  const uint32_t sw = __shfl_sync(0xFFFFFFFFu, w_ex, src_lane);
  const uint32_t s2 = e4m3x2_to_f16x2(prmt(sw, 0u, byte_sel | 0x4440u));   // {s, 0} as f16
  const uint32_t m = (s2 & 0xFFFFu) * 0x00010001u;               // {s, s}
  uint32_t h[4];
  e2m1x8_to_f16x8(w, h);
  return make_uint4(f16x2_mul(h[0], m), f16x2_mul(h[1], m), f16x2_mul(h[2], m),
                    f16x2_mul(h[3], m));
}
// Latent word w (elements 8w..8w+7) of a row whose scale words sit in lanes
// 0..7 of the warp (w_ex): the scale byte of its block (w/2) is byte
// (w/2)%4 of scale word w/8.
__device__ __forceinline__ uint4 dequant_latent_word(uint32_t w, uint32_t w_ex, int word) {
  return dequant_latent_part(w, w_ex, word >> 3, (word >> 1) & 3);
}
__device__ __forceinline__ uint2 dequant_rope(uint32_t w_ex) {
  return make_uint2(e4m3x2_to_f16x2(w_ex & 0xFFFFu), e4m3x2_to_f16x2(w_ex >> 16));
}

__device__ __forceinline__ DequantRow dequant_row_words(uint32_t w_lo, uint32_t w_hi,
                                                        uint32_t w_ex, int lane,
                                                        uint32_t scale_sel) {
  // scale byte of latent block lane/2 lives in word lane/8 (lane lane/8), and
  // that of block 16 + lane/2 in word 4 + lane/8.
  const uint32_t sw_lo = __shfl_sync(0xFFFFFFFFu, w_ex, lane >> 3);
  const uint32_t sw_hi = __shfl_sync(0xFFFFFFFFu, w_ex, 4 + (lane >> 3));
  const uint32_t s_pair = prmt(sw_lo, sw_hi, scale_sel);  // {s_lo byte, s_hi byte}
  const uint32_t s2 = e4m3x2_to_f16x2(s_pair);            // {s_lo, s_hi} as f16
  const uint32_t m_lo = (s2 & 0xFFFFu) * 0x00010001u;     // {s_lo, s_lo}
  const uint32_t m_hi = (s2 >> 16) * 0x00010001u;         // {s_hi, s_hi}

  DequantRow r;
  uint32_t h[4];
  e2m1x8_to_f16x8(w_lo, h);
  r.lat_lo.x = f16x2_mul(h[0], m_lo);
  r.lat_lo.y = f16x2_mul(h[1], m_lo);
  r.lat_lo.z = f16x2_mul(h[2], m_lo);
  r.lat_lo.w = f16x2_mul(h[3], m_lo);
  e2m1x8_to_f16x8(w_hi, h);
  r.lat_hi.x = f16x2_mul(h[0], m_hi);
  r.lat_hi.y = f16x2_mul(h[1], m_hi);
  r.lat_hi.z = f16x2_mul(h[2], m_hi);
  r.lat_hi.w = f16x2_mul(h[3], m_hi);
  r.rope.x = e4m3x2_to_f16x2(w_ex & 0xFFFFu);
  r.rope.y = e4m3x2_to_f16x2(w_ex >> 16);
  return r;
}

// ---------------------------------------------------------------------------
// top-k index -> pool slot (a2)
// ---------------------------------------------------------------------------
// Resolution runs in two stages so that a caller can overlap each dependent
// load with other work:
//   stage 1: top-k position -> page-table index, or -1 when the position is
//            padding (outside [0, l_eff): masked, no error) or the page index
//            is past the table (masked, flagged);
//   stage 2: page-table entry -> slot, or -1 when the entry is negative or the
//            slot is past the pool (masked, flagged).
__device__ __forceinline__ int32_t slot_page_index(int32_t idx, int64_t l_eff, int64_t pt_stride,
                                                   int32_t* dev_err) {
  if (idx < 0 || static_cast<int64_t>(idx) >= l_eff) return -1;
  const int32_t pi = idx >> 6;
  if (pi >= pt_stride) {
    flag_error(dev_err, kDevBadPage);
    return -1;
  }
  return pi;
}

__device__ __forceinline__ int32_t slot_from_page(int32_t page, int32_t idx, int64_t num_slots,
                                                  int32_t* dev_err) {
  const int64_t slot = static_cast<int64_t>(page) * kPage + (idx & (kPage - 1));
  if (page < 0 || slot >= num_slots) {
    flag_error(dev_err, kDevBadPage);
    return -1;
  }
  return static_cast<int32_t>(slot);
}

// Both stages at once: the slot of key k of one query, or -1 when masked.
__device__ __forceinline__ int32_t resolve_slot(const int32_t* __restrict__ topk_row, int k,
                                                int K, int64_t l_eff,
                                                const int32_t* __restrict__ pt_row,
                                                int64_t pt_stride, int64_t num_slots,
                                                int32_t* dev_err) {
  if (k >= K) return -1;
  const int32_t idx = __ldg(topk_row + k);
  const int32_t pi = slot_page_index(idx, l_eff, pt_stride, dev_err);
  if (pi < 0) return -1;
  return slot_from_page(__ldg(pt_row + pi), idx, num_slots, dev_err);
}

}  // namespace kv4
