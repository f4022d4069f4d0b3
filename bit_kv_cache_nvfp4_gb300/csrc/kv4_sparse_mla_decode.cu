// kv4_sparse_mla_decode.cu -- sparse MLA decode over the NVFP4 latent KV
// pool on the 5th-generation tensor core (numinousmuses
// "inference-optimizations" README: "4-bit KV cache" kv4mla bullet -- the
// 4-bit rows are dequantized in shared memory instead of an FP8 scratch copy
// in HBM; "Attention kernels" split-K sparse decode bullet; "Parallelism and
// disaggregation" (o, lse) merge).
//
// Work unit: one thread block per (request b, draft token s, head group g,
// split).  A head group holds HG = min(H, 64) query heads, which all share
// every gathered row.  The block (8 compute warps and one MMA-issue
// warpgroup) splits into its two roles at once; the issuer stages Q with one
// bulk copy while the compute warps resolve the slots of the first two tiles,
// convert Q and gather tile 0, then the block walks its share of the top-k
// list in tiles of 128 keys:
//   a2     slots are resolved two tiles ahead (top-k -> page table -> slot),
//          each dependent load spread over a tile's work; as soon as a
//          tile's slots are known its rows are prefetched into L2
//   a3     each warp gathers 16 rows of the next tile into registers (three
//          coalesced 4-byte loads per lane and row, without L1 allocation)
//          while QK runs
//   a4     and dequantizes them straight into the 128-byte-swizzled f16
//          operand tile in shared memory (576 columns per key; E2M1 x E4M3
//          and E4M3 values are exact in f16) in three passes -- latent
//          slabs 0-3, latent slabs 4-7, rope -- each into the
//          slabs that the previous tile's PV has already released; q is
//          converted to f16 with a per-head power-of-two scale folded into
//          the score scale
//   a5     as each pass lands, the QK issuer (lane 0 of warp 8) issues its
//          part of S^T[128 x HG] = K_tile . Q^T on tcgen05 (M = 128 keys,
//          N = HG, K = 576) into an fp32 TMEM accumulator
//   a6     the 8 compute warps read S from TMEM (one key per thread; warps
//          0..3 take the first half of the heads, warps 4..7 the second
//          half) and run the online softmax in base 2; the running maximum
//          is only raised
//          when a score exceeds it by more than 8 (so most tiles need no
//          cross-thread reduction and no rescale), p is rounded to f16 and
//          written as the PV operand over the tile's rope columns, which
//          QK^T no longer needs
//   a7     two issuers run O^T[512 x HG] += V^T . P^T (issuer 0 the
//          128-column slabs 0 then 2 of the latent columns, issuer 1 slabs 1
//          then 3; V^T is the same shared-memory tile read as an MN-major
//          operand) and signal each slab's release
//   a8     epilogue: O / sum(p) -> bf16 out, lse = ln 2 * (m + log2 sum(p));
//          two splits of a unit merge inside their 2-block cluster, more
//          write the normalized partial (o, lse) to the workspace and
//   a9     merge_kernel combines the partials by log-sum-exp.
// Mbarrier waits suspend the thread (try_wait with a time hint) and are
// bounded (KV4_DEV_TIMEOUT on expiry).
#include "kv4_device.cuh"
#include "kv4_launch.h"

#include <math.h>

#include <type_traits>
#include <utility>

namespace kv4 {
namespace {

// Block: warpgroups 0 and 1 (8 compute warps) gather, dequantize, run the
// softmax and the epilogue; warpgroup 2 issues the MMAs (lane 0 of warps 8
// and 9), so that no compute warp ever stalls behind the tensor-core queue.
// Registers are moved from the issue warpgroup to the compute warpgroups
// with setmaxnreg; per SM sub-partition (one warp of each warpgroup) that is
// 2 x 232 + 40 = 504 of the 3 x 168 the block is launched with.
constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kThreads = kComputeThreads + 128;
constexpr int kLaunchRegs = 168;          // 65536 / 384, rounded down to a multiple of 8
constexpr uint32_t kComputeRegs = 232;
constexpr uint32_t kIssueRegs = 40;
static_assert(2 * kComputeRegs + kIssueRegs <= 3 * kLaunchRegs, "register split exceeds the launch");
#ifndef KV4_PV_ISSUERS
#define KV4_PV_ISSUERS 2
#endif
constexpr int kPvIssuers = KV4_PV_ISSUERS;    // 2: slabs 0,1 are released half way through PV
static_assert(kPvIssuers == 2 || kPvIssuers == 4, "PV issuers");
// QK issuers, each accumulating its share of the 36 k-steps into its own
// partial S^T sum, which the softmax adds up.  One: the fully unrolled issue
// keeps the tensor pipe fed from one thread, and the softmax then reads one
// accumulator (TMEM reads share the shared-memory data stage with the MMA
// operand fetch: four sums measured 0.9 us slower at the long workload).
#ifndef KV4_QK_ISSUERS
#define KV4_QK_ISSUERS 1
#endif
constexpr int kQkIssuers = KV4_QK_ISSUERS;
static_assert(kQkIssuers == 1 || kQkIssuers == 2 || kQkIssuers == 4, "QK issuers");
constexpr int kBarCompute = 3;            // named barrier of the 256 compute threads (1, 2: softmax groups)
constexpr float kRaiseThreshold = 8.0f;   // log2 units: p <= 256 between raises

// FMT: the pool's row format (kv4_launch.h): 352-byte NVFP4 rows (QK over
// 576 columns), 288-byte latent-only NVFP4 rows (QK over the 512 latent
// columns) or 576-byte FP8 rows (QK over 576 columns).
template <int HG, int FMT>
struct Layout {
  static constexpr int HPT = HG / 2;                                  // heads per softmax group
  static constexpr int QK = FMT == kFmtNvfp4Latent ? kLatent : kQk;   // columns of QK^T
  static constexpr int row_bytes =
      FMT == kFmtNvfp4 ? kRowBytes : (FMT == kFmtNvfp4Latent ? kRowBytesLatent : kRowBytesFp8);
  static constexpr uint32_t q_slabs = QK / 64;                        // 64-column slabs of Q
  static constexpr uint32_t q_bytes = q_slabs * HG * 128u;            // Q
  static constexpr uint32_t kv_off = (q_bytes + 1023u) & ~1023u;
  static constexpr uint32_t kv_bytes = 9u * kChunkBytes;              // K/V tile
  static constexpr uint32_t ctl_off = kv_off + kv_bytes;
  // control block
  static constexpr uint32_t bar_off = ctl_off;                        // uint64 x 12
  static constexpr uint32_t tmem_off = ctl_off + 96;                  // uint32
  static constexpr uint32_t done_off = ctl_off + 104;                 // uint64: merge barrier
  static constexpr uint32_t slot_off = ctl_off + 112;                 // int32 [3][128]
  static constexpr uint32_t mref_off = slot_off + 3 * 128 * 4;        // float [HG]
  static constexpr uint32_t alpha_off = mref_off + HG * 4;            // float [HG]
  static constexpr uint32_t red_off = alpha_off + HG * 4;             // float [2][4][HPT]
  static constexpr uint32_t lsum_off = red_off + 4 * HG * 4;          // float [2][HG]
  static constexpr uint32_t qscale_off = lsum_off + 2 * HG * 4;       // float [HG]
  // cluster merge of two splits: this block's partial lse, the peer's (copied
  // in), and the two weights and 1/sum per head
  static constexpr uint32_t xlse_off = qscale_off + HG * 4;           // float [HG]
  static constexpr uint32_t xlse_in_off = xlse_off + HG * 4;          // float [HG]
  static constexpr uint32_t xw_off = xlse_in_off + HG * 4;            // float [2][HG]
  static constexpr uint32_t xinv_off = xw_off + 2 * HG * 4;           // float [HG]
  static constexpr uint32_t end = xinv_off + HG * 4;
  // The peer's half of this block's output slice of O lands in the Q region
  // (free after the last QK): half of HG x 512 fp32 fits in Q's 8 or 9 slabs
  // of HG x 128 B.
  static_assert(HG * kLatent * 4 / 2 <= q_bytes, "peer slice must fit in the Q region");
  // the merge stages the outgoing half (fp32) in the K/V region
  static_assert(HG * kLatent * 4 / 2 <= kv_bytes, "merge staging fits the K/V region");
  static_assert(xlse_off % 16 == 0 && xlse_in_off % 16 == 0, "bulk-copy operands are 16-byte aligned");
  static constexpr uint32_t smem_bytes = end + 1024;                  // + alignment slack
  // tensor memory: O^T slabs at columns [0, 4HG); S^T as kQkIssuers partial
  // sums (one per QK issuer) at [4HG + i HG, 5HG + i HG)
  static constexpr uint32_t tmem_cols = (8 * HG <= 128) ? 128 : (8 * HG <= 256 ? 256 : 512);
  static constexpr uint32_t col_o = 0;
  static constexpr uint32_t col_s = 4 * HG;
  // P^T operand (MN-major, N = HG): one swizzle atom per 8 keys
  static constexpr uint32_t p_row_bytes = 2 * HG;
  static constexpr uint32_t p_atom_bytes = 8 * p_row_bytes;
  static constexpr uint32_t p_swizzle_mode =
      HG == 64 ? kSwizzle128 : (HG == 32 ? kSwizzle64 : kSwizzle32);
  static constexpr int p_swizzle_bits = HG == 64 ? 3 : (HG == 32 ? 2 : 1);
};

// Reduce N values per lane across the 32 lanes of a warp by halving: after
// the call lane l holds max(N/32, 1) results, for heads reduced_head(l, j).
template <int N, bool IS_MAX>
__device__ __forceinline__ void warp_transpose_reduce(float (&v)[N], int lane) {
  int n = N;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (n > 1) {
      const int half = n / 2;
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < half) {
          const float keep = upper ? v[half + i] : v[i];
          const float send = upper ? v[i] : v[half + i];
          const float got = __shfl_xor_sync(0xFFFFFFFFu, send, off);
          v[i] = IS_MAX ? fmaxf(keep, got) : keep + got;
        }
      }
      n = half;
    } else {
      const float got = __shfl_xor_sync(0xFFFFFFFFu, v[0], off);
      v[0] = IS_MAX ? fmaxf(v[0], got) : v[0] + got;
    }
  }
}

template <int N>
__device__ __forceinline__ int reduced_head(int lane, int j) {
  int head = 0, n = N;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (n > 1) {
      n /= 2;
      if (lane & off) head += n;
    }
  }
  return head + j;
}

// Reduction of N per-thread values over the 128 threads of one softmax
// group (4 warps, named barrier bar_id); totals land in dst[N] (shared).
// v is destroyed.
template <int N, bool IS_MAX>
__device__ __forceinline__ void group_reduce(float (&v)[N], int quarter, int lane, float* red,
                                             float* dst, int bar_id) {
  warp_transpose_reduce<N, IS_MAX>(v, lane);
  constexpr int kPerLane = N >= 32 ? N / 32 : 1;
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) red[quarter * N + reduced_head<N>(lane, j)] = v[j];
  named_sync(bar_id, 128);
  const int r = quarter * 32 + lane;
  if (r < N) {
    float acc = red[r];
#pragma unroll
    for (int w = 1; w < 4; ++w) acc = IS_MAX ? fmaxf(acc, red[w * N + r]) : acc + red[w * N + r];
    dst[r] = acc;
  }
  named_sync(bar_id, 128);
}

// N consecutive fp32 TMEM columns of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float (&x)[N]) {
  __syncwarp();                        // tcgen05.ld is warp-collective (.sync.aligned)
  if constexpr (N == 8) {
    uint32_t v[8];
    tmem_ld8_sync(taddr, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = __uint_as_float(v[j]);
  } else {
#pragma unroll
    for (int c = 0; c < N / 16; ++c) {
      uint32_t v[16];
      tmem_ld16_sync(taddr + 16 * c, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) x[16 * c + j] = __uint_as_float(v[j]);
    }
  }
}

// Scores: the sum of the kQkIssuers partial S^T accumulators (columns
// c + i gap), added as (S0 + S1) + (S2 + S3).
template <int N>
__device__ __forceinline__ void load_scores(uint32_t taddr, uint32_t gap, float (&x)[N]) {
  __syncwarp();
  if constexpr (kQkIssuers == 1) {
    tmem_load_cols<N>(taddr, x);
  } else if constexpr (kQkIssuers == 2) {
    if constexpr (N == 32) {
      uint32_t va[32], vb[32];
      tmem_ld32x2_sync(taddr, taddr + gap, va, vb);
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(va[j]) + __uint_as_float(vb[j]);
    } else {
      float y[N];
      tmem_load_cols<N>(taddr, x);
      tmem_load_cols<N>(taddr + gap, y);
#pragma unroll
      for (int j = 0; j < N; ++j) x[j] += y[j];
    }
  } else if constexpr (N == 32) {
    uint32_t va[32], vb[32];
    tmem_ld32x2_sync(taddr, taddr + gap, va, vb);
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(va[j]) + __uint_as_float(vb[j]);
    tmem_ld32x2_sync(taddr + 2 * gap, taddr + 3 * gap, va, vb);
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] += __uint_as_float(va[j]) + __uint_as_float(vb[j]);
  } else {
    float y[N], z[N], u[N];
    tmem_load_cols<N>(taddr, x);
    tmem_load_cols<N>(taddr + gap, y);
    tmem_load_cols<N>(taddr + 2 * gap, z);
    tmem_load_cols<N>(taddr + 3 * gap, u);
#pragma unroll
    for (int j = 0; j < N; ++j) x[j] = (x[j] + y[j]) + (z[j] + u[j]);
  }
}

// Four consecutive output elements: bf16 (rounded to nearest even) or, for
// the fp32 partial output of a decode-context-parallel rank, fp32.
__device__ __forceinline__ void store_out4(void* out, int64_t idx, float4 v, bool f32) {
  if (f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + idx) = v;
  } else {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + idx) = pk;
  }
}

// N consecutive floats of shared memory (16-byte aligned) into registers.
template <int N>
__device__ __forceinline__ void lds_vec(const float* src, float (&v)[N]) {
#pragma unroll
  for (int j = 0; j < N; j += 4) {
    const float4 t = *reinterpret_cast<const float4*>(src + j);
    v[j] = t.x; v[j + 1] = t.y; v[j + 2] = t.z; v[j + 3] = t.w;
  }
}

template <int N>
__device__ __forceinline__ void tmem_scale_cols(uint32_t taddr, const float* alpha) {
  __syncwarp();
  if constexpr (N == 8) {
    uint32_t v[8];
    tmem_ld8_sync(taddr, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha[j]);
    tmem_st8(taddr, v);
  } else {
#pragma unroll
    for (int c = 0; c < N / 16; ++c) {
      uint32_t v[16];
      tmem_ld16_sync(taddr + 16 * c, v);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha[16 * c + j]);
      tmem_st16(taddr + 16 * c, v);
    }
  }
}

template <int HG, int FMT>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecodeArgs a) {
  using L = Layout<HG, FMT>;
  constexpr bool ROPE = FMT != kFmtNvfp4Latent;     // rows carry a rope part
  constexpr bool FP8 = FMT == kFmtFp8;
  constexpr int HPT = L::HPT;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int NG = a.H / HG;
  const int split = blockIdx.x % a.splits;
  const int unit = blockIdx.x / a.splits;          // (b, s, g)
  const int g = unit % NG;
  const int bs = unit / NG;                        // b * Sq + s
  const int b = bs / a.Sq;
  const int s = bs % a.Sq;
  const int32_t* topk_row = a.topk + static_cast<int64_t>(bs) * a.K;
  const int32_t* pt_row = a.page_table + static_cast<int64_t>(b) * a.pt_stride;

  uint8_t* q_s = smem;
  uint8_t* kv_s = smem + L::kv_off;
  // mbarriers: QK done (every QK issuer commits), PV done per 128-column
  // slab of O (slabs 0-1 from issuer 0, 2-3 from issuer 1), tile parts
  // written by the 8 compute warps (latent group a, latent group b, rope), P
  // written, the test hook's one, the cluster merge's and Q staged.
  const uint32_t bars = smem_addr(smem + L::bar_off);
  const uint32_t bar_qk = bars;
  const uint32_t bar_pv0 = bars + 8;              // + 8 * slab: PV slab (128 columns) done
  const uint32_t bar_part0 = bars + 40;           // + 8 * part: tile part written
  const uint32_t bar_p = bars + 64;
  const uint32_t bar_fault = bars + 72;
  const uint32_t bar_merge = bars + 80;           // cluster merge: the peer's data arrived
  const uint32_t bar_q = bars + 88;               // Q copied into the K/V region
  // cluster merge: the peer has received this block's outgoing half (so the
  // bulk copies that read it from this block's shared memory are done)
  const uint32_t bar_done = smem_addr(smem + L::done_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::tmem_off);
  int32_t* slot_s = reinterpret_cast<int32_t*>(smem + L::slot_off);
  float* m_ref = reinterpret_cast<float*>(smem + L::mref_off);
  float* alpha_s = reinterpret_cast<float*>(smem + L::alpha_off);
  float* red_all = reinterpret_cast<float*>(smem + L::red_off);
  float* lsum = reinterpret_cast<float*>(smem + L::lsum_off);
  float* qscale = reinterpret_cast<float*>(smem + L::qscale_off);

  // ---- prologue ------------------------------------------------------------
  bool timed_out = false;
  auto wait = [&](uint32_t bar, uint32_t parity) {
    if (!mbar_wait_bounded(bar, parity, a.timeout_ns)) timed_out = true;
  };
  const uint32_t kv_addr = smem_addr(kv_s);
  constexpr int kQThread = 32 * (kComputeWarps + 1);   // inits the barriers, copies Q
  if (warp == kComputeWarps) tmem_alloc(smem_addr(tmem_slot), L::tmem_cols);
  if (tid == kQThread) {
    mbar_init(bar_qk, kQkIssuers);
    for (int p = 0; p < 4; ++p) mbar_init(bar_pv0 + 8 * p, 1);
    for (int p = 0; p < 3; ++p) mbar_init(bar_part0 + 8 * p, kComputeWarps);
    mbar_init(bar_p, 1);
    mbar_init(bar_fault, 1);
    mbar_init(bar_merge, 1);
    mbar_init(bar_q, 1);
    mbar_init(bar_done, 1);
    fence_mbar_init();
  }
  // every barrier is initialised and the TMEM address is in place before any
  // thread waits on the one or reads the other
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // Everything above touches no global memory and may overlap the end of
  // the previous kernel of the stream, which may have produced any input.
  // When that kernel is known to be this call's own cache write (which
  // writes only the pool), the prologue below -- Q, top-k, page-table and
  // length reads, L2 prefetches -- overlaps it too, and each compute thread
  // waits just before its first read of pool rows.
  if (!a.early_inputs) grid_dependency_wait();
  grid_launch_dependents();
  // The entries of the top-k list this unit walks: all K, or only the first
  // k_count[b, s] of them (a context-parallel rank's own keys, moved to the
  // front of its list); entries at or past k_walk are masked like -1.
  // With a count, the unit's own tiles are shared evenly by its splits.
  const int k_walk = a.k_count != nullptr ? min(a.K, max(0, __ldg(a.k_count + bs))) : a.K;
  const int num_tiles = (k_walk + kTileKeys - 1) / kTileKeys;
  const int tiles_per_split =
      a.k_count != nullptr ? (num_tiles + a.splits - 1) / a.splits : a.tiles_per_split;
  const int tile_begin = split * tiles_per_split;
  const int tile_end = min(num_tiles, tile_begin + tiles_per_split);
  const int my_tiles = max(0, tile_end - tile_begin);
  // The HG x QK bf16 rows of Q (contiguous) go into the K/V region, which
  // holds no tile yet, by one bulk copy; the compute warps convert them.
  constexpr uint32_t kQBytes = HG * L::QK * 2;
  static_assert(kQBytes <= L::kv_bytes, "Q staging fits the K/V region");
  // (Compute warps.)  Rows of the next tile travel in registers: warp w
  // holds rows 16w..16w+15 as three 32-bit words per lane -- latent word
  // wa(l), latent word wb(l),
  // and word 64 + l (lanes 0..7: scales, 8..23: rope, which only 352-byte
  // rows have) -- where pass A covers slabs 0-3 and pass B slabs 4-7, each
  // as one contiguous 128-byte run of the row:
  //   wa(l) = l,   wb(l) = 32 + l.
  // All three groups are reloaded for the next tile after the last pass,
  // while QK finishes.
  // An NVFP4 row's latent word w (8 codes) and an FP8 row's 8-byte latent
  // unit w (8 E4M3 values) both become the f16 unit of columns 8w..8w+7.
  // The extra word of lane l is word 64 + l of an NVFP4 row (scales, rope)
  // and word 120 + l of an FP8 row (rope only, lanes 8..23).
  using LatWord = std::conditional_t<FP8, uint2, uint32_t>;
  constexpr int kExtraWord0 = FP8 ? 120 : 64;
  const bool extra_lane = FP8 ? (lane >= 8 && lane < 24) : (lane < (ROPE ? 24 : 8));
  const int word_a = lane;
  const int word_b = lane + 32;
  LatWord wa[16], wb[16];
  uint32_t wex[16];
  // the slots of this warp's 16 rows of the tile whose slots are at `slots`
  // (re-read from shared memory for every tile, so that they hold no
  // registers across it)
  auto read_slots = [&](const int32_t* slots, int32_t (&sv)[16]) {
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const int4 t = *reinterpret_cast<const int4*>(slots + warp * 16 + i);
      sv[i] = t.x; sv[i + 1] = t.y; sv[i + 2] = t.z; sv[i + 3] = t.w;
    }
  };
  // The three words of each of this warp's 16 rows of the tile whose slots
  // are at `slots` (read once), grouped by word -- every row's first word,
  // then every row's second, then the extra words; a masked key gives a
  // zero row.  (Issuing each row's three words back to back measured
  // slower.)
  auto load_rows = [&](const int32_t* slots) {
    int32_t sv[16];
    read_slots(slots, sv);
    auto word_ptr = [&](int i) {
      return reinterpret_cast<const uint32_t*>(a.pool + static_cast<int64_t>(sv[i]) * L::row_bytes);
    };
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if constexpr (FP8)
        wa[i] = sv[i] >= 0 ? ldg_stream_u64(reinterpret_cast<const uint2*>(word_ptr(i)) + word_a)
                           : make_uint2(0, 0);
      else
        wa[i] = sv[i] >= 0 ? ldg_stream_u32(word_ptr(i) + word_a) : 0u;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if constexpr (FP8)
        wb[i] = sv[i] >= 0 ? ldg_stream_u64(reinterpret_cast<const uint2*>(word_ptr(i)) + word_b)
                           : make_uint2(0, 0);
      else
        wb[i] = sv[i] >= 0 ? ldg_stream_u32(word_ptr(i) + word_b) : 0u;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
      wex[i] = (sv[i] >= 0 && extra_lane) ? ldg_stream_u32(word_ptr(i) + kExtraWord0 + lane) : 0u;
  };
  // Q -> f16, 128-byte-swizzled K-major operand, by the compute threads
  // while their first slot lookups are in flight.  Each head is scaled by
  // 2^-e_h (exact) so that its largest magnitude lies in [2^14, 2^15): every
  // bf16 element of at least 2^-31 of the head's maximum then converts to f16
  // without loss (smaller ones fall into f16's subnormal range); 2^e_h is
  // folded into the head's score scale.  TPH threads own a head (its QK/8 16-byte units interleaved
  // among them, the order rotated by head so that a warp's reads of the
  // staged rows spread over all banks) and reduce its maximum with shuffles.
  auto convert_q = [&] {
    constexpr int UNITS = L::QK / 8;               // 16-byte units of a head
    constexpr int TPH = HG == 64 ? 4 : 8;          // threads per head
    constexpr int UPT = UNITS / TPH;               // 16-byte units per thread
    static_assert(UNITS % TPH == 0, "units per thread");
    const int h = tid / TPH, part = tid % TPH;
    if (h >= HG) return;                           // HG = 16 uses 128 threads
    const uint4* qst = reinterpret_cast<const uint4*>(kv_s);
    uint32_t m = 0;
    wait(bar_q, 0);
    // two passes over the staged rows (maximum, then conversion), so that no
    // thread holds its whole share of Q in registers
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      const int gu = part + ((j + h) % UPT) * TPH;   // 16-byte unit of head h
      const uint4 qv = qst[h * UNITS + gu];
      const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        m = max(m, max((w[k] << 16) & 0x7FFFFFFFu, w[k] & 0x7FFF0000u));   // |bf16| as fp32 bits
    }
#pragma unroll
    for (int off = 1; off < TPH; off <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    // e = floor(log2 amax) + 1 - 15 from the bits of amax (|bf16| widened to
    // fp32: normal, subnormal or zero), kept in [-126, 126] so that 2^-e and
    // 2^e are normal floats built from their exponent fields
    const int lg = m >= 0x00800000u ? static_cast<int>(m >> 23) - 127
                                    : (m != 0u ? (31 - __clz(static_cast<int>(m))) - 149 : 14);
    const int e = min(126, max(-126, lg - 14));
    const float f = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    if (part == 0)
      qscale[h] = a.sm_scale * 1.4426950408889634f * __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      const int gu = part + ((j + h) % UPT) * TPH;
      const uint4 qv = qst[h * UNITS + gu];
      const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __half2 hv = __floats2half2_rn(__uint_as_float(w[k] << 16) * f,
                                             __uint_as_float(w[k] & 0xFFFF0000u) * f);
        o[k] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      const uint32_t off = (gu >> 3) * (HG * 128) + (h >> 3) * 1024 + (h & 7) * 128 + (gu & 7) * 16;
      *reinterpret_cast<uint4*>(q_s + swizzle<3>(off)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  };
  // The roles split here and never meet again before the epilogue; each
  // takes its register share first, while it has no load in flight (the
  // reallocation waits for the thread's outstanding loads).
  if (warp >= kComputeWarps) {
    if (tid == kQThread) {
      mbar_arrive_expect_tx(bar_q, kQBytes);
      bulk_copy_g2s(kv_addr,
                    static_cast<const __nv_bfloat16*>(a.q) + (static_cast<int64_t>(bs) * a.H + g * HG) * L::QK,
                    kQBytes, bar_q);
    }
    // ==== MMA issue warpgroup: lane 0 of each of its warps is an issuer ====
    // QK comes from kQkIssuers issuers (one partial sum of S^T each) and PV
    // from two (issuer 0: O slabs 0 then 2, issuer 1: slabs 1 then 3, so
    // that slabs 0 and 1 -- latent columns 0-255 -- are released half way
    // through).
    setmaxnreg_dec<kIssueRegs>();
    if (lane == 0) {
      const int qi = warp - kComputeWarps;         // issuer 0..3
      // descriptors built once, advanced by adding 16-byte-unit offsets to the
      // start-address field (addresses stay below 2^18, so no carry)
      const uint64_t desc_k = smem_desc(kv_addr, 16, 1024, kSwizzle128);             // K-major A
      const uint64_t desc_q = smem_desc(smem_addr(q_s), 16, 1024, kSwizzle128);      // K-major B
      const uint64_t desc_v = smem_desc(kv_addr, kChunkBytes, 1024, kSwizzle128);    // MN-major A
      const uint64_t desc_p = smem_desc(kv_addr + 8 * kChunkBytes, 8192, L::p_atom_bytes,
                                        L::p_swizzle_mode);                         // MN-major B
      // a5 for issuer QI: its share of S^T = K_tile . Q^T, each part as soon as
      // the compute warps wrote it.  Pass a writes latent chunks (64 columns =
      // 4 k-steps of 16) 0-3 and pass b chunks 4-7; issuer QI
      // takes kCpi of each pass's four, and kRpi of the four rope k-steps
      // (chunk 8).  Every operand offset is a compile-time constant.
      constexpr uint32_t idesc_qk = idesc_f16(128, HG, false, false);
      constexpr int kCpi = 4 / kQkIssuers;
      constexpr int kRpi = 4 / kQkIssuers;
      const uint32_t d_s = tmem + L::col_s + qi * HG;
      auto issue_qk = [&](auto qi_const, const uint32_t par) {
        constexpr int QI = decltype(qi_const)::value;
        auto chunk = [&](auto c_const, const bool first) {
          constexpr int c = decltype(c_const)::value;
          [&]<int... SUB>(std::integer_sequence<int, SUB...>) {
            ((mma_f16kind_at<((c * kChunkBytes + SUB * 32) >> 4), ((c * (HG * 128) + SUB * 32) >> 4)>(
                 d_s, desc_k, desc_q, idesc_qk, (first && SUB == 0) ? 0u : 1u)), ...);
          }(std::make_integer_sequence<int, 4>{});
        };
        wait(bar_part0, par);
        tc_fence_after_sync();
        [&]<int... I>(std::integer_sequence<int, I...>) {
          (chunk(std::integral_constant<int, QI * kCpi + I>{}, I == 0), ...);
        }(std::make_integer_sequence<int, kCpi>{});
        wait(bar_part0 + 8, par);
        tc_fence_after_sync();
        [&]<int... I>(std::integer_sequence<int, I...>) {
          (chunk(std::integral_constant<int, 4 + QI * kCpi + I>{}, false), ...);
        }(std::make_integer_sequence<int, kCpi>{});
        if constexpr (ROPE) {
          wait(bar_part0 + 16, par);
          tc_fence_after_sync();
          [&]<int... J>(std::integer_sequence<int, J...>) {
            ((mma_f16kind_at<((8 * kChunkBytes + (QI * kRpi + J) * 32) >> 4),
                             ((8 * (HG * 128) + (QI * kRpi + J) * 32) >> 4)>(
                 d_s, desc_k, desc_q, idesc_qk, 1u)), ...);
          }(std::make_integer_sequence<int, kRpi>{});
        }
        mma_commit(bar_qk);
      };
      // a7 for issuer QI: O slabs QI, QI + kPvIssuers, ... (128 latent
      // columns each, M = 128) += V^T . P^T over the tile's 128 keys (8
      // k-steps of 16 keys), every operand offset a compile-time constant;
      // each slab is committed on its own barrier.
      constexpr uint32_t idesc_pv = idesc_f16(128, HG, true, true);
      constexpr int kSlabsPerIssuer = 4 / kPvIssuers;
      auto issue_pv = [&](auto qi_const, const bool acc_prev) {
        constexpr int QI = decltype(qi_const)::value;
        [&]<int... J>(std::integer_sequence<int, J...>) {
          ([&] {
            constexpr int mb = QI + kPvIssuers * J;
            [&]<int... KS>(std::integer_sequence<int, KS...>) {
              ((mma_f16kind_at<(((2 * mb) * kChunkBytes + (2 * KS) * 1024) >> 4),
                               (((2 * KS) * L::p_atom_bytes) >> 4)>(
                   tmem + L::col_o + mb * HG, desc_v, desc_p, idesc_pv,
                   (acc_prev || KS > 0) ? 1u : 0u)), ...);
            }(std::make_integer_sequence<int, 8>{});
            mma_commit(bar_pv0 + 8 * mb);
          }(), ...);
        }(std::make_integer_sequence<int, kSlabsPerIssuer>{});
      };
      for (int it = 0; it < my_tiles; ++it) {
        const uint32_t par = it & 1;
        if (qi == 0) issue_qk(std::integral_constant<int, 0>{}, par);
        if constexpr (kQkIssuers >= 2) {
          if (qi == 1) issue_qk(std::integral_constant<int, 1>{}, par);
        }
        if constexpr (kQkIssuers == 4) {
          if (qi == 2) issue_qk(std::integral_constant<int, 2>{}, par);
          if (qi == 3) issue_qk(std::integral_constant<int, 3>{}, par);
        }
        if (qi >= kPvIssuers) continue;
        // a7: O^T += V^T . P^T, 4 / kPvIssuers O slabs (128 columns each) per
        // issuer, each committed on its own so that the next tile's
        // dequantization can reuse its shared memory as early as possible
        wait(bar_p, par);
        tc_fence_after_sync();
        if (qi == 0) issue_pv(std::integral_constant<int, 0>{}, it > 0);
        if (qi == 1) issue_pv(std::integral_constant<int, 1>{}, it > 0);
        if constexpr (kPvIssuers == 4) {
          if (qi == 2) issue_pv(std::integral_constant<int, 2>{}, it > 0);
          if (qi == 3) issue_pv(std::integral_constant<int, 3>{}, it > 0);
        }
      }
    }
    __syncwarp();
    if (a.cluster_merge) cluster_sync();       // the compute warps' merge barrier
  } else {
    // ==== compute warpgroups (warps 0..7) ====
    setmaxnreg_inc<kComputeRegs>();
    // The request's page-table row into L2 (up to 32 KB, one 128-byte line
    // per thread), so that the slot lookups two tiles ahead find their
    // second dependent load there.
    {
      const int64_t pt_lines = (a.pt_stride * 4 + 127) / 128;
      if (tid < pt_lines) prefetch_l2_line(reinterpret_cast<const uint8_t*>(pt_row) + tid * 128);
    }
    const int64_t l_eff = static_cast<int64_t>(__ldg(a.seq_lens + b)) - (a.Sq - 1 - s);
    if (tid < HG) m_ref[tid] = -INFINITY;
    // Slots of the first two tiles (a ring of three tiles, filled two
    // ahead): lane l of warp w resolves row 16w + (l mod 16) of tile l/16 --
    // the rows the warp gathers itself -- by its top-k entry, page-table
    // entry and slot, while Q is on its way; tile 0's rows are then started
    // into L2 (a row's bytes span at most four 128-byte lines), so that the
    // gather after the Q conversion finds them there.
    {
      const int t0 = lane >> 4, r0 = warp * 16 + (lane & 15);
      if (t0 < my_tiles) {
        const int k0 = (tile_begin + t0) * kTileKeys + r0;
        const int32_t idx = k0 < k_walk ? __ldg(topk_row + k0) : -1;
        const int32_t pi = slot_page_index(idx, l_eff, a.pt_stride, a.dev_err);
        const int32_t sl =
            pi >= 0 ? slot_from_page(__ldg(pt_row + pi), idx, a.num_slots, a.dev_err) : -1;
        slot_s[t0 * 128 + r0] = sl;
        if (t0 == 0 && sl >= 0) {
          const uint8_t* row = a.pool + static_cast<int64_t>(sl) * L::row_bytes;
          prefetch_l2_line(row);
          prefetch_l2_line(row + 128);
          prefetch_l2_line(row + 256);
          prefetch_l2_line(row + L::row_bytes - 1);
        }
      }
    }
    convert_q();
    fence_async_smem();                              // Q is read by the tensor core
    __syncwarp();                                    // this warp's slots are written
    if (a.early_inputs) grid_dependency_wait();      // the pool rows are written
    if (my_tiles > 0) load_rows(slot_s);
    // Q's scales, the reference maxima and the slots are in place for every
    // compute warp (the barrier also waits for this thread's gathers, which
    // the first pass needs anyway)
    named_sync(kBarCompute, kComputeThreads);

    // softmax roles: group G owns heads [G*HPT, G*HPT + HPT); thread (quarter,
    // lane) owns key row r = quarter*32 + lane of each tile = TMEM lane r.
    const int G = warp >> 2;
    const int quarter = warp & 3;
    const int r_key = quarter * 32 + lane;
    const int h0 = G * HPT;
    const int bar_group = 1 + G;
    float* red = red_all + G * 4 * HPT;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    // Running sum of p per head (fp32).  It normalizes O and gives lse; the
    // f16 rounding of p inside PV changes each weight by at most 2^-12.
    float l_sum[HPT];
#pragma unroll
    for (int h = 0; h < HPT; ++h) l_sum[h] = 0.0f;
    // Start this warp's 16 rows of a tile (slots at `slots`, written by its
    // lanes 0..15 a tile earlier) on their way into L2, so that the register
    // gather at the end of the current tile finds them there: lane l asks for
    // line (l & 3) of rows l/4 and 8 + l/4 (a row's bytes span at most four
    // 128-byte lines).
    auto prefetch_rows = [&](const int32_t* slots) {
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int32_t sl = slots[warp * 16 + 8 * k + (lane >> 2)];
        const uint32_t off = (lane & 3) == 3 ? L::row_bytes - 1 : 128u * (lane & 3);
        if (sl >= 0) prefetch_l2_line(a.pool + static_cast<int64_t>(sl) * L::row_bytes + off);
      }
    };
    auto dequant_latent = [&](const LatWord& w, uint32_t w_ex, int word) -> uint4 {
      if constexpr (FP8) {
        const uint2 lo = dequant_rope(w.x), hi = dequant_rope(w.y);
        return make_uint4(lo.x, lo.y, hi.x, hi.y);
      } else {
        return dequant_latent_word(w, w_ex, word);
      }
    };

    // dequant store addresses (shared-window): latent word w of row r goes to
    // slab w/8, unit (w%8) ^ (r%8) of the row's 128-byte line; rows of this
    // warp start at line 2*warp*1024; indexed by r%8 (the swizzle phase).
    uint32_t a_base[8], b_base[8], rope_base[8];
    {
      const uint32_t kv = kv_addr + warp * 2048;
      const uint32_t lr = (lane - 8) & 15;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        a_base[j] = kv + (word_a >> 3) * kChunkBytes + (((word_a & 7) ^ j) << 4);
        b_base[j] = kv + (word_b >> 3) * kChunkBytes + (((word_b & 7) ^ j) << 4);
        rope_base[j] = kv + 8 * kChunkBytes + ((((lr >> 1) ^ j) << 4) | ((lr & 1) << 3));
      }
    }

    for (int it = 0; it < my_tiles; ++it) {
      const int tile = tile_begin + it;
      const int ring = it % 3;
      const int32_t* next_slots = slot_s + ((it + 1) % 3) * 128;
      const uint32_t par = it & 1;                 // phase parity of this tile's barriers
      // slot of key (tile + 2, row warp*16 + lane) for lanes 0..15, resolved in
      // three steps spread over this iteration (top-k load, page-table load,
      // slot) so that neither dependent load stalls the warp
      const bool resolve_ahead = (it + 2 < my_tiles) && lane < 16;
      const int k_ahead = (tile + 2) * kTileKeys + warp * 16 + lane;
      int32_t idx_ahead = -1, page_ahead = -1, pi_ahead = -1;
      if (resolve_ahead && k_ahead < k_walk) idx_ahead = __ldg(topk_row + k_ahead);

      // ---- a3/a4 in three passes, each into slabs that the previous tile's
      // PV has released; QK starts on each part as soon as all warps wrote it.
      // the next tile's rows on their way into L2 while the previous PV runs
      // (the gather follows the last pass below)
      if (it + 1 < my_tiles) prefetch_rows(next_slots);
      // pass A: slabs 0-3 (O slabs 0 and 1, which PV runs first)
      if (it > 0) {
        wait(bar_pv0, par ^ 1);
        wait(bar_pv0 + 8, par ^ 1);
        __syncwarp();
        tc_fence_after_sync();
      }
#pragma unroll
      for (int i = 0; i < 16; ++i)
        st_shared_v4(a_base[i & 7] + (i >> 3) * 1024 + (i & 7) * 128,
                     dequant_latent(wa[i], wex[i], word_a));
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_part0);
      // pass B: slabs 4-7 (O slabs 2 and 3; PV is then complete)
      if (it > 0) {
        wait(bar_pv0 + 16, par ^ 1);
        wait(bar_pv0 + 24, par ^ 1);
        __syncwarp();
        tc_fence_after_sync();
      }
#pragma unroll
      for (int i = 0; i < 16; ++i)
        st_shared_v4(b_base[i & 7] + (i >> 3) * 1024 + (i & 7) * 128,
                     dequant_latent(wb[i], wex[i], word_b));
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_part0 + 8);
      if constexpr (ROPE) {
        // pass C: rope -> slab 8 (the previous tile's P lived there; PV is done)
        if (lane >= 8 && lane < 24) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            st_shared_v2(rope_base[i & 7] + (i >> 3) * 1024 + (i & 7) * 128, dequant_rope(wex[i]));
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_part0 + 16);
      }
      // the next tile's rows, gathered while QK finishes (the passes above
      // run back to back, so that QK receives its parts as early as possible)
      if (it + 1 < my_tiles) load_rows(next_slots);

      // ---- a2, second step: page-table entry of the key two tiles ahead
      if (resolve_ahead) {
        pi_ahead = slot_page_index(idx_ahead, l_eff, a.pt_stride, a.dev_err);
        if (pi_ahead >= 0) page_ahead = __ldg(pt_row + pi_ahead);
      }

      // ---- a6: online softmax (two head groups) ----
      {
        wait(bar_qk, par);               // QK done
        __syncwarp();                    // lanes may leave the wait at different times
        tc_fence_after_sync();
        const bool valid = slot_s[ring * 128 + r_key] >= 0;
        // x = log2-domain score relative to the head's reference maximum
        float x[HPT], c[HPT], mr[HPT];
        load_scores<HPT>(lane_base + L::col_s + h0, HG, x);
        lds_vec<HPT>(qscale + h0, c);
        lds_vec<HPT>(m_ref + h0, mr);
        float xmax = -INFINITY;
#pragma unroll
        for (int h = 0; h < HPT; ++h) {
          x[h] = fmaf(x[h], c[h], -mr[h]);
          xmax = fmaxf(xmax, x[h]);
        }
        const bool need = named_sync_or(bar_group, 128, valid && xmax > kRaiseThreshold);
        if (need) {
          // (rare) raise the reference maximum of every head to its tile maximum
          load_scores<HPT>(lane_base + L::col_s + h0, HG, x);
#pragma unroll
          for (int h = 0; h < HPT; ++h) x[h] = valid ? x[h] * c[h] : -INFINITY;
          float v[HPT];
#pragma unroll
          for (int h = 0; h < HPT; ++h) v[h] = x[h];
          group_reduce<HPT, true>(v, quarter, lane, red, alpha_s + h0, bar_group);
          if (r_key < HPT) {
            const float mo = m_ref[h0 + r_key];
            const float mn = fmaxf(mo, alpha_s[h0 + r_key]);
            alpha_s[h0 + r_key] = (mo == mn) ? 1.0f : fast_exp2(mo - mn);
            m_ref[h0 + r_key] = mn;
          }
          named_sync(bar_group, 128);
          float al[HPT];
          lds_vec<HPT>(alpha_s + h0, al);
          lds_vec<HPT>(m_ref + h0, mr);
#pragma unroll
          for (int h = 0; h < HPT; ++h) {
            l_sum[h] *= al[h];
            x[h] -= mr[h];
          }
          if (it > 0) {
#pragma unroll
            for (int mb = 0; mb < 4; ++mb)
              tmem_scale_cols<HPT>(lane_base + L::col_o + mb * HG + h0, alpha_s + h0);
            tmem_st_wait();
          }
        }
        // probabilities -> f16 P^T row r_key, heads [h0, h0 + HPT)
        uint32_t packed[HPT / 2];
        if (valid) {
#pragma unroll
          for (int h = 0; h < HPT; h += 2) {
            const float p0 = fast_exp2(x[h]);
            const float p1 = fast_exp2(x[h + 1]);
            l_sum[h] += p0;
            l_sum[h + 1] += p1;
            const __half2 ph = __floats2half2_rn(p0, p1);
            packed[h / 2] = *reinterpret_cast<const uint32_t*>(&ph);
          }
        } else {
#pragma unroll
          for (int h = 0; h < HPT / 2; ++h) packed[h] = 0u;
        }
        uint8_t* p_s = kv_s + 8 * kChunkBytes;
#pragma unroll
        for (int u = 0; u < HPT / 8; ++u) {
          const uint32_t off = (r_key >> 3) * L::p_atom_bytes + (r_key & 7) * L::p_row_bytes +
                               (h0 * 2) + u * 16;
          *reinterpret_cast<uint4*>(p_s + swizzle<L::p_swizzle_bits>(off)) =
              make_uint4(packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
        }
        // ---- a2, last step: the slot of the key two tiles ahead.  Its ring
        // entry was last read by the previous tile's softmax.
        if (resolve_ahead)
          slot_s[((it + 2) % 3) * 128 + warp * 16 + lane] =
              pi_ahead >= 0 ? slot_from_page(page_ahead, idx_ahead, a.num_slots, a.dev_err) : -1;
        fence_async_smem();
        tc_fence_before_sync();
      }
      // P of all 128 keys (and any O rescale) is in place: hand over to the issuers
      named_sync(kBarCompute, kComputeThreads);
      if (tid == 0) mbar_arrive(bar_p);
    }
    // ---- a8: epilogue ----
    // Normalized partial (o, lse) of this split: merged inside the cluster
    // when the splits of the unit form one (below), else into the workspace;
    // with one split, straight to out / lse.  l and lse need only the softmax
    // state, so they are computed while the last PV still runs.
    const bool cmerge = a.cluster_merge != 0;
    const bool partial = a.splits > 1;
    float* xlse = reinterpret_cast<float*>(smem + L::xlse_off);
    const int64_t out_head0 = static_cast<int64_t>(bs) * a.H + g * HG;   // first head row
    const int64_t part = static_cast<int64_t>(unit) * a.splits + split;
    group_reduce<HPT, false>(l_sum, quarter, lane, red, lsum + h0, bar_group);
    if (r_key < HPT) {
      const float lt = lsum[h0 + r_key];
      lsum[HG + h0 + r_key] = lt > 0.0f ? __frcp_rn(lt) : 0.0f;     // 1 / l
    }
    named_sync(bar_group, 128);
    if (r_key < HPT) {
      const int h = h0 + r_key;
      const float lt = lsum[h];
      const float lse = (lt > 0.0f) ? (m_ref[h] + log2f(lt)) * 0.69314718055994531f : -INFINITY;
      if (cmerge) xlse[h] = lse;
      else if (partial) a.ws_lse[part * HG + h] = lse;
      else a.lse[out_head0 + h] = lse;
    }
    if (cmerge) {
      // first half of the merge's first cluster barrier: this block's Q region
      // is free (its last QK is done) and its merge barrier is armed
      if (tid == 0) mbar_arrive_expect_tx(bar_merge, HG * kLatent * 4 / 2 + HG * 4);
      cluster_arrive();
    }
    // the last PV must be complete before O is read or TMEM is freed
    if (my_tiles > 0) {
      const uint32_t last = (my_tiles - 1) & 1;
      for (int p = 0; p < 4; ++p) wait(bar_pv0 + 8 * p, last);
      __syncwarp();
      tc_fence_after_sync();
    }

#pragma unroll
    for (int mb = 0; mb < 4; ++mb) {
      if (cmerge) break;
      const int d = mb * 128 + r_key;
      float o[HPT];
      if (my_tiles > 0) {
        tmem_load_cols<HPT>(lane_base + L::col_o + mb * HG + h0, o);
      } else {
#pragma unroll
        for (int j = 0; j < HPT; ++j) o[j] = 0.0f;
      }
      float inv[HPT];
      lds_vec<HPT>(lsum + HG + h0, inv);
#pragma unroll
      for (int j = 0; j < HPT; ++j) {
        const int h = h0 + j;
        const float v = o[j] * inv[j];
        if (partial) a.ws_o[(part * HG + h) * kLatent + d] = v;
        else if (a.out_f32) static_cast<float*>(a.out)[(out_head0 + h) * kLatent + d] = v;
        else static_cast<__nv_bfloat16*>(a.out)[(out_head0 + h) * kLatent + d] = __float2bfloat16_rn(v);
      }
    }
    if (a.fault_site == 1 && warp == 0) {
      // test hook, after all work of the block: warp 0 waits on a barrier that
      // nothing arrives on, so the wait runs out and reports a timeout
      const bool ok = mbar_wait_bounded(bar_fault, 0, a.timeout_ns);
      __syncwarp();
      if (!ok) timed_out = true;
    }

    // ---- a9 inside a cluster of the unit's two splits: block r produces
    // output columns [256 r, 256 r + 256) (O slabs 2r, 2r+1), out =
    // (w_0 o_0 + w_1 o_1) / (w_0 + w_1) with w_i = exp(lse_i - max lse) and
    // lse = max lse + log(w_0 + w_1), o_i the normalized partials.
    //   1. each thread normalizes its column of the peer's two slabs (from
    //      TMEM) into a staging area of this block's K/V region: a
    //      (slab, column) row of HG fp32 values, its 16-byte units
    //      XOR-swizzled by the column so that a warp's accesses spread over
    //      all banks;
    //   2. after a cluster barrier (the peer's Q region is free once its last
    //      QK is done; each block arrived on it before waiting for its last
    //      PV), one bulk copy moves the staged half and this block's lse into
    //      the peer; meanwhile the threads read their own half from TMEM;
    //   3. once the peer's half has arrived, each block tells the peer so
    //      (a remote mbarrier arrive: the peer's outgoing half has been read)
    //      and stores its merged columns straight to out (for each head a
    //      warp writes 32 consecutive columns);
    //   4. before exiting, each block waits for the peer's word that this
    //      block's outgoing half has arrived there.
    // (The issue warpgroup meets the same cluster barrier.)
    if (cmerge) {
      constexpr int U = HG / 4;                              // 16-byte units of a row
      constexpr uint32_t kHalfBytes = HG * kLatent * 4 / 2;
      const uint32_t rank = cluster_ctarank();
      const uint32_t peer = rank ^ 1u;
      float* xlse_in = reinterpret_cast<float*>(smem + L::xlse_in_off);
      float* xw = reinterpret_cast<float*>(smem + L::xw_off);
      float* xinv = reinterpret_cast<float*>(smem + L::xinv_off);
      uint8_t* stage_out = kv_s;                             // outgoing half, fp32
      auto row_unit = [&](int s2, int u) -> uint32_t {       // byte offset of a staged unit
        return static_cast<uint32_t>(((s2 * 128 + r_key) * U + (u ^ (r_key % U))) * 16);
      };
      float inv[HPT];
      lds_vec<HPT>(lsum + HG + h0, inv);
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        float v[HPT];
        if (my_tiles > 0) {
          tmem_load_cols<HPT>(lane_base + L::col_o + (2 * peer + s2) * HG + h0, v);
        } else {
#pragma unroll
          for (int j = 0; j < HPT; ++j) v[j] = 0.0f;
        }
#pragma unroll
        for (int k = 0; k < HPT / 4; ++k)
          *reinterpret_cast<float4*>(stage_out + row_unit(s2, h0 / 4 + k)) =
              make_float4(v[4 * k] * inv[4 * k], v[4 * k + 1] * inv[4 * k + 1],
                          v[4 * k + 2] * inv[4 * k + 2], v[4 * k + 3] * inv[4 * k + 3]);
      }
      fence_async_smem();                      // the staged half is read by the async proxy
      named_sync(kBarCompute, kComputeThreads);  // every thread's part is staged
      cluster_wait();                          // the peer's Q region is free, its barrier armed
      // the staged half leaves in kMergeCopies bulk copies issued by as many
      // threads (lane 0 of consecutive warps), so that they run side by side
      constexpr int kMergeCopies = 8;
      static_assert(kHalfBytes % (kMergeCopies * 16) == 0, "copy chunks of whole 16-byte units");
      constexpr uint32_t kChunk = kHalfBytes / kMergeCopies;
      if (lane == 0 && warp < kMergeCopies) {
        const uint32_t peer_bar = cluster_map(bar_merge, peer);
        bulk_copy_to_cluster(cluster_map(smem_addr(q_s) + warp * kChunk, peer),
                             smem_addr(stage_out) + warp * kChunk, kChunk, peer_bar);
        if (warp == 0)
          bulk_copy_to_cluster(cluster_map(smem_addr(xlse_in), peer), smem_addr(xlse), HG * 4,
                               peer_bar);
      }
      float mine[2][HPT];
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        if (my_tiles > 0) {
          tmem_load_cols<HPT>(lane_base + L::col_o + (2 * rank + s2) * HG + h0, mine[s2]);
        } else {
#pragma unroll
          for (int j = 0; j < HPT; ++j) mine[s2][j] = 0.0f;
        }
#pragma unroll
        for (int j = 0; j < HPT; ++j) mine[s2][j] *= inv[j];
      }
      wait(bar_merge, 0);                      // the peer's half and lse are here
      // the peer's copies into this block are complete, so its outgoing half
      // has been read: let it finish (and exit) whenever it is done
      if (tid == 0) mbar_remote_arrive(cluster_map(bar_done, peer));
      if (tid < HG) {
        const float l0 = rank == 0 ? xlse[tid] : xlse_in[tid];
        const float l1 = rank == 0 ? xlse_in[tid] : xlse[tid];
        const float m = fmaxf(l0, l1);
        // base-2 hardware exponent and logarithm (wsum lies in [1, 2])
        const float w0 = l0 != -INFINITY ? fast_exp2((l0 - m) * 1.4426950408889634f) : 0.0f;
        const float w1 = l1 != -INFINITY ? fast_exp2((l1 - m) * 1.4426950408889634f) : 0.0f;
        const float wsum = w0 + w1;
        xw[tid] = w0;
        xw[HG + tid] = w1;
        xinv[tid] = wsum > 0.0f ? __frcp_rn(wsum) : 0.0f;
        if (rank == 0)
          a.lse[out_head0 + tid] =
              wsum > 0.0f ? m + fast_log2(wsum) * 0.69314718055994531f : -INFINITY;
      }
      named_sync(kBarCompute, kComputeThreads);
      // merged values straight to out[head, 256 rank + column]: for each head
      // a warp's lanes store 32 consecutive columns (storing bf16 pairs after
      // a lane-pair exchange, or staging the rows for bulk copies, measured
      // no faster)
      {
        float w0[HPT], w1[HPT], xi[HPT];
        lds_vec<HPT>(xw + h0, w0);
        lds_vec<HPT>(xw + HG + h0, w1);
        lds_vec<HPT>(xinv + h0, xi);
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          const int64_t col = 256 * static_cast<int64_t>(rank) + s2 * 128 + r_key;
#pragma unroll
          for (int k = 0; k < HPT / 4; ++k) {
            const float4 t = *reinterpret_cast<const float4*>(q_s + row_unit(s2, h0 / 4 + k));
            const float theirs[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = 4 * k + i;
              // summed in split order, as the merge kernel does
              const float v0 = rank == 0 ? mine[s2][j] : theirs[i];
              const float v1 = rank == 0 ? theirs[i] : mine[s2][j];
              const float v = (w0[j] * v0 + w1[j] * v1) * xi[j];
              const int64_t o = (out_head0 + h0 + j) * kLatent + col;
              if (a.out_f32) static_cast<float*>(a.out)[o] = v;
              else static_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(v);
            }
          }
        }
      }
      // before exiting: the peer has received this block's outgoing half
      if (tid == 0) wait(bar_done, 0);
    }
  }  // compute warpgroups
  if (timed_out) flag_error(a.dev_err, kDevTimeout);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kComputeWarps) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::tmem_cols);
  }
}

// a9 for more than two splits: out = sum_i w_i o_i / sum_i w_i with
// w_i = exp(lse_i - max lse), lse = max lse + log(sum_i w_i), o_i the
// normalized partials.  A group of `group` warps (one block) takes one
// (unit, head, 128-column quarter of the latent) row: warp k accumulates the
// partials k, k + group, ... (at most eight per warp, so each lane has all
// its loads in flight at once), lane l the columns 4l..4l+3 of the quarter;
// the warps' sums then meet in shared memory and warp 0 adds them in warp
// order.  Every warp first takes the maximum lse over all splits itself.
constexpr int kMergeMaxWarps = 8;
__global__ void __launch_bounds__(32 * kMergeMaxWarps) merge_kernel(DecodeArgs a, int n_units,
                                                                     int group) {
  grid_dependency_wait();                      // the decode's partials
  grid_launch_dependents();
  __shared__ float4 part_acc[kMergeMaxWarps][32];
  __shared__ float part_w[kMergeMaxWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HG = a.HG;
  const int quarter = blockIdx.x & 3;
  const int rid = blockIdx.x >> 2;             // unit * HG + head
  const int unit = rid / HG, h = rid % HG;
  const int NG = a.H / HG;
  const int g = unit % NG, bs = unit / NG;
  const int S = a.splits;
  const float* lse_p = a.ws_lse + static_cast<int64_t>(unit) * S * HG + h;
  const float4* o_p = reinterpret_cast<const float4*>(
      a.ws_o + (static_cast<int64_t>(unit) * S * HG + h) * kLatent) + quarter * 32 + lane;
  const int64_t o_stride = static_cast<int64_t>(HG) * kLatent / 4;   // float4 per split
  float m = -INFINITY;
  for (int i = lane; i < S; i += 32) m = fmaxf(m, lse_p[i * HG]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.0f;
  if (m != -INFINITY) {
    // without branches (a split with no key has lse = -inf and weight 0;
    // its o is 0)
#pragma unroll 8
    for (int i = warp; i < S; i += group) {
      const float li = lse_p[i * HG];
      const float w = li != -INFINITY ? fast_exp2((li - m) * 1.4426950408889634f) : 0.0f;
      wsum += w;
      const float4 v = o_p[i * o_stride];
      acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
    }
  }
  part_acc[warp][lane] = acc;
  if (lane == 0) part_w[warp] = wsum;
  __syncthreads();
  if (warp != 0) return;
  for (int k = 1; k < group; ++k) {
    const float4 t = part_acc[k][lane];
    acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
    wsum += part_w[k];
  }
  const int64_t row = static_cast<int64_t>(bs) * a.H + g * HG + h;
  const float inv = wsum > 0.0f ? __frcp_rn(wsum) : 0.0f;
  store_out4(a.out, row * kLatent + quarter * 128 + lane * 4,
             make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv), a.out_f32 != 0);
  if (quarter == 0 && lane == 0)
    a.lse[row] = (wsum > 0.0f) ? m + fast_log2(wsum) * 0.69314718055994531f : -INFINITY;
}

// Debug: the decode's index resolution and dequantization (the f16 operand
// values) written to HBM.  One warp per (b, s, k) row; 576 columns per row
// for 352-byte pool rows, 512 for 288-byte (latent-only) rows.
__global__ void __launch_bounds__(256) debug_gather_kernel(GatherArgs a) {
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t n = static_cast<int64_t>(a.B) * a.Sq * a.K;
  if (gw >= n) return;
  const int k = static_cast<int>(gw % a.K);
  const int64_t bs = gw / a.K;
  const int b = static_cast<int>(bs / a.Sq), s = static_cast<int>(bs % a.Sq);
  const int64_t l_eff = static_cast<int64_t>(__ldg(a.seq_lens + b)) - (a.Sq - 1 - s);
  int32_t slot = 0;
  if (lane == 0)
    slot = resolve_slot(a.topk + bs * a.K, k, a.K, l_eff, a.page_table + static_cast<int64_t>(b) * a.pt_stride,
                        a.pt_stride, a.num_slots, a.dev_err);
  slot = __shfl_sync(0xFFFFFFFFu, slot, 0);
  const int row_bytes = a.rope ? kRowBytes : kRowBytesLatent;
  uint32_t wlo = 0, whi = 0, wex = 0;
  if (slot >= 0) {
    const uint32_t* row = reinterpret_cast<const uint32_t*>(a.pool + static_cast<int64_t>(slot) * row_bytes);
    wlo = __ldg(row + lane);
    whi = __ldg(row + 32 + lane);
    wex = lane < (a.rope ? 24 : 8) ? __ldg(row + 64 + lane) : 0u;
  }
  DequantRow d = dequant_row_words(wlo, whi, wex, lane, dequant_scale_selector(lane));
  if (slot < 0) {
    d.lat_lo = d.lat_hi = make_uint4(0, 0, 0, 0);
    d.rope = make_uint2(0, 0);
  }
  __half* out = static_cast<__half*>(a.rows) + gw * (a.rope ? kQk : kLatent);
  *reinterpret_cast<uint4*>(out + 8 * lane) = d.lat_lo;
  *reinterpret_cast<uint4*>(out + 256 + 8 * lane) = d.lat_hi;
  if (a.rope && lane >= 8 && lane < 24)
    *reinterpret_cast<uint2*>(out + 512 + 4 * (lane - 8)) = d.rope;
}

// The FP8 scratch copy (the comparison path the README's kv4mla bullet
// measures against): for every (b, s, k), the NVFP4 row the key selects,
// dequantized as in the decode and cast to E4M3, into a 576-byte row of
// a.rows; masked keys give zero rows.  One warp per (b, s, k) row.
__global__ void __launch_bounds__(256) fp8_scratch_kernel(GatherArgs a) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t n = static_cast<int64_t>(a.B) * a.Sq * a.K;
  if (gw >= n) return;
  const int k = static_cast<int>(gw % a.K);
  const int64_t bs = gw / a.K;
  const int b = static_cast<int>(bs / a.Sq), s = static_cast<int>(bs % a.Sq);
  const int64_t l_eff = static_cast<int64_t>(__ldg(a.seq_lens + b)) - (a.Sq - 1 - s);
  int32_t slot = 0;
  if (lane == 0)
    slot = resolve_slot(a.topk + bs * a.K, k, a.K, l_eff,
                        a.page_table + static_cast<int64_t>(b) * a.pt_stride, a.pt_stride,
                        a.num_slots, a.dev_err);
  slot = __shfl_sync(0xFFFFFFFFu, slot, 0);
  uint32_t wlo = 0, whi = 0, wex = 0;
  if (slot >= 0) {
    const uint32_t* row =
        reinterpret_cast<const uint32_t*>(a.pool + static_cast<int64_t>(slot) * kRowBytes);
    wlo = __ldg(row + lane);
    whi = __ldg(row + 32 + lane);
    wex = lane < 24 ? __ldg(row + 64 + lane) : 0u;
  }
  const DequantRow d = dequant_row_words(wlo, whi, wex, lane, dequant_scale_selector(lane));
  auto e4m3x8 = [](const uint4& h) {                     // 8 f16 -> 8 E4M3 bytes
    return make_uint2(f16x2_to_e4m3x2(h.x) | (f16x2_to_e4m3x2(h.y) << 16),
                      f16x2_to_e4m3x2(h.z) | (f16x2_to_e4m3x2(h.w) << 16));
  };
  uint2 lo = e4m3x8(d.lat_lo), hi = e4m3x8(d.lat_hi);
  uint32_t rope = f16x2_to_e4m3x2(d.rope.x) | (f16x2_to_e4m3x2(d.rope.y) << 16);
  if (slot < 0) {
    lo = hi = make_uint2(0, 0);
    rope = 0;
  }
  uint8_t* out = static_cast<uint8_t*>(a.rows) + gw * kRowBytesFp8;
  *reinterpret_cast<uint2*>(out + 8 * lane) = lo;
  *reinterpret_cast<uint2*>(out + 256 + 8 * lane) = hi;
  if (lane >= 8 && lane < 24) *reinterpret_cast<uint32_t*>(out + 512 + 4 * (lane - 8)) = rope;
}

// The scratch path's indexing: for n = b*Sq + s, page-table row n holds the
// pages n*(K/64) .. n*(K/64) + K/64 - 1 of the scratch buffer, and the top-k
// list of one-token request n keeps position k where key k of the original
// query is valid (0 <= topk[b,s,k] < L_eff) and -1 where it is masked; every
// such request has length K.  One thread per top-k entry.
__global__ void __launch_bounds__(256) fp8_scratch_index_kernel(const int32_t* topk,
                                                                const int32_t* seq_lens, int B,
                                                                int Sq, int K, int32_t* pt_out,
                                                                int32_t* topk_out,
                                                                int32_t* lens_out) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t n_keys = static_cast<int64_t>(B) * Sq * K;
  const int pages = K / kPage;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_keys;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = i / K;
    const int k = static_cast<int>(i % K);
    const int b = static_cast<int>(n / Sq), s = static_cast<int>(n % Sq);
    const int64_t l_eff = static_cast<int64_t>(seq_lens[b]) - (Sq - 1 - s);
    const int32_t idx = topk[i];
    topk_out[i] = (idx >= 0 && idx < l_eff) ? k : -1;
    if (k < pages) pt_out[n * pages + k] = static_cast<int32_t>(n * pages + k);
    if (k == 0) lens_out[n] = K;
  }
}

template <int HG, int FMT>
cudaError_t configure_decode() {
  static cudaError_t state = cudaErrorNotReady;   // per process; attributes are per kernel
  if (state == cudaErrorNotReady) {
    // The setmaxnreg split assumes the block is launched with exactly
    // kLaunchRegs registers per thread; with fewer the compute warpgroups'
    // increase could never be granted, so refuse to launch instead.
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, decode_kernel<HG, FMT>);
    if (e == cudaSuccess && (attr.numRegs != kLaunchRegs || attr.maxThreadsPerBlock < kThreads))
      e = cudaErrorInvalidConfiguration;
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_kernel<HG, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(Layout<HG, FMT>::smem_bytes));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_kernel<HG, FMT>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    state = e;
  }
  return state;
}

template <int HG, int FMT>
int max_active_clusters_hg(int splits) {
  static int known[kMaxClusterSplits + 1] = {};   // 0 unknown, else 1 + the count
  if (splits < 2 || splits > kMaxClusterSplits) return 0;
  if (known[splits] == 0) {
    int n = 0;
    if (configure_decode<HG, FMT>() == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(splits);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = Layout<HG, FMT>::smem_bytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = splits;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, decode_kernel<HG, FMT>, &cfg) != cudaSuccess) n = 0;
    }
    (void)cudaGetLastError();
    known[splits] = 1 + (n > 0 ? n : 0);
  }
  return known[splits] - 1;
}

template <int HG, int FMT>
cudaError_t launch_decode_hg(const DecodeArgs& a, cudaStream_t stream) {
  const size_t smem = Layout<HG, FMT>::smem_bytes;
  cudaError_t e = configure_decode<HG, FMT>();
  if (e != cudaSuccess) return e;
  const int units = a.B * a.Sq * (a.H / HG);
  e = launch_pdl(decode_kernel<HG, FMT>, static_cast<unsigned>(units * a.splits), kThreads, smem, stream,
                 a.cluster_merge ? a.splits : 1, a);
  if (e == cudaSuccess && a.after_decode != nullptr) e = cudaEventRecord(a.after_decode, stream);
  if (e != cudaSuccess || a.splits == 1 || a.cluster_merge) return e;
  // a group of warps per (unit, head, column quarter), at most eight
  // partials per warp
  const int group = (a.splits + 7) / 8 < kMergeMaxWarps ? (a.splits + 7) / 8 : kMergeMaxWarps;
  if (static_cast<int64_t>(units) * HG * 4 > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  return launch_pdl(merge_kernel, static_cast<unsigned>(units * HG * 4),
                    static_cast<unsigned>(32 * group), 0, stream, 1, a, units, group);
}

template <int FMT>
size_t decode_smem_bytes_r(int HG) {
  switch (HG) {
    case 16: return Layout<16, FMT>::smem_bytes;
    case 32: return Layout<32, FMT>::smem_bytes;
    case 64: return Layout<64, FMT>::smem_bytes;
    default: return 0;
  }
}

template <int FMT>
int decode_max_active_clusters_r(int HG, int splits) {
  switch (HG) {
    case 16: return max_active_clusters_hg<16, FMT>(splits);
    case 32: return max_active_clusters_hg<32, FMT>(splits);
    case 64: return max_active_clusters_hg<64, FMT>(splits);
    default: return 0;
  }
}

template <int FMT>
cudaError_t launch_decode_r(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.HG) {
    case 16: return launch_decode_hg<16, FMT>(a, stream);
    case 32: return launch_decode_hg<32, FMT>(a, stream);
    case 64: return launch_decode_hg<64, FMT>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t decode_smem_bytes(int HG, int fmt) {
  switch (fmt) {
    case kFmtNvfp4: return decode_smem_bytes_r<kFmtNvfp4>(HG);
    case kFmtNvfp4Latent: return decode_smem_bytes_r<kFmtNvfp4Latent>(HG);
    case kFmtFp8: return decode_smem_bytes_r<kFmtFp8>(HG);
    default: return 0;
  }
}

int decode_max_active_clusters(int HG, int splits, int fmt) {
  switch (fmt) {
    case kFmtNvfp4: return decode_max_active_clusters_r<kFmtNvfp4>(HG, splits);
    case kFmtNvfp4Latent: return decode_max_active_clusters_r<kFmtNvfp4Latent>(HG, splits);
    case kFmtFp8: return decode_max_active_clusters_r<kFmtFp8>(HG, splits);
    default: return 0;
  }
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.fmt) {
    case kFmtNvfp4: return launch_decode_r<kFmtNvfp4>(a, stream);
    case kFmtNvfp4Latent: return launch_decode_r<kFmtNvfp4Latent>(a, stream);
    case kFmtFp8: return launch_decode_r<kFmtFp8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fp8_scratch(const GatherArgs& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.Sq * a.K;
  if (rows <= 0) return cudaSuccess;
  return launch_pdl(fp8_scratch_kernel, static_cast<unsigned>((rows + 7) / 8), 256, 0, stream, 1,
                    a);
}

cudaError_t launch_fp8_scratch_index(const int32_t* topk, const int32_t* seq_lens, int B, int Sq,
                                     int K, int32_t* pt_out, int32_t* topk_out,
                                     int32_t* lens_out, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(B) * Sq * K;
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(fp8_scratch_index_kernel, static_cast<unsigned>(blocks), 256, 0, stream, 1,
                    topk, seq_lens, B, Sq, K, pt_out, topk_out, lens_out);
}

cudaError_t launch_debug_gather(const GatherArgs& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.Sq * a.K;
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;
  debug_gather_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kv4

