// kv4_dcp.cu -- decode-context parallelism over the NVFP4 pool (numinousmuses
// "inference-optimizations" README, "Parallelism and disaggregation": each
// rank attends over the part of the context it holds and the ranks' (o, lse)
// are merged).
//
// Ownership (this project's reading; the page names no rule): physical page p
// of the pool lives on rank p mod world, as page p / world of that rank's own
// pool, which therefore holds only about 1/world of the pages.  The rank's
// cache writes go to its local slots (dcp_local_slots_kernel), and its decode
// reads through a rank-local page table (dcp_local_page_table_kernel) that
// maps each owned page to its local index.  A rank's top-k list keeps the
// positions whose page it owns and replaces the others by -1 (masked), so
// the ranks partition every query's keys.  A position outside [0, L_eff)
// stays masked everywhere; a position whose page-table entry cannot be read
// (page index past the table or a negative entry) is kept on rank 0 only, so
// that exactly one rank's decode reports it.  After each rank's decode has
// written its normalized fp32 o and its lse, and the ranks have exchanged
// them (an all-gather), merge_partials_kernel combines the R partials of
// every (query token, head) row by log-sum-exp into the bf16 output.
#include "kv4_device.cuh"
#include "kv4_launch.h"

#include <math.h>

namespace kv4 {
namespace {

__global__ void __launch_bounds__(256) dcp_mask_topk_kernel(const int32_t* topk,
                                                            const int32_t* page_table,
                                                            int64_t pt_stride,
                                                            const int32_t* seq_lens, int B,
                                                            int Sq, int K, int world, int rank,
                                                            int32_t* topk_out) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t n = static_cast<int64_t>(B) * Sq * K;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t bs = i / K;
    const int b = static_cast<int>(bs / Sq), s = static_cast<int>(bs % Sq);
    const int64_t l_eff = static_cast<int64_t>(seq_lens[b]) - (Sq - 1 - s);
    const int32_t idx = topk[i];
    int32_t keep = -1;
    if (idx >= 0 && idx < l_eff) {
      const int64_t pi = idx / kPage;
      const int32_t page = pi < pt_stride ? page_table[static_cast<int64_t>(b) * pt_stride + pi] : -1;
      if (page < 0) keep = rank == 0 ? idx : -1;             // unreadable: rank 0 reports it
      else if (page % world == rank) keep = idx;
    }
    topk_out[i] = keep;
  }
}

// The same ownership rule, with the rank's kept positions moved to the front
// of each query's list in their order and -1 after them, and their number
// in count_out[b * Sq + s]: a decode that walks only that many entries
// (kv4_sparse_mla_decode_partial_counted) then does the rank's share of the
// keys instead of every tile of the list.  One block of 256 threads per
// query: thread t decides a contiguous run of kCompactPer entries at a time
// (all of their loads in flight), and a block-wide prefix sum of the kept
// counts places them.
constexpr int kCompactThreads = 256;
constexpr int kCompactPer = 8;

__global__ void __launch_bounds__(kCompactThreads) dcp_compact_topk_kernel(
    const int32_t* topk, const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
    int B, int Sq, int K, int world, int rank, int32_t* topk_out, int32_t* count_out) {
  grid_dependency_wait();
  grid_launch_dependents();
  __shared__ int warp_sums[kCompactThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t rows = static_cast<int64_t>(B) * Sq;
  for (int64_t bs = blockIdx.x; bs < rows; bs += gridDim.x) {
    const int b = static_cast<int>(bs / Sq), s = static_cast<int>(bs % Sq);
    const int64_t l_eff = static_cast<int64_t>(seq_lens[b]) - (Sq - 1 - s);
    const int32_t* in = topk + bs * K;
    int32_t* out = topk_out + bs * K;
    int base = 0;                                   // kept entries of earlier rounds
    for (int k0 = 0; k0 < K; k0 += kCompactThreads * kCompactPer) {
      int32_t keep[kCompactPer];
      int n = 0;
#pragma unroll
      for (int j = 0; j < kCompactPer; ++j) {
        const int k = k0 + tid * kCompactPer + j;
        keep[j] = -1;
        if (k < K) {
          const int32_t idx = in[k];
          if (idx >= 0 && idx < l_eff) {
            const int64_t pi = idx / kPage;
            const int32_t page =
                pi < pt_stride ? page_table[static_cast<int64_t>(b) * pt_stride + pi] : -1;
            if (page < 0) keep[j] = rank == 0 ? idx : -1;  // unreadable: rank 0 reports it
            else if (page % world == rank) keep[j] = idx;
          }
        }
        n += keep[j] >= 0;
      }
      // exclusive prefix of n over the block, in thread order
      int incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += v;
      }
      if (lane == 31) warp_sums[warp] = incl;
      __syncthreads();
      int before = 0, total = 0;
#pragma unroll
      for (int w2 = 0; w2 < kCompactThreads / 32; ++w2) {
        const int ws = warp_sums[w2];
        before += w2 < warp ? ws : 0;
        total += ws;
      }
      int pos = base + before + incl - n;
#pragma unroll
      for (int j = 0; j < kCompactPer; ++j)
        if (keep[j] >= 0) out[pos++] = keep[j];
      base += total;
      __syncthreads();                              // warp_sums is reused
    }
    for (int k = base + tid; k < K; k += kCompactThreads) out[k] = -1;
    if (tid == 0) count_out[bs] = base;
  }
}

// Rank-local page table: entry p (a physical page) becomes p / world where
// the rank owns it (p >= 0, p % world == rank) and -1 elsewhere -- a
// position on another rank's page never reaches this rank's decode (its
// top-k list masks it), and a negative entry stays unreadable, so the rank
// whose top-k keeps that position (rank 0) reports it.
__global__ void __launch_bounds__(256) dcp_local_page_table_kernel(const int32_t* page_table,
                                                                   int64_t n, int world,
                                                                   int rank, int32_t* out) {
  grid_dependency_wait();
  grid_launch_dependents();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t p = page_table[i];
    out[i] = (p >= 0 && p % world == rank) ? p / world : -1;
  }
}

// Rank-local cache-write slots: global slot s (page s / 64) becomes
// (page / world) * 64 + s % 64 on the page's owner and -1 (no write)
// elsewhere; a negative slot stays -1.
__global__ void __launch_bounds__(256) dcp_local_slots_kernel(const int64_t* slots, int64_t n,
                                                              int world, int rank,
                                                              int64_t* out) {
  grid_dependency_wait();
  grid_launch_dependents();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t s = slots[i];
    const int64_t page = s >= 0 ? s / kPage : -1;
    out[i] = (page >= 0 && page % world == rank) ? (page / world) * kPage + s % kPage : -1;
  }
}

// One warp per row: out = sum_r exp(lse_r - m) o_r / sum_r exp(lse_r - m),
// lse = m + log sum_r exp(lse_r - m), m = max_r lse_r; a partial with
// lse = -inf has weight 0; no finite lse gives out = 0, lse = -inf.
__global__ void __launch_bounds__(256) merge_partials_kernel(const float* o_parts,
                                                             const float* lse_parts, int R,
                                                             int64_t n_rows,
                                                             __nv_bfloat16* out, float* lse) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= n_rows) return;
  float m = -INFINITY;
  for (int r = 0; r < R; ++r) m = fmaxf(m, lse_parts[r * n_rows + row]);
  float4 acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.0f;
  if (m != -INFINITY) {
    for (int r = 0; r < R; ++r) {
      const float lr = lse_parts[r * n_rows + row];
      if (lr == -INFINITY) continue;
      const float w = expf(lr - m);
      wsum += w;
      const float4* o = reinterpret_cast<const float4*>(o_parts + (r * n_rows + row) * kLatent);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 v = o[j * 32 + lane];
        acc[j].x += w * v.x; acc[j].y += w * v.y; acc[j].z += w * v.z; acc[j].w += w * v.w;
      }
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[j].x * inv, acc[j].y * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[j].z * inv, acc[j].w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + row * kLatent + j * 128 + lane * 4) = pk;
  }
  if (lane == 0) lse[row] = wsum > 0.0f ? m + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_dcp_mask_topk(const int32_t* topk, const int32_t* page_table,
                                 int64_t pt_stride, const int32_t* seq_lens, int B, int Sq,
                                 int K, int world, int rank, int32_t* topk_out,
                                 cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(B) * Sq * K;
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(dcp_mask_topk_kernel, static_cast<unsigned>(blocks), 256, 0, stream, 1, topk,
                    page_table, pt_stride, seq_lens, B, Sq, K, world, rank, topk_out);
}

cudaError_t launch_dcp_compact_topk(const int32_t* topk, const int32_t* page_table,
                                    int64_t pt_stride, const int32_t* seq_lens, int B, int Sq,
                                    int K, int world, int rank, int32_t* topk_out,
                                    int32_t* count_out, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(B) * Sq;
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = rows < 4096 ? rows : 4096;      // one block per query
  return launch_pdl(dcp_compact_topk_kernel, static_cast<unsigned>(blocks), kCompactThreads, 0,
                    stream, 1,
                    topk, page_table, pt_stride, seq_lens, B, Sq, K, world, rank, topk_out,
                    count_out);
}

cudaError_t launch_dcp_local_page_table(const int32_t* page_table, int64_t n, int world,
                                        int rank, int32_t* out, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(dcp_local_page_table_kernel, static_cast<unsigned>(blocks), 256, 0, stream, 1,
                    page_table, n, world, rank, out);
}

cudaError_t launch_dcp_local_slots(const int64_t* slots, int64_t n, int world, int rank,
                                   int64_t* out, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(dcp_local_slots_kernel, static_cast<unsigned>(blocks), 256, 0, stream, 1,
                    slots, n, world, rank, out);
}

cudaError_t launch_merge_partials(const float* o_parts, const float* lse_parts, int R,
                                  int64_t n_rows, void* out_bf16, float* lse,
                                  cudaStream_t stream) {
  if (n_rows <= 0) return cudaSuccess;
  const int64_t blocks = (n_rows + 7) / 8;
  return launch_pdl(merge_partials_kernel, static_cast<unsigned>(blocks), 256, 0, stream, 1,
                    o_parts, lse_parts, R, n_rows, static_cast<__nv_bfloat16*>(out_bf16), lse);
}

}  // namespace kv4
