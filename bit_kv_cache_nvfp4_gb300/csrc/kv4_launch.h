// kv4_launch.h -- internal launch interface between the C ABI (kv4_capi.cu)
// and the kernels.  Not installed; the public interface is include/kv4mla.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace kv4 {

// Row formats of the pool:
//   kFmtNvfp4        352 B: E2M1 latent codes, E4M3 scales, E4M3 rope; q of 576
//   kFmtNvfp4Latent  288 B: the same without rope; q of 512
//   kFmtFp8          576 B: E4M3 latent and rope (the comparison row); q of 576
enum RowFormat : int { kFmtNvfp4 = 0, kFmtNvfp4Latent = 1, kFmtFp8 = 2 };

struct QuantizeArgs {
  const void* latent;
  int64_t latent_stride;
  const void* rope;
  int64_t rope_stride;
  const int64_t* slots;
  int64_t n_tokens;
  uint8_t* pool;
  int64_t num_slots;
  int row_bytes;               // 352 (latent + rope) or 288 (latent only; rope unused)
  int32_t* dev_err;
  int mse;                     // 1: MSE-searched block scales instead of amax/6
  int fp8;                     // 1: 576-byte FP8 rows (E4M3 of every value; row_bytes 576)
};

struct DecodeArgs {
  const void* q;               // bf16 [B, Sq, H, 576]
  const uint8_t* pool;
  int64_t num_slots;
  const int32_t* page_table;
  int64_t pt_stride;
  const int32_t* topk;         // int32 [B, Sq, K]
  int K;
  const int32_t* seq_lens;
  int B, Sq, H;
  int HG;                      // heads per thread block: 16, 32 or 64
  int splits;                  // split-K partitions (>= 1)
  int tiles_per_split;
  float sm_scale;
  void* out;                   // bf16 [B, Sq, H, 512]
  float* lse;                  // fp32 [B, Sq, H]
  float* ws_o;                 // fp32 [units, splits, HG, 512] when splits > 1
  float* ws_lse;               // fp32 [units, splits, HG]
  int32_t* dev_err;
  uint64_t timeout_ns;
  int fault_site;
  cudaEvent_t after_decode;    // recorded between the decode and merge kernels (may be null)
  int cluster_merge;           // splits > 1 merged inside a cluster of `splits` blocks
  int fmt;                     // row format: kFmtNvfp4, kFmtNvfp4Latent or kFmtFp8
  int out_f32;                 // 1: out is fp32 (a context-parallel rank's partial), else bf16
  int early_inputs;            // 1: q, page table, top-k and lengths may be read before the
                               //    previous kernel (this call's cache write) has finished
  const int32_t* k_count;      // int32 [B * Sq] or null: each query walks only the first
                               //    k_count[b * Sq + s] entries of its list (never with
                               //    early_inputs)
};

struct GatherArgs {
  const uint8_t* pool;
  int64_t num_slots;
  const int32_t* page_table;
  int64_t pt_stride;
  const int32_t* topk;
  int K;
  const int32_t* seq_lens;
  int B, Sq;
  void* rows;                  // f16 [B, Sq, K, 576] (rope) or [B, Sq, K, 512]
  int rope;                    // 1: 352-byte rows; 0: 288-byte latent-only rows
  int32_t* dev_err;
};

// Launch of one of the library's kernels with programmatic stream
// serialization allowed (the kernel may begin while the previous kernel of
// the stream finishes; it calls grid_dependency_wait() before touching
// global memory), optionally as clusters of `cluster_x` blocks.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_quantize_write(const QuantizeArgs& a, int num_sms, cudaStream_t stream);
// Decode-context parallelism: the top-k list of one rank (keys on pages it
// owns, page % world == rank), and the merge of the ranks' (o, lse).
cudaError_t launch_dcp_mask_topk(const int32_t* topk, const int32_t* page_table,
                                 int64_t pt_stride, const int32_t* seq_lens, int B, int Sq,
                                 int K, int world, int rank, int32_t* topk_out,
                                 cudaStream_t stream);
cudaError_t launch_dcp_compact_topk(const int32_t* topk, const int32_t* page_table,
                                    int64_t pt_stride, const int32_t* seq_lens, int B, int Sq,
                                    int K, int world, int rank, int32_t* topk_out,
                                    int32_t* count_out, cudaStream_t stream);
cudaError_t launch_dcp_local_page_table(const int32_t* page_table, int64_t n, int world,
                                        int rank, int32_t* out, cudaStream_t stream);
cudaError_t launch_dcp_local_slots(const int64_t* slots, int64_t n, int world, int rank,
                                   int64_t* out, cudaStream_t stream);
cudaError_t launch_merge_partials(const float* o_parts, const float* lse_parts, int R,
                                  int64_t n_rows, void* out_bf16, float* lse,
                                  cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_debug_gather(const GatherArgs& a, cudaStream_t stream);
// The FP8 scratch copy of the rows the keys select: a.rows is uint8
// [B*Sq*K, 576] (E4M3 of the dequantized NVFP4 values; masked keys 0).
cudaError_t launch_fp8_scratch(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_fp8_scratch_index(const int32_t* topk, const int32_t* seq_lens, int B, int Sq,
                                     int K, int32_t* pt_out, int32_t* topk_out,
                                     int32_t* lens_out, cudaStream_t stream);
size_t decode_smem_bytes(int HG, int fmt);
// How many clusters of `splits` blocks of the HG variant can be resident at
// once on this device (0: such clusters cannot run).  A unit split in two
// runs as a cluster of two blocks that merge through distributed shared
// memory; more splits merge through the workspace.
int decode_max_active_clusters(int HG, int splits, int fmt);
constexpr int kMaxClusterSplits = 2;

}  // namespace kv4
