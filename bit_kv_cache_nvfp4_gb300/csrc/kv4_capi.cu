// kv4_capi.cu -- the extern "C" entry points of libkv4mla.so declared in
// include/kv4mla.h: argument validation, the split-K planner and the
// stream-ordered launches.  The library never allocates device memory and
// never synchronizes.
#include "kv4mla.h"
#include "kv4_launch.h"

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <new>

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];          // 0 = not queried yet
std::atomic<int> g_cc[kMaxDevices];           // major*10 + minor
std::atomic<int64_t> g_timeout_ns{1000000000};  // bounded-wait limit: 1 s
std::atomic<int> g_fault_site{0};
std::atomic<void*> g_timing_event{nullptr};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count and compute capability of the current device (cached).
kv4_status device_info(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return KV4_ERR_LAUNCH;
  int n = g_sms[dev].load(std::memory_order_relaxed);
  int cc = g_cc[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return KV4_ERR_LAUNCH;
    cc = major * 10 + minor;
    g_cc[dev].store(cc, std::memory_order_relaxed);
    g_sms[dev].store(n, std::memory_order_relaxed);
  }
  if (cc != 103) return KV4_ERR_ARCH;           // built for sm_103a only
  *sms = n;
  return KV4_OK;
}

int heads_per_block(int H) {
  if (H == 16 || H == 32 || H == 64) return H;
  if (H > 64 && H <= 256 && H % 64 == 0) return 64;
  return 0;
}

constexpr double kBlockFixedTiles = 2.0;

struct Plan {
  int HG, units, tiles, splits, tiles_per_split;
  bool cluster_merge;          // the splits of a unit merge inside a thread-block cluster
  size_t ws_bytes;
};

// Split-K planner: pick the number of partitions S of each query's tiles
// that minimizes (waves of thread blocks) x (fixed cost of a block + tiles
// per partition), plus a charge for the merge when S > 1 -- half a tile,
// and 0.06 tile more for every partial beyond two (the merge kernel reads
// them one row per warp) -- ties going to the smaller S.  One block runs per
// SM.  The fixed cost (prologue: Q load and conversion, first dependent
// loads; epilogue: output or partial writes) is about two tiles of work.
// (Fitted to graph-timed sweeps of forced S on the five workloads.)
Plan make_plan(int B, int Sq, int H, int K, int force_splits, int sms, int fmt) {
  Plan p{};
  p.HG = heads_per_block(H);
  p.units = B * Sq * (H / p.HG);
  p.tiles = (K + KV4_TILE_KEYS - 1) / KV4_TILE_KEYS;
  int S = 1;
  if (p.tiles > 1) {
    if (force_splits > 0) {
      S = force_splits < p.tiles ? force_splits : p.tiles;
    } else {
      double best = 1e300;
      for (int c = 1; c <= p.tiles; ++c) {
        const long long waves = (static_cast<long long>(p.units) * c + sms - 1) / sms;
        const int per = (p.tiles + c - 1) / c;
        const double cost = static_cast<double>(waves) * (kBlockFixedTiles + per) +
                            (c > 1 ? 0.5 + 0.06 * (c > 2 ? c - 2 : 0) : 0.0);
        if (cost < best - 1e-9) { best = cost; S = c; }
      }
    }
  }
  p.tiles_per_split = p.tiles > 0 ? (p.tiles + S - 1) / S : 0;
  p.splits = p.tiles_per_split > 0 ? (p.tiles + p.tiles_per_split - 1) / p.tiles_per_split : 1;
  // Two splits of a unit run as one cluster and merge in distributed shared
  // memory (no workspace, no merge kernel) when all units' clusters fit on
  // the device at once; otherwise the partials go to the workspace for
  // merge_kernel.
  p.cluster_merge = p.splits > 1 && p.splits <= kv4::kMaxClusterSplits &&
                    p.units <= kv4::decode_max_active_clusters(p.HG, p.splits, fmt);
  p.ws_bytes = (p.splits > 1 && !p.cluster_merge)
                   ? static_cast<size_t>(p.units) * p.splits * p.HG * (KV4_LATENT + 1) *
                         sizeof(float)
                   : 0;
  return p;
}

kv4_status check_decode_shape(int B, int Sq, int H, int K) {
  if (B < 0 || Sq < 1 || K < 0) return KV4_ERR_INVALID_ARG;
  if (heads_per_block(H) == 0) return KV4_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Sq * H > (1LL << 30)) return KV4_ERR_INVALID_ARG;
  return KV4_OK;
}

}  // namespace

namespace {

// The entry points below share these bodies.  For the cache write, `rope`
// selects the 352-byte row (latent + rope) or the 288-byte latent-only row;
// for the decode, `fmt` is the row format (kv4_launch.h).
kv4_status quantize_impl(const void* latent_dev, int64_t latent_row_stride, const void* rope_dev,
                         int64_t rope_row_stride, const int64_t* slot_mapping_dev,
                         int64_t n_tokens, uint8_t* pool_dev, int64_t num_slots,
                         int32_t* dev_err, kv4_stream_t stream, bool rope, bool mse = false) {
  if (n_tokens < 0 || num_slots < 0) return KV4_ERR_INVALID_ARG;
  if (n_tokens == 0) return KV4_OK;
  if (!latent_dev || (rope && !rope_dev) || !slot_mapping_dev || !pool_dev)
    return KV4_ERR_INVALID_ARG;
  if (latent_row_stride < KV4_LATENT || latent_row_stride % 8 != 0 ||
      (rope && (rope_row_stride < KV4_ROPE || rope_row_stride % 8 != 0)))
    return KV4_ERR_INVALID_ARG;
  if (!aligned16(latent_dev) || (rope && !aligned16(rope_dev)) || !aligned16(pool_dev) ||
      (reinterpret_cast<uintptr_t>(slot_mapping_dev) & 7u) != 0)
    return KV4_ERR_INVALID_ARG;
  const int row_bytes = rope ? KV4_ROW_BYTES : KV4_ROW_BYTES_LATENT;
  if (num_slots > INT64_MAX / row_bytes) return KV4_ERR_INVALID_ARG;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  kv4::QuantizeArgs a{latent_dev, latent_row_stride, rope ? rope_dev : nullptr,
                      rope ? rope_row_stride : 0, slot_mapping_dev, n_tokens, pool_dev,
                      num_slots, row_bytes, dev_err, mse ? 1 : 0, 0};
  return kv4::launch_quantize_write(a, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KV4_OK
             : KV4_ERR_LAUNCH;
}

kv4_status plan_impl(int B, int Sq, int H, int K, int force_splits, int* splits,
                     size_t* workspace_bytes, int fmt) {
  const kv4_status shape = check_decode_shape(B, Sq, H, K);
  if (shape != KV4_OK) return shape;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  const Plan p = make_plan(B, Sq, H, K, force_splits, sms, fmt);
  if (splits) *splits = p.splits;
  if (workspace_bytes) *workspace_bytes = p.ws_bytes;
  return KV4_OK;
}

// The decode's host-side argument checks (shape, page size, pointers,
// ranges, alignment), shared by every decode entry point and run before any
// device call.  KV4_OK with B == 0 means there is nothing to launch.
kv4_status check_decode_args(const void* q_dev, const uint8_t* pool_dev, int64_t num_slots,
                             const int32_t* page_table_dev, int64_t pt_stride, int page_size,
                             const int32_t* topk_idx_dev, int K, const int32_t* seq_lens_dev,
                             int B, int Sq, int H, const void* out_dev, const float* lse_dev) {
  const kv4_status shape = check_decode_shape(B, Sq, H, K);
  if (shape != KV4_OK) return shape;
  if (page_size != KV4_PAGE) return KV4_ERR_UNSUPPORTED;
  if (B == 0) return KV4_OK;
  if (!q_dev || !pool_dev || !page_table_dev || (K > 0 && !topk_idx_dev) || !seq_lens_dev ||
      !out_dev || !lse_dev)
    return KV4_ERR_INVALID_ARG;
  if (num_slots < 0 || num_slots > INT32_MAX || pt_stride < 1 || pt_stride > INT32_MAX)
    return KV4_ERR_INVALID_ARG;
  if (!aligned16(q_dev) || !aligned16(pool_dev) || !aligned16(out_dev) ||
      (reinterpret_cast<uintptr_t>(lse_dev) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(page_table_dev) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(topk_idx_dev) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(seq_lens_dev) & 3u) != 0)
    return KV4_ERR_INVALID_ARG;
  return KV4_OK;
}

kv4_status decode_impl(const void* q_dev, const uint8_t* pool_dev, int64_t num_slots,
                       const int32_t* page_table_dev, int64_t pt_stride, int page_size,
                       const int32_t* topk_idx_dev, int K, const int32_t* seq_lens_dev, int B,
                       int Sq, int H, float sm_scale, void* out_dev, float* lse_dev,
                       void* workspace_dev, size_t workspace_bytes, int force_splits,
                       int32_t* dev_err, kv4_stream_t stream, int fmt, bool out_f32 = false,
                       bool early_inputs = false, bool launch = true,
                       const int32_t* k_count = nullptr) {
  const kv4_status args = check_decode_args(q_dev, pool_dev, num_slots, page_table_dev, pt_stride,
                                            page_size, topk_idx_dev, K, seq_lens_dev, B, Sq, H,
                                            out_dev, lse_dev);
  if (args != KV4_OK || B == 0) return args;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  const Plan p = make_plan(B, Sq, H, K, force_splits, sms, fmt);
  if (p.ws_bytes > 0 &&
      (workspace_dev == nullptr || workspace_bytes < p.ws_bytes || !aligned16(workspace_dev)))
    return KV4_ERR_WORKSPACE;

  kv4::DecodeArgs a{};
  a.q = q_dev;
  a.pool = pool_dev;
  a.num_slots = num_slots;
  a.page_table = page_table_dev;
  a.pt_stride = pt_stride;
  a.topk = topk_idx_dev;
  a.K = K;
  a.seq_lens = seq_lens_dev;
  a.B = B;
  a.Sq = Sq;
  a.H = H;
  a.HG = p.HG;
  a.splits = p.splits;
  a.tiles_per_split = p.tiles_per_split;
  a.sm_scale = sm_scale;
  a.out = out_dev;
  a.lse = lse_dev;
  a.cluster_merge = p.cluster_merge ? 1 : 0;
  a.fmt = fmt;
  a.out_f32 = out_f32 ? 1 : 0;
  a.early_inputs = early_inputs ? 1 : 0;
  a.k_count = k_count;
  if (p.splits > 1 && !p.cluster_merge) {
    a.ws_o = static_cast<float*>(workspace_dev);
    a.ws_lse = a.ws_o + static_cast<size_t>(p.units) * p.splits * p.HG * KV4_LATENT;
  }
  a.dev_err = dev_err;
  a.timeout_ns = static_cast<uint64_t>(g_timeout_ns.load());
  a.fault_site = g_fault_site.load();
  a.after_decode = static_cast<cudaEvent_t>(g_timing_event.load());
  if (!launch) return KV4_OK;                  // arguments checked only
  return kv4::launch_decode(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KV4_OK
             : KV4_ERR_LAUNCH;
}

kv4_status gather_impl(const uint8_t* pool_dev, int64_t num_slots, const int32_t* page_table_dev,
                       int64_t pt_stride, int page_size, const int32_t* topk_idx_dev, int K,
                       const int32_t* seq_lens_dev, int B, int Sq, void* rows_dev,
                       int32_t* dev_err, kv4_stream_t stream, bool rope) {
  if (B < 0 || Sq < 1 || K < 0) return KV4_ERR_INVALID_ARG;
  if (page_size != KV4_PAGE) return KV4_ERR_UNSUPPORTED;
  if (B == 0 || K == 0) return KV4_OK;
  if (!pool_dev || !page_table_dev || !topk_idx_dev || !seq_lens_dev || !rows_dev)
    return KV4_ERR_INVALID_ARG;
  if (num_slots < 0 || num_slots > INT32_MAX || pt_stride < 1 || pt_stride > INT32_MAX)
    return KV4_ERR_INVALID_ARG;
  if (!aligned16(pool_dev) || !aligned16(rows_dev)) return KV4_ERR_INVALID_ARG;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  kv4::GatherArgs a{pool_dev, num_slots,    page_table_dev, pt_stride,   topk_idx_dev, K,
                    seq_lens_dev, B,     Sq,             rows_dev,    rope ? 1 : 0, dev_err};
  return kv4::launch_debug_gather(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KV4_OK
             : KV4_ERR_LAUNCH;
}

}  // namespace

extern "C" {

kv4_status kv4_quantize_write(const void* latent_dev, int64_t latent_row_stride,
                              const void* rope_dev, int64_t rope_row_stride,
                              const int64_t* slot_mapping_dev, int64_t n_tokens,
                              uint8_t* pool_dev, int64_t num_slots, int32_t* dev_err,
                              kv4_stream_t stream) {
  return quantize_impl(latent_dev, latent_row_stride, rope_dev, rope_row_stride,
                       slot_mapping_dev, n_tokens, pool_dev, num_slots, dev_err, stream, true);
}

kv4_status kv4_decode_plan(int B, int Sq, int H, int K, int force_splits, int* splits,
                           size_t* workspace_bytes) {
  return plan_impl(B, Sq, H, K, force_splits, splits, workspace_bytes, kv4::kFmtNvfp4);
}

kv4_status kv4_sparse_mla_decode(const void* q_dev, const uint8_t* pool_dev, int64_t num_slots,
                                 const int32_t* page_table_dev, int64_t pt_stride, int page_size,
                                 const int32_t* topk_idx_dev, int K, const int32_t* seq_lens_dev,
                                 int B, int Sq, int H, float sm_scale, void* out_dev,
                                 float* lse_dev, void* workspace_dev, size_t workspace_bytes,
                                 int force_splits, int32_t* dev_err, kv4_stream_t stream) {
  return decode_impl(q_dev, pool_dev, num_slots, page_table_dev, pt_stride, page_size,
                     topk_idx_dev, K, seq_lens_dev, B, Sq, H, sm_scale, out_dev, lse_dev,
                     workspace_dev, workspace_bytes, force_splits, dev_err, stream,
                     kv4::kFmtNvfp4);
}

kv4_status kv4_quantize_write_and_decode(
    const void* latent_dev, int64_t latent_row_stride, const void* rope_dev,
    int64_t rope_row_stride, const int64_t* slot_mapping_dev, int64_t n_tokens, uint8_t* pool_dev,
    int64_t num_slots, const void* q_dev, const int32_t* page_table_dev, int64_t pt_stride,
    int page_size, const int32_t* topk_idx_dev, int K, const int32_t* seq_lens_dev, int B, int Sq,
    int H, float sm_scale, void* out_dev, float* lse_dev, void* workspace_dev,
    size_t workspace_bytes, int force_splits, int32_t* dev_err, kv4_stream_t stream) {
  // the decode's arguments are checked before anything is launched
  const kv4_status d = decode_impl(q_dev, pool_dev, num_slots, page_table_dev, pt_stride,
                                   page_size, topk_idx_dev, K, seq_lens_dev, B, Sq, H, sm_scale,
                                   out_dev, lse_dev, workspace_dev, workspace_bytes, force_splits,
                                   dev_err, stream, kv4::kFmtNvfp4, false, false, false);
  if (d != KV4_OK) return d;
  const kv4_status w = quantize_impl(latent_dev, latent_row_stride, rope_dev, rope_row_stride,
                                     slot_mapping_dev, n_tokens, pool_dev, num_slots, dev_err,
                                     stream, true);
  if (w != KV4_OK) return w;
  return decode_impl(q_dev, pool_dev, num_slots, page_table_dev, pt_stride, page_size,
                     topk_idx_dev, K, seq_lens_dev, B, Sq, H, sm_scale, out_dev, lse_dev,
                     workspace_dev, workspace_bytes, force_splits, dev_err, stream,
                     kv4::kFmtNvfp4, false, n_tokens > 0);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Host-buffer pipe: the write-and-decode step fed from host memory, two steps
// in flight over two device staging areas.
// ---------------------------------------------------------------------------
struct kv4_host_pipe {
  struct Area {
    void* q;
    int32_t* topk;
    int32_t* lens;
    void* latent;
    void* rope;
    int64_t* slots;
    void* out;
    float* lse;
  };
  int B, Sq, H, K, force_splits;
  int64_t max_new;
  size_t q_bytes, topk_bytes, lens_bytes, out_bytes, lse_bytes;
  Area area[2];
  void* ws;
  size_t ws_bytes;
  cudaStream_t s_in, s_comp, s_out;
  cudaEvent_t in_ready[2], comp_done[2], out_done[2];
  bool used[2];
  uint64_t steps;
};

namespace {

size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// A step's smaller inputs (lengths, new tokens, slots, the top-k list), read
// by one kernel straight from page-locked host memory (which the device can
// address) into device staging.  Each small cudaMemcpyAsync from the host
// carried a fixed cost of several microseconds, which the copy-in stream
// paid once per input; one launch pays it once.
constexpr int kGatherMax = 5;
struct HostGather {
  const uint8_t* src[kGatherMax];
  uint8_t* dst[kGatherMax];
  size_t bytes[kGatherMax];
  int n;
};

__global__ void __launch_bounds__(256) host_gather_kernel(HostGather g) {
  const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (int i = 0; i < g.n; ++i) {
    const size_t n = g.bytes[i];
    const bool vec = ((reinterpret_cast<uintptr_t>(g.src[i]) | reinterpret_cast<uintptr_t>(g.dst[i]) |
                       n) & 15u) == 0;
    if (vec) {
      const uint4* s4 = reinterpret_cast<const uint4*>(g.src[i]);
      uint4* d4 = reinterpret_cast<uint4*>(g.dst[i]);
      for (size_t k = tid; k < n / 16; k += stride) d4[k] = s4[k];
    } else {
      for (size_t k = tid; k < n; k += stride) g.dst[i][k] = g.src[i][k];
    }
  }
}

// The device address of page-locked host memory, or nullptr when `p` is not
// page-locked host memory that this device can address.
const void* mapped_host(const void* p) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return attr.type == cudaMemoryTypeHost ? attr.devicePointer : nullptr;
}

// Byte sizes of one staging area's buffers and of the whole staging memory.
struct PipeSizes {
  size_t q, topk, lens, latent, rope, slots, out, lse, area, ws, total;
};

kv4_status pipe_sizes(int B, int Sq, int H, int K, int64_t max_new, int force_splits,
                      PipeSizes* z) {
  const kv4_status shape = check_decode_shape(B, Sq, H, K);
  if (shape != KV4_OK) return shape;
  if (B < 1 || max_new < 0 || max_new > INT32_MAX || force_splits < 0)
    return KV4_ERR_INVALID_ARG;
  int splits = 0;
  size_t ws = 0;
  const kv4_status st = plan_impl(B, Sq, H, K, force_splits, &splits, &ws, kv4::kFmtNvfp4);
  if (st != KV4_OK) return st;
  const size_t rows = static_cast<size_t>(B) * Sq * H;
  z->q = rows * KV4_QK_DIM * 2;
  z->topk = static_cast<size_t>(B) * Sq * K * 4;
  z->lens = static_cast<size_t>(B) * 4;
  z->latent = static_cast<size_t>(max_new) * KV4_LATENT * 2;
  z->rope = static_cast<size_t>(max_new) * KV4_ROPE * 2;
  z->slots = static_cast<size_t>(max_new) * 8;
  z->out = rows * KV4_LATENT * 2;
  z->lse = rows * 4;
  z->area = round256(z->q) + round256(z->topk) + round256(z->lens) + round256(z->latent) +
            round256(z->rope) + round256(z->slots) + round256(z->out) + round256(z->lse);
  z->ws = round256(ws);
  z->total = 2 * z->area + z->ws;
  return KV4_OK;
}

void destroy_events(kv4_host_pipe* p) {
  for (int i = 0; i < 2; ++i) {
    if (p->in_ready[i]) cudaEventDestroy(p->in_ready[i]);
    if (p->comp_done[i]) cudaEventDestroy(p->comp_done[i]);
    if (p->out_done[i]) cudaEventDestroy(p->out_done[i]);
  }
}

}  // namespace

extern "C" {

kv4_status kv4_host_pipe_bytes(int B, int Sq, int H, int K, int64_t max_new, int force_splits,
                               size_t* staging_bytes) {
  if (!staging_bytes) return KV4_ERR_INVALID_ARG;
  PipeSizes z{};
  const kv4_status st = pipe_sizes(B, Sq, H, K, max_new, force_splits, &z);
  if (st != KV4_OK) return st;
  *staging_bytes = z.total;
  return KV4_OK;
}

kv4_status kv4_host_pipe_create(int B, int Sq, int H, int K, int64_t max_new, int force_splits,
                                void* staging_dev, size_t staging_bytes, kv4_stream_t copy_in,
                                kv4_stream_t compute, kv4_stream_t copy_out,
                                kv4_host_pipe** pipe) {
  if (!pipe) return KV4_ERR_INVALID_ARG;
  *pipe = nullptr;
  PipeSizes z{};
  const kv4_status st = pipe_sizes(B, Sq, H, K, max_new, force_splits, &z);
  if (st != KV4_OK) return st;
  if (!staging_dev || (reinterpret_cast<uintptr_t>(staging_dev) & 255u) != 0 ||
      staging_bytes < z.total)
    return KV4_ERR_INVALID_ARG;
  kv4_host_pipe* p = new (std::nothrow) kv4_host_pipe{};
  if (!p) return KV4_ERR_LAUNCH;
  p->B = B;
  p->Sq = Sq;
  p->H = H;
  p->K = K;
  p->force_splits = force_splits;
  p->max_new = max_new;
  p->q_bytes = z.q;
  p->topk_bytes = z.topk;
  p->lens_bytes = z.lens;
  p->out_bytes = z.out;
  p->lse_bytes = z.lse;
  uint8_t* cur = static_cast<uint8_t*>(staging_dev);
  auto take = [&](size_t n) {
    uint8_t* r = cur;
    cur += round256(n);
    return r;
  };
  for (int i = 0; i < 2; ++i) {
    kv4_host_pipe::Area& a = p->area[i];
    a.q = take(z.q);
    a.topk = reinterpret_cast<int32_t*>(take(z.topk));
    a.lens = reinterpret_cast<int32_t*>(take(z.lens));
    a.latent = take(z.latent);
    a.rope = take(z.rope);
    a.slots = reinterpret_cast<int64_t*>(take(z.slots));
    a.out = take(z.out);
    a.lse = reinterpret_cast<float*>(take(z.lse));
  }
  p->ws = z.ws > 0 ? take(z.ws) : nullptr;
  p->ws_bytes = z.ws;
  p->s_in = reinterpret_cast<cudaStream_t>(copy_in);
  p->s_comp = reinterpret_cast<cudaStream_t>(compute);
  p->s_out = reinterpret_cast<cudaStream_t>(copy_out);
  for (int i = 0; i < 2; ++i) {
    if (cudaEventCreateWithFlags(&p->in_ready[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->comp_done[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->out_done[i], cudaEventDisableTiming) != cudaSuccess) {
      destroy_events(p);
      delete p;
      return KV4_ERR_LAUNCH;
    }
  }
  *pipe = p;
  return KV4_OK;
}

kv4_status kv4_host_pipe_step(kv4_host_pipe* p, const void* latent_host, const void* rope_host,
                              const int64_t* slots_host, int64_t n_new, uint8_t* pool_dev,
                              int64_t num_slots, const int32_t* page_table_dev, int64_t pt_stride,
                              int page_size, const void* q_host, const int32_t* topk_host,
                              const int32_t* seq_lens_host, float sm_scale, void* out_host,
                              float* lse_host, int32_t* dev_err) {
  if (!p) return KV4_ERR_INVALID_ARG;
  if (n_new < 0 || n_new > p->max_new) return KV4_ERR_INVALID_ARG;
  if (!q_host || (p->K > 0 && !topk_host) || !seq_lens_host || !out_host || !lse_host ||
      (n_new > 0 && (!latent_host || !rope_host || !slots_host)))
    return KV4_ERR_INVALID_ARG;
  const int s = static_cast<int>(p->steps & 1);
  const kv4_host_pipe::Area& a = p->area[s];
  // every device-side argument is checked before anything is enqueued
  const kv4_status d = decode_impl(a.q, pool_dev, num_slots, page_table_dev, pt_stride, page_size,
                                   a.topk, p->K, a.lens, p->B, p->Sq, p->H, sm_scale, a.out,
                                   a.lse, p->ws, p->ws_bytes, p->force_splits, dev_err, p->s_comp,
                                   kv4::kFmtNvfp4, false, false, false);
  if (d != KV4_OK) return d;
  if (n_new > 0 && (!pool_dev || num_slots < 0 || num_slots > INT64_MAX / KV4_ROW_BYTES))
    return KV4_ERR_INVALID_ARG;

  const size_t latent_bytes = static_cast<size_t>(n_new) * KV4_LATENT * 2;
  const size_t rope_bytes = static_cast<size_t>(n_new) * KV4_ROPE * 2;
  const size_t slot_bytes = static_cast<size_t>(n_new) * 8;
  bool ok = true;
  auto h2d = [&](void* dst, const void* src, size_t n) {
    if (ok && n > 0)
      ok = cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, p->s_in) == cudaSuccess;
  };
  auto d2h = [&](void* dst, const void* src, size_t n) {
    if (ok && n > 0)
      ok = cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, p->s_out) == cudaSuccess;
  };
  auto wait_on = [&](cudaStream_t stream, cudaEvent_t ev) {
    if (ok) ok = cudaStreamWaitEvent(stream, ev, 0) == cudaSuccess;
  };
  auto record = [&](cudaEvent_t ev, cudaStream_t stream) {
    if (ok) ok = cudaEventRecord(ev, stream) == cudaSuccess;
  };
  // inputs into area s once the step two before has finished computing from it
  if (p->used[s]) wait_on(p->s_in, p->comp_done[s]);
  h2d(a.q, q_host, p->q_bytes);
  // the other inputs: one gather kernel when all are device-addressable
  // page-locked memory, else one copy each
  {
    HostGather gat{};
    const void* srcs[kGatherMax] = {topk_host, seq_lens_host, latent_host, rope_host, slots_host};
    void* dsts[kGatherMax] = {a.topk, a.lens, a.latent, a.rope, a.slots};
    const size_t sizes[kGatherMax] = {p->topk_bytes, p->lens_bytes, latent_bytes, rope_bytes,
                                      slot_bytes};
    bool mapped = true;
    size_t total = 0;
    for (int i = 0; i < kGatherMax && mapped; ++i) {
      if (sizes[i] == 0) continue;
      const void* dev = mapped_host(srcs[i]);
      if (dev == nullptr) {
        mapped = false;
        break;
      }
      gat.src[gat.n] = static_cast<const uint8_t*>(dev);
      gat.dst[gat.n] = static_cast<uint8_t*>(dsts[i]);
      gat.bytes[gat.n] = sizes[i];
      ++gat.n;
      total += sizes[i];
    }
    if (mapped) {
      if (ok && gat.n > 0) {
        const size_t blocks = (total / 16 + 255) / 256;
        host_gather_kernel<<<static_cast<unsigned>(blocks < 152 ? (blocks > 0 ? blocks : 1) : 152),
                             256, 0, p->s_in>>>(gat);
        ok = cudaGetLastError() == cudaSuccess;
      }
    } else {
      for (int i = 0; i < kGatherMax; ++i) h2d(dsts[i], srcs[i], sizes[i]);
    }
  }
  record(p->in_ready[s], p->s_in);
  // the step, once its inputs are in and the step two before has read its
  // results out of area s
  wait_on(p->s_comp, p->in_ready[s]);
  if (p->used[s]) wait_on(p->s_comp, p->out_done[s]);
  if (!ok) return KV4_ERR_LAUNCH;
  // lse (a few KB) is written by the decode straight into the host buffer
  // when that is device-addressable page-locked memory, instead of one more
  // small copy; out goes back by one copy
  float* lse_mapped = static_cast<float*>(const_cast<void*>(mapped_host(lse_host)));
  if ((reinterpret_cast<uintptr_t>(lse_mapped) & 3u) != 0) lse_mapped = nullptr;
  const kv4_status r = kv4_quantize_write_and_decode(
      a.latent, KV4_LATENT, a.rope, KV4_ROPE, a.slots, n_new, pool_dev, num_slots, a.q,
      page_table_dev, pt_stride, page_size, a.topk, p->K, a.lens, p->B, p->Sq, p->H, sm_scale,
      a.out, lse_mapped ? lse_mapped : a.lse, p->ws, p->ws_bytes, p->force_splits, dev_err,
      reinterpret_cast<kv4_stream_t>(p->s_comp));
  if (r != KV4_OK) return r;
  record(p->comp_done[s], p->s_comp);
  // results back to the host
  wait_on(p->s_out, p->comp_done[s]);
  d2h(out_host, a.out, p->out_bytes);
  if (!lse_mapped) d2h(lse_host, a.lse, p->lse_bytes);
  record(p->out_done[s], p->s_out);
  if (!ok) return KV4_ERR_LAUNCH;
  p->used[s] = true;
  ++p->steps;
  return KV4_OK;
}

kv4_status kv4_host_pipe_destroy(kv4_host_pipe* p) {
  if (!p) return KV4_ERR_INVALID_ARG;
  destroy_events(p);
  delete p;
  return KV4_OK;
}

kv4_status kv4_debug_gather_dequant(const uint8_t* pool_dev, int64_t num_slots,
                                    const int32_t* page_table_dev, int64_t pt_stride,
                                    int page_size, const int32_t* topk_idx_dev, int K,
                                    const int32_t* seq_lens_dev, int B, int Sq, void* rows_dev,
                                    int32_t* dev_err, kv4_stream_t stream) {
  return gather_impl(pool_dev, num_slots, page_table_dev, pt_stride, page_size, topk_idx_dev, K,
                     seq_lens_dev, B, Sq, rows_dev, dev_err, stream, true);
}

kv4_status kv4_quantize_write_mse(const void* latent_dev, int64_t latent_row_stride,
                                  const void* rope_dev, int64_t rope_row_stride,
                                  const int64_t* slot_mapping_dev, int64_t n_tokens,
                                  uint8_t* pool_dev, int64_t num_slots, int32_t* dev_err,
                                  kv4_stream_t stream) {
  return quantize_impl(latent_dev, latent_row_stride, rope_dev, rope_row_stride,
                       slot_mapping_dev, n_tokens, pool_dev, num_slots, dev_err, stream, true,
                       true);
}

kv4_status kv4_sparse_mla_decode_partial(const void* q_dev, const uint8_t* pool_dev,
                                         int64_t num_slots, const int32_t* page_table_dev,
                                         int64_t pt_stride, int page_size,
                                         const int32_t* topk_idx_dev, int K,
                                         const int32_t* seq_lens_dev, int B, int Sq, int H,
                                         float sm_scale, float* o_dev, float* lse_dev,
                                         void* workspace_dev, size_t workspace_bytes,
                                         int force_splits, int32_t* dev_err,
                                         kv4_stream_t stream) {
  return decode_impl(q_dev, pool_dev, num_slots, page_table_dev, pt_stride, page_size,
                     topk_idx_dev, K, seq_lens_dev, B, Sq, H, sm_scale, o_dev, lse_dev,
                     workspace_dev, workspace_bytes, force_splits, dev_err, stream,
                     kv4::kFmtNvfp4, true);
}

kv4_status kv4_sparse_mla_decode_partial_counted(
    const void* q_dev, const uint8_t* pool_dev, int64_t num_slots, const int32_t* page_table_dev,
    int64_t pt_stride, int page_size, const int32_t* topk_idx_dev, int K,
    const int32_t* k_count_dev, const int32_t* seq_lens_dev, int B, int Sq, int H, float sm_scale,
    float* o_dev, float* lse_dev, void* workspace_dev, size_t workspace_bytes, int force_splits,
    int32_t* dev_err, kv4_stream_t stream) {
  if (B > 0 && (k_count_dev == nullptr || (reinterpret_cast<uintptr_t>(k_count_dev) & 3u) != 0))
    return KV4_ERR_INVALID_ARG;
  return decode_impl(q_dev, pool_dev, num_slots, page_table_dev, pt_stride, page_size,
                     topk_idx_dev, K, seq_lens_dev, B, Sq, H, sm_scale, o_dev, lse_dev,
                     workspace_dev, workspace_bytes, force_splits, dev_err, stream,
                     kv4::kFmtNvfp4, true, false, true, k_count_dev);
}

kv4_status kv4_dcp_compact_topk(const int32_t* topk_idx_dev, const int32_t* page_table_dev,
                                int64_t pt_stride, const int32_t* seq_lens_dev, int B, int Sq,
                                int K, int world, int rank, int32_t* topk_out_dev,
                                int32_t* count_out_dev, kv4_stream_t stream) {
  if (B < 0 || Sq < 1 || K < 0 || pt_stride < 1 || world < 1 || rank < 0 || rank >= world)
    return KV4_ERR_INVALID_ARG;
  if (B == 0) return KV4_OK;
  if ((K > 0 && (!topk_idx_dev || !topk_out_dev)) || !page_table_dev || !seq_lens_dev ||
      !count_out_dev || (K > 0 && topk_idx_dev == topk_out_dev))
    return KV4_ERR_INVALID_ARG;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  return kv4::launch_dcp_compact_topk(topk_idx_dev, page_table_dev, pt_stride, seq_lens_dev, B,
                                      Sq, K, world, rank, topk_out_dev, count_out_dev,
                                      reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KV4_OK
             : KV4_ERR_LAUNCH;
}

kv4_status kv4_dcp_mask_topk(const int32_t* topk_idx_dev, const int32_t* page_table_dev,
                             int64_t pt_stride, const int32_t* seq_lens_dev, int B, int Sq,
                             int K, int world, int rank, int32_t* topk_out_dev,
                             kv4_stream_t stream) {
  if (B < 0 || Sq < 1 || K < 0 || pt_stride < 1 || world < 1 || rank < 0 || rank >= world)
    return KV4_ERR_INVALID_ARG;
  if (B == 0 || K == 0) return KV4_OK;
  if (!topk_idx_dev || !page_table_dev || !seq_lens_dev || !topk_out_dev)
    return KV4_ERR_INVALID_ARG;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  return kv4::launch_dcp_mask_topk(topk_idx_dev, page_table_dev, pt_stride, seq_lens_dev, B, Sq,
                                   K, world, rank, topk_out_dev,
                                   reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KV4_OK
             : KV4_ERR_LAUNCH;
}

kv4_status kv4_dcp_local_page_table(const int32_t* page_table_dev, int64_t pt_stride, int B,
                                   int world, int rank, int32_t* pt_local_dev,
                                   kv4_stream_t stream) {
  if (B < 0 || pt_stride < 1 || world < 1 || rank < 0 || rank >= world) return KV4_ERR_INVALID_ARG;
  if (B == 0) return KV4_OK;
  if (!page_table_dev || !pt_local_dev) return KV4_ERR_INVALID_ARG;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  return kv4::launch_dcp_local_page_table(page_table_dev, static_cast<int64_t>(B) * pt_stride,
                                          world, rank, pt_local_dev,
                                          reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KV4_OK
             : KV4_ERR_LAUNCH;
}

kv4_status kv4_dcp_local_slots(const int64_t* slot_mapping_dev, int64_t n_tokens, int world,
                               int rank, int64_t* slots_out_dev, kv4_stream_t stream) {
  if (n_tokens < 0 || world < 1 || rank < 0 || rank >= world) return KV4_ERR_INVALID_ARG;
  if (n_tokens == 0) return KV4_OK;
  if (!slot_mapping_dev || !slots_out_dev) return KV4_ERR_INVALID_ARG;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  return kv4::launch_dcp_local_slots(slot_mapping_dev, n_tokens, world, rank, slots_out_dev,
                                     reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KV4_OK
             : KV4_ERR_LAUNCH;
}

kv4_status kv4_merge_partials(const float* o_parts_dev, const float* lse_parts_dev, int R,
                              int64_t n_rows, void* out_dev, float* lse_dev,
                              kv4_stream_t stream) {
  if (R < 1 || n_rows < 0) return KV4_ERR_INVALID_ARG;
  if (n_rows == 0) return KV4_OK;
  if (!o_parts_dev || !lse_parts_dev || !out_dev || !lse_dev) return KV4_ERR_INVALID_ARG;
  if (!aligned16(o_parts_dev) || !aligned16(out_dev)) return KV4_ERR_INVALID_ARG;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  return kv4::launch_merge_partials(o_parts_dev, lse_parts_dev, R, n_rows, out_dev, lse_dev,
                                    reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KV4_OK
             : KV4_ERR_LAUNCH;
}

kv4_status kv4_quantize_write_fp8(const void* latent_dev, int64_t latent_row_stride,
                                  const void* rope_dev, int64_t rope_row_stride,
                                  const int64_t* slot_mapping_dev, int64_t n_tokens,
                                  uint8_t* pool_dev, int64_t num_slots, int32_t* dev_err,
                                  kv4_stream_t stream) {
  if (n_tokens < 0 || num_slots < 0) return KV4_ERR_INVALID_ARG;
  if (n_tokens == 0) return KV4_OK;
  if (!latent_dev || !rope_dev || !slot_mapping_dev || !pool_dev) return KV4_ERR_INVALID_ARG;
  if (latent_row_stride < KV4_LATENT || latent_row_stride % 8 != 0 ||
      rope_row_stride < KV4_ROPE || rope_row_stride % 8 != 0)
    return KV4_ERR_INVALID_ARG;
  if (!aligned16(latent_dev) || !aligned16(rope_dev) || !aligned16(pool_dev) ||
      (reinterpret_cast<uintptr_t>(slot_mapping_dev) & 7u) != 0)
    return KV4_ERR_INVALID_ARG;
  if (num_slots > INT64_MAX / KV4_ROW_BYTES_FP8) return KV4_ERR_INVALID_ARG;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  kv4::QuantizeArgs a{latent_dev, latent_row_stride, rope_dev,     rope_row_stride, slot_mapping_dev,
                      n_tokens,   pool_dev,          num_slots,    KV4_ROW_BYTES_FP8, dev_err,
                      0,          1};
  return kv4::launch_quantize_write(a, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KV4_OK
             : KV4_ERR_LAUNCH;
}

kv4_status kv4_decode_plan_fp8(int B, int Sq, int H, int K, int force_splits, int* splits,
                               size_t* workspace_bytes) {
  return plan_impl(B, Sq, H, K, force_splits, splits, workspace_bytes, kv4::kFmtFp8);
}

kv4_status kv4_sparse_mla_decode_fp8(const void* q_dev, const uint8_t* pool_dev,
                                     int64_t num_slots, const int32_t* page_table_dev,
                                     int64_t pt_stride, int page_size,
                                     const int32_t* topk_idx_dev, int K,
                                     const int32_t* seq_lens_dev, int B, int Sq, int H,
                                     float sm_scale, void* out_dev, float* lse_dev,
                                     void* workspace_dev, size_t workspace_bytes,
                                     int force_splits, int32_t* dev_err, kv4_stream_t stream) {
  return decode_impl(q_dev, pool_dev, num_slots, page_table_dev, pt_stride, page_size,
                     topk_idx_dev, K, seq_lens_dev, B, Sq, H, sm_scale, out_dev, lse_dev,
                     workspace_dev, workspace_bytes, force_splits, dev_err, stream,
                     kv4::kFmtFp8);
}

kv4_status kv4_fp8_scratch(const uint8_t* pool_dev, int64_t num_slots,
                           const int32_t* page_table_dev, int64_t pt_stride, int page_size,
                           const int32_t* topk_idx_dev, int K, const int32_t* seq_lens_dev,
                           int B, int Sq, uint8_t* scratch_dev, int32_t* dev_err,
                           kv4_stream_t stream) {
  if (B < 0 || Sq < 1 || K < 0) return KV4_ERR_INVALID_ARG;
  if (page_size != KV4_PAGE) return KV4_ERR_UNSUPPORTED;
  if (B == 0 || K == 0) return KV4_OK;
  if (!pool_dev || !page_table_dev || !topk_idx_dev || !seq_lens_dev || !scratch_dev)
    return KV4_ERR_INVALID_ARG;
  if (num_slots < 0 || num_slots > INT32_MAX || pt_stride < 1 || pt_stride > INT32_MAX)
    return KV4_ERR_INVALID_ARG;
  if (!aligned16(pool_dev) || !aligned16(scratch_dev)) return KV4_ERR_INVALID_ARG;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  kv4::GatherArgs a{pool_dev, num_slots,    page_table_dev, pt_stride, topk_idx_dev, K,
                    seq_lens_dev, B,         Sq,             scratch_dev, 1,          dev_err};
  return kv4::launch_fp8_scratch(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KV4_OK
             : KV4_ERR_LAUNCH;
}

kv4_status kv4_fp8_scratch_index(const int32_t* topk_idx_dev, int K, const int32_t* seq_lens_dev,
                                 int B, int Sq, int32_t* pt_out_dev, int32_t* topk_out_dev,
                                 int32_t* lens_out_dev, kv4_stream_t stream) {
  if (B < 0 || Sq < 1 || K < 0) return KV4_ERR_INVALID_ARG;
  if (K % KV4_PAGE != 0) return KV4_ERR_UNSUPPORTED;
  if (B == 0 || K == 0) return KV4_OK;
  if (!topk_idx_dev || !seq_lens_dev || !pt_out_dev || !topk_out_dev || !lens_out_dev)
    return KV4_ERR_INVALID_ARG;
  int sms = 0;
  const kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  return kv4::launch_fp8_scratch_index(topk_idx_dev, seq_lens_dev, B, Sq, K, pt_out_dev,
                                       topk_out_dev, lens_out_dev,
                                       reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KV4_OK
             : KV4_ERR_LAUNCH;
}

kv4_status kv4_quantize_write_latent(const void* latent_dev, int64_t latent_row_stride,
                                     const int64_t* slot_mapping_dev, int64_t n_tokens,
                                     uint8_t* pool_dev, int64_t num_slots, int32_t* dev_err,
                                     kv4_stream_t stream) {
  return quantize_impl(latent_dev, latent_row_stride, nullptr, 0, slot_mapping_dev, n_tokens,
                       pool_dev, num_slots, dev_err, stream, false);
}

kv4_status kv4_decode_plan_latent(int B, int Sq, int H, int K, int force_splits, int* splits,
                                  size_t* workspace_bytes) {
  return plan_impl(B, Sq, H, K, force_splits, splits, workspace_bytes, kv4::kFmtNvfp4Latent);
}

kv4_status kv4_sparse_mla_decode_latent(const void* q_dev, const uint8_t* pool_dev,
                                        int64_t num_slots, const int32_t* page_table_dev,
                                        int64_t pt_stride, int page_size,
                                        const int32_t* topk_idx_dev, int K,
                                        const int32_t* seq_lens_dev, int B, int Sq, int H,
                                        float sm_scale, void* out_dev, float* lse_dev,
                                        void* workspace_dev, size_t workspace_bytes,
                                        int force_splits, int32_t* dev_err,
                                        kv4_stream_t stream) {
  return decode_impl(q_dev, pool_dev, num_slots, page_table_dev, pt_stride, page_size,
                     topk_idx_dev, K, seq_lens_dev, B, Sq, H, sm_scale, out_dev, lse_dev,
                     workspace_dev, workspace_bytes, force_splits, dev_err, stream,
                     kv4::kFmtNvfp4Latent);
}

kv4_status kv4_debug_gather_dequant_latent(const uint8_t* pool_dev, int64_t num_slots,
                                           const int32_t* page_table_dev, int64_t pt_stride,
                                           int page_size, const int32_t* topk_idx_dev, int K,
                                           const int32_t* seq_lens_dev, int B, int Sq,
                                           void* rows_dev, int32_t* dev_err,
                                           kv4_stream_t stream) {
  return gather_impl(pool_dev, num_slots, page_table_dev, pt_stride, page_size, topk_idx_dev, K,
                     seq_lens_dev, B, Sq, rows_dev, dev_err, stream, false);
}

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// decode -- for example a plugin that its host engine hands only input and
// output buffers, while the engine owns and budgets every byte of device
// memory, or code that must not call cudaMalloc because it synchronizes the
// device.  For them the split-K partials go to a buffer that is part of the
// library itself: a file-scope device array, created when the library's
// module is loaded on a device and held by that device until the process
// exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = size_t(24) << 20;   // 24 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device.  In host code
// the symbol's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress with that device current.  It is looked up on every
// call (a host-side query that allocates nothing), so a context that was
// torn down and recreated -- and the array with it -- is always addressed
// correctly.
kv4_status static_scratch(void** ptr) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
    return KV4_ERR_LAUNCH;
  *ptr = p;
  return KV4_OK;
}

}  // namespace

kv4_status kv4_sparse_mla_decode_noalloc(const void* q_dev, const uint8_t* pool_dev,
                                         int64_t num_slots, const int32_t* page_table_dev,
                                         int64_t pt_stride, int page_size,
                                         const int32_t* topk_idx_dev, int K,
                                         const int32_t* seq_lens_dev, int B, int Sq, int H,
                                         float sm_scale, void* out_dev, float* lse_dev,
                                         int force_splits, int32_t* dev_err,
                                         kv4_stream_t stream) {
  // every argument is checked first, so that a bad pointer is reported as
  // such and not as a shape beyond the scratch array
  const kv4_status args = check_decode_args(q_dev, pool_dev, num_slots, page_table_dev, pt_stride,
                                            page_size, topk_idx_dev, K, seq_lens_dev, B, Sq, H,
                                            out_dev, lse_dev);
  if (args != KV4_OK || B == 0) return args;
  int sms = 0;
  kv4_status st = device_info(&sms);
  if (st != KV4_OK) return st;
  const Plan p = make_plan(B, Sq, H, K, force_splits, sms, kv4::kFmtNvfp4);
  if (p.ws_bytes > kStaticScratchBytes) return KV4_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  st = static_scratch(&scratch);
  if (st != KV4_OK) return st;
  return kv4_sparse_mla_decode(q_dev, pool_dev, num_slots, page_table_dev, pt_stride, page_size,
                               topk_idx_dev, K, seq_lens_dev, B, Sq, H, sm_scale, out_dev, lse_dev,
                               scratch, kStaticScratchBytes, force_splits, dev_err, stream);
}

size_t kv4_noalloc_scratch_bytes(void) { return kStaticScratchBytes; }

kv4_status kv4_set_wait_limit(int64_t timeout_ns, int fault_site) {
  if (timeout_ns < 0 || fault_site < 0 || fault_site > 1) return KV4_ERR_INVALID_ARG;
  g_timeout_ns.store(timeout_ns > 0 ? timeout_ns : 1000000000);
  g_fault_site.store(fault_site);
  return KV4_OK;
}

kv4_status kv4_set_timing_event(void* cuda_event) {
  g_timing_event.store(cuda_event);
  return KV4_OK;
}

const char* kv4_status_str(kv4_status status) {
  switch (status) {
    case KV4_OK: return "ok";
    case KV4_ERR_INVALID_ARG: return "invalid argument";
    case KV4_ERR_UNSUPPORTED: return "unsupported shape or page size";
    case KV4_ERR_ARCH: return "current device is not compute capability 10.3";
    case KV4_ERR_LAUNCH: return "kernel launch failed";
    case KV4_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case KV4_ERR_SCRATCH_LIMIT:
      return "split-K partials exceed the library's static scratch (see "
             "kv4_noalloc_scratch_bytes); pass a workspace or force fewer splits";
  }
  return "unknown status";
}

int kv4_version(void) { return 1; }

}  // extern "C"
