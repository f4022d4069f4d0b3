/*
 * kv4mla.h -- C ABI of libkv4mla.so: NVFP4 latent-KV cache write and
 * sparse MLA (DSA) decode on GB300 (sm_103a).
 *
 * The method (numinousmuses "inference-optimizations" README):
 *  - "4-bit KV cache", GLM-5.3 bullet: each cached token is one 352-byte
 *    NVFP4 row -- E2M1 values with one E4M3 scale per 16 values -- that
 *    replaces the 576-byte FP8 row used by DSA sparse attention.  This
 *    library fixes the byte order of the row:
 *        bytes [0,256)   512 latent E2M1 codes, byte j = code(2j) | code(2j+1)<<4
 *        bytes [256,288) 32 E4M3 scales, scale i covers latent 16i..16i+15
 *        bytes [288,352) 64 rope values as E4M3 (no scale)
 *    A row lives at pool + slot*352; slot = page*64 + offset (64-token pages,
 *    the page size of the sgl-amd-mono sparse-attention page table).
 *  - "4-bit KV cache", kv4mla bullet: the decode reads the 4-bit rows and
 *    dequantizes them in shared memory (no FP8 scratch copy in HBM).
 *  - "Attention kernels", split-K sparse decode bullet, and "Parallelism and
 *    disaggregation", (o, lse) merge bullet: when the batch is too small to
 *    fill the GPU the selected set is split and the partial (o, lse) are
 *    merged by log-sum-exp.
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev are DEVICE pointers of the current CUDA device;
 *    the caller allocates and owns every buffer (including the workspace).
 *    The library keeps no pointer after a call returns (apart from a host
 *    pipe, which keeps its staging memory and streams until destroyed),
 *    never allocates device memory and never synchronizes.  Pointers named
 *    *_host are host pointers.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously; outputs are valid once the stream has
 *    reached that point.
 *  - Host-detectable argument errors return a nonzero kv4_status and launch
 *    nothing.  Errors only the device can see (an index or page out of range,
 *    a bounded wait that gave up) OR a KV4_DEV_* flag into *dev_err (when
 *    non-NULL); the offending row is skipped / the offending key is masked.
 *    Read *dev_err after synchronizing.  Nothing traps.
 *  - bf16 tensors are raw IEEE bfloat16; all sizes are in elements unless
 *    named *_bytes.
 */
#ifndef KV4MLA_H
#define KV4MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kv4_stream_t;   /* same handle as cudaStream_t */

typedef enum {
  KV4_OK = 0,
  KV4_ERR_INVALID_ARG = 1,   /* null pointer, bad size, stride or alignment   */
  KV4_ERR_UNSUPPORTED = 2,   /* H or page size outside the supported set      */
  KV4_ERR_ARCH = 3,          /* current device is not compute capability 10.3 */
  KV4_ERR_LAUNCH = 4,        /* a kernel launch failed (cudaGetLastError)     */
  KV4_ERR_WORKSPACE = 5,     /* workspace missing or smaller than required    */
  KV4_ERR_SCRATCH_LIMIT = 6  /* kv4_sparse_mla_decode_noalloc: the split-K
                                partials would not fit the static scratch     */
} kv4_status;

/* Flags OR-ed into *dev_err by the kernels. */
enum {
  KV4_DEV_BAD_SLOT = 1,      /* write: slot >= num_slots; that row skipped     */
  KV4_DEV_BAD_PAGE = 2,      /* decode: page index >= pt_stride, negative page
                                entry or slot >= num_slots; that key masked    */
  KV4_DEV_TIMEOUT = 4        /* a bounded on-chip wait gave up; the outputs of
                                that thread block are not valid               */
};

enum {
  KV4_ROW_BYTES = 352, KV4_LATENT = 512, KV4_ROPE = 64, KV4_QK_DIM = 576,
  KV4_BLOCK = 16, KV4_PAGE = 64, KV4_TILE_KEYS = 128,
  KV4_ROW_BYTES_LATENT = 288,  /* latent-only row (the *_latent entry points) */
  KV4_ROW_BYTES_FP8 = 576      /* FP8 comparison row (the *_fp8 entry points)  */
};

/* ---------------------------------------------------------------------------
 * kv4_quantize_write -- quantize N new tokens into their cache rows.
 * Source: README "4-bit KV cache" (the quantized write of the NVFP4 row).
 *   latent_dev        bf16 [N, latent_row_stride]; first 512 used
 *   rope_dev          bf16 [N, rope_row_stride];   first 64 used
 *                     (both: base 16-byte aligned, stride a multiple of 8)
 *   slot_mapping_dev  int64 [N]; slot < 0 skips the token
 *   pool_dev          uint8 [num_slots, 352], base 16-byte aligned
 * Per 16-element block: scale byte = E4M3(amax/6) (IEEE fp32 division, round
 * half to even, saturate at 448); s = decoded scale; code = E2M1(x/s) (fp32
 * division, round half to even, saturate at 6, sign of x kept); s == 0 gives
 * all-zero codes.  Rope: E4M3(x).  Bit-identical to the CPU oracle.
 * ------------------------------------------------------------------------- */
kv4_status kv4_quantize_write(const void* latent_dev, int64_t latent_row_stride,
                              const void* rope_dev, int64_t rope_row_stride,
                              const int64_t* slot_mapping_dev, int64_t n_tokens,
                              uint8_t* pool_dev, int64_t num_slots,
                              int32_t* dev_err, kv4_stream_t stream);

/* ---------------------------------------------------------------------------
 * kv4_quantize_write_mse -- kv4_quantize_write with searched block scales.
 * Source: README "4-bit KV cache", DeepSeek V4 Pro bullet ("an MSE-searched
 * scale"); the page gives no rule, this is the project's reading.  Same
 * arguments, row layout and errors as kv4_quantize_write.  Per block: the
 * candidate scale bytes are c0-8 .. c0+1 (clipped to 0..126) around
 * c0 = E4M3(amax/6); each candidate s gives codes E2M1(x/s) (fp32 division,
 * round half to even; s == 0 gives zero codes) and the error
 * sum_i (x_i - dec(code_i) * s)^2 in IEEE fp32, element order, every
 * operation rounded to nearest; the smallest error wins, the lowest scale
 * byte on ties.  The rows decode with kv4_sparse_mla_decode unchanged.
 * Bit-identical to the CPU oracle.
 * ------------------------------------------------------------------------- */
kv4_status kv4_quantize_write_mse(const void* latent_dev, int64_t latent_row_stride,
                                  const void* rope_dev, int64_t rope_row_stride,
                                  const int64_t* slot_mapping_dev, int64_t n_tokens,
                                  uint8_t* pool_dev, int64_t num_slots,
                                  int32_t* dev_err, kv4_stream_t stream);

/* ---------------------------------------------------------------------------
 * kv4_decode_plan -- number of split-K partitions and workspace bytes that
 * kv4_sparse_mla_decode will use for this shape on the current device.
 * force_splits > 0 requests that many partitions (clamped to the number of
 * 128-key tiles); 0 lets the planner fill the SMs.
 * ------------------------------------------------------------------------- */
kv4_status kv4_decode_plan(int B, int Sq, int H, int K, int force_splits,
                           int* splits, size_t* workspace_bytes);

/* ---------------------------------------------------------------------------
 * kv4_sparse_mla_decode -- sparse MLA decode over the NVFP4 pool.
 * Source: README "4-bit KV cache" (kv4mla) and "Attention kernels"
 * (split-K); (o, lse) merge from "Parallelism and disaggregation".
 *   q_dev          bf16 [B, Sq, H, 576] contiguous (512 latent + 64 rope),
 *                  16-byte aligned
 *   pool_dev       uint8 [num_slots, 352] (num_slots < 2^31), 16-byte aligned
 *   page_table_dev int32 [B, pt_stride]: physical page of each 64-token
 *                  logical page; page_size must be 64
 *   topk_idx_dev   int32 [B, Sq, K]: logical token positions; a position
 *                  outside [0, L_eff) is masked (-1 = padding), with
 *                  L_eff = seq_lens[b] - (Sq-1-s) (causal within the draft)
 *   seq_lens_dev   int32 [B]: tokens of request b, including its Sq drafts
 *   H              16, 32, 64, or a multiple of 64 up to 256
 *   sm_scale       softmax scale applied to q.k
 *   out_dev        bf16 [B, Sq, H, 512]: softmax-weighted sum of the latent
 *                  part of the selected rows (0 if no key is valid),
 *                  16-byte aligned
 *   lse_dev        fp32 [B, Sq, H]: natural-log log-sum-exp of the scaled
 *                  scores (-inf if no key is valid)
 *   workspace_dev  device scratch of at least the bytes kv4_decode_plan
 *                  returns (may be NULL when that is 0), 16-byte aligned
 * Duplicated positions count once per occurrence.  Scores use all 576 dims;
 * the weighted sum uses the 512 latent dims of the same rows.  Arithmetic:
 * K/V rows are dequantized exactly to f16, q is converted to f16 after an
 * exact per-head power-of-two scaling, QK^T and PV accumulate in fp32 on the
 * tensor cores, softmax weights enter PV as f16.
 * ------------------------------------------------------------------------- */
kv4_status kv4_sparse_mla_decode(const void* q_dev, const uint8_t* pool_dev,
                                 int64_t num_slots, const int32_t* page_table_dev,
                                 int64_t pt_stride, int page_size,
                                 const int32_t* topk_idx_dev, int K,
                                 const int32_t* seq_lens_dev, int B, int Sq, int H,
                                 float sm_scale, void* out_dev, float* lse_dev,
                                 void* workspace_dev, size_t workspace_bytes,
                                 int force_splits, int32_t* dev_err,
                                 kv4_stream_t stream);

/* ---------------------------------------------------------------------------
 * kv4_quantize_write_and_decode -- one decode step: kv4_quantize_write of the
 * step's new tokens, then kv4_sparse_mla_decode over the pool, on `stream`.
 * Source: the write (README "4-bit KV cache", kv4mla bullet) followed by the
 * decode it feeds; the two are the step's hot path.
 * Arguments: those of kv4_quantize_write (latent_dev .. num_slots) followed
 * by those of kv4_sparse_mla_decode (q_dev .. stream), with the same
 * meanings, layouts and ownership; pool_dev and num_slots are shared.
 * Results are bit-identical to the two calls made one after the other.  The
 * difference: the decode kernel starts while the write is still running and
 * reads q, the page table, the top-k list and seq_lens at once; only its
 * reads of pool rows wait for the write.  So q_dev, page_table_dev,
 * topk_idx_dev and seq_lens_dev must not overlap the pool or the write's
 * inputs (they are otherwise as in kv4_sparse_mla_decode: ready in stream
 * order).  Every argument of both parts is checked before anything is
 * launched; errors are those of the two calls.
 * ------------------------------------------------------------------------- */
kv4_status kv4_quantize_write_and_decode(
    const void* latent_dev, int64_t latent_row_stride, const void* rope_dev,
    int64_t rope_row_stride, const int64_t* slot_mapping_dev, int64_t n_tokens,
    uint8_t* pool_dev, int64_t num_slots, const void* q_dev, const int32_t* page_table_dev,
    int64_t pt_stride, int page_size, const int32_t* topk_idx_dev, int K,
    const int32_t* seq_lens_dev, int B, int Sq, int H, float sm_scale, void* out_dev,
    float* lse_dev, void* workspace_dev, size_t workspace_bytes, int force_splits,
    int32_t* dev_err, kv4_stream_t stream);

/* ---------------------------------------------------------------------------
 * Host-buffer steps (kv4_host_pipe_*) -- the step of
 * kv4_quantize_write_and_decode fed from HOST memory, as a serving loop runs
 * it: each step's inputs (the new tokens and their slots, q, the top-k list,
 * seq_lens) are copied from host buffers into device staging, the write and
 * the decode run, and out / lse are copied back into host buffers.  The
 * pages have no counterpart: it is the same hot path (README "4-bit KV
 * cache", kv4mla bullet: the write, then the decode it feeds) with its
 * host<->device copies.
 *
 * A pipe keeps two steps in flight.  Step i's inputs are copied on copy_in
 * while step i-1 computes on `compute`, and step i-1's results are copied
 * back on copy_out while step i computes.  Steps alternate between two
 * staging areas; CUDA events order the three streams (a step's copies into
 * an area wait until the step two before it has finished computing from it,
 * and its compute waits until that step's results have left it).
 *
 *   kv4_host_pipe_bytes(B, Sq, H, K, max_new, force_splits, &bytes)
 *       device staging bytes of a pipe of this shape: two areas (q, top-k,
 *       seq_lens, new tokens and slots, out, lse) and the split-K workspace.
 *   kv4_host_pipe_create(B, Sq, H, K, max_new, force_splits, staging_dev,
 *                        staging_bytes, copy_in, compute, copy_out, &pipe)
 *       B, Sq, H, K: the decode shape of every step (as in
 *       kv4_sparse_mla_decode); max_new: the most new tokens one step
 *       writes; force_splits: as in kv4_decode_plan; staging_dev:
 *       caller-owned device memory of at least kv4_host_pipe_bytes bytes,
 *       256-byte aligned, which nothing else uses while the pipe lives;
 *       copy_in, compute, copy_out: the caller's streams (one stream for all
 *       three serializes the steps).  Creates six CUDA events and a small
 *       host object; allocates no device memory.
 *   kv4_host_pipe_step(pipe, latent_host, rope_host, slots_host, n_new,
 *                      pool_dev, num_slots, page_table_dev, pt_stride,
 *                      page_size, q_host, topk_host, seq_lens_host, sm_scale,
 *                      out_host, lse_host, dev_err)
 *       enqueues one step and returns.  Host buffers (contiguous):
 *       latent_host bf16 [n_new, 512], rope_host bf16 [n_new, 64],
 *       slots_host int64 [n_new] (0 <= n_new <= max_new), q_host bf16
 *       [B, Sq, H, 576], topk_host int32 [B, Sq, K], seq_lens_host int32 [B],
 *       out_host bf16 [B, Sq, H, 512], lse_host fp32 [B, Sq, H].  pool_dev
 *       and page_table_dev are device buffers, as in the device calls, and
 *       dev_err is a device word (or NULL).  Results equal those of
 *       kv4_quantize_write_and_decode on the same values bit for bit.
 *       Host buffers should be page-locked (cudaHostAlloc /
 *       cudaHostRegister): with pageable memory the copies still happen but
 *       block the calling thread.  q is copied on copy_in; the other inputs
 *       (the top-k list, seq_lens, the new tokens and their slots) are read
 *       there by one kernel through their device addresses when all of them
 *       are page-locked, and copied one by one otherwise.  out is copied back
 *       on copy_out; lse is written by the decode straight into lse_host when
 *       that is page-locked, and copied otherwise.  A step's host inputs must stay unchanged,
 *       and its host outputs unread, until copy_out has passed the step
 *       (synchronize copy_out, or wait on an event recorded on it after the
 *       call).  Argument errors return nonzero before anything is enqueued;
 *       KV4_ERR_LAUNCH (a failed copy or launch) leaves the pipe unusable:
 *       destroy it.
 *   kv4_host_pipe_destroy(pipe)
 *       releases the events and the host object; work already enqueued
 *       completes normally.  The staging memory stays the caller's.
 * ------------------------------------------------------------------------- */
typedef struct kv4_host_pipe kv4_host_pipe;
kv4_status kv4_host_pipe_bytes(int B, int Sq, int H, int K, int64_t max_new, int force_splits,
                               size_t* staging_bytes);
kv4_status kv4_host_pipe_create(int B, int Sq, int H, int K, int64_t max_new, int force_splits,
                                void* staging_dev, size_t staging_bytes, kv4_stream_t copy_in,
                                kv4_stream_t compute, kv4_stream_t copy_out,
                                kv4_host_pipe** pipe);
kv4_status kv4_host_pipe_step(kv4_host_pipe* pipe, const void* latent_host, const void* rope_host,
                              const int64_t* slots_host, int64_t n_new, uint8_t* pool_dev,
                              int64_t num_slots, const int32_t* page_table_dev, int64_t pt_stride,
                              int page_size, const void* q_host, const int32_t* topk_host,
                              const int32_t* seq_lens_host, float sm_scale, void* out_host,
                              float* lse_host, int32_t* dev_err);
kv4_status kv4_host_pipe_destroy(kv4_host_pipe* pipe);

/* ---------------------------------------------------------------------------
 * kv4_debug_gather_dequant -- the decode's own index resolution and
 * dequantization, written out: rows_dev f16 [B, Sq, K, 576] receives the
 * dequantized selected rows, i.e. the tensor-core operand values (every
 * E2M1 x E4M3 product and E4M3 value is exact in f16); a masked key gives an
 * all-zero row.  Exists so that the gather indexing can be checked bit for
 * bit; same argument meaning as kv4_sparse_mla_decode.
 * ------------------------------------------------------------------------- */
kv4_status kv4_debug_gather_dequant(const uint8_t* pool_dev, int64_t num_slots,
                                    const int32_t* page_table_dev, int64_t pt_stride,
                                    int page_size, const int32_t* topk_idx_dev, int K,
                                    const int32_t* seq_lens_dev, int B, int Sq,
                                    void* rows_dev, int32_t* dev_err,
                                    kv4_stream_t stream);

/* ---------------------------------------------------------------------------
 * Latent-only rows (288 bytes).
 * Source: README "4-bit KV cache", the GLM-5.3-Flash bullet (a 288-byte
 * rope-free row).  A row is the first 288 bytes of the 352-byte row above --
 * bytes [0,256) E2M1 codes, [256,288) the 32 E4M3 scales -- for models whose
 * cached keys carry no rope part.  QK^T then runs over the 512 latent
 * columns only, and PV over the same 512.  Arguments, layouts, ownership
 * and errors are those of the 352-byte calls, except:
 *   kv4_quantize_write_latent     no rope input; pool uint8 [num_slots, 288]
 *   kv4_decode_plan_latent        the plan of kv4_sparse_mla_decode_latent
 *   kv4_sparse_mla_decode_latent  q bf16 [B, Sq, H, 512]; pool [num_slots, 288]
 *   kv4_debug_gather_dequant_latent  rows f16 [B, Sq, K, 512]
 * Per byte of pool, 288-byte rows hold 2x the tokens of 576-byte FP8 rows
 * and 1.22x those of 352-byte rows.
 * ------------------------------------------------------------------------- */
kv4_status kv4_quantize_write_latent(const void* latent_dev, int64_t latent_row_stride,
                                     const int64_t* slot_mapping_dev, int64_t n_tokens,
                                     uint8_t* pool_dev, int64_t num_slots, int32_t* dev_err,
                                     kv4_stream_t stream);
kv4_status kv4_decode_plan_latent(int B, int Sq, int H, int K, int force_splits,
                                  int* splits, size_t* workspace_bytes);
kv4_status kv4_sparse_mla_decode_latent(const void* q_dev, const uint8_t* pool_dev,
                                        int64_t num_slots, const int32_t* page_table_dev,
                                        int64_t pt_stride, int page_size,
                                        const int32_t* topk_idx_dev, int K,
                                        const int32_t* seq_lens_dev, int B, int Sq, int H,
                                        float sm_scale, void* out_dev, float* lse_dev,
                                        void* workspace_dev, size_t workspace_bytes,
                                        int force_splits, int32_t* dev_err,
                                        kv4_stream_t stream);
kv4_status kv4_debug_gather_dequant_latent(const uint8_t* pool_dev, int64_t num_slots,
                                           const int32_t* page_table_dev, int64_t pt_stride,
                                           int page_size, const int32_t* topk_idx_dev, int K,
                                           const int32_t* seq_lens_dev, int B, int Sq,
                                           void* rows_dev, int32_t* dev_err,
                                           kv4_stream_t stream);

/* ---------------------------------------------------------------------------
 * FP8 comparison paths.
 * Source: README "4-bit KV cache", kv4mla bullet (the NVFP4 decode against
 * the 576-byte FP8 row it replaces, and against an "FP8 scratch" path that
 * first copies the selected rows, dequantized to FP8, into HBM).
 *   kv4_quantize_write_fp8     the FP8 row: 576 E4M3 bytes, latent [0,512)
 *                              then rope [512,576), each x rounded to
 *                              nearest even and saturated at 448, no scale;
 *                              pool uint8 [num_slots, 576]; otherwise as
 *                              kv4_quantize_write
 *   kv4_decode_plan_fp8 /
 *   kv4_sparse_mla_decode_fp8  the decode over a pool of 576-byte FP8 rows:
 *                              arguments, layouts, workspace and errors as
 *                              kv4_sparse_mla_decode
 *   kv4_fp8_scratch            for every (b, s, k) the NVFP4 row key k
 *                              selects, dequantized as the decode does and
 *                              cast to E4M3, into row (b*Sq + s)*K + k of
 *                              scratch_dev uint8 [B*Sq*K, 576] (16-byte
 *                              aligned); masked keys give zero rows; index
 *                              errors as in the decode
 *   kv4_fp8_scratch_index      the indexing that makes that scratch buffer
 *                              look like a paged pool, for a decode of
 *                              B*Sq one-token requests: pt_out int32
 *                              [B*Sq, K/64] (entry (n, p) = n*(K/64) + p),
 *                              topk_out int32 [B*Sq, 1, K] (k where key k
 *                              of the original query is valid, -1 where it
 *                              is masked), lens_out int32 [B*Sq] (= K).  K
 *                              must be a multiple of 64 (else
 *                              KV4_ERR_UNSUPPORTED).
 * ------------------------------------------------------------------------- */
kv4_status kv4_quantize_write_fp8(const void* latent_dev, int64_t latent_row_stride,
                                  const void* rope_dev, int64_t rope_row_stride,
                                  const int64_t* slot_mapping_dev, int64_t n_tokens,
                                  uint8_t* pool_dev, int64_t num_slots, int32_t* dev_err,
                                  kv4_stream_t stream);
kv4_status kv4_decode_plan_fp8(int B, int Sq, int H, int K, int force_splits, int* splits,
                               size_t* workspace_bytes);
kv4_status kv4_sparse_mla_decode_fp8(const void* q_dev, const uint8_t* pool_dev,
                                     int64_t num_slots, const int32_t* page_table_dev,
                                     int64_t pt_stride, int page_size,
                                     const int32_t* topk_idx_dev, int K,
                                     const int32_t* seq_lens_dev, int B, int Sq, int H,
                                     float sm_scale, void* out_dev, float* lse_dev,
                                     void* workspace_dev, size_t workspace_bytes,
                                     int force_splits, int32_t* dev_err, kv4_stream_t stream);
kv4_status kv4_fp8_scratch(const uint8_t* pool_dev, int64_t num_slots,
                           const int32_t* page_table_dev, int64_t pt_stride, int page_size,
                           const int32_t* topk_idx_dev, int K, const int32_t* seq_lens_dev,
                           int B, int Sq, uint8_t* scratch_dev, int32_t* dev_err,
                           kv4_stream_t stream);
kv4_status kv4_fp8_scratch_index(const int32_t* topk_idx_dev, int K, const int32_t* seq_lens_dev,
                                 int B, int Sq, int32_t* pt_out_dev, int32_t* topk_out_dev,
                                 int32_t* lens_out_dev, kv4_stream_t stream);

/* ---------------------------------------------------------------------------
 * Decode-context parallelism (DCP).
 * Source: README "Parallelism and disaggregation" (ranks attend over their
 * part of the context and merge (o, lse)).  Ownership rule (this project's
 * reading): physical page p lives on rank p mod world, as page p / world of
 * that rank's own pool -- a rank holds only its pages, about 1/world of the
 * cache.  The cache write of a token goes to its owner's pool at the local
 * slot kv4_dcp_local_slots gives (slot_out = (page / world) * 64 + slot % 64
 * on the owner, -1 -- no write -- elsewhere; int64 [N] in and out).  The
 * decode reads through the rank-local page table of kv4_dcp_local_page_table
 * (pt_local [B, pt_stride] int32: p / world where the rank owns page p,
 * -1 elsewhere and for negative entries).  One decode step on `world` ranks
 * is:
 *   1. kv4_dcp_mask_topk on every rank: topk_out [B,Sq,K] int32 keeps the
 *      positions whose page the rank owns and is -1 elsewhere.  Positions
 *      outside [0, L_eff) are -1 on every rank; a position whose page entry
 *      cannot be read (page index >= pt_stride or a negative entry) is kept
 *      on rank 0 only, whose decode then reports KV4_DEV_BAD_PAGE.
 *   2. kv4_sparse_mla_decode_partial on every rank with its own pool, its
 *      pt_local and its topk_out: the
 *      same decode as kv4_sparse_mla_decode (same arguments, workspace and
 *      errors), except that o_dev is fp32 [B,Sq,H,512] -- the normalized
 *      weighted sum over the rank's keys, not rounded to bf16 -- and lse_dev
 *      that partial's lse (-inf when the rank holds no key of the row).
 *   3. An all-gather of (o, lse) across the ranks (by the caller, e.g. NCCL)
 *      into o_parts [R, n_rows, 512] and lse_parts [R, n_rows], where
 *      n_rows = B*Sq*H.
 *   4. kv4_merge_partials: out bf16 [n_rows, 512] and lse [n_rows] by
 *      log-sum-exp over the R partials (a partial with lse = -inf has weight
 *      0; no finite lse gives out = 0, lse = -inf).  o_parts and out 16-byte
 *      aligned.
 * Steps 1-2 with each rank's work in proportion to its share of the keys:
 *   1'. kv4_dcp_compact_topk: the same kept positions, moved to the front of
 *      each query's list in their order, -1 after them (topk_out [B,Sq,K]
 *      int32, not overlapping topk_idx), and their number per query in
 *      count_out int32 [B*Sq].
 *   2'. kv4_sparse_mla_decode_partial_counted: kv4_sparse_mla_decode_partial
 *      walking only the first k_count_dev[b*Sq + s] entries of each query's
 *      list (k_count_dev int32 [B*Sq], 4-byte aligned, read on the device;
 *      values are clamped to [0, K]).  A split whose tiles lie past the
 *      count contributes lse = -inf.  With 1'.'s output a rank at world R
 *      walks about K/R keys instead of K.
 * ------------------------------------------------------------------------- */
kv4_status kv4_dcp_mask_topk(const int32_t* topk_idx_dev, const int32_t* page_table_dev,
                             int64_t pt_stride, const int32_t* seq_lens_dev, int B, int Sq,
                             int K, int world, int rank, int32_t* topk_out_dev,
                             kv4_stream_t stream);
kv4_status kv4_dcp_local_page_table(const int32_t* page_table_dev, int64_t pt_stride, int B,
                                   int world, int rank, int32_t* pt_local_dev,
                                   kv4_stream_t stream);
kv4_status kv4_dcp_local_slots(const int64_t* slot_mapping_dev, int64_t n_tokens, int world,
                               int rank, int64_t* slots_out_dev, kv4_stream_t stream);
kv4_status kv4_sparse_mla_decode_partial(const void* q_dev, const uint8_t* pool_dev,
                                         int64_t num_slots, const int32_t* page_table_dev,
                                         int64_t pt_stride, int page_size,
                                         const int32_t* topk_idx_dev, int K,
                                         const int32_t* seq_lens_dev, int B, int Sq, int H,
                                         float sm_scale, float* o_dev, float* lse_dev,
                                         void* workspace_dev, size_t workspace_bytes,
                                         int force_splits, int32_t* dev_err,
                                         kv4_stream_t stream);
kv4_status kv4_dcp_compact_topk(const int32_t* topk_idx_dev, const int32_t* page_table_dev,
                                int64_t pt_stride, const int32_t* seq_lens_dev, int B, int Sq,
                                int K, int world, int rank, int32_t* topk_out_dev,
                                int32_t* count_out_dev, kv4_stream_t stream);
kv4_status kv4_sparse_mla_decode_partial_counted(
    const void* q_dev, const uint8_t* pool_dev, int64_t num_slots, const int32_t* page_table_dev,
    int64_t pt_stride, int page_size, const int32_t* topk_idx_dev, int K,
    const int32_t* k_count_dev, const int32_t* seq_lens_dev, int B, int Sq, int H, float sm_scale,
    float* o_dev, float* lse_dev, void* workspace_dev, size_t workspace_bytes, int force_splits,
    int32_t* dev_err, kv4_stream_t stream);
kv4_status kv4_merge_partials(const float* o_parts_dev, const float* lse_parts_dev, int R,
                              int64_t n_rows, void* out_dev, float* lse_dev,
                              kv4_stream_t stream);

/* ---------------------------------------------------------------------------
 * kv4_sparse_mla_decode_noalloc -- the same decode for callers that cannot
 * allocate device memory when they call it (for example a plugin whose host
 * engine hands it only its input and output buffers and owns every byte of
 * device memory, or code that must not call cudaMalloc because cudaMalloc can
 * synchronize the device).  The pages have no counterpart: it is an interface
 * variant of kv4_sparse_mla_decode, with the same arguments except the
 * workspace, and the same results.
 *   - The split-K partials go to a file-scope device array inside the library
 *     of kv4_noalloc_scratch_bytes() bytes (24 MiB).  Every device that loads
 *     the library holds it until the process exits.
 *   - Arguments are checked first, as in kv4_sparse_mla_decode (null or
 *     misaligned pointers: KV4_ERR_INVALID_ARG; shapes and page sizes:
 *     KV4_ERR_UNSUPPORTED).  Then a shape whose planned partials need more
 *     than the array returns KV4_ERR_SCRATCH_LIMIT and launches nothing
 *     (force fewer splits, or use kv4_sparse_mla_decode with a workspace).
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress: a host-side query that allocates nothing), so
 *     the address stays right across a device reset.  The first call on a
 *     device may also load the library's kernels there; make that first
 *     call before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents;
 *     nothing in it needs to start at zero (every partial is written before
 *     it is read).  Calls whose kernels overlap on the GPU (two streams, or
 *     two threads) race on the array: serialize them.
 *   - This entry point itself calls no cudaMalloc, cudaFree or allocating
 *     library routine.
 * ------------------------------------------------------------------------- */
kv4_status kv4_sparse_mla_decode_noalloc(const void* q_dev, const uint8_t* pool_dev,
                                         int64_t num_slots, const int32_t* page_table_dev,
                                         int64_t pt_stride, int page_size,
                                         const int32_t* topk_idx_dev, int K,
                                         const int32_t* seq_lens_dev, int B, int Sq, int H,
                                         float sm_scale, void* out_dev, float* lse_dev,
                                         int force_splits, int32_t* dev_err,
                                         kv4_stream_t stream);
size_t kv4_noalloc_scratch_bytes(void);

/* Test hook: the next decode launches use this bounded-wait limit (ns; 0
 * keeps the 1 s default) and, when fault_site == 1, one warp of each block
 * finishes its work and then waits on an mbarrier that nothing arrives on,
 * so that the wait runs out and KV4_DEV_TIMEOUT is reported while the block
 * still exits normally.  fault_site must be 0 or 1.  0, 0 restores the
 * defaults. */
kv4_status kv4_set_wait_limit(int64_t timeout_ns, int fault_site);

/* Measurement hook: when `cuda_event` (a cudaEvent_t) is non-NULL, every
 * later kv4_sparse_mla_decode call records it on its stream right after the
 * decode kernel and before the split-K merge kernel, so that a caller can
 * time the decode kernel alone with events on the same stream.  NULL turns
 * it off.  The event must outlive its use. */
kv4_status kv4_set_timing_event(void* cuda_event);

const char* kv4_status_str(kv4_status status);
int kv4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KV4MLA_H */
