/*
 * kv4ref.h -- the CPU oracle for NVFP4 latent-KV sparse-MLA decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the plain, slow, single-threaded
 * definition that the GPU path is checked against.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path (the CUDA library and its Python binding) never calls it and shares no
 * source with it.
 *
 * What it computes (sources are the web pages collected for this project):
 *  - The 352-byte NVFP4 KV row of the numinousmuses "inference-optimizations"
 *    README, section "4-bit KV cache": E2M1 latent values with one E4M3 scale
 *    per 16 values, plus the 64-dim rope part; it replaces the 576-byte FP8
 *    row.  The page fixes only the sizes; the byte order below is this
 *    project's reading:
 *       bytes [0,256)   latent codes, byte j = code(2j) | code(2j+1) << 4
 *       bytes [256,288) E4M3 scale i for latent elements 16i..16i+15
 *       bytes [288,352) rope element r as E4M3 (no scale)
 *  - Quantize: scale byte = E4M3_RNE_satfinite(amax/6) with amax/6 an IEEE
 *    fp32 division; each code = E2M1_RNE_satfinite(x / s) with s the decoded
 *    scale (fp32 division); s == 0 gives all-zero codes; the code keeps the
 *    sign of x.
 *  - Sparse MLA decode ("kv4mla ... dequantizes the 4-bit rows", same README
 *    section; split-K and the (o, lse) merge, README sections "Attention
 *    kernels" and "Parallelism and disaggregation"): for each query token,
 *    its top-k logical positions are mapped through a 64-token page table,
 *    scores over 576 dims (512 latent + 64 rope), softmax, and a weighted sum
 *    over the 512 latent dims (V is the latent part of the same row).
 *    Attention arithmetic is fp32, accumulated in index order.
 *
 * All pointers are HOST pointers.  bf16 inputs are passed as raw uint16 bit
 * patterns.  Functions return KV4REF_OK (0) or a nonzero status.
 */
#ifndef KV4REF_H
#define KV4REF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  KV4REF_OK = 0,
  KV4REF_ERR_ARG = 1,      /* bad sizes or null pointers; nothing written   */
  KV4REF_ERR_SLOT = 2,     /* a slot >= num_slots was skipped (write)        */
  KV4REF_ERR_PAGE = 3      /* a page-table entry or page index out of range;
                              the key was masked (decode)                    */
};

/* ---- scalar codecs (finite inputs; NaN/Inf are outside the contract) ---- */
uint8_t kv4ref_enc_e4m3(float x);   /* E4M3fn, RNE, saturate to +-448        */
float   kv4ref_dec_e4m3(uint8_t c);
uint8_t kv4ref_enc_e2m1(float x);   /* E2M1 in the low nibble, RNE, sat +-6  */
float   kv4ref_dec_e2m1(uint8_t c); /* low nibble only                        */
/* element-wise array forms of the two encoders */
void kv4ref_enc_e4m3_n(const float* x, uint8_t* codes, int64_t n);
void kv4ref_enc_e2m1_n(const float* x, uint8_t* codes, int64_t n);

/* ---- one row: 512 latent + 64 rope bf16 -> 352 bytes, and back ---------- */
void kv4ref_quantize_row(const uint16_t* latent_bf16, const uint16_t* rope_bf16,
                         uint8_t* row);
void kv4ref_dequant_row(const uint8_t* row, float* out576);

/* ---- the same row with MSE-searched block scales ------------------------
 * README "4-bit KV cache", DeepSeek V4 Pro bullet ("an MSE-searched scale");
 * the page gives no search rule, and this project's reading is: for each
 * block, c0 = E4M3_RNE(amax/6) as above; the candidate scale bytes are
 * c0-8 .. c0+1 (clipped to 0..126: one binade below and one step above);
 * each candidate s gives codes E2M1_RNE(x/s) (s == 0: all zero) and the
 * error E = sum_i (x_i - dec(code_i)*s)^2, computed in IEEE fp32 in element
 * order (each difference, square and sum rounded to nearest); the block
 * takes the candidate with the smallest E, the lowest scale byte on ties.
 * The rope part is as above. */
void kv4ref_quantize_row_mse(const uint16_t* latent_bf16, const uint16_t* rope_bf16,
                             uint8_t* row);
int kv4ref_quantize_write_mse(const uint16_t* latent_bf16, int64_t latent_stride,
                              const uint16_t* rope_bf16, int64_t rope_stride,
                              const int64_t* slot_mapping, int64_t n_tokens,
                              uint8_t* pool, int64_t num_slots);

/* ---- quantized write into a paged pool [num_slots, 352] -----------------
 * Token t goes to pool[slot_mapping[t]]; slot < 0 is skipped; slot >=
 * num_slots is skipped and reported with KV4REF_ERR_SLOT. */
int kv4ref_quantize_write(const uint16_t* latent_bf16, int64_t latent_stride,
                          const uint16_t* rope_bf16, int64_t rope_stride,
                          const int64_t* slot_mapping, int64_t n_tokens,
                          uint8_t* pool, int64_t num_slots);

/* ---- index resolution -----------------------------------------------------
 * slots[b,s,k] = page_table[b*pt_stride + idx/64]*64 + idx%64 for
 * 0 <= idx < L_eff(b,s) = seq_lens[b] - (Sq-1-s), else -1 (masked).
 * A page index >= pt_stride, a negative page entry or a slot >= num_slots
 * masks the key and makes the call return KV4REF_ERR_PAGE. */
int kv4ref_resolve_slots(const int32_t* page_table, int64_t pt_stride,
                         int page_size, const int32_t* topk_idx, int K,
                         const int32_t* seq_lens, int B, int Sq,
                         int64_t num_slots, int64_t* slots);

/* ---- gathered, dequantized rows [B,Sq,K,576] fp32; masked rows are 0 ---- */
int kv4ref_gather_dequant(const uint8_t* pool, int64_t num_slots,
                          const int32_t* page_table, int64_t pt_stride,
                          int page_size, const int32_t* topk_idx, int K,
                          const int32_t* seq_lens, int B, int Sq, float* rows,
                          uint8_t* valid);

/* ---- sparse MLA decode ----------------------------------------------------
 * q [B,Sq,H,576] bf16; out [B,Sq,H,512] fp32; lse [B,Sq,H] natural log,
 * including sm_scale.  splits >= 1 partitions each query's k-list into that
 * many contiguous chunks of ceil(K/splits) keys, computes a normalized
 * (o_i, lse_i) per chunk and merges them; splits == 1 is the direct form.
 * No valid key gives out = 0, lse = -inf. */
int kv4ref_sparse_mla_decode(const uint16_t* q_bf16, const uint8_t* pool,
                             int64_t num_slots, const int32_t* page_table,
                             int64_t pt_stride, int page_size,
                             const int32_t* topk_idx, int K,
                             const int32_t* seq_lens, int B, int Sq, int H,
                             float sm_scale, int splits, float* out,
                             float* lse);

/* ---- FP8 rows (the comparison paths) --------------------------------------
 * README "4-bit KV cache": the 352-byte row "replaces the 576-byte FP8 row",
 * and kv4mla is compared with a path that builds "an FP8 scratch copy".  The
 * FP8 row is read here as 576 E4M3 bytes -- latent 0..511 then rope 0..63,
 * each E4M3_RNE_satfinite(x) with no scale (the page gives no scale).
 *   kv4ref_quantize_write_fp8   bf16 latent/rope -> pool [num_slots, 576]
 *   kv4ref_dequant_row_fp8      576 bytes -> 576 floats
 *   kv4ref_fp8_scratch          for every (b, s, k): the NVFP4 row the key
 *                               selects, dequantized and cast to E4M3 (the
 *                               FP8 scratch copy), into scratch
 *                               [B*Sq*K, 576]; masked keys give zero rows
 *   kv4ref_sparse_mla_decode_fp8  kv4ref_sparse_mla_decode over a pool of
 *                               576-byte FP8 rows */
int kv4ref_quantize_write_fp8(const uint16_t* latent_bf16, int64_t latent_stride,
                              const uint16_t* rope_bf16, int64_t rope_stride,
                              const int64_t* slot_mapping, int64_t n_tokens,
                              uint8_t* pool, int64_t num_slots);
void kv4ref_dequant_row_fp8(const uint8_t* row, float* out576);
int kv4ref_fp8_scratch(const uint8_t* pool, int64_t num_slots, const int32_t* page_table,
                       int64_t pt_stride, int page_size, const int32_t* topk_idx, int K,
                       const int32_t* seq_lens, int B, int Sq, uint8_t* scratch);
int kv4ref_sparse_mla_decode_fp8(const uint16_t* q_bf16, const uint8_t* pool,
                                 int64_t num_slots, const int32_t* page_table,
                                 int64_t pt_stride, int page_size,
                                 const int32_t* topk_idx, int K,
                                 const int32_t* seq_lens, int B, int Sq, int H,
                                 float sm_scale, int splits, float* out, float* lse);

/* ---- log-sum-exp merge of S partials -------------------------------------
 * o_parts [S, n, D] (each normalized), lse_parts [S, n] -> out [n, D],
 * lse [n].  Partials with lse = -inf carry weight 0. */
void kv4ref_merge(const float* o_parts, const float* lse_parts, int S, int n,
                  int D, float* out, float* lse);

#ifdef __cplusplus
}
#endif

#endif /* KV4REF_H */
