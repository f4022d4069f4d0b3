/*
 * kv4ref_attention.cpp -- oracle for index resolution, sparse MLA decode and
 * the split-K log-sum-exp merge.
 *
 * TEST INFRASTRUCTURE ONLY (see kv4ref.h).
 *
 * Sources (numinousmuses "inference-optimizations" README):
 *  - "4-bit KV cache", kv4mla bullet: a sparse MLA decode that reads the
 *    4-bit rows and dequantizes them; V is the latent part of the row.
 *  - "Attention kernels", split-K sparse decode bullet: the selected set is
 *    split into chunks that are attended separately.
 *  - "Parallelism and disaggregation", decode-context-parallel bullet: each
 *    part returns (o, lse) and a merge combines them.
 * The sgl-amd-mono PR text (a 64-token page table passed to the sparse
 * attention) fixes the page size.  Everything here is the plain definition:
 * a loop over queries, heads and keys, fp32 arithmetic accumulated in index
 * order, exp/log from the C library.
 */
#include "kv4ref.h"

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

constexpr int kRowBytes = 352;
constexpr int kQkDim = 576;
constexpr int kVDim = 512;

inline float bf16_to_float(uint16_t h) {
  uint32_t bits = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return f;
}

/* Attention of one query head over n dequantized rows (valid ones only).
 * Writes out[512] normalized and returns lse (natural log). */
float attend_one_head(const float* q576, const std::vector<const float*>& rows,
                      float sm_scale, float* out512) {
  const size_t n = rows.size();
  for (int d = 0; d < kVDim; ++d) out512[d] = 0.0f;
  if (n == 0) return -std::numeric_limits<float>::infinity();
  std::vector<float> score(n);
  float m = -std::numeric_limits<float>::infinity();
  for (size_t k = 0; k < n; ++k) {
    float acc = 0.0f;
    for (int d = 0; d < kQkDim; ++d) acc += q576[d] * rows[k][d];
    score[k] = sm_scale * acc;
    if (score[k] > m) m = score[k];
  }
  float l = 0.0f;
  std::vector<float> p(n);
  for (size_t k = 0; k < n; ++k) {
    p[k] = std::exp(score[k] - m);
    l += p[k];
  }
  for (size_t k = 0; k < n; ++k)
    for (int d = 0; d < kVDim; ++d) out512[d] += p[k] * rows[k][d];
  for (int d = 0; d < kVDim; ++d) out512[d] /= l;
  return m + std::log(l);
}

}  // namespace

namespace {

/* The decode over rows of either layout: row_bytes 352 (NVFP4) or 576
 * (FP8), dequantized by the matching row decoder. */
int decode_rows(const uint16_t* q_bf16, const uint8_t* pool, int64_t num_slots,
                const int32_t* page_table, int64_t pt_stride, int page_size,
                const int32_t* topk_idx, int K, const int32_t* seq_lens, int B, int Sq,
                int H, float sm_scale, int splits, float* out, float* lse, int row_bytes,
                void (*dequant)(const uint8_t*, float*)) {
  if (!q_bf16 || !pool || !page_table || !topk_idx || !seq_lens || !out ||
      !lse || B < 0 || Sq < 1 || H < 1 || K < 0 || splits < 1)
    return KV4REF_ERR_ARG;
  const int64_t n_keys = static_cast<int64_t>(B) * Sq * K;
  std::vector<int64_t> slots(static_cast<size_t>(n_keys));
  const int status =
      kv4ref_resolve_slots(page_table, pt_stride, page_size, topk_idx, K,
                           seq_lens, B, Sq, num_slots, slots.data());
  if (status == KV4REF_ERR_ARG) return status;

  const int chunk = (K + splits - 1) / (splits > 0 ? splits : 1);
  std::vector<float> kv(static_cast<size_t>(K) * kQkDim);
  std::vector<float> q(kQkDim);
  std::vector<float> o_parts(static_cast<size_t>(splits) * kVDim);
  std::vector<float> lse_parts(static_cast<size_t>(splits));
  for (int b = 0; b < B; ++b) {
    for (int s = 0; s < Sq; ++s) {
      const int64_t base = (static_cast<int64_t>(b) * Sq + s) * K;
      for (int k = 0; k < K; ++k)
        if (slots[base + k] >= 0)
          dequant(pool + slots[base + k] * row_bytes,
                  kv.data() + static_cast<size_t>(k) * kQkDim);
      for (int h = 0; h < H; ++h) {
        const int64_t qh = (static_cast<int64_t>(b) * Sq + s) * H + h;
        for (int d = 0; d < kQkDim; ++d) q[d] = bf16_to_float(q_bf16[qh * kQkDim + d]);
        for (int part = 0; part < splits; ++part) {
          std::vector<const float*> rows;
          const int k0 = part * chunk;
          const int k1 = (k0 + chunk < K) ? k0 + chunk : K;
          for (int k = k0; k < k1; ++k)
            if (slots[base + k] >= 0)
              rows.push_back(kv.data() + static_cast<size_t>(k) * kQkDim);
          lse_parts[part] = attend_one_head(q.data(), rows, sm_scale,
                                            o_parts.data() + part * kVDim);
        }
        if (splits == 1) {
          std::memcpy(out + qh * kVDim, o_parts.data(), kVDim * sizeof(float));
          lse[qh] = lse_parts[0];
        } else {
          kv4ref_merge(o_parts.data(), lse_parts.data(), splits, 1, kVDim,
                       out + qh * kVDim, lse + qh);
        }
      }
    }
  }
  return status;
}

}  // namespace

extern "C" {

int kv4ref_resolve_slots(const int32_t* page_table, int64_t pt_stride,
                         int page_size, const int32_t* topk_idx, int K,
                         const int32_t* seq_lens, int B, int Sq,
                         int64_t num_slots, int64_t* slots) {
  if (page_size != 64 || K < 0 || B < 0 || Sq < 1 || pt_stride < 1)
    return KV4REF_ERR_ARG;
  int status = KV4REF_OK;
  for (int b = 0; b < B; ++b) {
    for (int s = 0; s < Sq; ++s) {
      const int64_t l_eff = static_cast<int64_t>(seq_lens[b]) - (Sq - 1 - s);
      for (int k = 0; k < K; ++k) {
        const int64_t pos = (static_cast<int64_t>(b) * Sq + s) * K + k;
        const int64_t idx = topk_idx[pos];
        int64_t slot = -1;
        if (idx >= 0 && idx < l_eff) {
          const int64_t page_index = idx / page_size;
          if (page_index >= pt_stride) {
            status = KV4REF_ERR_PAGE;
          } else {
            const int64_t page = page_table[b * pt_stride + page_index];
            const int64_t cand = page * page_size + idx % page_size;
            if (page < 0 || cand >= num_slots) status = KV4REF_ERR_PAGE;
            else slot = cand;
          }
        }
        slots[pos] = slot;
      }
    }
  }
  return status;
}

int kv4ref_gather_dequant(const uint8_t* pool, int64_t num_slots,
                          const int32_t* page_table, int64_t pt_stride,
                          int page_size, const int32_t* topk_idx, int K,
                          const int32_t* seq_lens, int B, int Sq, float* rows,
                          uint8_t* valid) {
  const int64_t n = static_cast<int64_t>(B) * Sq * K;
  std::vector<int64_t> slots(static_cast<size_t>(n));
  const int status =
      kv4ref_resolve_slots(page_table, pt_stride, page_size, topk_idx, K,
                           seq_lens, B, Sq, num_slots, slots.data());
  if (status == KV4REF_ERR_ARG) return status;
  for (int64_t i = 0; i < n; ++i) {
    float* dst = rows + i * kQkDim;
    if (slots[i] < 0) {
      for (int d = 0; d < kQkDim; ++d) dst[d] = 0.0f;
      valid[i] = 0;
    } else {
      kv4ref_dequant_row(pool + slots[i] * kRowBytes, dst);
      valid[i] = 1;
    }
  }
  return status;
}

void kv4ref_merge(const float* o_parts, const float* lse_parts, int S, int n,
                  int D, float* out, float* lse) {
  const float ninf = -std::numeric_limits<float>::infinity();
  for (int i = 0; i < n; ++i) {
    float m = ninf;
    for (int s = 0; s < S; ++s) m = std::fmax(m, lse_parts[s * n + i]);
    for (int d = 0; d < D; ++d) out[i * D + d] = 0.0f;
    if (m == ninf) { lse[i] = ninf; continue; }
    float sum = 0.0f;
    for (int s = 0; s < S; ++s) {
      const float li = lse_parts[s * n + i];
      if (li == ninf) continue;
      sum += std::exp(li - m);
    }
    const float total = m + std::log(sum);
    lse[i] = total;
    for (int s = 0; s < S; ++s) {
      const float li = lse_parts[s * n + i];
      if (li == ninf) continue;
      const float w = std::exp(li - total);
      for (int d = 0; d < D; ++d)
        out[i * D + d] += w * o_parts[(static_cast<int64_t>(s) * n + i) * D + d];
    }
  }
}

int kv4ref_sparse_mla_decode(const uint16_t* q_bf16, const uint8_t* pool,
                             int64_t num_slots, const int32_t* page_table,
                             int64_t pt_stride, int page_size,
                             const int32_t* topk_idx, int K,
                             const int32_t* seq_lens, int B, int Sq, int H,
                             float sm_scale, int splits, float* out,
                             float* lse) {
  return decode_rows(q_bf16, pool, num_slots, page_table, pt_stride, page_size, topk_idx, K,
                     seq_lens, B, Sq, H, sm_scale, splits, out, lse, kRowBytes,
                     kv4ref_dequant_row);
}

int kv4ref_sparse_mla_decode_fp8(const uint16_t* q_bf16, const uint8_t* pool,
                                 int64_t num_slots, const int32_t* page_table,
                                 int64_t pt_stride, int page_size,
                                 const int32_t* topk_idx, int K,
                                 const int32_t* seq_lens, int B, int Sq, int H,
                                 float sm_scale, int splits, float* out, float* lse) {
  return decode_rows(q_bf16, pool, num_slots, page_table, pt_stride, page_size, topk_idx, K,
                     seq_lens, B, Sq, H, sm_scale, splits, out, lse, 576,
                     kv4ref_dequant_row_fp8);
}

int kv4ref_fp8_scratch(const uint8_t* pool, int64_t num_slots, const int32_t* page_table,
                       int64_t pt_stride, int page_size, const int32_t* topk_idx, int K,
                       const int32_t* seq_lens, int B, int Sq, uint8_t* scratch) {
  if (!pool || !page_table || !topk_idx || !seq_lens || !scratch || B < 0 || Sq < 1 || K < 0)
    return KV4REF_ERR_ARG;
  const int64_t n = static_cast<int64_t>(B) * Sq * K;
  std::vector<int64_t> slots(static_cast<size_t>(n));
  const int status = kv4ref_resolve_slots(page_table, pt_stride, page_size, topk_idx, K,
                                          seq_lens, B, Sq, num_slots, slots.data());
  if (status == KV4REF_ERR_ARG) return status;
  float row[kQkDim];
  for (int64_t i = 0; i < n; ++i) {
    uint8_t* dst = scratch + i * 576;
    if (slots[i] < 0) {
      std::memset(dst, 0, 576);
      continue;
    }
    kv4ref_dequant_row(pool + slots[i] * kRowBytes, row);
    for (int d = 0; d < kQkDim; ++d) dst[d] = kv4ref_enc_e4m3(row[d]);
  }
  return status;
}

}  // extern "C"
