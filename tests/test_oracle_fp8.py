"""Pins of the oracle's FP8-row comparison paths (README "4-bit KV cache": the
576-byte FP8 row that the NVFP4 row replaces, and the FP8 scratch copy that
kv4mla avoids).  Each is checked against PyTorch, not against the oracle:

- FP8 row bytes = PyTorch's float32 -> float8_e4m3fn conversion of the bf16
  values (saturated at +-448), latent then rope; the row decoder = PyTorch's
  float8_e4m3fn decode;
- the FP8 scratch row of a key = PyTorch's E4M3 conversion of the NVFP4 row's
  dequantized values (the dequantizer is pinned in test_oracle_codec.py);
  masked keys give zero rows;
- the decode over FP8 rows with top-k = the whole context = PyTorch float64
  scaled_dot_product_attention and logsumexp over the decoded rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from test_oracle_attention import bf16_bits, bf16_values, dense_reference, small_case


def torch_e4m3(values):
    t = torch.as_tensor(np.asarray(values, dtype=np.float32)).clamp(-448, 448)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def torch_e4m3_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(
        torch.float8_e4m3fn).double().numpy()


def fp8_pool(L, B, seed, rope_scale=1.0):
    rng = np.random.default_rng(seed)
    pages = (L + 63) // 64
    perm = rng.permutation(B * pages).astype(np.int32)
    pt = perm.reshape(B, pages).copy()
    pool = np.zeros((B * pages * 64, 576), dtype=np.uint8)
    lat = bf16_bits(rng.standard_normal((B * L, 512)) * 4)
    rope = bf16_bits(rng.standard_normal((B * L, 64)) * rope_scale)
    slots = np.array([pt[b, p // 64] * 64 + p % 64 for b in range(B) for p in range(L)],
                     dtype=np.int64)
    assert oracle.quantize_write_fp8(lat, rope, slots, pool) == oracle.OK
    return pool, pt, lat, rope, slots, rng


def test_fp8_rows_are_torch_e4m3():
    pool, pt, lat, rope, slots, _ = fp8_pool(200, 2, 1, rope_scale=300)   # some saturate
    vals = np.concatenate([bf16_values(lat), bf16_values(rope)], axis=1)
    ref = torch_e4m3(vals)
    assert np.array_equal(pool[slots], ref)
    for i in (0, 17, 399):
        row = pool[slots[i]]
        assert np.array_equal(oracle.dequant_row_fp8(row).astype(np.float64),
                              torch_e4m3_decode(row))


def test_scratch_rows_are_e4m3_of_dequantized_nvfp4():
    c = small_case(L=300, B=2, Sq=2, H=2, seed=5)
    rng = c["rng"]
    topk = rng.integers(0, 300, (2, 2, 40)).astype(np.int32)
    topk[0, 1, :5] = -1
    topk[1, 0, 7] = 299                       # last position: masked for draft token 0
    st, scratch = oracle.fp8_scratch(c["pool"], c["pt"], topk, c["seq"])
    assert st == oracle.OK
    st, rows, valid = oracle.gather_dequant(c["pool"], c["pt"], topk, c["seq"])
    ref = torch_e4m3(rows.reshape(-1, 576))
    ref[~valid.reshape(-1).astype(bool)] = 0
    assert np.array_equal(scratch, ref)


@pytest.mark.parametrize("H,L", [(1, 9), (4, 64), (16, 300)])
def test_fp8_decode_whole_context_equals_dense_attention(H, L):
    pool, pt, _, _, _, rng = fp8_pool(L, 1, L)
    q = bf16_bits(rng.standard_normal((1, 1, H, 576)))
    topk = rng.permutation(L).astype(np.int32).reshape(1, 1, L)
    seq = np.full(1, L, dtype=np.int32)
    scale = 1 / math.sqrt(576)
    st, out, lse = oracle.sparse_mla_decode(q, pool, pt, topk, seq, scale, fp8_rows=True)
    assert st == oracle.OK
    slots = np.array([pt[0, p // 64] * 64 + p % 64 for p in topk[0, 0]])
    rows = torch_e4m3_decode(pool[slots])
    ref_out, ref_lse = dense_reference(q[0, 0], rows, scale)
    np.testing.assert_allclose(out[0, 0], ref_out, rtol=2e-5, atol=2e-5)
    np.testing.assert_allclose(lse[0, 0], ref_lse, rtol=0, atol=2e-5)
