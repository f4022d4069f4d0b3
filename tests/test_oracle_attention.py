"""Pins of the oracle's index resolution, sparse attention and merge.

Reference points independent of the oracle:
- top-k = the whole context reduces to dense attention, checked against
  PyTorch's scaled_dot_product_attention and logsumexp in float64;
- closed forms: q = 0 gives the mean of the selected V rows and
  lse = ln(n_valid); a single valid key gives out = V and lse = its score;
  duplicates count once per occurrence;
- invariants: permutation of the top-k order, split-K with any number of
  chunks equal to the direct form, perturbing an unselected row changes
  nothing and perturbing a selected one changes the output (the
  perturbation checks of the sgl-amd-mono "check-keys" test);
- index resolution on a hand-built page table.
Sources: numinousmuses "inference-optimizations" README ("4-bit KV cache"
kv4mla bullet; "Attention kernels" split-K bullet; "Parallelism and
disaggregation" (o, lse) merge bullet).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_nvfp4_gb300 import workloads as wl


def bf16_bits(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def bf16_values(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .double().numpy()


def small_case(L=300, B=2, Sq=1, H=4, seed=0, pt_extra=0):
    """A tiny paged pool of B requests of L tokens with a shuffled page table."""
    rng = np.random.default_rng(seed)
    pages = (L + 63) // 64
    perm = rng.permutation(B * pages).astype(np.int32)
    pt = np.full((B, pages + pt_extra), -1, dtype=np.int32)
    pt[:, :pages] = perm.reshape(B, pages)
    num_slots = B * pages * 64
    pool = np.zeros((num_slots, 352), dtype=np.uint8)
    lat = bf16_bits(rng.standard_normal((B * L, 512)))
    rope = bf16_bits(rng.standard_normal((B * L, 64)))
    slots = np.array([pt[b, p // 64] * 64 + p % 64 for b in range(B) for p in range(L)],
                     dtype=np.int64)
    assert oracle.quantize_write(lat, rope, slots, pool) == oracle.OK
    q = bf16_bits(rng.standard_normal((B, Sq, H, 576)))
    seq = np.full(B, L, dtype=np.int32)
    return dict(pool=pool, pt=pt, q=q, seq=seq, lat=lat, rope=rope, rng=rng, L=L)


def test_quantize_write_matches_rows_and_skips():
    c = small_case(L=70, B=1)
    lat, rope = c["lat"], c["rope"]
    pool = np.zeros_like(c["pool"])
    slots = np.arange(70, dtype=np.int64)
    slots[3] = -1
    slots[5] = pool.shape[0]          # out of range: skipped, reported
    st = oracle.quantize_write(lat, rope, slots, pool)
    assert st == oracle.ERR_SLOT
    assert not pool[3].any()
    for t in (0, 1, 69):
        assert np.array_equal(pool[t], oracle.quantize_row(lat[t], rope[t]))


def test_resolve_slots_handbuilt():
    pt = np.array([[5, 2, 7, -1], [0, 1, 3, 4]], dtype=np.int32)
    topk = np.array([[[0, 63, 64, 130, 191, 192, -1, 10]],
                     [[255, 256, 100, 0, 65, 64, 5, 1]]], dtype=np.int32)
    seq = np.array([192, 200], dtype=np.int32)
    st, slots = oracle.resolve_slots(pt, topk, seq, num_slots=8 * 64)
    exp0 = [5 * 64 + 0, 5 * 64 + 63, 2 * 64 + 0, 7 * 64 + 2, 7 * 64 + 63, -1, -1, 5 * 64 + 10]
    exp1 = [-1, -1, 1 * 64 + 36, 0, 1 * 64 + 1, 1 * 64 + 0, 5, 1]
    assert st == oracle.OK
    assert slots[0, 0].tolist() == exp0 and slots[1, 0].tolist() == exp1
    # a page entry past the pool masks the key and reports
    st, slots = oracle.resolve_slots(pt, topk, seq, num_slots=7 * 64)
    assert st == oracle.ERR_PAGE and slots[0, 0, 3] == -1 and slots[0, 0, 4] == -1
    # page index past the table: masked and reported
    st, slots = oracle.resolve_slots(pt[:, :2], topk, seq, num_slots=8 * 64)
    assert st == oracle.ERR_PAGE and slots[0, 0, 3] == -1


def test_causal_draft_lengths():
    pt = np.arange(4, dtype=np.int32).reshape(1, 4)
    seq = np.array([200], dtype=np.int32)
    Sq = 4
    topk = np.tile(np.array([196, 197, 198, 199, 0], dtype=np.int32), (1, Sq, 1))
    st, slots = oracle.resolve_slots(pt, topk, seq, num_slots=256)
    # token s sees positions < 200 - (3 - s)
    for s in range(Sq):
        visible = [p < 200 - (3 - s) for p in (196, 197, 198, 199, 0)]
        assert [x >= 0 for x in slots[0, s].tolist()] == visible


def dense_reference(q_bits, rows, scale):
    """PyTorch float64 SDPA + logsumexp over all rows (library routines)."""
    q = torch.from_numpy(bf16_values(q_bits))                    # [H,576]
    k = torch.from_numpy(rows.astype(np.float64))                # [n,576]
    v = k[:, :512]
    out = torch.nn.functional.scaled_dot_product_attention(
        q[None, :, None, :], k[None, None].expand(1, q.shape[0], -1, -1),
        v[None, None].expand(1, q.shape[0], -1, -1), scale=scale)[0, :, 0]
    lse = torch.logsumexp(scale * (q @ k.T), dim=-1)
    return out.numpy(), lse.numpy()


@pytest.mark.parametrize("H,L", [(1, 5), (4, 64), (16, 300)])
def test_topk_whole_context_equals_dense_attention(H, L):
    c = small_case(L=L, B=1, H=H, seed=L)
    topk = c["rng"].permutation(L).astype(np.int32).reshape(1, 1, L)
    scale = 1 / math.sqrt(576)
    st, out, lse = oracle.sparse_mla_decode(c["q"], c["pool"], c["pt"], topk, c["seq"], scale)
    assert st == oracle.OK
    st, rows, valid = oracle.gather_dequant(c["pool"], c["pt"], topk, c["seq"])
    assert valid.all()
    ref_out, ref_lse = dense_reference(c["q"][0, 0], rows[0, 0], scale)
    np.testing.assert_allclose(out[0, 0], ref_out, rtol=2e-5, atol=2e-5)
    np.testing.assert_allclose(lse[0, 0], ref_lse, rtol=0, atol=2e-5)


def test_dequant_rows_are_the_quantized_values():
    c = small_case(L=64, B=1)
    topk = np.arange(64, dtype=np.int32).reshape(1, 1, 64)
    st, rows, valid = oracle.gather_dequant(c["pool"], c["pt"], topk, c["seq"])
    for p in (0, 17, 63):
        slot = c["pt"][0, 0] * 64 + p
        assert np.array_equal(rows[0, 0, p], oracle.dequant_row(c["pool"][slot]))
        # every dequantized value is exact in bf16 (<= 6 significant bits)
        r = torch.from_numpy(rows[0, 0, p])
        assert torch.equal(r.to(torch.bfloat16).float(), r)


def test_zero_query_gives_mean_and_log_count():
    c = small_case(L=200, B=1, H=2)
    q = np.zeros_like(c["q"])
    topk = np.array([[[3, 150, 7, 7, -1, 500, 199]]], dtype=np.int32)   # dup 7, two masked
    st, out, lse = oracle.sparse_mla_decode(q, c["pool"], c["pt"], topk, c["seq"], 0.125)
    st, rows, valid = oracle.gather_dequant(c["pool"], c["pt"], topk, c["seq"])
    sel = rows[0, 0][valid[0, 0] == 1]
    assert sel.shape[0] == 5
    np.testing.assert_allclose(out[0, 0, 0], sel[:, :512].astype(np.float64).mean(0),
                               rtol=1e-6, atol=1e-6)
    assert lse[0, 0, 0] == pytest.approx(math.log(5), abs=1e-6)


def test_single_valid_key():
    c = small_case(L=100, B=1, H=3)
    topk = np.array([[[-1, 42, 1000]]], dtype=np.int32)
    scale = 0.05
    st, out, lse = oracle.sparse_mla_decode(c["q"], c["pool"], c["pt"], topk, c["seq"], scale)
    st, rows, valid = oracle.gather_dequant(c["pool"], c["pt"], topk, c["seq"])
    v = rows[0, 0, 1]
    for h in range(3):
        assert np.array_equal(out[0, 0, h], v[:512])
        score = scale * float(bf16_values(c["q"][0, 0, h]) @ v.astype(np.float64))
        assert lse[0, 0, h] == pytest.approx(score, abs=1e-5)


def test_no_valid_key():
    c = small_case(L=100, B=1, H=2)
    topk = np.array([[[-1, 100, 5000]]], dtype=np.int32)
    st, out, lse = oracle.sparse_mla_decode(c["q"], c["pool"], c["pt"], topk, c["seq"], 0.1)
    assert not out.any() and np.all(np.isneginf(lse))


def test_permutation_invariance_and_split_merge():
    c = small_case(L=1000, B=2, Sq=2, H=4, seed=5)
    K = 300
    rng = c["rng"]
    topk = np.stack([np.stack([rng.choice(999, K, replace=False) for _ in range(2)])
                     for _ in range(2)]).astype(np.int32)
    topk[0, 0, :10] = -1
    scale = 1 / 24
    st, out1, lse1 = oracle.sparse_mla_decode(c["q"], c["pool"], c["pt"], topk, c["seq"], scale)
    perm = rng.permutation(K)
    st, out2, lse2 = oracle.sparse_mla_decode(c["q"], c["pool"], c["pt"],
                                              np.ascontiguousarray(topk[:, :, perm]),
                                              c["seq"], scale)
    np.testing.assert_allclose(out2, out1, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(lse2, lse1, rtol=0, atol=1e-5)
    for S in (2, 3, 7, 300, 400):
        st, out3, lse3 = oracle.sparse_mla_decode(c["q"], c["pool"], c["pt"], topk, c["seq"],
                                                  scale, splits=S)
        np.testing.assert_allclose(out3, out1, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(lse3, lse1, rtol=0, atol=1e-5)


def test_merge_closed_forms():
    o = np.stack([np.full((1, 8), 1.0), np.full((1, 8), 3.0)]).astype(np.float32)
    lse = np.array([[0.5], [0.5]], dtype=np.float32)
    out, l = oracle.merge(o, lse)
    np.testing.assert_allclose(out, 2.0, rtol=1e-6)
    assert l[0] == pytest.approx(0.5 + math.log(2), abs=1e-6)
    lse = np.array([[0.0], [-np.inf]], dtype=np.float32)
    out, l = oracle.merge(o, lse)
    np.testing.assert_allclose(out, 1.0) and l[0] == 0.0
    out, l = oracle.merge(o, np.full((2, 1), -np.inf, dtype=np.float32))
    assert not out.any() and np.isneginf(l[0])


def test_perturbation_of_selected_and_unselected_rows():
    c = small_case(L=400, B=1, H=4, seed=9)
    topk = np.array([[c["rng"].choice(400, 100, replace=False)]], dtype=np.int32)
    scale = 1 / 24
    st, out0, lse0 = oracle.sparse_mla_decode(c["q"], c["pool"], c["pt"], topk, c["seq"], scale)
    unselected = sorted(set(range(400)) - set(topk.ravel().tolist()))[:5]
    pool = c["pool"].copy()
    for p in unselected:
        pool[c["pt"][0, p // 64] * 64 + p % 64] ^= 0x5A
    st, out1, lse1 = oracle.sparse_mla_decode(c["q"], pool, c["pt"], topk, c["seq"], scale)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)
    p = int(topk[0, 0, 17])
    pool[c["pt"][0, p // 64] * 64 + p % 64, :256] ^= 0x33
    st, out2, lse2 = oracle.sparse_mla_decode(c["q"], pool, c["pt"], topk, c["seq"], scale)
    assert not np.array_equal(out0, out2)


def test_compact_pool_equals_full_pool():
    """The oracle computed on a compact pool of only the touched pages (used
    for sampled checks at full size) equals the full-pool result."""
    w = wl.make_workload("tiny")
    lat, rope = wl.token_rows(w, torch.arange(w.total_tokens))
    slots = torch.cat([wl.token_slots(w, b, torch.arange(int(w.seq_lens[b])))
                       for b in range(w.B)])
    pool = np.zeros((w.num_slots, 352), dtype=np.uint8)
    to_bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    assert oracle.quantize_write(to_bits(lat), to_bits(rope), slots.numpy(), pool) == oracle.OK
    q = to_bits(wl.queries(w))
    st, out_full, lse_full = oracle.sparse_mla_decode(q, pool, w.page_table.numpy(),
                                                      w.topk.numpy(), w.seq_lens.numpy(),
                                                      w.sm_scale)
    pt_c, pages, ns = wl.compact_pool_plan(w, [(0, 0)])
    ids, cslots = wl.compact_pool_tokens(w, pages)
    lat_c, rope_c = wl.token_rows(w, ids)
    pool_c = np.zeros((ns, 352), dtype=np.uint8)
    assert oracle.quantize_write(to_bits(lat_c), to_bits(rope_c), cslots.numpy(), pool_c) == 0
    st, out_c, lse_c = oracle.sparse_mla_decode(q, pool_c, pt_c.numpy(), w.topk.numpy(),
                                                w.seq_lens.numpy(), w.sm_scale)
    assert np.array_equal(out_full, out_c) and np.array_equal(lse_full, lse_c)
    # only the selected rows of the compact pages (the form used at full size)
    ids, cslots = wl.compact_pool_tokens(w, pages, [(0, 0)])
    assert ids.numel() == int(((w.topk >= 0) & (w.topk < int(w.seq_lens[0]))).sum())
    lat_s, rope_s = wl.token_rows(w, ids)
    pool_s = np.zeros((ns, 352), dtype=np.uint8)
    assert oracle.quantize_write(to_bits(lat_s), to_bits(rope_s), cslots.numpy(), pool_s) == 0
    st, out_s, lse_s = oracle.sparse_mla_decode(q, pool_s, pt_c.numpy(), w.topk.numpy(),
                                                w.seq_lens.numpy(), w.sm_scale)
    assert np.array_equal(out_full, out_s) and np.array_equal(lse_full, lse_s)
