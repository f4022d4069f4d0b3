"""GPU parity of the sparse MLA decode and the gather against the CPU oracle.

- gather indexing: kv4_debug_gather_dequant rows are bit-identical to the
  oracle's dequantized rows (masked keys give zero rows);
- attention: max |out err| <= 2e-2 on the bf16 output and |d lse| <= 1e-3,
  on the five workload shapes (all queries, or sampled requests at full
  size in the launch configuration the benchmark times), on ragged / masked
  / duplicated / padded index sets, every supported head count, several
  draft tokens and forced split counts;
- device-side errors: an out-of-range page entry masks the key and sets
  KV4_DEV_BAD_PAGE; a bounded wait that runs out sets KV4_DEV_TIMEOUT;
- determinism: repeated launches and CUDA-graph replays are bitwise equal.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_nvfp4_gb300 import workloads as wl
from gpu_common import (assert_close, bits, device_inputs, gpu_pool, need_gpu, oracle_decode,
                        oracle_decode_many, workload)

pytestmark = pytest.mark.gpu


def kv():
    import bit_kv_cache_nvfp4_gb300 as m
    return m


# ---------------------------------------------------------------------------
# full-size workloads
# ---------------------------------------------------------------------------
CASES = {
    "tiny": None,          # all requests
    "decode": None,
    "long": [0, 3, 7, 12, 17, 21, 26, 30, 33, 38, 40, 45, 50, 54, 59, 63],
    "specverify": [0, 2, 4, 6, 9, 11, 13, 15, 17, 19, 21, 23, 25, 27, 29, 31],
    "splitk": None,
}


@pytest.mark.parametrize("name", list(CASES))
def test_decode_matches_oracle(name):
    need_gpu()
    w = workload(name)
    pool = gpu_pool(w)
    q, pt, topk, lens = device_inputs(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = kv().sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    req = CASES[name] or list(range(w.B))
    out_ref, lse_ref = oracle_decode_many(w, req)
    mo, ml = assert_close(out[req], lse[req], out_ref, lse_ref, name)
    print(f"{name}: max|out err| {mo:.3g}  max|lse err| {ml:.3g}")
    # properties that hold for every request at full size
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("name", ["tiny", "decode", "splitk"])
def test_gather_bit_exact(name):
    need_gpu()
    w = workload(name)
    pool = gpu_pool(w)
    _, pt, topk, lens = device_inputs(w)
    rows = kv().debug_gather_dequant(pool, pt, topk, lens)
    torch.cuda.synchronize()
    got = rows.float().cpu().numpy()
    qids = [(b, s) for b in range(w.B) for s in range(w.Sq)]
    pt_c, pages, ns = wl.compact_pool_plan(w, qids)
    ids, cslots = wl.compact_pool_tokens(w, pages, qids)
    lat, rope = wl.token_rows(w, ids)
    cpool = np.zeros((ns, 352), dtype=np.uint8)
    assert oracle.quantize_write(bits(lat), bits(rope), cslots.numpy(), cpool) == 0
    st, ref, valid = oracle.gather_dequant(cpool, pt_c.numpy(), w.topk.numpy(),
                                           w.seq_lens.numpy())
    assert st == 0
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_long_context_launch_properties():
    """At full size in the benchmark's launch configuration: the planner's
    split count, and the same oracle agreement with a forced single split."""
    need_gpu()
    w = workload("long")
    pool = gpu_pool(w)
    q, pt, topk, lens = device_inputs(w)
    splits, ws = kv().decode_plan(w.B, w.Sq, w.H, w.K)
    out1, lse1 = kv().sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale)
    out2, lse2 = kv().sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale, force_splits=1)
    torch.cuda.synchronize()
    req = [3, 50]
    out_ref, lse_ref = oracle_decode(w, req)
    assert_close(out1[req], lse1[req], out_ref, lse_ref, f"long S={splits}")
    assert_close(out2[req], lse2[req], out_ref, lse_ref, "long S=1")
    print(f"long: planner splits={splits} workspace={ws} bytes")


# ---------------------------------------------------------------------------
# small hand-built cases with full pools
# ---------------------------------------------------------------------------
def small_problem(L, B, Sq, H, K, seed, kind="normal"):
    rng = np.random.default_rng(seed)
    pages = (L + 63) // 64
    perm = rng.permutation(B * pages + 3).astype(np.int32)[:B * pages]
    pt = perm.reshape(B, pages).copy()
    num_slots = (B * pages + 3) * 64
    lat = torch.from_numpy(rng.standard_normal((B * L, 512)).astype(np.float32))
    lat[:, rng.choice(512, 5, replace=False)] *= 8
    lat = lat.to(torch.bfloat16)
    rope = torch.from_numpy(rng.standard_normal((B * L, 64)).astype(np.float32)).to(torch.bfloat16)
    slots = np.array([pt[b, p // 64] * 64 + p % 64 for b in range(B) for p in range(L)],
                     dtype=np.int64)
    q = torch.from_numpy(rng.standard_normal((B, Sq, H, 576)).astype(np.float32)).to(torch.bfloat16)
    topk = np.stack([np.stack([rng.choice(L, K, replace=K > L) for _ in range(Sq)])
                     for _ in range(B)]).astype(np.int32)
    seq = np.full(B, L, dtype=np.int32)
    return dict(lat=lat, rope=rope, slots=slots, q=q, topk=topk, seq=seq, pt=pt,
                num_slots=num_slots, rng=rng)


def run_both(p, sm_scale=1 / 24, force_splits=0, expect_err=0):
    dev = torch.device("cuda")
    m = kv()
    pool = torch.zeros((p["num_slots"], 352), dtype=torch.uint8, device=dev)
    m.quantize_write(p["lat"].to(dev), p["rope"].to(dev), torch.from_numpy(p["slots"]).to(dev),
                     pool)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = m.sparse_mla_decode(p["q"].to(dev), pool, torch.from_numpy(p["pt"]).to(dev),
                                   torch.from_numpy(p["topk"]).to(dev),
                                   torch.from_numpy(p["seq"]).to(dev), sm_scale,
                                   force_splits=force_splits, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == expect_err
    hpool = np.zeros((p["num_slots"], 352), dtype=np.uint8)
    oracle.quantize_write(bits(p["lat"]), bits(p["rope"]), p["slots"], hpool)
    assert np.array_equal(pool.cpu().numpy(), hpool)
    st, out_ref, lse_ref = oracle.sparse_mla_decode(bits(p["q"]), hpool, p["pt"], p["topk"],
                                                    p["seq"], sm_scale)
    return out, lse, out_ref, lse_ref, st


@pytest.mark.parametrize("H", [16, 32, 64, 128])
@pytest.mark.parametrize("K", [1, 7, 128, 129, 300, 1000])
def test_heads_and_ragged_k(H, K):
    need_gpu()
    p = small_problem(L=1500, B=2, Sq=1, H=H, K=K, seed=H * 1000 + K)
    out, lse, out_ref, lse_ref, st = run_both(p)
    assert_close(out, lse, out_ref, lse_ref, f"H={H} K={K}")


# two splits merge inside a thread-block cluster (distributed shared
# memory); more go through the workspace and the merge kernel
@pytest.mark.parametrize("K,S", [(1000, 1), (1000, 2), (1000, 3), (1000, 4), (1000, 5),
                                 (1000, 8), (2000, 9), (2000, 16)])
def test_forced_splits(K, S):
    need_gpu()
    p = small_problem(L=3000, B=2, Sq=1, H=64, K=K, seed=77)
    out, lse, out_ref, lse_ref, st = run_both(p, force_splits=S)
    assert_close(out, lse, out_ref, lse_ref, f"K={K} S={S}")


def test_masking_padding_duplicates_and_draft():
    need_gpu()
    p = small_problem(L=700, B=3, Sq=3, H=32, K=260, seed=5)
    t = p["topk"]
    t[0, 0, :50] = -1                       # padding
    t[0, 1, 10:20] = 700 + np.arange(10)    # past the sequence
    t[1, :, 5:40] = t[1, :, 40:75]          # duplicates
    t[2, :, :4] = np.arange(696, 700)       # the draft positions: causal per token
    t[2, 2, :] = -1                         # a query with no valid key
    t[2, 2, 0] = 699                        # ... except a draft position it can see
    t[1, 2, :] = 699                        # one key, repeated
    out, lse, out_ref, lse_ref, st = run_both(p)
    assert_close(out, lse, out_ref, lse_ref, "masking")
    # a query with no valid key
    t[2, 1, :] = -1
    out, lse, out_ref, lse_ref, st = run_both(p)
    assert torch.all(out[2, 1] == 0) and torch.all(torch.isneginf(lse[2, 1]))
    assert_close(out, lse, out_ref, lse_ref, "no valid key")


def test_bad_page_entries_are_masked_and_flagged():
    need_gpu()
    p = small_problem(L=640, B=2, Sq=1, H=16, K=200, seed=9)
    p["pt"][1, 3] = p["num_slots"] // 64 + 5      # past the pool
    p["pt"][0, 2] = -7                            # negative
    p["topk"][0, 0, :3] = [130, 131, 140]         # land in page 2 of request 0
    p["topk"][1, 0, :3] = [200, 201, 250]         # land in page 3 of request 1
    out, lse, out_ref, lse_ref, st = run_both(p, expect_err=kv().DEV_BAD_PAGE)
    assert st == oracle.ERR_PAGE
    assert_close(out, lse, out_ref, lse_ref, "bad pages")


def test_page_index_past_table_is_flagged():
    need_gpu()
    p = small_problem(L=640, B=1, Sq=1, H=16, K=100, seed=10)
    p["seq"][0] = 10 * 64 + 100                   # longer than the table covers
    p["topk"][0, 0, :2] = [10 * 64 + 5, 10 * 64 + 50]
    out, lse, out_ref, lse_ref, st = run_both(p, expect_err=kv().DEV_BAD_PAGE)
    assert st == oracle.ERR_PAGE
    assert_close(out, lse, out_ref, lse_ref, "page index past table")


def test_sm_scale_and_large_scores():
    need_gpu()
    p = small_problem(L=900, B=1, Sq=1, H=64, K=512, seed=11)
    for scale in (1 / 24, 0.5, 2.0):           # sharper softmax exercises the running max
        out, lse, out_ref, lse_ref, st = run_both(p, sm_scale=scale)
        assert_close(out, lse, out_ref, lse_ref, f"scale {scale}")


def test_empty_shapes():
    need_gpu()
    m = kv()
    dev = torch.device("cuda")
    pool = torch.zeros((64, 352), dtype=torch.uint8, device=dev)
    pt = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    lens = torch.full((1,), 64, dtype=torch.int32, device=dev)
    q = torch.randn(1, 1, 16, 576, device=dev).to(torch.bfloat16)
    out, lse = m.sparse_mla_decode(q, pool, pt, torch.zeros((1, 1, 0), dtype=torch.int32,
                                                           device=dev), lens, 0.1)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    q0 = torch.zeros((0, 1, 16, 576), dtype=torch.bfloat16, device=dev)
    out, lse = m.sparse_mla_decode(q0, pool, pt[:0], torch.zeros((0, 1, 5), dtype=torch.int32,
                                                                 device=dev), lens[:0], 0.1)
    assert out.shape == (0, 1, 16, 512)


def test_invalid_arguments_raise():
    need_gpu()
    m = kv()
    dev = torch.device("cuda")
    pool = torch.zeros((64, 352), dtype=torch.uint8, device=dev)
    pt = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    lens = torch.full((1,), 64, dtype=torch.int32, device=dev)
    topk = torch.zeros((1, 1, 4), dtype=torch.int32, device=dev)
    q = torch.zeros((1, 1, 48, 576), dtype=torch.bfloat16, device=dev)
    with pytest.raises(m.Kv4Error) as e:
        m.sparse_mla_decode(q, pool, pt, topk, lens, 0.1)
    assert e.value.status == 2
    q16 = q[:, :, :16].contiguous()
    # 10 splits (more than a cluster merges) keep their partials in the
    # workspace: one that is too small is refused
    topk1200 = torch.zeros((1, 1, 1200), dtype=torch.int32, device=dev)
    with pytest.raises(m.Kv4Error) as e:
        m.sparse_mla_decode(q16, pool, pt, topk1200, lens, 0.1,
                            workspace=torch.zeros(4, dtype=torch.uint8, device=dev),
                            force_splits=10)
    assert e.value.status == 5
    # misaligned pool
    big = torch.zeros((65 * 352 + 1,), dtype=torch.uint8, device=dev)
    with pytest.raises(m.Kv4Error) as e:
        m.sparse_mla_decode(q16, big[1:].view(65, 352), pt, topk, lens, 0.1)
    assert e.value.status == 1


@pytest.mark.parametrize("S", [0, 2])
def test_determinism_and_graph_replay(S):
    """Planned splits (merge kernel) and 2 forced splits (merged inside a
    thread-block cluster)."""
    need_gpu()
    w = workload("decode")
    pool = gpu_pool(w)
    q, pt, topk, lens = device_inputs(w)
    m = kv()
    out_a, lse_a = m.sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale, force_splits=S)
    out_b, lse_b = m.sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale, force_splits=S)
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(lse_a, lse_b)
    out = torch.empty_like(out_a)
    lse = torch.empty_like(lse_a)
    splits, ws_bytes = m.decode_plan(w.B, w.Sq, w.H, w.K, S)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale, out=out, lse=lse, workspace=ws,
                            force_splits=S)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale, out=out, lse=lse, workspace=ws,
                            force_splits=S)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out_a.view(torch.int16))
        assert torch.equal(lse, lse_a)


def test_bounded_wait_reports_timeout():
    """A wait on an mbarrier nothing arrives on gives up after the limit and
    reports KV4_DEV_TIMEOUT; the context stays usable and results are right."""
    need_gpu()
    m = kv()
    p = small_problem(L=300, B=1, Sq=1, H=16, K=64, seed=12)
    try:
        m.set_wait_limit(2_000_000, 1)          # 2 ms, injected wait
        out, lse, out_ref, lse_ref, st = run_both(p, expect_err=m.DEV_TIMEOUT)
    finally:
        m.set_wait_limit(0, 0)
    assert_close(out, lse, out_ref, lse_ref, "after timeout")
    out, lse, out_ref, lse_ref, st = run_both(p)
    assert_close(out, lse, out_ref, lse_ref, "after reset")


@pytest.mark.parametrize("S", [0, 2])
def test_write_and_decode_matches_two_calls(S):
    """kv4_quantize_write_and_decode, whose decode reads q, the page table,
    the top-k list and the lengths while the write is still running, gives
    the pool bytes and the results of quantize_write then sparse_mla_decode.
    The new tokens' slots are zeroed first and every query selects its
    newest position, so a decode that read a row before the write landed
    would differ."""
    need_gpu()
    w = workload("decode")
    base = gpu_pool(w)
    q, pt, topk, lens = device_inputs(w)
    topk = topk.clone()
    topk[:, :, 0] = (lens - 1).view(-1, 1).to(torch.int32)      # the newest token
    m = kv()
    lat, rope, slots = wl.newest_tokens(w, device="cuda")
    results = []
    for fused in (False, True):
        pool = base.clone()
        pool[slots] = 0
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            out, lse = m.quantize_write_and_decode(lat, rope, slots, pool, q, pt, topk, lens,
                                                   w.sm_scale, force_splits=S, dev_err=err)
        else:
            m.quantize_write(lat, rope, slots, pool, err)
            out, lse = m.sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale, force_splits=S,
                                           dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        results.append((pool, out, lse))
    (pa, oa, la), (pb, ob, lb) = results
    assert torch.equal(pa, pb)
    assert torch.equal(pa, base)                    # the write restored the zeroed rows
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(la, lb)
