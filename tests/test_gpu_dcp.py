"""Decode-context parallelism kernels on one GPU, against the CPU oracle.

The ranks are emulated one after another on the same GPU (nothing waits on
another rank).  For R ranks, every rank holds only its own pages: its pool
has the pages p with p % R == rank, as page p // R, written through
kv4_dcp_local_slots; kv4_dcp_mask_topk gives it its keys,
kv4_dcp_local_page_table its page table over that pool,
kv4_sparse_mla_decode_partial its fp32 (o, lse) -- or, compacted,
kv4_dcp_compact_topk its keys at the front of its lists and
kv4_sparse_mla_decode_partial_counted a decode over those only -- and
kv4_merge_partials
combines the stacked partials -- which must agree with the oracle's decode
over all keys within the decode tolerances.  The mask, the local page table
and the local slots are checked bit for bit against the rules written out in
numpy."""
import numpy as np
import pytest
import torch

from gpu_common import assert_close, device_inputs, need_gpu, oracle_decode, workload
from bit_kv_cache_nvfp4_gb300 import workloads as wl
from test_dcp_cpu import local_page_table, local_slots, owned_topk

pytestmark = pytest.mark.gpu


def kv():
    import bit_kv_cache_nvfp4_gb300 as m
    return m


@pytest.mark.parametrize("world", [2, 3, 8])
def test_mask_matches_ownership_rule(world):
    need_gpu()
    w = workload("decode")
    _, pt, topk, lens = device_inputs(w)
    topk_np = w.topk.numpy().copy()
    topk_np[0, 0, :7] = -1                              # padding
    topk_np[1, 0, 3] = int(w.seq_lens[1]) + 5           # past the sequence
    t = torch.from_numpy(topk_np).cuda()
    seen = np.zeros(topk_np.shape, dtype=np.int64)
    for r in range(world):
        got = kv().dcp_mask_topk(t, pt, lens, world, r).cpu().numpy()
        ref = owned_topk(topk_np, w.page_table.numpy(), w.seq_lens.numpy(), world, r)
        assert np.array_equal(got, ref), r
        seen += got >= 0
    valid = (topk_np >= 0) & (topk_np < w.seq_lens.numpy()[:, None, None])
    assert np.array_equal(seen, valid.astype(np.int64))    # a partition of the valid keys


@pytest.mark.parametrize("world", [2, 3, 8])
def test_compaction_matches_ownership_rule(world):
    """kv4_dcp_compact_topk: each query's kept positions (the mask's rule) in
    their order at the front of its list, -1 after them, and their count."""
    need_gpu()
    w = workload("decode")
    _, pt, topk, lens = device_inputs(w)
    topk_np = w.topk.numpy().copy()
    topk_np[0, 0, :7] = -1                              # padding
    topk_np[1, 0, 3] = int(w.seq_lens[1]) + 5           # past the sequence
    t = torch.from_numpy(topk_np).cuda()
    for r in range(world):
        got, cnt = kv().dcp_compact_topk(t, pt, lens, world, r)
        got, cnt = got.cpu().numpy(), cnt.cpu().numpy()
        kept = owned_topk(topk_np, w.page_table.numpy(), w.seq_lens.numpy(), world, r)
        for bs in range(w.B * w.Sq):
            row = kept.reshape(-1, w.K)[bs]
            ref = row[row >= 0]
            n = int(cnt[bs])
            assert n == ref.size, (r, bs)
            assert np.array_equal(got.reshape(-1, w.K)[bs, :n], ref), (r, bs)
            assert np.all(got.reshape(-1, w.K)[bs, n:] == -1), (r, bs)


@pytest.mark.parametrize("K", [5, 3000])
def test_compaction_ragged_and_multi_round(K):
    """Lists shorter than one round and longer than one round of the
    compaction block (256 threads x 8 entries), with padding, duplicates and
    positions past the sequence."""
    need_gpu()
    w = workload("decode")
    _, pt, _, lens = device_inputs(w)
    g = torch.Generator().manual_seed(11)
    L = w.seq_lens.to(torch.int64).view(-1, 1, 1)
    topk = (torch.randint(0, 1 << 30, (w.B, w.Sq, K), generator=g) % (L + 8) - 4).to(torch.int32)
    topk_np = topk.numpy()
    t = topk.cuda()
    world = 3
    total = np.zeros(w.B * w.Sq, dtype=np.int64)
    for r in range(world):
        got, cnt = kv().dcp_compact_topk(t, pt, lens, world, r)
        got, cnt = got.cpu().numpy().reshape(-1, K), cnt.cpu().numpy()
        kept = owned_topk(topk_np, w.page_table.numpy(), w.seq_lens.numpy(), world, r)
        for bs in range(w.B * w.Sq):
            ref = kept.reshape(-1, K)[bs]
            ref = ref[ref >= 0]
            assert int(cnt[bs]) == ref.size and np.array_equal(got[bs, :ref.size], ref)
            assert np.all(got[bs, ref.size:] == -1)
        total += cnt
    valid = ((topk_np >= 0) & (topk_np < w.seq_lens.numpy()[:, None, None])).reshape(-1, K)
    assert np.array_equal(total, valid.sum(axis=1))      # the ranks partition the valid keys


@pytest.mark.parametrize("world", [2, 3, 8])
def test_local_addressing_matches_rule(world):
    need_gpu()
    w = workload("decode")
    pt = w.page_table.clone()
    pt[0, 1] = -3                                        # a negative entry stays unreadable
    slots = torch.cat([wl.token_slots(w, b, torch.arange(0, int(w.seq_lens[b]), 997))
                       for b in range(w.B)])
    slots[::11] = -1                                     # skipped tokens stay skipped
    for r in range(world):
        got_pt = kv().dcp_local_page_table(pt.cuda(), world, r).cpu().numpy()
        assert np.array_equal(got_pt, local_page_table(pt.numpy(), world, r)), r
        got_sl = kv().dcp_local_slots(slots.cuda(), world, r).cpu().numpy()
        assert np.array_equal(got_sl, local_slots(slots.numpy(), world, r)), r


def local_pool(w, world, rank, dev):
    """Rank `rank`'s own pool: the pages it owns, written at local slots."""
    m = kv()
    n_pages = m.dcp_local_pages(w.num_slots // 64, world, rank)
    pool = torch.zeros((n_pages * 64, 352), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for lat, rope, slots in wl.iter_pool_chunks(w, chunk=1 << 18, device=dev):
        m.quantize_write(lat, rope, m.dcp_local_slots(slots, world, rank), pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return pool


@pytest.mark.parametrize("name,world,compact", [("decode", 1, False), ("decode", 2, False),
                                                ("decode", 4, False), ("decode", 8, False),
                                                ("long", 8, False), ("decode", 2, True),
                                                ("decode", 8, True), ("long", 8, True)])
def test_emulated_ranks_match_oracle(name, world, compact):
    """compact: each rank's keys moved to the front of its lists and its
    decode walking only those (kv4_dcp_compact_topk and
    kv4_sparse_mla_decode_partial_counted); else the masked full lists."""
    need_gpu()
    w = workload(name)
    q, pt, topk, lens = device_inputs(w)
    m = kv()
    parts_o, parts_l = [], []
    pages = []
    for r in range(world):
        pool = local_pool(w, world, r, q.device)          # this rank's pages only
        pages.append(pool.shape[0] // 64)
        count = None
        if compact:
            mine, count = m.dcp_compact_topk(topk, pt, lens, world, r)
        else:
            mine = m.dcp_mask_topk(topk, pt, lens, world, r)
        pt_local = m.dcp_local_page_table(pt, world, r)
        err = torch.zeros(1, dtype=torch.int32, device=q.device)
        o, l = m.sparse_mla_decode_partial(q, pool, pt_local, mine, lens, w.sm_scale,
                                           dev_err=err, k_count=count)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert o.dtype == torch.float32
        parts_o.append(o)
        parts_l.append(l)
        del pool
    # the ranks' pools partition the cache's pages, about 1/world each
    assert sum(pages) == w.num_slots // 64
    assert max(pages) == -(-(w.num_slots // 64) // world)
    out, lse = m.merge_partials(torch.stack(parts_o), torch.stack(parts_l))
    torch.cuda.synchronize()
    req = [0, 7, 15] if name == "decode" else [0, 41]
    out_ref, lse_ref = oracle_decode(w, req)
    what = f"{name} world={world}" + (" compacted" if compact else "")
    mo, ml = assert_close(out[req], lse[req], out_ref, lse_ref, what)
    print(f"{what}: max|out err| {mo:.3g}  max|lse err| {ml:.3g}")


def test_merge_of_empty_partials():
    need_gpu()
    o = torch.randn(3, 5, 512, device="cuda")
    l = torch.full((3, 5), float("-inf"), device="cuda")
    l[1, 2] = 0.5                                           # one finite partial in row 2
    out, lse = kv().merge_partials(o, l)
    torch.cuda.synchronize()
    assert torch.all(torch.isneginf(lse[[0, 1, 3, 4]]))
    assert torch.all(out[[0, 1, 3, 4]] == 0)
    assert abs(float(lse[2]) - 0.5) < 1e-6
    assert torch.equal(out[2], o[1, 2].to(torch.bfloat16))


def test_counted_decode_walks_only_the_counted_entries():
    """kv4_sparse_mla_decode_partial_counted with arbitrary counts (0, 1, K,
    and values that are not multiples of 128): the same result as the
    oracle's decode of the lists with every entry past the count masked."""
    need_gpu()
    import oracle
    from gpu_common import bits, gpu_pool
    w = workload("decode")
    q, pt, topk, lens = device_inputs(w)
    counts = torch.tensor([0, 1, 2048, 130, 1000, 127, 128, 2047, 5, 700, 1500, 64, 2000, 333,
                           256, 1919], dtype=torch.int32)[: w.B * w.Sq]
    o, l = kv().sparse_mla_decode_partial(q, gpu_pool(w), pt, topk, lens, w.sm_scale,
                                          k_count=counts.cuda())
    torch.cuda.synchronize()
    trunc = w.topk.clone()
    for bs in range(w.B * w.Sq):
        trunc.view(-1, w.K)[bs, int(counts[bs]):] = -1
    req = [0, 1, 3, 5, 7]
    qids = [(b, s) for b in req for s in range(w.Sq)]
    pt_c, pages = wl.compact_pool_plan(w, qids)[:2]
    ns = wl.compact_pool_plan(w, qids)[2]
    ids, cslots = wl.compact_pool_tokens(w, pages, qids)
    pool = np.zeros((max(ns, 64), 352), dtype=np.uint8)
    lat, rope = wl.token_rows(w, ids)
    assert oracle.quantize_write(bits(lat), bits(rope), cslots.numpy(), pool) == oracle.OK
    qb = bits(wl.queries(w))
    outs, lses = [], []
    for b in req:
        st, out, lse = oracle.sparse_mla_decode(
            np.ascontiguousarray(qb[b:b + 1]), pool, np.ascontiguousarray(pt_c[b:b + 1].numpy()),
            np.ascontiguousarray(trunc[b:b + 1].numpy()),
            np.ascontiguousarray(w.seq_lens[b:b + 1].numpy()), w.sm_scale)
        assert st == oracle.OK
        outs.append(out[0])
        lses.append(lse[0])
    assert_close(o[req], l[req], np.stack(outs), np.stack(lses), "decode, counted walk")
