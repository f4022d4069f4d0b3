"""Negative controls: the parity checks must fail when the oracle computes
something else.

Each case plants one mistake on the oracle's side, on the CPU, and asserts
that the check used everywhere else (``assert_close`` for attention, byte
equality for the cache write) rejects the GPU's correct result against it:

- the oracle's softmax scale doubled (the pages' own negative control, a
  doubled scale that the check must catch);
- half of each query's selected keys dropped from the oracle's top-k list;
- one bit flipped in the oracle's copy of the written cache rows.

A check that passed any of these would be too loose to prove parity.  The
file also runs the pages' selection checks on the GPU path: the top-k order
does not matter, a row no query selects does not matter, a selected row
does.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_nvfp4_gb300 import workloads as wl
from gpu_common import assert_close, bits, device_inputs, gpu_pool, need_gpu, workload

pytestmark = pytest.mark.gpu


def _gpu_decode(w):
    import bit_kv_cache_nvfp4_gb300 as kv
    q, pt, topk, lens = device_inputs(w)
    out, lse = kv.sparse_mla_decode(q, gpu_pool(w), pt, topk, lens, w.sm_scale)
    torch.cuda.synchronize()
    return out, lse


def _oracle(w, sm_scale=None, topk=None):
    """The oracle's decode of every request of a small workload on its own
    copy of the whole pool, with the given scale and top-k list."""
    pool = np.zeros((w.num_slots, 352), dtype=np.uint8)
    for lat, rope, slots in wl.iter_pool_chunks(w):
        assert oracle.quantize_write(bits(lat), bits(rope), slots.numpy(), pool) == oracle.OK
    st, out, lse = oracle.sparse_mla_decode(
        bits(wl.queries(w)), pool, w.page_table.numpy(),
        np.ascontiguousarray((w.topk if topk is None else topk).numpy()), w.seq_lens.numpy(),
        w.sm_scale if sm_scale is None else sm_scale)
    assert st == oracle.OK
    return out, lse


def test_control_itself_passes():
    """The unaltered oracle passes the same check (so the failures below come
    from the planted mistakes)."""
    need_gpu()
    w = workload("tiny")
    out, lse = _gpu_decode(w)
    o_ref, l_ref = _oracle(w)
    assert_close(out, lse, o_ref, l_ref, "negative-control baseline (tiny)")


def test_doubled_scale_is_caught():
    need_gpu()
    w = workload("tiny")
    out, lse = _gpu_decode(w)
    o_ref, l_ref = _oracle(w, sm_scale=2.0 * w.sm_scale)
    with pytest.raises(AssertionError):
        assert_close(out, lse, o_ref, l_ref, "planted: doubled sm_scale")


def test_dropped_keys_are_caught():
    need_gpu()
    w = workload("tiny")
    out, lse = _gpu_decode(w)
    topk = w.topk.clone()
    topk[..., 1::2] = -1                   # every other selected key masked
    o_ref, l_ref = _oracle(w, topk=topk)
    with pytest.raises(AssertionError):
        assert_close(out, lse, o_ref, l_ref, "planted: half the keys dropped")


def test_flipped_cache_bit_is_caught():
    need_gpu()
    w = workload("tiny")
    host = np.zeros((w.num_slots, 352), dtype=np.uint8)
    for lat, rope, slots in wl.iter_pool_chunks(w):
        assert oracle.quantize_write(bits(lat), bits(rope), slots.numpy(), host) == oracle.OK
    gpu = gpu_pool(w).cpu().numpy()
    assert np.array_equal(gpu, host)
    slot = int(wl.newest_tokens(w)[2][0])
    host[slot, 7] ^= 0x10                  # one code bit of one written row
    assert not np.array_equal(gpu, host)


def test_topk_order_and_row_perturbations():
    """The pages' selection checks on the GPU path: the order of the top-k
    list does not matter (within the parity bound of the oracle); rewriting
    a row that no query selects leaves the output bit for bit unchanged;
    rewriting a selected row changes it."""
    need_gpu()
    import bit_kv_cache_nvfp4_gb300 as kv
    w = workload("tiny")
    dev = torch.device("cuda")
    q, pt, topk, lens = device_inputs(w)
    pool = gpu_pool(w).clone()
    out0, lse0 = kv.sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale)
    # a seeded permutation of each query's list
    g = torch.Generator().manual_seed(7)
    perm = torch.stack([torch.randperm(w.K, generator=g) for _ in range(w.B * w.Sq)])
    topk_p = torch.gather(w.topk.view(-1, w.K), 1, perm).view_as(w.topk)
    out_p, lse_p = kv.sparse_mla_decode(q, pool, pt, topk_p.to(dev), lens, w.sm_scale)
    torch.cuda.synchronize()
    o_ref, l_ref = _oracle(w)
    assert_close(out_p, lse_p, o_ref, l_ref, "tiny, top-k order permuted")

    # a position no query selects, and one that is selected
    chosen = set(int(x) for x in w.topk.flatten().tolist() if x >= 0)
    L = int(w.seq_lens[0])
    free = next(p for p in range(L) if p not in chosen)
    used = int(w.topk[0, 0, 0])
    def slot_of(p):
        return int(w.page_table[0, p // 64]) * 64 + p % 64
    lat = torch.full((1, 512), 3.0, dtype=torch.bfloat16, device=dev)
    rope = torch.full((1, 64), -2.0, dtype=torch.bfloat16, device=dev)
    kv.quantize_write(lat, rope, torch.tensor([slot_of(free)], dtype=torch.int64, device=dev),
                      pool)
    out_f, lse_f = kv.sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(out_f, out0) and torch.equal(lse_f, lse0)
    kv.quantize_write(lat, rope, torch.tensor([slot_of(used)], dtype=torch.int64, device=dev),
                      pool)
    out_u, lse_u = kv.sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale)
    torch.cuda.synchronize()
    assert not torch.equal(out_u, out0)
