"""GPU parity of the cache write with MSE-searched block scales
(kv4_quantize_write_mse) against the CPU oracle: bit-exact bytes on the four
sweep distributions (including round-half-even tie blocks and all-zero
blocks), and the decode over a pool written this way against the oracle's
decode over the oracle's own MSE-written rows."""
import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_nvfp4_gb300 import workloads as wl
from gpu_common import assert_close, bits, device_inputs, need_gpu, workload

pytestmark = pytest.mark.gpu


def kv():
    import bit_kv_cache_nvfp4_gb300 as m
    return m


@pytest.mark.parametrize("kind", wl.SWEEP_KINDS)
def test_mse_write_bit_exact(kind):
    need_gpu()
    n = 1 << 14                     # 524,288 blocks; the oracle's search is slow
    dev = torch.device("cuda")
    lat, rope = wl.sweep_rows(kind, 1, 0, n)
    slots = (np.arange(n, dtype=np.int64) * 7919) % n
    slots[::101] = -1
    pool = torch.full((n, 352), 0x5A, dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kv().quantize_write_mse(lat.to(dev), rope.to(dev), torch.from_numpy(slots).to(dev), pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = np.full((n, 352), 0x5A, dtype=np.uint8)
    assert oracle.quantize_write_mse(bits(lat), bits(rope), slots, ref) == oracle.OK
    got = pool.cpu().numpy()
    bad = np.nonzero((got != ref).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first slot {bad[:4]}"
    # how often the search moves a block's scale away from amax/6
    amax_ref = np.full((n, 352), 0x5A, dtype=np.uint8)
    assert oracle.quantize_write(bits(lat), bits(rope), slots, amax_ref) == oracle.OK
    changed = (amax_ref[:, 256:288] != ref[:, 256:288]).mean()
    print(f"{kind}: {100 * changed:.1f} % of block scales differ from amax/6")


def test_decode_over_mse_written_pool():
    need_gpu()
    w = workload("decode")
    dev = torch.device("cuda")
    pool = torch.zeros((w.num_slots, 352), dtype=torch.uint8, device=dev)
    for lat, rope, slots in wl.iter_pool_chunks(w, chunk=1 << 18, device=dev):
        kv().quantize_write_mse(lat, rope, slots, pool)
    q, pt, topk, lens = device_inputs(w)
    out, lse = kv().sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale)
    torch.cuda.synchronize()
    req = [0, 5, 15]
    qids = [(b, 0) for b in req]
    pt_c, pages, ns = wl.compact_pool_plan(w, qids)
    ids, cslots = wl.compact_pool_tokens(w, pages, qids)
    lat, rope = wl.token_rows(w, ids)
    cpool = np.zeros((max(ns, 64), 352), dtype=np.uint8)
    assert oracle.quantize_write_mse(bits(lat), bits(rope), cslots.numpy(), cpool) == oracle.OK
    qb = bits(wl.queries(w))
    outs, lses = [], []
    for b in req:
        st, o, l = oracle.sparse_mla_decode(
            np.ascontiguousarray(qb[b:b + 1]), cpool, np.ascontiguousarray(pt_c[b:b + 1].numpy()),
            np.ascontiguousarray(w.topk[b:b + 1].numpy()),
            np.ascontiguousarray(w.seq_lens[b:b + 1].numpy()), w.sm_scale)
        assert st == oracle.OK
        outs.append(o[0])
        lses.append(l[0])
    assert_close(out[req], lse[req], np.stack(outs), np.stack(lses), "decode over MSE rows")
