"""GPU parity of the FP8 comparison paths against the CPU oracle:

- the 576-byte FP8 row write: bit-exact bytes (including saturation);
- the FP8 scratch copy of the NVFP4 rows a query selects: bit-exact bytes;
- the decode over FP8 rows and the decode over the scratch copy (the path
  the README's kv4mla bullet compares against): within the decode
  tolerances of the oracle's decode over the same FP8 rows.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_nvfp4_gb300 import workloads as wl
from gpu_common import assert_close, bits, device_inputs, gpu_pool, need_gpu, workload

pytestmark = pytest.mark.gpu


def kv():
    import bit_kv_cache_nvfp4_gb300 as m
    return m


_FP8 = {}


def fp8_pool(w):
    key = (w.name, w.seed)
    if key not in _FP8:
        _FP8.clear()
        torch.cuda.empty_cache()
        dev = torch.device("cuda")
        pool = torch.zeros((w.num_slots, 576), dtype=torch.uint8, device=dev)
        for lat, rope, slots in wl.iter_pool_chunks(w, chunk=1 << 18, device=dev):
            kv().quantize_write_fp8(lat, rope, slots, pool)
        torch.cuda.synchronize()
        _FP8[key] = pool
    return _FP8[key]


def oracle_fp8_decode(w, requests):
    qids = [(b, s) for b in requests for s in range(w.Sq)]
    pt_c, pages, ns = wl.compact_pool_plan(w, qids)
    ids, cslots = wl.compact_pool_tokens(w, pages, qids)
    pool = np.zeros((max(ns, 64), 576), dtype=np.uint8)
    lat, rope = wl.token_rows(w, ids)
    assert oracle.quantize_write_fp8(bits(lat), bits(rope), cslots.numpy(), pool) == oracle.OK
    q = bits(wl.queries(w))
    outs, lses = [], []
    for b in requests:
        st, o, l = oracle.sparse_mla_decode(
            np.ascontiguousarray(q[b:b + 1]), pool, np.ascontiguousarray(pt_c[b:b + 1].numpy()),
            np.ascontiguousarray(w.topk[b:b + 1].numpy()),
            np.ascontiguousarray(w.seq_lens[b:b + 1].numpy()), w.sm_scale, fp8_rows=True)
        assert st == oracle.OK
        outs.append(o[0])
        lses.append(l[0])
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("kind,rope_scale", [("normal", 1.0), ("laplace", 1.0), ("normal", 300.0)])
def test_fp8_write_bit_exact(kind, rope_scale):
    need_gpu()
    n = 1 << 16
    dev = torch.device("cuda")
    lat, rope = wl.sweep_rows(kind, 2, 0, n)
    lat = (lat.float() * 40).to(torch.bfloat16)              # some latent values saturate too
    rope = (rope.float() * rope_scale).to(torch.bfloat16)
    slots = (np.arange(n, dtype=np.int64) * 7919) % n
    slots[::89] = -1
    pool = torch.full((n, 576), 0x3C, dtype=torch.uint8, device=dev)
    kv().quantize_write_fp8(lat.to(dev), rope.to(dev), torch.from_numpy(slots).to(dev), pool)
    torch.cuda.synchronize()
    ref = np.full((n, 576), 0x3C, dtype=np.uint8)
    assert oracle.quantize_write_fp8(bits(lat), bits(rope), slots, ref) == oracle.OK
    assert np.array_equal(pool.cpu().numpy(), ref)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_fp8_scratch_bit_exact(name):
    need_gpu()
    w = workload(name)
    pool = gpu_pool(w)
    _, pt, topk, lens = device_inputs(w)
    scratch = kv().fp8_scratch(pool, pt, topk, lens)
    torch.cuda.synchronize()
    qids = [(b, s) for b in range(w.B) for s in range(w.Sq)]
    pt_c, pages, ns = wl.compact_pool_plan(w, qids)
    ids, cslots = wl.compact_pool_tokens(w, pages, qids)
    lat, rope = wl.token_rows(w, ids)
    cpool = np.zeros((ns, 352), dtype=np.uint8)
    assert oracle.quantize_write(bits(lat), bits(rope), cslots.numpy(), cpool) == 0
    st, ref = oracle.fp8_scratch(cpool, pt_c.numpy(), w.topk.numpy(), w.seq_lens.numpy())
    assert st == 0
    assert np.array_equal(scratch.cpu().numpy(), ref)


@pytest.mark.parametrize("name,req", [("tiny", None), ("decode", None), ("long", [0, 31, 63])])
def test_fp8_decode_matches_oracle(name, req):
    need_gpu()
    w = workload(name)
    pool = fp8_pool(w)
    q, pt, topk, lens = device_inputs(w)
    out, lse = kv().sparse_mla_decode_fp8(q, pool, pt, topk, lens, w.sm_scale)
    torch.cuda.synchronize()
    req = req or list(range(w.B))
    out_ref, lse_ref = oracle_fp8_decode(w, req)
    assert_close(out[req], lse[req], out_ref, lse_ref, f"{name} FP8 rows")


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_scratch_path_matches_oracle(name):
    """Scratch copy + FP8 decode over it, against the oracle's decode over the
    oracle's scratch copy with the same indexing."""
    need_gpu()
    w = workload(name)
    pool = gpu_pool(w)
    q, pt, topk, lens = device_inputs(w)
    m = kv()
    scratch = m.fp8_scratch(pool, pt, topk, lens)
    s_pt, s_topk, s_lens = m.scratch_index(topk, lens)
    qs = q.reshape(w.B * w.Sq, 1, w.H, 576).contiguous()
    out, lse = m.sparse_mla_decode_fp8(qs, scratch, s_pt, s_topk, s_lens, w.sm_scale)
    torch.cuda.synchronize()
    qids = [(b, s) for b in range(w.B) for s in range(w.Sq)]
    pt_c, pages, ns = wl.compact_pool_plan(w, qids)
    ids, cslots = wl.compact_pool_tokens(w, pages, qids)
    lat, rope = wl.token_rows(w, ids)
    cpool = np.zeros((ns, 352), dtype=np.uint8)
    assert oracle.quantize_write(bits(lat), bits(rope), cslots.numpy(), cpool) == 0
    st, ref_scratch = oracle.fp8_scratch(cpool, pt_c.numpy(), w.topk.numpy(), w.seq_lens.numpy())
    st, o_ref, l_ref = oracle.sparse_mla_decode(
        bits(qs.cpu()), ref_scratch, s_pt.cpu().numpy(), s_topk.cpu().numpy(),
        s_lens.cpu().numpy(), w.sm_scale, fp8_rows=True)
    assert st == oracle.OK
    assert_close(out, lse, o_ref, l_ref, f"{name} scratch path")
