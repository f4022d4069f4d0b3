"""The decode entry point that allocates nothing (kv4_sparse_mla_decode_noalloc).

It exists for callers that cannot allocate device memory when they run the
decode -- e.g. a plugin whose host engine gives it only its inputs and
outputs and owns all device memory -- and keeps its split-K partials in a
static device array inside the library.  This test calls it through the
C ABI on a shape forced to 16 splits -- more than one thread block cluster
merges, so the partials do go to the array:

- first with other queries (negated), which fills the array with partials
  unlike the ones the next call must produce;
- then twice in a row with the real queries, each result checked against the
  regular entry point and against the CPU oracle, within the parity bound.

A call that read a stale partial instead of writing its own would fail the
first of those checks.  It also checks that a shape needing more partial
storage than the array holds is refused with KV4_ERR_SCRATCH_LIMIT.  The file
is collected last and builds everything it needs itself, so it passes both
alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from bit_kv_cache_nvfp4_gb300 import workloads as wl
from gpu_common import LSE_ATOL, need_gpu, oracle_decode, out_bound

pytestmark = pytest.mark.gpu

KV4_ERR_SCRATCH_LIMIT = 6


def _noalloc_fn(lib):
    f = lib.kv4_sparse_mla_decode_noalloc
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [P, P, i64, P, i64, i32, P, i32, P, i32, i32, i32, ctypes.c_float, P, P, i32,
                  P, P]
    f.restype = i32
    lib.kv4_noalloc_scratch_bytes.argtypes = []
    lib.kv4_noalloc_scratch_bytes.restype = ctypes.c_size_t
    return f


def _call(f, q, pool, pt, topk, lens, w, out, lse, err, force_splits=0):
    stream = torch.cuda.current_stream().cuda_stream
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return f(p(q), p(pool), pool.shape[0], p(pt), pt.shape[1], 64, p(topk), topk.shape[2],
             p(lens), q.shape[0], q.shape[1], q.shape[2], ctypes.c_float(w.sm_scale), p(out),
             p(lse), force_splits, p(err), ctypes.c_void_p(stream))


def test_noalloc_decode_matches_regular_entry_point():
    need_gpu()
    import bit_kv_cache_nvfp4_gb300 as kv
    lib = kv.load_library()
    f = _noalloc_fn(lib)
    dev = torch.device("cuda")
    w = wl.make_workload("splitk")           # 2 requests x 64 tiles of 128 keys
    pool = torch.zeros((w.num_slots, 352), dtype=torch.uint8, device=dev)
    for lat, rope, slots in wl.iter_pool_chunks(w, device=dev):
        kv.quantize_write(lat, rope, slots, pool)
    q = wl.queries(w, dev)
    pt, topk, lens = w.page_table.to(dev), w.topk.to(dev), w.seq_lens.to(dev)
    splits, ws_bytes = kv.decode_plan(w.B, w.Sq, w.H, w.K, 16)
    assert splits == 16 and 0 < ws_bytes <= lib.kv4_noalloc_scratch_bytes()

    ref_out, ref_lse = kv.sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale)
    torch.cuda.synchronize()
    ref_o = ref_out.float().cpu().numpy()
    ref_l = ref_lse.cpu().numpy()
    ora_o, ora_l = oracle_decode(w, list(range(w.B)))

    # other queries first: the array then holds partials unlike the next call's
    other_out, other_lse = torch.empty_like(ref_out), torch.empty_like(ref_lse)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    assert _call(f, q.neg(), pool, pt, topk, lens, w, other_out, other_lse, err,
                 force_splits=16) == 0
    torch.cuda.synchronize()
    assert not torch.equal(other_lse, ref_lse)

    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        assert _call(f, q, pool, pt, topk, lens, w, out, lse, err, force_splits=16) == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        assert np.isfinite(o).all() and np.isfinite(l).all(), f"call {call}"
        for what, ro, rl in (("regular entry point", ref_o, ref_l), ("oracle", ora_o, ora_l)):
            assert np.all(np.abs(o - ro) <= out_bound(ro)), f"call {call} vs {what}"
            assert np.all(np.abs(l - rl) <= LSE_ATOL), f"call {call} vs {what}"


def test_noalloc_refuses_shapes_beyond_its_scratch():
    need_gpu()
    import bit_kv_cache_nvfp4_gb300 as kv
    lib = kv.load_library()
    f = _noalloc_fn(lib)
    dev = torch.device("cuda")
    w = wl.make_workload("decode")
    # 16 splits of 16 requests x 64 heads need 33.6 MB of partials (> 24 MiB)
    _, ws_bytes = kv.decode_plan(w.B, w.Sq, w.H, w.K, 16)
    assert ws_bytes > lib.kv4_noalloc_scratch_bytes()
    pool = torch.zeros((w.num_slots, 352), dtype=torch.uint8, device=dev)
    q = wl.queries(w, dev)
    pt, topk, lens = w.page_table.to(dev), w.topk.to(dev), w.seq_lens.to(dev)
    out = torch.empty((w.B, w.Sq, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Sq, w.H), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    assert _call(f, q, pool, pt, topk, lens, w, out, lse, err, force_splits=16) == \
        KV4_ERR_SCRATCH_LIMIT
