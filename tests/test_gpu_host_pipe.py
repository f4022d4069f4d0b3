"""Host-buffer steps (kv4_host_pipe_*, ``HostPipe``): the write-and-decode
step fed from pinned host memory, two steps in flight.

Several steps with different inputs (q, top-k positions, new token values,
a step that writes nothing) run through the pipe; each step's host results
must equal, bit for bit, those of the device entry point
kv4_quantize_write_and_decode called step after step on a second pool with
the same inputs, and the two pools must end equal.  The first step's inputs
are the workload's own, so its results are also checked against the oracle.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_nvfp4_gb300 import workloads as wl
from gpu_common import assert_close, bits, gpu_pool, need_gpu, oracle_decode, workload

pytestmark = pytest.mark.gpu


def _host_steps(w, n, pinned=True):
    """Per-step host inputs: step 0 the workload's own; step i > 0 scales q
    and the new tokens' values and shifts the top-k positions; step 2 writes
    no token.  With pinned=False the small inputs (lengths, new tokens,
    slots) stay in pageable memory, which the pipe copies instead of reading
    them through their device address."""
    q = wl.queries(w)
    L = w.seq_lens.to(torch.int64).view(-1, 1, 1)
    lat, rope, slots = wl.newest_tokens(w)
    steps = []
    for i in range(n):
        f = 1.0 + 0.25 * i
        qi = q if i == 0 else (q.float() * f).to(torch.bfloat16)
        ti = w.topk if i == 0 else ((w.topk.to(torch.int64) + 131 * i) % L).to(torch.int32)
        k = 0 if i == 2 else slots.shape[0]
        li = lat[:k] if i == 0 else (lat[:k].float() * f).to(torch.bfloat16)
        ri = rope[:k] if i == 0 else (rope[:k].float() * f).to(torch.bfloat16)
        small = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
        steps.append(dict(q=qi.contiguous().pin_memory(), topk=ti.contiguous().pin_memory(),
                          lens=small(w.seq_lens.clone()), lat=small(li.contiguous()),
                          rope=small(ri.contiguous()), slots=small(slots[:k].clone())))
    return steps


@pytest.mark.parametrize("name,force_splits,pinned", [("tiny", 0, True), ("tiny", 0, False),
                                                       ("decode", 0, True), ("decode", 2, True)])
def test_host_pipe_matches_device_steps(name, force_splits, pinned):
    need_gpu()
    import bit_kv_cache_nvfp4_gb300 as kv
    dev = torch.device("cuda")
    w = workload(name)
    base = gpu_pool(w)
    pool_pipe, pool_ref = base.clone(), base.clone()
    pt = w.page_table.to(dev)
    steps = _host_steps(w, 5, pinned)
    n_max = max(s["slots"].shape[0] for s in steps)
    outs = [torch.full((w.B, w.Sq, w.H, 512), float("nan"), dtype=torch.bfloat16).pin_memory()
            for _ in steps]
    lses = [torch.full((w.B, w.Sq, w.H), float("nan"), dtype=torch.float32).pin_memory()
            for _ in steps]
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    pipe = kv.HostPipe(w.B, w.Sq, w.H, w.K, n_max, dev, force_splits=force_splits)
    for s, o, l in zip(steps, outs, lses):
        pipe.step(s["lat"], s["rope"], s["slots"], pool_pipe, s["q"], pt, s["topk"], s["lens"],
                  w.sm_scale, o, l, dev_err=err)
    pipe.synchronize()
    pipe.close()
    assert int(err.item()) == 0

    for i, s in enumerate(steps):
        ref_out, ref_lse = kv.quantize_write_and_decode(
            s["lat"].to(dev), s["rope"].to(dev), s["slots"].to(dev), pool_ref, s["q"].to(dev), pt,
            s["topk"].to(dev), s["lens"].to(dev), w.sm_scale, force_splits=force_splits)
        torch.cuda.synchronize()
        assert np.array_equal(bits(outs[i]), bits(ref_out)), f"step {i}: out differs"
        assert torch.equal(lses[i].view(torch.int32), ref_lse.cpu().view(torch.int32)), \
            f"step {i}: lse differs"
    assert torch.equal(pool_pipe, pool_ref)

    requests = [0, w.B - 1] if w.B > 1 else [0]
    o_ref, l_ref = oracle_decode(w, requests)
    assert_close(outs[0][requests], lses[0][requests], o_ref, l_ref,
                 f"{name} host pipe step 0 (S={force_splits or 'plan'}"
                 f"{'' if pinned else ', pageable small inputs'})")


def test_host_pipe_rejects_bad_arguments():
    need_gpu()
    import bit_kv_cache_nvfp4_gb300 as kv
    dev = torch.device("cuda")
    w = workload("tiny")
    pool = gpu_pool(w)
    pt = w.page_table.to(dev)
    s = _host_steps(w, 1)[0]
    n = s["slots"].shape[0]
    out = torch.empty((w.B, w.Sq, w.H, 512), dtype=torch.bfloat16).pin_memory()
    lse = torch.empty((w.B, w.Sq, w.H), dtype=torch.float32).pin_memory()
    pipe = kv.HostPipe(w.B, w.Sq, w.H, w.K, max(n - 1, 0), dev)
    try:
        # more new tokens than the pipe was created for: refused, nothing enqueued
        with pytest.raises(kv.Kv4Error) as e:
            pipe.step(s["lat"], s["rope"], s["slots"], pool, s["q"], pt, s["topk"], s["lens"],
                      w.sm_scale, out, lse)
        assert e.value.status == 1
        with pytest.raises(TypeError):
            pipe.step(s["lat"][:0], s["rope"][:0], s["slots"][:0], pool, s["q"].to(dev), pt,
                      s["topk"], s["lens"], w.sm_scale, out, lse)
    finally:
        pipe.close()
