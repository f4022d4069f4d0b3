"""GPU parity of the latent-only (288-byte) row layout against the CPU oracle.

The latent-only row (README "4-bit KV cache", the GLM-5.3-Flash bullet) is
the first 288 bytes of the 352-byte row: E2M1 codes and E4M3 scales, no rope.
The oracle needs no separate code for it:

- write bytes: the oracle's 352-byte row truncated to 288 bytes;
- gather: the oracle's dequantized 576-column row truncated to 512 columns;
- attention: the oracle's decode with the rope part of q set to zero.  The
  64 rope products are then +-0 and leave every fp32 score unchanged, so QK
  over 576 columns equals QK over the 512 latent columns.

The tolerances are the same as for the 352-byte rows.
"""
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


_POOL = {}


def latent_pool(w: wl.Workload) -> torch.Tensor:
    """The workload's 288-byte pool, written on the GPU by the library."""
    key = (w.name, w.seed)
    if key not in _POOL:
        _POOL.clear()
        torch.cuda.empty_cache()
        dev = torch.device("cuda")
        pool = torch.zeros((w.num_slots, 288), dtype=torch.uint8, device=dev)
        for lat, _rope, slots in wl.iter_pool_chunks(w, chunk=1 << 18, device=dev):
            kv().quantize_write_latent(lat, slots, pool)
        torch.cuda.synchronize()
        _POOL[key] = pool
    return _POOL[key]


def oracle_decode_latent(w: wl.Workload, requests, splits: int = 1):
    """Oracle (out, lse) for the listed requests with the rope part of q
    zeroed, on a compact 352-byte pool of the rows they select."""
    qids = [(b, s) for b in requests for s in range(w.Sq)]
    pt_c, pages, ns = wl.compact_pool_plan(w, qids)
    ids, cslots = wl.compact_pool_tokens(w, pages, qids)
    pool = np.zeros((max(ns, 64), 352), dtype=np.uint8)
    if ids.numel():
        lat, rope = wl.token_rows(w, ids)
        assert oracle.quantize_write(bits(lat), bits(rope), cslots.numpy(), pool) == oracle.OK
    q = bits(wl.queries(w)).copy()
    q[..., 512:] = 0                     # +0.0 in bf16
    outs, lses = [], []
    for b in requests:
        st, out, lse = oracle.sparse_mla_decode(
            np.ascontiguousarray(q[b:b + 1]), pool, np.ascontiguousarray(pt_c[b:b + 1].numpy()),
            np.ascontiguousarray(w.topk[b:b + 1].numpy()),
            np.ascontiguousarray(w.seq_lens[b:b + 1].numpy()), w.sm_scale, splits=splits)
        assert st == oracle.OK
        outs.append(out[0])
        lses.append(lse[0])
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("kind", wl.SWEEP_KINDS)
def test_quantize_latent_bit_exact(kind):
    need_gpu()
    n = 1 << 16
    dev = torch.device("cuda")
    lat, rope = wl.sweep_rows(kind, 0, 0, n)
    slots = (np.arange(n, dtype=np.int64) * 7919) % n         # a permutation
    slots[::97] = -1                                          # some tokens skipped
    pool = torch.full((n, 288), 0xA5, dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kv().quantize_write_latent(lat.to(dev), torch.from_numpy(slots).to(dev), pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = np.full((n, 352), 0xA5, dtype=np.uint8)
    assert oracle.quantize_write(bits(lat), bits(rope), slots, ref) == oracle.OK
    assert np.array_equal(pool.cpu().numpy(), ref[:, :288])


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_gather_latent_bit_exact(name):
    need_gpu()
    w = workload(name)
    pool = latent_pool(w)
    _, pt, topk, lens = device_inputs(w)
    rows = kv().debug_gather_dequant_latent(pool, pt, topk, lens)
    torch.cuda.synchronize()
    got = rows.float().cpu().numpy()
    qids = [(b, s) for b in range(w.B) for s in range(w.Sq)]
    pt_c, pages, ns = wl.compact_pool_plan(w, qids)
    ids, cslots = wl.compact_pool_tokens(w, pages, qids)
    lat, rope = wl.token_rows(w, ids)
    cpool = np.zeros((ns, 352), dtype=np.uint8)
    assert oracle.quantize_write(bits(lat), bits(rope), cslots.numpy(), cpool) == 0
    st, ref, _valid = oracle.gather_dequant(cpool, pt_c.numpy(), w.topk.numpy(),
                                            w.seq_lens.numpy())
    assert st == 0
    ref = np.ascontiguousarray(ref[..., :512])
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


CASES = {"tiny": None, "decode": None, "long": [0, 33, 63], "splitk": None}


@pytest.mark.parametrize("name", list(CASES))
def test_decode_latent_matches_oracle(name):
    need_gpu()
    w = workload(name)
    pool = latent_pool(w)
    q, pt, topk, lens = device_inputs(w)
    q512 = q[..., :512].contiguous()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = kv().sparse_mla_decode_latent(q512, pool, pt, topk, lens, w.sm_scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    req = CASES[name] or list(range(w.B))
    out_ref, lse_ref = oracle_decode_latent(w, req)
    mo, ml = assert_close(out[req], lse[req], out_ref, lse_ref, f"{name} (288-byte rows)")
    print(f"{name} latent rows: max|out err| {mo:.3g}  max|lse err| {ml:.3g}")


@pytest.mark.parametrize("S", [1, 2, 5, 16])
def test_decode_latent_forced_splits(S):
    """Every split path on 288-byte rows: one block, the 2-block cluster
    merge, and the workspace + merge kernel."""
    need_gpu()
    w = workload("decode")
    pool = latent_pool(w)
    q, pt, topk, lens = device_inputs(w)
    out, lse = kv().sparse_mla_decode_latent(q[..., :512].contiguous(), pool, pt, topk, lens,
                                             w.sm_scale, force_splits=S)
    torch.cuda.synchronize()
    req = [0, 7]
    out_ref, lse_ref = oracle_decode_latent(w, req)
    assert_close(out[req], lse[req], out_ref, lse_ref, f"S={S} (288-byte rows)")


def test_latent_argument_checks():
    need_gpu()
    m = kv()
    dev = torch.device("cuda")
    pool352 = torch.zeros((128, 352), dtype=torch.uint8, device=dev)
    pool288 = torch.zeros((128, 288), dtype=torch.uint8, device=dev)
    pt = torch.zeros((1, 2), dtype=torch.int32, device=dev)
    topk = torch.zeros((1, 1, 4), dtype=torch.int32, device=dev)
    lens = torch.full((1,), 64, dtype=torch.int32, device=dev)
    q512 = torch.zeros((1, 1, 64, 512), dtype=torch.bfloat16, device=dev)
    q576 = torch.zeros((1, 1, 64, 576), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        m.sparse_mla_decode_latent(q576, pool288, pt, topk, lens, 0.1)
    with pytest.raises(ValueError):
        m.sparse_mla_decode_latent(q512, pool352, pt, topk, lens, 0.1)
    with pytest.raises(ValueError):
        m.sparse_mla_decode(q576, pool288, pt, topk, lens, 0.1)
    out, lse = m.sparse_mla_decode_latent(q512, pool288, pt, topk, lens, 0.1)
    torch.cuda.synchronize()
    # all-zero rows: every score is 0, so out = 0 and lse = ln 4
    assert torch.all(out == 0)
    assert torch.allclose(lse, torch.full_like(lse, float(np.log(4.0))), atol=1e-6)
