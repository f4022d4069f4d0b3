"""Helpers shared by the GPU parity tests: pools built on the device by the
library, and oracle results for the same seeded inputs on the host."""
from __future__ import annotations

import functools
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_nvfp4_gb300 import workloads as wl

# Tolerances.  Every lse must be within 1e-3 of the oracle's, and every
# output element within 2e-2 -- plainly, wherever the oracle's value is below
# 8 in magnitude.  At |out| >= 8 (the x8 outlier channels of the workloads
# reach it) half a bf16 ulp is itself more than 2e-2 (1/32 at [8, 16)): the
# rounding of the exact value to the bf16 output alone can exceed the bound,
# so there, and only there, each element is allowed 2e-2 for the computation
# plus half a bf16 ulp at its magnitude for the output rounding.
OUT_ATOL = 2e-2
LSE_ATOL = 1e-3
ROUNDING_ALLOWANCE_FROM = 8.0
MARGIN = 0.9

# Per-case parity records (largest errors, the oracle value at the worst
# element, the share of the bound used), printed at the end of the session by
# conftest.py and written as JSON where KV4_PARITY_LOG names a file.
PARITY_RECORDS: list = []


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |x| (2^(e-8) for |x| in [2^e, 2^(e+1)))."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def out_bound(out_ref: np.ndarray) -> np.ndarray:
    """Per-element bound on |out_gpu - out_ref|: 2e-2, plus half a bf16 ulp
    only where |out_ref| >= 8."""
    a = np.abs(np.asarray(out_ref, dtype=np.float64))
    return OUT_ATOL + np.where(a >= ROUNDING_ALLOWANCE_FROM, bf16_half_ulp(a), 0.0)


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy of its bit patterns (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@functools.lru_cache(maxsize=2)
def workload(name: str, seed: int = 0) -> wl.Workload:
    return wl.make_workload(name, seed)


_POOLS: dict = {}


def gpu_pool(w: wl.Workload) -> torch.Tensor:
    """The workload's NVFP4 pool, written on the GPU by kv4_quantize_write."""
    import bit_kv_cache_nvfp4_gb300 as kv
    key = (w.name, w.seed)
    if key not in _POOLS:
        _POOLS.clear()                       # keep one large pool at a time
        torch.cuda.empty_cache()
        dev = torch.device("cuda")
        pool = torch.zeros((w.num_slots, 352), dtype=torch.uint8, device=dev)
        for lat, rope, slots in wl.iter_pool_chunks(w, chunk=1 << 18, device=dev):
            kv.quantize_write(lat, rope, slots, pool)
        torch.cuda.synchronize()
        _POOLS[key] = pool
    return _POOLS[key]


def device_inputs(w: wl.Workload):
    dev = torch.device("cuda")
    q = wl.queries(w, dev)
    return (q, w.page_table.to(dev), w.topk.to(dev), w.seq_lens.to(dev))


def oracle_decode(w: wl.Workload, requests, splits: int = 1):
    """Oracle (out fp32 [n,Sq,H,512], lse [n,Sq,H]) for the listed requests,
    computed on a compact pool holding only the rows those requests select."""
    qids = [(b, s) for b in requests for s in range(w.Sq)]
    pt_c, pages, ns = wl.compact_pool_plan(w, qids)
    ids, cslots = wl.compact_pool_tokens(w, pages, qids)
    pool = np.zeros((max(ns, 64), 352), dtype=np.uint8)
    if ids.numel():
        lat, rope = wl.token_rows(w, ids)
        assert oracle.quantize_write(bits(lat), bits(rope), cslots.numpy(), pool) == oracle.OK
    q = bits(wl.queries(w))
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


def _oracle_decode_job(args):
    name, seed, requests = args
    torch.set_num_threads(1)
    return requests, oracle_decode(workload(name, seed), requests)


_ORACLE_POOL = None


def oracle_decode_many(w: wl.Workload, requests):
    """oracle_decode for many requests of a named workload, one request per
    job on a pool of single-threaded worker processes (started with spawn, so
    they hold no CUDA state); results in the order of `requests`."""
    global _ORACLE_POOL
    if _ORACLE_POOL is None:
        _ORACLE_POOL = mp.get_context("spawn").Pool(max(1, min(16, os.cpu_count() or 1)))
    jobs = [(w.name, w.seed // 1000, [b]) for b in requests]
    got = {}
    for reqs, (o, l) in _ORACLE_POOL.imap_unordered(_oracle_decode_job, jobs):
        got[reqs[0]] = (o[0], l[0])
    return (np.stack([got[b][0] for b in requests]), np.stack([got[b][1] for b in requests]))


def assert_close(out_gpu: torch.Tensor, lse_gpu: torch.Tensor, out_ref: np.ndarray,
                 lse_ref: np.ndarray, what: str = ""):
    o = out_gpu.float().cpu().numpy()
    l = lse_gpu.float().cpu().numpy()
    assert o.shape == out_ref.shape and l.shape == lse_ref.shape
    both_inf = np.isneginf(l) & np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(l), np.isneginf(lse_ref)), f"{what}: -inf lse pattern differs"
    err_o = np.abs(o.astype(np.float64) - out_ref)
    err_l = np.abs(np.where(both_inf, 0.0, l) - np.where(both_inf, 0.0, lse_ref))
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    bound = out_bound(out_ref)
    excess = err_o - bound
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess[i] <= 0, (f"{what}: |out err| {err_o[i]:.4g} > {bound[i]:.4g} at {i} "
                            f"(oracle {out_ref[i]:.5g}, gpu {o[i]:.5g})")
    mo, ml = float(err_o.max()), float(err_l.max())
    assert ml <= LSE_ATOL, f"{what}: max |lse err| {ml:.4g} > {LSE_ATOL}"
    used = err_o / bound
    j = np.unravel_index(np.argmax(used), used.shape)
    # headroom: no element uses more than 90 % of its bound (output rounding
    # alone takes up to 0.0156 of the 0.02 at |out| in [4, 8))
    assert used[j] <= MARGIN, (f"{what}: |out err| {err_o[j]:.4g} uses {used[j]:.3f} of its "
                               f"bound {bound[j]:.4g} (oracle {out_ref[j]:.5g})")
    small = np.abs(out_ref) < ROUNDING_ALLOWANCE_FROM
    PARITY_RECORDS.append({
        "case": what, "elements": int(o.size),
        "max_out_err": mo,
        "out_ref_at_max_err": float(out_ref[np.unravel_index(np.argmax(err_o), err_o.shape)]),
        "max_out_err_below_8": float(err_o[small].max()) if small.any() else 0.0,
        "max_out_err_at_8_and_above": float(err_o[~small].max()) if (~small).any() else 0.0,
        "max_share_of_out_bound": float(used[j]),
        "max_lse_err": ml, "share_of_lse_bound": ml / LSE_ATOL,
    })
    return mo, ml
