"""Decode-context parallelism on CPU (gloo, world size 2 and 3): every rank
holds only its own pages -- physical page p (p % world == rank) as page
p // world of a rank-local pool, written at the local slots -- takes the keys
on its pages, computes its partial (o, lse) with the oracle over that local
pool through the rank-local page table, the ranks exchange the partials with
the library's gather_partials over torch.distributed, and the oracle's
log-sum-exp merge of the gathered partials must equal the oracle's decode
over all keys on one global pool.  This covers the multi-rank exchange, the
ownership partition and the local addressing; the GPU kernels of the same
steps are covered by tests/test_gpu_dcp.py on one GPU."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def owned_topk(topk, page_table, seq_lens, world, rank):
    """The ownership rule written out: keep position idx of (b, s) when it is
    valid and its physical page is owned by `rank`; -1 elsewhere."""
    B, Sq, K = topk.shape
    out = np.full_like(topk, -1)
    for b in range(B):
        for s in range(Sq):
            l_eff = int(seq_lens[b]) - (Sq - 1 - s)
            for k in range(K):
                idx = int(topk[b, s, k])
                if 0 <= idx < l_eff and page_table[b, idx // 64] % world == rank:
                    out[b, s, k] = idx
    return out


def local_page_table(page_table, world, rank):
    """The rank-local page table written out: p // world where the rank owns
    physical page p, -1 elsewhere (and for negative entries)."""
    pt = np.asarray(page_table)
    return np.where((pt >= 0) & (pt % world == rank), pt // world, -1).astype(np.int32)


def local_slots(slots, world, rank):
    """Rank-local cache-write slots written out: (page // world) * 64 +
    slot % 64 on the page's owner, -1 elsewhere."""
    out = np.full(len(slots), -1, dtype=np.int64)
    for i, sl in enumerate(np.asarray(slots).tolist()):
        if sl >= 0 and (sl // 64) % world == rank:
            out[i] = (sl // 64 // world) * 64 + sl % 64
    return out


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from bit_kv_cache_nvfp4_gb300 import gather_partials
    from bit_kv_cache_nvfp4_gb300 import workloads as wl
    from gpu_common import bits
    w = wl.make_workload("tiny", seed=0)
    qids = [(b, s) for b in range(w.B) for s in range(w.Sq)]
    pt_c, pages, ns = wl.compact_pool_plan(w, qids)
    ids, cslots = wl.compact_pool_tokens(w, pages, qids)
    lat, rope = wl.token_rows(w, ids)
    pool = np.zeros((max(ns, 64), 352), dtype=np.uint8)
    assert oracle.quantize_write(bits(lat), bits(rope), cslots.numpy(), pool) == oracle.OK
    q = bits(wl.queries(w))
    # this rank's own pool: the tokens of every page it owns, at local slots
    # (ownership follows the workload's own, physical, page table)
    num_pages = w.num_slots // 64
    n_local = (num_pages - rank + world - 1) // world
    L = int(w.seq_lens[0])
    pos = torch.arange(L, dtype=torch.int64)
    lslots = local_slots(wl.token_slots(w, 0, pos).numpy(), world, rank)
    keep = lslots >= 0
    llat, lrope = wl.token_rows(w, pos[torch.from_numpy(keep)] + int(w.token_offset[0]))
    local_pool = np.zeros((n_local * 64, 352), dtype=np.uint8)
    assert oracle.quantize_write(bits(llat), bits(lrope), lslots[keep], local_pool) == oracle.OK
    mine = owned_topk(w.topk.numpy(), w.page_table.numpy(), w.seq_lens.numpy(), world, rank)
    st, o, lse = oracle.sparse_mla_decode(q, local_pool,
                                          local_page_table(w.page_table.numpy(), world, rank),
                                          mine, w.seq_lens.numpy(), w.sm_scale)
    assert st == oracle.OK
    out[rank, 4] = float(n_local)
    out[rank, 5] = float(num_pages)
    o_parts, lse_parts = gather_partials(torch.from_numpy(o), torch.from_numpy(lse))
    R, n = o_parts.shape[0], lse.size
    m_out, m_lse = oracle.merge(np.ascontiguousarray(o_parts.numpy().reshape(R, n, 512)),
                                np.ascontiguousarray(lse_parts.numpy().reshape(R, n)))
    st, o_all, lse_all = oracle.sparse_mla_decode(q, pool, pt_c.numpy(), w.topk.numpy(),
                                                  w.seq_lens.numpy(), w.sm_scale)
    out[rank, 0] = float(np.abs(m_out.reshape(o_all.shape) - o_all).max())
    out[rank, 1] = float(np.abs(m_lse.reshape(lse_all.shape) - lse_all).max())
    # the ranks' key sets partition the valid keys
    out[rank, 2] = float((mine >= 0).sum())
    out[rank, 3] = float(((w.topk.numpy() >= 0)).sum())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_dcp_exchange_and_merge_gloo(world):
    port = _free_port()
    out = torch.zeros(world, 6, dtype=torch.float64).share_memory_()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    assert torch.all(out[:, 0] <= 1e-5), out[:, 0]       # merged o equals the direct decode
    assert torch.all(out[:, 1] <= 1e-5), out[:, 1]
    assert float(out[:, 2].sum()) == float(out[0, 3])   # every valid key on exactly one rank
    # the local pools partition the pages: each holds about 1/world of them
    assert float(out[:, 4].sum()) == float(out[0, 5])
    assert float(out[:, 4].max()) <= math.ceil(float(out[0, 5]) / world)
