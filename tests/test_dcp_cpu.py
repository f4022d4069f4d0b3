"""Decode-context parallelism on CPU (gloo, world size 2 and 3): every rank
takes the keys on its pages (physical page p % world == rank), computes its
partial (o, lse) with the oracle, the ranks exchange them with the library's
gather_partials over torch.distributed, and the oracle's log-sum-exp merge of
the gathered partials must equal the oracle's decode over all keys.  This
covers the multi-rank exchange and the ownership partition; the GPU kernels
of the same steps are covered by tests/test_gpu_dcp.py on one GPU."""
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
    # ownership follows the workload's own (physical) page table
    mine = owned_topk(w.topk.numpy(), w.page_table.numpy(), w.seq_lens.numpy(), world, rank)
    st, o, lse = oracle.sparse_mla_decode(q, pool, pt_c.numpy(), mine, w.seq_lens.numpy(),
                                          w.sm_scale)
    assert st == oracle.OK
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
    out = torch.zeros(world, 4, dtype=torch.float64).share_memory_()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    assert torch.all(out[:, 0] <= 1e-5), out[:, 0]       # merged o equals the direct decode
    assert torch.all(out[:, 1] <= 1e-5), out[:, 1]
    assert float(out[:, 2].sum()) == float(out[0, 3])   # every valid key on exactly one rank
