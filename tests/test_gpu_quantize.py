"""GPU parity of kv4_quantize_write against the CPU oracle: bit-exact bytes.

The 1,048,576-token sweeps (N(0,1), Laplace(0,1), 25 % zero blocks, and
round-half-even tie blocks) are written on the GPU in one launch and compared
in full: oracle workers (a spawn process pool, each single-threaded) rebuild
the same seeded inputs from the generator and hash their rows chunk by chunk.
"""
import hashlib
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

from bit_kv_cache_nvfp4_gb300 import workloads as wl
from gpu_common import bits, need_gpu, gpu_pool, workload

pytestmark = pytest.mark.gpu

N_SWEEP = 1 << 20
CHUNK = 1 << 15


def _slot_of(t: np.ndarray) -> np.ndarray:
    """A fixed permutation of [0, N_SWEEP) (odd multiplier mod 2^20)."""
    return (t.astype(np.int64) * 7919) % N_SWEEP


def _oracle_chunk_digest(args):
    kind, first, n = args
    torch.set_num_threads(1)
    import oracle
    lat, rope = wl.sweep_rows(kind, 0, first, n)
    pool = np.zeros((n, 352), dtype=np.uint8)
    st = oracle.quantize_write(bits(lat), bits(rope), np.arange(n, dtype=np.int64), pool)
    assert st == 0
    return first, hashlib.sha256(pool.tobytes()).hexdigest()


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = mp.get_context("spawn").Pool(max(1, min(16, os.cpu_count() or 1)))
    return _POOL


@pytest.mark.parametrize("kind", wl.SWEEP_KINDS)
def test_quantize_sweep_bit_exact(kind):
    need_gpu()
    import bit_kv_cache_nvfp4_gb300 as kv
    dev = torch.device("cuda")
    lat, rope = wl.sweep_rows(kind, 0, 0, N_SWEEP, device=dev)
    tokens = np.arange(N_SWEEP)
    slots = torch.from_numpy(_slot_of(tokens)).to(dev)
    pool = torch.zeros((N_SWEEP, 352), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kv.quantize_write(lat, rope, slots, pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    host = pool.cpu().numpy()
    rows = host[_slot_of(tokens)]                       # back to token order
    jobs = [(kind, f, min(CHUNK, N_SWEEP - f)) for f in range(0, N_SWEEP, CHUNK)]
    for first, digest in _pool().imap_unordered(_oracle_chunk_digest, jobs):
        n = min(CHUNK, N_SWEEP - first)
        got = hashlib.sha256(rows[first:first + n].tobytes()).hexdigest()
        if got != digest:
            import oracle
            lat_c, rope_c = wl.sweep_rows(kind, 0, first, n)
            ref = np.zeros((n, 352), dtype=np.uint8)
            oracle.quantize_write(bits(lat_c), bits(rope_c), np.arange(n, dtype=np.int64), ref)
            bad = np.nonzero((ref != rows[first:first + n]).any(1))[0]
            i = int(bad[0])
            col = int(np.nonzero(ref[i] != rows[first + i])[0][0])
            pytest.fail(f"{kind}: {bad.size} rows differ in chunk {first}; first token "
                        f"{first + i} byte {col}: gpu {rows[first + i, col]:#x} "
                        f"oracle {ref[i, col]:#x}")


def test_skip_and_bad_slots():
    need_gpu()
    import bit_kv_cache_nvfp4_gb300 as kv
    import oracle
    dev = torch.device("cuda")
    n = 1000
    lat, rope = wl.sweep_rows("normal", 3, 0, n, device=dev)
    slots = torch.arange(n, dtype=torch.int64)
    slots[::7] = -1
    slots[5] = n + 10                                   # past the pool: skipped + flagged
    pool = torch.zeros((n, 352), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kv.quantize_write(lat, rope, slots.to(dev), pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) & kv.DEV_BAD_SLOT
    ref = np.zeros((n, 352), dtype=np.uint8)
    st = oracle.quantize_write(bits(lat), bits(rope), slots.numpy(), ref)
    assert st == oracle.ERR_SLOT
    assert np.array_equal(pool.cpu().numpy(), ref)


def test_strided_inputs_and_per_step_write():
    """The decode workload's per-step write: 16 new tokens (one per request),
    taken from wider strided buffers, equal the oracle rows; and the GPU-built
    pool of that workload matches the oracle at sampled slots."""
    need_gpu()
    import bit_kv_cache_nvfp4_gb300 as kv
    import oracle
    dev = torch.device("cuda")
    w = workload("decode")
    lat, rope, slots = wl.newest_tokens(w, dev)
    wide_lat = torch.zeros((lat.shape[0], 640), dtype=torch.bfloat16, device=dev)
    wide_rope = torch.zeros((rope.shape[0], 72), dtype=torch.bfloat16, device=dev)
    wide_lat[:, :512] = lat
    wide_rope[:, :64] = rope
    pool = gpu_pool(w).clone()
    pool[slots] = 0
    kv.quantize_write(wide_lat[:, :512], wide_rope[:, :64], slots, pool)
    torch.cuda.synchronize()
    got = pool[slots].cpu().numpy()
    for i in range(lat.shape[0]):
        ref = oracle.quantize_row(bits(lat[i]), bits(rope[i]))
        assert np.array_equal(got[i], ref), i
    # sampled rows of the whole pool
    g = torch.Generator().manual_seed(5)
    host_pool = gpu_pool(w)
    for b in range(w.B):
        pos = torch.randint(0, int(w.seq_lens[b]), (8,), generator=g)
        ids = pos + int(w.token_offset[b])
        l2, r2 = wl.token_rows(w, ids)
        sl = wl.token_slots(w, b, pos)
        rows = host_pool[sl.to(dev)].cpu().numpy()
        for i in range(8):
            assert np.array_equal(rows[i], oracle.quantize_row(bits(l2[i]), bits(r2[i])))
