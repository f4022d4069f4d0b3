"""The seeded input generator: determinism, shapes and index-set structure."""
import numpy as np
import torch

from bit_kv_cache_nvfp4_gb300 import workloads as wl


def test_hash_is_exact_uint32_mix():
    # fmix32 of a few values against a plain Python-integer evaluation
    def ref(x):
        x ^= x >> 16
        x = (x * 0x85EBCA6B) & 0xFFFFFFFF
        x ^= x >> 13
        x = (x * 0xC2B2AE35) & 0xFFFFFFFF
        x ^= x >> 16
        return x
    vals = [0, 1, 2, 0xDEADBEEF, 0xFFFFFFFF, 123456789]
    got = wl.fmix32(torch.tensor(vals, dtype=torch.int64)).tolist()
    assert got == [ref(v) for v in vals]


def test_quantile_tables():
    t = wl.quantile_table("normal", "cpu").double()
    assert t.shape == (65536,)
    assert abs(float(t.mean())) < 1e-3 and abs(float(t.std()) - 1.0) < 2e-3
    assert torch.all(t[1:] >= t[:-1])
    lap = wl.quantile_table("laplace", "cpu").double()
    assert abs(float(lap.abs().mean()) - 1.0) < 2e-3


def test_configs_structure():
    for name in wl.CONFIG_NAMES:
        w = wl.make_workload(name)
        assert w.topk.shape == (w.B, w.Sq, w.K) and w.topk.dtype == torch.int32
        for b in range(w.B):
            L = int(w.seq_lens[b])
            for s in range(w.Sq):
                row = w.topk[b, s]
                assert torch.unique(row).numel() == w.K
                assert int(row.min()) >= 0 and int(row.max()) < L
        # every position of every request has a distinct physical page
        used = torch.cat([w.page_table[b, :(int(w.seq_lens[b]) + 63) // 64]
                          for b in range(w.B)])
        assert torch.unique(used).numel() == used.numel()
        assert int(used.max()) * 64 < w.num_slots
    long = wl.make_workload("long")
    recent = (long.topk >= 204800 - 4096).sum(-1)
    assert torch.all(recent == 1024)
    sv = wl.make_workload("specverify")
    shared = set(sv.topk[0, 0].tolist()) & set(sv.topk[0, 3].tolist())
    assert len(shared) == 1024 + 4


def test_generation_is_deterministic_and_device_independent():
    w = wl.make_workload("tiny")
    a1, r1 = wl.token_rows(w, torch.arange(100))
    a2, r2 = wl.token_rows(w, torch.arange(100))
    assert torch.equal(a1.view(torch.int16), a2.view(torch.int16))
    w2 = wl.make_workload("tiny")
    assert torch.equal(w.topk, w2.topk) and torch.equal(w.page_table, w2.page_table)
    # a row drawn alone equals the same row drawn in a batch
    a3, _ = wl.token_rows(w, torch.tensor([57]))
    assert torch.equal(a3[0].view(torch.int16), a1[57].view(torch.int16))
    # outlier channels are 8x
    big = wl.token_rows(w, torch.arange(4000))[0].float()
    sd = big.std(0)
    ch = w.outlier_channels
    assert torch.all(sd[ch] > 6) and float(np.median(sd.numpy())) < 1.2


def test_sweep_kinds():
    for kind in wl.SWEEP_KINDS:
        lat, rope = wl.sweep_rows(kind, 0, 10, 256)
        assert lat.shape == (256, 512) and rope.shape == (256, 64)
        assert torch.isfinite(lat.float()).all()
    lat, _ = wl.sweep_rows("zeroblocks", 0, 0, 4096)
    zero = (lat.view(4096, 32, 16).float().abs().amax(-1) == 0).float().mean()
    assert 0.2 < float(zero) < 0.3
