"""Pins of the oracle's MSE-searched block scale (README "4-bit KV cache",
DeepSeek V4 Pro bullet: "an MSE-searched scale"; the search rule is this
project's reading, written in oracle/kv4ref.h).

Each check compares against something other than the oracle itself:
- a brute force in float64: every candidate scale of the window (decoded by
  PyTorch's float8_e4m3fn), codes by nearest-grid search with ties to even,
  squared error summed in float64.  The oracle's pick must reach the
  smallest error (up to fp32 rounding of near-ties), and its codes must be
  the brute-force codes for the scale it picked;
- the amax/6 quantizer (pinned in test_oracle_codec.py): the searched row
  never reconstructs a block worse than it;
- closed cases: an all-zero block, and a block on the grid of a scale s with
  amax = 6 s, which reconstructs exactly with that scale.
"""
import numpy as np
import torch

import oracle
from test_oracle_codec import E2M1_GRID, bf16_bits, brute_force_encode, e4m3_grid_from_torch

GRID = e4m3_grid_from_torch()                  # E4M3 magnitudes by code 0..126


def _block_values(lat_bits16):
    return torch.from_numpy(lat_bits16.view(np.int16)).view(torch.bfloat16).double().numpy()


def _amax6_code(x):
    amax = np.float32(np.abs(x).max())
    s_f = np.float32(amax / np.float32(6.0))   # IEEE fp32 division
    s_f = min(s_f, np.float32(448.0))          # E4M3 saturates at 448
    return int(torch.tensor([s_f]).to(torch.float8_e4m3fn).view(torch.uint8)[0])


def _brute_force_block(x):
    """(errors by candidate code, codes by candidate) over the window."""
    c0 = _amax6_code(x)
    out = {}
    for c in range(max(0, c0 - 8), min(126, c0 + 1) + 1):
        s = GRID[c]
        if s == 0:
            codes = np.zeros(16, dtype=np.int64)
        else:
            r = (x.astype(np.float32) / np.float32(s)).astype(np.float64)
            codes = brute_force_encode(r, E2M1_GRID, 0x8)
        vals = E2M1_GRID[codes & 7] * np.where(codes & 8, -1.0, 1.0) * s
        out[c] = (float(np.sum((x - vals) ** 2)), codes)
    return out


def _unpack(row, blk):
    return np.array([(row[(16 * blk + j) // 2] >> (4 * ((16 * blk + j) % 2))) & 0xF
                     for j in range(16)])


def test_brute_force_window_search():
    rng = np.random.default_rng(11)
    checked = 0
    improved = 0
    for trial in range(120):
        kind = trial % 3
        scale = 10.0 ** rng.uniform(-2.5, 2.5)
        if kind == 0:
            xs = rng.standard_normal(512)
        elif kind == 1:
            xs = rng.laplace(size=512)
        else:
            xs = rng.standard_normal(512)
            xs[rng.integers(0, 512, 40)] *= 8        # outliers
        lat = bf16_bits((xs * scale).astype(np.float32))
        row = oracle.quantize_row_mse(lat, np.zeros(64, dtype=np.uint16))
        x_all = _block_values(lat)
        for blk in range(32):
            x = x_all[16 * blk:16 * blk + 16]
            cands = _brute_force_block(x)
            best = min(e for e, _ in cands.values())
            c = int(row[256 + blk])
            assert c in cands, (trial, blk, c)
            err, codes = cands[c]
            assert err <= best * (1 + 1e-5) + 1e-300, (trial, blk, c, err, best)
            assert np.array_equal(_unpack(row, blk), codes), (trial, blk)
            if err < cands[_amax6_code(x)][0]:
                improved += 1
            checked += 1
    assert checked == 120 * 32
    assert improved > checked // 10              # the search does change scales


def test_never_worse_than_amax_over_6():
    rng = np.random.default_rng(12)
    for _ in range(60):
        xs = (rng.standard_normal(512) * 10.0 ** rng.uniform(-2, 2)).astype(np.float32)
        lat = bf16_bits(xs)
        x = _block_values(lat)
        d_mse = oracle.dequant_row(oracle.quantize_row_mse(lat, np.zeros(64, np.uint16)))
        d_amx = oracle.dequant_row(oracle.quantize_row(lat, np.zeros(64, np.uint16)))
        e_mse = ((x - d_mse[:512].astype(np.float64)) ** 2).reshape(32, 16).sum(1)
        e_amx = ((x - d_amx[:512].astype(np.float64)) ** 2).reshape(32, 16).sum(1)
        assert np.all(e_mse <= e_amx * (1 + 1e-5) + 1e-300)


def test_zero_block_on_grid_block_and_rope():
    lat = np.zeros(512, dtype=np.uint16)
    rope = bf16_bits(np.linspace(-3, 3, 64).astype(np.float32))
    row = oracle.quantize_row_mse(lat, rope)
    assert not row[:288].any()
    assert np.array_equal(row[288:], oracle.quantize_row(lat, rope)[288:])
    rng = np.random.default_rng(13)
    done = 0
    while done < 100:
        c = int(rng.integers(9, 120))
        s = float(GRID[c])
        mags = E2M1_GRID[rng.integers(0, 8, 16)]
        mags[rng.integers(0, 16)] = 6.0                      # amax = 6 s
        x = mags * np.where(rng.random(16) < 0.5, -1, 1) * s
        lat = np.zeros(512, dtype=np.uint16)
        lat[:16] = bf16_bits(x)
        if not np.array_equal(_block_values(lat[:16]), x):
            continue                                           # not bf16-exact
        row = oracle.quantize_row_mse(lat, np.zeros(64, dtype=np.uint16))
        assert row[256] == c
        assert np.array_equal(oracle.dequant_row(row)[:16].astype(np.float64), x)
        done += 1
