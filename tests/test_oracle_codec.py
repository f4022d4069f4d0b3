"""Pins of the oracle's codecs against things other than the oracle itself.

- hand-worked encodings (tests/golden/minifloat_handworked.txt);
- the E4M3 decoder against PyTorch's float8_e4m3fn dtype (a library routine);
- both encoders against an independent brute-force nearest-value search with
  ties to the even code, over random floats and every grid midpoint;
- the E4M3 encoder against PyTorch's float32 -> float8_e4m3fn conversion;
- exhaustive round trips of every finite code;
- a hand-worked block quantization (tests/golden/quantize_row_handworked.txt),
  the all-zero block, the reconstruction error bound and exact re-encoding of
  on-grid blocks, for the 352-byte row of the numinousmuses
  "inference-optimizations" README, "4-bit KV cache" section.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# E2M1 magnitudes by code 0..7, from the format's definition (1 sign,
# 2 exponent bits with bias 1, 1 mantissa bit).
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e4m3_grid_from_torch():
    """Positive finite E4M3 magnitudes by code 0..126, decoded by PyTorch."""
    codes = torch.arange(0, 127, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def brute_force_encode(x, grid, sign_bit):
    """Nearest grid magnitude, ties to the even code, saturating; sign kept."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    out = np.empty(x.shape, dtype=np.int64)
    for lo in range(0, x.size, 100_000):
        blk = a.ravel()[lo:lo + 100_000]
        d = np.abs(blk[:, None] - grid[None, :])
        best = d.min(axis=1, keepdims=True)
        cand = d == best
        # among the (at most two) nearest codes take the even one
        codes = np.arange(grid.size)
        even = cand & (codes[None, :] % 2 == 0)
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        pick = np.where(blk >= grid[-1], grid.size - 1, pick)   # saturate
        out.ravel()[lo:lo + 100_000] = pick
    return out | np.where(np.signbit(x), sign_bit, 0)


def load_handworked():
    rows = []
    with open(os.path.join(GOLDEN, "minifloat_handworked.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            fmt, val, code = line.split()[:3]
            rows.append((fmt, float(val), int(code, 16)))
    return rows


@pytest.mark.parametrize("fmt,val,code", load_handworked())
def test_handworked_encodings(fmt, val, code):
    enc = oracle.enc_e4m3 if fmt == "e4m3" else oracle.enc_e2m1
    assert enc(np.float32(val)) == code, (fmt, val, hex(code))


def test_e4m3_decode_matches_torch_float8():
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]      # 0x7F/0xFF are NaN
    ref = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.dec_e4m3(c) for c in codes], dtype=np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))  # incl. -0


def test_e2m1_decode_matches_format_table():
    for c in range(16):
        v = E2M1_GRID[c & 7] * (-1.0 if c & 8 else 1.0)
        got = oracle.dec_e2m1(c)
        assert got == v and np.signbit(got) == bool(c & 8)


def test_round_trip_all_finite_codes():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.enc_e4m3(oracle.dec_e4m3(c)) == c, hex(c)
    for c in range(16):
        assert oracle.enc_e2m1(oracle.dec_e2m1(c)) == c, hex(c)


def _adversarial_floats(grid, n_random, rng, scale):
    mids = (grid[1:] + grid[:-1]) / 2
    pts = np.concatenate([grid, mids, np.nextafter(mids.astype(np.float32), 0),
                          np.nextafter(mids.astype(np.float32), np.inf)])
    rnd = rng.standard_normal(n_random) * scale * rng.choice([1e-3, 1e-1, 1, 10], n_random)
    x = np.concatenate([pts, -pts, rnd, grid[-1] * np.array([1.01, 2.0, 1e6])])
    return x.astype(np.float32)


def test_e4m3_encoder_brute_force():
    rng = np.random.default_rng(0)
    grid = e4m3_grid_from_torch()
    x = _adversarial_floats(grid, 1_000_000, rng, 64.0)
    got = oracle.enc_e4m3_array(x)
    ref = brute_force_encode(x, grid, 0x80)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_e4m3_encoder_matches_torch_conversion():
    rng = np.random.default_rng(1)
    grid = e4m3_grid_from_torch()
    x = _adversarial_floats(grid, 1_000_000, rng, 32.0)
    x = x[np.abs(x) < 464.0]             # torch does not saturate beyond 464
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.enc_e4m3_array(x)
    assert np.array_equal(got, ref)


def test_e2m1_encoder_brute_force():
    rng = np.random.default_rng(2)
    x = _adversarial_floats(E2M1_GRID, 1_000_000, rng, 3.0)
    got = oracle.enc_e2m1_array(x)
    ref = brute_force_encode(x, E2M1_GRID, 0x8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def bf16_bits(values):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_quantize_row_handworked_block():
    fields = {}
    with open(os.path.join(GOLDEN, "quantize_row_handworked.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *v = line.split()
            fields[k] = v
    x = [float(v) for v in fields["latent_block0"]]
    lat = np.zeros(512, dtype=np.uint16)
    lat[:16] = bf16_bits(x)
    assert np.array_equal(torch.from_numpy(lat[:16].view(np.int16)).view(torch.bfloat16)
                          .float().numpy(), np.array(x, dtype=np.float32))
    row = oracle.quantize_row(lat, np.zeros(64, dtype=np.uint16))
    assert row[256] == int(fields["scale_byte0"][0], 16)
    assert list(row[:8]) == [int(b, 16) for b in fields["bytes_0_8"]]
    codes = [int(c, 16) for c in fields["codes_block0"]]
    unpacked = [(row[j // 2] >> (4 * (j % 2))) & 0xF for j in range(16)]
    assert unpacked == codes
    assert not row[8:256].any() and not row[257:].any()        # zero blocks, zero rope


def test_zero_block_and_tiny_block():
    lat = np.zeros(512, dtype=np.uint16)
    lat[16:32] = bf16_bits([1e-3] * 16)          # amax/6 below half of 2^-9 -> scale 0
    row = oracle.quantize_row(lat, np.zeros(64, dtype=np.uint16))
    assert not row.any()


def test_reconstruction_error_bound_and_layout():
    rng = np.random.default_rng(3)
    for trial in range(50):
        scale = 10.0 ** rng.uniform(-2, 2)
        xl = (rng.standard_normal(512) * scale).astype(np.float32)
        xr = (rng.standard_normal(64) * scale).astype(np.float32)
        lat, rope = bf16_bits(xl), bf16_bits(xr)
        xl = torch.from_numpy(lat.view(np.int16)).view(torch.bfloat16).double().numpy()
        xr = torch.from_numpy(rope.view(np.int16)).view(torch.bfloat16).double().numpy()
        row = oracle.quantize_row(lat, rope)
        deq = oracle.dequant_row(row).astype(np.float64)
        s = torch.from_numpy(row[256:288].copy()).view(torch.float8_e4m3fn).double().numpy()
        for blk in range(32):
            xb = xl[16 * blk:16 * blk + 16]
            db = deq[16 * blk:16 * blk + 16]
            sb = s[blk]
            if sb == 0:
                assert not db.any()
                continue
            r = np.abs(xb) / sb
            half_step = np.where(r < 2, 0.25, np.where(r < 4, 0.5, 1.0))
            err = np.abs(db - xb)
            bound = np.where(r <= 6, half_step * sb, np.abs(xb) - 6 * sb) * (1 + 1e-6)
            assert np.all(err <= bound + 1e-30), (trial, blk)
        # rope is a direct E4M3 cast: compare with torch's conversion of the bf16 values
        ref = torch.from_numpy(xr.astype(np.float32)).clamp(-448, 448).to(torch.float8_e4m3fn)
        assert np.array_equal(row[288:], ref.view(torch.uint8).numpy())
        # dequant of the rope part is the E4M3 value itself
        assert np.array_equal(deq[512:], ref.double().numpy())


def test_on_grid_block_reencodes_exactly():
    rng = np.random.default_rng(4)
    grid = e4m3_grid_from_torch()
    for _ in range(200):
        s = float(grid[rng.integers(1, 127)])
        mags = E2M1_GRID[rng.integers(0, 8, 16)]
        mags[rng.integers(0, 16)] = 6.0                      # amax = 6 s
        x = mags * np.where(rng.random(16) < 0.5, -1, 1) * s
        if not np.all(np.isfinite(x)) or np.abs(x).max() > 3e38:
            continue
        lat = np.zeros(512, dtype=np.uint16)
        lat[:16] = bf16_bits(x)
        back = torch.from_numpy(lat[:16].view(np.int16)).view(torch.bfloat16).double().numpy()
        if not np.array_equal(back, x):
            continue                                           # not bf16-exact; skip
        row = oracle.quantize_row(lat, np.zeros(64, dtype=np.uint16))
        deq = oracle.dequant_row(row)
        assert np.array_equal(deq[:16].astype(np.float64), x)
        row2 = oracle.quantize_row(bf16_bits(deq[:512]), np.zeros(64, dtype=np.uint16))
        assert np.array_equal(row, row2)
