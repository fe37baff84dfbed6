"""Pins for the oracle's element formats, against the format specifications (golden
tables), brute force and an independent library (torch's float32 -> bfloat16 cast,
mpmath)."""
import numpy as np
import pytest
import torch

from conftest import golden_path
from oracle import formats as F


def _table(name):
    rows = []
    for line in open(golden_path(name)):
        line = line.strip()
        if line and not line.startswith("#"):
            a, b = line.split()
            rows.append((a, b))
    return rows


def test_e2m1_code_table_matches_spec():
    for code, val in _table("e2m1_codes.txt"):
        got = F.e2m1_decode(np.array([int(code)]))[0]
        assert got == float(val) and np.signbit(got) == val.startswith("-"), (code, got, val)


def test_e4m3_codes_match_spec():
    for code, val in _table("e4m3_codes.txt"):
        got = F.e4m3_decode(np.array([int(code, 16)]))[0]
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val) and np.signbit(got) == val.startswith("-"), (code, got, val)


def test_e4m3_monotone_and_symmetric():
    pos = F.e4m3_decode(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0)                         # strictly increasing codes
    neg = F.e4m3_decode(np.arange(0x80, 0xFF))
    assert np.array_equal(-pos, neg)


def _brute_nearest(values, grid_vals, grid_codes, x):
    """Nearest grid value by exhaustive distance, ties to the even code."""
    d = np.abs(x[:, None] - grid_vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = np.where(d == best, grid_codes[None, :], 1 << 30)
    even = np.where(cand % 2 == 0, cand, 1 << 30).min(axis=1)
    anyc = cand.min(axis=1)
    return np.where(even < (1 << 30), even, anyc)


def test_e2m1_rne_exhaustive_over_bf16():
    """All 65,536 BF16 patterns (finite ones) at unit scale against brute force."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = F.bf16_to_f32(bits)
    x = x[np.isfinite(x)]
    codes = F.e2m1_encode_rne(x)
    a = np.abs(x).astype(np.float64)
    grid = F.E2M1_MAGNITUDES.copy()
    mag_code = _brute_nearest(None, grid, np.arange(8), np.minimum(a, 6.0))
    sign = (x < 0) & (mag_code != 0)
    expect = (mag_code | (sign.astype(np.int64) << 3)).astype(np.uint8)
    assert np.array_equal(codes, expect)


def test_e2m1_rne_ties():
    v = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -5.0, 6.5, -100.0, -0.1, -0.0], np.float32)
    expect = [0, 2, 2, 4, 4, 6, 6, 0xE, 7, 0xF, 0, 0]
    assert list(F.e2m1_encode_rne(v)) == expect


def test_e4m3_encode_brute_force():
    """Every finite code's value, every midpoint, and their float32 neighbours."""
    pos = F.e4m3_decode(np.arange(0x7F))
    mids = (pos[1:] + pos[:-1]) / 2
    base = np.concatenate([pos, mids, [448.0, 460.0, 464.0, 500.0, 1e6, 1e-30, 2.0 ** -10]])
    b32 = base.astype(np.float32)
    xs = np.concatenate([b32, np.nextafter(b32, np.float32(0)), np.nextafter(b32, np.float32(np.inf))])
    xs = xs[xs >= 0]
    got = F.e4m3_encode_rne_satfinite(xs)
    expect = _brute_nearest(None, pos, np.arange(0x7F), np.minimum(xs.astype(np.float64), 448.0))
    assert np.array_equal(got, expect.astype(np.uint8))


def test_bf16_round_matches_torch_on_float32():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-40, 38, 100000),
                        [0.0, -0.0, 1e-45, -1e-45, 3.3e38, -3.39e38, 1.17e-38]]).astype(np.float32)
    ours = F.bf16_round(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_round_from_float64_single_rounding():
    """A float64 value just above a BF16 midpoint must round up even where a float32
    intermediate would land exactly on the midpoint (checked with mpmath)."""
    mpmath = pytest.importorskip("mpmath")
    mid = 1.0 + 2.0 ** -8                      # midpoint between 1 and 1 + 2^-7
    vals = np.array([mid + 2.0 ** -40, mid - 2.0 ** -40, mid, 1.0 + 3 * 2.0 ** -8])
    got = F.bf16_round(vals)
    for v, g in zip(vals, got):
        f32 = np.float32(v)
        b = (f32.view(np.uint32) >> 16).astype(np.uint16)
        cands = [b - 1, b, b + 1, b + 2]
        cv = [float(F.bf16_to_f32(np.array([c], np.uint16))[0]) for c in cands]
        d = [abs(mpmath.mpf(v) - mpmath.mpf(c)) for c in cv]
        best = min(d)
        winners = [c for c, di in zip(cands, d) if di == best]
        even = [c for c in winners if c % 2 == 0]
        assert g == (even[0] if even else winners[0])


def test_pack_roundtrip_and_nibble_order():
    codes = np.array([[1, 2, 3, 4]], np.uint8)
    p = F.pack_e2m1(codes)
    assert list(p[0]) == [0x21, 0x43]
    assert np.array_equal(F.unpack_e2m1(p), codes)


def test_sf_swizzle_layout_is_a_bijection_with_known_offsets():
    rows, cols = 256, 8
    sf = np.arange(rows * cols, dtype=np.int64).reshape(rows, cols) % 251
    buf = F.sf_swizzle(sf.astype(np.uint8))
    assert buf.size == 2 * 2 * 512
    assert np.array_equal(F.sf_unswizzle(buf, rows, cols), sf.astype(np.uint8))
    offs = F.sf_swizzle_offset(*np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij"), cols)
    assert np.unique(offs).size == rows * cols
    # hand-computed positions: (row, col) -> byte
    known = {(0, 0): 0, (0, 3): 3, (1, 0): 16, (31, 0): 496, (32, 0): 4, (96, 1): 13,
             (0, 4): 512, (127, 7): 512 + 31 * 16 + 12 + 3, (128, 0): 1024, (200, 5): 1024 + 512 + (200 % 32) * 16 + 2 * 4 + 1}
    for (r, c), o in known.items():
        assert F.sf_swizzle_offset(r, c, cols) == o, (r, c)
