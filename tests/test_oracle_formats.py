"""Pins for the oracle's number formats (E2M1, E4M3, bf16).

Each check ties ``oracle.nvfp4`` to something outside it: values written out
by hand from the bit-field definitions, torch's own float8_e4m3fn and
bfloat16 conversions, and an independent formula for round-to-nearest-even.
"""

import math

import numpy as np
import pytest
import torch

from oracle import nvfp4


def test_e2m1_table_by_hand():
    # sign | exponent(2) | mantissa(1), bias 1, exponent 0 subnormal.
    expect = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert nvfp4.E2M1_VALUES[:8].tolist() == expect
    assert nvfp4.E2M1_VALUES[8:].tolist() == [-v for v in expect]
    assert math.copysign(1.0, nvfp4.E2M1_VALUES[8]) == -1.0


def test_e4m3_table_spot_values():
    v = nvfp4.E4M3_VALUES
    assert v[0x00] == 0.0
    assert v[0x01] == 2.0 ** -9            # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert v[0x08] == 2.0 ** -6            # smallest normal
    assert v[0x38] == 1.0
    assert v[0x40] == 2.0
    assert v[0x61] == 36.0
    assert v[0x7E] == 448.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0xFE] == -448.0
    finite = v[:127]
    assert np.all(np.diff(finite) > 0)     # codes 0..126 ascending


def _e4m3_probe_values():
    grid = nvfp4.E4M3_VALUES[:127].astype(np.float32)
    mids = ((grid[:-1].astype(np.float64) + grid[1:]) / 2).astype(np.float32)
    up = np.nextafter(mids, np.float32(np.inf))
    down = np.nextafter(mids, np.float32(0))
    rng = np.random.default_rng(7)
    rand = np.exp2(rng.uniform(-14, math.log2(464.0), 200_000)).astype(np.float32)
    tiny = np.float32([2.0 ** -10, 2.0 ** -11, 1e-30, 0.0, 3 * 2.0 ** -11])
    vals = np.concatenate([grid, mids, up, down, rand, tiny, np.float32([464.0, 460.0])])
    return vals[vals <= 464.0]


def test_e4m3_encode_matches_torch_float8():
    # torch rounds to nearest even; it saturates only up to 464 (beyond that it
    # makes NaN), so the comparison stays at or below 464.
    vals = _e4m3_probe_values()
    vals = np.concatenate([vals, -vals])
    ours = nvfp4.e4m3_encode(vals)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first {vals[bad[:5]]} -> {ours[bad[:5]]} vs {ref[bad[:5]]}"


def test_e4m3_encode_saturates():
    big = np.float32([448.0, 449.0, 480.0, 1e6, 3e38, np.inf])
    assert (nvfp4.e4m3_encode(big) == 0x7E).all()
    assert (nvfp4.e4m3_encode(-big) == 0xFE).all()


def _e2m1_rne_formula(a: np.ndarray) -> np.ndarray:
    """Round |a| to E2M1 by the generic binary rounding formula: spacing 0.5
    below 2 (subnormals and the first binade), 2^(e-1) above; numpy's rint is
    round-half-even; then saturate at 6."""
    a = np.abs(a.astype(np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    spacing = np.where(a < 2.0, 0.5, np.exp2(e - 1))
    r = np.rint(a / spacing) * spacing
    return np.minimum(r, 6.0)


def test_e2m1_ties_by_hand():
    cases = [(0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6),
             (5.0, 0x6), (6.5, 0x7), (7.0, 0x7), (100.0, 0x7), (0.2499, 0x0), (0.2501, 0x1),
             (4.99, 0x6), (5.01, 0x7), (-0.1, 0x8), (-0.0, 0x8), (0.0, 0x0), (-3.5, 0xE),
             (-5.0, 0xE)]
    got = nvfp4.e2m1_encode(np.float32([v for v, _ in cases]))
    assert got.tolist() == [c for _, c in cases]


def test_e2m1_encode_matches_formula_dense():
    # float32 bit patterns in [0, 8] at a stride of 997, plus +-4 ulps around
    # each tie point of the grid
    lo = np.float32(0).view(np.uint32)
    hi = np.float32(8).view(np.uint32)
    pats = np.arange(lo, hi, 997, dtype=np.uint64).astype(np.uint32)
    vals = pats.view(np.float32)
    ties = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    near = [ties]
    for _ in range(4):
        near.append(np.nextafter(near[-1], np.float32(np.inf)))
    down = [ties]
    for _ in range(4):
        down.append(np.nextafter(down[-1], np.float32(0)))
    vals = np.concatenate([vals] + near + down)
    vals = np.concatenate([vals, -vals])
    codes = nvfp4.e2m1_encode(vals)
    decoded = np.abs(nvfp4.e2m1_decode(codes))
    assert np.array_equal(decoded, _e2m1_rne_formula(vals))
    neg = np.signbit(vals)
    assert np.array_equal((codes >> 3).astype(bool), neg)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100_000) * np.exp2(rng.uniform(-40, 40, 100_000))).astype(np.float32)
    # exact ties: bit 15 set, bits 0..14 clear
    ties = (rng.integers(0, 2 ** 31, 1000, dtype=np.uint64).astype(np.uint32) & 0xFFFF0000) | 0x8000
    x = np.concatenate([x, ties.view(np.float32)[np.isfinite(ties.view(np.float32))]])
    ours = nvfp4.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_pack_unpack_roundtrip():
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 16, (5, 64), dtype=np.uint8)
    packed = nvfp4.pack_e2m1(codes)
    assert packed.shape == (5, 32)
    assert packed[0, 0] == (codes[0, 0] | (codes[0, 1] << 4))
    assert np.array_equal(nvfp4.unpack_e2m1(packed), codes)


@pytest.mark.parametrize("amax,gs", [(6.0, 448.0), (12.0, 224.0), (1024.0, 2.625), (0.0, 1.0), (2688.0, 1.0)])
def test_global_scale_closed_form(amax, gs):
    assert nvfp4.global_scale(np.float32([amax]))[0] == np.float32(gs)


def test_global_scale_overflow_clamps():
    g = nvfp4.global_scale(np.float32([1e-37]))
    assert g[0] == np.finfo(np.float32).max
