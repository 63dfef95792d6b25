"""Pins for the oracle's per-token / per-expert NVFP4 quantizer.

* hand-derived worked examples in ``tests/golden/quant_ex*.txt``;
* invariants that hold for any correct implementation of the stated rules:
  power-of-two scaling, zero rows, the dequantization error bound, the
  saturation bound, and independence of rows.
"""

import glob
import os

import numpy as np
import pytest

from oracle import nvfp4


def _load_fixture(path):
    d = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            d[key.strip()] = val.split()
    return d


def _fixtures(golden_dir):
    return sorted(glob.glob(os.path.join(golden_dir, "quant_ex*.txt")))


def test_fixtures_present(golden_dir):
    assert len(_fixtures(golden_dir)) >= 5


@pytest.mark.parametrize("idx", range(5))
def test_worked_example(golden_dir, idx):
    path = _fixtures(golden_dir)[idx]
    fx = _load_fixture(path)
    x = np.float32([float(v) for v in fx["x"]])
    # the inputs are exact bf16 values
    assert np.array_equal(nvfp4.bf16_to_f32(nvfp4.bf16_round(x)), x), path
    codes, sf, gs = nvfp4.quantize_rows(x[None, :])
    assert gs[0] == np.float32(float(fx["gs"][0])), path
    assert sf[0].tolist() == [int(b, 16) for b in fx["sf"]], path
    assert codes[0].tolist() == [int(c, 16) for c in fx["codes"]], path
    assert nvfp4.pack_e2m1(codes)[0].tolist() == [int(b, 16) for b in fx["packed"]], path
    if "dequant" in fx:
        deq = nvfp4.dequantize(codes, sf, gs)[0]
        np.testing.assert_allclose(deq, [float(v) for v in fx["dequant"]], rtol=1e-12, atol=0)


def _random_rows(rng, rows, K):
    scale = np.exp2(rng.uniform(-10, 10, (rows, 1)))
    x = rng.standard_normal((rows, K)) * scale
    x[0, :] = 0.0                                    # a zero row
    x[1, 16:32] = 0.0                                # a zero block
    return nvfp4.bf16_to_f32(nvfp4.bf16_round(x.astype(np.float32)))


def test_power_of_two_scaling_invariance():
    rng = np.random.default_rng(1)
    x = _random_rows(rng, 64, 256)
    codes, sf, gs = nvfp4.quantize_rows(x)
    for k in (-12, -3, -1, 1, 5, 20):
        c2, s2, g2 = nvfp4.quantize_rows((x * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(c2, codes)
        assert np.array_equal(s2, sf)
        nz = np.abs(x).max(axis=1) > 0
        assert np.array_equal(g2[nz], (gs[nz] * np.float32(2.0 ** -k)).astype(np.float32))


def test_zero_row_and_zero_block():
    rng = np.random.default_rng(2)
    x = _random_rows(rng, 4, 64)
    codes, sf, gs = nvfp4.quantize_rows(x)
    assert gs[0] == 1.0 and not sf[0].any() and not codes[0].any()
    assert sf[1, 1] == 0 and not codes[1, 16:32].any()


def test_dequant_error_and_saturation_bounds():
    rng = np.random.default_rng(4)
    x = _random_rows(rng, 256, 512)
    codes, sf, gs = nvfp4.quantize_rows(x)
    xd = nvfp4.dequantize(codes, sf, gs)
    blocks = np.abs(x.astype(np.float64)).reshape(256, -1, 16)
    amax_b = blocks.max(axis=2)
    sfv = nvfp4.e4m3_decode(sf)
    step = sfv / gs[:, None].astype(np.float64)        # value of one unit of the E2M1 grid
    err = np.abs(xd - x).reshape(256, -1, 16)
    # |code - x*q| is at most 1 grid unit (half the widest gap, or the
    # saturation excess); each block's error is at most one unit of its scale
    assert np.all(err <= step[:, :, None] * (1 + 1e-6))
    # the block scale rounds up by at most 2^-4 relative, so |xd| <= amax_b (1 + 2^-4)
    assert np.all(np.abs(xd).reshape(256, -1, 16).max(axis=2) <= amax_b * (1 + 2.0 ** -4) * (1 + 1e-6))
    # global relative error of NVFP4 on gaussian rows is a few percent
    rel = np.linalg.norm(xd[2:] - x[2:]) / np.linalg.norm(x[2:])
    assert 0.02 < rel < 0.15


def test_rows_are_independent():
    rng = np.random.default_rng(5)
    x = _random_rows(rng, 32, 128)
    full = nvfp4.quantize_rows(x)
    for r in (0, 7, 31):
        one = nvfp4.quantize_rows(x[r:r + 1])
        for a, b in zip(full, one):
            assert np.array_equal(a[r:r + 1] if a.ndim > 1 else a[r:r + 1], b)


def test_tensor_scale_matches_row_rule_on_a_single_row():
    rng = np.random.default_rng(6)
    w = _random_rows(rng, 3, 64)[2:3]
    c1, s1, g1 = nvfp4.quantize_tensor(w)
    c2, s2, g2 = nvfp4.quantize_rows(w)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2) and g1 == g2[0]


def test_tensor_scale_uses_whole_matrix_amax():
    w = np.zeros((4, 32), np.float32)
    w[0, 0] = 6.0
    w[3, 5] = 0.75
    codes, sf, gs = nvfp4.quantize_tensor(w)
    assert gs == np.float32(448.0)
    # row 3: block amax 0.75 -> sf32 = 0.75*448/6 = 56 = 1.75*2^5 -> E4M3 0x66, q = 8, v = 6
    assert sf[3, 0] == 0x66 and codes[3, 5] == 0x7
