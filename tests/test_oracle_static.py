"""Pins of the oracle's per-tensor static activation-scale contract (the
contract "CuTe DSL backend gets per-token NVFP4 online quantization and
reload" keeps apart from the per-token one, Summary and Implementation
item 2): calibrated global scales are given instead of derived per token and
per expanded row.

* a hand-derived worked example with saturation and a rounding tie;
* power-of-two invariance (exact scaling);
* reduction to the per-token path: one token whose static scales equal its
  own per-token scales gives the per-token forward bit for bit (a dropped or
  misindexed scale anywhere in the path fails it).
"""

import glob
import os

import numpy as np

import synthetic
from oracle import moe as omoe
from oracle import nvfp4

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(path):
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.split()
    return out


def test_static_worked_example():
    paths = sorted(glob.glob(os.path.join(GOLDEN, "static_ex*.txt")))
    assert paths
    for path in paths:
        fx = _load(path)
        x = np.float32([float(v) for v in fx["x"]])
        assert np.array_equal(nvfp4.bf16_to_f32(nvfp4.bf16_round(x)), x), path
        codes, sf, gs = nvfp4.quantize_rows_static(x[None, :], np.float32(float(fx["gs"][0])))
        assert sf[0].tolist() == [int(b, 16) for b in fx["sf"]], path
        assert codes[0].tolist() == [int(c, 16) for c in fx["codes"]], path
        assert nvfp4.pack_e2m1(codes)[0].tolist() == [int(b, 16) for b in fx["packed"]], path
        deq = nvfp4.dequantize(codes, sf, gs)[0]
        np.testing.assert_allclose(deq, [float(v) for v in fx["dequant"]], rtol=1e-12, atol=0)


def test_static_power_of_two_invariance():
    rng = np.random.default_rng(3)
    x = nvfp4.bf16_to_f32(nvfp4.bf16_round(rng.standard_normal((4, 64)).astype(np.float32)))
    c1, s1, _ = nvfp4.quantize_rows_static(x, np.float32(300.0))
    c2, s2, _ = nvfp4.quantize_rows_static(x * np.float32(8.0), np.float32(300.0 / 8.0))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def _tiny():
    wl = synthetic.make_workload("c0_tiny")
    x = omoe.as_f32(wl.x)
    wg = omoe.as_f32(wl.gate_w)
    w13 = omoe.quantize_weights(omoe.as_f32(wl.w13))
    w2 = omoe.quantize_weights(omoe.as_f32(wl.w2))
    return wl, x, wg, w13, w2


def test_static_reduces_to_per_token_for_one_token():
    wl, x, wg, w13, w2 = _tiny()
    K, E = wl.shape.K, wl.shape.E
    dyn = omoe.moe_forward(x[:1], wg, w13, w2, K)
    h_gs = np.ones(E, np.float32)
    for j in range(K):
        h_gs[dyn.ids[0, j]] = dyn.h_gs[(0, j)]
    sta = omoe.moe_forward(x[:1], wg, w13, w2, K, static_scales=(dyn.x_gs[0], h_gs))
    assert np.array_equal(sta.x_codes, dyn.x_codes) and np.array_equal(sta.x_sf, dyn.x_sf)
    assert np.array_equal(sta.out_bits, dyn.out_bits)
    # and the forward does use them: an h scale 64x too large saturates the
    # intermediate's blocks and changes the output
    sat = omoe.moe_forward(x[:1], wg, w13, w2, K, static_scales=(dyn.x_gs[0], h_gs * np.float32(64)))
    assert not np.array_equal(sat.out_bits, dyn.out_bits)

