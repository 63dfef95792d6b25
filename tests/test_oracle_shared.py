"""Pins for the oracle's shared expert and its combination with the routed
output (the Cohere2MoE sparse-block listing of "SM10X Command-A-Plus decode
2.3x faster, BCG capture memory -78%": routed + shared, halved under the
'average' strategy).

* a shared expert equal to the only routed expert (one expert, top-1, weight
  one) computes the same FP32 rows as the routed path, which is itself pinned
  to a dense SwiGLU MLP: the sum is exactly twice the routed output, the
  average exactly the routed output;
* an all-zero shared expert adds exactly zero: the sum equals the routed
  output, the average is exactly half of it;
* the shared rows equal a dense SwiGLU MLP on the dequantized operands
  computed here from the quantizer alone.
"""

import numpy as np

from oracle import moe, nvfp4


def _bf16(a):
    return nvfp4.bf16_to_f32(nvfp4.bf16_round(np.asarray(a, dtype=np.float32)))


def _layer(seed, E=1, T=6, H=256, I=64):
    rng = np.random.default_rng(seed)
    x = _bf16(rng.standard_normal((T, H)))
    wg = _bf16(rng.standard_normal((H, E)) * 0.02)
    w13 = moe.quantize_weights(_bf16(rng.standard_normal((E, 2 * I, H)) * 0.02))
    w2 = moe.quantize_weights(_bf16(rng.standard_normal((E, H, I)) * 0.02))
    return x, wg, w13, w2


def test_shared_equal_to_routed_doubles_or_keeps():
    x, wg, w13, w2 = _layer(31)
    base = moe.moe_forward(x, wg, w13, w2, 1)
    summed = moe.moe_forward(x, wg, w13, w2, 1, shared=(w13, w2))
    avg = moe.moe_forward(x, wg, w13, w2, 1, shared=(w13, w2), shared_average=True)
    assert np.array_equal(summed.out_f32, (base.out_f32 * np.float32(2)).astype(np.float32))
    assert np.array_equal(avg.out_f32, base.out_f32)


def test_zero_shared_expert_adds_nothing():
    x, wg, w13, w2 = _layer(32, E=4)
    H = x.shape[1]
    zero13 = moe.quantize_weights(np.zeros((1, 2 * 64, H), np.float32))
    zero2 = moe.quantize_weights(np.zeros((1, H, 64), np.float32))
    base = moe.moe_forward(x, wg, w13, w2, 2)
    summed = moe.moe_forward(x, wg, w13, w2, 2, shared=(zero13, zero2))
    avg = moe.moe_forward(x, wg, w13, w2, 2, shared=(zero13, zero2), shared_average=True)
    assert np.array_equal(summed.out_f32, base.out_f32)
    assert np.array_equal(avg.out_f32, (base.out_f32 * np.float32(0.5)).astype(np.float32))


def test_shared_rows_are_a_dense_swiglu_mlp():
    x, wg, w13, w2 = _layer(33, E=4)
    _, _, s13, s2 = _layer(34)
    xc, xsf, xgs = nvfp4.quantize_rows(x)
    rows = moe.shared_expert_rows(xc, xsf, xgs, s13, s2)
    xq = nvfp4.dequantize(xc, xsf, xgs)
    W13 = nvfp4.dequantize(s13.codes[0], s13.sf[0], s13.gs[0])
    gu = (xq @ W13.T).astype(np.float32).astype(np.float64)
    I = gu.shape[1] // 2
    h = (gu[:, :I] / (1 + np.exp(-gu[:, :I])) * gu[:, I:]).astype(np.float32)
    hq = nvfp4.dequantize(*nvfp4.quantize_rows(h))
    W2 = nvfp4.dequantize(s2.codes[0], s2.sf[0], s2.gs[0])
    y = (hq @ W2.T).astype(np.float32)
    np.testing.assert_allclose(rows, y, rtol=1e-5, atol=1e-7)
