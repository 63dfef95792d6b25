"""Pins for the oracle's whole forward (expert GEMMs, SwiGLU, requantization,
finalize).

* brute force: every operand fully dequantized, each output an exactly summed
  FP64 dot product (math.fsum), token by token - a different route from the
  oracle's grouped FP64 matmuls with the scales applied afterwards;
* closed forms: inputs on the FP4 grid with unit scales make the GEMM an exact
  integer matmul; one expert with top-1 reduces the layer to a dense SwiGLU
  MLP; zero tokens give exactly zero rows;
* the FP32 finalize order, by hand;
* the quantized layer stays close to the unquantized FP64 layer.
"""

import math

import numpy as np
import pytest

import synthetic
from oracle import moe, nvfp4


def _bf16(a):
    return nvfp4.bf16_to_f32(nvfp4.bf16_round(np.asarray(a, dtype=np.float32)))


def _tiny(seed=0, T=None, name="c0_tiny"):
    wl = synthetic.make_workload(name, T=T, seed=seed)
    x = moe.as_f32(wl.x)
    wg = moe.as_f32(wl.gate_w)
    w13 = moe.quantize_weights(moe.as_f32(wl.w13))
    w2 = moe.quantize_weights(moe.as_f32(wl.w2))
    bias = None if wl.bias is None else wl.bias.numpy()
    return wl, x, wg, w13, w2, bias


def _fsum_matvec(W, v):
    return np.array([math.fsum(W[n] * v) for n in range(W.shape[0])])


def test_brute_force_tiny():
    wl, x, wg, w13, w2, _ = _tiny()
    K = wl.shape.K
    res = moe.moe_forward(x, wg, w13, w2, K)
    T, H = x.shape
    I = wl.shape.I
    xq = nvfp4.dequantize(res.x_codes, res.x_sf, res.x_gs)          # [T, H] f64, /gs applied
    out = np.zeros((T, H), np.float32)
    for t in range(T):
        acc = None
        for j in range(K):
            e = int(res.ids[t, j])
            W13 = nvfp4.dequantize(w13.codes[e], w13.sf[e], w13.gs[e])
            y1 = _fsum_matvec(W13, xq[t]).astype(np.float32)
            g, u = y1[:I].astype(np.float64), y1[I:].astype(np.float64)
            h = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
            hc, hs, hg = nvfp4.quantize_rows(h[None, :])
            hq = nvfp4.dequantize(hc, hs, hg)[0]
            W2 = nvfp4.dequantize(w2.codes[e], w2.sf[e], w2.gs[e])
            y2 = _fsum_matvec(W2, hq).astype(np.float32)
            np.testing.assert_allclose(y2, res.y2[(t, j)], rtol=2e-6, atol=1e-30)
            assert hg[0] == res.h_gs[(t, j)]
            term = (res.weights[t, j] * y2).astype(np.float32)
            acc = term if acc is None else (acc + term).astype(np.float32)
        out[t] = acc
    np.testing.assert_allclose(res.out_f32, out, rtol=1e-5, atol=1e-6 * np.abs(out).max())


def test_exact_grid_gemm_is_integer_matmul():
    # Activations and weights on the E2M1 grid, each 16-block holding a +-6 and
    # the whole row / matrix amax 6: gs = 448, every block scale 448 (0x7E),
    # q = 1, so quantization is lossless and w13 output = exact matmul.
    rng = np.random.default_rng(21)
    grid = nvfp4.E2M1_VALUES
    n, H, N = 5, 64, 32

    def grid_matrix(rows, cols):
        m = grid[rng.integers(0, 16, (rows, cols))]
        m[:, ::16] = 6.0 * rng.choice([-1.0, 1.0], (rows, cols // 16))
        return m.astype(np.float32)

    x = grid_matrix(n, H)
    w = grid_matrix(N, H)[None]
    codes, sf, gs = nvfp4.quantize_rows(x)
    assert (gs == 448).all() and (sf == 0x7E).all()
    assert np.array_equal(nvfp4.dequantize(codes, sf, gs), x)
    wq = moe.quantize_weights(w)
    assert wq.gs[0] == 448
    exact = (np.rint(2 * x).astype(np.int64) @ np.rint(2 * w[0]).astype(np.int64).T) / 4.0
    A = nvfp4.decode_scaled(codes, sf)
    B = nvfp4.decode_scaled(wq.codes[0], wq.sf[0])
    y = ((A @ B.T) * (1.0 / (gs[:, None].astype(np.float64) * np.float64(wq.gs[0])))).astype(np.float32)
    assert np.array_equal(y.astype(np.float64), exact)


def test_single_expert_top1_is_dense_swiglu_mlp():
    rng = np.random.default_rng(22)
    T, H, I = 6, 256, 64
    x = _bf16(rng.standard_normal((T, H)))
    wg = _bf16(rng.standard_normal((H, 1)) * 0.02)
    w13 = moe.quantize_weights(_bf16(rng.standard_normal((1, 2 * I, H)) * 0.02))
    w2 = moe.quantize_weights(_bf16(rng.standard_normal((1, H, I)) * 0.02))
    res = moe.moe_forward(x, wg, w13, w2, 1)
    assert (res.ids == 0).all() and (res.weights == 1.0).all()
    # dense MLP on the dequantized operands: y = W2q . Q(silu(G x) * (U x))
    xq = nvfp4.dequantize(*nvfp4.quantize_rows(x))
    W13 = nvfp4.dequantize(w13.codes[0], w13.sf[0], w13.gs[0])
    gu = (xq @ W13.T).astype(np.float32).astype(np.float64)
    h = (gu[:, :I] / (1 + np.exp(-gu[:, :I])) * gu[:, I:]).astype(np.float32)
    hq = nvfp4.dequantize(*nvfp4.quantize_rows(h))
    W2 = nvfp4.dequantize(w2.codes[0], w2.sf[0], w2.gs[0])
    y = (hq @ W2.T).astype(np.float32)
    np.testing.assert_allclose(res.out_f32, y, rtol=1e-5, atol=1e-7)


def test_zero_tokens_give_zero_rows():
    wl, x, wg, w13, w2, _ = _tiny()
    x = x.copy()
    x[3] = 0.0
    x[9] = 0.0
    res = moe.moe_forward(x, wg, w13, w2, wl.shape.K)
    assert not res.out_bits[3].any() and not res.out_bits[9].any()
    assert res.x_gs[3] == 1.0 and not res.x_codes[3].any() and not res.x_sf[3].any()
    assert res.out_bits[0].any()


def test_finalize_order_by_hand():
    # (2^24 + 1) + 1 with FP32 partial sums: each +1 ties to even and is lost.
    y = np.float32([[[2.0 ** 24], [1.0], [1.0]]])          # [T=1, K=3, H=1]
    w = np.float32([[1.0, 1.0, 1.0]])
    assert moe.finalize(y, w)[0, 0] == np.float32(2.0 ** 24)
    y_rev = y[:, ::-1, :]
    assert moe.finalize(y_rev, w)[0, 0] == np.float32(2.0 ** 24 + 2)


def test_token_subset_matches_full_batch():
    wl, x, wg, w13, w2, _ = _tiny()
    full = moe.moe_forward(x, wg, w13, w2, wl.shape.K)
    sub = moe.moe_forward(x, wg, w13, w2, wl.shape.K, tokens=[3, 7, 15])
    assert np.array_equal(sub.out_bits, full.out_bits[[3, 7, 15]])
    assert np.array_equal(sub.ids, full.ids[[3, 7, 15]])


def test_empty_batch():
    wl, x, wg, w13, w2, _ = _tiny()
    res = moe.moe_forward(x[:0], wg, w13, w2, wl.shape.K)
    assert res.out_bits.shape == (0, x.shape[1])


def test_close_to_unquantized_layer():
    wl, x, wg, w13, w2, _ = _tiny()
    K, I = wl.shape.K, wl.shape.I
    res = moe.moe_forward(x, wg, w13, w2, K)
    W13 = moe.as_f32(wl.w13).astype(np.float64)
    W2 = moe.as_f32(wl.w2).astype(np.float64)
    ref = np.zeros_like(res.out_f32, dtype=np.float64)
    for t in range(x.shape[0]):
        for j in range(K):
            e = res.ids[t, j]
            gu = W13[e] @ x[t].astype(np.float64)
            h = gu[:I] / (1 + np.exp(-gu[:I])) * gu[I:]
            ref[t] += res.weights[t, j] * (W2[e] @ h)
    rel = np.linalg.norm(res.out - ref) / np.linalg.norm(ref)
    assert rel < 0.25, rel


def test_swapped_gate_up_would_be_detected():
    # A planted mistake in a copy of the oracle (gate and up halves swapped)
    # must move the output far outside the parity tolerance.
    wl, x, wg, w13, w2, _ = _tiny()
    K, I = wl.shape.K, wl.shape.I
    good = moe.moe_forward(x, wg, w13, w2, K)
    swapped = moe.QuantWeights(np.concatenate([w13.codes[:, I:], w13.codes[:, :I]], axis=1),
                               np.concatenate([w13.sf[:, I:], w13.sf[:, :I]], axis=1), w13.gs)
    bad = moe.moe_forward(x, wg, swapped, w2, K)
    rms = np.sqrt(np.mean(good.out.astype(np.float64) ** 2))
    err = np.abs(bad.out - good.out)
    assert np.any(err > 2e-2 * rms + 5e-2 * np.abs(good.out))


def test_silu_hand_values():
    """silu(g) = g * sigmoid(g) at points worked out on paper: sigmoid(0) = 1/2;
    e^(-ln 3) = 1/3 gives sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4;
    e^(-ln 4) = 1/4 gives sigmoid(ln 4) = 4/5.  Large negative gates vanish,
    large positive gates pass through."""
    ln3, ln4 = math.log(3.0), math.log(4.0)
    got = moe.silu(np.array([0.0, ln3, -ln3, ln4, -ln4, -60.0, 60.0]))
    want = np.array([0.0, 0.75 * ln3, -0.25 * ln3, 0.8 * ln4, -0.2 * ln4, 0.0, 60.0])
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=1e-24)
    assert got[0] == 0.0
    assert abs(got[5]) < 1e-24  # -60 * e^-60
