"""GPU parity of the layer with a shared expert (the Cohere2MoE sparse block
of "SM10X Command-A-Plus decode 2.3x faster, BCG capture memory -78%": a
dense SwiGLU expert on every token next to the routed experts, combined by
sum or by the 'average' strategy).

The library runs the shared expert on a second stream (quantize, w13 GEMM
with the fused requantization, w2 GEMM into bf16 rows) and joins it before
the finalize, which adds the shared row to the routed FP32 sum.  Checked
through the C ABI against the oracle with ``shared=(w13s, w2s)``:

* the shared branch's own per-token quantization of x, bit for bit;
* the shared rows and the layer output against the oracle, with the
  shared intermediate's rare near-tie requantization decisions taken from
  the GPU on both sides (see _check);
* small batches (the single-kernel front and the 64-row GEMMs) and batches
  above 64 tokens (the expanded layout and 128-row cluster GEMMs), each
  with sum and average;
* a shared width that is not a multiple of 256 (Is = 384: the w2 GEMM's K
  is zero-padded to 512);
* deterministic mode gives the same bits on every run, and a CUDA graph
  capture of the forked forward replays to the eager output;
* a handle with a shared expert refuses to run before its shared weights
  are loaded;
* the widest shapes (I = Is = 2048, top-16) above 64 tokens.
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import moe as omoe
from oracle import nvfp4 as onv
from tests.parity import assert_close, built, gpu, needs_gpu, to_dev

pytestmark = [gpu, needs_gpu]

MID = synthetic.MoEShape(name="shared_mid", T=200, H=512, E=16, K=4, I=256, max_num_tokens=256)


def _bf16(a):
    return onv.bf16_to_f32(onv.bf16_round(np.asarray(a, dtype=np.float32)))


def _run(shape, T, Is, average, deterministic=False, seed=3, accurate=False):
    from nvfp4_token_quantized_gb300 import MoE

    built()
    wl = synthetic.make_workload(shape, T=T, seed=seed)
    w13s, w2s = synthetic.make_shared_weights(shape, Is, seed=seed)
    d = to_dev(wl)
    layer = MoE(shape.H, shape.I, shape.E, shape.K, shape.max_num_tokens, device=0, deterministic=deterministic,
                shared_inter=Is, shared_average=average, accurate_sigmoid=accurate)
    layer.load_weights(d["w13"], d["w2"])
    layer.load_shared_weights(w13s.cuda(), w2s.cuda())
    out = layer.forward(d["x"], d["gate_w"])
    torch.cuda.synchronize()
    q13 = omoe.quantize_weights(omoe.as_f32(wl.w13))
    q2 = omoe.quantize_weights(omoe.as_f32(wl.w2))
    q13s = omoe.quantize_weights(omoe.as_f32(w13s)[None])
    q2s = omoe.quantize_weights(omoe.as_f32(w2s)[None])
    ref = omoe.moe_forward(omoe.as_f32(wl.x), omoe.as_f32(wl.gate_w), q13, q2, shape.K,
                           shared=(q13s, q2s), shared_average=average)
    routed = omoe.moe_forward(omoe.as_f32(wl.x), omoe.as_f32(wl.gate_w), q13, q2, shape.K)
    return layer, d, out, ref, routed, q2s, q13s


def _check(layer, out, ref, routed, q2s, q13s, average, what):
    """Output parity, separating the requantization decisions of the shared
    intermediate.

    The GPU forms SwiGLU in FP32 (with a hardware tanh for the sigmoid) from
    FP32 tensor-core sums; the oracle in FP64.  A block whose maximum or an
    element lies within that difference of an E4M3 or E2M1 rounding boundary
    can take the neighbouring code, and with weight one (the shared expert is
    not scaled by a routing weight) one such block moves a few outputs of its
    row by up to ~15 % of the row's rms.  So: the global scales agree, such
    blocks are rare, the layer output equals the oracle's second GEMM and
    combination applied to the GPU's own intermediate (the same decisions on
    both sides), and every row whose intermediate matches exactly equals the
    oracle's full forward."""
    T = out.shape[0]
    # the shared branch quantizes x itself: bit for bit the per-token rules
    ac, asf, ags = (t.cpu().numpy() for t in layer.debug_shared_act_quant())
    assert np.array_equal(ags.view(np.uint32), ref.x_gs.view(np.uint32)), f"{what}: shared input global scales"
    assert np.array_equal(asf, ref.x_sf), f"{what}: shared input block scales"
    assert np.array_equal(ac, onv.pack_e2m1(ref.x_codes)), f"{what}: shared input codes"
    rows, hc, hsf, hgs = (t.cpu() for t in layer.debug_shared())
    sr = omoe.expert_rows(ref.x_codes, ref.x_sf, ref.x_gs, q13s, q2s, 0)
    hgs = hgs.numpy()
    np.testing.assert_allclose(hgs, sr["h_gs"], rtol=1e-4)
    packed = hc.numpy()
    codes = np.stack([packed & 0xF, packed >> 4], -1).reshape(T, -1)
    hsf = hsf.numpy()
    code_diff = codes != sr["h_codes"]
    assert code_diff.mean() <= 1e-3, f"{what}: {int(code_diff.sum())} intermediate codes differ"
    flipped = code_diff.any(1) | (hsf != sr["h_sf"]).any(1)
    assert flipped.sum() <= max(1, T // 50), f"{what}: {int(flipped.sum())} intermediate rows differ"
    y2 = omoe.expert_w2(codes, hsf, hgs, q2s, 0)
    assert_close(rows.float().numpy(), y2, what=f"{what}: shared rows")
    same = _bf16(omoe.combine_shared(routed.out_f32, y2, average))
    got = out.float().cpu().numpy()
    assert_close(got, same, what=f"{what}: downstream of the GPU intermediate")
    keep = ~flipped
    assert_close(got[keep], ref.out[keep], what=f"{what}: rows with an exactly matching intermediate")


@pytest.mark.parametrize("T,Is,average,deterministic", [
    (16, 128, False, False),     # small batch, atomic finalize
    (16, 128, True, True),       # small batch, ordered finalize, average
    (48, 384, False, False),     # Is not a multiple of 256
    (200, 256, False, False),    # above 64 tokens: cluster GEMMs, ordered finalize
    (200, 384, True, False),
    (129, 128, False, True),     # a ragged second 128-row tile
])
def test_shared_expert_parity(T, Is, average, deterministic):
    layer, _, out, ref, routed, q2s, q13s = _run(MID, T, Is, average, deterministic)
    _check(layer, out, ref, routed, q2s, q13s, average, f"shared Is={Is}, T={T}, average={average}")
    layer.close()


def test_shared_expert_changes_the_output():
    """The shared expert's contribution is visible: the sum differs from the
    routed-only output of the same layer by far more than the tolerance."""
    from nvfp4_token_quantized_gb300 import MoE

    layer, d, out, ref, _, _, _ = _run(MID, 40, 256, False)
    routed = MoE(MID.H, MID.I, MID.E, MID.K, MID.max_num_tokens, device=0)
    routed.load_weights(d["w13"], d["w2"])
    base = routed.forward(d["x"], d["gate_w"]).float()
    torch.cuda.synchronize()
    diff = (out.float() - base).abs().max().item()
    assert diff > 0.1 * base.abs().max().item()
    routed.close()
    layer.close()


def test_shared_expert_deterministic_and_graph():
    layer, d, out, ref, routed, q2s, q13s = _run(MID, 200, 256, True, deterministic=True)
    outs = [layer.forward(d["x"], d["gate_w"]).clone() for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), out.view(torch.int16)), "deterministic mode differs between runs"
    s = torch.cuda.Stream()
    buf = torch.empty_like(out)
    with torch.cuda.stream(s):
        layer.forward(d["x"], d["gate_w"], out=buf, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(d["x"], d["gate_w"], out=buf, stream=s)
    buf.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(buf.view(torch.int16), out.view(torch.int16)), "graph replay differs from eager"
    _check(layer, buf, ref, routed, q2s, q13s, True, "shared expert, graph replay")
    layer.close()


def test_shared_weights_required():
    from nvfp4_token_quantized_gb300 import MoE, MoEError
    from nvfp4_token_quantized_gb300.binding import MOE_ERR_INVALID_ARG, MOE_ERR_NOT_LOADED

    built()
    wl = synthetic.make_workload(MID, T=8)
    d = to_dev(wl)
    layer = MoE(MID.H, MID.I, MID.E, MID.K, MID.max_num_tokens, device=0, shared_inter=128)
    layer.load_weights(d["w13"], d["w2"])
    with pytest.raises(MoEError) as ei:
        layer.forward(d["x"], d["gate_w"])
    assert ei.value.status == MOE_ERR_NOT_LOADED
    w13s, w2s = synthetic.make_shared_weights(MID, 256)           # wrong width
    with pytest.raises(MoEError) as ei:
        layer.load_shared_weights(w13s.cuda(), w2s.cuda())
    assert ei.value.status == MOE_ERR_INVALID_ARG
    layer.close()
    plain = MoE(MID.H, MID.I, MID.E, MID.K, MID.max_num_tokens, device=0)
    w13s, w2s = synthetic.make_shared_weights(MID, 128)
    with pytest.raises(MoEError):
        plain.load_shared_weights(w13s.cuda(), w2s.cuda())
    plain.close()


@pytest.mark.parametrize("T", [100])
def test_maximum_widths(T):
    """The widest supported layer shapes in one handle, above 64 tokens:
    I = 2048 (w13 clusters of 16 CTAs exchanging row maxima), top-16 (the
    wide finalize variant), and a 2048-wide shared expert (its own 16-CTA
    clusters)."""
    shape = synthetic.MoEShape(name="max_widths", T=T, H=256, E=32, K=16, I=2048, max_num_tokens=128)
    layer, _, out, ref, routed, q2s, q13s = _run(shape, T, 2048, False)
    r = layer.debug_routing()
    assert np.array_equal(r["topk_ids"].cpu().numpy(), ref.ids)
    _check(layer, out, ref, routed, q2s, q13s, False, f"maximum widths, T={T}")
    layer.close()


FLIP = synthetic.MoEShape(name="flip_rate", T=2048, H=2048, E=8, K=1, I=128, max_num_tokens=2048)


@pytest.mark.parametrize("T", [64, 2048])
def test_sigmoid_forms_flip_rate(T):
    """How often the SwiGLU's sigmoid form moves a requantization decision of
    the intermediate away from the oracle's FP64 evaluation: the shared
    expert (weight one, 1536 features per row) of T tokens, once with the
    hardware-tanh sigmoid (the default) and once with the accurate one
    (MOE_FLAG_ACCURATE_SIGMOID).  T = 64 runs the small-batch w13 GEMM and the
    row requantization kernel, T = 2048 the cluster GEMM with the fused
    requantization.  The counts are printed for the record; the accurate
    form must not flip more blocks."""
    from nvfp4_token_quantized_gb300 import MoE

    built()
    Is = 1536
    wl = synthetic.make_workload(FLIP, T=T, seed=11)
    w13s, w2s = synthetic.make_shared_weights(FLIP, Is, seed=11)
    q13s = omoe.quantize_weights(omoe.as_f32(w13s)[None])
    q2s = omoe.quantize_weights(omoe.as_f32(w2s)[None])
    xc, xs, xg = onv.quantize_rows(omoe.as_f32(wl.x))
    sr = omoe.expert_rows(xc, xs, xg, q13s, q2s, 0)
    d = to_dev(wl)
    counts = {}
    for accurate in (False, True):
        layer = MoE(FLIP.H, FLIP.I, FLIP.E, FLIP.K, FLIP.max_num_tokens, device=0, shared_inter=Is,
                    accurate_sigmoid=accurate)
        layer.load_weights(d["w13"], d["w2"])
        layer.load_shared_weights(w13s.cuda(), w2s.cuda())
        layer.forward(d["x"], d["gate_w"])
        torch.cuda.synchronize()
        hc, hsf, hgs = (t.cpu().numpy() for t in layer.debug_shared()[1:])
        layer.close()
        np.testing.assert_allclose(hgs, sr["h_gs"], rtol=1e-4)
        codes = np.stack([hc & 0xF, hc >> 4], -1).reshape(T, -1)
        blk = (codes != sr["h_codes"]).reshape(T, -1, 16).any(2) | (hsf != sr["h_sf"])
        counts[accurate] = (int(blk.any(1).sum()), int(blk.sum()), blk.size)
    print(f"\nflip rate T={T}: tanh.approx rows {counts[False][0]}/{T}, blocks {counts[False][1]}/"
          f"{counts[False][2]}; accurate rows {counts[True][0]}/{T}, blocks {counts[True][1]}/{counts[True][2]}")
    assert counts[True][1] <= counts[False][1]
