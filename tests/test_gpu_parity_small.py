"""End-to-end GPU parity on the tiny layer (T=16, H=256, E=8, top-2, I=128)
and small variations, through the C ABI, against the oracle on every token:

bit-exact: router logits, top-k ids, the permutation, expert offsets,
activation codes / block scales / global scales, weight codes / block scales /
global scales.  Within tolerance: top-k weights, the requantized intermediate's
global scales, and the bf16 output.
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import moe as omoe
from oracle import nvfp4 as onv
from tests.parity import assert_close, built, gpu, needs_gpu, to_dev

pytestmark = [gpu, needs_gpu]


def _layer(shape, deterministic=None, max_num_tokens=None):
    from nvfp4_token_quantized_gb300 import MoE

    built()
    return MoE.from_shape(shape, device=0, deterministic=deterministic, max_num_tokens=max_num_tokens)


def _oracle_full(wl):
    x = omoe.as_f32(wl.x)
    q13 = omoe.quantize_weights(omoe.as_f32(wl.w13))
    q2 = omoe.quantize_weights(omoe.as_f32(wl.w2))
    bias = None if wl.bias is None else wl.bias.numpy()
    return omoe.moe_forward(x, omoe.as_f32(wl.gate_w), q13, q2, wl.shape.K, bias), q13, q2


@pytest.mark.parametrize("deterministic", [False, True])
def test_tiny_layer_parity(deterministic):
    wl = synthetic.make_workload("c0_tiny")
    d = to_dev(wl)
    layer = _layer(wl.shape, deterministic=deterministic)
    layer.load_weights(d["w13"], d["w2"])
    out = layer.forward(d["x"], d["gate_w"])
    torch.cuda.synchronize()
    ref, q13, q2 = _oracle_full(wl)

    logits = layer.debug_logits().cpu().numpy()
    assert np.array_equal(logits.view(np.uint32), ref.logits.view(np.uint32)), "router logits differ"
    r = layer.debug_routing()
    ids = r["topk_ids"].cpu().numpy()
    assert np.array_equal(ids, ref.ids)
    np.testing.assert_allclose(r["topk_w"].cpu().numpy(), ref.weights, rtol=2e-6, atol=1e-7)
    off, src, _ = omoe.permute(ref.ids, wl.shape.E)
    assert np.array_equal(r["expert_offsets"].cpu().numpy(), off)
    assert np.array_equal(r["src_of_row"].cpu().numpy(), src)

    codes, sf, gs = (t.cpu().numpy() for t in layer.debug_act_quant())
    assert np.array_equal(codes, onv.pack_e2m1(ref.x_codes))
    assert np.array_equal(sf, ref.x_sf)
    assert np.array_equal(gs.view(np.uint32), ref.x_gs.view(np.uint32))

    for which, q in ((0, q13), (1, q2)):
        wc, wsf, wgs = (t.cpu().numpy() for t in layer.debug_weight_quant(which))
        assert np.array_equal(wc, onv.pack_e2m1(q.codes)), f"weight codes {which}"
        assert np.array_equal(wsf, q.sf), f"weight block scales {which}"
        assert np.array_equal(wgs.view(np.uint32), q.gs.view(np.uint32)), f"weight global scales {which}"

    hc, hsf, hgs = (t.cpu().numpy() for t in layer.debug_intermediate())
    K = wl.shape.K
    ref_hgs = np.array([ref.h_gs[(t, j)] for t in range(wl.T) for j in range(K)], np.float32)
    np.testing.assert_allclose(hgs, ref_hgs, rtol=1e-4)

    got = out.float().cpu().numpy()
    assert_close(got, ref.out)
    layer.close()


def test_deterministic_mode_is_bitwise_repeatable():
    wl = synthetic.make_workload("c0_tiny")
    d = to_dev(wl)
    layer = _layer(wl.shape, deterministic=True)
    layer.load_weights(d["w13"], d["w2"])
    outs = [layer.forward(d["x"], d["gate_w"]).clone() for _ in range(10)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    layer.close()


def test_token_counts_on_one_instance():
    shape = synthetic.CONFIGS["c0_tiny"]
    layer = _layer(shape, max_num_tokens=64)
    wl = synthetic.make_workload(shape, T=16)
    d = to_dev(wl)
    layer.load_weights(d["w13"], d["w2"])
    q13 = omoe.quantize_weights(omoe.as_f32(wl.w13))
    q2 = omoe.quantize_weights(omoe.as_f32(wl.w2))
    for T in (1, 3, 16, 64, 0, 17):
        x = synthetic.make_activations(shape, T=T, seed=T + 100)
        out = layer.forward(x.cuda(), d["gate_w"])
        torch.cuda.synchronize()
        if T == 0:
            continue
        ref = omoe.moe_forward(omoe.as_f32(x), omoe.as_f32(wl.gate_w), q13, q2, shape.K)
        assert np.array_equal(layer.debug_routing()["topk_ids"].cpu().numpy(), ref.ids)
        assert_close(out.float().cpu().numpy(), ref.out, what=f"T={T}")
    layer.close()


def test_zero_tokens_give_zero_rows_on_gpu():
    wl = synthetic.make_workload("c0_tiny")
    x = wl.x.clone()
    x[2] = 0
    x[11] = 0
    d = to_dev(wl)
    layer = _layer(wl.shape)
    layer.load_weights(d["w13"], d["w2"])
    out = layer.forward(x.cuda(), d["gate_w"])
    torch.cuda.synchronize()
    o = out.cpu()
    assert torch.count_nonzero(o[2]) == 0 and torch.count_nonzero(o[11]) == 0
    assert torch.count_nonzero(o[0]) > 0
    layer.close()


@pytest.mark.parametrize("E,K,T", [(16, 4, 16), (16, 4, 100), (256, 12, 24), (256, 12, 100), (136, 8, 70)])
def test_tied_logits_take_the_lower_expert(E, K, T):
    """Router columns duplicated in pairs give every token's logits in exact
    pairs (the canonical FP32 order computes both the same way), so the top-k
    meets a tie at every step: the lower expert id must come first, as in the
    oracle.  Covers both per-lane candidate counts of the warp top-k (E <= 128
    and above) on the fused small-batch front end and on the top-k kernel."""
    shape = synthetic.MoEShape(name="ties", T=T, H=256, E=E, K=K, I=128, max_num_tokens=128)
    wl = synthetic.make_workload(shape, T=T, seed=11)
    gate = wl.gate_w.clone()
    gate[:, 1::2] = gate[:, 0::2]
    layer = _layer(shape)
    layer.load_weights(wl.w13.cuda(), wl.w2.cuda())
    layer.forward(wl.x.cuda(), gate.cuda())
    torch.cuda.synchronize()
    logits = omoe.router_logits(omoe.as_f32(wl.x), omoe.as_f32(gate))
    assert np.array_equal(logits[:, 0::2], logits[:, 1::2])
    ids, weights = omoe.topk_route(logits, K)
    r = layer.debug_routing()
    got = r["topk_ids"].cpu().numpy()
    assert np.array_equal(got, ids), "tie order differs from the oracle"
    np.testing.assert_allclose(r["topk_w"].cpu().numpy(), weights, rtol=1e-5, atol=1e-7)
    layer.close()

