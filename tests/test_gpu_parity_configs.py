"""GPU parity at the full workload sizes, through the C ABI.

* decode (T=64, H=2048, E=128, top-8, I=768) captured in a CUDA graph and
  replayed;
* speculative-decode batch (T=256) with Zipf-skewed routing in deterministic
  mode, bitwise identical over 10 runs;
* prefill on one instance sized for 4096 tokens, forwards of 1, 17, 2048, 4073
  and 4096 tokens, and a refused 4097-token forward;
* per-token-scale stress (T=2048, H=4096, E=64, top-6, I=1536) with an
  in-place weight reload under a captured graph, compared with a fresh
  instance.

Bit-exact: router logits and top-k ids, the permutation and expert offsets
(the whole batch at every token count of at least 17), the activation codes /
block scales / global scales of every token (all forwards above 64 tokens run
the per-token quantize kernel; up to 64 tokens the fused front kernel), and
weight codes / block scales / global scales (sampled experts).  Outputs within
the parity tolerance: every token up to 256 tokens; above that, a set of
tokens that puts at least one checked row - the first and the last - in every
128-row GEMM tile of every expert with rows, each expert's ragged last tile
included, so that every tile, every cluster rank's features and every
expert's weights feed a checked output.
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import moe as omoe
from oracle import nvfp4 as onv
from tests.parity import (assert_close, built, gpu, needs_gpu, oracle_forward_parallel, oracle_route,
                          quantize_experts, tile_covering_tokens, to_dev)

pytestmark = [gpu, needs_gpu]


def _layer(shape, **kw):
    from nvfp4_token_quantized_gb300 import MoE

    built()
    return MoE.from_shape(shape, device=0, **kw)


def _check_routing(layer, wl, tokens=None, full_permutation=False):
    logits_ref, ids_ref, w_ref = oracle_route(wl, tokens)
    tok = np.arange(wl.T) if tokens is None else np.asarray(tokens)
    logits = layer.debug_logits().cpu().numpy()[tok]
    assert np.array_equal(logits.view(np.uint32), logits_ref.view(np.uint32)), "router logits differ"
    r = layer.debug_routing()
    ids = r["topk_ids"].cpu().numpy()
    assert np.array_equal(ids[tok], ids_ref), "top-k ids differ"
    np.testing.assert_allclose(r["topk_w"].cpu().numpy()[tok], w_ref, rtol=3e-6, atol=1e-7)
    if full_permutation:
        off, src, _ = omoe.permute(ids_ref, wl.shape.E)
        assert np.array_equal(r["expert_offsets"].cpu().numpy(), off)
        assert np.array_equal(r["src_of_row"].cpu().numpy(), src)
    return ids_ref, r


def _check_act_quant(layer, wl, tokens=None, what="activations"):
    """Codes, block-scale bytes and global-scale bits of the tokens (all by
    default) equal the oracle's per-token quantization."""
    tok = np.arange(wl.T) if tokens is None else np.asarray(tokens)
    codes, sf, gs = (t.cpu().numpy() for t in layer.debug_act_quant())
    rc, rs, rg = onv.quantize_rows(omoe.as_f32(wl.x)[tok])
    assert np.array_equal(gs[tok].view(np.uint32), rg.view(np.uint32)), f"{what}: global scales differ"
    assert np.array_equal(sf[tok], rs), f"{what}: block scales differ"
    assert np.array_equal(codes[tok], onv.pack_e2m1(rc)), f"{what}: codes differ"


def _check_weight_quant(layer, wl, experts):
    q13 = quantize_experts(wl.w13, experts)
    q2 = quantize_experts(wl.w2, experts)
    for which, q in ((0, q13), (1, q2)):
        codes, sf, gs = (t.cpu().numpy() for t in layer.debug_weight_quant(which))
        for e in experts:
            assert np.array_equal(codes[e], onv.pack_e2m1(q.codes[e])), f"weight codes {which} expert {e}"
            assert np.array_equal(sf[e], q.sf[e]), f"weight block scales {which} expert {e}"
            assert gs[e] == q.gs[e], f"weight global scale {which} expert {e}"


# Requantization decisions of the intermediate are not bit-exact targets (the
# GPU sums in FP32 on the tensor cores and forms SwiGLU in FP32, the oracle
# in FP64): a block whose maximum or an element sits within that difference
# of an E4M3 or E2M1 rounding boundary can take the neighbouring code.  Such
# blocks must stay this rare.
MAX_FLIPPED_BLOCK_FRACTION = 2e-3


def _check_output(out, wl, tokens, what, layer):
    """The output of the tokens against the oracle, with the intermediate's
    requantization decisions separated:
    * the intermediate's global scales agree (rtol 1e-4) and blocks whose
      codes or scale differ from the oracle's are rare;
    * every token's output equals, within the tolerance, the oracle's second
      GEMM and finalize applied to the GPU's own intermediate (the same
      decisions on both sides);
    * every token whose K intermediate rows all match the oracle's exactly
      equals the oracle's whole forward within the tolerance."""
    h = tuple(t.cpu().numpy() for t in layer.debug_intermediate())
    res = oracle_forward_parallel(wl, tokens, h_gpu=h)
    got = out.float().cpu().numpy()[np.asarray(tokens)]
    np.testing.assert_allclose(res.h_gs_gpu, res.h_gs_ref, rtol=1e-4, err_msg=f"{what}: intermediate global scales")
    tok_flipped = res.flipped.any(1)
    print(f"\n{what}: intermediate blocks differing from the oracle {res.flipped_blocks}/{res.blocks}, "
          f"rows {int(res.flipped.sum())}/{res.flipped.size}, tokens {int(tok_flipped.sum())}/{len(tok_flipped)}")
    assert res.flipped_blocks <= max(4, MAX_FLIPPED_BLOCK_FRACTION * res.blocks), f"{what}: too many flipped blocks"
    assert_close(got, res.out_gpu_h, what=f"{what} (downstream of the GPU intermediate)")
    return assert_close(got[~tok_flipped], res.out[~tok_flipped], what=f"{what} (tokens whose intermediate matches)")


def test_decode_graph_replay():
    wl = synthetic.make_workload("c1_decode")
    d = to_dev(wl)
    layer = _layer(wl.shape)
    layer.load_weights(d["w13"], d["w2"])
    out = torch.empty_like(d["x"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward(d["x"], d["gate_w"], out=out)
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(d["x"], d["gate_w"], out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    replay = out.clone()
    _check_routing(layer, wl, full_permutation=True)
    _check_act_quant(layer, wl)
    tokens = np.arange(wl.T)
    _check_output(replay, wl, tokens, "graph replay", layer)
    if not torch.equal(eager, replay):  # the atomic finalize adds in arrival order
        _check_output(eager, wl, tokens, "eager", layer)
    _check_weight_quant(layer, wl, [0, 77, 127])
    layer.close()


def test_specdecode_deterministic_zipf():
    wl = synthetic.make_workload("c2_specdecode")
    d = to_dev(wl)
    layer = _layer(wl.shape)
    assert layer.deterministic
    layer.load_weights(d["w13"], d["w2"])
    outs = [layer.forward(d["x"], d["gate_w"], bias=d["bias"]).clone() for _ in range(10)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16)), "deterministic mode differs between runs"
    ids, r = _check_routing(layer, wl, full_permutation=True)
    counts = np.diff(r["expert_offsets"].cpu().numpy())
    assert (counts == 0).sum() >= 4, "skewed routing should leave experts without rows"
    assert counts.max() > 4 * counts.mean()
    _check_act_quant(layer, wl, what="zipf deterministic activations")
    _check_output(outs[0], wl, np.arange(wl.T), "zipf deterministic", layer)


def test_prefill_token_sweep_one_instance():
    from nvfp4_token_quantized_gb300 import MoEError

    shape = synthetic.CONFIGS["c3_prefill"]
    wl = synthetic.make_workload(shape, T=1)
    gate = wl.gate_w.cuda()
    layer = _layer(shape)
    layer.load_weights(wl.w13.cuda(), wl.w2.cuda())
    ptrs = layer.debug_buffer_ptrs()
    for T in (1, 17, 2048, 4073, 4096):
        # new activations for every token count, the instance's weights
        xT = synthetic.make_activations(shape, T=T, seed=T)
        wlT = synthetic.Workload(shape=shape, x=xT, gate_w=wl.gate_w, w13=wl.w13, w2=wl.w2, bias=None)
        out = layer.forward(xT.cuda(), gate)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        _check_act_quant(layer, wlT, what=f"T={T} activations")
        if T == 1:
            _check_routing(layer, wlT, None)
            tokens = np.arange(T)
        else:  # the whole batch: every token's route and the full permutation
            ids, _ = _check_routing(layer, wlT, None, full_permutation=True)
            tokens = np.arange(T) if T <= 256 else tile_covering_tokens(ids, shape.E)
        _check_output(out, wlT, tokens, f"T={T}", layer)
    assert layer.debug_buffer_ptrs() == ptrs, "a forward moved a device buffer"
    with pytest.raises(MoEError) as ei:
        layer.forward(torch.zeros(4097, shape.H, dtype=torch.bfloat16, device="cuda"), gate)
    assert ei.value.status == 2  # MOE_ERR_TOO_MANY_TOKENS
    layer.close()


def test_stress_refresh_replay_equals_fresh():
    from nvfp4_token_quantized_gb300 import MoEError

    shape = synthetic.CONFIGS["c4_stress"]
    wl = synthetic.make_workload(shape)
    w13_b, w2_b = synthetic.make_weights(shape, seed=shape.refresh_seed)
    x, gate = wl.x.cuda(), wl.gate_w.cuda()
    layer = _layer(shape)
    assert layer.deterministic
    layer.load_weights(wl.w13.cuda(), wl.w2.cuda())
    out = torch.empty_like(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward(x, gate, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(x, gate, out=out)
    g.replay()
    torch.cuda.synchronize()
    before = out.clone()
    ptrs = layer.debug_buffer_ptrs()
    # every row: zero rows, norms over six decades, the x100 outlier channels
    _check_act_quant(layer, wl, what="stress activations")

    w13_b_dev, w2_b_dev = w13_b.cuda(), w2_b.cuda()
    layer.refresh_scales_inplace(w13_b_dev, w2_b_dev)
    g.replay()
    torch.cuda.synchronize()
    refreshed = out.clone()
    assert layer.debug_buffer_ptrs() == ptrs, "refresh moved a device buffer"
    _check_act_quant(layer, wl, what="stress activations after the refresh")
    assert not torch.equal(refreshed, before)

    fresh = _layer(shape)
    fresh.load_weights(w13_b_dev, w2_b_dev)
    expect = fresh.forward(x, gate)
    torch.cuda.synchronize()
    assert torch.equal(refreshed.view(torch.int16), expect.view(torch.int16)), "replay after refresh != fresh load"
    fresh.close()

    # changed metadata is refused and leaves the loaded weights in place
    with pytest.raises(MoEError) as ei:
        layer.refresh_scales_inplace(w13_b_dev[:, :-128].contiguous(), w2_b_dev)
    assert ei.value.status == 4  # MOE_ERR_METADATA_CHANGED

    # zero rows stay exactly zero; sampled rows (zero, smallest and largest
    # norms, and a spread) match the oracle with the reloaded weights
    xf = wl.x.float()
    norms = xf.norm(dim=1)
    zero = torch.nonzero(norms == 0).flatten()
    assert zero.numel() == synthetic.workloads.expected_zero_rows(shape, wl.T)
    assert torch.count_nonzero(refreshed[zero.cuda()]) == 0
    nz = torch.nonzero(norms > 0).flatten()
    extra = [int(zero[0]), int(nz[norms[nz].argmin()]), int(nz[norms[nz].argmax()])]
    _, ids_all, _ = oracle_route(wl)
    tokens = np.union1d(tile_covering_tokens(ids_all, shape.E), extra)
    wl_b = synthetic.Workload(shape=shape, x=wl.x, gate_w=wl.gate_w, w13=w13_b, w2=w2_b, bias=None)
    _check_output(refreshed, wl_b, tokens, "stress after refresh", layer)
    _check_weight_quant(layer, wl_b, [0, 63])
    layer.close()


@pytest.mark.parametrize("T,H,E,K", [(5000, 256, 16, 4), (80, 4352, 8, 2), (600, 512, 32, 4)])
def test_long_batch_and_wide_rows(T, H, E, K):
    """Paths the benchmark shapes do not reach: more than 4096 tokens (the
    permutation counts its experts in a pass of its own before ranking),
    rows wider than 4096 elements (the activation quantizer forms codes after
    its dependency wait instead of holding them in registers), and the
    router's 32-expert blocks with streamed activations (more than 512
    tokens, H <= 1536).  Routing, the whole permutation and every token's
    quantization are bit-exact; every token's output is checked as in the
    other workloads."""
    shape = synthetic.MoEShape(name="edge", T=T, H=H, E=E, K=K, I=128, max_num_tokens=T)
    wl = synthetic.make_workload(shape, T=T, seed=5)
    d = to_dev(wl)
    layer = _layer(shape)
    layer.load_weights(d["w13"], d["w2"])
    out = layer.forward(d["x"], d["gate_w"])
    torch.cuda.synchronize()
    _check_routing(layer, wl, full_permutation=True)
    _check_act_quant(layer, wl)
    _check_output(out, wl, np.arange(T), f"T={T} H={H}", layer)
    layer.close()
