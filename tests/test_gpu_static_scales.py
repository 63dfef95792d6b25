"""The static per-tensor activation-scale contract on the GPU, against the
oracle's static forward ("CuTe DSL backend gets per-token NVFP4 online
quantization and reload" keeps it apart from per-token scales: Summary,
Implementation item 2).

Calibrated scales: x_gs = 2688 / max|x| over the batch; h_gs[e] varies with
the expert (so a dropped or misindexed scale fails).  Covered: the
small-batch path (fused front kernel, w13 without clusters), decode size,
a 256-token batch (the clustered w13 with its row exchange skipped), a
saturating scale, and the handle's state errors.  Activation codes and block
scales are compared bit for bit; outputs within the parity tolerance.
"""

import numpy as np
import pytest
import torch

from oracle import moe as omoe
from oracle import nvfp4 as onv
from tests.parity import (assert_close, built, gpu, needs_gpu, oracle_forward, sample_tokens, to_dev,
                          workload)

pytestmark = [gpu, needs_gpu]


def _scales(wl, x_factor=1.0):
    x = omoe.as_f32(wl.x)
    x_gs = np.float32(onv.global_scale(np.max(np.abs(x))) * np.float32(x_factor))
    E = wl.shape.E
    h_gs = np.float32(2688.0) / (np.float32(4.0) + (np.arange(E, dtype=np.float32) % np.float32(7)))
    return x_gs, h_gs.astype(np.float32)


def _run(name, T=None, x_factor=1.0, n_check=8):
    from nvfp4_token_quantized_gb300 import MoE

    built()
    wl = workload(name, T)
    d = to_dev(wl)
    x_gs, h_gs = _scales(wl, x_factor)
    layer = MoE.from_shape(wl.shape, device=0, static_scales=True, max_num_tokens=wl.shape.max_num_tokens)
    layer.load_weights(d["w13"], d["w2"])
    layer.set_static_scales(torch.tensor([x_gs], device="cuda"), torch.from_numpy(h_gs).cuda())
    out = layer.forward(d["x"], d["gate_w"], bias=d["bias"])
    torch.cuda.synchronize()
    tokens = sample_tokens(wl.T, n_check)
    ref = oracle_forward(wl, tokens, static_scales=(x_gs, h_gs))
    codes, sf, gs = (t.cpu().numpy() for t in layer.debug_act_quant())
    assert np.array_equal(codes[tokens], onv.pack_e2m1(ref.x_codes)), "static activation codes differ"
    assert np.array_equal(sf[tokens], ref.x_sf), "static activation block scales differ"
    assert np.all(gs[tokens] == x_gs)
    assert_close(out.float().cpu().numpy()[tokens], ref.out, what=f"static {name}")
    layer.close()
    return ref


def test_static_small_batch():
    _run("c0_tiny")


def test_static_decode():
    _run("c1_decode")


def test_static_large_batch_clustered_w13():
    _run("c2_specdecode", n_check=6)


def test_static_saturating_scale_matches_oracle():
    ref = _run("c0_tiny", x_factor=16.0)
    assert np.any(ref.x_sf == 0x7E)  # the 16x scale saturates block scales


def test_static_state_errors():
    from nvfp4_token_quantized_gb300 import MoE, MoEError

    built()
    wl = workload("c0_tiny")
    d = to_dev(wl)
    layer = MoE.from_shape(wl.shape, device=0, static_scales=True)
    layer.load_weights(d["w13"], d["w2"])
    with pytest.raises(MoEError) as ei:
        layer.forward(d["x"], d["gate_w"])
    assert ei.value.status == 3  # MOE_ERR_NOT_LOADED: scales not set
    layer.close()
    plain = MoE.from_shape(wl.shape, device=0)
    with pytest.raises(MoEError) as ei:
        plain.set_static_scales(torch.ones(1, device="cuda"), torch.ones(wl.shape.E, device="cuda"))
    assert ei.value.status == 1  # MOE_ERR_INVALID_ARG: not a static handle
    plain.close()
