"""GPU parity with more than eight experts per token (top-12 of 32): the
finalize's wide-top-k variant on both of its paths, a forward above 64
tokens (the prefill kernels) and a deterministic small batch, through the C
ABI against the oracle: bit-exact top-k ids and permutation, bf16 output
within the tolerance of tests/parity.py.
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import moe as omoe
from tests.parity import assert_close, built, gpu, needs_gpu, to_dev

pytestmark = [gpu, needs_gpu]

WIDE = synthetic.MoEShape(name="wide_topk", T=80, H=256, E=32, K=12, I=128, max_num_tokens=96)


@pytest.mark.parametrize("T,deterministic", [(80, False), (24, True)])
def test_wide_topk_parity(T, deterministic):
    from nvfp4_token_quantized_gb300 import MoE

    built()
    wl = synthetic.make_workload(WIDE, T=T, seed=7)
    d = to_dev(wl)
    layer = MoE.from_shape(WIDE, device=0, deterministic=deterministic, max_num_tokens=WIDE.max_num_tokens)
    layer.load_weights(d["w13"], d["w2"])
    out = layer.forward(d["x"], d["gate_w"])
    torch.cuda.synchronize()
    q13 = omoe.quantize_weights(omoe.as_f32(wl.w13))
    q2 = omoe.quantize_weights(omoe.as_f32(wl.w2))
    ref = omoe.moe_forward(omoe.as_f32(wl.x), omoe.as_f32(wl.gate_w), q13, q2, WIDE.K)
    r = layer.debug_routing()
    assert np.array_equal(r["topk_ids"].cpu().numpy(), ref.ids), "top-k ids differ"
    off, src, _ = omoe.permute(ref.ids, WIDE.E)
    assert np.array_equal(r["expert_offsets"].cpu().numpy(), off)
    assert np.array_equal(r["src_of_row"].cpu().numpy(), src)
    assert_close(out.float().cpu().numpy(), ref.out, what=f"top-12, T={T}")
    layer.close()
