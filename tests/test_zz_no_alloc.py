"""moe_route_noalloc: routing with no handle and no device allocation.

Its scratch (the router logits) is a fixed array in the
library's device code.  Checked against the routing the handle-based forward
computes for the same inputs (moe_forward_ex, read back with
moe_debug_routing), on two calls in a row; the size limit is refused before
any device work; at the limit itself, routing the whole batch equals routing
its two halves.  This file is collected last so that it also runs after every
other test in one process.
"""

import gc

import numpy as np
import pytest
import torch

import synthetic
from tests.parity import built, gpu, needs_gpu, to_dev

MAX_LOGITS = 1 << 20


def _lib():
    from nvfp4_token_quantized_gb300 import build, load_library

    build()
    return load_library()


def test_limits_refused_without_a_device():
    # argument and size checks come before any CUDA call, so they hold here
    lib = _lib()
    call = lib.moe_route_noalloc
    assert call(None, None, None, 8193, 2048, 128, 8, None, None, None) == 2  # MOE_ERR_TOO_MANY_TOKENS
    assert call(None, None, None, -1, 2048, 128, 8, None, None, None) == 1  # MOE_ERR_INVALID_ARG
    assert call(None, None, None, 16, 2000, 128, 8, None, None, None) == 8  # hidden % 256
    assert call(None, None, None, 16, 2048, 260, 8, None, None, None) == 8  # num_experts > 256
    assert call(None, None, None, 16, 2048, 128, 17, None, None, None) == 8  # top_k > 16


def _handle_routing(wl, bias):
    from nvfp4_token_quantized_gb300 import MoE

    d = to_dev(wl)
    layer = MoE.from_shape(wl.shape, device=0)
    layer.load_weights(d["w13"], d["w2"])
    layer.forward(d["x"], d["gate_w"], bias=bias)
    r = layer.debug_routing()
    torch.cuda.synchronize()
    ids, w = r["topk_ids"].clone(), r["topk_w"].clone()
    layer.close()
    return d, ids, w


@gpu
@needs_gpu
@pytest.mark.parametrize("name", ["c1_decode", "c2_specdecode"])
def test_noalloc_routing_matches_the_forward(name):
    from nvfp4_token_quantized_gb300 import moe_route_noalloc

    built()
    wl = synthetic.make_workload(name)
    bias = wl.bias.cuda() if wl.bias is not None else None
    d, ids_ref, w_ref = _handle_routing(wl, bias)
    T, K = wl.T, wl.shape.K
    ids = torch.empty(T, K, dtype=torch.int32, device="cuda")
    w = torch.empty(T, K, dtype=torch.float32, device="cuda")
    for call in range(2):
        ids.fill_(-1)
        w.fill_(float("nan"))
        torch.cuda.synchronize()
        # no collection of other tests' garbage inside the measured window
        gc.collect()
        gc.disable()
        try:
            allocated = torch.cuda.memory_allocated()
            free_before = torch.cuda.mem_get_info()[0]
            moe_route_noalloc(d["x"], d["gate_w"], K, bias=bias, topk_ids=ids, topk_w=w)
            torch.cuda.synchronize()
            allocated_after = torch.cuda.memory_allocated()
            free_after = torch.cuda.mem_get_info()[0]
        finally:
            gc.enable()
        assert allocated_after == allocated
        # Call 0 may be the first on this device when the file runs alone: it
        # loads the library's device code there (lazy module loading), which
        # reserves the fixed scratch array.  Every later call allocates nothing.
        if call == 1:
            assert free_after == free_before, "device memory changed during the call"
        assert torch.equal(ids, ids_ref), f"call {call}: top-k ids differ from the forward's routing"
        # the same device functions on the same inputs: the weights agree bit for bit
        assert torch.equal(w.view(torch.int32), w_ref.view(torch.int32)), f"call {call}: routing weights differ"


@gpu
@needs_gpu
def test_noalloc_at_the_size_limit():
    from nvfp4_token_quantized_gb300 import MoEError, moe_route_noalloc

    built()
    shape = synthetic.CONFIGS["c1_decode"]
    E, K = shape.E, shape.K
    T = MAX_LOGITS // E  # exactly at the limit
    x = synthetic.make_activations(shape, T=T, seed=5).cuda()
    gate = synthetic.make_router(shape).cuda()
    ids, w = moe_route_noalloc(x, gate, K)
    h = T // 2
    ids_a, w_a = moe_route_noalloc(x[:h], gate, K)
    ids_b, w_b = moe_route_noalloc(x[h:], gate, K)
    torch.cuda.synchronize()
    assert torch.equal(ids, torch.cat([ids_a, ids_b]))
    assert torch.equal(w.view(torch.int32), torch.cat([w_a, w_b]).view(torch.int32))
    assert bool(((ids >= 0) & (ids < E)).all())
    with pytest.raises(MoEError) as ei:
        moe_route_noalloc(torch.zeros(T + 1, shape.H, dtype=torch.bfloat16, device="cuda"), gate, K)
    assert ei.value.status == 2
