"""C-ABI contract on a GPU: argument checks, the lifecycle state machine, the
aliasing rule, the host-buffer entry point, and stage timing.  Every failure
here is a returned status; nothing faults or waits on the device."""

import numpy as np
import pytest
import torch

import synthetic
from tests.parity import built, gpu, needs_gpu, to_dev

pytestmark = [gpu, needs_gpu]

OK, INVALID, TOO_MANY, NOT_LOADED, META, ALIAS = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def tiny():
    from nvfp4_token_quantized_gb300 import MoE

    built()
    wl = synthetic.make_workload("c0_tiny")
    layer = MoE.from_shape(wl.shape, device=0, max_num_tokens=32)
    return wl, layer


def _status(fn, *a):
    from nvfp4_token_quantized_gb300 import MoEError

    try:
        fn(*a)
    except MoEError as e:
        return e.status
    return OK


def test_state_machine_and_errors(tiny):
    from nvfp4_token_quantized_gb300 import MoE
    from nvfp4_token_quantized_gb300.binding import load_library

    wl, layer = tiny
    d = to_dev(wl)
    fresh = MoE.from_shape(wl.shape, device=0)
    assert _status(fresh.forward, d["x"], d["gate_w"]) == NOT_LOADED
    assert _status(fresh.refresh_scales_inplace, d["w13"], d["w2"]) == NOT_LOADED
    fresh.close()

    layer.load_weights(d["w13"], d["w2"])
    # wrong weight shape at load
    assert _status(layer.load_weights, d["w13"][:, :128].contiguous(), d["w2"]) == INVALID
    # over capacity (the instance holds 32 tokens)
    big = torch.zeros(33, wl.shape.H, dtype=torch.bfloat16, device="cuda")
    assert _status(layer.forward, big, d["gate_w"]) == TOO_MANY
    # out aliasing x is refused
    assert _status(layer.forward, d["x"], d["gate_w"], d["x"]) == ALIAS
    # zero tokens is a no-op
    lib = load_library()
    assert lib.moe_forward(layer.handle, None, None, None, 0, None) == OK
    assert layer.status == OK
    assert lib.moe_get_workspace_bytes(layer.handle) > 0


def test_forward_host_matches_device(tiny):
    wl, layer = tiny
    d = to_dev(wl)
    layer.load_weights(d["w13"], d["w2"])
    dev_out = layer.forward(d["x"], d["gate_w"])
    torch.cuda.synchronize()
    host_out = torch.empty_like(wl.x).pin_memory()
    layer.forward_host(wl.x.pin_memory(), wl.gate_w.pin_memory(), host_out)
    ref = dev_out.cpu().float()
    err = (host_out.float() - ref).abs().max().item()
    assert err <= 1e-2 * ref.abs().max().item()


def test_stage_timing(tiny):
    wl, layer = tiny
    d = to_dev(wl)
    layer.load_weights(d["w13"], d["w2"])
    layer.set_stage_timing(True)
    layer.forward(d["x"], d["gate_w"])
    torch.cuda.synchronize()
    st = layer.stage_times()
    layer.set_stage_timing(False)
    assert list(st) == ["router", "topk", "permute", "quantize", "gemm_w13", "gemm_w2", "finalize"]
    assert all(v >= 0 for v in st.values())


def test_hardware_conversion_of_the_worked_examples():
    # the device quantizer's conversions reproduce the hand-derived bytes
    from nvfp4_token_quantized_gb300 import moe_debug_convert

    built()
    vals = np.float32([6, 3, 1.5, 0.75, 0.25, -0.25, -1, -2, 5, 2.5, 1.25, 0, -6, -3, 4, 1])
    e2, e4 = moe_debug_convert(torch.from_numpy(vals).cuda())
    assert e2.cpu().tolist() == [0x7, 0x5, 0x3, 0x2, 0x0, 0x8, 0xA, 0xC, 0x6, 0x4, 0x2, 0x0, 0xF, 0xD, 0x6, 0x2]
    _, e4 = moe_debug_convert(torch.tensor([448.0, 37.333333, 2.0 ** -10, 0.0013020833], device="cuda"))
    assert e4.cpu().tolist() == [0x7E, 0x61, 0x00, 0x01]


def test_narrower_handle_leaves_wider_one_working():
    # kernel launch limits are per kernel, not per handle: creating a handle
    # with a smaller hidden and intermediate size must not break the forward
    # of a wider handle created before it
    import dataclasses

    from nvfp4_token_quantized_gb300 import MoE

    built()
    wide = dataclasses.replace(synthetic.CONFIGS["c0_tiny"], name="wide", H=1024, I=512, deterministic=True)
    wl = synthetic.make_workload(wide)
    d = to_dev(wl)
    a = MoE.from_shape(wide, device=0)
    a.load_weights(d["w13"], d["w2"])
    before = a.forward(d["x"], d["gate_w"]).clone()
    narrow = dataclasses.replace(wide, name="narrow", H=256, I=128)
    b = MoE.from_shape(narrow, device=0)
    after = a.forward(d["x"], d["gate_w"])
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), after.view(torch.int16))
    b.close()
    a.close()


def test_hidden_beyond_the_router_tile_is_refused():
    # the router keeps a [hidden x 8] slice of its weight and 48 KB of
    # activation rings in one CTA's shared memory: hidden 11520 needs 228 KB
    # in all, over the 227 KB a CTA may hold; the create and the no-handle
    # routing refuse it before any allocation or launch
    from nvfp4_token_quantized_gb300 import MoE
    from nvfp4_token_quantized_gb300.binding import load_library

    built()
    UNSUPPORTED = 8
    assert _status(lambda: MoE(hidden=11520, inter=256, num_experts=64, top_k=4, max_num_tokens=16)) == UNSUPPORTED
    x = torch.zeros(2, 11520, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(11520, 64, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(2, 4, dtype=torch.int32, device="cuda")
    w = torch.empty(2, 4, dtype=torch.float32, device="cuda")
    lib = load_library()
    assert lib.moe_route_noalloc(x.data_ptr(), g.data_ptr(), None, 2, 11520, 64, 4, ids.data_ptr(), w.data_ptr(),
                                 None) == UNSUPPORTED
