"""The C ABI without a GPU: the library builds, loads, exports every entry point
that ``include/moe_nvfp4.h`` declares, and its argument checks return status
codes (no compute call is made)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "moe_nvfp4.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from nvfp4_token_quantized_gb300 import build, load_library

    build()
    return load_library()


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("moe_create", "moe_load_weights", "moe_refresh_scales_inplace", "moe_forward",
                     "moe_forward_ex", "moe_destroy", "moe_get_workspace_bytes", "moe_get_last_error",
                     "moe_debug_routing", "moe_debug_act_quant", "moe_debug_weight_quant",
                     "moe_debug_buffer_ptrs"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} not exported"


def test_binding_covers_the_header():
    from nvfp4_token_quantized_gb300.binding import EXPORTED

    assert sorted(EXPORTED) == _declared()


def test_status_strings(lib):
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(2) == b"MOE_ERR_TOO_MANY_TOKENS"
    assert lib.moe_status_string(4) == b"MOE_ERR_METADATA_CHANGED"


def test_argument_checks_without_gpu(lib):
    from nvfp4_token_quantized_gb300.binding import moe_config

    h = ctypes.c_void_p()
    assert lib.moe_create(None, ctypes.byref(h)) == 1                    # INVALID_ARG
    bad = moe_config(255, 768, 128, 8, 64, 0, 0)                         # H not a multiple of 256
    assert lib.moe_create(ctypes.byref(bad), ctypes.byref(h)) == 8       # UNSUPPORTED
    assert not h.value
    neg = moe_config(2048, 768, 128, 8, 0, 0, 0)                         # no tokens
    assert lib.moe_create(ctypes.byref(neg), ctypes.byref(h)) == 1
    odd_shared = moe_config(2048, 768, 128, 8, 64, 0, 0, 100)            # Is not a multiple of 128
    assert lib.moe_create(ctypes.byref(odd_shared), ctypes.byref(h)) == 8
    static_shared = moe_config(2048, 768, 128, 8, 64, 0, 2, 256)         # shared expert with static scales
    assert lib.moe_create(ctypes.byref(static_shared), ctypes.byref(h)) == 8
    assert not h.value
    assert lib.moe_load_shared_weights(None, None, None, None, None, None) == 1
    assert lib.moe_forward(None, None, None, None, 4, None) == 1
    assert lib.moe_destroy(None) == 0
    assert lib.moe_get_workspace_bytes(None) == 0


def test_no_gpu_means_unsupported(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from nvfp4_token_quantized_gb300.binding import moe_config

    h = ctypes.c_void_p()
    cfg = moe_config(2048, 768, 128, 8, 64, 0, 0)
    assert lib.moe_create(ctypes.byref(cfg), ctypes.byref(h)) == 8
    assert not h.value


def test_python_binding_refuses_without_library(tmp_path, monkeypatch):
    import nvfp4_token_quantized_gb300.binding as b

    monkeypatch.setattr(b, "_LIB", None)
    monkeypatch.setattr(b, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        b.load_library()
