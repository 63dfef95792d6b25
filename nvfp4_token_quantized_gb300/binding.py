"""Thin ctypes binding of the C ABI in ``include/moe_nvfp4.h``.

Argument marshalling only: every step of the forward runs in the CUDA
library.  Functions carry the C names; ``MoE`` is a small owner object around
a handle.  If the library has not been built, loading raises - there is no
fallback of any kind.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import builder as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_TOO_MANY_TOKENS = 2
MOE_ERR_NOT_LOADED = 3
MOE_ERR_METADATA_CHANGED = 4
MOE_ERR_ALIAS = 5
MOE_ERR_CUDA = 6
MOE_ERR_DEVICE_TIMEOUT = 7
MOE_ERR_UNSUPPORTED = 8
MOE_FLAG_DETERMINISTIC = 1
MOE_FLAG_STATIC_ACT_SCALES = 2
MOE_FLAG_SHARED_AVERAGE = 4
MOE_FLAG_ACCURATE_SIGMOID = 8
MOE_DTYPE_BF16 = 1

EXPORTED = (
    "moe_create", "moe_destroy", "moe_load_weights", "moe_refresh_scales_inplace", "moe_forward",
    "moe_forward_ex", "moe_forward_host", "moe_get_workspace_bytes", "moe_get_last_error",
    "moe_status_string", "moe_get_status", "moe_debug_routing", "moe_debug_logits",
    "moe_debug_act_quant", "moe_debug_weight_quant", "moe_debug_intermediate", "moe_debug_buffer_ptrs",
    "moe_debug_convert", "moe_debug_block_scaled_gemm", "moe_set_stage_timing", "moe_get_stage_times",
    "moe_stage_name", "moe_route_noalloc", "moe_set_static_scales", "moe_load_shared_weights",
    "moe_debug_shared", "moe_debug_shared_act_quant",
)
MOE_ROUTE_NOALLOC_MAX_LOGITS = 1 << 20
MOE_NUM_STAGES = 7


class moe_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("num_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("max_num_tokens", ctypes.c_int), ("device", ctypes.c_int),
                ("flags", ctypes.c_uint), ("shared_inter", ctypes.c_int)]


class moe_weight_desc(ctypes.Structure):
    _fields_ = [("dims", ctypes.c_int64 * 3), ("dtype", ctypes.c_int), ("device", ctypes.c_int)]


class MoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


_LIB = None


def lib_path() -> str:
    return _build.LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load the built library (``build()`` must have run)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    P, I, U, L, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "moe_create": (I, [ctypes.POINTER(moe_config), ctypes.POINTER(P)]),
        "moe_destroy": (I, [P]),
        "moe_load_weights": (I, [P, P, ctypes.POINTER(moe_weight_desc), P, ctypes.POINTER(moe_weight_desc), P]),
        "moe_load_shared_weights": (I, [P, P, ctypes.POINTER(moe_weight_desc), P, ctypes.POINTER(moe_weight_desc),
                                        P]),
        "moe_refresh_scales_inplace": (I, [P, P, ctypes.POINTER(moe_weight_desc), P,
                                           ctypes.POINTER(moe_weight_desc), P]),
        "moe_forward": (I, [P, P, P, P, I, P]),
        "moe_forward_ex": (I, [P, P, P, P, P, I, P]),
        "moe_forward_host": (I, [P, P, P, P, P, I, P]),
        "moe_get_workspace_bytes": (S, [P]),
        "moe_get_last_error": (ctypes.c_char_p, [P]),
        "moe_status_string": (ctypes.c_char_p, [I]),
        "moe_get_status": (I, [P]),
        "moe_debug_routing": (I, [P, P, P, P, P, P]),
        "moe_debug_logits": (I, [P, P, P]),
        "moe_debug_act_quant": (I, [P, P, P, P, P]),
        "moe_debug_weight_quant": (I, [P, I, P, P, P, P]),
        "moe_debug_intermediate": (I, [P, P, P, P, P]),
        "moe_debug_buffer_ptrs": (I, [P, ctypes.POINTER(P), ctypes.POINTER(I)]),
        "moe_debug_convert": (I, [P, P, P, L, P]),
        "moe_debug_block_scaled_gemm": (I, [P, P, P, P, P, I, I, I, P]),
        "moe_set_stage_timing": (I, [P, I]),
        "moe_get_stage_times": (I, [P, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(I)]),
        "moe_stage_name": (ctypes.c_char_p, [I]),
        "moe_route_noalloc": (I, [P, P, P, I, I, I, I, P, P, P]),
        "moe_set_static_scales": (I, [P, P, P, P]),
        "moe_debug_shared": (I, [P, P, P, P, P, P]),
        "moe_debug_shared_act_quant": (I, [P, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _ = U
    _LIB = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().moe_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check_dev(t: torch.Tensor, dtype, name: str, device: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype or t.device.type != "cuda" or t.device.index != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor on cuda:{device}")


def _wdesc(t: torch.Tensor) -> moe_weight_desc:
    d = moe_weight_desc()
    for i in range(3):
        d.dims[i] = int(t.shape[i]) if t.dim() == 3 else -1
    d.dtype = MOE_DTYPE_BF16 if t.dtype == torch.bfloat16 else 0
    d.device = t.device.index if t.device.type == "cuda" else -1
    return d


# ---- functions with the C names (handles are ctypes c_void_p) ----

def moe_create(hidden: int, inter: int, num_experts: int, top_k: int, max_num_tokens: int, device: int = 0,
               flags: int = 0, shared_inter: int = 0) -> ctypes.c_void_p:
    lib = load_library()
    cfg = moe_config(hidden, inter, num_experts, top_k, max_num_tokens, device, flags, shared_inter)
    h = ctypes.c_void_p()
    st = lib.moe_create(ctypes.byref(cfg), ctypes.byref(h))
    if st != MOE_OK:
        raise MoEError(st, "moe_create failed")
    return h


def moe_destroy(h) -> None:
    load_library().moe_destroy(h)


def _raise(h, st: int):
    if st != MOE_OK:
        msg = load_library().moe_get_last_error(h).decode() if h else ""
        raise MoEError(st, msg)


def moe_load_weights(h, w13: torch.Tensor, w2: torch.Tensor, stream=None) -> None:
    d13, d2 = _wdesc(w13), _wdesc(w2)
    _raise(h, load_library().moe_load_weights(h, _ptr(w13), ctypes.byref(d13), _ptr(w2), ctypes.byref(d2),
                                              _stream(stream)))


def moe_load_shared_weights(h, w13s: torch.Tensor, w2s: torch.Tensor, stream=None) -> None:
    """The shared expert's bf16 weights: w13s [2*Is, H] (gate rows, then up rows), w2s [H, Is]."""
    w13s = w13s.unsqueeze(0) if w13s.dim() == 2 else w13s
    w2s = w2s.unsqueeze(0) if w2s.dim() == 2 else w2s
    d13, d2 = _wdesc(w13s), _wdesc(w2s)
    _raise(h, load_library().moe_load_shared_weights(h, _ptr(w13s), ctypes.byref(d13), _ptr(w2s), ctypes.byref(d2),
                                                     _stream(stream)))


def moe_refresh_scales_inplace(h, w13: torch.Tensor, w2: torch.Tensor, stream=None) -> None:
    d13, d2 = _wdesc(w13), _wdesc(w2)
    _raise(h, load_library().moe_refresh_scales_inplace(h, _ptr(w13), ctypes.byref(d13), _ptr(w2),
                                                        ctypes.byref(d2), _stream(stream)))


def moe_set_static_scales(h, x_gs: torch.Tensor, h_gs: torch.Tensor, stream=None) -> None:
    """Calibrated global scales of the static per-tensor contract: x_gs float32
    [1] (the w13 input, all tokens), h_gs float32 [E] (each expert's w2 input),
    CUDA tensors on the handle's device."""
    _raise(h, load_library().moe_set_static_scales(h, _ptr(x_gs), _ptr(h_gs), _stream(stream)))


def moe_forward(h, x: torch.Tensor, gate_w: torch.Tensor, out: torch.Tensor, num_tokens: int, stream=None) -> None:
    _raise(h, load_library().moe_forward(h, _ptr(x), _ptr(gate_w), _ptr(out), int(num_tokens), _stream(stream)))


def moe_forward_ex(h, x, gate_w, gate_bias, out, num_tokens: int, stream=None) -> None:
    _raise(h, load_library().moe_forward_ex(h, _ptr(x), _ptr(gate_w), _ptr(gate_bias), _ptr(out), int(num_tokens),
                                            _stream(stream)))


def moe_forward_host(h, x, gate_w, gate_bias, out, num_tokens: int, stream=None) -> None:
    _raise(h, load_library().moe_forward_host(h, _ptr(x), _ptr(gate_w), _ptr(gate_bias), _ptr(out),
                                              int(num_tokens), _stream(stream)))


def moe_get_workspace_bytes(h) -> int:
    return int(load_library().moe_get_workspace_bytes(h))


def moe_get_last_error(h) -> str:
    return load_library().moe_get_last_error(h).decode()


def moe_get_status(h) -> int:
    return int(load_library().moe_get_status(h))


def moe_debug_convert(x: torch.Tensor, stream=None):
    """Hardware E2M1 / E4M3 conversion of a float32 CUDA tensor (uint8 codes)."""
    e2m1 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    e4m3 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    st = load_library().moe_debug_convert(_ptr(x), _ptr(e2m1), _ptr(e4m3), x.numel(), _stream(stream))
    if st != MOE_OK:
        raise MoEError(st, "moe_debug_convert")
    return e2m1, e4m3


def moe_debug_block_scaled_gemm(a_codes, a_sf, b_codes, b_sf, M: int, N: int, K: int, stream=None) -> torch.Tensor:
    d = torch.empty(M, N, dtype=torch.float32, device=a_codes.device)
    st = load_library().moe_debug_block_scaled_gemm(_ptr(a_codes), _ptr(a_sf), _ptr(b_codes), _ptr(b_sf), _ptr(d),
                                                    M, N, K, _stream(stream))
    if st != MOE_OK:
        raise MoEError(st, "moe_debug_block_scaled_gemm")
    return d


def moe_route_noalloc(x: torch.Tensor, gate_w: torch.Tensor, top_k: int, bias: Optional[torch.Tensor] = None,
                      topk_ids: Optional[torch.Tensor] = None, topk_w: Optional[torch.Tensor] = None,
                      stream=None):
    """Routing (logits, top-k, renormalised weights) with no handle and no
    device allocation inside the library call.  ``topk_ids`` (int32 [T, K])
    and ``topk_w`` (float32 [T, K]) may be passed in to be filled; otherwise
    they are created here, before the call.  Every tensor must be contiguous
    and on x's device, which must be the current CUDA device (the library
    launches there); anything else raises before the library is called."""
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a 2-D tensor [num_tokens, hidden]")
    if x.device.type != "cuda":
        raise ValueError("x must be a CUDA tensor")
    dev = x.device.index
    if dev != torch.cuda.current_device():
        raise ValueError(f"x is on cuda:{dev} but the current device is cuda:{torch.cuda.current_device()}")
    _check_dev(x, torch.bfloat16, "x", dev)
    _check_dev(gate_w, torch.bfloat16, "gate_w", dev)
    T, H = x.shape
    if gate_w.dim() != 2 or gate_w.shape[0] != H:
        raise ValueError(f"gate_w must be [hidden={H}, num_experts], got {tuple(gate_w.shape)}")
    E = gate_w.shape[1]
    if bias is not None:
        _check_dev(bias, torch.float32, "bias", dev)
        if tuple(bias.shape) != (E,):
            raise ValueError(f"bias must be [{E}], got {tuple(bias.shape)}")
    if topk_ids is None:
        topk_ids = torch.empty(T, top_k, dtype=torch.int32, device=x.device)
    if topk_w is None:
        topk_w = torch.empty(T, top_k, dtype=torch.float32, device=x.device)
    _check_dev(topk_ids, torch.int32, "topk_ids", dev)
    _check_dev(topk_w, torch.float32, "topk_w", dev)
    for name, t in (("topk_ids", topk_ids), ("topk_w", topk_w)):
        if tuple(t.shape) != (T, top_k):
            raise ValueError(f"{name} must be [{T}, {top_k}], got {tuple(t.shape)}")
    st = load_library().moe_route_noalloc(_ptr(x), _ptr(gate_w), _ptr(bias), T, H, E, top_k, _ptr(topk_ids),
                                          _ptr(topk_w), _stream(stream))
    if st != MOE_OK:
        what = f"moe_route_noalloc(T={T}, H={H}, E={E}, K={top_k})"
        if st == MOE_ERR_TOO_MANY_TOKENS:
            what += f": T*E = {T * E} exceeds the fixed scratch of {MOE_ROUTE_NOALLOC_MAX_LOGITS} logits"
        raise MoEError(st, what)
    return topk_ids, topk_w


class MoE:
    """Owner of one library handle: a routed-MoE layer with fixed sizes."""

    def __init__(self, hidden: int, inter: int, num_experts: int, top_k: int, max_num_tokens: int,
                 device: int = 0, deterministic: bool = False, static_scales: bool = False,
                 shared_inter: int = 0, shared_average: bool = False, accurate_sigmoid: bool = False):
        self.H, self.I, self.E, self.K, self.Tmax = hidden, inter, num_experts, top_k, max_num_tokens
        self.device = device
        self.deterministic = deterministic
        self.static_scales = static_scales
        self.shared_inter, self.shared_average = shared_inter, shared_average
        flags = (MOE_FLAG_DETERMINISTIC if deterministic else 0) | (MOE_FLAG_STATIC_ACT_SCALES if static_scales else 0)
        flags |= MOE_FLAG_SHARED_AVERAGE if shared_average else 0
        flags |= MOE_FLAG_ACCURATE_SIGMOID if accurate_sigmoid else 0
        self.accurate_sigmoid = accurate_sigmoid
        self._h = moe_create(hidden, inter, num_experts, top_k, max_num_tokens, device, flags, shared_inter)
        self.last_T = None

    @classmethod
    def from_shape(cls, shape, device: int = 0, deterministic: Optional[bool] = None, max_num_tokens=None,
                   static_scales: bool = False, accurate_sigmoid: bool = False):
        return cls(shape.H, shape.I, shape.E, shape.K, max_num_tokens or shape.max_num_tokens, device,
                   shape.deterministic if deterministic is None else deterministic, static_scales,
                   accurate_sigmoid=accurate_sigmoid)

    def set_static_scales(self, x_gs: torch.Tensor, h_gs: torch.Tensor, stream=None):
        moe_set_static_scales(self._h, x_gs, h_gs, stream)

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            moe_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown
            pass

    def load_weights(self, w13: torch.Tensor, w2: torch.Tensor, stream=None):
        moe_load_weights(self._h, w13, w2, stream)

    def load_shared_weights(self, w13s: torch.Tensor, w2s: torch.Tensor, stream=None):
        moe_load_shared_weights(self._h, w13s, w2s, stream)

    def refresh_scales_inplace(self, w13: torch.Tensor, w2: torch.Tensor, stream=None):
        moe_refresh_scales_inplace(self._h, w13, w2, stream)

    def forward(self, x: torch.Tensor, gate_w: torch.Tensor, out: Optional[torch.Tensor] = None,
                bias: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        _check_dev(x, torch.bfloat16, "x", self.device)
        _check_dev(gate_w, torch.bfloat16, "gate_w", self.device)
        if bias is not None:
            _check_dev(bias, torch.float32, "bias", self.device)
        T = int(x.shape[0])
        if out is None:
            out = torch.empty_like(x)
        moe_forward_ex(self._h, x, gate_w, bias, out, T, stream)
        self.last_T = T
        return out

    def forward_host(self, x: torch.Tensor, gate_w: torch.Tensor, out: torch.Tensor,
                     bias: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        moe_forward_host(self._h, x, gate_w, bias, out, int(x.shape[0]), stream)
        return out

    @property
    def workspace_bytes(self) -> int:
        return moe_get_workspace_bytes(self._h)

    @property
    def status(self) -> int:
        return moe_get_status(self._h)

    def _dev(self, shape, dtype):
        return torch.empty(shape, dtype=dtype, device=f"cuda:{self.device}")

    def debug_routing(self, stream=None):
        T = self.last_T or 0
        ids = self._dev((T, self.K), torch.int32)
        w = self._dev((T, self.K), torch.float32)
        src = self._dev((T * self.K,), torch.int32)
        off = self._dev((self.E + 1,), torch.int32)
        _raise(self._h, load_library().moe_debug_routing(self._h, _ptr(ids), _ptr(w), _ptr(src), _ptr(off),
                                                         _stream(stream)))
        return dict(topk_ids=ids, topk_w=w, src_of_row=src, expert_offsets=off)

    def debug_logits(self, stream=None):
        T = self.last_T or 0
        l = self._dev((T, self.E), torch.float32)
        _raise(self._h, load_library().moe_debug_logits(self._h, _ptr(l), _stream(stream)))
        return l

    def debug_act_quant(self, stream=None):
        T = self.last_T or 0
        codes = self._dev((T, self.H // 2), torch.uint8)
        sf = self._dev((T, self.H // 16), torch.uint8)
        gs = self._dev((T,), torch.float32)
        _raise(self._h, load_library().moe_debug_act_quant(self._h, _ptr(codes), _ptr(sf), _ptr(gs), _stream(stream)))
        return codes, sf, gs

    def debug_weight_quant(self, which: int, stream=None):
        if which == 0:
            N, Kd = 2 * self.I, self.H
        else:
            N, Kd = self.H, self.I
        codes = self._dev((self.E, N, Kd // 2), torch.uint8)
        sf = self._dev((self.E, N, Kd // 16), torch.uint8)
        gs = self._dev((self.E,), torch.float32)
        _raise(self._h, load_library().moe_debug_weight_quant(self._h, which, _ptr(codes), _ptr(sf), _ptr(gs),
                                                              _stream(stream)))
        return codes, sf, gs

    def debug_intermediate(self, stream=None):
        R = (self.last_T or 0) * self.K
        codes = self._dev((R, self.I // 2), torch.uint8)
        sf = self._dev((R, self.I // 16), torch.uint8)
        gs = self._dev((R,), torch.float32)
        _raise(self._h, load_library().moe_debug_intermediate(self._h, _ptr(codes), _ptr(sf), _ptr(gs),
                                                              _stream(stream)))
        return codes, sf, gs

    def debug_shared(self, stream=None):
        """The shared expert's bf16 rows [T, H] and requantized intermediate
        (codes [T, Is/2], block scales [T, Is/16], global scales [T]) of the
        last forward."""
        T = self.last_T or 0
        rows = self._dev((T, self.H), torch.bfloat16)
        codes = self._dev((T, self.shared_inter // 2), torch.uint8)
        sf = self._dev((T, self.shared_inter // 16), torch.uint8)
        gs = self._dev((T,), torch.float32)
        _raise(self._h, load_library().moe_debug_shared(self._h, _ptr(rows), _ptr(codes), _ptr(sf), _ptr(gs),
                                                        _stream(stream)))
        return rows, codes, sf, gs

    def debug_shared_act_quant(self, stream=None):
        """The shared expert's per-token quantization of x in the last
        forward: codes [T, H/2], block scales [T, H/16], global scales [T]."""
        T = self.last_T or 0
        codes = self._dev((T, self.H // 2), torch.uint8)
        sf = self._dev((T, self.H // 16), torch.uint8)
        gs = self._dev((T,), torch.float32)
        _raise(self._h, load_library().moe_debug_shared_act_quant(self._h, _ptr(codes), _ptr(sf), _ptr(gs),
                                                                  _stream(stream)))
        return codes, sf, gs

    def set_stage_timing(self, enable: bool = True):
        _raise(self._h, load_library().moe_set_stage_timing(self._h, int(enable)))

    def stage_times(self) -> dict:
        """Durations (ms) of the stages of the last completed forward / replay."""
        lib = load_library()
        arr = (ctypes.c_float * MOE_NUM_STAGES)()
        n = ctypes.c_int(MOE_NUM_STAGES)
        _raise(self._h, lib.moe_get_stage_times(self._h, arr, ctypes.byref(n)))
        return {lib.moe_stage_name(i).decode(): float(arr[i]) for i in range(n.value)}

    def debug_buffer_ptrs(self):
        n = ctypes.c_int(0)
        lib = load_library()
        _raise(self._h, lib.moe_debug_buffer_ptrs(self._h, None, ctypes.byref(n)))
        arr = (ctypes.c_void_p * n.value)()
        _raise(self._h, lib.moe_debug_buffer_ptrs(self._h, arr, ctypes.byref(n)))
        return [int(p or 0) for p in arr]
