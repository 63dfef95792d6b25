"""GPU parity of the building blocks, through the C ABI:

* the hardware E2M1 / E4M3 conversions the quantizer uses, against the
  oracle's encoders, exhaustively over every FP32 pattern where E2M1 makes a
  decision and densely for E4M3;
* the tcgen05 block-scaled FP4 GEMM main loop in isolation, against an FP64
  product of the decoded operands.
"""

import numpy as np
import pytest
import torch

from oracle import nvfp4 as onv
from tests.parity import built, gpu, needs_gpu

pytestmark = [gpu, needs_gpu]


def _cvt(vals: np.ndarray):
    from nvfp4_token_quantized_gb300 import moe_debug_convert

    built()
    x = torch.from_numpy(np.ascontiguousarray(vals, dtype=np.float32)).cuda()
    e2, e4 = moe_debug_convert(x)
    torch.cuda.synchronize()
    return e2.cpu().numpy(), e4.cpu().numpy()


def test_e2m1_conversion_exhaustive_decision_range():
    # every FP32 bit pattern in [2^-3, 2^3): all E2M1 thresholds lie inside;
    # below it everything rounds to 0, above it everything saturates
    lo = np.float32(0.125).view(np.uint32)
    hi = np.float32(8.0).view(np.uint32)
    step = 1 << 24
    for start in range(int(lo), int(hi), step):
        pats = np.arange(start, min(start + step, int(hi)), dtype=np.uint32)
        vals = pats.view(np.float32)
        vals = np.concatenate([vals, -vals[::97]])
        e2, _ = _cvt(vals)
        ref = onv.e2m1_encode(vals)
        bad = np.nonzero(e2 != ref)[0]
        assert bad.size == 0, f"{bad.size} mismatches, e.g. {vals[bad[:4]]}: hw {e2[bad[:4]]} oracle {ref[bad[:4]]}"


def test_e2m1_conversion_outside_range():
    rng = np.random.default_rng(0)
    small = np.exp2(rng.uniform(-149, -3, 200_000)).astype(np.float32)
    big = np.exp2(rng.uniform(3, 127.9, 200_000)).astype(np.float32)
    vals = np.concatenate([small, big, np.float32([0.0, -0.0, 3.4e38, 1e-45])])
    vals = np.concatenate([vals, -vals])
    e2, _ = _cvt(vals)
    assert np.array_equal(e2, onv.e2m1_encode(vals))


def test_e4m3_conversion_dense():
    # every 3rd FP32 pattern in [2^-12, 2^9) plus every E4M3 midpoint +-2 ulps
    lo = np.float32(2.0 ** -12).view(np.uint32)
    hi = np.float32(512.0).view(np.uint32)
    grid = onv.E4M3_VALUES[:127]
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    near = [mids]
    for d in (np.inf, 0.0):
        v = mids
        for _ in range(2):
            v = np.nextafter(v, np.float32(d))
            near.append(v)
    extra = np.concatenate(near + [np.float32([0.0, 448.0, 464.0, 480.0, 1e30, 1e-40])])
    step = 3 << 22
    for start in range(int(lo), int(hi), step):
        pats = np.arange(start, min(start + step, int(hi)), 3, dtype=np.uint32)
        vals = np.concatenate([pats.view(np.float32), extra])
        vals = np.concatenate([vals, -vals[::101]])
        _, e4 = _cvt(vals)
        ref = onv.e4m3_encode(vals)
        bad = np.nonzero(e4 != ref)[0]
        assert bad.size == 0, f"{bad.size} mismatches, e.g. {vals[bad[:4]]}: hw {e4[bad[:4]]} oracle {ref[bad[:4]]}"


def _gemm(a_codes, a_sf, b_codes, b_sf):
    from nvfp4_token_quantized_gb300 import moe_debug_block_scaled_gemm

    built()
    M, K = a_codes.shape
    N = b_codes.shape[0]
    ac = torch.from_numpy(onv.pack_e2m1(a_codes)).cuda()
    bc = torch.from_numpy(onv.pack_e2m1(b_codes)).cuda()
    asf = torch.from_numpy(np.ascontiguousarray(a_sf)).cuda()
    bsf = torch.from_numpy(np.ascontiguousarray(b_sf)).cuda()
    d = moe_debug_block_scaled_gemm(ac, asf, bc, bsf, M, N, K)
    return d.cpu().numpy().astype(np.float64)


def _ref(a_codes, a_sf, b_codes, b_sf):
    A = onv.decode_scaled(a_codes, a_sf)
    B = onv.decode_scaled(b_codes, b_sf)
    return A @ B.T, np.abs(A) @ np.abs(B).T


def _check(d, ref, mag, what):
    err = np.abs(d - ref)
    tol = 1e-5 * mag + 1e-30
    bad = err > tol
    if bad.any():
        r, c = np.nonzero(bad)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} wrong; first (row, col) {list(zip(r[:6], c[:6]))}; "
                             f"got {d[r[:3], c[:3]]} want {ref[r[:3], c[:3]]}; rows wrong {np.unique(r)[:12]} "
                             f"cols wrong {np.unique(c)[:12]}")


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 768)])
def test_block_scaled_gemm_unit_scales(M, N, K):
    rng = np.random.default_rng(M + N + K)
    a = rng.integers(0, 16, (M, K), dtype=np.uint8)
    b = rng.integers(0, 16, (N, K), dtype=np.uint8)
    sa = np.full((M, K // 16), 0x38, np.uint8)     # 1.0
    sb = np.full((N, K // 16), 0x38, np.uint8)
    ref, mag = _ref(a, sa, b, sb)
    _check(_gemm(a, sa, b, sb), ref, mag, "codes with unit block scales")


def test_block_scaled_gemm_scales_only():
    rng = np.random.default_rng(1)
    M, N, K = 128, 256, 512
    a = np.full((M, K), 2, np.uint8)               # 1.0
    b = np.full((N, K), 2, np.uint8)
    sa = rng.integers(0x20, 0x50, (M, K // 16), dtype=np.uint8)
    sb = rng.integers(0x20, 0x50, (N, K // 16), dtype=np.uint8)
    ref, mag = _ref(a, sa, b, sb)
    _check(_gemm(a, sa, b, sb), ref, mag, "block scales with unit codes")


def test_block_scaled_gemm_random():
    rng = np.random.default_rng(2)
    M, N, K = 384, 768, 1024
    a = rng.integers(0, 16, (M, K), dtype=np.uint8)
    b = rng.integers(0, 16, (N, K), dtype=np.uint8)
    sa = rng.integers(0x18, 0x58, (M, K // 16), dtype=np.uint8)
    sb = rng.integers(0x18, 0x58, (N, K // 16), dtype=np.uint8)
    ref, mag = _ref(a, sa, b, sb)
    _check(_gemm(a, sa, b, sb), ref, mag, "random operands and scales")
