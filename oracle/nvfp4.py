"""CPU oracle, part 1: the NVFP4 number formats and the quantizer.

TEST INFRASTRUCTURE.  This module is a plain, slow restatement of what the
per-token NVFP4 path computes, used only by ``tests/``, by
``__graft_entry__.smoke()`` and by the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``.  The library under test never imports it, and it never
imports the library.

Sources (the pages' titles; no formula is printed on them, so every numeric
rule below is a stated reading):

* "CuTe DSL backend gets per-token NVFP4 online quantization and reload",
  Implementation item 2 and the ``_make_per_token_global_scale`` snippet: the
  activation global scale is a dynamic FP32 value per token; data are E2M1
  codes with E4M3 block scale factors.
* Same page, Review ("numeric constants"): scale-factor vector size 16 and an
  ``e4m3_max`` constant.

Readings (the pages are silent on the arithmetic):

* gs = fl32(2688 / amax), 2688 = 448 (largest finite E4M3) x 6 (largest
  E2M1); amax == 0 gives gs = 1; a quotient that overflows is clamped to
  FLT_MAX.
* block scale: sf32 = fl32(fl32(amax_b * gs) / 6), sf = E4M3 round-to-nearest-
  even, saturating at 448, subnormals kept.
* element code: if dec(sf) == 0 every code of the block is +0; else
  q = fl32(gs / dec(sf)), v = fl32(x * q), code = E2M1 round-to-nearest-even,
  saturating at 6, the sign bit kept (so -0.1 gives 0x8).
* packing: element 2i in the low nibble, 2i+1 in the high nibble.
* dequant: dec(code) * dec(sf) / gs.

All FP32 steps are numpy float32 operations (IEEE single, round to nearest
even, subnormals kept), one operation at a time, exactly as written above.
"""

from __future__ import annotations

import numpy as np

F32 = np.float32
SF_VEC = 16                       # elements per E4M3 block scale
E2M1_MAX = 6.0
E4M3_MAX = 448.0
GS_NUMERATOR = F32(448.0 * 6.0)   # 2688
FLT_MAX = np.finfo(np.float32).max


# --------------------------------------------------------------------------
# E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf/nan.
# --------------------------------------------------------------------------

def e2m1_decode_table() -> np.ndarray:
    """Value of each of the 16 E2M1 codes, from the bit fields.

    exponent field 0 is subnormal: 0.m * 2^0; otherwise 1.m * 2^(e-1).
    """
    vals = np.zeros(16, dtype=np.float64)
    for code in range(16):
        s = -1.0 if code & 0x8 else 1.0
        e = (code >> 1) & 0x3
        m = code & 0x1
        mag = (m / 2.0) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
        vals[code] = s * mag
    return vals


E2M1_VALUES = e2m1_decode_table()


# --------------------------------------------------------------------------
# E4M3 (the "fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
# 0x7F / 0xFF are NaN, no infinities, largest finite 448.
# --------------------------------------------------------------------------

def e4m3_decode_table() -> np.ndarray:
    vals = np.zeros(256, dtype=np.float64)
    for b in range(256):
        s = -1.0 if b & 0x80 else 1.0
        e = (b >> 3) & 0xF
        m = b & 0x7
        if e == 0xF and m == 0x7:
            vals[b] = np.nan
        elif e == 0:
            vals[b] = s * (m / 8.0) * 2.0 ** -6
        else:
            vals[b] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


E4M3_VALUES = e4m3_decode_table()


def _round_to_grid_rne(a: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid value to each a >= 0, ties to the even index.

    ``grid`` is the ascending list of non-negative finite values of a format
    whose codes are consecutive integers in the same order (true for both E2M1
    and E4M3), so "even index" is "even mantissa".  Values above the last grid
    point saturate to it.
    """
    a = np.asarray(a, dtype=np.float64)
    hi = np.searchsorted(grid, a, side="left")          # first grid >= a
    hi = np.clip(hi, 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_lo = np.abs(a - grid[lo])
    d_hi = np.abs(grid[hi] - a)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(a >= grid[-1], len(grid) - 1, idx)   # saturate
    return idx.astype(np.int64)


_E2M1_GRID = E2M1_VALUES[:8]            # 0, .5, 1, 1.5, 2, 3, 4, 6
_E4M3_GRID = E4M3_VALUES[:127]          # 0x00 .. 0x7E, ascending


def e2m1_encode(v) -> np.ndarray:
    """FP32 -> E2M1 code, round to nearest even, saturating, sign kept."""
    v = np.asarray(v, dtype=np.float32)
    mag = _round_to_grid_rne(np.abs(v.astype(np.float64)), _E2M1_GRID)
    sign = np.signbit(v).astype(np.int64)
    return (mag | (sign << 3)).astype(np.uint8)


def e4m3_encode(v) -> np.ndarray:
    """FP32 -> E4M3 byte, round to nearest even, saturating at +-448."""
    v = np.asarray(v, dtype=np.float32)
    if np.isnan(v).any():
        raise ValueError("e4m3_encode: NaN input")
    mag = _round_to_grid_rne(np.abs(v.astype(np.float64)), _E4M3_GRID)
    sign = np.signbit(v).astype(np.int64)
    return (mag | (sign << 7)).astype(np.uint8)


def e2m1_decode(codes) -> np.ndarray:
    return E2M1_VALUES[np.asarray(codes, dtype=np.int64)]


def e4m3_decode(b) -> np.ndarray:
    return E4M3_VALUES[np.asarray(b, dtype=np.int64)]


# --------------------------------------------------------------------------
# Global scale, block scales and codes.
# --------------------------------------------------------------------------

def global_scale(amax) -> np.ndarray:
    """gs = fl32(2688 / amax); 1 where amax == 0; FLT_MAX where it overflows."""
    amax = np.asarray(amax, dtype=np.float32)
    with np.errstate(divide="ignore", over="ignore"):
        gs = np.where(amax > 0, GS_NUMERATOR / np.where(amax > 0, amax, F32(1)), F32(1)).astype(np.float32)
    gs = np.where(np.isinf(gs), F32(FLT_MAX), gs).astype(np.float32)
    return gs


def quantize_blocks(x: np.ndarray, gs: np.ndarray):
    """Block scales and codes of rows ``x`` (float32 [rows, K]) given one
    global scale per row (``gs`` float32 [rows]).

    Returns (codes uint8 [rows, K] one code per element, sf uint8 [rows, K/16]).
    """
    x = np.asarray(x, dtype=np.float32)
    rows, K = x.shape
    if K % SF_VEC:
        raise ValueError(f"K={K} is not a multiple of {SF_VEC}")
    gs = np.asarray(gs, dtype=np.float32).reshape(rows, 1)
    blocks = x.reshape(rows, K // SF_VEC, SF_VEC)
    amax_b = np.max(np.abs(blocks), axis=2)                       # float32, exact
    sf32 = (amax_b * gs) / F32(6.0)                              # two fl32 steps
    sf = e4m3_encode(sf32)
    sf_val = e4m3_decode(sf).astype(np.float32)                  # exact in fp32
    nonzero = sf_val > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(nonzero, gs / np.where(nonzero, sf_val, F32(1)), F32(0)).astype(np.float32)
    v = (blocks * q[:, :, None]).astype(np.float32)             # fl32(x * q)
    codes = e2m1_encode(v)
    codes = np.where(nonzero[:, :, None], codes, np.uint8(0)).astype(np.uint8)
    return codes.reshape(rows, K), sf


def quantize_rows(x: np.ndarray):
    """Per-row (per-token) quantization: one global scale per row.

    Returns (codes uint8 [rows, K], sf uint8 [rows, K/16], gs float32 [rows]).
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    gs = global_scale(amax)
    codes, sf = quantize_blocks(x, gs)
    return codes, sf, gs


def quantize_rows_static(x: np.ndarray, gs):
    """Per-tensor static quantization: every row uses the given global scale
    ``gs`` (a calibrated FP32 scalar) instead of one derived from the row's
    maximum.  Blocks whose scaled maximum exceeds the formats saturate (block
    scale 448, codes +-6).

    Returns (codes uint8 [rows, K], sf uint8 [rows, K/16], gs float32 [rows]).
    """
    x = np.asarray(x, dtype=np.float32)
    g = np.full(x.shape[0], np.float32(gs), dtype=np.float32)
    codes, sf = quantize_blocks(x, g)
    return codes, sf, g


def quantize_tensor(w: np.ndarray):
    """One global scale for the whole matrix (an expert's weight).

    Returns (codes uint8 [N, K], sf uint8 [N, K/16], gs float32 scalar).
    """
    w = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w)) if w.size else np.float32(0)
    gs = global_scale(np.float32(amax)).reshape(())
    codes, sf = quantize_blocks(w, np.full(w.shape[0], gs, dtype=np.float32))
    return codes, sf, np.float32(gs)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Two codes per byte along the last axis: element 2i low nibble, 2i+1 high."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] & 0xF) | ((codes[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def decode_scaled(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """dec(code) * dec(sf) in float64 (exact), without the global scale."""
    codes = np.asarray(codes)
    rows, K = codes.shape
    vals = e2m1_decode(codes).reshape(rows, K // SF_VEC, SF_VEC)
    scales = e4m3_decode(sf).reshape(rows, K // SF_VEC, 1)
    return (vals * scales).reshape(rows, K)


def dequantize(codes: np.ndarray, sf: np.ndarray, gs) -> np.ndarray:
    """dec(code) * dec(sf) / gs in float64, gs per row or scalar."""
    gs = np.asarray(gs, dtype=np.float64)
    if gs.ndim == 1:
        gs = gs[:, None]
    return decode_scaled(codes, sf) / gs


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit pattern (uint16), round to nearest even.

    Keep the upper 16 bits after adding 0x7FFF plus the lowest kept bit.
    Inputs must be finite.
    """
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if not np.isfinite(x).all():
        raise ValueError("bf16_round: non-finite input")
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    return ((bits + 0x7FFF + lsb) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32)
