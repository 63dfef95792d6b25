"""Shared helpers of the GPU parity tests: the library handle, oracle runs
(cached per session), and the output tolerance.

Tolerance (the stated reading of "max|err| <= 2e-2 rms(ref) plus elementwise
relative error <= 5e-2"): every element satisfies
|gpu - ref| <= 2e-2 * rms(ref) + 5e-2 * |ref|, and every output is finite.
The same check is also applied row by row with the row's own rms, which is
stricter for the small rows of the per-token-scale stress inputs.
"""

from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import synthetic
from oracle import moe as omoe
from oracle import nvfp4 as onv

ABS_RMS = 2e-2
REL = 5e-2


def have_gpu() -> bool:
    return torch.cuda.is_available()


@functools.lru_cache(maxsize=None)
def built():
    from nvfp4_token_quantized_gb300 import build

    return build()


def tolerance_report(got: np.ndarray, ref: np.ndarray, per_row: bool = True):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(got - ref)
    ok_global = bool(np.all(err <= ABS_RMS * rms + REL * np.abs(ref)))
    row_rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True)) if ref.ndim == 2 else rms
    ok_rows = bool(np.all(err <= ABS_RMS * row_rms + REL * np.abs(ref)))
    return dict(finite=bool(np.isfinite(got).all()), ok=ok_global, ok_rows=ok_rows,
                max_err=float(err.max()) if err.size else 0.0, rms=rms,
                max_err_over_rms=float(err.max() / rms) if err.size and rms > 0 else 0.0)


def assert_close(got, ref, per_row=True, what="output"):
    r = tolerance_report(got, ref)
    assert r["finite"], f"{what}: non-finite values"
    assert r["ok"], f"{what}: outside tolerance {r}"
    if per_row:
        assert r["ok_rows"], f"{what}: outside per-row tolerance {r}"
    return r


@functools.lru_cache(maxsize=8)
def workload(name: str, T=None, seed: int = 0, weight_seed=None):
    return synthetic.make_workload(name, T=T, seed=seed, weight_seed=weight_seed)


_POOL = None


def _pool():
    # spawn, never fork: the parent may already hold a CUDA context
    global _POOL
    if _POOL is None:
        import concurrent.futures as cf
        import multiprocessing as mp
        import os as _os

        _POOL = cf.ProcessPoolExecutor(max_workers=max(1, min(16, (_os.cpu_count() or 2) - 1)),
                                       mp_context=mp.get_context("spawn"))
    return _POOL


def quantize_experts(w: torch.Tensor, experts) -> omoe.QuantWeights:
    """Oracle quantization of the listed experts of w [E, N, K] (others left
    zero with gs = 1), one expert per worker process."""
    E, N, Kd = w.shape
    codes = np.zeros((E, N, Kd), np.uint8)
    sf = np.zeros((E, N, Kd // 16), np.uint8)
    gs = np.ones(E, np.float32)
    experts = [int(e) for e in experts]
    arrays = [omoe.as_f32(w[e]) for e in experts]
    if len(experts) <= 1:
        results = [onv.quantize_tensor(a) for a in arrays]
    else:
        # workers import only the oracle's numpy code
        results = list(_pool().map(onv.quantize_tensor, arrays))
    for e, (c, s_, g) in zip(experts, results):
        codes[e], sf[e], gs[e] = c, s_, g
    return omoe.QuantWeights(codes, sf, gs)


def oracle_route(wl, tokens=None):
    x = omoe.as_f32(wl.x)
    tok = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    bias = None if wl.bias is None else wl.bias.numpy()
    logits = omoe.router_logits(x[tok], omoe.as_f32(wl.gate_w), bias)
    ids, w = omoe.topk_route(logits, wl.shape.K)
    return logits, ids, w


def oracle_forward(wl, tokens=None, static_scales=None):
    """Oracle forward for all tokens or a subset; only the experts those tokens
    route to are quantized.  static_scales: (x_gs, h_gs[E]) for the static
    per-tensor contract, or None for per-token scales."""
    x = omoe.as_f32(wl.x)
    wg = omoe.as_f32(wl.gate_w)
    bias = None if wl.bias is None else wl.bias.numpy()
    _, ids, _ = oracle_route(wl, tokens)
    experts = np.unique(ids)
    q13 = quantize_experts(wl.w13, experts)
    q2 = quantize_experts(wl.w2, experts)
    return omoe.moe_forward(x, wg, q13, q2, wl.shape.K, bias, tokens=tokens, static_scales=static_scales)


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


class ParallelResult:
    """Result of ``oracle_forward_parallel`` for n tokens.

    out       float32 [n, H]  the oracle's forward (bf16 values widened)
    ids       int32 [n, K]    its top-k choice
    h_gs      {(token, slot): float32} its intermediate's global scales
    With the GPU's intermediate given:
    out_gpu_h float32 [n, H]  the oracle's second GEMM and finalize applied to
                              the GPU's requantized intermediate (the same
                              requantization decisions on both sides)
    h_gs_gpu, h_gs_ref float32 [n, K]  the two sides' intermediate global scales
    flipped   bool [n, K]     rows whose intermediate codes or block scales
                              differ from the oracle's
    flipped_blocks, blocks    16-element blocks that differ, and all blocks
    """


def oracle_forward_parallel(wl, tokens, h_gpu=None):
    """``oracle_forward(wl, tokens)`` (per-token scales) computed expert by
    expert in worker processes: routing, per-token quantization and the
    finalize here, each expert's weight quantization and GEMMs in a worker
    (``tests/oracle_jobs.py``).

    ``h_gpu``: optionally the GPU's requantized intermediate of the whole
    batch, (packed codes [T*K, I/2], block scales [T*K, I/16], global scales
    [T*K]) indexed by token * K + slot (``MoE.debug_intermediate``).
    Returns a ``ParallelResult``."""
    from tests import oracle_jobs

    tok = np.asarray(tokens, dtype=np.int64)
    K, H = wl.shape.K, wl.shape.H
    _, ids, w = oracle_route(wl, tok)
    xs = omoe.as_f32(wl.x)[tok]
    codes, sf, gs = onv.quantize_rows(xs)
    if h_gpu is not None:
        hc_all, hs_all, hg_all = (np.asarray(a) for a in h_gpu)
    jobs, where = [], []
    for e in np.unique(ids):
        sel_t, sel_j = np.nonzero(ids == e)          # token-ascending, as the oracle's forward
        hj = None
        if h_gpu is not None:
            src = tok[sel_t] * K + sel_j
            hj = (onv.unpack_e2m1(hc_all[src]), hs_all[src], hg_all[src])
        jobs.append((_bf16_bits(wl.w13[int(e)]), _bf16_bits(wl.w2[int(e)]), codes[sel_t], sf[sel_t], gs[sel_t], hj))
        where.append((sel_t, sel_j))
    results = list(_pool().map(oracle_jobs.expert_job, jobs)) if len(jobs) > 1 else \
        [oracle_jobs.expert_job(j) for j in jobs]
    n = len(tok)
    y_rows = np.zeros((n, K, H), np.float32)
    res = ParallelResult()
    res.ids, res.h_gs = ids, {}
    if h_gpu is not None:
        y_gpu = np.zeros((n, K, H), np.float32)
        res.h_gs_ref = np.zeros((n, K), np.float32)
        res.h_gs_gpu = hg_all[tok[:, None] * K + np.arange(K)[None, :]].astype(np.float32)
        res.flipped = np.zeros((n, K), bool)
        res.flipped_blocks = res.blocks = 0
    for (sel_t, sel_j), r, job in zip(where, results, jobs):
        y_rows[sel_t, sel_j] = r["y2"]
        for i, (t, j) in enumerate(zip(sel_t, sel_j)):
            res.h_gs[(int(tok[t]), int(j))] = r["h_gs"][i]
        if h_gpu is not None:
            y_gpu[sel_t, sel_j] = r["y2_gpu_h"]
            res.h_gs_ref[sel_t, sel_j] = r["h_gs"]
            gc, gsf, _ = job[5]
            nb = gsf.shape[1]
            blk = (gc != r["h_codes"]).reshape(len(sel_t), nb, 16).any(2) | (gsf != r["h_sf"])
            res.flipped[sel_t, sel_j] = blk.any(1)
            res.flipped_blocks += int(blk.sum())
            res.blocks += blk.size
    res.out = onv.bf16_to_f32(onv.bf16_round(omoe.finalize(y_rows, w)))
    if h_gpu is not None:
        res.out_gpu_h = onv.bf16_to_f32(onv.bf16_round(omoe.finalize(y_gpu, w)))
    return res


def tile_covering_tokens(ids: np.ndarray, num_experts: int, tile_rows: int = 128):
    """Tokens whose rows include the first and the last row of every
    tile_rows-row GEMM tile of every expert with rows (each expert's ragged
    last tile included), in the expert-grouped, token-ordered row order of
    the permutation; ids int [T, K] is the whole batch's top-k choice."""
    ids = np.asarray(ids)
    K = ids.shape[1]
    off, src, _ = omoe.permute(ids, num_experts)
    toks = set()
    for e in range(num_experts):
        n = int(off[e + 1] - off[e])
        for r0 in range(0, n, tile_rows):
            for r in (r0, min(r0 + tile_rows, n) - 1):
                toks.add(int(src[off[e] + r]) // K)
    return np.array(sorted(toks), dtype=np.int64)


def sample_tokens(T: int, n: int, extra=()):
    """n evenly spread token indices (always the first and last) plus extras."""
    base = np.linspace(0, T - 1, min(n, T)).astype(np.int64)
    return np.unique(np.concatenate([base, np.asarray(list(extra), dtype=np.int64)]))


def to_dev(wl, dev="cuda:0"):
    return dict(x=wl.x.to(dev), gate_w=wl.gate_w.to(dev), w13=wl.w13.to(dev), w2=wl.w2.to(dev),
                bias=None if wl.bias is None else wl.bias.to(dev))


gpu = pytest.mark.gpu
needs_gpu = pytest.mark.skipif(not have_gpu(), reason="needs a CUDA device")
