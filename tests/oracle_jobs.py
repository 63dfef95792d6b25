"""Worker-process jobs of the parallel oracle runs in the GPU parity tests.

Imports only numpy and the oracle, so that spawned workers start quickly.
Each job is one expert of the oracle's forward: its NVFP4 weights are
quantized from the bf16 bit patterns passed in, and ``oracle.moe.expert_rows``
runs the expert on its already-quantized input rows.  The parent process
does the routing, the per-token quantization and the finalize with the same
oracle functions ``oracle.moe.moe_forward`` uses, so the assembled result is
that function's, expert by expert.

Optionally the job also runs the expert's second GEMM on the GPU's own
requantized intermediate of the same rows (``oracle.moe.expert_w2``), and
returns the oracle's intermediate so that the parent can count the blocks
whose requantization decisions differ.
"""

from __future__ import annotations

import numpy as np

from oracle import moe as omoe
from oracle import nvfp4 as onv


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def expert_job(args):
    """(w13 bf16 bits [2I, H], w2 bf16 bits [H, I], x codes [n, H], x block
    scales [n, H/16], x global scales [n], GPU intermediate or None) -> dict
    with the expert's FP32 output rows ``y2`` [n, H] and the global scales of
    its requantized intermediate ``h_gs`` [n]; with a GPU intermediate (codes
    [n, I], block scales [n, I/16], global scales [n]) also ``y2_gpu_h`` (the
    second GEMM on it) and the oracle's ``h_codes`` / ``h_sf``."""
    w13_bits, w2_bits, codes, sf, gs, h_gpu = args
    c13, s13, g13 = onv.quantize_tensor(bf16_bits_to_f32(w13_bits))
    c2, s2, g2 = onv.quantize_tensor(bf16_bits_to_f32(w2_bits))
    q13 = omoe.QuantWeights(c13[None], s13[None], np.array([g13], np.float32))
    q2 = omoe.QuantWeights(c2[None], s2[None], np.array([g2], np.float32))
    r = omoe.expert_rows(codes, sf, gs, q13, q2, 0)
    out = {"y2": r["y2"], "h_gs": r["h_gs"]}
    if h_gpu is not None:
        hc, hs, hg = h_gpu
        out["y2_gpu_h"] = omoe.expert_w2(hc, hs, hg, q2, 0)
        out["h_codes"], out["h_sf"] = r["h_codes"], r["h_sf"]
    return out
