"""CPU oracle, part 2: the routed-MoE forward with per-token NVFP4 activations.

TEST INFRASTRUCTURE.  Plain, slow restatement of the hot path, used only by
``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``.  It
shares no code with the CUDA library and never imports it.

Steps, in the order the pages list the fused MoE operations ("SM10X
Command-A-Plus decode 2.3x faster", Motivation: routing, expandInputRows,
activation and finalize around the expert GEMMs) and the per-token contract
("CuTe DSL backend gets per-token NVFP4 online quantization and reload",
Implementation item 2):

1. router: FP32 logits x.Wg (+ bias), top-k by logit, softmax weights of the
   chosen experts renormalised to sum to one;
2. expand / permute: rows grouped by expert, stable in token order;
3. per-token NVFP4 quantization of x (``oracle.nvfp4``);
4. grouped GEMM on w13 in FP64 over exactly decoded operands;
5. SwiGLU h = silu(gate) * up;
6. per-row NVFP4 requantization of h;
7. grouped GEMM on w2 in FP64;
8. finalize: top-k-weighted sum of each token's expert rows, rounded to bf16.

Readings where the pages give no arithmetic (each is also listed in the
design notes):

* router logits use a canonical FP32 order so that CPU and GPU pick the same
  experts bit for bit: H is cut into 8-element chunks; partial p (0..31)
  accumulates chunks c = p, p+32, p+64, ... in ascending order and elements
  inside a chunk in ascending order, each step one fused multiply-add
  acc <- fl32(acc + x*w) starting from +0; the 32 partials are then combined
  pairwise, partial p with partial p xor o for o = 16, 8, 4, 2, 1; the logit is
  the result, plus the bias (one FP32 add) when a bias is given.  H must be a
  multiple of 256.
* top-k is taken on the logits, larger logit first, ties to the lower expert
  index.  Weights: softmax over all E logits in FP64, the K chosen
  probabilities divided by their sum, rounded to FP32.
* the intermediate h is requantized per expanded row with a dynamic global
  scale (the same rules as the activations).  The pages keep a separate
  second-GEMM input scale but never say how it is formed; this is the reading
  that keeps the whole path per-token.
* GEMM outputs: FP64 sum of exactly decoded products, times
  1 / (gs_row * gs_expert) in FP64, rounded to FP32.  SwiGLU in FP64 from the
  FP32 gate/up values, rounded to FP32.
* finalize: out[t] = bf16( sum over j = 0..K-1 ascending of fl32(w_j * y_j) )
  with FP32 partial sums, the first term taken as is.
* rows [0, I) of w13[e] are the gate projection, rows [I, 2I) the up
  projection.

Optional shared expert ("SM10X Command-A-Plus decode 2.3x faster, BCG capture
memory -78%", the Cohere2MoE sparse-block listing: the shared experts read the
same post-norm input as the routed experts, their output is added to the
routed output, and the 'average' combination strategy halves the sum):

* the shared expert is one more NVFP4 SwiGLU MLP (w13s [2Is, H], w2s [H, Is],
  one global scale per tensor) on every token, with the same per-token
  quantized input as the routed experts and the same requantization of its
  intermediate (the pages do not say how it is quantized; this reading keeps
  one activation contract for the layer);
* combination in FP32 with one bf16 rounding at the end:
  out = bf16( fl32(routed + shared) ), or bf16( fl32(fl32(routed + shared)
  * 0.5) ) for 'average' (the pages add two bf16 tensors; the reading keeps
  FP32 until the single rounding the layer output needs).
"""

from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

from . import nvfp4

F32 = np.float32
CHUNK = 8        # elements per router chunk
PARTIALS = 32    # router partial sums


# --------------------------------------------------------------------------
# 1. Router
# --------------------------------------------------------------------------

def router_logits(x: np.ndarray, wg: np.ndarray, bias: Optional[np.ndarray] = None) -> np.ndarray:
    """FP32 router logits [T, E] in the canonical order described above.

    ``x`` float32 [T, H] and ``wg`` float32 [H, E] hold bf16 values.  Each
    fused multiply-add is evaluated in float64 and rounded once to float32
    (the float64 sum of a float32 accumulator and a bf16*bf16 product rounds
    to float32 exactly as a single-rounding FMA does).
    """
    x = np.asarray(x, dtype=np.float32)
    wg = np.asarray(wg, dtype=np.float32)
    T, H = x.shape
    E = wg.shape[1]
    if H % (CHUNK * PARTIALS):
        raise ValueError(f"H={H} must be a multiple of {CHUNK * PARTIALS}")
    x64 = x.astype(np.float64)
    w64 = wg.astype(np.float64)
    parts = np.zeros((PARTIALS, T, E), dtype=np.float32)
    for c in range(H // CHUNK):
        p = c % PARTIALS
        for k in range(CHUNK):
            h = CHUNK * c + k
            prod = x64[:, h, None] * w64[None, h, :]
            parts[p] = (parts[p].astype(np.float64) + prod).astype(np.float32)
    lane = np.arange(PARTIALS)
    for o in (16, 8, 4, 2, 1):
        parts = (parts + parts[lane ^ o]).astype(np.float32)
    logits = parts[0]
    if bias is not None:
        logits = (logits + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
    return logits


def topk_route(logits: np.ndarray, k: int):
    """Top-k experts per token and their renormalised softmax weights.

    Returns (ids int32 [T, k] in selection order, weights float32 [T, k]).
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError(f"top_k={k} out of range for E={E}")
    ids = np.zeros((T, k), dtype=np.int32)
    weights = np.zeros((T, k), dtype=np.float32)
    idx = np.arange(E)
    for t in range(T):
        order = np.lexsort((idx, -logits[t].astype(np.float64)))   # logit desc, index asc
        chosen = order[:k]
        l64 = logits[t].astype(np.float64)
        p = np.exp(l64 - l64.max())
        p = p / p.sum()
        pc = p[chosen]
        ids[t] = chosen
        weights[t] = (pc / pc.sum()).astype(np.float32)
    return ids, weights


# --------------------------------------------------------------------------
# 2. Expand / permute
# --------------------------------------------------------------------------

def permute(ids: np.ndarray, num_experts: int):
    """Expert-grouped row order, stable in token order.

    Returns (expert_offsets int32 [E+1], src_of_row int32 [T*K],
    row_of_src int32 [T*K]); src = t*K + j names slot j of token t, and row r
    of expert e lies in [expert_offsets[e], expert_offsets[e+1]).
    """
    ids = np.asarray(ids, dtype=np.int64)
    T, K = ids.shape
    src = np.arange(T * K)
    flat = ids.reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= num_experts):
        raise ValueError("expert id out of range")
    order = np.lexsort((src // K, flat))            # expert asc, then token asc
    counts = np.bincount(flat, minlength=num_experts)
    offsets = np.zeros(num_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    src_of_row = order.astype(np.int32)
    row_of_src = np.empty(T * K, dtype=np.int32)
    row_of_src[src_of_row] = np.arange(T * K, dtype=np.int32)
    return offsets.astype(np.int32), src_of_row, row_of_src


# --------------------------------------------------------------------------
# Weights, quantized once per expert
# --------------------------------------------------------------------------

@dataclasses.dataclass
class QuantWeights:
    """Per-expert NVFP4 weights: codes (one per element), E4M3 block scales
    along K, one FP32 global scale per expert."""

    codes: np.ndarray   # uint8 [E, N, K]
    sf: np.ndarray      # uint8 [E, N, K/16]
    gs: np.ndarray      # float32 [E]

    @property
    def num_experts(self) -> int:
        return int(self.codes.shape[0])


def quantize_weights(w: np.ndarray) -> QuantWeights:
    """Quantize expert weights ``w`` float32 [E, N, K] (bf16 values), one
    global scale per expert over the whole [N, K] matrix."""
    w = np.asarray(w, dtype=np.float32)
    E, N, K = w.shape
    codes = np.empty((E, N, K), dtype=np.uint8)
    sf = np.empty((E, N, K // nvfp4.SF_VEC), dtype=np.uint8)
    gs = np.empty(E, dtype=np.float32)
    for e in range(E):
        codes[e], sf[e], gs[e] = nvfp4.quantize_tensor(w[e])
    return QuantWeights(codes, sf, gs)


# --------------------------------------------------------------------------
# 4-7. Expert computation for one expert's rows
# --------------------------------------------------------------------------

def silu(g: np.ndarray) -> np.ndarray:
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def expert_rows(a_codes, a_sf, a_gs, w13: QuantWeights, w2: QuantWeights, e: int, h_gs_static=None):
    """Run one expert on already-quantized input rows.

    ``h_gs_static``: None for the per-row (dynamic) requantization of the
    SwiGLU output; otherwise the expert's calibrated FP32 global scale, used
    for all its rows (the static per-tensor contract).

    Returns a dict with the FP32 w13 output ``y1`` [n, 2I], the FP32 SwiGLU
    output ``h`` [n, I], its quantization (``h_codes``, ``h_sf``, ``h_gs``)
    and the FP32 w2 output ``y2`` [n, H].
    """
    A = nvfp4.decode_scaled(a_codes, a_sf)                       # [n, H] f64
    B = nvfp4.decode_scaled(w13.codes[e], w13.sf[e])             # [2I, H] f64
    acc = A @ B.T
    scale = 1.0 / (np.asarray(a_gs, np.float64)[:, None] * np.float64(w13.gs[e]))
    y1 = (acc * scale).astype(np.float32)
    I = y1.shape[1] // 2
    gate, up = y1[:, :I], y1[:, I:]
    h = (silu(gate) * up.astype(np.float64)).astype(np.float32)
    if h_gs_static is None:
        h_codes, h_sf, h_gs = nvfp4.quantize_rows(h)
    else:
        h_codes, h_sf, h_gs = nvfp4.quantize_rows_static(h, h_gs_static)
    y2 = expert_w2(h_codes, h_sf, h_gs, w2, e)
    return dict(y1=y1, h=h, h_codes=h_codes, h_sf=h_sf, h_gs=h_gs, y2=y2)


def expert_w2(h_codes, h_sf, h_gs, w2: QuantWeights, e: int) -> np.ndarray:
    """The second GEMM of expert ``e`` on quantized intermediate rows (codes
    [n, I], block scales [n, I/16], global scales [n]): the FP32 output
    [n, H], from FP64 sums over the exactly decoded operands."""
    A2 = nvfp4.decode_scaled(h_codes, h_sf)                      # [n, I]
    B2 = nvfp4.decode_scaled(w2.codes[e], w2.sf[e])              # [H, I]
    acc2 = A2 @ B2.T
    scale2 = 1.0 / (np.asarray(h_gs, np.float64)[:, None] * np.float64(w2.gs[e]))
    return (acc2 * scale2).astype(np.float32)


def finalize(y_rows: np.ndarray, weights: np.ndarray) -> np.ndarray:
    """out = sum_j fl32(w_j * y_j) in ascending j with FP32 partial sums.

    ``y_rows`` float32 [T, K, H] (row j of token t), ``weights`` float32
    [T, K].  Returns float32 [T, H] (before the bf16 rounding).
    """
    y_rows = np.asarray(y_rows, dtype=np.float32)
    weights = np.asarray(weights, dtype=np.float32)
    acc = (weights[:, 0, None] * y_rows[:, 0, :]).astype(np.float32)
    for j in range(1, y_rows.shape[1]):
        acc = (acc + (weights[:, j, None] * y_rows[:, j, :]).astype(np.float32)).astype(np.float32)
    return acc


# --------------------------------------------------------------------------
# Whole forward
# --------------------------------------------------------------------------

@dataclasses.dataclass
class ForwardResult:
    out_bits: np.ndarray        # uint16 [n, H] bf16 bit patterns
    out: np.ndarray             # float32 [n, H] (bf16 values widened)
    out_f32: np.ndarray         # float32 [n, H] before bf16 rounding
    logits: np.ndarray          # float32 [n, E]
    ids: np.ndarray             # int32 [n, K]
    weights: np.ndarray         # float32 [n, K]
    x_codes: np.ndarray         # uint8 [n, H]
    x_sf: np.ndarray            # uint8 [n, H/16]
    x_gs: np.ndarray            # float32 [n]
    tokens: np.ndarray          # int64 [n] token indices computed
    h_gs: dict                  # (t, j) -> float32 requant global scale
    y2: dict                    # (t, j) -> float32 [H]


def shared_expert_rows(x_codes, x_sf, x_gs, w13s: QuantWeights, w2s: QuantWeights) -> np.ndarray:
    """The shared expert on every token's quantized input: the FP32 w2
    output [n, H] of its NVFP4 SwiGLU MLP (one expert, weight 1)."""
    return expert_rows(x_codes, x_sf, x_gs, w13s, w2s, 0)["y2"]


def combine_shared(routed_f32: np.ndarray, shared_f32: np.ndarray, average: bool) -> np.ndarray:
    """fl32(routed + shared), halved (one more FP32 rounding) for 'average'."""
    s = (np.asarray(routed_f32, np.float32) + np.asarray(shared_f32, np.float32)).astype(np.float32)
    if average:
        s = (s * np.float32(0.5)).astype(np.float32)
    return s


def moe_forward(x: np.ndarray, wg: np.ndarray, w13: QuantWeights, w2: QuantWeights,
                top_k: int, bias: Optional[np.ndarray] = None,
                tokens: Optional[Sequence[int]] = None, static_scales=None,
                shared=None, shared_average: bool = False) -> ForwardResult:
    """Forward of the routed MoE layer for all tokens, or for ``tokens`` only.

    Tokens are independent in this layer, so a subset gives the same rows as
    the full batch (the permutation is needed only by the GPU's layout).
    ``x`` float32 [T, H] and ``wg`` float32 [H, E] hold bf16 values.

    ``static_scales``: None for the per-token contract (activation global
    scales from each token's and each expanded row's maximum), or a pair
    (x_gs, h_gs) for the per-tensor static contract the pages keep separate
    ("CuTe DSL backend gets per-token NVFP4 online quantization and reload",
    Summary and Implementation item 2): one calibrated FP32 global scale for
    the first GEMM's input, and one per expert (``h_gs`` [E]) for the second
    GEMM's input.

    ``shared``: None, or a pair (w13s, w2s) of single-expert QuantWeights for
    the shared expert, combined with the routed output by sum or, with
    ``shared_average``, by the average (see the module notes).
    """
    x = np.asarray(x, dtype=np.float32)
    tok = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens, dtype=np.int64)
    xs = x[tok]
    n, H = xs.shape
    logits = router_logits(xs, wg, bias)
    ids, weights = topk_route(logits, top_k)
    if static_scales is None:
        x_codes, x_sf, x_gs = nvfp4.quantize_rows(xs)
    else:
        x_codes, x_sf, x_gs = nvfp4.quantize_rows_static(xs, static_scales[0])
    y_rows = np.zeros((n, top_k, H), dtype=np.float32)
    h_gs, y2_map = {}, {}
    for e in range(w13.num_experts):
        sel_t, sel_j = np.nonzero(ids == e)          # token-ascending
        if sel_t.size == 0:
            continue
        h_static = None if static_scales is None else np.float32(np.asarray(static_scales[1])[e])
        r = expert_rows(x_codes[sel_t], x_sf[sel_t], x_gs[sel_t], w13, w2, e, h_static)
        y_rows[sel_t, sel_j] = r["y2"]
        for i, (t, j) in enumerate(zip(sel_t, sel_j)):
            h_gs[(int(tok[t]), int(j))] = r["h_gs"][i]
            y2_map[(int(tok[t]), int(j))] = r["y2"][i]
    out_f32 = finalize(y_rows, weights) if n else np.zeros((0, H), np.float32)
    if shared is not None and n:
        out_f32 = combine_shared(out_f32, shared_expert_rows(x_codes, x_sf, x_gs, shared[0], shared[1]),
                                 shared_average)
    bits = nvfp4.bf16_round(out_f32)
    return ForwardResult(out_bits=bits, out=nvfp4.bf16_to_f32(bits), out_f32=out_f32,
                         logits=logits, ids=ids, weights=weights, x_codes=x_codes,
                         x_sf=x_sf, x_gs=x_gs, tokens=tok, h_gs=h_gs, y2=y2_map)


def as_f32(t) -> np.ndarray:
    """A bf16 torch tensor (or any array) as float32 numpy."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu", torch.float32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float32)
